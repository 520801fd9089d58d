"""The forward entry point that allocates nothing (hstu_attn_fwd_noalloc).

It exists for callers that are not allowed to allocate device memory -- a
framework that owns all device memory through its own pool, a latency-bound
server that cannot afford an allocation, an integration with no allocator --
and takes its scratch from a buffer built into the library instead of a
caller workspace.  These tests call it through the C ABI and compare it with
the ordinary workspace forward (bit for bit: both run the same deterministic
kernels on the same plan) and with the FP64 oracle.  This file is collected
last on purpose.
"""
import math

import numpy as np
import pytest

from hstu_jagged_attention_02_gb300 import binding as C
from hstu_jagged_attention_02_gb300 import synth

TOL_BF16 = 1e-2   # max abs error <= 1e-2 x RMS of the oracle output, as for BF16 parity


def test_noalloc_rejects_problems_beyond_its_buffer():
    # host-side check, nothing is launched: 2M tokens need more than 1 MiB of plan scratch
    d = C.make_desc(dtype="bf16", out_dtype="fp32", B=8, H=4, d_qk=128, d_v=128,
                    total_tokens=2_000_000, max_seq_len=300_000 // 4, alpha=0.1)
    args = C.hstu_attn_fwd_args()
    for name in ("seq_offsets", "q", "k", "v", "o"):
        setattr(args, name, 4096)
    with pytest.raises(C.HSTUError) as e:
        C.hstu_attn_fwd_noalloc(d, args, None)
    assert e.value.status == C.HSTU_ERR_WORKSPACE
    assert "bytes of forward scratch" in C.hstu_last_error_detail()


def _close_to_oracle(got, want, tol):
    got = got.double().cpu().numpy().reshape(want.shape)
    rms = math.sqrt(float(np.mean(want * want)))
    assert np.all(np.isfinite(got))
    assert float(np.max(np.abs(got - want))) <= tol * rms


def _batches():
    small = synth.make_batch([40, 300, 7, 129], H=2, d_qk=64, d_v=64, dtype="bf16",
                             num_contexts=[2, 4, 0, 1], num_targets=[3, 16, 2, 8], seed=77)
    large = synth.heavy_tailed(5)
    return small, large


@pytest.mark.gpu
@pytest.mark.parametrize("order", ["small_first", "large_first"])
def test_noalloc_forward_matches_the_workspace_forward_twice_in_a_row(order):
    torch = pytest.importorskip("torch")
    from hstu_jagged_attention_02_gb300.attention import Problem, _stream_handle
    from oracle import oracle as O
    small, large = _batches()
    batches = [small, large] if order == "small_first" else [large, small]
    # two different problems, one call each, back to back: the second call
    # reuses the built-in buffer the first one left behind (a larger plan
    # after a smaller one, or the reverse)
    probs = [Problem(b, out_dtype="fp32") for b in batches]
    refs = []
    for pr in probs:
        pr.forward()
        torch.cuda.synchronize()
        assert pr.device_error() == 0
        refs.append((pr.o.clone(), pr.y.clone()))
        pr.o.fill_(float("nan"))
        pr.y.fill_(float("nan"))
    for pr in probs:
        code = C.hstu_attn_fwd_noalloc(pr.desc, pr.fwd_args, _stream_handle())
        assert code == 0
    torch.cuda.synchronize()
    for pr, (o_ref, y_ref) in zip(probs, refs):
        assert torch.equal(pr.o, o_ref)
        assert torch.equal(pr.y, y_ref)
    # the small problem against the oracle directly
    i = batches.index(small)
    f = O.forward(small)
    _close_to_oracle(probs[i].o, f["o"], TOL_BF16)
    _close_to_oracle(probs[i].y, f["y"], TOL_BF16)
