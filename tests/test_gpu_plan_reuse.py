"""One planner launch per training step: the forward called with
HSTU_FLAG_PLAN_BWD plans the backward too (a second CTA of its planner
launch) and the backward called with HSTU_FLAG_REUSE_PLAN uses that plan.

The results are checked against the FP64 oracle at the path's bar; a kept
plan that does not match the backward's descriptor or metadata must be
refused on the device (HSTU_ERR_DEVICE_CHECK, no work done), never used."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from hstu_jagged_attention_02_gb300 import binding as C  # noqa: E402
from hstu_jagged_attention_02_gb300 import synth  # noqa: E402
from hstu_jagged_attention_02_gb300.attention import Problem  # noqa: E402

from tests.test_gpu_parity import TOL, _ragged_batch, check, run_oracle  # noqa: E402

pytestmark = pytest.mark.gpu


def _grads(pr):
    out = {"o": pr.o, "y": pr.y, "dq": pr.dq, "dk": pr.dk, "dv": pr.dvv, "du": pr.du,
           "d_rab_pos": pr.d_rab_pos, "d_rab_time": pr.d_rab_time}
    return {k: (None if v is None else v.double().cpu().numpy()) for k, v in out.items()}


@pytest.mark.parametrize("case", ["heavy_tailed", "ragged_bf16", "ragged_fp32"])
def test_plan_once_matches_the_oracle(case):
    if case == "heavy_tailed":
        b = synth.by_name("heavy_tailed", 3)   # the batch with the longest work item
    else:
        dtype = case.split("_")[1]
        b = _ragged_batch(dtype, 128, seed=140)
    pr = Problem(b, plan_once=True)
    pr.forward()
    fwd_launches = C.hstu_last_launch_count()
    pr.backward()
    bwd_launches = C.hstu_last_launch_count()
    torch.cuda.synchronize()
    assert pr.device_error() == 0
    # planner + attention + norm-gate forward; norm-gate + attention backward
    assert (fwd_launches, bwd_launches) == (3, 2)
    check(_grads(pr), run_oracle(b), TOL[b.dtype])


def test_kept_plan_serves_repeated_backwards():
    b = _ragged_batch("bf16", 128, seed=141)
    pr = Problem(b, plan_once=True)
    pr.forward()
    pr.backward()
    torch.cuda.synchronize()
    first = _grads(pr)
    pr.backward()   # the work counter is re-armed by the check
    torch.cuda.synchronize()
    assert pr.device_error() == 0
    second = _grads(pr)
    want = run_oracle(b)
    check(first, want, TOL["bf16"])
    check(second, want, TOL["bf16"])
    # dq is summed by reduce-adds in no fixed order; everything else repeats exactly
    for k in ("dk", "dv", "du"):
        assert np.array_equal(first[k], second[k]), k


def _bwd_into(pr_ws, pr_args, flags):
    """pr_args' backward on pr_ws's workspace, with extra flags."""
    d = C.hstu_attn_desc.from_buffer_copy(pr_args.desc)
    d.flags |= flags
    C.hstu_attn_bwd(d, pr_args.bwd_args, pr_ws.ws.data_ptr(), pr_ws.ws_bytes, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("other", ["offsets", "targets", "timestamps", "fewer_tokens", "simt_path"])
def test_mismatched_kept_plan_is_refused(other):
    lengths = [200, 130, 64, 300, 17]
    a = _ragged_batch("bf16", 128, seed=142, lengths=lengths)
    pa = Problem(a, plan_once=True)
    pa.forward()
    flags = 0
    if other == "offsets":      # same B, T and longest sequence; two lengths swapped
        b = _ragged_batch("bf16", 128, seed=142, lengths=[130, 200, 64, 300, 17])
        assert (b.T, b.max_seq_len) == (a.T, a.max_seq_len)
    elif other == "targets":    # same lengths: one target of a sequence becomes history
        nt = a.num_targets.astype(np.int64).copy()
        hist = np.array(lengths, np.int64)
        j = int(np.flatnonzero(nt)[0])
        nt[j] -= 1
        hist[j] += 1
        b = synth.make_batch(hist, H=2, d_qk=128, d_v=128, dtype="bf16", num_contexts=a.num_contexts,
                             num_targets=nt, seed=142)
        assert np.array_equal(b.offsets, a.offsets)
    elif other == "timestamps":
        b = _ragged_batch("bf16", 128, seed=142, lengths=lengths)
        b.timestamps = b.timestamps + 7
    elif other == "fewer_tokens":
        b = _ragged_batch("bf16", 128, seed=142, lengths=lengths[:-1] + [5])
    else:                       # same metadata, the CUDA-core backward's tiling
        b = a
        flags = C.HSTU_FLAG_FORCE_SIMT
    pb = Problem(b)
    assert pb.ws_bytes <= pa.ws_bytes
    _bwd_into(pa, pb, C.HSTU_FLAG_REUSE_PLAN | flags)
    torch.cuda.synchronize()
    assert pa.device_error() == C.HSTU_ERR_DEVICE_CHECK
    # nothing was computed: the zeroed accumulators stay zero
    assert float(pb.d_rab_pos.abs().max()) == 0.0


def test_plain_forward_voids_the_kept_plan():
    b = _ragged_batch("bf16", 128, seed=144)
    pr = Problem(b, plan_once=True)
    pr.forward()
    C.hstu_attn_fwd(pr.desc, pr.fwd_args, pr.ws.data_ptr(), pr.ws_bytes, torch.cuda.current_stream().cuda_stream)
    pr.backward()
    torch.cuda.synchronize()
    assert pr.device_error() == C.HSTU_ERR_DEVICE_CHECK
    # a matching pair afterwards works again
    pr.forward()
    pr.backward()
    torch.cuda.synchronize()
    assert pr.device_error() == 0
    check(_grads(pr), run_oracle(b), TOL["bf16"])


def test_packed_inputs_match_the_oracle():
    # the benchmark's step: every input in one device buffer, one planner launch
    b = _ragged_batch("bf16", 128, seed=150)
    pr = Problem(b, plan_once=True, packed_inputs=True)
    base = pr.input_buffer.data_ptr()
    for t in (pr.offsets, pr.timestamps, pr.q, pr.k, pr.v, pr.u, pr.dy):
        assert base <= t.data_ptr() < base + pr.input_buffer.numel() and t.data_ptr() % 256 == 0
    pr.forward()
    pr.backward()
    torch.cuda.synchronize()
    assert pr.device_error() == 0
    check(_grads(pr), run_oracle(b), TOL["bf16"])
