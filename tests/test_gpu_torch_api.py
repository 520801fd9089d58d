"""The PyTorch entry point (hstu_attention / HSTUAttnFunction) under
torch.autograd, against the FP64 oracle and against the direct C-ABI path.

The library computes y and every gradient in FP32 for BF16 inputs (the
default out_dtype); autograd then hands each gradient back in the dtype of
its input, so the BF16 q, k, v, u receive the FP32 results rounded once to
BF16.  Their bar is the parity bar plus that one rounding: max error
<= 1e-2 x RMS + 2^-8 x max |oracle|.  y and the bias-table gradients stay
FP32 and meet the parity bar itself.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from hstu_jagged_attention_02_gb300 import binding as C  # noqa: E402
from hstu_jagged_attention_02_gb300 import synth  # noqa: E402
from oracle import oracle as O  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _batch(seed):
    r = np.random.default_rng(seed)
    hist = np.array([1, 40, 129, 300, 700, 57])
    return synth.make_batch(hist, H=2, d_qk=128, d_v=128, dtype="bf16",
                            num_contexts=r.integers(0, 9, size=len(hist)),
                            num_targets=r.integers(0, 40, size=len(hist)), seed=seed)


def _max_err_ok(got, want, tol, extra_rel=0.0, name=""):
    got = got.detach().double().cpu().numpy().reshape(want.shape)
    rms = math.sqrt(float(np.mean(want * want)))
    err = float(np.max(np.abs(got - want)))
    bound = tol * rms + extra_rel * float(np.max(np.abs(want)))
    assert np.all(np.isfinite(got)), name
    assert err <= bound, f"{name}: max abs err {err:.3e} > {bound:.3e}"


def _run_autograd(b, u_fp32=False):
    from hstu_jagged_attention_02_gb300.attention import hstu_attention
    dev = torch.device("cuda")
    leaf = lambda a, dt: torch.tensor(np.asarray(a), device=dev, dtype=dt).requires_grad_(True)
    q, k, v = (leaf(x, torch.bfloat16) for x in (b.q, b.k, b.v))
    u = leaf(b.u, torch.float32 if u_fp32 else torch.bfloat16)
    rab_pos, rab_time = leaf(b.rab_pos, torch.float32), leaf(b.rab_time, torch.float32)
    off = torch.tensor(b.offsets, device=dev, dtype=torch.int64)
    nt = torch.tensor(b.num_targets, device=dev, dtype=torch.int32)
    nc = torch.tensor(b.num_contexts, device=dev, dtype=torch.int32)
    ts = torch.tensor(b.timestamps, device=dev, dtype=torch.int64)
    y = hstu_attention(q, k, v, u, off, b.max_seq_len, b.alpha, num_targets=nt, num_contexts=nc,
                       timestamps=ts, rab_pos=rab_pos, rab_time=rab_time)
    assert y.dtype == torch.float32
    dy = torch.tensor(np.asarray(b.dy, np.float32), device=dev).reshape(y.shape)
    (y * dy).sum().backward()
    torch.cuda.synchronize()
    return y, {"dq": q.grad, "dk": k.grad, "dv": v.grad, "du": u.grad,
               "d_rab_pos": rab_pos.grad, "d_rab_time": rab_time.grad}


@pytest.mark.parametrize("u_fp32", [False, True])
def test_autograd_matches_the_oracle(u_fp32):
    b = _batch(301)
    if u_fp32:   # a gate with more than 8 significant bits, read as FP32
        b.u = (np.asarray(b.u, np.float32) * np.float32(1.0 + 2.0 ** -12)).astype(np.float32)
    y, grads = _run_autograd(b, u_fp32=u_fp32)
    f = O.forward(b)
    g = O.backward(b, o=f["o"])
    _max_err_ok(y, f["y"], TOL, name="y")
    for name in ("d_rab_pos", "d_rab_time"):
        assert grads[name].dtype == torch.float32
        _max_err_ok(grads[name], g[name], TOL, name=name)
    for name in ("dq", "dk", "dv", "du"):
        extra = 0.0 if (name == "du" and u_fp32) else 2.0 ** -8
        _max_err_ok(grads[name], g[name], TOL, extra_rel=extra, name=name)


def test_autograd_is_the_c_abi_path():
    # the wrapper only marshals: y and the deterministic gradients equal the
    # direct C-ABI call's, rounded the same way
    from hstu_jagged_attention_02_gb300.attention import Problem
    b = _batch(302)
    y, grads = _run_autograd(b)
    pr = Problem(b, out_dtype="fp32")
    pr.forward()
    pr.backward()
    torch.cuda.synchronize()
    assert torch.equal(y, pr.y)
    for name, ref in (("dk", pr.dk), ("dv", pr.dvv), ("du", pr.du)):
        assert torch.equal(grads[name], ref.to(torch.bfloat16)), name


def test_bf16_outputs_on_request():
    from hstu_jagged_attention_02_gb300.attention import hstu_attention
    b = _batch(303)
    dev = torch.device("cuda")
    t = lambda a, dt: torch.tensor(np.asarray(a), device=dev, dtype=dt)
    y = hstu_attention(t(b.q, torch.bfloat16), t(b.k, torch.bfloat16), t(b.v, torch.bfloat16),
                       t(b.u, torch.bfloat16), t(b.offsets, torch.int64), b.max_seq_len, b.alpha,
                       num_targets=t(b.num_targets, torch.int32), num_contexts=t(b.num_contexts, torch.int32),
                       timestamps=t(b.timestamps, torch.int64), rab_pos=t(b.rab_pos, torch.float32),
                       rab_time=t(b.rab_time, torch.float32), out_dtype="bf16")
    torch.cuda.synchronize()
    assert y.dtype == torch.bfloat16
    f = O.forward(b)
    _max_err_ok(y, f["y"], TOL, extra_rel=2.0 ** -8, name="y")
