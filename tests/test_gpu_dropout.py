"""GPU parity of the fused dropout on y = dropout(Norm(o) * u) through the C
ABI, against the oracle on the same seeded inputs.

* the keep mask bit for bit: every element the oracle drops is exactly 0 on
  the GPU, every element it keeps is not, for row widths F = H d_v that take
  the 4-wide path (F % 128 == 0) and the 1-wide path;
* the kept values and the backward (dq, dk, dv, du, d-rab) within the
  path's bar (1e-2 x RMS for BF16 inputs, 1e-4 x RMS for FP32);
* p = 0 reproduces the run without dropout bit for bit, and another offset
  draws another mask;
* the full layer with dropout against the oracle layer.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from hstu_jagged_attention_02_gb300 import synth  # noqa: E402
from oracle import oracle as O  # noqa: E402
from tests.test_gpu_parity import TOL, check  # noqa: E402

pytestmark = pytest.mark.gpu


def _batch(seed, dtype, H, d, lengths):
    r = np.random.default_rng(seed)
    hist = np.asarray(lengths)
    return synth.make_batch(hist, H=H, d_qk=d, d_v=d, dtype=dtype, num_contexts=r.integers(0, 9, size=len(hist)),
                            num_targets=r.integers(0, 40, size=len(hist)), with_time=True, with_rab=True, seed=seed)


def _run(batch, dropout, out_dtype="fp32"):
    from hstu_jagged_attention_02_gb300.attention import Problem
    pr = Problem(batch, out_dtype=out_dtype, dropout=dropout)
    pr.forward()
    pr.backward()
    torch.cuda.synchronize()
    assert pr.device_error() == 0
    got = {"o": pr.o, "y": pr.y, "dq": pr.dq, "dk": pr.dk, "dv": pr.dvv, "du": pr.du,
           "d_rab_pos": pr.d_rab_pos, "d_rab_time": pr.d_rab_time}
    return {k: (None if v is None else v.double().cpu().numpy()) for k, v in got.items()}


def _oracle(batch, dropout):
    f = O.forward(batch, dropout=dropout)
    g = O.backward(batch, o=f["o"], dropout=dropout)
    return {"o": f["o"], "y": f["y"], "dq": g["dq"], "dk": g["dk"], "dv": g["dv"], "du": g["du"],
            "d_rab_pos": g["d_rab_pos"], "d_rab_time": g["d_rab_time"]}


def _mask_matches(y_gpu, batch, dropout):
    keep, _ = O.dropout_mask(batch.T, batch.H * batch.d_v, *dropout)
    y = y_gpu.reshape(keep.shape)
    assert np.all(y[~keep] == 0.0)
    assert np.all(y[keep] != 0.0)


# (dtype, H, d): F = 512 and 256 take the 4-wide path, F = 96 the 1-wide one
@pytest.mark.parametrize("dtype,H,d", [("bf16", 4, 128), ("bf16", 2, 128), ("fp32", 4, 64), ("fp32", 3, 32)])
@pytest.mark.parametrize("p", [0.1, 0.5])
def test_dropout_parity(dtype, H, d, p):
    b = _batch(61, dtype, H, d, [300, 77, 1, 190, 129])
    drop = (p, 1234 + H, 17)
    got = _run(b, drop)
    _mask_matches(got["y"], b, drop)
    check(got, _oracle(b, drop), TOL[dtype])


def test_dropout_p_zero_is_bit_identical_and_offsets_differ():
    b = _batch(62, "bf16", 4, 128, [200, 64, 333])
    plain = _run(b, None)
    zero = _run(b, (0.0, 99, 3))
    for k in plain:
        if plain[k] is not None and k not in ("dq", "d_rab_pos", "d_rab_time"):   # atomics: order varies
            assert np.array_equal(plain[k], zero[k]), k
    a = _run(b, (0.5, 7, 0))["y"]
    c = _run(b, (0.5, 7, 1))["y"]
    agree = float(np.mean((a == 0) == (c == 0)))
    assert 0.45 < agree < 0.55


def test_dropout_heavy_tailed_config():
    b = synth.by_name("heavy_tailed", 0)
    drop = (0.1, 2024, 5)
    got = _run(b, drop)
    _mask_matches(got["y"], b, drop)
    check(got, _oracle(b, drop), TOL["bf16"])


def test_layer_with_dropout():
    from tests.test_gpu_layer import _close, _np, _small_layer, layer_problem
    b = _small_layer(44, [300, 131, 77, 1, 260])
    drop = (0.2, 555, 9)
    pr = layer_problem(b, dropout=drop)
    pr.forward()
    pr.backward()
    torch.cuda.synchronize()
    assert pr.device_error() == 0
    f = O.layer_forward(b, act_dtype="bf16", dropout=drop)
    g = O.layer_backward(b, f, act_dtype="bf16")
    keep, _ = O.dropout_mask(b.T, b.H * b.d_v, *drop)
    y = _np(pr.y)
    assert np.all(y[~keep] == 0.0) and np.all(y[keep] != 0.0)
    x, dout = b.x.astype(np.float64), b.dout.astype(np.float64)
    _close("y", y, f["y"])
    _close("out - x", _np(pr.out) - x, f["out"] - x)
    _close("dx - dout", _np(pr.dx) - dout, g["dx"] - dout)
    _close("dw1", _np(pr.dw1), g["dw1"])
    _close("dw2", _np(pr.dw2), g["dw2"])
    _close("d_rab_pos", _np(pr.d_rab_pos), g["d_rab_pos"])
