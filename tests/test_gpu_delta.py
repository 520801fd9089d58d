"""GPU parity of the delta forward (KV-cached, candidate-only inference): the
candidates' o and y from hstu_attn_fwd_delta against the candidate rows of
the FP64 oracle's forward on the whole sequences (the definition the delta
call must reproduce).  Bar: max abs err <= 1e-2 x RMS (BF16 inputs)."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from hstu_jagged_attention_02_gb300 import binding as C  # noqa: E402
from hstu_jagged_attention_02_gb300 import synth  # noqa: E402
from oracle import oracle as O  # noqa: E402

pytestmark = pytest.mark.gpu


def _close(name, got, want, tol=1e-2):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert np.all(np.isfinite(got)), name
    rms = math.sqrt(float(np.mean(want * want)))
    err = float(np.max(np.abs(got - want)))
    assert err <= tol * rms, f"{name}: max abs err {err:.3e} > {tol:g} x rms {rms:.3e}"


def _run(b, flags=0):
    from hstu_jagged_attention_02_gb300.delta import DeltaProblem
    pr = DeltaProblem(b, flags=flags)
    pr.forward()
    torch.cuda.synchronize()
    assert pr.device_error() == 0
    rows = np.zeros(b.T, bool)
    rows[pr.cand_rows] = True
    f = O.forward(b, rows=rows)
    D = b.H * b.d_v
    _close("o", pr.o.double().cpu().numpy().reshape(-1, D), f["o"].reshape(b.T, D)[pr.cand_rows])
    _close("y", pr.y.double().cpu().numpy(), f["y"][pr.cand_rows])
    return pr


@pytest.mark.parametrize("d", [64, 128])
def test_delta_matches_candidate_rows_ragged(d):
    # contexts, targets from 0 to 150 (two candidate blocks), one sequence whose
    # cache is empty (all of it candidates)
    hist = [300, 131, 0, 77, 520, 12]
    nt = [40, 150, 20, 0, 64, 9]
    b = synth.make_batch(hist, H=2, d_qk=d, d_v=d, dtype="bf16", num_contexts=[3, 0, 0, 5, 8, 1],
                         num_targets=nt, seed=140 + d)
    _run(b)


def test_delta_wide_timestamps():
    b = synth.make_batch([400, 250], H=2, d_qk=128, d_v=128, dtype="bf16", num_targets=[70, 90], seed=151)
    ts, o = b.timestamps.copy(), b.offsets
    ts[int(o[0]) + 100:int(o[1])] += np.int64(1) << 35     # candidates and late history far ahead
    b.timestamps = ts
    _run(b)


def test_delta_ranking_scale():
    # 16 sequences of U[256, 3968] history + 8 context + 64 candidates, 4 heads x 128
    b = synth.ranking(0)
    pr = _run(b)
    assert pr.T_cand == 16 * 64


def test_delta_rejects_what_it_does_not_support():
    b = synth.make_batch([300, 200], H=2, d_qk=32, d_v=32, dtype="bf16", num_targets=[70, 90], seed=152)
    from hstu_jagged_attention_02_gb300.delta import DeltaProblem
    with pytest.raises(C.HSTUError) as e:
        DeltaProblem(b).forward()
    assert e.value.status == C.HSTU_ERR_UNSUPPORTED
