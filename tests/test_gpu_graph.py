"""The path is stream-ordered and CUDA-graph capturable: the forward and
backward (attention, with and without dropout; the full layer) are captured
into one graph, replayed, and give the eager results.

Outputs written by plain stores must match bit for bit.  dq and d-rab are
summed with atomics in a run-dependent order, and the layer's dx, dW1, dW2
inherit that through dZ1, so those are compared to 1e-4 of their RMS.
"""
import math

import pytest

torch = pytest.importorskip("torch")

from hstu_jagged_attention_02_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

ATOMIC = {"dq", "d_rab_pos", "d_rab_time", "dx", "dw1", "dw2"}


def _snapshot(named):
    return {k: v.detach().clone() for k, v in named.items() if v is not None}


def _compare(eager, replay):
    for k, a in eager.items():
        b = replay[k]
        if k in ATOMIC:
            a64, b64 = a.double(), b.double()
            rms = math.sqrt(float((a64 * a64).mean()))
            assert float((a64 - b64).abs().max()) <= 1e-4 * max(rms, 1e-30), k
        else:
            assert torch.equal(a, b), k


def _capture_and_replay(step, outputs):
    step()                                   # eager run (also creates any library handle)
    torch.cuda.synchronize()
    eager = _snapshot(outputs())
    for t in outputs().values():             # poison the outputs: the replay must rewrite them
        if t is not None:
            t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    _compare(eager, _snapshot(outputs()))


@pytest.mark.parametrize("dropout,plan_once", [(None, False), ((0.2, 31, 7), False), (None, True)])
def test_attention_forward_backward_in_a_graph(dropout, plan_once):
    # plan_once: the benchmark's step (one planner launch, inputs in one buffer)
    from hstu_jagged_attention_02_gb300.attention import Problem
    b = synth.by_name("heavy_tailed", 3)
    pr = Problem(b, dropout=dropout, plan_once=plan_once, packed_inputs=plan_once)

    def step():
        pr.forward()
        pr.backward()

    def outputs():
        return {"o": pr.o, "y": pr.y, "dq": pr.dq, "dk": pr.dk, "dv": pr.dvv, "du": pr.du,
                "d_rab_pos": pr.d_rab_pos, "d_rab_time": pr.d_rab_time}

    _capture_and_replay(step, outputs)
    assert pr.device_error() == 0


def test_layer_forward_backward_in_a_graph():
    from hstu_jagged_attention_02_gb300.layer import LayerProblem
    from tests.test_gpu_layer import _small_layer
    b = _small_layer(45, [300, 131, 77, 260], H=2, d=128)
    pr = LayerProblem(b)

    def step():
        pr.forward()
        pr.backward()

    def outputs():
        return {"out": pr.out, "z1": pr.z1, "u": pr.u, "o": pr.o, "y": pr.y, "dx": pr.dx, "dw1": pr.dw1,
                "dw2": pr.dw2, "d_rab_pos": pr.d_rab_pos, "d_rab_time": pr.d_rab_time}

    _capture_and_replay(step, outputs)
    assert pr.device_error() == 0
