"""Failure detection without a GPU fault: every pipeline wait of the
tensor-core kernels has a time limit.  The test-only flag makes the forward
withhold one TMA load, so a wait runs out (after ~1 ms), the kernel records
HSTU_ERR_TIMEOUT in the workspace and every role exits cleanly; the context
stays usable for the next call."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from hstu_jagged_attention_02_gb300 import binding as C  # noqa: E402
from hstu_jagged_attention_02_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu


def test_forward_wait_times_out_and_context_survives():
    from hstu_jagged_attention_02_gb300.attention import Problem
    b = synth.make_batch([300, 129, 700], H=2, d_qk=128, d_v=128, dtype="bf16", num_targets=8, seed=90)
    pr = Problem(b, flags=C.HSTU_FLAG_TEST_TIMEOUT)
    pr.forward()
    torch.cuda.synchronize()
    assert pr.device_error() == C.HSTU_ERR_TIMEOUT
    # same inputs without the flag: clean run, and a finite result
    pr2 = Problem(b)
    pr2.forward()
    pr2.backward()
    torch.cuda.synchronize()
    assert pr2.device_error() == 0
    assert torch.isfinite(pr2.o).all() and torch.isfinite(pr2.dq).all()


def test_layer_projection_wait_times_out_and_context_survives():
    # the layer's tensor-core input projection in its test mode: CTA 0 skips
    # its first load, the MMA warp's wait runs out, every role exits, and the
    # error (kept in the layer's own header word while the attention runs)
    # is raised into the workspace error word by the output projection
    from tests.test_gpu_layer import _small_layer, layer_problem
    b = _small_layer(91, [300, 131, 260], H=2, d=64)
    pr = layer_problem(b)
    pr.desc.flags |= C.HSTU_FLAG_TEST_TIMEOUT
    pr.forward()
    torch.cuda.synchronize()
    assert pr.device_error() == C.HSTU_ERR_TIMEOUT
    with pytest.raises(C.HSTUError) as e:   # a forward-only test mode
        pr.backward()
    assert e.value.status == C.HSTU_ERR_UNSUPPORTED
    pr.desc.flags &= ~C.HSTU_FLAG_TEST_TIMEOUT
    pr.forward()
    pr.backward()
    torch.cuda.synchronize()
    assert pr.device_error() == 0
    assert torch.isfinite(pr.out).all() and torch.isfinite(pr.dx).all()
