"""Failure detection without a GPU fault: every wait inside the kernels is
bounded.  exattn_watchdog_selftest launches one warp whose wait on a barrier
nothing arrives on runs out after 2 ms; the host must then read
EXATTN_ERR_TIMEOUT from exattn_device_error(), the word must clear, and the
context must stay usable for real work."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_67_gb300 as ex
    from exact_attention_67_gb300 import _lib
    from exact_attention_67_gb300 import build
    from exact_attention_67_gb300.synth import WORKLOADS, make_inputs
    build.build()
    assert ex.device_error() == 0
    _lib.watchdog_selftest(2000)
    assert ex.device_error() == 8          # EXATTN_ERR_TIMEOUT, read and cleared
    assert ex.device_error() == 0
    w = WORKLOADS[1]
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    o, lse = ex.forward(q, k, v, w.causal, w.scale)
    dq, dk, dv = ex.backward(q, k, v, o, lse, do, w.causal, w.scale)
    torch.cuda.synchronize()
    assert ex.device_error() == 0
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t.float()).all()


def test_selftest_rejects_bad_timeout():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_67_gb300 import _lib
    assert _lib.load().exattn_watchdog_selftest(0, None) == 9
    assert _lib.load().exattn_watchdog_selftest(2000000, None) == 9


def test_python_helpers_raise_after_a_fired_wait():
    """The helpers poll the watchdog word without synchronising: after a wait
    gave up, the next helper call whose poll has landed raises
    ExattnError(EXATTN_ERR_TIMEOUT), which also clears the word."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_67_gb300 as ex
    from exact_attention_67_gb300 import _lib
    from exact_attention_67_gb300.synth import WORKLOADS, make_inputs
    w = WORKLOADS[1]
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    assert ex.device_error() == 0
    _lib.watchdog_selftest(2000)
    torch.cuda.synchronize()
    with pytest.raises(ex.ExattnError) as ei:
        ex.forward(q, k, v, w.causal, w.scale)
    assert ei.value.status == 8
    assert ex.device_error() == 0
    o, lse = ex.forward(q, k, v, w.causal, w.scale)   # clean again
    ex.backward(q, k, v, o, lse, do, w.causal, w.scale)
    torch.cuda.synchronize()
    ex.forward(q, k, v, w.causal, w.scale)
    assert ex.device_error() == 0
