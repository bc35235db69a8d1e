"""Calls from a host thread that has made no CUDA call of its own: such a
thread has no current CUDA context, and the library makes the device's
primary context current before its driver calls (the TMA tensor-map
encoder).  Results match the same calls on the main thread bit for bit; the
autograd backward runs on PyTorch's device thread."""
import threading

import pytest
import torch

from exact_attention_67_gb300.synth import custom

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_67_gb300 import build
    build.build()


def in_fresh_thread(fn):
    box = {}

    def run():
        try:
            box["out"] = fn()
            torch.cuda.synchronize()
        except BaseException as e:  # re-raised on the calling thread
            box["err"] = e

    t = threading.Thread(target=run)
    t.start()
    t.join()
    if "err" in box:
        raise box["err"]
    return box["out"]


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_forward_and_backward_from_a_fresh_thread(d, causal):
    import exact_attention_67_gb300 as ex
    w, ins = custom(1, 2, 300, d, causal, seed=71 + d)
    q, k, v, do = (t.to(DEV) for t in ins)
    o, lse = ex.forward(q, k, v, causal)
    dq, dk, dv = ex.backward(q, k, v, o, lse, do, causal)
    o2, lse2 = in_fresh_thread(lambda: ex.forward(q, k, v, causal))
    dq2, dk2, dv2 = in_fresh_thread(lambda: ex.backward(q, k, v, o, lse, do, causal))
    o3, lse3, o32 = in_fresh_thread(lambda: ex.forward(q, k, v, causal, fp32_o=True))
    torch.cuda.synchronize()
    assert ex.device_error() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2) and torch.equal(o, o3) and torch.equal(lse, lse3)
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_last_cuda_error_is_per_thread_and_empty_after_success():
    import exact_attention_67_gb300 as ex
    from exact_attention_67_gb300 import _lib
    w, ins = custom(1, 1, 128, 64, False, seed=5)
    q, k, v, _ = (t.to(DEV) for t in ins)
    assert in_fresh_thread(lambda: (ex.forward(q, k, v, False), _lib.last_cuda_error())[1]) == ""
