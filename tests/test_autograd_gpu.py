"""The differentiable wrappers (attention, flash_attn_func) return exactly
what the explicit forward/backward calls return, in both layouts."""
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


def test_attention_autograd_equals_explicit_calls():
    import exact_attention_67_gb300 as ex
    w, ins = custom(2, 3, 333, 128, True, seed=91)
    q, k, v, do = (t.to(DEV) for t in ins)
    qr, kr, vr = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = ex.attention(qr, kr, vr, causal=True, scale=w.scale)
    out.backward(do)
    o, lse = ex.forward(q, k, v, True, w.scale)
    dq, dk, dv = ex.backward(q, k, v, o, lse, do, True, w.scale)
    assert torch.equal(out, o)
    for name, a, b in (("dq", qr.grad, dq), ("dk", kr.grad, dk), ("dv", vr.grad, dv)):
        assert torch.equal(a, b), name


def test_flash_attn_func_layout_and_expanded_gradient():
    import exact_attention_67_gb300 as ex
    w, ins = custom(1, 4, 200, 64, True, seed=92, dtype=torch.float16)
    q, k, v, _ = (t.to(DEV) for t in ins)                        # [B, H, N, d]
    qn, kn, vn = (t.transpose(1, 2).contiguous().requires_grad_(True) for t in (q, k, v))  # [B, N, H, d]
    out = ex.flash_attn_func(qn, kn, vn, causal=True, softmax_scale=w.scale)
    assert out.shape == qn.shape
    out.float().sum().backward()                                   # an expanded gradient of ones
    o, lse = ex.forward(q, k, v, True, w.scale)
    ones = torch.ones_like(o)
    dq, dk, dv = ex.backward(q, k, v, o, lse, ones, True, w.scale)
    assert torch.equal(out.transpose(1, 2), o)
    for name, a, b in (("dq", qn.grad, dq), ("dk", kn.grad, dk), ("dv", vn.grad, dv)):
        assert torch.equal(a.transpose(1, 2), b), name
    with pytest.raises(ValueError):
        ex.flash_attn_func(qn, kn, vn, dropout_p=0.1)
