"""GPU parity of the fp32-O path (attn_fwd_o32 / attn_bwd_o32): the forward's
fp32 copy of O rounds to the O it returns, the backward that takes the row
terms D_i = dO_i . O_i from it matches the fp64 oracle -- including on rows
whose softmax is nearly one-hot, where D from the 16-bit O is not accurate
enough for the relative gradient bound -- and the autograd option runs it."""
import pytest
import torch

from exact_attention_67_gb300.synth import custom
from tests.parity import TOL_GRAD_REL, check_fwd, check_grads, out_bits, rel_fro, to_f64
from tests.test_layouts_gpu import empty_like_layout, place
from tests.test_varlen_gpu import packed_inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_67_gb300 import build
    build.build()


def run_o32(ins, causal, scale, layouts, window=0):
    import exact_attention_67_gb300 as ex
    q, k, v, do = (place(t, lay) for t, lay in zip(ins, layouts[:4]))
    B, H, N, d = q.shape
    o = empty_like_layout(ins[0], layouts[4])
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    o32 = torch.empty(B, H, N, d, dtype=torch.float32, device=DEV)
    ex.attn_fwd_o32(q, k, v, o, lse, o32, causal, scale, window=window)
    dq, dk, dv = (empty_like_layout(ins[0], lay) for lay in layouts[5:8])
    ws = torch.empty(ex.attn_bwd_workspace_size(B, H, N, d, causal), dtype=torch.uint8, device=DEV)
    ex.attn_bwd_o32(q, k, v, o32, do, lse, dq, dk, dv, causal, scale, ws, window=window)
    torch.cuda.synchronize()
    assert ex.device_error() == 0
    return {"o": o.cpu(), "lse": lse.cpu(), "o32": o32.cpu(), "dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu()}


CASES = [
    # (B, H, N, d, causal, window, dtype, layouts of q, k, v, dO, O, dQ, dK, dV)
    (2, 3, 333, 128, True, 0, torch.bfloat16, ["bhnd"] * 8),
    (1, 2, 520, 64, False, 100, torch.float16, ["bnhd", "pad", "bhnd", "bnhd", "bhnd", "pad", "bnhd", "bhnd"]),
    (1, 80, 200, 128, False, 0, torch.bfloat16, ["bhnd"] * 8),
]


@pytest.mark.parametrize("B,H,N,d,causal,window,dtype,layouts", CASES, ids=lambda x: str(x).replace(" ", "")[:40])
def test_o32_parity(orc, B, H, N, d, causal, window, dtype, layouts):
    w, ins = custom(B, H, N, d, causal, seed=600 + N + d, dtype=dtype)
    res = run_o32(ins, causal, w.scale, layouts, window)
    # O is the fp32 copy rounded to the output type, element for element.
    assert torch.equal(res["o"], res["o32"].to(dtype))
    qf, kf, vf, dof = (to_f64(t) for t in ins)
    o_ref, lse_ref = orc.attention_fwd(qf, kf, vf, causal, w.scale, window=window)
    msg = check_fwd(to_f64(res["o"]), res["lse"].double().numpy(), o_ref, lse_ref, "o32 path", out_bits(res["o"]))
    dq_ref, dk_ref, dv_ref = orc.attention_bwd(qf, kf, vf, dof, causal, w.scale, window=window)
    msg += " | " + check_grads([("dQ", to_f64(res["dq"]), dq_ref), ("dK", to_f64(res["dk"]), dk_ref),
                                ("dV", to_f64(res["dv"]), dv_ref)], "o32 path")
    print(msg)


def test_nearly_one_hot_rows():
    """Two tokens, causal, second row's weights 0.96 / 0.04 on both heads: dQ
    is a small difference.  D from the bf16 O gives it a relative error near
    0.1; D from the fp32 copy keeps it within the bound."""
    import exact_attention_67_gb300 as ex
    import oracle
    orc = oracle._load()
    lens = [12, 994, 934, 79, 2]
    ins_p, cu = packed_inputs(lens, 2, 64, seed=3000 + sum(lens), dtype=torch.bfloat16)
    a, z = int(cu[4]), int(cu[5])
    ins = [t[a:z].permute(1, 0, 2).unsqueeze(0).contiguous() for t in ins_p]  # [1, 2, 2, 64]
    scale = float(torch.tensor(64 ** -0.5, dtype=torch.float32))
    q, k, v, do = (t.to(DEV) for t in ins)
    qf, kf, vf, dof = (to_f64(t) for t in ins)
    dq_ref, dk_ref, dv_ref = orc.attention_bwd(qf, kf, vf, dof, True, scale)
    o, lse = ex.forward(q, k, v, True, scale)
    dq16, _, _ = ex.backward(q, k, v, o, lse, do, True, scale)
    o2, lse2, o32 = ex.forward(q, k, v, True, scale, fp32_o=True)
    dq32, dk32, dv32 = ex.backward(q, k, v, None, lse2, do, True, scale, o32=o32)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    e16, e32 = rel_fro(to_f64(dq16.cpu()), dq_ref), rel_fro(to_f64(dq32.cpu()), dq_ref)
    print(f"nearly one-hot rows: dQ rel-Fro {e16:.3e} with D from the bf16 O, {e32:.3e} from the fp32 copy")
    assert e32 <= TOL_GRAD_REL
    assert rel_fro(to_f64(dk32.cpu()), dk_ref) <= TOL_GRAD_REL and rel_fro(to_f64(dv32.cpu()), dv_ref) <= TOL_GRAD_REL


def test_autograd_fp32_o_matches_the_o32_calls():
    import exact_attention_67_gb300 as ex
    w, ins = custom(1, 2, 300, 128, True, seed=61)
    q, k, v, do = (t.to(DEV) for t in ins)
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = ex.attention(qa, ka, va, causal=True, fp32_o=True)
    out.backward(do)
    o, lse, o32 = ex.forward(q, k, v, True, fp32_o=True)
    dq, dk, dv = ex.backward(q, k, v, None, lse, do, True, o32=o32)
    torch.cuda.synchronize()
    assert torch.equal(out.detach(), o)
    assert torch.equal(qa.grad, dq) and torch.equal(ka.grad, dk) and torch.equal(va.grad, dv)


@pytest.mark.parametrize("d,causal,window", [(64, True, 100), (128, False, 57)])
def test_autograd_fp32_o_with_window_against_the_oracle(orc, d, causal, window):
    """attention(..., fp32_o=True) with a sliding window, f16 inputs in the
    [B, N, H, d] layout: gradients match the fp64 oracle, and the output
    equals the default path's (the fp32 copy changes only the row terms)."""
    import exact_attention_67_gb300 as ex
    w, ins = custom(1, 3, 410, d, causal, seed=71 + d, dtype=torch.float16)
    q, k, v, do = (t.to(DEV) for t in ins)
    qn, kn, vn = (t.transpose(1, 2).contiguous().transpose(1, 2).requires_grad_(True) for t in (q, k, v))
    out = ex.attention(qn, kn, vn, causal=causal, scale=w.scale, window=window, fp32_o=True)
    out.backward(do)
    o_default = ex.attention(q, k, v, causal=causal, scale=w.scale, window=window)
    torch.cuda.synchronize()
    assert torch.equal(out.detach(), o_default)
    qf, kf, vf, dof = (to_f64(t) for t in ins)
    dq_ref, dk_ref, dv_ref = orc.attention_bwd(qf, kf, vf, dof, causal, w.scale, window=window)
    print(check_grads([("dQ", to_f64(qn.grad.cpu()), dq_ref), ("dK", to_f64(kn.grad.cpu()), dk_ref),
                       ("dV", to_f64(vn.grad.cpu()), dv_ref)], f"fp32_o autograd d{d} window {window}"))
