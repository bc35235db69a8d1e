"""GPU parity of the strided / f16 entry points (attn_fwd_ex, attn_bwd_ex):
f16 inputs, the [B, N, H, d] layout of the flash_attn_func example
("提示词再优也救不了的性能黑洞…", 第一章), padded rows and mixed layouts, all
against the fp64 oracle, plus bit-identity with the contiguous bf16 path."""
import pytest
import torch

from exact_attention_67_gb300.synth import custom
from tests.parity import check_fwd, check_grads, out_bits, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_67_gb300 import build
    build.build()


def place(x: torch.Tensor, layout: str) -> torch.Tensor:
    """The CPU [B, H, N, d] tensor x on the GPU as a [B, H, N, d] view with the
    given memory layout: 'bhnd' (contiguous), 'bnhd' (x.transpose(1, 2) of a
    contiguous [B, N, H, d] tensor) or 'pad' (rows padded to d + 64)."""
    if layout == "bhnd":
        return x.to(DEV)
    if layout == "bnhd":
        return x.transpose(1, 2).contiguous().to(DEV).transpose(1, 2)
    if layout == "pad":
        B, H, N, d = x.shape
        buf = torch.zeros(B, H, N, d + 64, dtype=x.dtype, device=DEV)
        buf[..., :d] = x.to(DEV)
        return buf[..., :d]
    raise ValueError(layout)


def empty_like_layout(x: torch.Tensor, layout: str) -> torch.Tensor:
    return place(torch.empty(x.shape, dtype=x.dtype), layout).fill_(float("nan"))


def run_ex(ins, causal, scale, layouts, window=0):
    """attn_fwd_ex + attn_bwd_ex with q, k, v, dO and every output in the given layouts."""
    import exact_attention_67_gb300 as ex
    q, k, v, do = (place(t, lay) for t, lay in zip(ins, layouts[:4]))
    B, H, N, d = q.shape
    o = empty_like_layout(ins[0], layouts[4])
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    ex.attn_fwd_ex(q, k, v, o, lse, causal, scale, window=window)
    dq, dk, dv = (empty_like_layout(ins[0], lay) for lay in layouts[5:8])
    ws = torch.empty(ex.attn_bwd_workspace_size(B, H, N, d, causal), dtype=torch.uint8, device=DEV)
    ex.attn_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, causal, scale, ws, window=window)
    torch.cuda.synchronize()
    assert ex.device_error() == 0
    return {n: t.cpu() for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}


def check_against_oracle(orc, ins, res, causal, scale, what, window=0):
    qf, kf, vf, dof = (to_f64(t) for t in ins)
    o_ref, lse_ref = orc.attention_fwd(qf, kf, vf, causal, scale, window=window)
    msg = check_fwd(to_f64(res["o"]), res["lse"].double().numpy(), o_ref, lse_ref, what, out_bits(res["o"]))
    dq_ref, dk_ref, dv_ref = orc.attention_bwd(qf, kf, vf, dof, causal, scale, window=window)
    msg += " | " + check_grads([("dQ", to_f64(res["dq"]), dq_ref), ("dK", to_f64(res["dk"]), dk_ref),
                                ("dV", to_f64(res["dv"]), dv_ref)], what)
    return msg


CASES = [
    # (B, H, N, d, causal, dtype, layouts of q, k, v, dO, O, dQ, dK, dV)
    (1, 2, 256, 64, False, torch.float16, ["bhnd"] * 8),
    (2, 3, 300, 128, True, torch.float16, ["bhnd"] * 8),
    (1, 4, 384, 128, True, torch.bfloat16, ["bnhd"] * 8),
    (2, 2, 257, 64, True, torch.float16, ["bnhd"] * 8),
    (1, 3, 200, 128, False, torch.bfloat16, ["pad"] * 8),
    (2, 2, 320, 64, True, torch.bfloat16, ["bhnd", "bnhd", "pad", "bnhd", "pad", "bnhd", "bhnd", "pad"]),
    (1, 2, 129, 128, True, torch.float16, ["pad", "bhnd", "bnhd", "pad", "bnhd", "pad", "bnhd", "bhnd"]),
]


@pytest.mark.parametrize("B,H,N,d,causal,dtype,layouts", CASES, ids=lambda x: str(x).replace(" ", ""))
def test_strided_and_f16_parity(orc, B, H, N, d, causal, dtype, layouts):
    w, ins = custom(B, H, N, d, causal, seed=500 + N + d, dtype=dtype)
    res = run_ex(ins, causal, w.scale, layouts)
    assert res["o"].dtype == dtype and res["dq"].dtype == dtype
    print(check_against_oracle(orc, ins, res, causal, w.scale, f"{B},{H},{N},{d},{causal},{dtype},{layouts}"))


def test_f16_at_scale(orc):
    """A larger causal f16 problem in [B, N, H, d] layout (several waves of CTAs)."""
    w, ins = custom(1, 16, 2048, 128, True, seed=4242, dtype=torch.float16)
    res = run_ex(ins, True, w.scale, ["bnhd"] * 8)
    print(check_against_oracle(orc, ins, res, True, w.scale, "f16 B1 H16 N2048 d128 causal bnhd"))


def test_layout_does_not_change_bits():
    """The strided path reads and writes through different addresses only: for
    bf16 its results equal the contiguous attn_fwd / attn_bwd bit for bit."""
    import exact_attention_67_gb300 as ex
    w, ins = custom(2, 4, 520, 128, True, seed=91)
    q, k, v, do = (t.to(DEV) for t in ins)
    o, lse = ex.forward(q, k, v, True, w.scale)
    dq, dk, dv = ex.backward(q, k, v, o, lse, do, True, w.scale)
    res = run_ex(ins, True, w.scale, ["bnhd", "pad", "bnhd", "pad", "bnhd", "pad", "bnhd", "pad"])
    for name, ref in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(res[name], ref.cpu()), name


@pytest.mark.parametrize("dtype,groups", [(torch.bfloat16, 2), (torch.float16, 3), (torch.bfloat16, 1)])
def test_host_path_equals_device_path(dtype, groups):
    """fwd_bwd_from_host (host tensors in and out, copies overlapped with the
    kernels in groups of heads) gives the device path's results bit for bit."""
    import exact_attention_67_gb300 as ex
    from exact_attention_67_gb300.host import fwd_bwd_from_host
    w, ins = custom(2, 3, 300, 128, True, seed=61, dtype=dtype)
    pin = [t.pin_memory() for t in ins]
    outs = fwd_bwd_from_host(*pin, True, w.scale, groups=groups, device=DEV)
    torch.cuda.synchronize()
    q, k, v, do = (t.to(DEV) for t in ins)
    o, lse = ex.forward(q, k, v, True, w.scale)
    dq, dk, dv = ex.backward(q, k, v, o, lse, do, True, w.scale)
    torch.cuda.synchronize()
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), outs, (o, lse, dq, dk, dv)):
        assert torch.equal(a, b.cpu()), name


def test_host_step_replays_current_inputs():
    """HostStep (the host path as one CUDA graph) matches the device path bit
    for bit, and a replay picks up new contents of the pinned inputs."""
    import exact_attention_67_gb300 as ex
    w, ins = custom(1, 5, 700, 64, True, seed=71)
    w2, ins2 = custom(1, 5, 700, 64, True, seed=72)
    pin = [t.pin_memory() for t in ins]
    step = ex.HostStep(*pin, True, w.scale, groups=3, streams=2, device=DEV)
    for src in (ins, ins2):
        for p_, t in zip(pin, src):
            p_.copy_(t)
        outs = step()
        torch.cuda.synchronize()
        q, k, v, do = (t.to(DEV) for t in src)
        o, lse = ex.forward(q, k, v, True, w.scale)
        dq, dk, dv = ex.backward(q, k, v, o, lse, do, True, w.scale)
        torch.cuda.synchronize()
        for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), outs, (o, lse, dq, dk, dv)):
            assert torch.equal(a, b.cpu()), name


@pytest.mark.parametrize("B,H,N,d,causal,groups,side,dtype", [
    (3, 1, 77, 64, True, 5, False, torch.bfloat16),     # more groups than problems; every role on one stream
    (1, 1, 300, 128, False, 1, True, torch.bfloat16),   # one problem, ragged N
    (2, 3, 129, 64, True, 4, True, torch.float16),      # f16 backward in one call per group
])
def test_host_entry_point_edge_cases(B, H, N, d, causal, groups, side, dtype):
    """attn_fwd_bwd_host (the C ABI's host-buffer call) on awkward shapes and
    stream set-ups gives the device path's results bit for bit."""
    import exact_attention_67_gb300 as ex
    w, ins = custom(B, H, N, d, causal, seed=81 + N, dtype=dtype)
    pin = [t.pin_memory() for t in ins]
    outs = (torch.empty_like(ins[0]).pin_memory(), torch.empty(B, H, N).pin_memory(),
            torch.empty_like(ins[0]).pin_memory(), torch.empty_like(ins[0]).pin_memory(),
            torch.empty_like(ins[0]).pin_memory())
    ws = torch.empty(ex.attn_fwd_bwd_host_workspace_size(B, H, N, d, causal), dtype=torch.uint8, device=DEV)
    streams = [torch.cuda.Stream(device=DEV) for _ in range(3)] if side else [None, None, None]
    ex.attn_fwd_bwd_host(*pin, outs[0], outs[1], outs[2], outs[3], outs[4], causal, w.scale, ws, groups=groups,
                         copy_in_stream=streams[0], copy_out_stream=streams[1], stream2=streams[2])
    torch.cuda.synchronize()
    q, k, v, do = (t.to(DEV) for t in ins)
    o, lse = ex.forward(q, k, v, causal, w.scale)
    dq, dk, dv = ex.backward(q, k, v, o, lse, do, causal, w.scale)
    torch.cuda.synchronize()
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), outs, (o, lse, dq, dk, dv)):
        assert torch.equal(a, b.cpu()), name
    assert ex.device_error() == 0
