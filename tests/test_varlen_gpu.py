"""GPU parity of packed variable-length batches (attn_fwd_varlen /
attn_bwd_varlen): every sequence of the pack is its own attention problem.
Each sequence is compared with the fp64 oracle run on that sequence alone,
and with the same sequence run by itself through the fixed-length path (bit
for bit: same tiles, same arithmetic)."""
import numpy as np
import pytest
import torch

from exact_attention_67_gb300.synth import seeded_bf16
from tests.parity import check_fwd, check_grads, out_bits, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_67_gb300 import build
    build.build()


def packed_inputs(lens, H, d, seed, dtype):
    total = int(sum(lens))
    ins = [seeded_bf16((total, H, d), seed + t, 1.0, dtype) for t in range(4)]  # q, k, v, dO on the CPU
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    return ins, cu


def run_varlen(ins, cu, lens, causal, scale, window):
    import exact_attention_67_gb300 as ex
    q, k, v, do = (t.to(DEV) for t in ins)
    cud = cu.to(DEV)
    o, lse = ex.forward_varlen(q, k, v, cud, max(lens), causal, scale, window=window)
    dq, dk, dv = ex.backward_varlen(q, k, v, o, lse, do, cud, max(lens), causal, scale, window=window)
    torch.cuda.synchronize()
    assert ex.device_error() == 0
    return {n: t.cpu() for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}


CASES = [
    # (lens, H, d, causal, window, dtype)
    ([300, 1, 128, 129, 513, 64, 127], 3, 128, True, 0, torch.bfloat16),
    ([257, 700, 2, 256], 2, 64, False, 0, torch.bfloat16),
    ([1000, 33, 400], 2, 128, True, 100, torch.float16),
    ([640, 5, 300], 2, 64, False, 129, torch.float16),
]


@pytest.mark.parametrize("lens,H,d,causal,window,dtype", CASES, ids=lambda x: str(x).replace(" ", ""))
def test_varlen_parity(orc, lens, H, d, causal, window, dtype):
    ins, cu = packed_inputs(lens, H, d, seed=3000 + sum(lens), dtype=dtype)
    scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    res = run_varlen(ins, cu, lens, causal, scale, window)
    msgs = []
    for b, n in enumerate(lens):
        a, z = int(cu[b]), int(cu[b + 1])
        # this sequence as [1, H, n, d] for the oracle
        q, k, v, do = (to_f64(t[a:z].permute(1, 0, 2).unsqueeze(0)) for t in ins)
        o_ref, lse_ref = orc.attention_fwd(q, k, v, causal, scale, window=window)
        o = to_f64(res["o"][a:z].permute(1, 0, 2).unsqueeze(0))
        lse = res["lse"][:, a:z].unsqueeze(0).double().numpy()
        msgs.append(check_fwd(o, lse, o_ref, lse_ref, f"seq {b} (n={n})", out_bits(res["o"])))
        dq_ref, dk_ref, dv_ref = orc.attention_bwd(q, k, v, do, causal, scale, window=window)
        g = {nm: to_f64(res[nm][a:z].permute(1, 0, 2).unsqueeze(0)) for nm in ("dq", "dk", "dv")}
        msgs.append(check_grads([("dQ", g["dq"], dq_ref), ("dK", g["dk"], dk_ref), ("dV", g["dv"], dv_ref)],
                                f"seq {b} (n={n})"))
    print("\n".join(msgs))


def test_varlen_equals_each_sequence_alone():
    """The pack gives, per sequence, exactly what the fixed-length path gives
    for that sequence by itself ([1, H, n, d] views of the packed rows)."""
    import exact_attention_67_gb300 as ex
    lens = [129, 384, 1, 250]
    H, d, causal, window = 2, 128, True, 0
    ins, cu = packed_inputs(lens, H, d, seed=77, dtype=torch.bfloat16)
    scale = d ** -0.5
    res = run_varlen(ins, cu, lens, causal, scale, window)
    for b, n in enumerate(lens):
        a, z = int(cu[b]), int(cu[b + 1])
        q, k, v, do = (t[a:z].to(DEV).permute(1, 0, 2).unsqueeze(0) for t in ins)  # strided [1, H, n, d] views
        o, lse = ex.forward(q, k, v, causal, scale)
        dq, dk, dv = ex.backward(q, k, v, o, lse, do, causal, scale)
        torch.cuda.synchronize()
        assert torch.equal(res["o"][a:z], o[0].permute(1, 0, 2).cpu()), b
        assert torch.equal(res["lse"][:, a:z], lse[0].cpu()), b
        for nm, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            assert torch.equal(res[nm][a:z], t[0].permute(1, 0, 2).cpu()), (b, nm)
