"""GPU parity of the decode-shaped forward (attn_fwd_decode): Nq queries
against Nk keys, the queries being the last Nq positions of the sequence
(at d = 128 with at most 12 queries through the decode kernel, otherwise
through the forward kernel with split keys).
Reference: the fp64 oracle on the square problem whose last Nq query rows
are these queries (the oracle's rows= selection), so the alignment, the
causal mask and the window are checked with no new oracle arithmetic.  Small
B*H forces the key split and the merge."""
import pytest
import torch

from exact_attention_67_gb300.synth import seeded_bf16
from tests.parity import check_fwd, out_bits, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_67_gb300 import build
    build.build()


CASES = [
    # (B, H, Nq, Nk, d, causal, window, dtype)
    (1, 2, 1, 777, 128, True, 0, torch.bfloat16),
    (1, 1, 1, 20000, 128, True, 0, torch.bfloat16),
    (2, 2, 4, 4096, 64, True, 0, torch.float16),
    (1, 2, 130, 5000, 128, True, 0, torch.bfloat16),
    (1, 3, 7, 3000, 128, False, 0, torch.bfloat16),
    (1, 2, 16, 9000, 64, True, 300, torch.bfloat16),
    (1, 1, 1, 1, 128, True, 0, torch.bfloat16),
    (2, 2, 300, 300, 128, True, 0, torch.float16),
    # d = 128 and at most 12 queries: the decode kernel (keys on the MMA's M side)
    (2, 3, 5, 6000, 128, False, 700, torch.float16),
    (1, 2, 8, 50000, 128, True, 0, torch.bfloat16),
    (3, 110, 2, 1100, 128, True, 0, torch.bfloat16),
    (1, 1, 3, 129, 128, True, 64, torch.bfloat16),
    (2, 2, 12, 7000, 128, True, 0, torch.float16),
    (1, 3, 11, 2500, 128, False, 900, torch.bfloat16),
    # Many key splits: the merge's batched loads over several rounds and a
    # ragged last batch (147 splits of a one-head sequence), at both head
    # sizes, and its 256-thread form (400 merged rows, 32 splits).
    (1, 1, 1, 131072, 128, True, 0, torch.bfloat16),
    (1, 1, 16, 131072, 64, False, 0, torch.float16),
    (1, 4, 100, 20000, 128, True, 0, torch.bfloat16),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,window,dtype", CASES, ids=lambda x: str(x).replace(" ", ""))
def test_decode_parity(orc, B, H, Nq, Nk, d, causal, window, dtype):
    import exact_attention_67_gb300 as ex
    seed = 7000 + Nq + Nk + d
    q_full = seeded_bf16((B, H, Nk, d), seed, 1.0, dtype)
    k = seeded_bf16((B, H, Nk, d), seed + 1, 1.0, dtype)
    v = seeded_bf16((B, H, Nk, d), seed + 2, 1.0, dtype)
    q = q_full[:, :, Nk - Nq:, :].contiguous()
    scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    o, lse = ex.forward_decode(q.to(DEV), k.to(DEV), v.to(DEV), causal, scale, window=window)
    torch.cuda.synchronize()
    assert ex.device_error() == 0
    rows = list(range(Nk - Nq, Nk))
    o_ref = torch.empty(B, H, Nq, d, dtype=torch.float64).numpy()
    lse_ref = torch.empty(B, H, Nq, dtype=torch.float64).numpy()
    for b in range(B):
        for h in range(H):
            o_ref[b, h], lse_ref[b, h] = orc.head_fwd(to_f64(q_full[b, h]), to_f64(k[b, h]), to_f64(v[b, h]), causal,
                                                      scale, rows=rows, window=window)
    splits = ex.attn_fwd_decode_workspace_size(B, H, Nq, Nk, d)
    print(check_fwd(to_f64(o.cpu()), lse.cpu().double().numpy(), o_ref, lse_ref,
                    f"decode B{B} H{H} Nq{Nq} Nk{Nk} d{d} causal={causal} window={window} ws={splits}",
                    out_bits(o)))
