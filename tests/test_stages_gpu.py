"""The backward's stage calls against attn_bwd: attn_bwd_d_and_dq (dQ kernel
forming the row terms D_i itself) followed by attn_bwd_dkdv, and
attn_bwd_preprocess followed by attn_bwd_dkdv and attn_bwd_dq, give D and
dQ, dK, dV bit-identical to attn_bwd; dQ also matches the fp64 oracle."""
import pytest
import torch

from exact_attention_67_gb300.synth import custom
from tests.parity import TOL_GRAD_REL, rel_fro, to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_67_gb300 import build
    build.build()


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 3, 333, 128, True), (2, 2, 200, 64, False), (1, 1, 1, 64, True),
                                            (1, 2, 700, 128, False), (2, 1, 520, 64, True)])
def test_stage_calls_match_attn_bwd(orc, B, H, N, d, causal):
    import exact_attention_67_gb300 as ex
    w, ins = custom(B, H, N, d, causal, seed=900 + N + d)
    q, k, v, do = (t.to(DEV) for t in ins)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    ex.attn_fwd(q, k, v, o, lse, causal, w.scale)
    ws = torch.empty(ex.attn_bwd_workspace_size(B, H, N, d, causal), dtype=torch.uint8, device=DEV)
    g0 = [torch.empty_like(q) for _ in range(3)]
    ex.attn_bwd(q, k, v, o, do, lse, *g0, causal, w.scale, ws)
    # Three launches: row dots, dK/dV, dQ.
    D1 = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=DEV)
    g1 = [torch.empty_like(q) for _ in range(3)]
    ex.attn_bwd_preprocess(o, do, D1)
    ex.attn_bwd_dkdv(q, k, v, do, lse, D1, g1[1], g1[2], causal, w.scale)
    ex.attn_bwd_dq(q, k, v, do, lse, D1, g1[0], causal, w.scale)
    # Two launches: dQ with the row dots, then dK/dV.
    D2 = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=DEV)
    g2 = [torch.empty_like(q) for _ in range(3)]
    ex.attn_bwd_d_and_dq(q, k, v, o, do, lse, D2, g2[0], causal, w.scale)
    ex.attn_bwd_dkdv(q, k, v, do, lse, D2, g2[1], g2[2], causal, w.scale)
    torch.cuda.synchronize()
    assert ex.device_error() == 0
    assert torch.equal(D1, D2), "D from the dQ kernel differs from the row-dot kernel's"
    for a, b, c, name in zip(g0, g1, g2, ("dQ", "dK", "dV")):
        assert torch.equal(a, b) and torch.equal(a, c), name
    # D against its definition in fp64 (sum of products of the bf16 values).
    D_ref = (to_f64(o.cpu()) * to_f64(do.cpu())).sum(-1)
    assert abs(D2.double().cpu().numpy() - D_ref).max() <= 1e-4 * max(1.0, abs(D_ref).max())
    qf, kf, vf, dof = (to_f64(t) for t in ins)
    dq_ref, _, _ = orc.attention_bwd(qf, kf, vf, dof, causal, w.scale)
    assert rel_fro(to_f64(g2[0].cpu()), dq_ref) <= TOL_GRAD_REL
