"""GPU parity of sliding-window (local) attention through attn_fwd_ex /
attn_bwd_ex: key j visible to query i iff i - j < W (and j - i < W without the
causal mask), the reading of the local attention of "Flash Attention V3：大模型
加速的核心网络算子优化实践", §三.1.  Windows below, at and across the 128-key
tile, ragged N, both input types, against the fp64 oracle with the same window."""
import pytest
import torch

from exact_attention_67_gb300.synth import custom
from tests.test_layouts_gpu import check_against_oracle, run_ex

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_67_gb300 import build
    build.build()


CASES = [
    # (B, H, N, d, causal, window, dtype)
    (1, 2, 700, 128, True, 1, torch.bfloat16),
    (1, 2, 700, 128, True, 64, torch.bfloat16),
    (2, 2, 1100, 64, True, 129, torch.bfloat16),
    (1, 3, 1024, 128, True, 256, torch.float16),
    (1, 2, 777, 128, True, 300, torch.bfloat16),
    (1, 2, 650, 64, False, 100, torch.bfloat16),
    (1, 2, 900, 128, False, 257, torch.float16),
    (1, 1, 300, 128, True, 5000, torch.bfloat16),
]


@pytest.mark.parametrize("B,H,N,d,causal,window,dtype", CASES, ids=lambda x: str(x).replace(" ", ""))
def test_window_parity(orc, B, H, N, d, causal, window, dtype):
    w, ins = custom(B, H, N, d, causal, seed=900 + N + window, dtype=dtype)
    res = run_ex(ins, causal, w.scale, ["bhnd"] * 8, window=window)
    print(check_against_oracle(orc, ins, res, causal, w.scale, f"window {window} {B},{H},{N},{d},{causal}",
                               window=window))


def test_window_of_n_is_no_window():
    """A window of N or more hides no key: results equal the windowless call
    bit for bit (same tiles, same arithmetic)."""
    w, ins = custom(1, 4, 520, 128, True, seed=31)
    a = run_ex(ins, True, w.scale, ["bhnd"] * 8, window=0)
    b = run_ex(ins, True, w.scale, ["bhnd"] * 8, window=520)
    for name in a:
        assert torch.equal(a[name], b[name]), name
