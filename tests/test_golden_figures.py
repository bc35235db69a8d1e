"""Workload accounting against figures printed on the pages (CPU only)."""
import os

from exact_attention_67_gb300.synth import WORKLOADS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.txt")


def _golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = int(v)
    return out


def test_score_matrix_size_matches_page():
    g = _golden()
    w = WORKLOADS[5]
    assert w.N == 16384 and w.H == 8
    assert w.N * w.N == g["score_elements_per_head_N16384"]
    assert 2 * w.N * w.N == g["score_bytes_fp16_per_head_N16384"]
    assert 2 * w.N * w.N * w.H == g["score_bytes_fp16_8heads_N16384"]


def test_causal_flops_are_half():
    g = _golden()
    for w in WORKLOADS.values():
        full = 4.0 * w.B * w.H * w.N * w.N * w.d
        kept = w.flops_fwd() / full * 100
        assert kept == (g["causal_work_percent"] if w.causal else 100)
        assert w.flops_bwd() == 2.5 * w.flops_fwd()
