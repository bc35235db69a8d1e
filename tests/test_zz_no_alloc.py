"""attn_bwd_noalloc: the backward entry point for callers that cannot
allocate device memory (a plugin handed only its input and output buffers by
a runtime that owns all device memory, or code on a path where an allocation
is not allowed).  It keeps its row terms in a fixed array inside the library
instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row, on two different
problems, and checks each result against attn_bwd (the entry point with a
caller-allocated workspace) within the gradient tolerance the parity tests
use.  This file is collected last so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_67_gb300.synth import WORKLOADS, custom, make_inputs
from tests.parity import TOL_GRAD_REL, rel_fro, to_f64


@pytest.fixture(scope="module")
def lib():
    from exact_attention_67_gb300 import _lib
    from exact_attention_67_gb300 import build as b
    b.build()
    return _lib.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_rejects_more_rows_than_its_scratch(lib):
    # 2 * 64 * 32768 = 4,194,304 rows is the limit; one more head is too many.
    fake = [0x100000 * (i + 1) for i in range(9)]
    assert lib.attn_bwd_noalloc(*fake, 2, 65, 32768, 128, 1, 0.088, None) == 6  # EXATTN_ERR_WORKSPACE
    assert lib.attn_bwd_noalloc(*fake, 1, 1, 0, 128, 1, 0.088, None) == 2      # invalid shape
    assert lib.attn_bwd_noalloc(None, *fake[1:], 1, 1, 8, 128, 1, 0.088, None) == 1


@pytest.mark.gpu
def test_noalloc_matches_attn_bwd_twice(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_67_gb300 as ex
    dev = torch.device("cuda:0")
    w2 = WORKLOADS[2]
    problems = [(w2, make_inputs(w2)), custom(1, 3, 777, 64, False, seed=4242)]
    stream = torch.cuda.current_stream().cuda_stream
    for call, (w, (q, k, v, do)) in enumerate(problems):
        q, k, v, do = (t.to(dev) for t in (q, k, v, do))
        o, lse = ex.forward(q, k, v, w.causal, w.scale)
        ref = ex.backward(q, k, v, o, lse, do, w.causal, w.scale)   # caller workspace
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = lib.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(got[0]), _p(got[1]),
                                  _p(got[2]), w.B, w.H, w.N, w.d, int(w.causal), w.scale, stream)
        assert rc == 0, ex.status_string(rc)
        torch.cuda.synchronize()
        assert ex.device_error() == 0
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            gf, rf = to_f64(g), to_f64(r)
            assert np.all(np.isfinite(gf)), f"call {call}: {name} not finite"
            assert rel_fro(gf, rf) <= TOL_GRAD_REL, f"call {call}: {name} rel-Fro {rel_fro(gf, rf):.3e}"
