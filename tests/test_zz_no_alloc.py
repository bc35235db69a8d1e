"""attn_bwd_noalloc: the backward entry point for callers that cannot
allocate device memory (a plugin handed only its input and output buffers by
a runtime that owns all device memory, or code on a path where an allocation
is not allowed).  It keeps its row terms in a fixed array inside the library
instead of a caller workspace.

The GPU tests call it through the C ABI twice in a row, on two different
problems, and check each result against the fp64 oracle and against
attn_bwd (the entry point with a caller-allocated workspace) within the
gradient tolerance the parity tests use; then once more at exactly its row
limit, after those calls left their contents in its array.  This file is
collected last so that a run stopping at the first failure has already run
every other test."""
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
def test_noalloc_matches_oracle_and_attn_bwd_twice(lib, orc):
    """Two calls in a row on different problems: each result against the fp64
    oracle (gradient tolerance of the parity tests) and against attn_bwd."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_67_gb300 as ex
    dev = torch.device("cuda:0")
    w2 = WORKLOADS[2]
    problems = [(w2, make_inputs(w2)), custom(1, 3, 777, 64, False, seed=4242)]
    stream = torch.cuda.current_stream().cuda_stream
    for call, (w, (q, k, v, do)) in enumerate(problems):
        dq_ref, dk_ref, dv_ref = orc.attention_bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(do), w.causal, w.scale)
        q, k, v, do = (t.to(dev) for t in (q, k, v, do))
        o, lse = ex.forward(q, k, v, w.causal, w.scale)
        lib_ref = ex.backward(q, k, v, o, lse, do, w.causal, w.scale)   # caller workspace
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = lib.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(got[0]), _p(got[1]),
                                  _p(got[2]), w.B, w.H, w.N, w.d, int(w.causal), w.scale, stream)
        assert rc == 0, ex.status_string(rc)
        torch.cuda.synchronize()
        assert ex.device_error() == 0
        for name, g, r, oref in zip(("dQ", "dK", "dV"), got, lib_ref, (dq_ref, dk_ref, dv_ref)):
            gf = to_f64(g)
            assert np.all(np.isfinite(gf)), f"call {call}: {name} not finite"
            e = rel_fro(gf, oref)
            assert e <= TOL_GRAD_REL, f"call {call}: {name} rel-Fro vs oracle {e:.3e}"
            e = rel_fro(gf, to_f64(r))
            assert e <= TOL_GRAD_REL, f"call {call}: {name} rel-Fro vs attn_bwd {e:.3e}"


@pytest.mark.gpu
def test_noalloc_at_its_row_limit_after_smaller_calls(lib, orc):
    """B*H*N exactly at the 4,194,304-row limit (the whole 16 MiB array), run
    after the smaller calls above left their contents in it: bit-identical to
    the three-kernel backward with a caller workspace (the same kernels), and
    sampled dQ rows of the first and last head against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_67_gb300 as ex
    B, H, N, d, causal = 1, 64, 65536, 64, True
    assert B * H * N == 1 << 22
    scale = float(torch.tensor(d ** -0.5, dtype=torch.float32))
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(777)
    q, k, v, do = (torch.randn((B, H, N, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(4))
    o, lse = ex.forward(q, k, v, causal, scale)
    ws = torch.empty(ex.attn_bwd_workspace_size(B, H, N, d, causal), dtype=torch.uint8, device=dev)
    ref = [torch.empty_like(q) for _ in range(3)]
    stream = torch.cuda.current_stream().cuda_stream
    # d = 64: attn_bwd takes the same three-kernel path as the allocation-free call.
    ex.attn_bwd(q, k, v, o, do, lse, *ref, causal, scale, ws)
    got = [torch.full_like(q, float("nan")) for _ in range(3)]
    rc = lib.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(got[0]), _p(got[1]), _p(got[2]),
                              B, H, N, d, int(causal), scale, stream)
    assert rc == 0, ex.status_string(rc)
    torch.cuda.synchronize()
    assert ex.device_error() == 0
    for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
        assert torch.equal(a, b), f"{name} differs from attn_bwd at the row limit"
    rng = np.random.default_rng(5)
    rows = np.array(sorted({0, 1, N - 1} | set(int(x) for x in rng.choice(N, 40, replace=False))), dtype=np.int32)
    for h in (0, H - 1):
        f = [to_f64(t[0, h].cpu()) for t in (q, k, v, do)]
        dq_ref, _, _ = orc.head_bwd(*f, causal, scale, qrows=rows, krows=np.zeros(0, np.int32))
        e = rel_fro(to_f64(got[0][0, h].cpu())[rows], dq_ref)
        assert e <= TOL_GRAD_REL, f"head {h}: sampled dQ rel-Fro {e:.3e}"
