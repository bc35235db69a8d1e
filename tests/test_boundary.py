"""The C-ABI boundary on the host: the library loads, exports every entry point
include/exattn.h declares, and rejects bad arguments before touching CUDA.

No test here launches a kernel or needs a GPU: every call below fails
validation, which happens before the first CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "exattn.h")


@pytest.fixture(scope="module")
def lib():
    from exact_attention_67_gb300 import build as b
    b.build()
    from exact_attention_67_gb300 import _lib
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\**\s+\**([a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    from exact_attention_67_gb300._lib import EXPORTS
    assert sorted(EXPORTS) == names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    from exact_attention_67_gb300 import _lib
    for code in range(0, 10):
        s = _lib.status_string(code)
        assert s and s != "unknown exattn status"
    assert _lib.status_string(12345) == "unknown exattn status"
    assert lib.exattn_version() >= 100


# fake, never dereferenced, 256-byte aligned "device" addresses
P = [0x100000 + 0x100000 * i for i in range(12)]


def fwd(lib, q=P[0], k=P[1], v=P[2], o=P[3], lse=P[4], B=1, H=2, N=256, d=64, causal=0, scale=0.125):
    return lib.attn_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, None)


def bwd(lib, ptrs=None, B=1, H=2, N=256, d=64, causal=0, scale=0.125, ws=P[11], ws_bytes=1 << 20):
    p = list(P[:9]) if ptrs is None else ptrs
    return lib.attn_bwd(*p, B, H, N, d, causal, scale, ws, ws_bytes, None)


def test_fwd_validation(lib):
    assert fwd(lib, q=None) == 1
    assert fwd(lib, lse=None) == 1
    assert fwd(lib, B=0) == 2
    assert fwd(lib, H=-1) == 2
    assert fwd(lib, N=0) == 2
    assert fwd(lib, B=1 << 16, H=1 << 10, N=1 << 10) == 2   # B*H*N >= 2^31
    assert fwd(lib, d=96) == 4
    assert fwd(lib, d=256) == 4
    assert fwd(lib, scale=0.0) == 9
    assert fwd(lib, scale=-1.0) == 9
    assert fwd(lib, scale=float("inf")) == 9
    assert fwd(lib, scale=float("nan")) == 9
    assert fwd(lib, q=P[0] + 8) == 3
    assert fwd(lib, o=P[3] + 2) == 3
    assert fwd(lib, lse=P[4] + 2) == 3


def test_bwd_validation(lib):
    for i in range(9):
        p = list(P[:9])
        p[i] = None
        assert bwd(lib, ptrs=p) == 1
    assert bwd(lib, N=0) == 2
    assert bwd(lib, d=32) == 4
    assert bwd(lib, scale=float("nan")) == 9
    for i in (0, 1, 2, 3, 4, 6, 7, 8):
        p = list(P[:9])
        p[i] += 4
        assert bwd(lib, ptrs=p) == 3
    assert bwd(lib, ws=None) == 6
    assert bwd(lib, ws_bytes=16) == 6
    assert bwd(lib, ws=P[11] + 4) == 3


def test_workspace_size(lib):
    assert lib.attn_bwd_workspace_size(1, 2, 256, 64, 0) == 2048
    assert lib.attn_bwd_workspace_size(1, 16, 8192, 128, 1) == 16 * 8192 * 4
    assert lib.attn_bwd_workspace_size(1, 1, 3, 64, 0) == 256
    assert lib.attn_bwd_workspace_size(0, 1, 3, 64, 0) == 0
    assert lib.attn_bwd_workspace_size(1, 1, 3, 80, 0) == 0


def test_python_binding_rejects_bad_tensors():
    import torch
    from exact_attention_67_gb300 import _lib
    q = torch.zeros(1, 1, 8, 64, dtype=torch.float32)
    with pytest.raises(TypeError):
        _lib._shape4(q, "q")
    with pytest.raises(ValueError):
        _lib._shape4(torch.zeros(8, 64, dtype=torch.bfloat16), "q")
    with pytest.raises(ValueError):  # CPU tensor: the library has no CPU path
        _lib._shape4(torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16), "q")


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from exact_attention_67_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "library_path", lambda: str(tmp_path / "nope.so"))
    with pytest.raises(ImportError):
        _lib.load()


def test_stage_validation(lib):
    # attn_bwd_preprocess(o, dO, D, B, H, N, d, stream)
    assert lib.attn_bwd_preprocess(None, P[1], P[2], 1, 1, 8, 64, None) == 1
    assert lib.attn_bwd_preprocess(P[0], P[1], P[2], 1, 1, 0, 64, None) == 2
    assert lib.attn_bwd_preprocess(P[0], P[1], P[2], 1, 1, 8, 48, None) == 4
    assert lib.attn_bwd_preprocess(P[0] + 2, P[1], P[2], 1, 1, 8, 64, None) == 3
    assert lib.attn_bwd_preprocess(P[0], P[1], P[2] + 2, 1, 1, 8, 64, None) == 3
    # attn_bwd_dkdv(q, k, v, dO, lse, D, dk, dv, B, H, N, d, causal, scale, stream)
    args = list(P[:8])
    assert lib.attn_bwd_dkdv(*args[:5], None, *args[6:8], 1, 1, 8, 64, 0, 0.1, None) == 1
    assert lib.attn_bwd_dkdv(*args, 1, 1, 8, 64, 0, 0.0, None) == 9
    bad = list(args)
    bad[6] += 8
    assert lib.attn_bwd_dkdv(*bad, 1, 1, 8, 64, 0, 0.1, None) == 3
    # attn_bwd_dq(q, k, v, dO, lse, D, dq, B, H, N, d, causal, scale, stream)
    args = list(P[:7])
    assert lib.attn_bwd_dq(*args[:6], None, 1, 1, 8, 64, 0, 0.1, None) == 1
    assert lib.attn_bwd_dq(*args, 1, 1, 8, 128, 1, float("inf"), None) == 9
    assert lib.attn_bwd_dq(*args, -1, 1, 8, 128, 1, 0.1, None) == 2
    # attn_bwd_d_and_dq(q, k, v, o, dO, lse, D, dq, B, H, N, d, causal, scale, stream)
    args = list(P[:8])
    for i in range(8):
        nul = list(args)
        nul[i] = None
        assert lib.attn_bwd_d_and_dq(*nul, 1, 1, 8, 64, 0, 0.1, None) == 1
    assert lib.attn_bwd_d_and_dq(*args, 1, 1, 8, 64, 0, float("nan"), None) == 9
    assert lib.attn_bwd_d_and_dq(*args, 1, 1, 8, 96, 0, 0.1, None) == 4
    assert lib.attn_bwd_d_and_dq(*args, 1, 0, 8, 64, 0, 0.1, None) == 2
    for i, off in ((3, 8), (4, 8), (6, 2), (7, 8)):  # o, dO, D, dq misaligned
        bad = list(args)
        bad[i] += off
        assert lib.attn_bwd_d_and_dq(*bad, 1, 1, 8, 64, 0, 0.1, None) == 3


def test_ex_validation(lib):
    """attn_fwd_ex / attn_bwd_ex reject a bad type code and bad strides before
    any CUDA call (fake, 16-byte-aligned pointers; nothing is launched)."""
    from exact_attention_67_gb300._lib import Strides
    P = [0x10000 * (i + 1) for i in range(10)]
    B, H, N, d = 1, 2, 8, 64
    good = Strides(H * N * d, N * d, d)
    bnhd = Strides(N * H * d, d, H * d)

    def fwd(dt=0, s=(good, good, good, good), d_=d, N_=N, window=0):
        return lib.attn_fwd_ex(dt, P[0], s[0], P[1], s[1], P[2], s[2], P[3], s[3], P[4], B, H, N_, d_, 1, window,
                               0.125, None)

    assert fwd(dt=2) == 4 and fwd(dt=-1) == 4
    assert fwd(window=-1) == 9
    assert fwd(d_=80) == 4
    assert fwd(s=(good, Strides(H * N * d, N * d, 60), good, good)) == 3   # not a multiple of 8 elements
    assert fwd(s=(good, good, Strides(-8, N * d, d), good)) == 3          # negative
    assert fwd(s=(good, good, good, Strides(H * N * d, N * d, 1 << 36))) == 3
    assert fwd(s=(good, good, good, Strides(H * N * d, N * d, 0))) == 2   # zero along N > 1
    assert fwd(s=(Strides(0, 0, d), good, good, good), N_=N) == 2         # zero along H = 2
    assert lib.attn_fwd_ex(0, None, good, P[1], good, P[2], good, P[3], good, P[4], B, H, N, d, 1, 0, 0.125,
                           None) == 1
    assert lib.attn_fwd_ex(1, P[0] + 8, bnhd, P[1], good, P[2], good, P[3], good, P[4], B, H, N, d, 1, 0, 0.125,
                           None) == 3

    def bwd(dt=0, ss=None, ws_bytes=1 << 20, scale=0.125, window=0):
        s = ss or [good] * 8
        return lib.attn_bwd_ex(dt, P[0], s[0], P[1], s[1], P[2], s[2], P[3], s[3], P[4], s[4], P[5], P[6], s[5],
                               P[7], s[6], P[8], s[7], B, H, N, d, 0, window, scale, P[9], ws_bytes, None)

    assert bwd(dt=3) == 4
    assert bwd(window=-5) == 9
    assert bwd(scale=0.0) == 9
    bad = [good] * 8
    bad[6] = Strides(H * N * d, N * d + 4, d)
    assert bwd(ss=bad) == 3
    assert bwd(ws_bytes=16) == 6


def test_o32_validation(lib):
    """attn_fwd_o32 / attn_bwd_o32 reject a missing or misaligned fp32 O, and
    otherwise validate like the _ex calls (fake pointers; nothing launched)."""
    from exact_attention_67_gb300._lib import Strides
    P = [0x10000 * (i + 1) for i in range(10)]
    B, H, N, d = 1, 2, 8, 64
    good = Strides(H * N * d, N * d, d)

    def fwd(o32=P[5], dt=0, window=0):
        return lib.attn_fwd_o32(dt, P[0], good, P[1], good, P[2], good, P[3], good, P[4], o32, B, H, N, d, 1,
                                window, 0.125, None)

    assert fwd(o32=None) == 1
    assert fwd(o32=P[5] + 4) == 3
    assert fwd(dt=2) == 4
    assert fwd(window=-1) == 9

    def bwd(o32=P[3], ws_bytes=1 << 20, scale=0.125):
        return lib.attn_bwd_o32(0, P[0], good, P[1], good, P[2], good, o32, P[4], good, P[5], P[6], good, P[7],
                                good, P[8], good, B, H, N, d, 0, 0, scale, P[9], ws_bytes, None)

    assert bwd(o32=None) == 1
    assert bwd(o32=P[3] + 8) == 3
    assert bwd(scale=0.0) == 9
    assert bwd(ws_bytes=16) == 6


def test_varlen_validation(lib):
    """attn_fwd_varlen / attn_bwd_varlen reject a missing or misaligned offset
    table and bad sizes before any CUDA call (nothing is launched)."""
    from exact_attention_67_gb300._lib import Strides
    P = [0x10000 * (i + 1) for i in range(12)]
    H, d, total = 2, 64, 40
    s = Strides(0, d, H * d)

    def fwd(cu=P[5], B=3, maxlen=20, tot=total, window=0, dt=0):
        return lib.attn_fwd_varlen(dt, P[0], s, P[1], s, P[2], s, P[3], s, P[4], cu, B, H, maxlen, tot, d, 1,
                                   window, 0.125, None)

    assert fwd(cu=None) == 1
    assert fwd(cu=P[5] + 2) == 3
    assert fwd(tot=0) == 2 and fwd(B=0) == 2 and fwd(maxlen=0) == 2
    assert fwd(window=-1) == 9 and fwd(dt=7) == 4
    assert lib.attn_fwd_varlen(0, P[0], Strides(0, d, 60), P[1], s, P[2], s, P[3], s, P[4], P[5], 3, H, 20, total,
                               d, 1, 0, 0.125, None) == 3

    def bwd(cu=P[10], ws=1 << 20):
        return lib.attn_bwd_varlen(0, P[0], s, P[1], s, P[2], s, P[3], s, P[4], s, P[5], P[6], s, P[7], s, P[8],
                                   s, cu, 3, H, 20, total, d, 1, 0, 0.125, P[9], ws, None)

    assert bwd(cu=None) == 1
    assert bwd(ws=8) == 6


def test_decode_validation(lib):
    """attn_fwd_decode rejects queries that would see no key and bad sizes
    before any CUDA call; the workspace is zero when no key split is needed."""
    from exact_attention_67_gb300._lib import Strides
    P = [0x10000 * (i + 1) for i in range(8)]
    d = 128

    def st(H, n):
        return Strides(H * n * d, n * d, d)

    def dec(B=1, H=2, Nq=4, Nk=8, causal=1, window=0, ws=None, wsb=0):
        return lib.attn_fwd_decode(0, P[0], st(H, Nq), P[1], st(H, Nk), P[2], st(H, Nk), P[3], st(H, Nq), P[4], B, H,
                                   Nq, Nk, d, causal, window, 0.125, ws, wsb, None)

    assert dec(Nq=9, Nk=8) == 2                       # causal: query 0 would see no key
    assert dec(Nq=9, Nk=8, causal=0, window=3) == 2
    assert dec(Nq=0) == 2 and dec(Nk=0) == 2
    assert dec(window=-1) == 9
    assert lib.attn_fwd_decode_workspace_size(1, 2, 4, 8, 80) == 0
    assert lib.attn_fwd_decode_workspace_size(64, 16, 1, 1024, d) == 0   # enough CTAs without a split
    ws = lib.attn_fwd_decode_workspace_size(1, 1, 1, 32768, d)
    assert ws > 0
    assert dec(B=1, H=1, Nq=1, Nk=32768, ws=None) == 6
    assert dec(B=1, H=1, Nq=1, Nk=32768, ws=P[5], wsb=ws - 1) == 6


def test_decode_plan_sizes(lib):
    """The decode call's workspace follows its plan: at d = 128 with at most
    12 queries the decode kernel (16 query columns per split row), otherwise
    the forward kernel with split keys (256-row query pairs).  The split
    count is the one whose grid ends first when a CTA costs its key tiles
    plus three, CTAs run in waves of 152 (one per SM), at most about two
    waves of CTAs, at least four key tiles per split for the decode kernel
    and two for the forward's.  Sizes: split partials fp32
    [splits, B*H, rows, d] plus two fp32 logsumexps [splits, B*H, rows], each
    256-byte aligned; no workspace without a split."""
    def size(splits, bh, rows, d):
        n = splits * bh * rows
        up = lambda x: (x + 255) // 256 * 256
        return up(n * d * 4) + 2 * up(n * 4)
    # B4 H32 Nk32768 d128: 128 heads fill one wave unsplit (3 + 256 = 259);
    # two splits would take two waves of 3 + 128 (262).
    assert lib.attn_fwd_decode_workspace_size(4, 32, 1, 32768, 128) == 0
    assert lib.attn_fwd_decode_workspace_size(4, 32, 12, 32768, 128) == 0
    assert lib.attn_fwd_decode_workspace_size(4, 32, 13, 32768, 128) == 0
    # d = 64 takes the forward kernel; 128 heads, 128 key tiles: unsplit.
    assert lib.attn_fwd_decode_workspace_size(8, 16, 1, 16384, 64) == 0
    # One head, 1024 key tiles: 147 splits of 7 tiles fill one wave (cost
    # 10); 8 tiles cost 11, and 4-6 tiles need a second wave (14 or more).
    assert lib.attn_fwd_decode_workspace_size(1, 1, 1, 131072, 128) == size(147, 1, 16, 128)
    assert lib.attn_fwd_decode_workspace_size(1, 1, 16, 131072, 128) == size(147, 1, 256, 128)
    # 16 heads, 256 tiles: 9 splits of 29 tiles are 144 CTAs in one wave
    # (32); 10 splits make 160 CTAs, two waves (58); 19 make two full
    # waves (34).
    assert lib.attn_fwd_decode_workspace_size(2, 8, 1, 32768, 128) == size(9, 16, 16, 128)
    # 8 heads, 512 tiles: 19 splits of 27 tiles, exactly 152 CTAs.
    assert lib.attn_fwd_decode_workspace_size(1, 8, 1, 65536, 128) == size(19, 8, 16, 128)
    # 8 tiles: two splits of four (3 + 4) beat one CTA of eight (3 + 8).
    assert lib.attn_fwd_decode_workspace_size(1, 1, 1, 1000, 128) == size(2, 1, 16, 128)


def test_decode_plan_properties(lib):
    """Over a sweep of shapes the plan the workspace implies keeps its
    limits: at most 512 splits (the merge's limit) and about two waves of
    152 CTAs, every split holding at least four key tiles in the decode
    kernel (two in the forward's) unless there is one split, and the
    workspace exactly the partials' layout."""
    def split_count(B, H, Nq, Nk, d):
        rows = 16 if (Nq <= 12 and d == 128) else (Nq + 255) // 256 * 256
        per = B * H * rows * (d * 4 + 8)
        ws = lib.attn_fwd_decode_workspace_size(B, H, Nq, Nk, d)
        if ws == 0:
            return 1
        for s in range(2, 513):
            n = s * B * H * rows
            if ws == (n * d * 4 + 255) // 256 * 256 + 2 * ((n * 4 + 255) // 256 * 256):
                return s
        raise AssertionError(f"workspace {ws} matches no split count ({per} bytes per split)")
    for B, H in ((1, 1), (1, 3), (2, 8), (1, 40), (4, 32), (8, 64)):
        for Nk in (1, 127, 128, 1000, 5000, 32768, 131072, 1 << 20):
            if B * H * Nk >= 1 << 31:
                continue
            for Nq, d in ((1, 128), (12, 128), (13, 128), (1, 64), (300, 128)):
                s = split_count(B, H, Nq, Nk, d)
                nkt = (Nk + 127) // 128
                units = B * H * ((Nq + 255) // 256 if not (Nq <= 12 and d == 128) else 1)
                floor = 4 if (Nq <= 12 and d == 128) else 2
                assert 1 <= s <= 512
                assert s == 1 or units * s <= 2 * 152, (B, H, Nq, Nk, d, s)
                assert s == 1 or -(-nkt // s) >= floor, (B, H, Nq, Nk, d, s)


def test_host_path_rejects_bad_tensors():
    """fwd_bwd_from_host checks its host tensors before any device work."""
    import torch
    from exact_attention_67_gb300.host import fwd_bwd_from_host
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fwd_bwd_from_host(q, q, q[:, :1], q)  # shape mismatch
    with pytest.raises(ValueError):
        fwd_bwd_from_host(q.float(), q.float(), q.float(), q.float())  # fp32
    with pytest.raises(ValueError):
        t = q.transpose(1, 2)
        fwd_bwd_from_host(t, t, t, t)  # not contiguous
    with pytest.raises(ValueError):
        fwd_bwd_from_host(q, q, q, q, out=(q, q, q, q, q))  # lse of the wrong type and shape


def test_host_entry_point_validates_before_any_copy():
    """attn_fwd_bwd_host rejects bad arguments before touching the device."""
    import torch
    from exact_attention_67_gb300 import _lib
    lib = _lib.load()
    assert lib.attn_fwd_bwd_host_workspace_size(1, 2, 128, 96, 1) == 0     # d not 64 or 128
    need = lib.attn_fwd_bwd_host_workspace_size(1, 2, 128, 64, 1)
    assert need >= 8 * 2 * 128 * 64 * 2 + 2 * 2 * 128 * 4
    x = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 128)
    small = torch.zeros(16, dtype=torch.uint8)  # far too small (and not device memory: never touched)
    p = [t.data_ptr() for t in (x, x, x, x, x, lse, x, x, x)]
    W, V, N_ = _lib.EXATTN_OK + 6, _lib.EXATTN_OK + 9, _lib.EXATTN_OK + 1
    assert lib.attn_fwd_bwd_host(0, *p, 1, 2, 128, 64, 1, 0.125, small.data_ptr(), 16, 2, None, None, None, None) == W
    assert lib.attn_fwd_bwd_host(0, *p, 1, 2, 128, 64, 1, 0.125, small.data_ptr(), need, 0, None, None, None, None) == V
    assert lib.attn_fwd_bwd_host(0, *p, 1, 2, 128, 64, 1, -1.0, small.data_ptr(), need, 2, None, None, None, None) == V
    assert lib.attn_fwd_bwd_host(0, None, *p[1:], 1, 2, 128, 64, 1, 0.125, small.data_ptr(), need, 2, None, None,
                                 None, None) == N_
    assert lib.attn_fwd_bwd_host(7, *p, 1, 2, 128, 64, 1, 0.125, small.data_ptr(), need, 2, None, None, None,
                                 None) == _lib.EXATTN_OK + 4


def test_binding_argument_counts_match_the_header():
    """Every C prototype in include/exattn.h has as many parameters as the
    ctypes binding declares for it (a mismatch would pass wrong arguments)."""
    import re
    from exact_attention_67_gb300 import _lib
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = open(os.path.join(root, "include", "exattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)  # drop comments
    protos = re.findall(r"^\s*(?:const\s+)?[\w]+\s*\**\s*(\w+)\s*\(([^;{]*?)\)\s*;", src, flags=re.M | re.S)
    lib = _lib.load()
    seen = 0
    for name, params in protos:
        if name not in _lib.EXPORTS:
            continue
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(getattr(lib, name).argtypes) == n, name
        seen += 1
    assert seen == len(_lib.EXPORTS)
