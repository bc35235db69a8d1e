"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library and its Python binding never touch it, and it never touches them:
the two sides share nothing but the seeded input generator, which holds none
of the method's arithmetic.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, POSIX threads);
this module compiles it with gcc on first use (or via :func:`build`) and
wraps it with ctypes.  Arrays are numpy float64, laid out [B, H, N, d].

Functions and what they follow (pages cited by title and section):

* :func:`attention_fwd` -- the standard three-step attention of
  "Gemini 3 Flash的注意力内核重写：算子融合如何实现亚毫秒级推理"
  §传统注意力计算的内存带宽瓶颈, with the max-subtracted softmax of
  "提示词再优也救不了的性能黑洞：Transformer注意力计算冗余分析（含FlashAttention-3
  内核级优化验证数据）" §2.2 and its causal flag (第一章); returns O and the
  per-row natural-log logsumexp (the row statistics kept by the
  "Gemini 3 Flash…" page §4 重计算).
* :func:`attention_bwd` -- the analytic gradient (textbook softmax VJP).
* :func:`attention_fwd_online` -- the one-pass running-max/running-sum form of
  "Gemini 3 Flash…" §3 在线softmax算法, for the equivalence pin only.

Parity pins: every function here is checked against closed forms,
invariants, central finite differences and an independent library routine in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc -O2, no fast-math, no FMA contraction (x86 and Arm hosts agree)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


class OracleLib:
    """ctypes view of one compiled copy of attn_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        i, d = ctypes.c_int, ctypes.c_double
        lib.oracle_head_fwd_rows.argtypes = [dp, dp, dp, i, i, i, i, d, ip, i, dp, dp, i]
        lib.oracle_head_fwd_rows.restype = i
        lib.oracle_head_fwd_online.argtypes = [dp, dp, dp, i, i, i, i, d, i, dp, dp]
        lib.oracle_head_fwd_online.restype = i
        lib.oracle_head_bwd_rows.argtypes = [dp, dp, dp, dp, i, i, i, i, d, ip, i, ip, i,
                                             dp, dp, dp, dp, dp, i]
        lib.oracle_head_bwd_rows.restype = i
        lib.oracle_default_threads.argtypes = []
        lib.oracle_default_threads.restype = i
        self.lib = lib
        self.path = path

    def default_threads(self) -> int:
        return int(self.lib.oracle_default_threads())

    def head_fwd(self, q, k, v, causal: bool, scale: float, rows=None, nthreads=None, window: int = 0):
        """One head: q, k, v are [N, d].  Returns (o[len(rows), d], lse[len(rows)]).
        ``window`` W > 0 keeps only keys with i - j < W (and j - i < W when not causal)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        N, dd = q.shape
        assert k.shape == (N, dd) and v.shape == (N, dd)
        r = _idx(rows, N)
        o = np.empty((r.size, dd), np.float64)
        lse = np.empty((r.size,), np.float64)
        nt = self.default_threads() if nthreads is None else int(nthreads)
        _check(self.lib.oracle_head_fwd_rows(_dptr(q), _dptr(k), _dptr(v), N, dd,
                                             int(bool(causal)), int(window), float(scale), _iptr(r),
                                             r.size, _dptr(o), _dptr(lse), nt), "fwd")
        return o, lse

    def head_bwd(self, q, k, v, dO, causal: bool, scale: float, qrows=None, krows=None,
                 nthreads=None, want_stats=False, window: int = 0):
        """One head.  Returns (dq[len(qrows), d], dk[len(krows), d], dv[len(krows), d])
        and, if want_stats, also (lse[N], D[N]) (NaN where not computed)."""
        q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
        N, dd = q.shape
        qr = _idx(qrows, N)
        kr = _idx(krows, N)
        dq = np.empty((qr.size, dd), np.float64)
        dk = np.empty((kr.size, dd), np.float64)
        dv = np.empty((kr.size, dd), np.float64)
        lse = np.empty((N,), np.float64)
        D = np.empty((N,), np.float64)
        nt = self.default_threads() if nthreads is None else int(nthreads)
        _check(self.lib.oracle_head_bwd_rows(_dptr(q), _dptr(k), _dptr(v), _dptr(dO), N, dd,
                                             int(bool(causal)), int(window), float(scale), _iptr(qr),
                                             qr.size, _iptr(kr), kr.size, _dptr(dq), _dptr(dk), _dptr(dv),
                                             _dptr(lse), _dptr(D), nt), "bwd")
        if want_stats:
            return dq, dk, dv, lse, D
        return dq, dk, dv

    def head_fwd_online(self, q, k, v, causal: bool, scale: float, tile_cols: int, window: int = 0):
        """One head, one-pass online-softmax forward with key tiles of tile_cols."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        N, dd = q.shape
        o = np.empty((N, dd), np.float64)
        lse = np.empty((N,), np.float64)
        _check(self.lib.oracle_head_fwd_online(_dptr(q), _dptr(k), _dptr(v), N, dd,
                                               int(bool(causal)), int(window), float(scale),
                                               int(tile_cols), _dptr(o), _dptr(lse)), "fwd_online")
        return o, lse

    # ---- whole-tensor helpers, [B, H, N, d] ----
    def attention_fwd(self, q, k, v, causal: bool, scale: float, nthreads=None, window: int = 0):
        """[B, H, N, d] fp64 -> (O [B, H, N, d], lse [B, H, N]), natural log."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, dd = q.shape
        o = np.empty_like(q)
        lse = np.empty((B, H, N), np.float64)
        for b in range(B):
            for h in range(H):
                o[b, h], lse[b, h] = self.head_fwd(q[b, h], k[b, h], v[b, h], causal, scale,
                                                   nthreads=nthreads, window=window)
        return o, lse

    def attention_bwd(self, q, k, v, dO, causal: bool, scale: float, nthreads=None, window: int = 0):
        """[B, H, N, d] fp64 -> (dQ, dK, dV), each [B, H, N, d]."""
        q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
        B, H, N, dd = q.shape
        dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
        for b in range(B):
            for h in range(H):
                dq[b, h], dk[b, h], dv[b, h] = self.head_bwd(q[b, h], k[b, h], v[b, h],
                                                             dO[b, h], causal, scale,
                                                             nthreads=nthreads, window=window)
        return dq, dk, dv

    def attention_fwd_online(self, q, k, v, causal: bool, scale: float, tile_cols: int, window: int = 0):
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, dd = q.shape
        o = np.empty_like(q)
        lse = np.empty((B, H, N), np.float64)
        for b in range(B):
            for h in range(H):
                o[b, h], lse[b, h] = self.head_fwd_online(q[b, h], k[b, h], v[b, h], causal,
                                                          scale, tile_cols, window)
        return o, lse


def _load() -> OracleLib:
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build())
        return _lib


def default_threads() -> int:
    return _load().default_threads()


def _dptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _idx(rows, N) -> np.ndarray:
    if rows is None:
        return np.arange(N, dtype=np.int32)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1))


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with status {rc}")


def head_fwd(*a, **kw):
    return _load().head_fwd(*a, **kw)


def head_bwd(*a, **kw):
    return _load().head_bwd(*a, **kw)


def head_fwd_online(*a, **kw):
    return _load().head_fwd_online(*a, **kw)


def attention_fwd(*a, **kw):
    return _load().attention_fwd(*a, **kw)


def attention_bwd(*a, **kw):
    return _load().attention_bwd(*a, **kw)


def attention_fwd_online(*a, **kw):
    return _load().attention_fwd_online(*a, **kw)
