"""ctypes binding of libexattn.so: the C ABI of include/exattn.h under the
same names, argument marshalling only.  Every step of the computation runs
in the library's CUDA kernels; there is no other implementation to fall back
to, and a missing library raises instead of degrading."""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

EXATTN_OK = 0
EXATTN_ERR_CUDA = 7
STATUS_NAMES = {
    0: "EXATTN_OK", 1: "EXATTN_ERR_NULL", 2: "EXATTN_ERR_SHAPE", 3: "EXATTN_ERR_ALIGN",
    4: "EXATTN_ERR_UNSUPPORTED", 5: "EXATTN_ERR_ARCH", 6: "EXATTN_ERR_WORKSPACE",
    7: "EXATTN_ERR_CUDA", 8: "EXATTN_ERR_TIMEOUT", 9: "EXATTN_ERR_VALUE",
}
# Every entry point include/exattn.h declares.
EXPORTS = ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_bwd_preprocess", "attn_bwd_dkdv",
           "attn_bwd_dq", "attn_bwd_d_and_dq", "attn_fwd_ex", "attn_bwd_ex", "attn_fwd_o32", "attn_bwd_o32", "attn_fwd_varlen",
           "attn_bwd_varlen",
           "attn_fwd_decode_workspace_size", "attn_fwd_decode", "attn_bwd_noalloc",
           "attn_fwd_bwd_host_workspace_size", "attn_fwd_bwd_host",
           "exattn_status_string", "exattn_last_cuda_error",
           "exattn_device_error", "exattn_device_error_poll", "exattn_watchdog_selftest", "exattn_version")

EXATTN_DTYPE_BF16 = 0
EXATTN_DTYPE_F16 = 1


class Strides(ctypes.Structure):
    """C ``exattn_strides``: element strides of a [B, H, N, d] view (d contiguous)."""
    _fields_ = [("b_stride", ctypes.c_longlong), ("h_stride", ctypes.c_longlong),
                ("n_stride", ctypes.c_longlong)]


class ExattnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libexattn.so; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise ImportError(
                    f"{path} is missing: build it with `python -m exact_attention_67_gb300.build` "
                    "(the CUDA library is the only implementation)")
            _build.build()
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        lib.attn_fwd.restype = i
        lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
        lib.attn_bwd.restype = i
        lib.attn_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, vp]
        lib.attn_bwd_preprocess.restype = i
        lib.attn_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        lib.attn_bwd_dkdv.restype = i
        lib.attn_bwd_dq.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        lib.attn_bwd_dq.restype = i
        lib.attn_bwd_d_and_dq.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        lib.attn_bwd_d_and_dq.restype = i
        lib.exattn_device_error_poll.argtypes = [vp, vp]
        lib.exattn_device_error_poll.restype = i
        S = Strides
        lib.attn_fwd_ex.argtypes = [i, vp, S, vp, S, vp, S, vp, S, vp, i, i, i, i, i, i, f, vp]
        lib.attn_fwd_ex.restype = i
        lib.attn_bwd_ex.argtypes = [i, vp, S, vp, S, vp, S, vp, S, vp, S, vp, vp, S, vp, S, vp, S, i, i, i, i, i, i,
                                    f, vp, sz, vp]
        lib.attn_bwd_ex.restype = i
        lib.attn_fwd_o32.argtypes = [i, vp, S, vp, S, vp, S, vp, S, vp, vp, i, i, i, i, i, i, f, vp]
        lib.attn_fwd_o32.restype = i
        lib.attn_bwd_o32.argtypes = [i, vp, S, vp, S, vp, S, vp, vp, S, vp, vp, S, vp, S, vp, S, i, i, i, i, i, i, f,
                                     vp, sz, vp]
        lib.attn_bwd_o32.restype = i
        lib.attn_fwd_varlen.argtypes = [i, vp, S, vp, S, vp, S, vp, S, vp, vp, i, i, i, i, i, i, i, f, vp]
        lib.attn_fwd_varlen.restype = i
        lib.attn_bwd_varlen.argtypes = [i, vp, S, vp, S, vp, S, vp, S, vp, S, vp, vp, S, vp, S, vp, S, vp, i, i, i, i,
                                        i, i, i, f, vp, sz, vp]
        lib.attn_bwd_varlen.restype = i
        lib.attn_fwd_decode_workspace_size.argtypes = [i, i, i, i, i]
        lib.attn_fwd_decode_workspace_size.restype = sz
        lib.attn_fwd_decode.argtypes = [i, vp, S, vp, S, vp, S, vp, S, vp, i, i, i, i, i, i, i, f, vp, sz, vp]
        lib.attn_fwd_decode.restype = i
        lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        lib.attn_bwd_noalloc.restype = i
        lib.attn_fwd_bwd_host_workspace_size.argtypes = [i, i, i, i, i]
        lib.attn_fwd_bwd_host_workspace_size.restype = sz
        lib.attn_fwd_bwd_host.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, i, vp, vp, vp,
                                          vp]
        lib.attn_fwd_bwd_host.restype = i
        lib.attn_bwd_workspace_size.argtypes = [i, i, i, i, i]
        lib.attn_bwd_workspace_size.restype = sz
        lib.exattn_status_string.argtypes = [i]
        lib.exattn_status_string.restype = ctypes.c_char_p
        lib.exattn_last_cuda_error.argtypes = []
        lib.exattn_last_cuda_error.restype = ctypes.c_char_p
        lib.exattn_device_error.argtypes = []
        lib.exattn_device_error.restype = i
        lib.exattn_watchdog_selftest.argtypes = [ctypes.c_uint, vp]
        lib.exattn_watchdog_selftest.restype = i
        lib.exattn_version.argtypes = []
        lib.exattn_version.restype = i
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().exattn_status_string(int(status)).decode()


def last_cuda_error() -> str:
    """C ``exattn_last_cuda_error``: the failing CUDA call behind the calling
    thread's last EXATTN_ERR_CUDA ("" if none)."""
    return load().exattn_last_cuda_error().decode()


def _check(status: int):
    if status != EXATTN_OK:
        msg = status_string(status)
        if status == EXATTN_ERR_CUDA:
            msg += f" ({last_cuda_error()})"
        raise ExattnError(status, msg)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, device=None):
    """The cudaStream_t of a torch stream (or a raw handle); None is the
    current stream of ``device`` (of the current device if None)."""
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _device_of(*ts):
    """The one CUDA device of the given tensors (None entries skipped).  The
    C ABI runs on the current device, so operands on another device, or on
    several, are rejected here, before anything is launched."""
    dev = None
    for t in ts:
        if t is None or isinstance(t, int):
            continue
        if not t.is_cuda:
            raise ValueError("all device operands must be CUDA tensors")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"operands are on different devices ({dev} and {t.device})")
    return dev


def _shape4(t: torch.Tensor, name: str):
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, H, N, d], got {tuple(t.shape)}")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous [B, H, N, d]")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return tuple(t.shape)


_DTYPES = {torch.bfloat16: EXATTN_DTYPE_BF16, torch.float16: EXATTN_DTYPE_F16}


def _view4(t: torch.Tensor, name: str):
    """Shape, element type code and C strides of a [B, H, N, d] view whose d
    axis is contiguous (any b, h, n strides the library accepts)."""
    if t.dim() != 4:
        raise ValueError(f"{name} must be a [B, H, N, d] view, got {tuple(t.shape)}")
    if t.dtype not in _DTYPES:
        raise TypeError(f"{name} must be bfloat16 or float16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.shape[3] > 1 and t.stride(3) != 1:
        raise ValueError(f"{name}: the d axis must be contiguous (stride 1), got stride {t.stride(3)}")
    return tuple(t.shape), _DTYPES[t.dtype], Strides(t.stride(0), t.stride(1), t.stride(2))


def attn_fwd_ex(q, k, v, o, lse, causal: bool, scale: float, stream=None, window: int = 0) -> None:
    """C ``attn_fwd_ex``: q, k, v, o are [B, H, N, d] views (d contiguous) of one
    type, bf16 or f16 (a [B, N, H, d] tensor passes as ``x.transpose(1, 2)``);
    lse fp32 contiguous [B, H, N]; ``window`` > 0 for sliding-window attention."""
    (B, H, N, d), dt, sq = _view4(q, "q")
    views = [_view4(t, n) for n, t in (("k", k), ("v", v), ("o", o))]
    for n, (shape, dtn, _) in zip(("k", "v", "o"), views):
        if shape != (B, H, N, d) or dtn != dt:
            raise ValueError(f"{n} shape/dtype differs from q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, H, N]")
    dev = _device_of(q, k, v, o, lse)
    with torch.cuda.device(dev):
        _check(load().attn_fwd_ex(dt, _ptr(q), sq, _ptr(k), views[0][2], _ptr(v), views[1][2], _ptr(o), views[2][2],
                                  _ptr(lse), B, H, N, d, int(bool(causal)), int(window), float(scale),
                                  _stream(stream, dev)))


def attn_bwd_ex(q, k, v, o, dO, lse, dq, dk, dv, causal: bool, scale: float, workspace, stream=None,
                window: int = 0) -> None:
    """C ``attn_bwd_ex`` on [B, H, N, d] views of one 16-bit type (``window`` as
    in the forward)."""
    (B, H, N, d), dt, sq = _view4(q, "q")
    names = ("k", "v", "o", "dO", "dq", "dk", "dv")
    views = [_view4(t, n) for n, t in zip(names, (k, v, o, dO, dq, dk, dv))]
    for n, (shape, dtn, _) in zip(names, views):
        if shape != (B, H, N, d) or dtn != dt:
            raise ValueError(f"{n} shape/dtype differs from q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, H, N]")
    s = [vw[2] for vw in views]
    ws_bytes = workspace.numel() * workspace.element_size()
    dev = _device_of(q, k, v, o, dO, lse, dq, dk, dv, workspace)
    with torch.cuda.device(dev):
        _check(load().attn_bwd_ex(dt, _ptr(q), sq, _ptr(k), s[0], _ptr(v), s[1], _ptr(o), s[2], _ptr(dO), s[3],
                                  _ptr(lse), _ptr(dq), s[4], _ptr(dk), s[5], _ptr(dv), s[6], B, H, N, d,
                                  int(bool(causal)), int(window), float(scale), _ptr(workspace), ws_bytes,
                                  _stream(stream, dev)))


def _check_o32(o32, B, H, N, d):
    if o32.dtype != torch.float32 or tuple(o32.shape) != (B, H, N, d) or not o32.is_contiguous():
        raise ValueError("o32 must be contiguous float32 [B, H, N, d]")


def attn_fwd_o32(q, k, v, o, lse, o32, causal: bool, scale: float, stream=None, window: int = 0) -> None:
    """C ``attn_fwd_o32``: ``attn_fwd_ex`` that also writes ``o32``, an fp32
    contiguous [B, H, N, d] copy of O before its rounding (for ``attn_bwd_o32``)."""
    (B, H, N, d), dt, sq = _view4(q, "q")
    views = [_view4(t, n) for n, t in (("k", k), ("v", v), ("o", o))]
    for n, (shape, dtn, _) in zip(("k", "v", "o"), views):
        if shape != (B, H, N, d) or dtn != dt:
            raise ValueError(f"{n} shape/dtype differs from q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, H, N]")
    _check_o32(o32, B, H, N, d)
    dev = _device_of(q, k, v, o, lse, o32)
    with torch.cuda.device(dev):
        _check(load().attn_fwd_o32(dt, _ptr(q), sq, _ptr(k), views[0][2], _ptr(v), views[1][2], _ptr(o),
                                   views[2][2], _ptr(lse), _ptr(o32), B, H, N, d, int(bool(causal)), int(window),
                                   float(scale), _stream(stream, dev)))


def attn_bwd_o32(q, k, v, o32, dO, lse, dq, dk, dv, causal: bool, scale: float, workspace, stream=None,
                 window: int = 0) -> None:
    """C ``attn_bwd_o32``: ``attn_bwd_ex`` with the row terms D_i taken from the
    fp32 ``o32`` that ``attn_fwd_o32`` wrote (O itself is not needed)."""
    (B, H, N, d), dt, sq = _view4(q, "q")
    names = ("k", "v", "dO", "dq", "dk", "dv")
    views = [_view4(t, n) for n, t in zip(names, (k, v, dO, dq, dk, dv))]
    for n, (shape, dtn, _) in zip(names, views):
        if shape != (B, H, N, d) or dtn != dt:
            raise ValueError(f"{n} shape/dtype differs from q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, H, N]")
    _check_o32(o32, B, H, N, d)
    s = [vw[2] for vw in views]
    ws_bytes = workspace.numel() * workspace.element_size()
    dev = _device_of(q, k, v, o32, dO, lse, dq, dk, dv, workspace)
    with torch.cuda.device(dev):
        _check(load().attn_bwd_o32(dt, _ptr(q), sq, _ptr(k), s[0], _ptr(v), s[1], _ptr(o32), _ptr(dO), s[2],
                                   _ptr(lse), _ptr(dq), s[3], _ptr(dk), s[4], _ptr(dv), s[5], B, H, N, d,
                                   int(bool(causal)), int(window), float(scale), _ptr(workspace), ws_bytes,
                                   _stream(stream, dev)))


def _packed3(t: torch.Tensor, name: str):
    """Shape, type code and C strides of a packed [total, H, d] tensor (d contiguous)."""
    if t.dim() != 3:
        raise ValueError(f"{name} must be a packed [total, H, d] tensor, got {tuple(t.shape)}")
    if t.dtype not in _DTYPES:
        raise TypeError(f"{name} must be bfloat16 or float16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.shape[2] > 1 and t.stride(2) != 1:
        raise ValueError(f"{name}: the d axis must be contiguous")
    return tuple(t.shape), _DTYPES[t.dtype], Strides(0, t.stride(1), t.stride(0))


def _cu(cu_seqlens):
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_cuda:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor of B + 1 offsets")
    return cu_seqlens.numel() - 1


def attn_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen: int, causal: bool, scale: float, stream=None,
                    window: int = 0) -> None:
    """C ``attn_fwd_varlen``: packed [total, H, d] q, k, v, o of one 16-bit type,
    lse fp32 [H, total], cu_seqlens int32 [B + 1] on the device."""
    (total, H, d), dt, sq = _packed3(q, "q")
    views = [_packed3(t, n) for n, t in (("k", k), ("v", v), ("o", o))]
    for n, (shape, dtn, _) in zip(("k", "v", "o"), views):
        if shape != (total, H, d) or dtn != dt:
            raise ValueError(f"{n} shape/dtype differs from q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, total) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [H, total]")
    B = _cu(cu_seqlens)
    dev = _device_of(q, k, v, o, lse, cu_seqlens)
    with torch.cuda.device(dev):
        _check(load().attn_fwd_varlen(dt, _ptr(q), sq, _ptr(k), views[0][2], _ptr(v), views[1][2], _ptr(o),
                                      views[2][2], _ptr(lse), _ptr(cu_seqlens), B, H, int(max_seqlen), total, d,
                                      int(bool(causal)), int(window), float(scale), _stream(stream, dev)))


def attn_bwd_varlen(q, k, v, o, dO, lse, dq, dk, dv, cu_seqlens, max_seqlen: int, causal: bool, scale: float,
                    workspace, stream=None, window: int = 0) -> None:
    """C ``attn_bwd_varlen`` on packed [total, H, d] tensors."""
    (total, H, d), dt, sq = _packed3(q, "q")
    names = ("k", "v", "o", "dO", "dq", "dk", "dv")
    views = [_packed3(t, n) for n, t in zip(names, (k, v, o, dO, dq, dk, dv))]
    for n, (shape, dtn, _) in zip(names, views):
        if shape != (total, H, d) or dtn != dt:
            raise ValueError(f"{n} shape/dtype differs from q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, total) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [H, total]")
    B = _cu(cu_seqlens)
    s = [vw[2] for vw in views]
    ws_bytes = workspace.numel() * workspace.element_size()
    dev = _device_of(q, k, v, o, dO, lse, dq, dk, dv, cu_seqlens, workspace)
    with torch.cuda.device(dev):
        _check(load().attn_bwd_varlen(dt, _ptr(q), sq, _ptr(k), s[0], _ptr(v), s[1], _ptr(o), s[2], _ptr(dO), s[3],
                                      _ptr(lse), _ptr(dq), s[4], _ptr(dk), s[5], _ptr(dv), s[6], _ptr(cu_seqlens), B, H,
                                      int(max_seqlen), total, d, int(bool(causal)), int(window), float(scale),
                                      _ptr(workspace), ws_bytes, _stream(stream, dev)))


def attn_fwd_decode_workspace_size(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(load().attn_fwd_decode_workspace_size(B, H, Nq, Nk, d))


def attn_fwd_decode(q, k, v, o, lse, causal: bool, scale: float, workspace=None, stream=None,
                    window: int = 0) -> None:
    """C ``attn_fwd_decode``: q, o [B, H, Nq, d] and k, v [B, H, Nk, d] views of
    one 16-bit type (d contiguous), lse fp32 [B, H, Nq]; queries aligned to
    the last Nq keys."""
    (B, H, Nq, d), dt, sq = _view4(q, "q")
    (Bk, Hk, Nk, dk_), dtk, sk = _view4(k, "k")
    (Bv, Hv, Nv, dv_), dtv, sv = _view4(v, "v")
    (Bo, Ho, No, do_), dto, so = _view4(o, "o")
    if (Bk, Hk, dk_) != (B, H, d) or (Bv, Hv, Nv, dv_) != (B, H, Nk, d) or (Bo, Ho, No, do_) != (B, H, Nq, d):
        raise ValueError("shapes must be q, o [B, H, Nq, d] and k, v [B, H, Nk, d]")
    if len({dt, dtk, dtv, dto}) != 1:
        raise ValueError("q, k, v, o must share one dtype")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, H, Nq]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dev = _device_of(q, k, v, o, lse, workspace)
    with torch.cuda.device(dev):
        _check(load().attn_fwd_decode(dt, _ptr(q), sq, _ptr(k), sk, _ptr(v), sv, _ptr(o), so, _ptr(lse), B, H, Nq, Nk,
                                      d, int(bool(causal)), int(window), float(scale), _ptr(workspace), ws_bytes,
                                      _stream(stream, dev)))


def attn_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """C ``attn_fwd`` on torch tensors: q, k, v, o bf16 [B, H, N, d]; lse fp32
    [B, H, N].  Asynchronous on ``stream`` (default: torch's current stream)."""
    B, H, N, d = _shape4(q, "q")
    for n, t in (("k", k), ("v", v), ("o", o)):
        if _shape4(t, n) != (B, H, N, d):
            raise ValueError(f"{n} shape {tuple(t.shape)} != q shape {(B, H, N, d)}")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, H, N]")
    dev = _device_of(q, k, v, o, lse)
    with torch.cuda.device(dev):
        _check(load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, int(bool(causal)),
                               float(scale), _stream(stream, dev)))


def attn_bwd_workspace_size(B: int, H: int, N: int, d: int, causal: bool) -> int:
    return int(load().attn_bwd_workspace_size(B, H, N, d, int(bool(causal))))


def attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, causal: bool, scale: float, workspace, stream=None) -> None:
    """C ``attn_bwd`` on torch tensors.  ``workspace`` is a CUDA tensor of at
    least ``attn_bwd_workspace_size`` bytes."""
    B, H, N, d = _shape4(q, "q")
    for n, t in (("k", k), ("v", v), ("o", o), ("dO", dO), ("dq", dq), ("dk", dk), ("dv", dv)):
        if _shape4(t, n) != (B, H, N, d):
            raise ValueError(f"{n} shape {tuple(t.shape)} != q shape {(B, H, N, d)}")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, H, N]")
    ws_bytes = workspace.numel() * workspace.element_size()
    dev = _device_of(q, k, v, o, dO, lse, dq, dk, dv, workspace)
    with torch.cuda.device(dev):
        _check(load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
                               _ptr(dv), B, H, N, d, int(bool(causal)), float(scale), _ptr(workspace), ws_bytes,
                               _stream(stream, dev)))


def _check_rows(t, shape, name):
    if t.dtype != torch.float32 or tuple(t.shape) != shape or not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous float32 {list(shape)}")


def attn_bwd_preprocess(o, dO, D, stream=None) -> None:
    """C ``attn_bwd_preprocess``: D (fp32 [B, H, N]) = rowsum(dO * O)."""
    B, H, N, d = _shape4(o, "o")
    if _shape4(dO, "dO") != (B, H, N, d):
        raise ValueError("dO shape != o shape")
    _check_rows(D, (B, H, N), "D")
    dev = _device_of(o, dO, D)
    with torch.cuda.device(dev):
        _check(load().attn_bwd_preprocess(_ptr(o), _ptr(dO), _ptr(D), B, H, N, d, _stream(stream, dev)))


def attn_bwd_dkdv(q, k, v, dO, lse, D, dk, dv, causal: bool, scale: float, stream=None) -> None:
    """C ``attn_bwd_dkdv``."""
    B, H, N, d = _shape4(q, "q")
    for n, t in (("k", k), ("v", v), ("dO", dO), ("dk", dk), ("dv", dv)):
        if _shape4(t, n) != (B, H, N, d):
            raise ValueError(f"{n} shape != q shape")
    _check_rows(lse, (B, H, N), "lse")
    _check_rows(D, (B, H, N), "D")
    dev = _device_of(q, k, v, dO, lse, D, dk, dv)
    with torch.cuda.device(dev):
        _check(load().attn_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(D), _ptr(dk), _ptr(dv),
                                    B, H, N, d, int(bool(causal)), float(scale), _stream(stream, dev)))


def attn_bwd_dq(q, k, v, dO, lse, D, dq, causal: bool, scale: float, stream=None) -> None:
    """C ``attn_bwd_dq``."""
    B, H, N, d = _shape4(q, "q")
    for n, t in (("k", k), ("v", v), ("dO", dO), ("dq", dq)):
        if _shape4(t, n) != (B, H, N, d):
            raise ValueError(f"{n} shape != q shape")
    _check_rows(lse, (B, H, N), "lse")
    _check_rows(D, (B, H, N), "D")
    dev = _device_of(q, k, v, dO, lse, D, dq)
    with torch.cuda.device(dev):
        _check(load().attn_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(D), _ptr(dq), B, H, N, d,
                                  int(bool(causal)), float(scale), _stream(stream, dev)))


def attn_bwd_d_and_dq(q, k, v, o, dO, lse, D, dq, causal: bool, scale: float, stream=None) -> None:
    """C ``attn_bwd_d_and_dq``: D (fp32 [B, H, N], written) and dQ in one kernel."""
    B, H, N, d = _shape4(q, "q")
    for n, t in (("k", k), ("v", v), ("o", o), ("dO", dO), ("dq", dq)):
        if _shape4(t, n) != (B, H, N, d):
            raise ValueError(f"{n} shape != q shape")
    _check_rows(lse, (B, H, N), "lse")
    _check_rows(D, (B, H, N), "D")
    dev = _device_of(q, k, v, o, dO, lse, D, dq)
    with torch.cuda.device(dev):
        _check(load().attn_bwd_d_and_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(D), _ptr(dq),
                                        B, H, N, d, int(bool(causal)), float(scale), _stream(stream, dev)))


def attn_fwd_bwd_host_workspace_size(B: int, H: int, N: int, d: int, causal: bool) -> int:
    """C ``attn_fwd_bwd_host_workspace_size`` (bytes; 0 for invalid sizes)."""
    return int(load().attn_fwd_bwd_host_workspace_size(int(B), int(H), int(N), int(d), int(bool(causal))))


def attn_fwd_bwd_host(q, k, v, dO, o, lse, dq, dk, dv, causal: bool, scale: float, workspace, groups: int = 4,
                      stream=None, copy_in_stream=None, copy_out_stream=None, stream2=None) -> None:
    """C ``attn_fwd_bwd_host``: q, k, v, dO and the outputs o, lse, dq, dk, dv
    are contiguous HOST tensors (pinned, for the copies to overlap the
    kernels); ``workspace`` is a device tensor of at least
    ``attn_fwd_bwd_host_workspace_size`` bytes.  Streams: torch streams, or
    None (``stream``: the current stream; the others: run on ``stream``)."""
    if q.dim() != 4:
        raise ValueError(f"q must be [B, H, N, d], got {tuple(q.shape)}")
    B, H, N, d = q.shape
    for n, t in (("q", q), ("k", k), ("v", v), ("dO", dO), ("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        if tuple(t.shape) != (B, H, N, d) or t.dtype != q.dtype or t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{n}: expected a contiguous host tensor like q")
    if tuple(lse.shape) != (B, H, N) or lse.dtype != torch.float32 or lse.device.type != "cpu" or \
            not lse.is_contiguous():
        raise ValueError("lse: expected a contiguous fp32 host tensor [B, H, N]")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q: bf16 or f16")
    dtype = EXATTN_DTYPE_F16 if q.dtype == torch.float16 else EXATTN_DTYPE_BF16
    ws_bytes = workspace.numel() * workspace.element_size()

    def side(s):
        return None if s is None else _stream(s, dev)

    dev = _device_of(workspace)
    with torch.cuda.device(dev):
        _check(load().attn_fwd_bwd_host(dtype, _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(o), _ptr(lse), _ptr(dq),
                                        _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), float(scale),
                                        _ptr(workspace), ws_bytes, int(groups), _stream(stream, dev),
                                        side(copy_in_stream), side(copy_out_stream), side(stream2)))


def device_error() -> int:
    """Synchronise and read/clear the kernels' watchdog word of the current
    device (0 = clean); a pending poll of that word (watchdog_poll) is
    dropped with it."""
    rc = int(load().exattn_device_error())
    w = _watch.get(torch.device("cuda", torch.cuda.current_device()))
    if w is not None:
        w.word[0] = 0
        w.event = None
    return rc


class _Watch:
    """Per device: a page-locked word that the last poll copies the
    watchdog word into, and an event recorded after that copy."""

    def __init__(self, dev):
        self.word = torch.zeros(1, dtype=torch.int32, pin_memory=True)
        self.event = None


_watch: dict = {}


def watchdog_check(device) -> None:
    """Raise ExattnError(EXATTN_ERR_TIMEOUT) if the last completed poll on
    ``device`` saw a bounded wait give up (then read and clear the word).
    Never waits: a poll still in flight is checked by a later call."""
    w = _watch.get(device)
    if w is None or w.event is None or not w.event.query():
        return
    if int(w.word[0]) != 0:
        w.word[0] = 0
        w.event = None
        with torch.cuda.device(device):
            device_error()  # synchronises, clears the word
        raise ExattnError(8, "a kernel's bounded internal wait gave up; outputs of the calls since the last "
                             "check are invalid")


def watchdog_poll(device, stream=None) -> None:
    """Queue a copy of the watchdog word into page-locked memory after the
    work on ``stream`` (default: the device's current stream); a later
    watchdog_check reads it once it has landed.  No synchronisation."""
    w = _watch.get(device)
    if w is None:
        w = _watch[device] = _Watch(device)
    with torch.cuda.device(device):
        if stream is None:
            st = torch.cuda.current_stream(device)
        elif isinstance(stream, int):
            st = torch.cuda.ExternalStream(stream, device=device)
        else:
            st = stream
        _check(load().exattn_device_error_poll(w.word.data_ptr(), st.cuda_stream))
        ev = torch.cuda.Event()
        ev.record(st)
        w.event = ev


def watchdog_selftest(timeout_us: int = 2000, stream=None) -> None:
    """C ``exattn_watchdog_selftest``: a deliberately unsatisfied bounded wait
    on the current device, followed by a watchdog poll (watchdog_poll)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    _check(load().exattn_watchdog_selftest(int(timeout_us), _stream(stream, dev)))
    watchdog_poll(dev, stream)


def version() -> int:
    return int(load().exattn_version())
