"""GB300-native FP8 amax / scale selection / scaled cast / scaled GEMM.

A thin ctypes binding over ``libfp8q.so`` (``include/fp8q.h``).  Every function
has the name of the C entry point it calls and only marshals arguments: it
reads shapes, strides and data pointers from torch tensors (or takes raw device
pointers as ints), passes the caller's current CUDA stream, and raises
``FP8Error`` on a non-OK status.  All computation runs in the library's CUDA
kernels; there is no other code path.  If the library is not built, importing
works but every call raises.

Build it with ``python -m scaling_quantization_gemm_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Union

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8q.so")

# enums of include/fp8q.h
FP8_OK, FP8_ERR_INVALID_ARG, FP8_ERR_UNSUPPORTED, FP8_ERR_CUDA, FP8_ERR_TIMEOUT = 0, 1, 2, 3, 4
E4M3, E5M2 = 0, 1
TENSOR, BLOCK_1x128, BLOCK_128x128, MX_1x32, MX_1x32_OCP = 0, 1, 2, 3, 4
FPROP, DGRAD, WGRAD = 0, 1, 2
OUT_F32, OUT_BF16 = 0, 1
STATUS_NONFINITE_AMAX, STATUS_TIMEOUT, STATUS_BAD_BLOCK_SCALE = 1, 2, 4

# every entry point declared in include/fp8q.h
ENTRY_POINTS = ("fp8_amax", "fp8_compute_scale", "fp8_compute_scale_ratio", "fp8_amax_history_update",
                "fp8_amax_history_update_batch",
                "fp8_set_bias", "fp8_cast_stats", "fp8_quantize", "fp8_quantize_batch", "fp8_quantize_f32",
                "fp8_quantize_current",
                "fp8_quantize_current_noalloc",
                "fp8_scaled_gemm", "fp8_scaled_gemm_quantize", "fp8_status_string", "fp8_last_error_detail")
QUANTIZE_CURRENT_WORKSPACE_BYTES = 4096  # FP8_QUANTIZE_CURRENT_WORKSPACE_BYTES


class FP8Error(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn}: {status_name(status)}: {detail}")
        self.status = status
        self.detail = detail


_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded libfp8q.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built; run `python -m scaling_quantization_gemm_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            for name, args in {
                "fp8_amax": [vp, i64, i64, i64, vp, vp],
                "fp8_compute_scale": [vp, i32, i32, vp, vp, vp, vp, vp],
                "fp8_compute_scale_ratio": [vp, i32, vp, vp, vp, vp],
                "fp8_amax_history_update": [vp, i32, vp, vp, i32, i32, vp, vp, vp, vp, vp],
                "fp8_amax_history_update_batch": [vp, i32, vp],
                "fp8_quantize": [vp, i64, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp],
                "fp8_quantize_batch": [vp, i32, vp],
                "fp8_quantize_f32": [vp, i64, i32, vp, vp, vp, vp],
                "fp8_set_bias": [i32, vp, vp, vp, vp],
                "fp8_cast_stats": [vp, i64, i64, i64, i32, vp, i32, vp, vp, vp],
                "fp8_quantize_current": [vp, i64, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp],
                "fp8_quantize_current_noalloc": [vp, i64, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp],
                "fp8_scaled_gemm": [i32, i64, i64, i64, vp, i64, i32, i32, vp, vp, i64, i32, i32, vp, vp, i32, i64,
                                    vp, vp],
                "fp8_scaled_gemm_quantize": [i32, i64, i64, i64, vp, i64, i32, vp, vp, i64, i32, vp, vp, i64, i32, vp,
                                             vp, vp, vp],
            }.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = ctypes.c_int
            L.fp8_status_string.argtypes = [ctypes.c_int]
            L.fp8_status_string.restype = ctypes.c_char_p
            L.fp8_last_error_detail.argtypes = []
            L.fp8_last_error_detail.restype = ctypes.c_char_p
            _lib = L
    return _lib


def status_name(s: int) -> str:
    return lib().fp8_status_string(int(s)).decode()


Ptr = Union[None, int, torch.Tensor]


def _p(t: Ptr) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr() if t.numel() > 0 else None
    return int(t)


def _stream(stream) -> Optional[int]:
    if stream is None:
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream or None
        return None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, st: int) -> None:
    if st != FP8_OK:
        raise FP8Error(fn, st, lib().fp8_last_error_detail().decode())


def _matrix(x: torch.Tensor):
    if x.dim() != 2 or (x.size(1) > 1 and x.stride(1) != 1):
        raise ValueError("expected a 2-D row-major tensor (unit column stride)")
    return x.size(0), x.size(1), x.stride(0) if x.size(0) > 1 else max(x.size(1), 1)


def fp8_amax(x: torch.Tensor, amax: Ptr, stream=None) -> None:
    """amax <- max(amax, max|x|) for a bf16 [rows x cols] tensor (see fp8_amax in fp8q.h)."""
    rows, cols, ld = _matrix(x)
    _check("fp8_amax", lib().fp8_amax(_p(x), rows, cols, ld, _p(amax), _stream(stream)))


def fp8_compute_scale(amax: Ptr, fmt: int, margin: int, bias: Ptr = None, scale: Ptr = None,
                      scale_inv: Ptr = None, status: Ptr = None, stream=None) -> None:
    _check("fp8_compute_scale", lib().fp8_compute_scale(_p(amax), fmt, margin, _p(bias), _p(scale), _p(scale_inv),
                                                        _p(status), _stream(stream)))


def fp8_compute_scale_ratio(amax: Ptr, fmt: int, scale: Ptr = None, scale_inv: Ptr = None, status: Ptr = None,
                            stream=None) -> None:
    """The non-power-of-two alternative: scale = fmax / amax, scale_inv = 1 / scale (fp32, nearest)."""
    _check("fp8_compute_scale_ratio", lib().fp8_compute_scale_ratio(_p(amax), fmt, _p(scale), _p(scale_inv),
                                                                    _p(status), _stream(stream)))


def fp8_amax_history_update(history: torch.Tensor, pos: Ptr, amax: Ptr, fmt: int, margin: int, bias: Ptr,
                            scale: Ptr, scale_inv: Ptr, status: Ptr = None, stream=None) -> None:
    _check("fp8_amax_history_update",
           lib().fp8_amax_history_update(_p(history), history.numel(), _p(pos), _p(amax), fmt, margin, _p(bias),
                                         _p(scale), _p(scale_inv), _p(status), _stream(stream)))


class HistoryStateRecord(ctypes.Structure):
    """One record of fp8_amax_history_update_batch (fp8_history_state in fp8q.h)."""
    _fields_ = [("history", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("amax", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("scale_inv", ctypes.c_void_p),
                ("status", ctypes.c_void_p), ("len", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("margin", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def fp8_amax_history_update_batch(states, stream=None) -> None:
    """fp8_amax_history_update for every state in `states` in one launch per 48.  Each state is an object
    with tensors history, pos, amax, bias, scale, scale_inv (and optionally status) and ints fmt, margin."""
    states = list(states)
    recs = (HistoryStateRecord * max(len(states), 1))()
    for r, st in zip(recs, states):
        r.history, r.pos, r.amax = _p(st.history), _p(st.pos), _p(st.amax)
        r.bias, r.scale, r.scale_inv = _p(st.bias), _p(st.scale), _p(st.scale_inv)
        r.status = _p(getattr(st, "status", None))
        r.len, r.fmt, r.margin, r.reserved = st.history.numel(), int(st.fmt), int(st.margin), 0
    _check("fp8_amax_history_update_batch",
           lib().fp8_amax_history_update_batch(ctypes.cast(recs, ctypes.c_void_p), len(states), _stream(stream)))


def fp8_set_bias(e: int, bias: Ptr = None, scale: Ptr = None, scale_inv: Ptr = None, stream=None) -> None:
    """A fixed (FP8-CSCALE) bias: bias = e, scale = 2^e, scale_inv = 2^-e on the device."""
    _check("fp8_set_bias", lib().fp8_set_bias(int(e), _p(bias), _p(scale), _p(scale_inv), _stream(stream)))


def fp8_cast_stats(x: torch.Tensor, fmt: int, scales: torch.Tensor, saturated: torch.Tensor, underflow: torch.Tensor,
                   stream=None) -> None:
    """Accumulate, per scale, the elements the cast would saturate and flush to zero (int64 counters)."""
    rows, cols, ld = _matrix(x)
    _check("fp8_cast_stats", lib().fp8_cast_stats(_p(x), rows, cols, ld, fmt, _p(scales), scales.numel(),
                                                  _p(saturated), _p(underflow), _stream(stream)))


def fp8_quantize(x: torch.Tensor, fmt: int, gran: int, margin: int = 0, scale: Ptr = None, q_row: Ptr = None,
                 q_col: Ptr = None, sf_row: Ptr = None, sf_col: Ptr = None, amax: Ptr = None, stream=None) -> None:
    rows, cols, ld = _matrix(x)
    _check("fp8_quantize", lib().fp8_quantize(_p(x), rows, cols, ld, fmt, gran, margin, _p(scale), _p(q_row),
                                              _p(q_col), _p(sf_row), _p(sf_col), _p(amax), _stream(stream)))


class QuantizeDesc(ctypes.Structure):
    """One cast of fp8_quantize_batch (fp8_quantize_desc in fp8q.h)."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("ld", ctypes.c_int64),
                ("fmt", ctypes.c_int32), ("gran", ctypes.c_int32), ("margin", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("scale", ctypes.c_void_p), ("q_row", ctypes.c_void_p),
                ("q_col", ctypes.c_void_p), ("sf_row", ctypes.c_void_p), ("sf_col", ctypes.c_void_p),
                ("amax", ctypes.c_void_p)]


QUANTIZE_BATCH_MAX = 4  # FP8_QUANTIZE_BATCH_MAX


def fp8_quantize_batch(casts, stream=None) -> None:
    """Up to QUANTIZE_BATCH_MAX fp8_quantize casts in one launch.  Each cast is a dict with the keyword
    arguments of fp8_quantize: x, fmt, gran and optionally margin, scale, q_row, q_col, sf_row, sf_col,
    amax (see fp8_quantize_batch in fp8q.h)."""
    casts = list(casts)
    descs = (QuantizeDesc * max(len(casts), 1))()
    for d, c in zip(descs, casts):
        d.rows, d.cols, d.ld = _matrix(c["x"])
        d.x = _p(c["x"])
        d.fmt, d.gran, d.margin, d.reserved = int(c["fmt"]), int(c["gran"]), int(c.get("margin", 0)), 0
        d.scale, d.amax = _p(c.get("scale")), _p(c.get("amax"))
        d.q_row, d.q_col = _p(c.get("q_row")), _p(c.get("q_col"))
        d.sf_row, d.sf_col = _p(c.get("sf_row")), _p(c.get("sf_col"))
    _check("fp8_quantize_batch", lib().fp8_quantize_batch(ctypes.cast(descs, ctypes.c_void_p), len(casts),
                                                          _stream(stream)))


def fp8_quantize_f32(x: torch.Tensor, fmt: int, q: torch.Tensor, scale: Ptr = None, amax: Ptr = None,
                     stream=None) -> None:
    """q = RNE_sat(fl32(x * scale)) for a dense fp32 tensor x (any shape) into u8 q of the same size."""
    if x.dtype != torch.float32 or not x.is_contiguous() or q.dtype != torch.uint8 or q.numel() != x.numel():
        raise ValueError("expected a dense float32 x and a uint8 q with as many elements")
    _check("fp8_quantize_f32", lib().fp8_quantize_f32(_p(x), x.numel(), fmt, _p(scale), _p(q), _p(amax),
                                                      _stream(stream)))


def current_workspace(device=None) -> torch.Tensor:
    """A zeroed workspace for fp8_quantize_current (one per stream that calls it)."""
    return torch.zeros(QUANTIZE_CURRENT_WORKSPACE_BYTES, dtype=torch.uint8, device=device or "cuda")


def fp8_quantize_current(x: torch.Tensor, fmt: int, margin: int, workspace: Ptr, q_row: Ptr = None,
                         q_col: Ptr = None, amax: Ptr = None, bias: Ptr = None, scale: Ptr = None,
                         scale_inv: Ptr = None, status: Ptr = None, stream=None) -> None:
    """amax, compute_bias and the per-tensor cast in one launch (see fp8_quantize_current in fp8q.h)."""
    rows, cols, ld = _matrix(x)
    _check("fp8_quantize_current",
           lib().fp8_quantize_current(_p(x), rows, cols, ld, fmt, margin, _p(q_row), _p(q_col), _p(amax), _p(bias),
                                      _p(scale), _p(scale_inv), _p(workspace), _p(status), _stream(stream)))


def fp8_quantize_current_noalloc(x: torch.Tensor, fmt: int, margin: int, q_row: Ptr = None, q_col: Ptr = None,
                                 amax: Ptr = None, bias: Ptr = None, scale: Ptr = None, scale_inv: Ptr = None,
                                 status: Ptr = None, stream=None) -> None:
    """fp8_quantize_current with the library's static scratch instead of a workspace (allocates nothing)."""
    rows, cols, ld = _matrix(x)
    _check("fp8_quantize_current_noalloc",
           lib().fp8_quantize_current_noalloc(_p(x), rows, cols, ld, fmt, margin, _p(q_row), _p(q_col), _p(amax),
                                              _p(bias), _p(scale), _p(scale_inv), _p(status), _stream(stream)))


def fp8_scaled_gemm(op: int, A: torch.Tensor, fa: int, ga: int, sfa: Ptr, B: torch.Tensor, fb: int, gb: int,
                    sfb: Ptr, D: torch.Tensor, status: Ptr = None, stream=None) -> None:
    """D[M x N] = unscale(A[M x K] . B[N x K]^T); out dtype from D (float32 or bfloat16)."""
    M, K, lda = _matrix(A)
    N, K2, ldb = _matrix(B)
    if K != K2:
        raise ValueError("A and B disagree on K")
    Dm, Dn, ldd = _matrix(D)
    if (Dm, Dn) != (M, N):
        raise ValueError("D must be [M x N]")
    out = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}[D.dtype]
    _check("fp8_scaled_gemm", lib().fp8_scaled_gemm(op, M, N, K, _p(A), lda, fa, ga, _p(sfa), _p(B), ldb, fb, gb,
                                                    _p(sfb), _p(D), out, ldd, _p(status), _stream(stream)))


def fp8_scaled_gemm_quantize(op: int, A: torch.Tensor, fa: int, sfa: Ptr, B: torch.Tensor, fb: int, sfb: Ptr,
                             Dq: torch.Tensor, fd: int, scale_d: Ptr, amax_d: Ptr = None, status: Ptr = None,
                             stream=None) -> None:
    """Dq[M x N] (u8) = RNE_sat(unscale(A . B^T) * scale_d); max |unscale(A . B^T)| folded into amax_d."""
    M, K, lda = _matrix(A)
    N, K2, ldb = _matrix(B)
    if K != K2:
        raise ValueError("A and B disagree on K")
    Dm, Dn, ldd = _matrix(Dq)
    if (Dm, Dn) != (M, N) or Dq.dtype != torch.uint8:
        raise ValueError("Dq must be uint8 [M x N]")
    _check("fp8_scaled_gemm_quantize",
           lib().fp8_scaled_gemm_quantize(op, M, N, K, _p(A), lda, fa, _p(sfa), _p(B), ldb, fb, _p(sfb), _p(Dq), ldd,
                                          fd, _p(scale_d), _p(amax_d), _p(status), _stream(stream)))


__all__ = ["lib", "FP8Error", "status_name", "fp8_amax", "fp8_compute_scale", "fp8_compute_scale_ratio",
           "fp8_amax_history_update", "fp8_amax_history_update_batch", "HistoryStateRecord",
           "fp8_set_bias", "fp8_cast_stats",
           "fp8_quantize", "fp8_quantize_f32", "fp8_quantize_current", "fp8_quantize_current_noalloc",
           "current_workspace", "fp8_scaled_gemm", "fp8_scaled_gemm_quantize", "ENTRY_POINTS",
           "QUANTIZE_CURRENT_WORKSPACE_BYTES", "LIB_PATH", "E4M3", "E5M2", "TENSOR", "BLOCK_1x128",
           "BLOCK_128x128", "MX_1x32", "MX_1x32_OCP", "FPROP", "DGRAD", "WGRAD", "OUT_F32", "OUT_BF16"]
