"""CPU oracle for the FP8 amax / scale / cast / scaled-GEMM path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (``bench.py``) may import this package.  The
product library (``scaling_quantization_gemm_gb300``) never imports it, and the
two share no code: the arithmetic here is plain C in ``fp8_oracle.c`` (compiled
with gcc, no fast-math, no FMA contraction) driven through ctypes.

What each function computes, and the passage it follows, is stated in
``fp8_oracle.c``.  In short:

* ``encode`` / ``decode`` -- the OFP8 E4M3 / E5M2 codec ("FP8_E4" for weights
  and activations, "FP8_E5" for gradients: "Training and inference of large
  language models using 8-bit floating point", "Proposed method"), RNE with
  saturation to the largest finite magnitude.
* ``compute_bias`` -- floor(log2(fmax / amax)) - margin (same section);
  ``compute_bias_ocp`` and ``scale_ratio`` are the two alternatives kept
  behind options (the OCP MX rule for 1x32 blocks, and s = fmax / amax).
* ``quantize_tensor`` / ``quantize_block`` -- Encode(x * 2^e), per tensor or per
  block ("Per-Tensor and Per-Block Scaling Strategies for Effective FP8
  Training", "Key Questions Answered"); ``quantize_f32`` / ``amax_f32`` -- the
  per-tensor cast and amax of an fp32 array.
* ``history_update`` -- delayed scaling from an amax window (same page).
* ``gemm_sample`` / ``gemm_full`` -- fp64 product of the dequantised operands.
* ``gemm_quantize_bracket`` -- the FP8 codes a GEMM whose output is cast for the
  next layer may write (the cast of "Proposed method" applied to D).
* ``cast_stats`` -- how many elements a given (e.g. fixed, FP8-CSCALE) scale
  saturates and flushes to zero.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against closed forms, exhaustive tables, brute force
in exact rational arithmetic and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

E4M3, E5M2 = 0, 1
TENSOR, BLOCK_1x128, BLOCK_128x128, MX_1x32, MX_1x32_OCP = 0, 1, 2, 3, 4
FMAX = {E4M3: 448.0, E5M2: 57344.0}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``fp8_oracle.c`` into ``liboracle.so`` (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
            L.fp8o_decode.restype = ctypes.c_double
            L.fp8o_decode.argtypes = [i32, i32]
            L.fp8o_encode.restype = i32
            L.fp8o_encode.argtypes = [f32, i32]
            L.fp8o_encode_array.argtypes = [vp, i64, i32, vp]
            L.fp8o_decode_array.argtypes = [vp, i64, i32, vp]
            L.fp8o_compute_bias.restype = i32
            L.fp8o_compute_bias.argtypes = [f32, i32, i32, ctypes.POINTER(ctypes.c_int)]
            L.fp8o_compute_bias_ocp.restype = i32
            L.fp8o_compute_bias_ocp.argtypes = [f32, i32, i32, ctypes.POINTER(ctypes.c_int)]
            L.fp8o_compute_scale_ratio.restype = i32
            L.fp8o_compute_scale_ratio.argtypes = [f32, i32, vp, vp]
            L.fp8o_amax.restype = f32
            L.fp8o_amax.argtypes = [vp, i64, i64, i64]
            L.fp8o_quantize_tensor.argtypes = [vp, i64, i64, i64, i32, f32, vp, vp]
            L.fp8o_quantize_f32.argtypes = [vp, i64, i32, f32, vp]
            L.fp8o_amax_f32.restype = f32
            L.fp8o_amax_f32.argtypes = [vp, i64]
            L.fp8o_quantize_block.restype = i32
            L.fp8o_quantize_block.argtypes = [vp, i64, i64, i64, i32, i32, i32, vp, vp, vp, vp]
            L.fp8o_history_update.restype = i32
            L.fp8o_history_update.argtypes = [vp, ctypes.c_int32, vp, vp, i32, i32, vp, vp, vp]
            L.fp8o_cast_stats.argtypes = [vp, i64, i64, i64, i32, vp, i32, vp, vp]
            L.fp8o_gemm_sample.argtypes = [i64, i64, i64, vp, i64, i32, i32, vp, vp, i64, i32, i32, vp,
                                           i64, vp, vp, vp, vp]
            L.fp8o_gemm_full.argtypes = [i64, i64, i64, vp, i64, i32, i32, vp, vp, i64, i32, i32, vp, vp, vp]
            L.fp8o_max_threads.restype = i32
            L.fp8o_set_threads.argtypes = [i32]
            L.fp8o_maxcode.restype = i32
            L.fp8o_maxcode.argtypes = [i32]
            _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def set_threads(n: int) -> None:
    lib().fp8o_set_threads(int(n))


def max_threads() -> int:
    return int(lib().fp8o_max_threads())


# ----------------------------------------------------------------- codec

def decode(code: int, fmt: int) -> float:
    return float(lib().fp8o_decode(int(code), int(fmt)))


def encode(v: float, fmt: int) -> int:
    return int(lib().fp8o_encode(float(np.float32(v)), int(fmt)))


def encode_array(v: np.ndarray, fmt: int) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().fp8o_encode_array(_p(v), v.size, fmt, _p(out))
    return out


def decode_array(c: np.ndarray, fmt: int) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().fp8o_decode_array(_p(c), c.size, fmt, _p(out))
    return out


def maxcode(fmt: int) -> int:
    return int(lib().fp8o_maxcode(fmt))


# -------------------------------------------------------------- scaling

def compute_bias(amax: float, fmt: int, margin: int = 0) -> tuple[int, bool]:
    """Return (e, nonfinite_flag)."""
    nf = ctypes.c_int(0)
    e = lib().fp8o_compute_bias(float(np.float32(amax)), fmt, int(margin), ctypes.byref(nf))
    return int(e), bool(nf.value)


def pow2f(e: int) -> np.float32:
    return np.float32(np.ldexp(np.float32(1.0), int(e)))


def compute_bias_ocp(amax: float, fmt: int, margin: int = 0) -> tuple[int, bool]:
    """The OCP MX alternative: e = emax - floor(log2 amax) - margin (emax 8 for E4M3, 15 for E5M2)."""
    nf = ctypes.c_int(0)
    e = lib().fp8o_compute_bias_ocp(float(np.float32(amax)), fmt, int(margin), ctypes.byref(nf))
    return int(e), bool(nf.value)


def scale_ratio(amax: float, fmt: int) -> tuple[np.float32, np.float32, bool]:
    """The non-power-of-two alternative: (s = fmax / amax, 1 / s, nonfinite), fp32 divisions."""
    s = np.zeros(1, np.float32)
    si = np.zeros(1, np.float32)
    nf = lib().fp8o_compute_scale_ratio(float(np.float32(amax)), fmt, _p(s), _p(si))
    return s[0], si[0], bool(nf)


def scale_triple(amax: float, fmt: int, margin: int = 0) -> tuple[int, np.float32, np.float32]:
    e, _ = compute_bias(amax, fmt, margin)
    return e, pow2f(e), pow2f(-e)


def amax(x_bf16: np.ndarray) -> np.float32:
    """max |x| over a 2-D bf16 array given as uint16/int16 bits."""
    x = np.ascontiguousarray(x_bf16).view(np.uint16)
    r, c = x.shape
    return np.float32(lib().fp8o_amax(_p(x), r, c, c))


# ------------------------------------------------------------- quantise

def quantize_f32(x: np.ndarray, fmt: int, scale: float = 1.0) -> np.ndarray:
    """Per-tensor cast of an fp32 array: Encode(fl32(x * scale)), same shape, uint8 codes."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    lib().fp8o_quantize_f32(_p(x), x.size, fmt, float(np.float32(scale)), _p(q))
    return q


def amax_f32(x: np.ndarray) -> np.float32:
    """max |x| of an fp32 array (NaN if any element is NaN)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return np.float32(lib().fp8o_amax_f32(_p(x), x.size))


def quantize_tensor(x_bf16: np.ndarray, fmt: int, scale: float, row: bool = True, col: bool = False):
    """Per-tensor cast with scale s: returns (q_row or None, q_col or None)."""
    x = np.ascontiguousarray(x_bf16).view(np.uint16)
    r, c = x.shape
    qr = np.empty((r, c), np.uint8) if row else None
    qc = np.empty((c, r), np.uint8) if col else None
    lib().fp8o_quantize_tensor(_p(x), r, c, c, fmt, float(np.float32(scale)),
                               _p(qr) if row else None, _p(qc) if col else None)
    return qr, qc


def block_shape(gran: int) -> tuple[int, int]:
    return {BLOCK_1x128: (1, 128), BLOCK_128x128: (128, 128), MX_1x32: (1, 32), MX_1x32_OCP: (1, 32)}[gran]


def scale_shapes(rows: int, cols: int, gran: int) -> tuple[tuple[int, int], tuple[int, int]]:
    """Shapes of the row-wise and column-wise scale tensors of a block granularity."""
    br, bc = block_shape(gran)
    cdiv = lambda a, b: (a + b - 1) // b
    return (cdiv(rows, br), cdiv(cols, bc)), (cdiv(cols, br), cdiv(rows, bc))


def quantize_block(x_bf16: np.ndarray, fmt: int, gran: int, margin: int = 0, row: bool = True,
                   col: bool = False):
    """Block-scaled cast.  Returns (q_row, sf_row, q_col, sf_col, nonfinite); absent parts are None."""
    x = np.ascontiguousarray(x_bf16).view(np.uint16)
    r, c = x.shape
    srow, scol = scale_shapes(r, c, gran)
    sdt = np.uint8 if gran in (MX_1x32, MX_1x32_OCP) else np.float32
    qr = np.empty((r, c), np.uint8) if row else None
    sr = np.empty(srow, sdt) if row else None
    qc = np.empty((c, r), np.uint8) if col else None
    sc = np.empty(scol, sdt) if col else None
    nf = lib().fp8o_quantize_block(_p(x), r, c, c, fmt, gran, int(margin),
                                   _p(qr) if row else None, _p(sr) if row else None,
                                   _p(qc) if col else None, _p(sc) if col else None)
    return qr, sr, qc, sc, bool(nf)


# ----------------------------------------------------- delayed scaling

class HistoryState:
    """Delayed-scaling state: amax ring (float[L]), position, bias, scale, scale_inv."""

    def __init__(self, L: int):
        self.hist = np.zeros(L, np.float32)
        self.pos = np.zeros(1, np.int64)
        self.bias = np.zeros(1, np.int32)
        self.scale = np.ones(1, np.float32)
        self.scale_inv = np.ones(1, np.float32)

    def update(self, amax_value: float, fmt: int, margin: int) -> bool:
        a = np.array([amax_value], np.float32)
        nf = lib().fp8o_history_update(_p(self.hist), self.hist.size, _p(self.pos), _p(a), fmt, int(margin),
                                       _p(self.bias), _p(self.scale), _p(self.scale_inv))
        assert a[0] == 0.0
        return bool(nf)


# ----------------------------------------------------------------- GEMM

def _sf_arg(gran: int, sf) -> np.ndarray:
    if gran == TENSOR:
        return np.array([sf], np.float32).reshape(1) if np.isscalar(sf) else np.ascontiguousarray(sf, np.float32)
    if gran in (MX_1x32, MX_1x32_OCP):
        return np.ascontiguousarray(sf, np.uint8)
    return np.ascontiguousarray(sf, np.float32)


def gemm_sample(A: np.ndarray, fa: int, ga: int, sfa, B: np.ndarray, fb: int, gb: int, sfb,
                ms: np.ndarray, ns: np.ndarray):
    """fp64 y[m_i, n_i] and sum_k |a b| for sampled output coordinates."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    sfa_a, sfb_a = _sf_arg(ga, sfa), _sf_arg(gb, sfb)
    ms = np.ascontiguousarray(ms, np.int64)
    ns = np.ascontiguousarray(ns, np.int64)
    out = np.empty(ms.size, np.float64)
    mag = np.empty(ms.size, np.float64)
    lib().fp8o_gemm_sample(M, N, K, _p(A), K, fa, ga, _p(sfa_a), _p(B), K, fb, gb, _p(sfb_a), ms.size,
                           _p(ms), _p(ns), _p(out), _p(mag))
    return out, mag


def gemm_full(A: np.ndarray, fa: int, ga: int, sfa, B: np.ndarray, fb: int, gb: int, sfb):
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    sfa_a, sfb_a = _sf_arg(ga, sfa), _sf_arg(gb, sfb)
    out = np.empty((M, N), np.float64)
    mag = np.empty((M, N), np.float64)
    lib().fp8o_gemm_full(M, N, K, _p(A), K, fa, ga, _p(sfa_a), _p(B), K, fb, gb, _p(sfb_a), _p(out), _p(mag))
    return out, mag


def gemm_tolerance(y_ref: np.ndarray, mag: np.ndarray, out_bf16: bool) -> np.ndarray:
    """Allowed |y - y_ref|: 1e-3 * sum_k |a_k b_k| (the stated GEMM tolerance), plus, for a
    bf16 output, half a bf16 ulp of y_ref (the output rounding alone)."""
    tol = 1e-3 * mag
    if out_bf16:
        a = np.abs(y_ref)
        _, x = np.frexp(a)  # a = f 2^x, f in [0.5, 1): floor(log2 a) = x - 1
        ulp = np.where(a > 0, np.ldexp(1.0, (x - 1 - 7).astype(np.int64)), 0.0)
        tol = tol + 0.5 * ulp
    return tol


def round_bf16(v: np.ndarray) -> np.ndarray:
    """fp32 values rounded to the nearest bf16 (ties to even), returned as fp32; NaN stays NaN."""
    u = np.ascontiguousarray(v, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    return np.where(np.isnan(v), np.float32(np.nan), out)


def gemm_quantize_bracket(y_ref: np.ndarray, tol: np.ndarray, fmt: int, scale_d: float, via_bf16: bool = False):
    """Codes a GEMM with an FP8 output may write: Encode(fl32(v * scale_d)) for some fp32 v with
    |v - y_ref| <= tol (with via_bf16, v is first rounded to bf16: a bf16 output cast afterwards).
    Encode, the fp32 product and the bf16 rounding are monotone in v, so the admissible codes are
    exactly those between the codes of the two ends of the interval (the ends rounded outward to
    fp32 never narrow it).  Returns (lo, hi, nearest): code arrays for y_ref - tol, y_ref + tol
    and y_ref itself."""
    s = np.float32(scale_d)
    y_ref = np.asarray(y_ref, np.float64)
    tol = np.asarray(tol, np.float64)

    def codes(v):
        v32 = np.asarray(v, np.float64).astype(np.float32)
        if via_bf16:
            v32 = round_bf16(v32)
        return encode_array(v32 * s, fmt)

    return codes(y_ref - tol), codes(y_ref + tol), codes(y_ref)


def cast_stats(x_bf16: np.ndarray, fmt: int, scales) -> tuple[np.ndarray, np.ndarray]:
    """(saturated[j], underflow[j]) for each scale s_j: elements with |fl32(x s_j)| > fmax, and
    non-zero elements whose cast is +-0 (NaN elements count in neither)."""
    x = np.ascontiguousarray(x_bf16).view(np.uint16)
    sc = np.ascontiguousarray(scales, np.float32).reshape(-1)
    sat = np.zeros(sc.size, np.uint64)
    und = np.zeros(sc.size, np.uint64)
    lib().fp8o_cast_stats(_p(x), x.shape[0], x.shape[1], x.shape[1], fmt, _p(sc), sc.size, _p(sat), _p(und))
    return sat, und

