"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and rounds them to bf16; it holds none
of the FP8 method's arithmetic.  Both the CPU oracle and the CUDA path take the
arrays it returns as their inputs.

Recipe (all draws from numpy's PCG64 ``default_rng(seed)``; fp64 -> fp32 by
round-to-nearest -> bf16 by round-to-nearest-even on the bit pattern):

* linear forward, per-tensor current scaling (256x1024 activations, 1024x1024
  weights): X ~ N(0, 0.02^2) from seed 0; then 8 distinct positions of X drawn
  without replacement from the same stream are set to +-30 (sign drawn next);
  W ~ N(0, 0.02^2) drawn next from the same stream.
* delayed scaling, 4096x4096: activation at iteration t ~ N(0,1) * (1 + 0.1 t)
  from seed t; gradient at iteration t ~ Laplace(0, 1e-4) from seed 100 + t.
* per-block, Llama-2-7B MLP up-projection: X 8192x4096 ~ 0.5 * Student-t(3)
  (seed 0); W 11008x4096 ~ N(0, 0.02^2) (seed 1).
* MXFP8: X 16384x8192 ~ N(0,1) (seed 0), then a Bernoulli(0.001) mask from the
  same stream multiplies the selected entries by 100; W 28672x8192 ~
  N(0, 0.01^2) (seed 1).
* 13B-class FFN forward + backward: X 16384x5120 ~ N(0,1) (seed 0), W
  20480x5120 ~ N(0, 0.02^2) (seed 1), dY 16384x20480 ~ Laplace(0, 1e-5) (seed 2).

Large arrays are drawn in row chunks; numpy's generators give the same stream
whether a sample is drawn at once or in consecutive pieces (checked by a test).
Arrays are returned as ``uint16`` bf16 bit patterns.
"""
from __future__ import annotations

import numpy as np

CHUNK_ELEMS = 1 << 24


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp64/fp32 array -> bf16 bit patterns (uint16): fp32 round-to-nearest first,
    then round-to-nearest-even to the top 16 bits.  Inputs here are finite."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b).view(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _chunked(rows: int, cols: int, draw) -> np.ndarray:
    out = np.empty((rows, cols), np.uint16)
    step = max(1, CHUNK_ELEMS // cols)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = bf16_bits(draw((r1 - r0, cols)))
    return out


def normal(rng: np.random.Generator, rows: int, cols: int, std: float = 1.0) -> np.ndarray:
    return _chunked(rows, cols, lambda shp: rng.standard_normal(shp) * std)


def laplace(rng: np.random.Generator, rows: int, cols: int, b: float) -> np.ndarray:
    return _chunked(rows, cols, lambda shp: rng.laplace(0.0, b, shp))


def student_t(rng: np.random.Generator, rows: int, cols: int, dof: float, mult: float) -> np.ndarray:
    return _chunked(rows, cols, lambda shp: rng.standard_t(dof, shp) * mult)


# ------------------------------------------------------------------ configs

def linear_fwd_current(seed: int = 0, m: int = 256, k: int = 1024, n: int = 1024, outliers: int = 8,
                       outlier_value: float = 30.0):
    """X [m x k] and W [n x k] for the per-tensor current-scaling linear forward."""
    rng = np.random.default_rng(seed)
    xf = rng.standard_normal((m, k)) * 0.02
    pos = rng.choice(m * k, size=outliers, replace=False)
    sgn = np.where(rng.random(outliers) < 0.5, -1.0, 1.0)
    xf.reshape(-1)[pos] = sgn * outlier_value
    wf = rng.standard_normal((n, k)) * 0.02
    return bf16_bits(xf), bf16_bits(wf)


def delayed_activation(t: int, rows: int = 4096, cols: int = 4096) -> np.ndarray:
    rng = np.random.default_rng(t)
    return normal(rng, rows, cols, 1.0 + 0.1 * t)


def delayed_gradient(t: int, rows: int = 4096, cols: int = 4096, b: float = 1e-4) -> np.ndarray:
    rng = np.random.default_rng(100 + t)
    return laplace(rng, rows, cols, b)


def per_block_up_proj(m: int = 8192, k: int = 4096, n: int = 11008):
    X = student_t(np.random.default_rng(0), m, k, 3.0, 0.5)
    W = normal(np.random.default_rng(1), n, k, 0.02)
    return X, W


def mxfp8_inputs(m: int = 16384, k: int = 8192, n: int = 28672, p: float = 0.001, mult: float = 100.0):
    rng = np.random.default_rng(0)
    step = max(1, CHUNK_ELEMS // k)
    xs = []
    for r0 in range(0, m, step):
        xs.append(rng.standard_normal((min(m, r0 + step) - r0, k)))
    X = np.empty((m, k), np.uint16)
    r0 = 0
    for blk in xs:
        mask = rng.random(blk.shape) < p
        blk = np.where(mask, blk * mult, blk)
        X[r0:r0 + blk.shape[0]] = bf16_bits(blk)
        r0 += blk.shape[0]
    W = normal(np.random.default_rng(1), n, k, 0.01)
    return X, W


def ffn_fwd_bwd(m: int = 16384, k: int = 5120, n: int = 20480):
    """X [m x k], W [n x k], dY [m x n] for the FFN layer forward + backward."""
    X = normal(np.random.default_rng(0), m, k, 1.0)
    W = normal(np.random.default_rng(1), n, k, 0.02)
    dY = laplace(np.random.default_rng(2), m, n, 1e-5)
    return X, W, dY


# ---------------------------------------------------------- test helpers

def ptq_ffn(t: int = 8192, h: int = 5120, f: int = 13824, seed: int = 0):
    """Inference through a 13B-class FFN (hidden 5120, intermediate 13824): X [t x h] N(0,1),
    W1 [f x h] and W2 [h x f] N(0, 0.02^2); seeds seed, seed+1, seed+2."""
    X = normal(np.random.default_rng(seed), t, h, 1.0)
    W1 = normal(np.random.default_rng(seed + 1), f, h, 0.02)
    W2 = normal(np.random.default_rng(seed + 2), h, f, 0.02)
    return X, W1, W2


def random_bf16(seed: int, rows: int, cols: int, kind: str = "normal", scale: float = 1.0) -> np.ndarray:
    """Small seeded bf16 matrices for parity tests of odd shapes.
    kind: normal | laplace | t3 | wide (log-uniform magnitudes over ~2^-40..2^40) | zeros."""
    rng = np.random.default_rng(seed)
    if kind == "normal":
        a = rng.standard_normal((rows, cols)) * scale
    elif kind == "laplace":
        a = rng.laplace(0.0, scale, (rows, cols))
    elif kind == "t3":
        a = rng.standard_t(3.0, (rows, cols)) * scale
    elif kind == "wide":
        mag = np.exp2(rng.uniform(-40, 40, (rows, cols)))
        a = np.where(rng.random((rows, cols)) < 0.5, -mag, mag) * scale
    elif kind == "zeros":
        a = np.zeros((rows, cols))
    else:
        raise ValueError(kind)
    return bf16_bits(a)
