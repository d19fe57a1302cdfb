"""Pins for the oracle's scaled cast (per tensor and per block) and amax.

Independent checks: a pure-Python brute-force quantiser (block amax by numpy,
bias by searching the bracket amax 2^e <= fmax < amax 2^(e+1) with exact
rationals, nearest code by scanning all codes), the closed form of the
outlier workload (amax = 30 exactly, e = 3), the RNE error bound, and
structural invariants (column-wise = transpose for a shared scale, equal block
scales reduce to per-tensor).
"""
from fractions import Fraction

import numpy as np
import pytest

import workloads as wl


def _bias_by_search(amax: float, fmt: int, margin: int = 0) -> int:
    if amax == 0:
        return 0
    fmax = Fraction(448 if fmt == 0 else 57344)
    a = Fraction(amax)
    e = 0
    while a * Fraction(2) ** e > fmax:
        e -= 1
    while a * Fraction(2) ** (e + 1) <= fmax:
        e += 1
    return max(-126, min(127, e - margin))


def _nearest_code_table(oracle, fmt):
    mc = oracle.maxcode(fmt)
    return np.array([oracle.decode(c, fmt) for c in range(mc + 1)])


def _brute_encode(vals: np.ndarray, fmt: int, table: np.ndarray) -> np.ndarray:
    """Nearest code by full scan (ties to even), saturating, sign kept."""
    a = np.minimum(np.abs(vals.astype(np.float64)), table[-1])
    d = np.abs(a[:, None] - table[None, :])
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    idx = np.arange(table.size)
    # among tied candidates pick the even code
    pick = np.where(cand & (idx % 2 == 0), idx, 10_000).min(axis=1)
    pick = np.where(pick == 10_000, np.argmax(cand, axis=1), pick)
    sign = np.signbit(vals.astype(np.float32))
    return (pick | np.where(sign, 0x80, 0)).astype(np.uint8)


def _brute_block(x_bits, fmt, br, bc, margin, table):
    x = wl.bf16_to_f32(x_bits)
    R, C = x.shape
    q = np.zeros((R, C), np.uint8)
    nbr, nbc = -(-R // br), -(-C // bc)
    es = np.zeros((nbr, nbc), np.int64)
    for bi in range(nbr):
        for bj in range(nbc):
            blk = x[bi * br:(bi + 1) * br, bj * bc:(bj + 1) * bc]
            e = _bias_by_search(float(np.abs(blk).max()), fmt, margin)
            es[bi, bj] = e
            s = np.float32(2.0 ** e)
            p = (blk * s).astype(np.float32)
            q[bi * br:(bi + 1) * br, bj * bc:(bj + 1) * bc] = _brute_encode(p.reshape(-1), fmt, table).reshape(p.shape)
    return q, es


@pytest.mark.parametrize("gran", [1, 2, 3])
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shape", [(3, 160), (130, 96), (40, 64)])
def test_block_quant_brute_force(oracle, gran, fmt, shape):
    R, C = shape
    x = wl.random_bf16(100 + gran * 10 + fmt, R, C, "wide")
    table = _nearest_code_table(oracle, fmt)
    br, bc = oracle.block_shape(gran)
    margin = 1 if fmt == 1 else 0
    qr, sr, qc, sc, nf = oracle.quantize_block(x, fmt, gran, margin, row=True, col=True)
    assert not nf
    q_ref, e_ref = _brute_block(x, fmt, br, bc, margin, table)
    assert np.array_equal(qr, q_ref)
    qT_ref, eT_ref = _brute_block(np.ascontiguousarray(x.T), fmt, br, bc, margin, table)
    assert np.array_equal(qc, qT_ref)
    if gran == oracle.MX_1x32:
        assert np.array_equal(sr.astype(np.int64), 127 - e_ref)
        assert np.array_equal(sc.astype(np.int64), 127 - eT_ref)
    else:
        assert np.array_equal(sr, np.ldexp(np.float32(1), -e_ref).astype(np.float32))
        assert np.array_equal(sc, np.ldexp(np.float32(1), -eT_ref).astype(np.float32))
    if gran == oracle.BLOCK_128x128:
        assert np.array_equal(sc, sr.T)


@pytest.mark.parametrize("fmt", [0, 1])
def test_tensor_quant_brute_force(oracle, fmt):
    x = wl.random_bf16(5 + fmt, 37, 48, "wide", 1e-3)
    table = _nearest_code_table(oracle, fmt)
    amax = float(np.abs(wl.bf16_to_f32(x)).max())
    e = _bias_by_search(amax, fmt)
    s = np.float32(2.0 ** e)
    qr, qc = oracle.quantize_tensor(x, fmt, s, row=True, col=True)
    ref = _brute_encode((wl.bf16_to_f32(x) * s).astype(np.float32).reshape(-1), fmt, table).reshape(x.shape)
    assert np.array_equal(qr, ref)
    assert np.array_equal(qc, qr.T)


def test_amax_matches_numpy(oracle):
    for kind in ["normal", "wide", "zeros", "t3"]:
        x = wl.random_bf16(9, 33, 70, kind)
        assert oracle.amax(x) == np.float32(np.abs(wl.bf16_to_f32(x)).max())
    x = wl.random_bf16(9, 4, 8, "normal")
    x[2, 3] = 0x7FC0  # NaN propagates
    assert np.isnan(oracle.amax(x))


def test_outlier_workload_closed_form(oracle):
    """Eight +-30 outliers dominate N(0, 0.02^2): amax_X = 30 and e_X = 3 whatever the draw."""
    X, W = wl.linear_fwd_current()
    assert X.shape == (256, 1024) and W.shape == (1024, 1024)
    assert oracle.amax(X) == np.float32(30.0)
    assert oracle.compute_bias(30.0, 0, 0) == (3, False)
    xf = wl.bf16_to_f32(X)
    assert int((np.abs(xf) == 30.0).sum()) == 8


@pytest.mark.parametrize("fmt", [0, 1])
def test_rne_error_bound(oracle, fmt):
    """|decode(q) 2^-e - x| <= half the FP8 spacing at x 2^e (saturation excluded: amax scaling keeps
    x 2^e <= fmax)."""
    x = wl.random_bf16(21 + fmt, 64, 256, "laplace", 3.0)
    xf = wl.bf16_to_f32(x).astype(np.float64)
    e, s, si = oracle.scale_triple(float(np.abs(xf).max()), fmt)
    qr, _ = oracle.quantize_tensor(x, fmt, s)
    deq = oracle.decode_array(qr, fmt)
    p = xf * float(s)
    assert np.abs(p).max() <= oracle.FMAX[fmt]
    mb, bias = (3, 7) if fmt == 0 else (2, 15)
    expo = np.floor(np.log2(np.maximum(np.abs(p), 2.0 ** (1 - bias))))
    half_spacing = np.ldexp(0.5, (expo - mb).astype(np.int64))
    assert np.all(np.abs(deq - p) <= half_spacing)


def test_equal_block_scales_reduce_to_tensor(oracle):
    """If every 1x128 block has the same amax, block quantisation equals per-tensor quantisation."""
    x = wl.random_bf16(4, 16, 256, "normal")
    x[:, ::128] = wl.bf16_bits(np.full((16, 2), 7.5))  # every block's amax is 7.5
    qb, sb, _, _, _ = oracle.quantize_block(x, 0, oracle.BLOCK_1x128)
    e, s, si = oracle.scale_triple(7.5, 0)
    qt, _ = oracle.quantize_tensor(x, 0, s)
    assert np.array_equal(qb, qt)
    assert np.all(sb == si)


def test_generator_chunk_invariance():
    """The chunked generators give the same stream as a single draw."""
    old = wl.CHUNK_ELEMS
    try:
        wl.CHUNK_ELEMS = 1000
        a = wl.normal(np.random.default_rng(3), 70, 64, 0.02)
        b = wl.laplace(np.random.default_rng(4), 70, 64, 1e-5)
        c = wl.student_t(np.random.default_rng(5), 70, 64, 3.0, 0.5)
    finally:
        wl.CHUNK_ELEMS = old
    assert np.array_equal(a, wl.bf16_bits(np.random.default_rng(3).standard_normal((70, 64)) * 0.02))
    assert np.array_equal(b, wl.bf16_bits(np.random.default_rng(4).laplace(0.0, 1e-5, (70, 64))))
    assert np.array_equal(c, wl.bf16_bits(np.random.default_rng(5).standard_t(3.0, (70, 64)) * 0.5))


def test_bf16_rounding_rne():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, -2.5], np.float64)
    got = wl.bf16_bits(v)
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7: ties to even (1.0)
    assert list(got) == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC020]
