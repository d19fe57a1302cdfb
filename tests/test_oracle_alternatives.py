"""Pins for the two scale rules kept behind options: the OCP MX bias for 1x32 blocks and the
non-power-of-two ratio scale s = fmax / amax.

OCP bias: hand-worked values; the defining property (the block's largest magnitude lands in the
format's top binade, 2^emax <= amax 2^e < 2^(emax+1)) in exact rational arithmetic; its relation
to compute_bias (one larger exactly when amax's significand exceeds 1.75, the case that
saturates); the block cast against a pure-Python brute force.  Ratio scale: every result within
half an fp32 ulp of the exact quotient (correct rounding), exact for powers of two."""
from fractions import Fraction

import numpy as np
import pytest

import workloads as wl
from test_oracle_quant import _brute_encode, _nearest_code_table

EMAX = {0: 8, 1: 15}
FMAX = {0: 448.0, 1: 57344.0}


def _samples():
    rng = np.random.default_rng(17)
    s = list(np.exp2(rng.uniform(-120, 120, 2000)).astype(np.float32))
    for k in range(-100, 100, 9):
        for sig in (1.0, 1.5, 1.75, 1.8, 1.9921875):
            s.append(np.float32(sig * 2.0 ** k))
            s.append(np.nextafter(np.float32(sig * 2.0 ** k), np.float32(np.inf)))
    return [float(x) for x in s if np.isfinite(x) and x > 0]


@pytest.mark.parametrize("fmt,amax,e", [(0, 448.0, 0), (0, 480.0, 0), (0, 1.0, 8), (0, 1.9, 8), (0, 0.5, 9),
                                        (1, 1.0, 15), (1, 57344.0, 0), (1, 61440.0, 0)])
def test_ocp_hand_values(oracle, fmt, amax, e):
    assert oracle.compute_bias_ocp(amax, fmt) == (e, False)


@pytest.mark.parametrize("fmt", [0, 1])
def test_ocp_top_binade_and_relation(oracle, fmt):
    for a in _samples():
        e, nf = oracle.compute_bias_ocp(a, fmt)
        assert not nf
        if -126 < e < 127:
            v = Fraction(a) * Fraction(2) ** e
            assert Fraction(2) ** EMAX[fmt] <= v < Fraction(2) ** (EMAX[fmt] + 1), (a, e)
            e_cb, _ = oracle.compute_bias(a, fmt)
            if -126 < e_cb < 127:
                k = Fraction(a).numerator.bit_length() - Fraction(a).denominator.bit_length()
                sig = Fraction(a) / Fraction(2) ** k
                if sig < 1:
                    sig *= 2
                assert e - e_cb == (1 if sig > Fraction(7, 4) else 0), (a, e, e_cb)
    assert oracle.compute_bias_ocp(0.0, fmt) == (0, False)
    assert oracle.compute_bias_ocp(float("nan"), fmt) == (0, True)
    assert oracle.compute_bias_ocp(1.0, fmt, 3) == (EMAX[fmt] - 3, False)


def _ocp_by_search(amax, fmt):
    if amax == 0:
        return 0
    a, lo, e = Fraction(amax), Fraction(2) ** EMAX[fmt], 0
    while a * Fraction(2) ** e >= 2 * lo:
        e -= 1
    while a * Fraction(2) ** e < lo:
        e += 1
    return max(-126, min(127, e))


@pytest.mark.parametrize("fmt", [0, 1])
def test_ocp_block_cast_brute_force(oracle, fmt):
    x_bits = wl.random_bf16(600 + fmt, 24, 96, "wide")
    x = wl.bf16_to_f32(x_bits)
    table = _nearest_code_table(oracle, fmt)
    qr, sr, qc, sc, nf = oracle.quantize_block(x_bits, fmt, oracle.MX_1x32_OCP, 0, row=True, col=True)
    assert not nf
    for q, s, m in ((qr, sr, x), (qc, sc, np.ascontiguousarray(x.T))):
        R, C = m.shape
        for r in range(R):
            for b in range(C // 32):
                blk = m[r, 32 * b:32 * (b + 1)]
                e = _ocp_by_search(float(np.abs(blk).max()), fmt)
                assert int(s[r, b]) == 127 - e
                ref = _brute_encode((blk * np.float32(2.0 ** e)).astype(np.float32), fmt, table)
                assert np.array_equal(q[r, 32 * b:32 * (b + 1)], ref)
    # the same blocks under the default rule differ only where the OCP rule is one larger
    _, sr_d, _, _, _ = oracle.quantize_block(x_bits, fmt, oracle.MX_1x32, 0)
    assert set(np.unique(sr_d.astype(int) - sr.astype(int))) <= {0, 1}


def _is_rn(q: np.float32, exact: Fraction) -> bool:
    """q is exact rounded to the nearest fp32."""
    lo, hi = np.nextafter(q, np.float32(0)), np.nextafter(q, np.float32(np.inf))
    d = abs(Fraction(float(q)) - exact)
    return d <= abs(Fraction(float(lo)) - exact) and d <= abs(Fraction(float(hi)) - exact)


@pytest.mark.parametrize("fmt", [0, 1])
def test_ratio_scale_correctly_rounded(oracle, fmt):
    for a in _samples()[::7]:
        s, si, nf = oracle.scale_ratio(a, fmt)
        assert not nf
        if not np.isfinite(s) or s == 0:
            continue
        assert _is_rn(s, Fraction(FMAX[fmt]) / Fraction(a)), a
        if np.isfinite(si) and si != 0:
            assert _is_rn(si, 1 / Fraction(float(s))), a
    s, si, _ = oracle.scale_ratio(2.0 ** -4, fmt)  # a power-of-two amax: s is exact
    assert s == np.float32(FMAX[fmt] * 16) and si == np.float32(1 / (FMAX[fmt] * 16))
    assert oracle.scale_ratio(0.0, fmt)[:2] == (1.0, 1.0)
    assert oracle.scale_ratio(float("inf"), fmt)[2]
