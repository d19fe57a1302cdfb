"""Pins for the oracle's compute_bias: e = floor(log2(fmax/amax)) - margin.

Pinned against hand-worked values (``golden/compute_bias_cases.txt``), against
the defining bracket amax * 2^e <= fmax < amax * 2^(e+1) checked in exact
rational arithmetic (no logarithm), the margin shift, monotonicity and the
documented special cases.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMTS = {"E4M3": 0, "E5M2": 1}


def _cases():
    out = []
    with open(os.path.join(GOLDEN, "compute_bias_cases.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                fmt, amax, margin, e = line.split()
                out.append((FMTS[fmt], float(amax), int(margin), int(e)))
    return out


@pytest.mark.parametrize("fmt,amax,margin,e", _cases())
def test_hand_worked(oracle, fmt, amax, margin, e):
    assert oracle.compute_bias(amax, fmt, margin) == (e, False)


def _bracket_ok(amax32: np.float32, fmt: int, e: int) -> bool:
    a = Fraction(float(amax32))
    fmax = Fraction(oracle_fmax(fmt))
    return a * Fraction(2) ** e <= fmax < a * Fraction(2) ** (e + 1)


def oracle_fmax(fmt):
    return 448 if fmt == 0 else 57344


def _amax_samples():
    rng = np.random.default_rng(3)
    s = list(np.exp2(rng.uniform(-125, 120, 3000)).astype(np.float32))
    # powers of two, their neighbours, and the fmax/2^k boundaries
    for k in range(-120, 120, 7):
        p = np.float32(2.0 ** k)
        s += [p, np.nextafter(p, np.float32(0)), np.nextafter(p, np.float32(np.inf))]
        for fmax in (448.0, 57344.0):
            if fmax * 2.0 ** k > 3e38:
                continue
            b = np.float32(fmax * 2.0 ** k)
            if b > 0:
                s += [b, np.nextafter(b, np.float32(0)), np.nextafter(b, np.float32(np.inf))]
    return [x for x in s if np.isfinite(x) and x > 0]


@pytest.mark.parametrize("fmt", [0, 1])
def test_bracket_property(oracle, fmt):
    for a in _amax_samples():
        e, nf = oracle.compute_bias(float(a), fmt, 0)
        assert not nf
        if -126 < e < 127:
            assert _bracket_ok(a, fmt, e), (float(a), e)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("margin", [-2, 1, 3])
def test_margin_shift(oracle, fmt, margin):
    for a in _amax_samples()[::17]:
        e0, _ = oracle.compute_bias(float(a), fmt, 0)
        e, _ = oracle.compute_bias(float(a), fmt, margin)
        if -126 < e0 < 127:  # e0 not clamped, so it is the exact floor(log2(fmax/amax))
            assert e == max(-126, min(127, e0 - margin))


@pytest.mark.parametrize("fmt", [0, 1])
def test_monotone_non_increasing(oracle, fmt):
    a = np.sort(np.array(_amax_samples(), np.float32))
    es = [oracle.compute_bias(float(x), fmt, 0)[0] for x in a]
    assert all(x >= y for x, y in zip(es, es[1:]))


def test_special_cases(oracle):
    for fmt in (0, 1):
        assert oracle.compute_bias(0.0, fmt, 0) == (0, False)
        assert oracle.compute_bias(float("inf"), fmt, 0) == (0, True)
        assert oracle.compute_bias(float("nan"), fmt, 0) == (0, True)
        assert oracle.compute_bias(1e-45, fmt, 0) == (127, False)  # clamped high
    assert oracle.compute_bias(1.0, 0, 200) == (-126, False)  # clamped low
    # the largest bf16 magnitude stays in range
    big = float(np.float32(3.3895313892515355e38))
    e, _ = oracle.compute_bias(big, 0, 0)
    assert e == math.floor(math.log2(448 / big))


def test_scale_triple_exact(oracle):
    for e in range(-126, 128):
        s, si = oracle.pow2f(e), oracle.pow2f(-e)
        assert Fraction(float(s)) == Fraction(2) ** e
        assert Fraction(float(si)) == Fraction(2) ** (-e)
