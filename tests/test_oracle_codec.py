"""Pins for the oracle's FP8 codec (CPU only).

The codec is pinned against: the named format values in
``golden/fp8_format_values.txt``; PyTorch's own float8 casts (an independent
implementation) for every code and for in-range fp32 inputs; brute force over
all 256 codes for the nearest-value rule; and the saturation / sign / tie rules.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMTS = {"E4M3": 0, "E5M2": 1}
TORCH_DT = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}


def _golden_formats():
    rows = []
    with open(os.path.join(GOLDEN, "fp8_format_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            fmt, code, val = line.split()
            rows.append((FMTS[fmt], int(code, 16), float(val)))
    return rows


@pytest.mark.parametrize("fmt,code,val", _golden_formats())
def test_named_values(oracle, fmt, code, val):
    got = oracle.decode(code, fmt)
    if math.isnan(val):
        assert math.isnan(got)
    else:
        assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val)


@pytest.mark.parametrize("fmt", [0, 1])
def test_decode_matches_torch_all_codes(oracle, fmt):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(TORCH_DT[fmt]).to(torch.float64).numpy()
    got = oracle.decode_array(codes, fmt)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("fmt,n_finite", [(0, 254), (1, 248)])
def test_code_space(oracle, fmt, n_finite):
    vals = oracle.decode_array(np.arange(256, dtype=np.uint8), fmt)
    assert np.isfinite(vals).sum() == n_finite
    pos = vals[: oracle.maxcode(fmt) + 1]
    assert np.all(np.diff(pos) > 0), "non-negative codes must be strictly increasing"
    assert pos.max() == oracle.FMAX[fmt]


@pytest.mark.parametrize("fmt", [0, 1])
def test_roundtrip_every_finite_code(oracle, fmt):
    for c in range(256):
        v = oracle.decode(c, fmt)
        if math.isnan(v) or math.isinf(v):
            continue
        assert oracle.encode(v, fmt) == c, hex(c)


def _brute_nearest(v: float, fmt: int, oracle) -> int:
    """Nearest finite code by scanning all of them; ties to the even code; saturating."""
    fmax = oracle.FMAX[fmt]
    a = min(abs(v), fmax)
    best, bestd = None, None
    for c in range(oracle.maxcode(fmt) + 1):
        d = abs(oracle.decode(c, fmt) - a)
        if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
            best, bestd = c, d
    return best | (0x80 if math.copysign(1.0, v) < 0 else 0)


@pytest.mark.parametrize("fmt", [0, 1])
def test_encode_brute_force(oracle, fmt):
    rng = np.random.default_rng(7 + fmt)
    emax = 9 if fmt == 0 else 16
    emin = -12 if fmt == 0 else -19
    vals = np.exp2(rng.uniform(emin, emax, 600)) * np.where(rng.random(600) < 0.5, -1, 1)
    vals = vals.astype(np.float32)
    for v in vals:
        assert oracle.encode(float(v), fmt) == _brute_nearest(float(v), fmt, oracle), float(v)


@pytest.mark.parametrize("fmt", [0, 1])
def test_midpoints_tie_to_even(oracle, fmt):
    mc = oracle.maxcode(fmt)
    for c in range(mc):
        lo, hi = oracle.decode(c, fmt), oracle.decode(c + 1, fmt)
        mid = np.float32(0.5 * (lo + hi))
        assert float(mid) == 0.5 * (lo + hi)  # representable in fp32
        even = c if c % 2 == 0 else c + 1
        assert oracle.encode(float(mid), fmt) == even
        assert oracle.encode(float(np.nextafter(mid, np.float32(0))), fmt) == c
        assert oracle.encode(float(np.nextafter(mid, np.float32(np.inf))), fmt) == c + 1
        assert oracle.encode(-float(mid), fmt) == 0x80 | even


@pytest.mark.parametrize("fmt", [0, 1])
def test_saturation_and_specials(oracle, fmt):
    mc = oracle.maxcode(fmt)
    fmax = oracle.FMAX[fmt]
    for v in [fmax, fmax * 1.0001, fmax * 1.5, 1e30, float("inf")]:
        assert oracle.encode(v, fmt) == mc
        assert oracle.encode(-v, fmt) == 0x80 | mc
    assert oracle.encode(float("nan"), fmt) == 0x7F and math.isnan(oracle.decode(0x7F, fmt))
    assert oracle.encode(0.0, fmt) == 0x00
    assert oracle.encode(-0.0, fmt) == 0x80
    tiny = oracle.decode(1, fmt)
    assert oracle.encode(-tiny * 0.25, fmt) == 0x80  # underflow keeps the sign
    assert oracle.encode(tiny * 0.5, fmt) == 0x00  # exact half of the min subnormal ties to 0
    assert oracle.encode(float(np.nextafter(np.float32(tiny * 0.5), np.float32(1))), fmt) == 0x01
    assert oracle.encode(1e-45, fmt) == 0  # fp32 subnormal input


@pytest.mark.parametrize("fmt", [0, 1])
def test_encode_matches_torch_in_range(oracle, fmt):
    """PyTorch's float8 casts round to nearest-even but do not saturate, so compare
    only on |v| <= fmax, over random magnitudes spanning the whole FP8 range."""
    rng = np.random.default_rng(11 + fmt)
    n = 400_000
    lo, hi = (-12, 8.8) if fmt == 0 else (-19, 15.8)
    v = (np.exp2(rng.uniform(lo, hi, n)) * np.where(rng.random(n) < 0.5, -1, 1)).astype(np.float32)
    v = v[np.abs(v) <= oracle.FMAX[fmt]]
    ref = torch.from_numpy(v).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    got = oracle.encode_array(v, fmt)
    assert np.array_equal(got, ref)
