"""Pins for the oracle's per-tensor cast and amax of fp32 arrays.

Inside the format's range the cast is checked against torch: its fp32 multiply and its own
float32 -> float8 conversion (round to nearest even), which share no code with the oracle.  Outside
the range, where torch's conversion does not saturate, the expected codes are worked by hand:
+-Inf and every product beyond fmax give +-fmax, NaN a NaN code, a negative underflow 0x80.  The
amax against numpy's max of |x|."""
import numpy as np
import pytest
import torch

TORCH_DT = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}
FMAX = {0: 448.0, 1: 57344.0}
MAXCODE = {0: 0x7E, 1: 0x7B}


def _values(rng, n):
    mag = np.exp2(rng.uniform(-40, 40, n))
    return (mag * rng.choice([-1.0, 1.0], n)).astype(np.float32)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("scale", [1.0, 2.0 ** -7, 2.0 ** 9, 0.3, 1234.5678])
def test_matches_torch_in_range(oracle, fmt, scale):
    rng = np.random.default_rng(fmt * 10 + int(scale * 7) % 97)
    x = _values(rng, 200_000)
    s = np.float32(scale)
    p = (torch.from_numpy(x) * torch.tensor(s)).numpy()  # torch's fp32 product
    keep = np.abs(p) <= FMAX[fmt]
    ref = torch.from_numpy(p[keep]).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    got = oracle.quantize_f32(x, fmt, s)[keep]
    assert keep.sum() > 50_000
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt", [0, 1])
def test_saturation_and_specials(oracle, fmt):
    f = FMAX[fmt]
    big = np.float32(np.nextafter(np.float32(f), np.float32(np.inf)))
    x = np.array([np.inf, -np.inf, big, -big, 3.0e38, -3.0e38, f, -f, 0.0, -0.0, -1e-30, 1e-30, np.nan],
                 np.float32)
    q = oracle.quantize_f32(x, fmt, 1.0)
    mc = MAXCODE[fmt]
    assert list(q[:8]) == [mc, 0x80 | mc] * 4
    assert list(q[8:12]) == [0x00, 0x80, 0x80, 0x00]
    nan = q[12] & 0x7F
    assert (nan == 0x7F) if fmt == 0 else (nan > 0x7C)
    # a finite product that overflows fp32 saturates too
    assert oracle.quantize_f32(np.array([1e30, -1e30], np.float32), fmt, 1e30).tolist() == [mc, 0x80 | mc]


def test_amax_f32(oracle):
    rng = np.random.default_rng(5)
    x = _values(rng, 100_001)
    assert oracle.amax_f32(x) == np.max(np.abs(x))
    assert oracle.amax_f32(np.array([-0.0, 0.0], np.float32)) == 0.0
    assert oracle.amax_f32(np.array([1.0, -np.inf, 2.0], np.float32)) == np.inf
    x[777] = np.nan
    assert np.isnan(oracle.amax_f32(x))
