"""Pins for the oracle's cast statistics (saturated / flushed-to-zero counts at a given scale).

Power-of-two scales over all 65536 bf16 patterns are counted in exact rational arithmetic with no
FP8 encoder at all (a product beyond fmax saturates; a non-zero product at or below half the
smallest subnormal rounds to zero, the tie going to the even code 0).  Arbitrary scales are checked
against torch's CPU float8 conversion, and NaN / zero elements count in neither."""
from fractions import Fraction

import numpy as np
import pytest

FMAX = {0: Fraction(448), 1: Fraction(57344)}
HALF_MIN_SUB = {0: Fraction(1, 2 ** 10), 1: Fraction(1, 2 ** 17)}


def _bf16_fraction(p: int):
    """Exact value of a positive bf16 bit pattern (None for inf)."""
    e, m = p >> 7, p & 0x7F
    if e == 0xFF:
        return None
    if e == 0:
        return Fraction(m, 2 ** 7) * Fraction(1, 2 ** 126)
    return (1 + Fraction(m, 2 ** 7)) * (Fraction(2) ** (e - 127))


POS = [p for p in range(0x7F81)]  # +0 .. +inf (NaN patterns excluded)
VALS = [_bf16_fraction(p) for p in POS]


@pytest.mark.parametrize("fmt", [0, 1])
def test_power_of_two_scales_exhaustive(oracle, fmt):
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    es = list(range(-20, 21, 3)) + [-126, 127]
    sat, und = oracle.cast_stats(x, fmt, [float(2.0 ** e) for e in es])
    for j, e in enumerate(es):
        s = Fraction(2) ** e
        n_sat = sum(1 for v in VALS if v is None or v * s > FMAX[fmt])
        n_und = sum(1 for v in VALS if v is not None and v != 0 and v * s <= HALF_MIN_SUB[fmt])
        assert sat[j] == 2 * n_sat, (e, int(sat[j]), 2 * n_sat)  # both signs
        assert und[j] == 2 * n_und, (e, int(und[j]), 2 * n_und)


@pytest.mark.parametrize("fmt", [0, 1])
def test_arbitrary_scales_against_torch(oracle, fmt):
    import torch
    rng = np.random.default_rng(5 + fmt)
    bits = rng.integers(0, 65536, (64, 256)).astype(np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] = 0x3F80  # no inf / NaN here
    xf = (bits.astype(np.uint32) << 16).view(np.float32)
    scales = [0.3, 3.7, 1e-3, 1234.5, 2.0 ** -30]
    sat, und = oracle.cast_stats(bits, fmt, scales)
    t8 = torch.float8_e4m3fn if fmt == 0 else torch.float8_e5m2
    fmax = 448.0 if fmt == 0 else 57344.0
    for j, s in enumerate(scales):
        with np.errstate(over="ignore"):
            v = xf * np.float32(s)
        assert sat[j] == int((np.abs(v.astype(np.float64)) > fmax).sum())
        inr = np.abs(v) <= fmax  # torch's conversion is RNE inside the range
        zero = torch.from_numpy(v[inr]).to(t8).to(torch.float32).numpy() == 0
        assert und[j] == int((zero & (xf[inr] != 0)).sum())


def test_nan_and_zero_count_in_neither(oracle):
    x = np.array([[0x7FC0, 0xFFC1, 0x0000, 0x8000, 0x7F80, 0x0001]], np.uint16)  # NaN, NaN, +0, -0, inf, tiny
    sat, und = oracle.cast_stats(x, 0, [1.0])
    assert int(sat[0]) == 1 and int(und[0]) == 1  # inf saturates; the bf16 subnormal flushes
