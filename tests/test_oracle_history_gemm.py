"""Pins for the oracle's delayed-scaling history and its fp64 GEMM.

History: the window-max invariant against an independent deque, checkpoint /
restore equivalence, the first-step reading.  GEMM: exact rational brute force
on tiny shapes, W = 2^j I (result = dequantised A exactly), equal block / MX
scales reduce to per-tensor, and the tolerance helper.
"""
import collections
from fractions import Fraction

import numpy as np
import pytest

import workloads as wl


@pytest.mark.parametrize("L", [1, 4, 16])
@pytest.mark.parametrize("fmt,margin", [(0, 0), (1, 1)])
def test_history_window_invariant(oracle, L, fmt, margin):
    rng = np.random.default_rng(L)
    st = oracle.HistoryState(L)
    window = collections.deque(maxlen=L)
    for t in range(3 * L + 5):
        a = np.float32(np.exp2(rng.uniform(-20, 10)))
        st.update(float(a), fmt, margin)
        window.append(a)
        e_ref, _ = oracle.compute_bias(float(max(window)), fmt, margin)
        assert st.bias[0] == e_ref
        assert st.scale[0] == np.float32(2.0 ** e_ref) and st.scale_inv[0] == np.float32(2.0 ** -e_ref)
        assert st.pos[0] == t + 1


def test_history_checkpoint_restore(oracle):
    rng = np.random.default_rng(1)
    amaxes = np.exp2(rng.uniform(-5, 5, 40)).astype(np.float32)
    a = oracle.HistoryState(8)
    for v in amaxes:
        a.update(float(v), 0, 0)
    b = oracle.HistoryState(8)
    for v in amaxes[:17]:
        b.update(float(v), 0, 0)
    c = oracle.HistoryState(8)  # restore b's state into a fresh object, continue
    c.hist[:], c.pos[:], c.bias[:], c.scale[:], c.scale_inv[:] = b.hist, b.pos, b.bias, b.scale, b.scale_inv
    for v in amaxes[17:]:
        c.update(float(v), 0, 0)
    for f in ("hist", "pos", "bias", "scale", "scale_inv"):
        assert np.array_equal(getattr(a, f), getattr(c, f))


def test_history_nonfinite(oracle):
    st = oracle.HistoryState(4)
    assert not st.update(2.0, 0, 0)
    assert st.update(float("inf"), 0, 0)
    assert st.bias[0] == 0


def test_history_nan_stays_in_window(oracle):
    """A NaN amax is flagged and gives e = 0 for as long as it stays in the window (L = 3 steps)."""
    st = oracle.HistoryState(3)
    assert not st.update(2.0, 0, 0)
    flags = [st.update(v, 0, 0) for v in (float("nan"), 1.0, 1.0)]
    assert flags == [True, True, True] and st.bias[0] == 0  # NaN recorded at step 1, still in the window
    assert not st.update(1.0, 0, 0)  # overwritten: window {1, 1, 1}
    assert st.bias[0] == oracle.compute_bias(1.0, 0, 0)[0] == 8


def test_delayed_activation_sequence(oracle):
    """The growing-activation sequence (1 + 0.1 t) at a reduced 512x512 size: after each step the
    bias is compute_bias of the window max, recomputed here from numpy amaxes."""
    st = oracle.HistoryState(16)
    seen = []
    for t in range(16):
        x = wl.delayed_activation(t, 512, 512)
        a = np.float32(np.abs(wl.bf16_to_f32(x)).max())
        assert oracle.amax(x) == a
        seen.append(a)
        st.update(float(a), 0, 0)
        assert st.bias[0] == oracle.compute_bias(float(max(seen[-16:])), 0, 0)[0]


# ------------------------------------------------------------------ GEMM

def _exact_gemm(A, fa, sa, B, fb, sb, oracle):
    M, K = A.shape
    N = B.shape[0]
    da = [[Fraction(oracle.decode(int(A[m, k]), fa)) * sa(m, k) for k in range(K)] for m in range(M)]
    db = [[Fraction(oracle.decode(int(B[n, k]), fb)) * sb(n, k) for k in range(K)] for n in range(N)]
    return [[sum(da[m][k] * db[n][k] for k in range(K)) for n in range(N)] for m in range(M)]


def _finite_codes(rng, shape, fmt):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    if fmt == 0:
        c[(c & 0x7F) == 0x7F] = 0x38
    else:
        c[(c & 0x7C) == 0x7C] = 0x3C
    return c


@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0)])
def test_gemm_exact_tensor(oracle, fa, fb):
    rng = np.random.default_rng(fa * 2 + fb)
    A = _finite_codes(rng, (3, 40), fa)
    B = _finite_codes(rng, (5, 40), fb)
    sa, sb = np.float32(2.0 ** -3), np.float32(2.0 ** 5)
    y, mag = oracle.gemm_full(A, fa, 0, sa, B, fb, 0, sb)
    ref = _exact_gemm(A, fa, lambda m, k: Fraction(float(sa)), B, fb, lambda n, k: Fraction(float(sb)), oracle)
    for m in range(3):
        for n in range(5):
            assert abs(Fraction(y[m, n]) - ref[m][n]) <= abs(ref[m][n]) * Fraction(1, 2 ** 50)
    assert np.all(mag >= np.abs(y))


@pytest.mark.parametrize("ga,gb", [(3, 3), (1, 2), (1, 1)])
def test_gemm_exact_block(oracle, ga, gb):
    rng = np.random.default_rng(ga + 10 * gb)
    M, N, K = 3, 130, 256
    A = _finite_codes(rng, (M, K), 0)
    B = _finite_codes(rng, (N, K), 0)
    if ga == 3:
        sfa = rng.integers(120, 135, (M, K // 32)).astype(np.uint8)
        sfb = rng.integers(120, 135, (N, K // 32)).astype(np.uint8)
        fa_ = lambda m, k: Fraction(2) ** (int(sfa[m, k // 32]) - 127)
        fb_ = lambda n, k: Fraction(2) ** (int(sfb[n, k // 32]) - 127)
    else:
        sfa = np.ldexp(np.float32(1), rng.integers(-6, 6, (M, K // 128))).astype(np.float32)
        rb = N if gb == 1 else -(-N // 128)
        sfb = np.ldexp(np.float32(1), rng.integers(-6, 6, (rb, K // 128))).astype(np.float32)
        fa_ = lambda m, k: Fraction(float(sfa[m, k // 128]))
        fb_ = (lambda n, k: Fraction(float(sfb[n, k // 128]))) if gb == 1 else \
              (lambda n, k: Fraction(float(sfb[n // 128, k // 128])))
    ms = np.array([0, 1, 2, 2, 0], np.int64)
    ns = np.array([0, 7, 127, 128, 129], np.int64)
    y, _ = oracle.gemm_sample(A, 0, ga, sfa, B, 0, gb, sfb, ms, ns)
    ref = _exact_gemm(A, 0, fa_, B[: N], 0, fb_, oracle)
    for i, (m, n) in enumerate(zip(ms, ns)):
        assert abs(Fraction(y[i]) - ref[m][n]) <= abs(ref[m][n]) * Fraction(1, 2 ** 50)


@pytest.mark.parametrize("ga,gb", [(3, 3), (1, 2), (1, 1)])
def test_gemm_full_exact_block(oracle, ga, gb):
    """The whole product with distinct block scales per row and per K block, element by element
    against exact rational arithmetic (rows and K blocks both cross the scale-block edges)."""
    rng = np.random.default_rng(30 + ga + 10 * gb)
    M, N, K = 5, 133, 256
    A = _finite_codes(rng, (M, K), 0)
    B = _finite_codes(rng, (N, K), 1)
    if ga == 3:
        sfa = rng.integers(118, 137, (M, K // 32)).astype(np.uint8)
        sfb = rng.integers(118, 137, (N, K // 32)).astype(np.uint8)
        fa_ = lambda m, k: Fraction(2) ** (int(sfa[m, k // 32]) - 127)
        fb_ = lambda n, k: Fraction(2) ** (int(sfb[n, k // 32]) - 127)
    else:
        sfa = np.ldexp(np.float32(1), rng.integers(-6, 7, (M, K // 128))).astype(np.float32)
        rb = N if gb == 1 else -(-N // 128)
        sfb = np.ldexp(np.float32(1), rng.integers(-6, 7, (rb, K // 128))).astype(np.float32)
        fa_ = lambda m, k: Fraction(float(sfa[m, k // 128]))
        fb_ = (lambda n, k: Fraction(float(sfb[n, k // 128]))) if gb == 1 else \
              (lambda n, k: Fraction(float(sfb[n // 128, k // 128])))
    y, mag = oracle.gemm_full(A, 0, ga, sfa, B, 1, gb, sfb)
    ref = _exact_gemm(A, 0, fa_, B, 1, fb_, oracle)
    for m in range(M):
        for n in range(N):
            # fp64 summation of K products with cancellation: within K ulps of sum |a b|
            assert abs(Fraction(y[m, n]) - ref[m][n]) <= Fraction(float(mag[m, n])) * K * Fraction(1, 2 ** 52), (m, n)
    assert np.all(mag >= np.abs(y))


def test_gemm_identity_weight(oracle):
    """B = 2^j I: y = deq(A) 2^j exactly."""
    rng = np.random.default_rng(0)
    K = 64
    A = _finite_codes(rng, (7, K), 0)
    B = np.zeros((K, K), np.uint8)
    np.fill_diagonal(B, 0x38)  # 1.0
    sa = np.float32(2.0 ** -4)
    y, _ = oracle.gemm_full(A, 0, 0, sa, B, 0, 0, np.float32(8.0))
    assert np.array_equal(y, oracle.decode_array(A, 0) * float(sa) * 8.0)


def test_gemm_equal_scales_reduce_to_tensor(oracle):
    rng = np.random.default_rng(5)
    M, N, K = 4, 6, 128
    A = _finite_codes(rng, (M, K), 0)
    B = _finite_codes(rng, (N, K), 0)
    yt, _ = oracle.gemm_full(A, 0, 0, np.float32(0.25), B, 0, 0, np.float32(4.0))
    ym, _ = oracle.gemm_full(A, 0, 3, np.full((M, K // 32), 125, np.uint8), B, 0, 3,
                             np.full((N, K // 32), 129, np.uint8))
    yb, _ = oracle.gemm_full(A, 0, 1, np.full((M, 1), 0.25, np.float32), B, 0, 2,
                             np.full((1, 1), 4.0, np.float32))
    assert np.array_equal(yt, ym) and np.array_equal(yt, yb)


def test_gemm_tolerance_helper(oracle):
    y_ref = np.array([1.0, 3.0, -1000.0, 0.0])
    mag = np.array([1.0, 3.0, 1000.0, 0.0])
    t = oracle.gemm_tolerance(y_ref, mag, out_bf16=False)
    assert np.allclose(t, 1e-3 * mag)
    tb = oracle.gemm_tolerance(y_ref, mag, out_bf16=True)
    # bf16 ulp of 1.0 is 2^-7, of 3.0 is 2^-6, of 1000 is 4
    assert np.allclose(tb - t, [2 ** -8, 2 ** -7, 2.0, 0.0])


# ------------------------------------------------ FP8-output bracket

@pytest.mark.parametrize("fmt", [0, 1])
def test_gemm_quantize_bracket_brute_force(oracle, fmt):
    """Every fp32 v in a narrow interval around y is walked one ulp at a time: every
    Encode(fl32(v s)) lies between the bracket's ends (by value).  Half the y sit exactly on a
    rounding midpoint (after scaling), where both neighbouring codes must be admitted."""
    rng = np.random.default_rng(40 + fmt)
    s = np.float32(2.0 ** 3)
    fmax = 448.0 if fmt == 0 else 57344.0
    ys = list(rng.uniform(fmax / 64, fmax / 8, 30) * rng.choice([-1, 1], 30))
    for c in rng.integers(1, 0x7E if fmt == 0 else 0x7B, 30):  # midpoints between code c and c+1
        mid = (oracle.decode(int(c), fmt) + oracle.decode(int(c) + 1, fmt)) / 2
        ys.append(mid / float(s))
    for k, y in enumerate(ys):
        tol = abs(y) * 2e-6
        lo, hi, near = oracle.gemm_quantize_bracket(np.array([y]), np.array([tol]), fmt, s)
        dlo, dhi = oracle.decode(int(lo[0]), fmt), oracle.decode(int(hi[0]), fmt)
        assert dlo <= oracle.decode(int(near[0]), fmt) <= dhi
        v = np.float32(y - tol)
        seen = set()
        while float(v) <= y + tol:
            if float(v) >= y - tol:
                d = oracle.decode(oracle.encode(float(np.float32(v * s)), fmt), fmt)
                assert dlo <= d <= dhi, (y, float(v), d)
                seen.add(d)
            v = np.nextafter(v, np.float32(np.inf))
        assert seen <= {dlo, dhi}
        if k >= 30:  # on a midpoint: both neighbours are reachable and admitted
            assert seen == {dlo, dhi} and dlo < dhi


def test_gemm_quantize_bracket_exact_values(oracle):
    """tol = 0 on values exactly representable after scaling: lo = hi = the code of y s."""
    for fmt in (0, 1):
        codes = np.array([c for c in range(256) if not np.isnan(oracle.decode(c, fmt))], np.uint8)
        y = oracle.decode_array(codes, fmt) / 4.0  # scale 4 maps y back onto the codes
        lo, hi, near = oracle.gemm_quantize_bracket(y, np.zeros_like(y), fmt, 4.0)
        keep = np.abs(y * 4) < (448 if fmt == 0 else 57344) + 1  # Inf codes of E5M2 saturate
        assert np.array_equal(lo[keep] & 0x7F, codes[keep] & 0x7F)
        # by value: -0 - 0 and -0 + 0 differ in sign only
        dl, dh, dn = (oracle.decode_array(c, fmt) for c in (lo, hi, near))
        assert np.array_equal(dl, dh) and np.array_equal(dn, dl)


def test_round_bf16_matches_torch(oracle):
    """bf16 rounding (ties to even) against torch's CPU float32 -> bfloat16 conversion."""
    import torch
    rng = np.random.default_rng(77)
    v = np.concatenate([rng.standard_normal(20000).astype(np.float32) * np.float32(1e3),
                        np.exp2(rng.uniform(-130, 120, 20000)).astype(np.float32),
                        # exact ties: bf16 value plus half a bf16 ulp
                        (np.arange(1, 5000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(oracle.round_bf16(v).view(np.uint32), ref.view(np.uint32))
