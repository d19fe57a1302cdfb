"""GPU parity: the per-tensor FP8 GEMM whose epilogue casts D to FP8 (fp8_scaled_gemm_quantize).

D itself is only known to within the GEMM tolerance (fp32 accumulation in another order than the
fp64 oracle), so a code is correct when it is the cast of some value inside that tolerance: it
must lie between the oracle's codes for y_ref - tol and y_ref + tol.  Away from rounding
boundaries that bracket is one code, so nearly every code must equal the cast of y_ref itself.
The fused amax must lie within the same tolerance of max |y_ref|."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import host, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return require_gpu()


def realistic_codes(rng, shape, fmt):
    v = (rng.standard_normal(shape) * (100.0 if fmt == 0 else 8000.0)).astype(np.float32)
    return oracle.encode_array(v, fmt)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(q, A, fa, sa, B, fb, sb, fd, sd, amax0=0.0, with_amax=True, ldd=None):
    M, N = A.shape[0], B.shape[0]
    ldd = ldd or N
    Dq = torch.full((M, ldd), 0xAB, dtype=torch.uint8, device="cuda")
    amax = torch.tensor([amax0], dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.fp8_scaled_gemm_quantize(q.FPROP, _dev(A), fa, _dev(sa), _dev(B), fb, _dev(sb), Dq[:, :N], fd,
                               _dev(np.array([sd], np.float32)), amax if with_amax else None, status)
    return host(Dq), float(host(amax)[0]), int(host(status)[0])


def check(Dq, amax, y_ref, mag, fd, sd, min_exact=0.999):
    tol = oracle.gemm_tolerance(y_ref, mag, False)
    lo, hi, near = oracle.gemm_quantize_bracket(y_ref, tol, fd, sd)
    d, dl, dh, dn = (oracle.decode_array(c, fd) for c in (Dq, lo, hi, near))
    bad = ~((dl <= d) & (d <= dh))
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{int(bad.sum())} codes outside the bracket; first {i.tolist()}: "
                             f"got {[float(d[tuple(k)]) for k in i]} lo {[float(dl[tuple(k)]) for k in i]} "
                             f"hi {[float(dh[tuple(k)]) for k in i]}")
    assert np.mean(d == dn) >= min_exact
    a = np.abs(y_ref)
    assert (a - tol).max() <= amax <= (a + tol).max()


def delayed_like_scale(y_ref, fd):
    """The scale delayed scaling would pick if the history held this output's own amax."""
    return float(oracle.scale_triple(np.float32(np.abs(y_ref).max()), fd)[1])


SHAPES = [(128, 256, 256), (200, 272, 384), (512, 512, 1024), (96, 48, 128), (384, 16, 64), (129, 48, 512),
          (257, 1008, 512)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("fa,fb,fd", [(0, 0, 0), (1, 0, 0), (0, 0, 1)])
def test_fused_output_cast(q, M, N, K, fa, fb, fd):
    rng = np.random.default_rng(M + 3 * N + 7 * K + fa + 2 * fd)
    A, B = realistic_codes(rng, (M, K), fa), realistic_codes(rng, (N, K), fb)
    sa, sb = np.array([2.0 ** -6], np.float32), np.array([2.0 ** -5], np.float32)
    y_ref, mag = oracle.gemm_full(A, fa, 0, sa, B, fb, 0, sb)
    sd = delayed_like_scale(y_ref, fd)
    Dq, amax, st = run(q, A, fa, sa, B, fb, sb, fd, sd)
    assert st == 0
    check(Dq, amax, y_ref, mag, fd, sd)


@pytest.mark.parametrize("fd", [0, 1])
def test_saturating_and_underflowing_scales(q, fd):
    """A scale 16x too large saturates the tail (codes at +-max); one 2^20 too small flushes most
    outputs to zero.  Both must still be the cast of an admissible value."""
    rng = np.random.default_rng(9 + fd)
    A, B = realistic_codes(rng, (256, 512), 0), realistic_codes(rng, (512, 512), 0)
    sa, sb = np.array([2.0 ** -6], np.float32), np.array([2.0 ** -6], np.float32)
    y_ref, mag = oracle.gemm_full(A, 0, 0, sa, B, 0, 0, sb)
    s0 = delayed_like_scale(y_ref, fd)
    for sd in (s0 * 16, s0 * 2.0 ** -20):
        Dq, amax, st = run(q, A, 0, sa, B, 0, sb, fd, sd)
        check(Dq, amax, y_ref, mag, fd, sd)
    maxcode = oracle.maxcode(fd)
    Dq, _, _ = run(q, A, 0, sa, B, 0, sb, fd, s0 * 16)
    assert ((Dq & 0x7F) == maxcode).sum() > 0


def test_amax_accumulates_and_is_optional_and_ld(q):
    rng = np.random.default_rng(3)
    A, B = realistic_codes(rng, (256, 128), 0), realistic_codes(rng, (512, 128), 0)
    sa = sb = np.array([2.0 ** -7], np.float32)
    y_ref, mag = oracle.gemm_full(A, 0, 0, sa, B, 0, 0, sb)
    sd = delayed_like_scale(y_ref, 0)
    _, amax, _ = run(q, A, 0, sa, B, 0, sb, 0, sd, amax0=1e30)
    assert amax == np.float32(1e30)
    Dq, amax, st = run(q, A, 0, sa, B, 0, sb, 0, sd, amax0=-5.0, with_amax=False, ldd=576)
    assert st == 0 and amax == -5.0
    assert (Dq[:, 512:] == 0xAB).all()  # the padding beyond N is not written
    check(Dq[:, :512], float(np.abs(y_ref).max()), y_ref, mag, 0, sd)


def test_k_zero_writes_zero_codes(q):
    A = np.zeros((64, 0), np.uint8)
    B = np.zeros((32, 0), np.uint8)
    one = np.array([1.0], np.float32)
    Dq, amax, st = run(q, A, 0, one, B, 0, one, 0, 1.0, amax0=2.5)
    assert st == 0 and not Dq.any() and amax == 2.5
