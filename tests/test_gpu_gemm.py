"""GPU parity: the scaled FP8 GEMM (tcgen05) against the fp64 oracle.

Every element must satisfy |y - y_ref| <= 1e-3 sum_k |a_k b_k| (plus half a
bf16 ulp of y_ref when the output is bf16)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_gemm_close, bf16_out_to_f64, host, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return require_gpu()


def finite_codes(rng, shape, fmt):
    """Seeded random FP8 codes, NaN/Inf codes replaced by 1.0."""
    c = rng.integers(0, 256, shape).astype(np.uint8)
    if fmt == 0:
        c[(c & 0x7F) == 0x7F] = 0x38
    else:
        c[(c & 0x7C) == 0x7C] = 0x3C
    return c


def realistic_codes(rng, shape, fmt):
    """Codes of quantised Gaussian data (most mass at mid exponents, like real operands)."""
    v = (rng.standard_normal(shape) * (100.0 if fmt == 0 else 8000.0)).astype(np.float32)
    return oracle.encode_array(v, fmt)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gemm(q, A, fa, ga, sfa, B, fb, gb, sfb, out_bf16, op=0):
    M, N = A.shape[0], B.shape[0]
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16 if out_bf16 else torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.fp8_scaled_gemm(op, _dev(A), fa, ga, _dev(sfa), _dev(B), fb, gb, _dev(sfb), D, status=status)
    y = bf16_out_to_f64(D) if out_bf16 else host(D).astype(np.float64)
    return y, int(host(status)[0])


TENSOR_SHAPES = [(128, 256, 128), (256, 512, 1024), (200, 272, 160), (1, 16, 16), (384, 768, 2048),
                 (130, 1040, 4096), (512, 256, 64)]


@pytest.mark.parametrize("M,N,K", TENSOR_SHAPES)
@pytest.mark.parametrize("fa,fb,out_bf16", [(0, 0, False), (1, 0, True), (0, 0, True)])
def test_gemm_per_tensor(q, M, N, K, fa, fb, out_bf16):
    rng = np.random.default_rng(M * 7 + N * 3 + K + fa)
    A = realistic_codes(rng, (M, K), fa)
    B = realistic_codes(rng, (N, K), fb)
    sa = np.array([2.0 ** -5], np.float32)
    sb = np.array([2.0 ** 3], np.float32)
    y, st = run_gemm(q, A, fa, 0, sa, B, fb, 0, sb, out_bf16)
    assert st == 0
    y_ref, mag = oracle.gemm_full(A, fa, 0, sa, B, fb, 0, sb)
    assert_gemm_close(y, y_ref, mag, out_bf16)


def test_gemm_random_codes_full_range(q):
    """Every finite code (subnormals, max magnitude) as operands."""
    rng = np.random.default_rng(5)
    A, B = finite_codes(rng, (256, 512), 0), finite_codes(rng, (256, 512), 1)
    sa, sb = np.array([2.0 ** -9], np.float32), np.array([2.0 ** -14], np.float32)
    y, st = run_gemm(q, A, 0, 0, sa, B, 1, 0, sb, False)
    y_ref, mag = oracle.gemm_full(A, 0, 0, sa, B, 1, 0, sb)
    assert st == 0
    assert_gemm_close(y, y_ref, mag, False)


def test_gemm_identity_weight_is_exact(q):
    """B = I (1.0 codes) with sb = 2^4: fp32 D equals deq(A) * 2^4 bit for bit."""
    rng = np.random.default_rng(1)
    K = 256
    A = finite_codes(rng, (384, K), 0)
    B = np.zeros((K, K), np.uint8)
    np.fill_diagonal(B, 0x38)
    sa, sb = np.array([2.0 ** -6], np.float32), np.array([16.0], np.float32)
    y, _ = run_gemm(q, A, 0, 0, sa, B, 0, 0, sb, False)
    assert np.array_equal(y, oracle.decode_array(A, 0) * 2.0 ** -6 * 16.0)


def test_gemm_k_zero_writes_zeros(q):
    A = np.zeros((64, 0), np.uint8)
    D = torch.full((64, 32), 7.0, device="cuda")
    q.fp8_scaled_gemm(0, torch.empty(64, 0, dtype=torch.uint8, device="cuda"), 0, 0,
                      torch.ones(1, device="cuda"), torch.empty(32, 0, dtype=torch.uint8, device="cuda"), 0, 0,
                      torch.ones(1, device="cuda"), D)
    assert not host(D).any()
    del A


def test_gemm_ops_and_ld(q):
    """Strided operands (lda > K) and output (ldd > N); DGRAD/WGRAD labels run the same TN product."""
    rng = np.random.default_rng(3)
    M, N, K, pad = 256, 256, 384, 64
    A = realistic_codes(rng, (M, K + pad), 0)
    B = realistic_codes(rng, (N, K + pad), 0)
    Ad, Bd = _dev(A)[:, :K], _dev(B)[:, :K]
    sa = torch.tensor([0.5], device="cuda")
    sb = torch.tensor([0.25], device="cuda")
    y_ref, mag = oracle.gemm_full(A[:, :K], 0, 0, np.float32(0.5), B[:, :K], 0, 0, np.float32(0.25))
    for op in (q.FPROP, q.DGRAD, q.WGRAD):
        Dfull = torch.zeros(M, N + 32, dtype=torch.float32, device="cuda")
        D = Dfull[:, :N]
        q.fp8_scaled_gemm(op, Ad, 0, 0, sa, Bd, 0, 0, sb, D)
        assert_gemm_close(host(D).astype(np.float64), y_ref, mag, False)
        assert not host(Dfull)[:, N:].any(), "wrote past N"


# ------------------------------------------------------------- block-scaled

def mx_scales(rng, rows, K):
    return rng.integers(118, 137, (rows, K // 32)).astype(np.uint8)


def pow2_scales(rng, shape):
    return np.ldexp(np.float32(1), rng.integers(-10, 10, shape)).astype(np.float32)


BS_SHAPES = [(128, 256, 128), (256, 512, 512), (200, 272, 384), (384, 1024, 1024), (128, 256, 2048),
             (520, 784, 2048), (384, 480, 1536)]


@pytest.mark.parametrize("M,N,K", BS_SHAPES)
@pytest.mark.parametrize("out_bf16", [False, True])
def test_gemm_mx(q, M, N, K, out_bf16):
    rng = np.random.default_rng(M + N + K)
    A, B = realistic_codes(rng, (M, K), 0), realistic_codes(rng, (N, K), 0)
    sfa, sfb = mx_scales(rng, M, K), mx_scales(rng, N, K)
    y, st = run_gemm(q, A, 0, q.MX_1x32, sfa, B, 0, q.MX_1x32, sfb, out_bf16)
    assert st == 0
    y_ref, mag = oracle.gemm_full(A, 0, 3, sfa, B, 0, 3, sfb)
    assert_gemm_close(y, y_ref, mag, out_bf16)


@pytest.mark.parametrize("M,N,K", BS_SHAPES)
@pytest.mark.parametrize("gb", [1, 2])
def test_gemm_block(q, M, N, K, gb):
    rng = np.random.default_rng(M + N + K + gb)
    A, B = realistic_codes(rng, (M, K), 0), realistic_codes(rng, (N, K), 0)
    sfa = pow2_scales(rng, (M, K // 128))
    sfb = pow2_scales(rng, (N, K // 128) if gb == 1 else (-(-N // 128), K // 128))
    y, st = run_gemm(q, A, 0, 1, sfa, B, 0, gb, sfb, True)
    assert st == 0
    y_ref, mag = oracle.gemm_full(A, 0, 1, sfa, B, 0, gb, sfb)
    assert_gemm_close(y, y_ref, mag, True)


def test_gemm_mx_e5m2_a(q):
    rng = np.random.default_rng(11)
    M, N, K = 256, 256, 512
    A, B = realistic_codes(rng, (M, K), 1), realistic_codes(rng, (N, K), 0)
    sfa, sfb = mx_scales(rng, M, K), mx_scales(rng, N, K)
    y, st = run_gemm(q, A, 1, 3, sfa, B, 0, 3, sfb, False)
    y_ref, mag = oracle.gemm_full(A, 1, 3, sfa, B, 0, 3, sfb)
    assert st == 0
    assert_gemm_close(y, y_ref, mag, False)


def test_gemm_block_equal_scales_match_per_tensor(q):
    rng = np.random.default_rng(2)
    M, N, K = 256, 512, 512
    A, B = realistic_codes(rng, (M, K), 0), realistic_codes(rng, (N, K), 0)
    yt, _ = run_gemm(q, A, 0, 0, np.array([0.25], np.float32), B, 0, 0, np.array([2.0], np.float32), False)
    ym, _ = run_gemm(q, A, 0, 3, np.full((M, K // 32), 125, np.uint8), B, 0, 3, np.full((N, K // 32), 128, np.uint8),
                     False)
    y_ref, mag = oracle.gemm_full(A, 0, 0, np.float32(0.25), B, 0, 0, np.float32(2.0))
    assert_gemm_close(yt, y_ref, mag, False)
    assert_gemm_close(ym, y_ref, mag, False)


def test_gemm_bad_block_scale_sets_status(q):
    rng = np.random.default_rng(4)
    M, N, K = 128, 256, 256
    A, B = realistic_codes(rng, (M, K), 0), realistic_codes(rng, (N, K), 0)
    sfa = pow2_scales(rng, (M, K // 128))
    sfa[3, 1] = 0.3  # not a power of two
    sfb = pow2_scales(rng, (N // 128 + 1, K // 128))
    _, st = run_gemm(q, A, 0, 1, sfa, B, 0, 2, sfb, True)
    assert st == q.STATUS_BAD_BLOCK_SCALE


@pytest.mark.parametrize("gb", [1, 2])
def test_gemm_block_pair_kernel_edge_scales_and_bad_scale(q, gb):
    """The CTA-pair block-scaled kernel (M > 128, K a multiple of 512) with fp32 block scales at the
    ends of the E8M0 range (2^-127, 2^127) next to ordinary ones in the same rows (they take the
    word-by-word conversion) matches the oracle exactly as usual; a scale that is not a power of two
    raises FP8_STATUS_BAD_BLOCK_SCALE, also when it sits beside valid scales."""
    rng = np.random.default_rng(40 + gb)
    M, N, K = 512, 768, 1024
    A, B = realistic_codes(rng, (M, K), 0), realistic_codes(rng, (N, K), 0)
    sfa = pow2_scales(rng, (M, K // 128))
    sfb = pow2_scales(rng, (N if gb == 1 else N // 128, K // 128))
    sfa[5, 2], sfa[300, 0], sfb[1, 3] = np.float32(2.0 ** -127), np.float32(2.0 ** 127), np.float32(2.0 ** -127)
    A[300, :128] = 0  # the 2^127 block multiplies zeros (any finite product of it would overflow fp32)
    y, st = run_gemm(q, A, 0, 1, sfa, B, 0, gb, sfb, True)
    assert st == 0
    y_ref, mag = oracle.gemm_full(A, 0, 1, sfa, B, 0, gb, sfb)
    assert_gemm_close(y, y_ref, mag, True)
    for bad in (np.float32(0.3), np.float32(-2.0), np.float32(0.0), np.float32(np.inf)):
        s2 = sfa.copy()
        s2[200, 1] = bad
        _, st = run_gemm(q, A, 0, 1, s2, B, 0, gb, sfb, True)
        assert st == q.STATUS_BAD_BLOCK_SCALE, bad


@pytest.mark.parametrize("w,ga,gb", [(32, 1, 2), (48, 1, 1), (112, 3, 3), (192, 1, 2), (208, 1, 2), (16, 3, 3)])
def test_gemm_block_pair_ragged_last_column(q, w, ga, gb):
    """The CTA-pair block-scaled kernel with a last tile column w columns wide (N = 4 x 224 + w) and
    80 pair tiles, more than the grid's pairs (a second, partial round of the persistent loop).
    Every output element is written (D starts as NaN); sampled rows of every tile row, and all the
    rows of the last tile row, match the oracle."""
    rng = np.random.default_rng(60 + w + ga)
    M, N, K = 4096, 4 * 224 + w, 512
    A, B = realistic_codes(rng, (M, K), 0), realistic_codes(rng, (N, K), 0)
    if ga == 3:
        sfa, sfb = mx_scales(rng, M, K), mx_scales(rng, N, K)
    else:
        sfa = pow2_scales(rng, (M, K // 128))
        sfb = pow2_scales(rng, (N if gb == 1 else -(-N // 128), K // 128))
    y, st = run_gemm(q, A, 0, ga, sfa, B, 0, gb, sfb, True)
    assert st == 0
    assert not np.isnan(y).any(), "an output tile was not written"
    rows = np.unique(np.concatenate([np.arange(0, M, 37), np.arange(M - 256, M, 5), [M - 1]]))
    y_ref, mag = oracle.gemm_full(A[rows], 0, ga, sfa[rows], B, 0, gb, sfb)
    assert_gemm_close(y[rows], y_ref, mag, True)


@pytest.mark.parametrize("out_bf16", [False, True])
@pytest.mark.parametrize("offset", [0, 16])
def test_gemm_block_pair_output_pitch_and_offset(q, out_bf16, offset):
    """The CTA-pair block-scaled kernel, whose epilogue writes D with TMA stores of 32 x 32 boxes,
    into a strided D (ldd = N + 64) starting `offset` columns into each padded row, with ragged edges
    (M = 520, N = 784: partial boxes in both directions).  Values match the oracle, and nothing
    outside the N columns of D is written."""
    rng = np.random.default_rng(80 + offset + out_bf16)
    M, N, K = 520, 784, 1024
    A, B = realistic_codes(rng, (M, K), 0), realistic_codes(rng, (N, K), 0)
    sfa, sfb = mx_scales(rng, M, K), mx_scales(rng, N, K)
    dt = torch.bfloat16 if out_bf16 else torch.float32
    Dfull = torch.zeros(M, N + 64, dtype=dt, device="cuda")
    D = Dfull[:, offset:offset + N]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.fp8_scaled_gemm(0, _dev(A), 0, q.MX_1x32, _dev(sfa), _dev(B), 0, q.MX_1x32, _dev(sfb), D, status=status)
    y = bf16_out_to_f64(D) if out_bf16 else host(D).astype(np.float64)
    assert int(host(status)[0]) == 0
    y_ref, mag = oracle.gemm_full(A, 0, 3, sfa, B, 0, 3, sfb)
    assert_gemm_close(y, y_ref, mag, out_bf16)
    full = host(Dfull.float() if out_bf16 else Dfull)
    assert not full[:, :offset].any() and not full[:, offset + N:].any(), "wrote outside D"


@pytest.mark.parametrize("M,N", [(129, 16), (384, 48), (136, 1008), (257, 32)])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_gemm_pair_epilogue_edges(q, M, N, out_bf16):
    """The CTA-pair kernels' TMA-store epilogue at its edges: N narrower than one 32-column box (16) or
    not a multiple of 32, and M just past one 256-row pair tile (129, 257: the second CTA of the last
    pair, or all of its rows but one, outside D), per-tensor and MX, fp32 and bf16 out.  D matches
    the oracle and nothing past the N columns of each row is touched."""
    rng = np.random.default_rng(M * 7 + N + out_bf16)
    K = 512
    A, B = realistic_codes(rng, (M, K), 0), realistic_codes(rng, (N, K), 0)
    dt = torch.bfloat16 if out_bf16 else torch.float32
    for gran in (0, q.MX_1x32):
        Dfull = torch.full((M, N + 32), 7.0, dtype=dt, device="cuda")
        D = Dfull[:, :N]
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if gran == 0:
            sa, sb = np.float32(0.5), np.float32(0.25)
            q.fp8_scaled_gemm(0, _dev(A), 0, 0, torch.tensor([sa], device="cuda"), _dev(B), 0, 0,
                              torch.tensor([sb], device="cuda"), D, status=status)
            y_ref, mag = oracle.gemm_full(A, 0, 0, sa, B, 0, 0, sb)
        else:
            sfa, sfb = mx_scales(rng, M, K), mx_scales(rng, N, K)
            q.fp8_scaled_gemm(0, _dev(A), 0, gran, _dev(sfa), _dev(B), 0, gran, _dev(sfb), D, status=status)
            y_ref, mag = oracle.gemm_full(A, 0, 3, sfa, B, 0, 3, sfb)
        assert int(host(status)[0]) == 0
        y = bf16_out_to_f64(D) if out_bf16 else host(D).astype(np.float64)
        assert_gemm_close(y, y_ref, mag, out_bf16)
        assert (host(Dfull.float())[:, N:] == 7.0).all(), "wrote past N"


@pytest.mark.parametrize("out_bf16", [False, True])
def test_gemm_nan_operand_poisons_its_row_only(q, out_bf16):
    """A NaN code in A makes its output row NaN (the fp64 oracle agrees); every other row is finite
    and within tolerance."""
    rng = np.random.default_rng(12)
    A = realistic_codes(rng, (256, 512), 0)
    B = realistic_codes(rng, (256, 512), 0)
    A[3, 10] = 0x7F  # E4M3 NaN
    sa, sb = np.array([2.0 ** -6], np.float32), np.array([2.0 ** -6], np.float32)
    y, st = run_gemm(q, A, 0, 0, sa, B, 0, 0, sb, out_bf16)
    y_ref, mag = oracle.gemm_full(A, 0, 0, sa, B, 0, 0, sb)
    assert st == 0
    assert np.isnan(y[3]).all() and np.isnan(y_ref[3]).all()
    keep = np.ones(256, bool)
    keep[3] = False
    assert np.isfinite(y[keep]).all()
    assert_gemm_close(y[keep], y_ref[keep], mag[keep], out_bf16)
