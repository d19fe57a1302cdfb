"""Tensors past 2^31 elements (64-bit index paths): a 65536 x 32768 cast (4 GB of bf16) and GEMM
outputs of 65536 x 40960 (2.7 G elements), checked on sampled rows, columns and outputs against
the oracle.  The large input is a seeded 2048 x 32768 tile repeated 32 times down the rows, so the
oracle needs only the tile."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_codes_equal, assert_gemm_close, bf16_out_to_f64, dev_bf16, host, require_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TR, C, REP = 2048, 32768, 32  # 65536 x 32768 = 2^31 elements


@pytest.fixture(scope="module")
def big():
    q = require_gpu()
    tile = wl.random_bf16(404, TR, C, "t3", 0.5)
    x = dev_bf16(tile).repeat(REP, 1)
    assert x.shape == (TR * REP, C) and x.numel() == 1 << 31
    return q, tile, x


def test_per_tensor_cast_2g_elements(big):
    q, tile, x = big
    R = TR * REP
    amax = torch.zeros(1, device="cuda")
    q.fp8_amax(x, amax)
    assert host(amax)[0] == oracle.amax(tile)
    _, s, _ = oracle.scale_triple(oracle.amax(tile), 0)
    qr = torch.empty(R, C, dtype=torch.uint8, device="cuda")
    qc = torch.empty(C, R, dtype=torch.uint8, device="cuda")
    q.fp8_quantize(x, q.E4M3, q.TENSOR, scale=torch.tensor([s], device="cuda"), q_row=qr, q_col=qc)
    ref_r, ref_c = oracle.quantize_tensor(tile, 0, s, row=True, col=True)
    for r in (0, 1, R // 2 + 7, R - 1):  # rows in the first and last 2^31 bytes of the outputs
        assert_codes_equal(host(qr[r]), ref_r[r % TR], 0, f"row {r}")
    for c in (0, 5, C // 2 + 3, C - 1):
        assert_codes_equal(host(qc[c]), np.tile(ref_c[c], REP), 0, f"col {c}")
    del qr, qc


def test_mx_cast_2g_elements(big):
    q, tile, x = big
    R = TR * REP
    qr = torch.empty(R, C, dtype=torch.uint8, device="cuda")
    sr = torch.empty(R, C // 32, dtype=torch.uint8, device="cuda")
    qc = torch.empty(C, R, dtype=torch.uint8, device="cuda")
    sc = torch.empty(C, R // 32, dtype=torch.uint8, device="cuda")
    q.fp8_quantize(x, q.E4M3, q.MX_1x32, q_row=qr, q_col=qc, sf_row=sr, sf_col=sc)
    rr, rsr, rc, rsc, _ = oracle.quantize_block(tile, 0, 3, 0, row=True, col=True)
    for r in (3, R // 2, R - 1):
        assert_codes_equal(host(qr[r]), rr[r % TR], 0, f"row {r}")
        assert np.array_equal(host(sr[r]), rsr[r % TR])
    for c in (0, C // 3, C - 1):
        assert_codes_equal(host(qc[c]), np.tile(rc[c], REP), 0, f"col {c}")
        assert np.array_equal(host(sc[c]), np.tile(rsc[c], REP))
    del qr, qc, sr, sc


@pytest.mark.parametrize("mx", [False, True])
def test_gemm_output_past_2g_elements(mx):
    q = require_gpu()
    M, N, K = 65536, 40960, 256
    rng = np.random.default_rng(77 + mx)
    A = oracle.encode_array((rng.standard_normal((M, K)) * 60).astype(np.float32), 0)
    B = oracle.encode_array((rng.standard_normal((N, K)) * 60).astype(np.float32), 0)
    if mx:
        sa = rng.integers(118, 128, (M, K // 32)).astype(np.uint8)
        sb = rng.integers(118, 128, (N, K // 32)).astype(np.uint8)
        ga = gb = q.MX_1x32
    else:
        sa, sb = np.array([2.0 ** -6], np.float32), np.array([2.0 ** -5], np.float32)
        ga = gb = q.TENSOR
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q.fp8_scaled_gemm(q.FPROP, dev(A), 0, ga, dev(sa), dev(B), 0, gb, dev(sb), D, status=status)
    rng2 = np.random.default_rng(5)
    ms = np.concatenate([[0, M - 1, M - 1, M // 2], rng2.integers(0, M, 3000)]).astype(np.int64)
    ns = np.concatenate([[0, N - 1, 0, N // 2 + 1], rng2.integers(0, N, 3000)]).astype(np.int64)
    y_ref, mag = oracle.gemm_sample(A, 0, 3 if mx else 0, sa, B, 0, 3 if mx else 0, sb, ms, ns)
    y = D[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()].double().cpu().numpy()
    assert int(host(status)[0]) == 0
    assert_gemm_close(y, y_ref, mag, True)
    del D


def test_cast_stats_past_the_counter_fold():
    """2^34 elements (34 GB of bf16): every thread of the statistics kernel runs more than the 2048
    steps after which it folds its packed 16-bit lane counters into the CTA's counts.  The tensor is a
    4-row tile (a saturating row, a row that flushes at the small scales, zeros, the negated second
    row) repeated down the rows, so the exact counts are the oracle's on the tile times the repeats."""
    q = require_gpu()
    C, reps = 32768, 1 << 17
    a, b = (int(v) for v in wl.bf16_bits(np.array([60000.0, 2.0 ** -18], np.float32)))
    tile = np.zeros((4, C), np.uint16)
    tile[0], tile[1], tile[3] = a, b, b | 0x8000
    tile[0, ::7] = b  # rows that mix both kinds of element
    x = dev_bf16(tile).repeat(reps, 1)
    assert x.numel() == 1 << 34
    for scales in ([2.0 ** e for e in range(-3, 4)], [2.0 ** e for e in (-1, 0, 1, 2)], [1.0, 4.0]):
        sc = torch.tensor(np.asarray(scales, np.float32), device="cuda")
        sat = torch.zeros(len(scales), dtype=torch.int64, device="cuda")
        und = torch.zeros(len(scales), dtype=torch.int64, device="cuda")
        q.fp8_cast_stats(x, q.E5M2, sc, sat, und)
        ref_s, ref_u = oracle.cast_stats(tile, 1, scales)
        assert np.array_equal(host(sat).astype(np.uint64), ref_s * np.uint64(reps)), scales
        assert np.array_equal(host(und).astype(np.uint64), ref_u * np.uint64(reps)), scales
    del x
