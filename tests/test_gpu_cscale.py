"""GPU parity of fixed biases (FP8-CSCALE) and of the cast statistics against the oracle.

Counts are integers and must be exact: the number of elements a scale saturates and the number of
non-zero elements it flushes to zero, for several scales in one pass."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_codes_equal, dev_bf16, host, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return require_gpu()


def gpu_stats(q, x, fmt, scales):
    sc = torch.tensor(np.asarray(scales, np.float32), device="cuda")
    sat = torch.zeros(len(scales), dtype=torch.int64, device="cuda")
    und = torch.zeros(len(scales), dtype=torch.int64, device="cuda")
    q.fp8_cast_stats(x, fmt, sc, sat, und)
    return host(sat).astype(np.uint64), host(und).astype(np.uint64)


def test_set_bias_every_e(q):
    b = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.zeros(1, device="cuda")
    si = torch.zeros(1, device="cuda")
    for e in range(-126, 128):
        q.fp8_set_bias(e, b, s, si)
        assert host(b)[0] == e and host(s)[0] == oracle.pow2f(e) and host(si)[0] == oracle.pow2f(-e)


@pytest.mark.parametrize("fmt", [0, 1])
def test_stats_every_bf16(q, fmt):
    """All 65536 bf16 patterns (NaN, inf, subnormals) at powers of two and at arbitrary scales."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    x = dev_bf16(bits)
    for scales in ([2.0 ** e for e in (-126, -20, -3, 0, 3, 20, 127)],
                   [0.3, 3.7, 1e-3, 1234.5, 0.0, float("inf"), -2.0, float("nan")], [1.0]):
        got = gpu_stats(q, x, fmt, scales)
        ref = oracle.cast_stats(bits, fmt, scales)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), scales


@pytest.mark.parametrize("n", range(1, 9))
def test_stats_every_scale_count(q, n):
    """Each count of scales (1 to 8) has its own kernel instantiation: all 65536 bf16 patterns, the
    first n of a list that mixes powers of two with other scales, both formats."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    x = dev_bf16(bits)
    scales = [2.0 ** -3, 0.7, 2.0 ** 5, 1.0, 2.0 ** -20, 3.0, 2.0 ** 12, 1e-3][:n]
    for fmt in (0, 1):
        got = gpu_stats(q, x, fmt, scales)
        ref = oracle.cast_stats(bits, fmt, scales)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), (fmt, scales)


@pytest.mark.parametrize("shape,ld", [((48, 136), 136), ((130, 264), 280), ((1000, 1024), 1024)])
def test_stats_shapes_and_accumulation(q, shape, ld):
    r, c = shape
    full = wl.random_bf16(r + c, r, ld, "wide")
    xb = np.ascontiguousarray(full[:, :c])
    x = dev_bf16(full)[:, :c]
    scales = [2.0 ** e for e in range(-3, 4)]
    sc = torch.tensor(np.asarray(scales, np.float32), device="cuda")
    sat = torch.zeros(7, dtype=torch.int64, device="cuda")
    und = torch.zeros(7, dtype=torch.int64, device="cuda")
    q.fp8_cast_stats(x, 0, sc, sat, und)
    q.fp8_cast_stats(x, 0, sc, sat, und)  # accumulates
    ref = oracle.cast_stats(xb, 0, scales)
    assert np.array_equal(host(sat).astype(np.uint64), 2 * ref[0])
    assert np.array_equal(host(und).astype(np.uint64), 2 * ref[1])


def test_stats_counts_match_the_cast(q):
    """The counts are what fp8_quantize clips and flushes at that scale."""
    xb = wl.random_bf16(31, 512, 1024, "wide")
    x = dev_bf16(xb)
    out = torch.empty(512, 1024, dtype=torch.uint8, device="cuda")
    for fmt in (0, 1):
        for e in (-2, 0, 5):
            s = float(2.0 ** e)
            q.fp8_quantize(x, fmt, q.TENSOR, scale=torch.tensor([s], device="cuda"), q_row=out)
            codes = host(out)
            sat, und = gpu_stats(q, x, fmt, [s])
            xf = (xb.astype(np.uint32) << 16).view(np.float32)
            assert und[0] == int((((codes & 0x7F) == 0) & (xf != 0)).sum())
            assert sat[0] <= int(((codes & 0x7F) == oracle.maxcode(fmt)).sum())


def test_bias_sweep_harness(q):
    """The sweep over fixed biases e in [-3, 3] on the 13B FFN gradient (Laplace(0, 1e-5), E5M2):
    counts per e equal the oracle's."""
    from scaling_quantization_gemm_gb300.step import bias_sweep
    X = wl.random_bf16(2, 2048, 2048, "laplace", 1e-5)
    res = bias_sweep(dev_bf16(X), q.E5M2, list(range(-3, 4)))
    sat, und = oracle.cast_stats(X, 1, [2.0 ** e for e in range(-3, 4)])
    assert [r["e"] for r in res] == list(range(-3, 4))
    assert [r["saturated"] for r in res] == [int(v) for v in sat]
    assert [r["underflow"] for r in res] == [int(v) for v in und]
    assert all(0.0 <= r["underflow_frac"] <= 1.0 for r in res)
