"""GPU parity of the fp32 cast (fp8_quantize_f32) against the oracle: every one of the 2^32 fp32
bit patterns at scale 1 in both formats (NaN compared by class), arbitrary and power-of-two scales
on ragged lengths, and the fused amax."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_codes_equal, host, require_gpu

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


@pytest.fixture(scope="module")
def q():
    return require_gpu()


@pytest.mark.parametrize("fmt", [0, 1])
def test_every_fp32_pattern(q, fmt):
    x_dev = torch.empty(CHUNK, dtype=torch.float32, device="cuda")
    q_dev = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    bits = np.arange(CHUNK, dtype=np.uint32)
    for k in range(1 << 32 >> 28):
        x = (bits + np.uint32(k * CHUNK)).view(np.float32)
        x_dev.copy_(torch.from_numpy(x))
        q.fp8_quantize_f32(x_dev, fmt, q_dev)
        assert_codes_equal(host(q_dev), oracle.quantize_f32(x, fmt), fmt, f"patterns {k * CHUNK:#x}..")


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("n", [1, 7, 8, 4099, 1_000_003])
@pytest.mark.parametrize("scale", [None, 2.0 ** 5, 2.0 ** -20, 0.7071, 3.3e3])
def test_scaled_ragged(q, fmt, n, scale):
    rng = np.random.default_rng(n + fmt)
    x = (np.exp2(rng.uniform(-30, 30, n)) * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    qd = torch.full((n,), 0xAA, dtype=torch.uint8, device="cuda")
    sd = None if scale is None else torch.tensor([scale], dtype=torch.float32, device="cuda")
    q.fp8_quantize_f32(xd, fmt, qd, scale=sd)
    ref = oracle.quantize_f32(x, fmt, 1.0 if scale is None else scale)
    assert_codes_equal(host(qd), ref, fmt)


def test_amax_fused(q):
    rng = np.random.default_rng(9)
    x = rng.standard_normal(3_000_001).astype(np.float32)
    x[1234] = -77.5
    xd = torch.from_numpy(x).cuda()
    qd = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, device="cuda")
    q.fp8_quantize_f32(xd, 0, qd, amax=amax)
    assert host(amax)[0] == oracle.amax_f32(x) == np.float32(77.5)
    q.fp8_quantize_f32(xd[:5].clone(), 0, qd[:5], amax=amax)  # accumulated: stays 77.5
    assert host(amax)[0] == np.float32(77.5)
    x[2_999_999] = np.nan  # in the ragged tail
    q.fp8_quantize_f32(torch.from_numpy(x).cuda(), 0, qd, amax=amax)
    assert np.isnan(host(amax)[0]) and np.isnan(oracle.amax_f32(x))


def test_empty(q):
    x = torch.empty(0, dtype=torch.float32, device="cuda")
    q.fp8_quantize_f32(x, 0, torch.empty(0, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
