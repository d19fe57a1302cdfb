"""GPU parity of the scale rules kept behind options, against the oracle: the OCP MX bias for 1x32
blocks (cast and block-scaled GEMM), the ratio scale s = fmax / amax (scale, fp32-path cast,
GEMM), and a delayed-scaling first step with the fixed bias e = 0."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_codes_equal, assert_gemm_close, bf16_out_to_f64, dev_bf16, host, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return require_gpu()


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shape", [(48, 136), (144, 264), (256, 1024)])
def test_ocp_mx_cast(q, fmt, shape):
    r, c = shape
    x = wl.random_bf16(700 + r + fmt, r, c, "wide", 0.5)
    margin = 1 if fmt else 0
    srow, scol = oracle.scale_shapes(r, c, oracle.MX_1x32_OCP)
    u8 = dict(dtype=torch.uint8, device="cuda")
    qr, qc = torch.empty(r, c, **u8), torch.empty(c, r, **u8)
    sr, sc = torch.empty(srow, **u8), torch.empty(scol, **u8)
    q.fp8_quantize(dev_bf16(x), fmt, q.MX_1x32_OCP, margin, q_row=qr, q_col=qc, sf_row=sr, sf_col=sc)
    rr, rsr, rc, rsc, _ = oracle.quantize_block(x, fmt, oracle.MX_1x32_OCP, margin, row=True, col=True)
    assert_codes_equal(host(qr), rr, fmt, "row")
    assert_codes_equal(host(qc), rc, fmt, "col")
    assert np.array_equal(host(sr), rsr) and np.array_equal(host(sc), rsc)


def test_ocp_mx_forward(q):
    """The MX forward with OCP-rule scales: casts bit-exact, block-scaled GEMM within tolerance."""
    from scaling_quantization_gemm_gb300.step import BlockLinearFwd
    X = wl.random_bf16(71, 512, 1024, "normal")
    W = wl.random_bf16(72, 768, 1024, "normal", 0.02)
    f = BlockLinearFwd(dev_bf16(X), dev_bf16(W), mx=True, mx_rule="ocp")
    f.run()
    torch.cuda.synchronize()
    rx, sx, _, _, _ = oracle.quantize_block(X, 0, oracle.MX_1x32_OCP)
    rw, sw, _, _, _ = oracle.quantize_block(W, 0, oracle.MX_1x32_OCP)
    assert_codes_equal(host(f.qx_row), rx, 0, "X")
    assert_codes_equal(host(f.qw_row), rw, 0, "W")
    assert np.array_equal(host(f.sx_row), sx) and np.array_equal(host(f.sw_row), sw)
    y_ref, mag = oracle.gemm_full(rx, 0, oracle.MX_1x32_OCP, sx, rw, 0, oracle.MX_1x32_OCP, sw)
    assert_gemm_close(bf16_out_to_f64(f.Y), y_ref, mag, True)


def test_ratio_scale_values(q):
    rng = np.random.default_rng(3)
    vals = np.concatenate([np.exp2(rng.uniform(-120, 120, 500)), [0.0, 1.0, 448.0, 30.0, 3e38, 1e-40]]).astype(np.float32)
    a = torch.zeros(1, device="cuda")
    s = torch.zeros(1, device="cuda")
    si = torch.zeros(1, device="cuda")
    for fmt in (0, 1):
        for v in vals:
            a.fill_(float(v))
            q.fp8_compute_scale_ratio(a, fmt, s, si)
            rs, rsi, _ = oracle.scale_ratio(float(v), fmt)
            assert host(s)[0] == rs and host(si)[0] == rsi, (fmt, float(v))


def test_ratio_scale_forward(q):
    """Current scaling with s = fmax / amax: codes equal the oracle's cast at that scale (fp32
    product, then the encoding); the GEMM with the non-power-of-two dequantisation factors is within
    tolerance."""
    from scaling_quantization_gemm_gb300.step import PerTensorFwd
    Xb, Wb = wl.linear_fwd_current()
    f = PerTensorFwd(dev_bf16(Xb), dev_bf16(Wb), scale_rule="ratio")
    f.run()
    torch.cuda.synchronize()
    sx, ix, _ = oracle.scale_ratio(oracle.amax(Xb), 0)
    sw, iw, _ = oracle.scale_ratio(oracle.amax(Wb), 0)
    assert host(f.sx.scale)[0] == sx and host(f.sw.scale_inv)[0] == iw
    qx = oracle.quantize_tensor(Xb, 0, sx)[0]
    qw = oracle.quantize_tensor(Wb, 0, sw)[0]
    assert_codes_equal(host(f.qx), qx, 0, "QX")
    assert_codes_equal(host(f.qw), qw, 0, "QW")
    y_ref, mag = oracle.gemm_full(qx, 0, 0, ix, qw, 0, 0, iw)
    assert_gemm_close(host(f.Y).astype(np.float64), y_ref, mag, False)


def test_fixed_first_step(q):
    """Delayed scaling whose empty-history step uses e = 0 (scale 1): that step's codes are the cast at
    scale 1, its amax is recorded, and the next step scales from the history."""
    from scaling_quantization_gemm_gb300.step import LinearFwdBwd
    X = wl.random_bf16(81, 256, 512, "normal", 100.0)
    W = wl.random_bf16(82, 384, 512, "normal", 0.02)
    dY = wl.random_bf16(83, 256, 384, "laplace", 1e-3)
    f = LinearFwdBwd(dev_bf16(X), dev_bf16(W), dev_bf16(dY), history_len=4, first_step="fixed")
    f.run()
    torch.cuda.synchronize()
    for got, x, fmt in ((f.qx_row, X, 0), (f.qw_row, W, 0), (f.qg_row, dY, 1)):
        assert_codes_equal(host(got), oracle.quantize_tensor(x, fmt, np.float32(1.0))[0], fmt, "first step")
    for st, x, fmt in ((f.sx, X, 0), (f.sw, W, 0), (f.sg, dY, 1)):
        ref = oracle.HistoryState(4)
        ref.update(float(oracle.amax(x)), fmt, 0)
        assert np.array_equal(host(st.history), ref.hist) and host(st.scale)[0] == ref.scale[0]
    f.run()
    torch.cuda.synchronize()
    _, s2, _ = oracle.scale_triple(oracle.amax(X), 0)
    assert_codes_equal(host(f.qx_row), oracle.quantize_tensor(X, 0, s2)[0], 0, "second step")
