"""GPU parity at the full workload sizes, through the same step objects bench.py times.

Quantisation outputs (codes, scales, amax, bias, history) are compared bit for
bit over the whole tensors; GEMM outputs on sampled coordinates (four corner
blocks plus 4096 seeded random elements) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_codes_equal, assert_gemm_close, dev_bf16, host, require_gpu, sample_coords

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return require_gpu()


def sampled(D: torch.Tensor, ms, ns) -> np.ndarray:
    idx_m = torch.from_numpy(ms).cuda()
    idx_n = torch.from_numpy(ns).cuda()
    return D[idx_m, idx_n].double().cpu().numpy()


def test_linear_fwd_current_scaling(q):
    """X 256x1024 (N(0, 0.02^2) + eight +-30 outliers), W 1024x1024, E4M3, margin 0, fp32 Y."""
    from scaling_quantization_gemm_gb300.step import PerTensorFwd
    Xb, Wb = wl.linear_fwd_current()
    f = PerTensorFwd(dev_bf16(Xb), dev_bf16(Wb))
    f.run()
    torch.cuda.synchronize()
    assert host(f.sx.bias)[0] == 3  # closed form: amax = 30
    ex, sx, ix = oracle.scale_triple(oracle.amax(Xb), 0)
    ew, sw, iw = oracle.scale_triple(oracle.amax(Wb), 0)
    assert host(f.sw.bias)[0] == ew and host(f.sx.scale_inv)[0] == ix and host(f.sw.scale_inv)[0] == iw
    qx, _ = oracle.quantize_tensor(Xb, 0, sx)
    qw, _ = oracle.quantize_tensor(Wb, 0, sw)
    assert_codes_equal(host(f.qx), qx, 0, "QX")
    assert_codes_equal(host(f.qw), qw, 0, "QW")
    y_ref, mag = oracle.gemm_full(qx, 0, 0, ix, qw, 0, 0, iw)
    assert_gemm_close(host(f.Y).astype(np.float64), y_ref, mag, False)


def test_delayed_scaling_16_iterations(q):
    """Activation 4096x4096 N(0,1)(1+0.1t), E4M3 margin 0; gradient Laplace(0,1e-4), E5M2 margin 1;
    history 16.  Iteration 0 scales from its own amax (empty history).  Codes, amax, history and
    the per-iteration saturated / flushed-to-zero counts are exact."""
    from scaling_quantization_gemm_gb300.step import ScaleState, current_scaling
    L = 16
    sa, sg = ScaleState(0, 0, L), ScaleState(1, 1, L)
    ra, rg = oracle.HistoryState(L), oracle.HistoryState(L)
    qa = torch.empty(4096, 4096, dtype=torch.uint8, device="cuda")
    qg = torch.empty_like(qa)
    latest_is_max = []
    for t in range(16):
        xa, xg = wl.delayed_activation(t), wl.delayed_gradient(t)
        da, dg = dev_bf16(xa), dev_bf16(xg)
        saturated, underflow = {}, {}
        for d, st, out in ((da, sa, qa), (dg, sg, qg)):
            if t == 0:
                current_scaling(d, st)
            q.fp8_quantize(d, st.fmt, q.TENSOR, scale=st.scale, q_row=out, amax=st.amax)
            cnt = torch.zeros(2, dtype=torch.int64, device="cuda")
            q.fp8_cast_stats(d, st.fmt, st.scale, cnt[0:1], cnt[1:2])
            saturated[st.fmt], underflow[st.fmt] = (int(v) for v in host(cnt))
        got_amax = (host(sa.amax)[0], host(sg.amax)[0])
        ga, gg = host(qa), host(qg)
        for x, st, ref, g, fmt, margin, am in ((xa, sa, ra, ga, 0, 0, got_amax[0]),
                                               (xg, sg, rg, gg, 1, 1, got_amax[1])):
            amax = oracle.amax(x)
            assert am == amax, t
            scale = oracle.scale_triple(amax, fmt, margin)[1] if t == 0 else ref.scale[0]
            codes, _ = oracle.quantize_tensor(x, fmt, scale)
            assert_codes_equal(g, codes, fmt, f"iteration {t}")
            # saturated and flushed counts of this iteration's cast, exact
            sat_ref, und_ref = oracle.cast_stats(x, fmt, [scale])
            assert (saturated[fmt], underflow[fmt]) == (int(sat_ref[0]), int(und_ref[0])), t
            ref.update(float(amax), fmt, margin)
            st.advance()
            assert host(st.bias)[0] == ref.bias[0] and host(st.scale)[0] == ref.scale[0]
            assert np.array_equal(host(st.history), ref.hist)
        latest_is_max.append(bool(ra.hist[t] == ra.hist[: t + 1].max()))
    # the activation grows by 10 % per iteration: record whether the window max was the newest amax
    print("activation window max == latest amax per iteration:", latest_is_max)


def _block_fwd_check(q, X, W, mx, col, seed):
    from scaling_quantization_gemm_gb300.step import BlockLinearFwd
    f = BlockLinearFwd(dev_bf16(X), dev_bf16(W), mx=mx, col=col)
    f.run()
    torch.cuda.synchronize()
    gx, gw = (3, 3) if mx else (1, 2)
    rx, sxr, cx, sxc, _ = oracle.quantize_block(X, 0, gx, 0, row=True, col=col)
    rw, swr, cw, swc, _ = oracle.quantize_block(W, 0, gw, 0, row=True, col=col)
    assert_codes_equal(host(f.qx_row), rx, 0, "X row")
    assert_codes_equal(host(f.qw_row), rw, 0, "W row")
    assert np.array_equal(host(f.sx_row), sxr) and np.array_equal(host(f.sw_row), swr)
    if col:
        assert_codes_equal(host(f.qx_col), cx, 0, "X col")
        assert_codes_equal(host(f.qw_col), cw, 0, "W col")
        assert np.array_equal(host(f.sx_col), sxc) and np.array_equal(host(f.sw_col), swc)
    assert host(f.status)[0] == 0
    M, N = X.shape[0], W.shape[0]
    ms, ns = sample_coords(M, N, seed)
    y_ref, mag = oracle.gemm_sample(rx, 0, gx, sxr, rw, 0, gw, swr, ms, ns)
    assert_gemm_close(sampled(f.Y, ms, ns), y_ref, mag, True)


def test_per_block_llama2_7b_up_proj(q):
    """X 8192x4096 (0.5 Student-t(3)) 1x128 blocks, W 11008x4096 N(0, 0.02^2) 128x128 blocks, bf16 Y."""
    X, W = wl.per_block_up_proj()
    _block_fwd_check(q, X, W, mx=False, col=False, seed=3)


def test_mxfp8_row_and_col(q):
    """X 16384x8192 (N(0,1), 0.1% x100), W 28672x8192 N(0, 0.01^2); 1x32 E8M0, row- and column-wise;
    block-scaled GEMM M=16384 N=28672 K=8192, bf16 Y."""
    X, W = wl.mxfp8_inputs()
    _block_fwd_check(q, X, W, mx=True, col=True, seed=4)


def test_ffn_fwd_bwd_delayed(q):
    """X 16384x5120, W 20480x5120 (E4M3), dY 16384x20480 (E5M2), delayed scaling L=1024: two steps
    (the first scales from its own amax), all casts bit-exact, fprop/dgrad/wgrad sampled."""
    from scaling_quantization_gemm_gb300.step import LinearFwdBwd
    X, W, dY = wl.ffn_fwd_bwd()
    f = LinearFwdBwd(dev_bf16(X), dev_bf16(W), dev_bf16(dY), history_len=1024)
    refs = {k: oracle.HistoryState(1024) for k in "xwg"}
    amax = {"x": oracle.amax(X), "w": oracle.amax(W), "g": oracle.amax(dY)}
    fmts = {"x": 0, "w": 0, "g": 1}
    for _ in range(2):
        f.run()
        torch.cuda.synchronize()
        for k in "xwg":
            refs[k].update(float(amax[k]), fmts[k], 0)
    scale = {k: oracle.scale_triple(amax[k], fmts[k])[1:] for k in "xwg"}  # same tensors each step
    for k, st in (("x", f.sx), ("w", f.sw), ("g", f.sg)):
        assert host(st.bias)[0] == refs[k].bias[0] and host(st.pos)[0] == 2
        assert np.array_equal(host(st.history), refs[k].hist)
        assert host(st.scale_inv)[0] == scale[k][1]
    qx_r, qx_c = oracle.quantize_tensor(X, 0, scale["x"][0], row=True, col=True)
    qw_r, qw_c = oracle.quantize_tensor(W, 0, scale["w"][0], row=True, col=True)
    qg_r, qg_c = oracle.quantize_tensor(dY, 1, scale["g"][0], row=True, col=True)
    for got, ref, fmt, name in ((f.qx_row, qx_r, 0, "X row"), (f.qx_col, qx_c, 0, "X col"),
                                (f.qw_row, qw_r, 0, "W row"), (f.qw_col, qw_c, 0, "W col"),
                                (f.qg_row, qg_r, 1, "dY row"), (f.qg_col, qg_c, 1, "dY col")):
        assert_codes_equal(host(got), ref, fmt, name)
    ix, iw, ig = scale["x"][1], scale["w"][1], scale["g"][1]
    for D, A, fa, ia, B, fb, ib, bf16, seed in ((f.Y, qx_r, 0, ix, qw_r, 0, iw, True, 5),
                                                 (f.dX, qg_r, 1, ig, qw_c, 0, iw, True, 6),
                                                 (f.dW, qg_c, 1, ig, qx_c, 0, ix, False, 7)):
        ms, ns = sample_coords(D.shape[0], D.shape[1], seed)
        y_ref, mag = oracle.gemm_sample(A, fa, 0, ia, B, fb, 0, ib, ms, ns)
        assert_gemm_close(sampled(D, ms, ns), y_ref, mag, bf16)
