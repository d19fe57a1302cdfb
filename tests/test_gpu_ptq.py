"""GPU parity of the post-training-quantised inference stack (two FP8 linear layers, the hidden
activation cast in the first GEMM's epilogue) against the oracle.

Weight and input codes are bit-exact.  The hidden activation comes from a GEMM output known only
to within the GEMM tolerance, so it is checked for validity rather than equality: its recorded
amax must lie within tolerance of max |H_ref| (bounded only from below when a sample of rows is
checked), its scale must be the one compute_bias gives for such an amax, each hidden code must be
the cast of an admissible value (the oracle's bracket), and nearly all codes must equal the cast
of the exact product.  Y is compared with the oracle's product of the oracle's own hidden codes,
on the rows whose hidden codes all equal them."""
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


def _cast_tensor(Xb):
    _, s, si = oracle.scale_triple(oracle.amax(Xb), 0)
    return oracle.quantize_tensor(Xb, 0, s)[0], si


def _check_hidden(hq, sd, amax_h, amax_for_scale, h_ref, tol, via_bf16, all_rows):
    a = np.abs(h_ref)
    assert (a - tol).max() <= amax_h, "hidden amax below the sampled rows' magnitudes"
    if all_rows:  # the upper bound needs every row of H
        assert amax_h <= (a + tol).max(), "hidden amax above tolerance"
    assert sd == oracle.scale_triple(np.float32(amax_for_scale), 0)[1], "hidden scale is not compute_bias(amax)"
    lo, hi, near = oracle.gemm_quantize_bracket(h_ref, tol, 0, sd, via_bf16=via_bf16)
    d, dl, dh, dn = (oracle.decode_array(c, 0) for c in (hq, lo, hi, near))
    bad = ~((dl <= d) & (d <= dh))
    assert not bad.any(), f"{int(bad.sum())} hidden codes outside the bracket"
    assert np.mean(d == dn) >= 0.999
    return near


def _run_and_check(stack, x, Xb, W1b, W2b, rows, steps):
    qw1, iw1 = _cast_tensor(W1b)
    qw2, iw2 = _cast_tensor(W2b)
    qx, ix = _cast_tensor(Xb)
    F = W1b.shape[0]
    ms = np.repeat(rows, F)
    ns = np.tile(np.arange(F), rows.size)
    h_ref, h_mag = oracle.gemm_sample(qx, 0, 0, ix, qw1, 0, 0, iw1, ms, ns)
    h_ref, h_mag = h_ref.reshape(rows.size, F), h_mag.reshape(rows.size, F)
    for step in range(steps):
        stack.forward(x)
        torch.cuda.synchronize()
        assert_codes_equal(host(stack.qw1), qw1, 0, "QW1")
        assert_codes_equal(host(stack.qw2), qw2, 0, "QW2")
        assert_codes_equal(host(stack.qx), qx, 0, "QX")
        # step 0 casts GEMM 1's bf16 output from its own amax (two roundings: bf16, then FP8); later
        # steps cast the fp32 accumulator in the epilogue with the delayed scale (one rounding)
        tol = oracle.gemm_tolerance(h_ref, h_mag, step == 0)
        hist = host(stack.sh.history)
        amax_h = float(hist[step])  # this forward's hidden amax, recorded by the history update
        # the scale this forward cast with: from its own amax at step 0, else from the earlier window
        amax_for_scale = hist[0] if step == 0 else hist[:step].max()
        sd = np.float32(1.0) / host(stack.sh.scale_inv)[0] if step == 0 else sd_next
        hq = host(stack.qh)[rows]
        near = _check_hidden(hq, np.float32(sd), amax_h, amax_for_scale, h_ref, tol, step == 0,
                             rows.size == Xb.shape[0])
        sd_next = np.float32(host(stack.sh.scale)[0])
        # Y on the rows whose hidden codes are all the oracle's nearest codes
        keep = np.where((hq == near).all(axis=1))[0]
        assert keep.size >= 0.8 * rows.size
        H = W2b.shape[0]
        ms2 = np.repeat(np.arange(keep.size), H)
        ns2 = np.tile(np.arange(H), keep.size)
        y_ref, y_mag = oracle.gemm_sample(near[keep], 0, 0, np.float32(1.0) / np.float32(sd), qw2, 0, 0, iw2, ms2, ns2)
        y = bf16_out_to_f64(stack.Y)[rows[keep]]
        assert_gemm_close(y, y_ref.reshape(keep.size, H), y_mag.reshape(keep.size, H), True, f"Y step {step}")
        assert host(stack.sh.status)[0] == 0


@pytest.mark.parametrize("act", ["current", "delayed"])
def test_ptq_stack_small(q, act):
    from scaling_quantization_gemm_gb300.step import PTQStack
    T, H, F = 256, 512, 1024
    Xb, W1b, W2b = wl.ptq_ffn(T, H, F, seed=10)
    stack = PTQStack(dev_bf16(W1b), dev_bf16(W2b), T, act=act, history_len=4)
    _run_and_check(stack, dev_bf16(Xb), Xb, W1b, W2b, np.arange(T), 3)


def test_ptq_stack_13b_ffn_sampled_rows(q):
    """8192 tokens through the 5120 -> 13824 -> 5120 stack; 48 seeded rows checked in full."""
    from scaling_quantization_gemm_gb300.step import PTQStack
    Xb, W1b, W2b = wl.ptq_ffn()
    stack = PTQStack(dev_bf16(W1b), dev_bf16(W2b), Xb.shape[0], act="current")
    rows = np.sort(np.random.default_rng(8).choice(Xb.shape[0], 48, replace=False))
    rows[0], rows[-1] = 0, Xb.shape[0] - 1
    _run_and_check(stack, dev_bf16(Xb), Xb, W1b, W2b, rows, 2)
