"""GPU parity of the fused current-scaling cast (fp8_quantize_current) against the oracle.

amax, bias, scale, scale_inv and every code must be bit-exact with the oracle's
amax -> compute_bias -> per-tensor cast, the same result as the three separate
entry points give."""
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


class Out:
    def __init__(self, r, c, row=True, col=True):
        u8 = dict(dtype=torch.uint8, device="cuda")
        self.qr = torch.full((r, c), 0xAB, **u8) if row else None
        self.qc = torch.full((c, r), 0xAB, **u8) if col else None
        self.amax = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        self.bias = torch.full((1,), 999, dtype=torch.int32, device="cuda")
        self.scale = torch.zeros(1, dtype=torch.float32, device="cuda")
        self.scale_inv = torch.zeros(1, dtype=torch.float32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(self, q, x, fmt, margin, ws):
        q.fp8_quantize_current(x, fmt, margin, ws, q_row=self.qr, q_col=self.qc, amax=self.amax, bias=self.bias,
                               scale=self.scale, scale_inv=self.scale_inv, status=self.status)


def check(o: Out, x_bits: np.ndarray, fmt: int, margin: int):
    amax = oracle.amax(x_bits)
    e, s, si = oracle.scale_triple(amax, fmt, margin)
    assert host(o.amax)[0] == amax
    assert host(o.bias)[0] == e and host(o.scale)[0] == s and host(o.scale_inv)[0] == si
    assert host(o.status)[0] == 0
    rr, rc = oracle.quantize_tensor(x_bits, fmt, s, row=o.qr is not None, col=o.qc is not None)
    if o.qr is not None:
        assert_codes_equal(host(o.qr), rr, fmt, "row")
    if o.qc is not None:
        assert_codes_equal(host(o.qc), rc, fmt, "col")


SHAPES = [(16, 8), (48, 136), (144, 264), (256, 1024), (272, 520), (1040, 96)]


@pytest.mark.parametrize("fmt,margin", [(0, 0), (1, 1), (0, -2)])
@pytest.mark.parametrize("shape", SHAPES)
def test_parity(q, shape, fmt, margin):
    r, c = shape
    kind = ["normal", "t3", "wide", "laplace"][(r + c) % 4]
    x = wl.random_bf16(3000 + r + c + fmt, r, c, kind, 0.5)
    ws = q.current_workspace()
    o = Out(r, c)
    o.run(q, dev_bf16(x), fmt, margin, ws)
    check(o, x, fmt, margin)


def test_ld_row_only_col_only(q):
    r, c, ld = 160, 392, 520
    full = wl.random_bf16(91, r, ld, "t3", 2.0)
    x = dev_bf16(full)[:, :c]
    xb = np.ascontiguousarray(full[:, :c])
    ws = q.current_workspace()
    for row, col in ((True, False), (False, True)):
        o = Out(r, c, row, col)
        o.run(q, x, 0, 0, ws)
        check(o, xb, 0, 0)


def test_many_ctas_and_repeated_calls_share_a_workspace(q):
    """4096 x 4096 has 1024 tiles, more than one CTA per SM can hold at once: the grid is the
    resident maximum and the barrier spans it.  Ten calls in a row on one workspace, each on a
    tensor with a different amax, check that it resets itself."""
    ws = q.current_workspace()
    o = Out(4096, 4096)
    for t in range(10):
        xb = wl.delayed_activation(t) if t % 2 == 0 else wl.random_bf16(500 + t, 4096, 4096, "laplace", 10.0 ** (t - 5))
        o.run(q, dev_bf16(xb), t % 2, t % 2, ws)
        check(o, xb, t % 2, t % 2)
    hdr = host(ws[:16].view(torch.int32))
    assert hdr[0] == 0  # arrival count back to zero
    assert hdr[1] == 10  # one barrier generation per call
    assert hdr[3] == 0  # the running max (the CTAs' atomic max) zeroed for the next call


def test_matches_the_three_call_path(q):
    """Same result as fp8_amax + fp8_compute_scale + fp8_quantize (1x linear forward activation)."""
    Xb, _ = wl.linear_fwd_current()
    x = dev_bf16(Xb)
    r, c = Xb.shape
    o = Out(r, c)
    o.run(q, x, 0, 0, q.current_workspace())
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    bias = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = torch.zeros(1, dtype=torch.float32, device="cuda")
    si = torch.zeros(1, dtype=torch.float32, device="cuda")
    q.fp8_amax(x, amax)
    q.fp8_compute_scale(amax, 0, 0, bias, scale, si)
    qr = torch.empty(r, c, dtype=torch.uint8, device="cuda")
    qc = torch.empty(c, r, dtype=torch.uint8, device="cuda")
    q.fp8_quantize(x, 0, q.TENSOR, scale=scale, q_row=qr, q_col=qc)
    assert host(o.bias)[0] == host(bias)[0] == 3
    assert host(o.amax)[0] == host(amax)[0] and host(o.scale_inv)[0] == host(si)[0]
    assert np.array_equal(host(o.qr), host(qr)) and np.array_equal(host(o.qc), host(qc))
    check(o, Xb, 0, 0)


def test_nan_zero_and_empty(q):
    ws = q.current_workspace()
    xb = wl.random_bf16(7, 128, 256, "normal")
    xb[100, 3] = 0x7FC0
    o = Out(128, 256)
    o.run(q, dev_bf16(xb), 0, 0, ws)
    assert np.isnan(host(o.amax)[0]) and host(o.bias)[0] == 0 and host(o.scale)[0] == 1.0
    assert host(o.status)[0] & q.STATUS_NONFINITE_AMAX
    z = wl.random_bf16(0, 128, 256, "zeros")
    o = Out(128, 256)
    o.run(q, dev_bf16(z), 1, 0, ws)
    check(o, z, 1, 0)
    assert not host(o.qr).any()
    o = Out(0, 64, row=True, col=False)
    o.run(q, torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"), 0, 0, ws)
    assert host(o.amax)[0] == 0 and host(o.bias)[0] == 0 and host(o.scale)[0] == 1 and host(o.scale_inv)[0] == 1
