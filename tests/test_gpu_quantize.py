"""GPU parity: amax, compute_scale, history update and the scaled cast against the CPU oracle.

Codes, scales and amax must be bit-exact (NaN codes by class)."""
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


# ------------------------------------------------------------ exhaustive cast

@pytest.mark.parametrize("fmt", [0, 1])
def test_cast_every_bf16_at_every_scale(q, fmt):
    """All 65536 bf16 bit patterns times every scale 2^e, e in [-126, 127]: every value the
    per-tensor cast can see."""
    x_bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    x = dev_bf16(x_bits)
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    out = torch.empty(512, 128, dtype=torch.uint8, device="cuda")
    gpu = []
    for e in range(-126, 128):
        scale.fill_(float(oracle.pow2f(e)))
        q.fp8_quantize(x, fmt, q.TENSOR, scale=scale, q_row=out)
        gpu.append(host(out).copy())
    for e, g in zip(range(-126, 128), gpu):
        ref, _ = oracle.quantize_tensor(x_bits, fmt, oracle.pow2f(e))
        assert_codes_equal(g, ref, fmt, f"e={e}")


# ----------------------------------------------------------------------- amax

@pytest.mark.parametrize("shape,ld", [((1, 8), 8), ((37, 136), 136), ((130, 264), 280), ((1000, 1024), 1024),
                                      ((4097, 64), 64)])
def test_amax(q, shape, ld):
    r, c = shape
    full = wl.random_bf16(r * 7 + c, r, ld, "t3")
    x = dev_bf16(full)[:, :c]
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    q.fp8_amax(x, amax)
    assert host(amax)[0] == oracle.amax(np.ascontiguousarray(full[:, :c]))
    big = torch.full((1,), 1e30, dtype=torch.float32, device="cuda")  # accumulates with max
    q.fp8_amax(x, big)
    assert host(big)[0] == np.float32(1e30)


def test_amax_nan_and_empty(q):
    xb = wl.random_bf16(3, 64, 64, "normal")
    xb[10, 17] = 0xFFC1  # a negative NaN
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    q.fp8_amax(dev_bf16(xb), amax)
    assert np.isnan(host(amax)[0])
    amax.zero_()
    q.fp8_amax(torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"), amax)
    assert host(amax)[0] == 0


# -------------------------------------------------------------- compute_scale

def _amax_values():
    rng = np.random.default_rng(0)
    v = list(np.exp2(rng.uniform(-140, 127, 300)).astype(np.float32))
    v += [np.float32(x) for x in (0.0, 448.0, 450.0, 30.0, 1.0, 1.75, 224.0, 57344.0, 65536.0, 1e-45, 3.3e38)]
    for k in range(-60, 60, 9):
        b = np.float32(448.0 * 2.0 ** k)
        v += [b, np.nextafter(b, np.float32(0)), np.nextafter(b, np.float32(np.inf))]
    return v


@pytest.mark.parametrize("fmt,margin", [(0, 0), (1, 0), (1, 1), (0, -3)])
def test_compute_scale(q, fmt, margin):
    vals = _amax_values()
    amax = torch.tensor(np.array(vals, np.float32), device="cuda")
    bias = torch.empty(len(vals), dtype=torch.int32, device="cuda")
    scale = torch.empty(len(vals), dtype=torch.float32, device="cuda")
    sinv = torch.empty(len(vals), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    esz = 4
    for i in range(len(vals)):
        q.fp8_compute_scale(amax.data_ptr() + esz * i, fmt, margin, bias.data_ptr() + 4 * i,
                            scale.data_ptr() + 4 * i, sinv.data_ptr() + 4 * i, status)
    b, s, si = host(bias), host(scale), host(sinv)
    for i, a in enumerate(vals):
        e, _ = oracle.compute_bias(float(a), fmt, margin)
        assert b[i] == e, (float(a), b[i], e)
        assert s[i] == oracle.pow2f(e) and si[i] == oracle.pow2f(-e)
    assert host(status)[0] == 0


def test_compute_scale_nonfinite(q):
    for bad in (np.inf, np.nan):
        amax = torch.tensor([bad], dtype=torch.float32, device="cuda")
        bias = torch.full((1,), 99, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        q.fp8_compute_scale(amax, 0, 0, bias, None, None, status)
        assert host(bias)[0] == 0 and host(status)[0] == q.STATUS_NONFINITE_AMAX


# -------------------------------------------------------------------- history

@pytest.mark.parametrize("L", [1, 16, 1024, 1500])
@pytest.mark.parametrize("fmt,margin", [(0, 0), (1, 1)])
def test_history_sequence(q, L, fmt, margin):
    rng = np.random.default_rng(L + fmt)
    steps = min(3 * L + 7, 200) if L < 1024 else 40
    amaxes = np.exp2(rng.uniform(-30, 12, steps)).astype(np.float32)
    ref = oracle.HistoryState(L)
    from scaling_quantization_gemm_gb300.step import ScaleState
    st = ScaleState(fmt, margin, L)
    for t, a in enumerate(amaxes):
        st.amax.fill_(float(a))
        st.advance()
        ref.update(float(a), fmt, margin)
        assert host(st.bias)[0] == ref.bias[0], t
        assert host(st.scale)[0] == ref.scale[0] and host(st.scale_inv)[0] == ref.scale_inv[0]
        assert host(st.pos)[0] == ref.pos[0] and host(st.amax)[0] == 0
    assert np.array_equal(host(st.history), ref.hist)


def test_history_checkpoint_restore(q):
    from scaling_quantization_gemm_gb300.step import ScaleState
    rng = np.random.default_rng(9)
    amaxes = np.exp2(rng.uniform(-8, 8, 50)).astype(np.float32)
    a, b = ScaleState(0, 0, 16), ScaleState(0, 0, 16)
    for v in amaxes:
        a.amax.fill_(float(v))
        a.advance()
    for v in amaxes[:23]:
        b.amax.fill_(float(v))
        b.advance()
    saved = {k: host(getattr(b, k)).copy() for k in ("history", "pos", "bias", "scale", "scale_inv")}
    c = ScaleState(0, 0, 16)
    for k, v in saved.items():
        getattr(c, k).copy_(torch.from_numpy(v))
    for v in amaxes[23:]:
        c.amax.fill_(float(v))
        c.advance()
    for k in saved:
        assert np.array_equal(host(getattr(a, k)), host(getattr(c, k))), k


# ------------------------------------------------------------------ quantise

SHAPES = [(16, 8), (48, 136), (144, 264), (256, 1024), (272, 520), (1040, 96)]


def _run_gpu_quant(q, x_bits, fmt, gran, margin, row, col, ld=None, scale_val=None):
    r, c = x_bits.shape
    if ld is not None and ld != c:
        wide = np.zeros((r, ld), np.uint16)
        wide[:, :c] = x_bits
        x = dev_bf16(wide)[:, :c]
    else:
        x = dev_bf16(x_bits)
    srow, scol = oracle.scale_shapes(r, c, gran) if gran else ((0, 0), (0, 0))
    sdt = torch.uint8 if gran == q.MX_1x32 else torch.float32
    qr = torch.full((r, c), 0xAB, dtype=torch.uint8, device="cuda") if row else None
    qc = torch.full((c, r), 0xAB, dtype=torch.uint8, device="cuda") if col else None
    sr = torch.empty(srow, dtype=sdt, device="cuda") if (row and gran) else None
    sc = torch.empty(scol, dtype=sdt, device="cuda") if (col and gran) else None
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    scale = torch.tensor([scale_val], dtype=torch.float32, device="cuda") if gran == 0 else None
    q.fp8_quantize(x, fmt, gran, margin, scale=scale, q_row=qr, q_col=qc, sf_row=sr, sf_col=sc, amax=amax)
    return (host(qr) if row else None, host(sr) if sr is not None else None, host(qc) if col else None,
            host(sc) if sc is not None else None, host(amax)[0])


@pytest.mark.parametrize("gran", [0, 1, 2, 3])
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shape", SHAPES)
def test_quantize_parity(q, gran, fmt, shape):
    r, c = shape
    kind = ["normal", "t3", "wide", "laplace"][(r + c + gran) % 4]
    x = wl.random_bf16(1000 + r + c + 10 * gran + fmt, r, c, kind, 0.5)
    margin = 1 if fmt == 1 else 0
    amax_ref = oracle.amax(x)
    if gran == 0:
        e, s, _ = oracle.scale_triple(amax_ref, fmt, margin)
        qr, _, qc, _, am = _run_gpu_quant(q, x, fmt, gran, margin, True, True, scale_val=float(s))
        rr, rc = oracle.quantize_tensor(x, fmt, s, row=True, col=True)
        assert_codes_equal(qr, rr, fmt, "row")
        assert_codes_equal(qc, rc, fmt, "col")
    else:
        qr, sr, qc, sc, am = _run_gpu_quant(q, x, fmt, gran, margin, True, True)
        rr, rsr, rc, rsc, _ = oracle.quantize_block(x, fmt, gran, margin, row=True, col=True)
        assert_codes_equal(qr, rr, fmt, "row")
        assert_codes_equal(qc, rc, fmt, "col")
        assert np.array_equal(sr, rsr), "row scales"
        assert np.array_equal(sc, rsc), "col scales"
    assert am == amax_ref


@pytest.mark.parametrize("gran", [0, 1, 2, 3])
def test_quantize_row_only_col_only_and_ld(q, gran):
    r, c, ld = 160, 392, 520
    x = wl.random_bf16(77 + gran, r, c, "normal", 3.0)
    s = float(oracle.scale_triple(oracle.amax(x), 0)[1]) if gran == 0 else None
    qr, sr, _, _, _ = _run_gpu_quant(q, x, 0, gran, 0, True, False, ld=ld, scale_val=s)
    _, _, qc, sc, _ = _run_gpu_quant(q, x, 0, gran, 0, False, True, ld=ld, scale_val=s)
    if gran == 0:
        rr, rc = oracle.quantize_tensor(x, 0, np.float32(s), row=True, col=True)
    else:
        rr, rsr, rc, rsc, _ = oracle.quantize_block(x, 0, gran, 0, row=True, col=True)
        assert np.array_equal(sr, rsr) and np.array_equal(sc, rsc)
    assert_codes_equal(qr, rr, 0, "row")
    assert_codes_equal(qc, rc, 0, "col")


def test_quantize_all_zero_blocks(q):
    x = wl.random_bf16(0, 128, 256, "zeros")
    qr, sr, qc, sc, am = _run_gpu_quant(q, x, 0, q.MX_1x32, 0, True, True)
    assert am == 0 and not qr.any() and not qc.any()
    assert (sr == 127).all() and (sc == 127).all()


def test_quantize_empty_is_noop(q):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(0, 64, dtype=torch.uint8, device="cuda")
    q.fp8_quantize(x, 0, q.TENSOR, scale=torch.ones(1, device="cuda"), q_row=out)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("scale_val", [0.3, 3.7, -2.0, 1e-30, 2.0 ** -130])
def test_quantize_tensor_arbitrary_scale(q, fmt, scale_val):
    """A per-tensor scale that is not a positive normal power of two takes the fp32 multiply path."""
    x = wl.random_bf16(55 + fmt, 144, 264, "wide", 1.0)
    qr, _, qc, _, _ = _run_gpu_quant(q, x, fmt, 0, 0, True, True, scale_val=float(np.float32(scale_val)))
    rr, rc = oracle.quantize_tensor(x, fmt, np.float32(scale_val), row=True, col=True)
    assert_codes_equal(qr, rr, fmt, "row")
    assert_codes_equal(qc, rc, fmt, "col")


def test_calls_run_on_the_callers_stream(q):
    """Work is enqueued on the caller's (current) stream: each call sees the producer that ran just
    before it on the same side stream, without any synchronisation with other streams."""
    xb = wl.random_bf16(61, 4096, 4096, "normal")
    amax_ref = oracle.amax(xb)
    base = dev_bf16(xb)
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        x = torch.zeros_like(base)
        for _ in range(20):  # keep the producer busy for a while
            x.copy_(base * 1.0)
        amax = torch.zeros(1, dtype=torch.float32, device="cuda")
        q.fp8_amax(x, amax)
        out = torch.empty(4096, 4096, dtype=torch.uint8, device="cuda")
        scale = torch.tensor([float(oracle.scale_triple(amax_ref, 0)[1])], device="cuda")
        q.fp8_quantize(x, 0, q.TENSOR, scale=scale, q_row=out)
    side.synchronize()
    assert host(amax)[0] == amax_ref
    assert_codes_equal(host(out), oracle.quantize_tensor(xb, 0, oracle.scale_triple(amax_ref, 0)[1])[0], 0)


@pytest.mark.parametrize("gran", [0, 1, 2, 3])
@pytest.mark.parametrize("shape", [(48, 136), (272, 520)])
def test_quantize_col_bounds_and_offset(q, gran, shape):
    """The column-wise copy written at a 16-byte (not 128-byte) aligned offset inside a larger buffer:
    the codes match the oracle and no byte before or after the [cols x rows] block changes (the tile
    stores are clipped at the tensor's edge)."""
    r, c = shape
    x_bits = wl.random_bf16(300 + r + gran, r, c, "normal", 2.0)
    x = dev_bf16(x_bits)
    off, pad = 48, 4096
    buf = torch.full((off + c * r + pad,), 0x5A, dtype=torch.uint8, device="cuda")
    qc = buf[off:off + c * r].view(c, r)
    srow, scol = oracle.scale_shapes(r, c, gran) if gran else ((0, 0), (0, 0))
    sdt = torch.uint8 if gran == q.MX_1x32 else torch.float32
    sc = torch.empty(scol, dtype=sdt, device="cuda") if gran else None
    if gran == 0:
        s = oracle.scale_triple(oracle.amax(x_bits), 0)[1]
        q.fp8_quantize(x, 0, gran, 0, scale=torch.tensor([float(s)], device="cuda"), q_col=qc)
        _, rc = oracle.quantize_tensor(x_bits, 0, s, row=False, col=True)
    else:
        q.fp8_quantize(x, 0, gran, 0, q_col=qc, sf_col=sc)
        _, _, rc, rsc, _ = oracle.quantize_block(x_bits, 0, gran, 0, row=False, col=True)
        assert np.array_equal(host(sc), rsc)
    assert_codes_equal(host(qc), rc, 0, "col")
    b = host(buf)
    assert (b[:off] == 0x5A).all() and (b[off + c * r:] == 0x5A).all()
