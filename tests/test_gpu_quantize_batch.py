"""fp8_quantize_batch: several casts in one launch give, bit for bit, what the same fp8_quantize calls
give one after another, and what the oracle gives -- codes of both copies, block scales, amax.

Batches mix granularities and formats (the per-block recipe: 1x128 activations with 128x128
weights; a linear layer's three per-tensor casts, E4M3 and E5M2, row- and column-wise with the fused
amax; MX and OCP-MX blocks), use ragged shapes and leading dimensions, an empty tensor, and two casts
that share one amax (which then holds the maximum over both)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_codes_equal, dev_bf16, host, require_gpu

pytestmark = pytest.mark.gpu

TENSOR, B1x128, B128, MX, MXOCP = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def q():
    return require_gpu()


def _padded(xb, ld):
    """bf16 bits [r x c] -> device tensor view [r x c] with leading dimension ld (padding holds garbage)."""
    r, c = xb.shape
    full = np.full((r, ld), 0x7FC0, np.uint16)  # NaN padding: must never be read
    full[:, :c] = xb
    return dev_bf16(full)[:, :c]


def _outputs(xb, gran, row, col):
    r, c = xb.shape
    u8 = dict(dtype=torch.uint8, device="cuda")
    o = {}
    if row:
        o["q_row"] = torch.full((r, c), 0xAB, **u8)
    if col:
        o["q_col"] = torch.full((c, r), 0xAB, **u8)
    if gran != TENSOR:
        srow, scol = oracle.scale_shapes(r, c, gran)
        dt = torch.uint8 if gran in (MX, MXOCP) else torch.float32
        if row:
            o["sf_row"] = torch.full(srow, 7, dtype=dt, device="cuda")
        if col:
            o["sf_col"] = torch.full(scol, 7, dtype=dt, device="cuda")
    return o


def _cast_spec(x, fmt, gran, margin, out, scale=None, amax=None):
    d = dict(x=x, fmt=fmt, gran=gran, margin=margin, **out)
    if scale is not None:
        d["scale"] = scale
    if amax is not None:
        d["amax"] = amax
    return d


def _check_against_oracle(xb, fmt, gran, margin, out, scale=None):
    row, col = "q_row" in out, "q_col" in out
    if gran == TENSOR:
        rr, rc = oracle.quantize_tensor(xb, fmt, scale, row=row, col=col)
    else:
        rr, rsr, rc, rsc, _ = oracle.quantize_block(xb, fmt, gran, margin, row=row, col=col)
        if row:
            assert np.array_equal(host(out["sf_row"]), rsr), "row scales"
        if col:
            assert np.array_equal(host(out["sf_col"]), rsc), "column scales"
    if row:
        assert_codes_equal(host(out["q_row"]), rr, fmt, "row codes")
    if col:
        assert_codes_equal(host(out["q_col"]), rc, fmt, "column codes")


def _run(q, casts):
    """casts: list of (xb bits, ld, fmt, gran, margin, row, col, with_amax).  Runs them as one batch and
    as separate calls; checks both agree bit for bit and match the oracle.  Returns the batch's amaxes."""
    batch, single, meta = [], [], []
    for xb, ld, fmt, gran, margin, row, col, with_amax in casts:
        x = _padded(xb, ld)
        scale_t = None
        s = None
        if gran == TENSOR:
            _, s, _ = oracle.scale_triple(oracle.amax(xb), fmt, margin)
            scale_t = torch.full((1,), float(s), device="cuda")
        ob, os_ = _outputs(xb, gran, row, col), _outputs(xb, gran, row, col)
        ab = torch.zeros(1, device="cuda") if with_amax else None
        as_ = torch.zeros(1, device="cuda") if with_amax else None
        batch.append(_cast_spec(x, fmt, gran, margin, ob, scale_t, ab))
        single.append(_cast_spec(x, fmt, gran, margin, os_, scale_t, as_))
        meta.append((xb, fmt, gran, margin, s, ob, os_, ab, as_))
    q.fp8_quantize_batch(batch)
    for c in single:
        q.fp8_quantize(**c)
    torch.cuda.synchronize()
    for xb, fmt, gran, margin, s, ob, os_, ab, as_ in meta:
        for k in ob:
            assert torch.equal(ob[k], os_[k]), k
        if ab is not None:
            assert host(ab)[0] == host(as_)[0] == oracle.amax(xb)
        _check_against_oracle(xb, fmt, gran, margin, ob, s)


def test_batch_per_block_recipe(q):
    """1x128 activations and 128x128 weights in one launch (ragged rows and columns)."""
    X = wl.random_bf16(41, 1000, 4104, "t3", 0.5)
    W = wl.random_bf16(42, 1480, 4104, "normal", 0.02)
    _run(q, [(X, 4104, 0, B1x128, 0, True, False, False), (W, 4104, 0, B128, 0, True, False, False)])


def test_batch_linear_layer_per_tensor(q):
    """A layer's three per-tensor casts: X and W in E4M3, dY in E5M2 (margin 1), row- and column-wise,
    each with its fused amax; W with a leading dimension larger than its columns."""
    X = wl.random_bf16(43, 768, 1024, "normal")
    W = wl.random_bf16(44, 1536, 1024, "normal", 0.02)
    G = wl.random_bf16(45, 768, 1536, "laplace", 1e-4)
    _run(q, [(X, 1024, 0, TENSOR, 0, True, True, True), (W, 1040, 0, TENSOR, 0, True, True, True),
             (G, 1536, 1, TENSOR, 1, True, True, True)])


def test_batch_mx_and_ocp(q):
    """MX and OCP-MX blocks, row- and column-wise, in both formats, four casts (the maximum)."""
    a = wl.random_bf16(46, 512, 2048, "wide")
    b = wl.random_bf16(47, 1024, 2048, "normal", 0.01)
    c = wl.random_bf16(48, 336, 776, "t3")
    d = wl.random_bf16(49, 272, 1040, "laplace", 3.0)
    _run(q, [(a, 2048, 0, MX, 0, True, True, False), (b, 2048, 0, MX, 0, True, True, False),
             (c, 776, 1, MXOCP, 0, True, True, False), (d, 1048, 1, MX, 1, True, True, False)])


def test_batch_mixed_kinds_with_an_empty_tensor(q):
    """Every granularity kind across batches, an empty tensor skipped, row-only and column-only casts."""
    t = wl.random_bf16(50, 400, 520, "normal", 2.0)
    u = wl.random_bf16(51, 640, 136, "t3")
    v = wl.random_bf16(52, 144, 904, "wide")
    _run(q, [(t, 520, 1, TENSOR, 0, True, False, True), (u, 136, 0, B1x128, 0, False, True, False),
             (v, 904, 0, B128, 2, True, True, False)])
    empty = np.zeros((0, 64), np.uint16)
    x = dev_bf16(wl.random_bf16(53, 256, 256, "normal"))
    qr = torch.empty(256, 256, dtype=torch.uint8, device="cuda")
    sr = torch.empty(256, 8, dtype=torch.uint8, device="cuda")
    q.fp8_quantize_batch([dict(x=dev_bf16(np.zeros((1, 64), np.uint16))[:0], fmt=0, gran=MX),
                          dict(x=x, fmt=0, gran=MX, q_row=qr, sf_row=sr)])
    torch.cuda.synchronize()
    rr, rsr, _, _, _ = oracle.quantize_block(wl.random_bf16(53, 256, 256, "normal"), 0, MX)
    assert_codes_equal(host(qr), rr, 0, "row codes next to an empty tensor")
    assert np.array_equal(host(sr), rsr)
    assert empty.size == 0


def test_batch_shared_amax_holds_the_maximum_over_both(q):
    a = wl.random_bf16(54, 256, 512, "normal", 1.0)
    b = wl.random_bf16(55, 512, 256, "normal", 8.0)
    amax = torch.zeros(1, device="cuda")
    one = torch.ones(1, device="cuda")
    qa = torch.empty(256, 512, dtype=torch.uint8, device="cuda")
    qb = torch.empty(512, 256, dtype=torch.uint8, device="cuda")
    q.fp8_quantize_batch([dict(x=dev_bf16(a), fmt=0, gran=TENSOR, scale=one, q_row=qa, amax=amax),
                          dict(x=dev_bf16(b), fmt=1, gran=TENSOR, scale=one, q_row=qb, amax=amax)])
    torch.cuda.synchronize()
    assert host(amax)[0] == max(oracle.amax(a), oracle.amax(b))
    assert_codes_equal(host(qa), oracle.quantize_tensor(a, 0, 1.0)[0], 0)
    assert_codes_equal(host(qb), oracle.quantize_tensor(b, 1, 1.0)[0], 1)


def test_batch_full_size_per_block_workload(q):
    """The Llama-2-7B up-projection casts (X 8192x4096 1x128, W 11008x4096 128x128) in one launch."""
    X, W = wl.per_block_up_proj()
    _run(q, [(X, 4096, 0, B1x128, 0, True, False, False), (W, 4096, 0, B128, 0, True, False, False)])
