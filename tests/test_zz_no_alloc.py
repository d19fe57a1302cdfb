"""fp8_quantize_current_noalloc (static scratch, no allocation) against fp8_quantize_current (caller
workspace), called through the C ABI.  Collected last on purpose: it must pass after the other
GPU tests have used the library in this process, and alone in a fresh one.

Two calls in a row on different tensors, formats and margins: amax, bias, scale, scale_inv and
every code must match the workspace entry point bit for bit (the tolerance of all cast tests),
and the oracle's amax, bias and codes.  Across the two calls the torch caching allocator's
allocated and reserved bytes stay where they were: the call itself asks for no device memory."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import assert_codes_equal, dev_bf16, host, require_gpu

pytestmark = pytest.mark.gpu


def _outputs(r, c):
    u8 = dict(dtype=torch.uint8, device="cuda")
    return dict(q_row=torch.full((r, c), 0xAB, **u8), q_col=torch.full((c, r), 0xAB, **u8),
                amax=torch.full((1,), -1.0, device="cuda"), bias=torch.full((1,), 999, dtype=torch.int32, device="cuda"),
                scale=torch.zeros(1, device="cuda"), scale_inv=torch.zeros(1, device="cuda"),
                status=torch.zeros(1, dtype=torch.int32, device="cuda"))


def _ptrs(o):
    return [o[k].data_ptr() for k in ("q_row", "q_col", "amax", "bias", "scale", "scale_inv")]


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(oracle):
    q = require_gpu()
    L = q.lib()
    stream = torch.cuda.current_stream().cuda_stream or None
    ws = q.current_workspace()
    cases = [(2048, 3072, 0, 0, wl.random_bf16(11, 2048, 3072, "t3", 0.5)),
             (4096, 4096, 1, 1, wl.random_bf16(12, 4096, 4096, "laplace", 1e-4))]
    xs = [dev_bf16(xb) for *_, xb in cases]
    got = [_outputs(r, c) for r, c, *_ in cases]
    ref = [_outputs(r, c) for r, c, *_ in cases]

    def noalloc(i):
        r, c, fmt, margin, _ = cases[i]
        st = L.fp8_quantize_current_noalloc(xs[i].data_ptr(), r, c, c, fmt, margin, *_ptrs(got[i]),
                                            got[i]["status"].data_ptr(), stream)
        assert st == 0, L.fp8_last_error_detail().decode()

    noalloc(1)  # warm-up: the first call on this device may look up the scratch address
    torch.cuda.synchronize()
    mem = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved())
    noalloc(0)  # the two calls in a row: the second finds the first's contents in the scratch
    noalloc(1)
    torch.cuda.synchronize()
    assert (torch.cuda.memory_allocated(), torch.cuda.memory_reserved()) == mem
    for i, (r, c, fmt, margin, _) in enumerate(cases):
        st = L.fp8_quantize_current(xs[i].data_ptr(), r, c, c, fmt, margin, *_ptrs(ref[i]), ws.data_ptr(),
                                    ref[i]["status"].data_ptr(), stream)
        assert st == 0, L.fp8_last_error_detail().decode()
    torch.cuda.synchronize()
    for (r, c, fmt, margin, xb), g, rf in zip(cases, got, ref):
        for k in ("amax", "bias", "scale", "scale_inv", "status"):
            assert np.array_equal(host(g[k]), host(rf[k])), k
        assert host(g["status"])[0] == 0 and host(g["amax"])[0] > 0
        assert_codes_equal(host(g["q_row"]), host(rf["q_row"]), fmt, "row")
        assert_codes_equal(host(g["q_col"]), host(rf["q_col"]), fmt, "col")
        # and the oracle's: amax, bias, scale and the codes of both copies
        amax = oracle.amax(xb)
        e, s, si = oracle.scale_triple(amax, fmt, margin)
        assert host(g["amax"])[0] == np.float32(amax) and int(host(g["bias"])[0]) == e
        assert host(g["scale"])[0] == np.float32(s) and host(g["scale_inv"])[0] == np.float32(si)
        r_ref, c_ref = oracle.quantize_tensor(xb, fmt, s, row=True, col=True)
        assert_codes_equal(host(g["q_row"]), r_ref, fmt, "row vs oracle")
        assert_codes_equal(host(g["q_col"]), c_ref, fmt, "col vs oracle")
