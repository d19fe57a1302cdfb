"""fp8_quantize_current_noalloc (static scratch, no allocation) against fp8_quantize_current (caller
workspace), called through the C ABI.  Collected last on purpose: it must pass after the other
GPU tests have used the library in this process, and alone in a fresh one.

Two calls in a row on different tensors, formats and margins: amax, bias, scale, scale_inv and
every code must match the workspace entry point bit for bit (the tolerance of all cast tests)."""
import ctypes

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


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    q = require_gpu()
    L = q.lib()
    stream = torch.cuda.current_stream().cuda_stream or None
    ws = q.current_workspace()
    cases = [(2048, 3072, 0, 0, wl.random_bf16(11, 2048, 3072, "t3", 0.5)),
             (4096, 4096, 1, 1, wl.random_bf16(12, 4096, 4096, "laplace", 1e-4))]
    for r, c, fmt, margin, xb in cases:
        x = dev_bf16(xb)
        got, ref = _outputs(r, c), _outputs(r, c)
        st = L.fp8_quantize_current_noalloc(x.data_ptr(), r, c, c, fmt, margin, *_ptrs(got),
                                            got["status"].data_ptr(), stream)
        assert st == 0, L.fp8_last_error_detail().decode()
        st = L.fp8_quantize_current(x.data_ptr(), r, c, c, fmt, margin, *_ptrs(ref), ws.data_ptr(),
                                    ref["status"].data_ptr(), stream)
        assert st == 0, L.fp8_last_error_detail().decode()
        torch.cuda.synchronize()
        for k in ("amax", "bias", "scale", "scale_inv", "status"):
            assert np.array_equal(host(got[k]), host(ref[k])), k
        assert host(got["status"])[0] == 0 and host(got["amax"])[0] > 0
        assert_codes_equal(host(got["q_row"]), host(ref["q_row"]), fmt, "row")
        assert_codes_equal(host(got["q_col"]), host(ref["q_col"]), fmt, "col")
