"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The fused current-scaling cast waits at a grid barrier for the last CTA to
publish the scale.  With the workspace's arrival count poisoned, no CTA is ever
the last one, so every CTA's wait runs out (about 2 s); the kernel must return,
report FP8_STATUS_TIMEOUT in the status word and leave the context usable: after
the workspace is zeroed again the same call gives the right result."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_codes_equal, dev_bf16, host, require_gpu

pytestmark = pytest.mark.gpu


def test_barrier_timeout_is_reported_and_recoverable():
    q = require_gpu()
    xb = wl.random_bf16(21, 1024, 1024, "normal")
    x = dev_bf16(xb)
    ws = q.current_workspace()
    ws[:4].view(torch.int32).fill_(1 << 30)  # arrival count no CTA can complete
    out = torch.full((1024, 1024), 0xAB, dtype=torch.uint8, device="cuda")
    bias = torch.full((1,), 999, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.time()
    q.fp8_quantize_current(x, q.E4M3, 0, ws, q_row=out, bias=bias, status=status)
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert host(status)[0] & q.STATUS_TIMEOUT
    assert 1.5 < waited < 30.0
    assert (host(out) == 0xAB).all() and host(bias)[0] == 999  # nothing was cast or published

    ws.zero_()
    status.zero_()
    amax = torch.zeros(1, device="cuda")
    q.fp8_quantize_current(x, q.E4M3, 0, ws, q_row=out, amax=amax, bias=bias, status=status)
    torch.cuda.synchronize()
    assert host(status)[0] == 0
    e, s, _ = oracle.scale_triple(oracle.amax(xb), 0)
    assert host(bias)[0] == e and host(amax)[0] == oracle.amax(xb)
    assert_codes_equal(host(out), oracle.quantize_tensor(xb, 0, s)[0], 0, "after recovery")
