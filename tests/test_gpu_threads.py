"""Calls from several host threads at once, each on its own CUDA stream: the library keeps no state
between calls beyond per-device caches (kernel attributes, occupancy), so concurrent casts and GEMMs
on different streams must each give the oracle's result."""
import threading

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_codes_equal, assert_gemm_close, bf16_out_to_f64, dev_bf16, host, require_gpu

pytestmark = pytest.mark.gpu


def _work(q, seed, results, errors):
    try:
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            X = wl.random_bf16(seed, 384, 512, "normal")
            W = wl.random_bf16(seed + 1, 256, 512, "normal", 0.05)
            x, w = dev_bf16(X), dev_bf16(W)
            out = {}
            for rep in range(3):
                # MX casts (fresh kernels on the first call from this thread) and the MX GEMM
                qx = torch.empty(384, 512, dtype=torch.uint8, device="cuda")
                qw = torch.empty(256, 512, dtype=torch.uint8, device="cuda")
                sx = torch.empty(384, 16, dtype=torch.uint8, device="cuda")
                sw = torch.empty(256, 16, dtype=torch.uint8, device="cuda")
                q.fp8_quantize(x, 0, q.MX_1x32, q_row=qx, sf_row=sx)
                q.fp8_quantize(w, 0, q.MX_1x32, q_row=qw, sf_row=sw)
                y = torch.empty(384, 256, dtype=torch.bfloat16, device="cuda")
                q.fp8_scaled_gemm(q.FPROP, qx, 0, q.MX_1x32, sx, qw, 0, q.MX_1x32, sw, y)
                # per-tensor current scaling with its own workspace
                ws = q.current_workspace()
                qc = torch.empty(384, 512, dtype=torch.uint8, device="cuda")
                am = torch.zeros(1, device="cuda")
                q.fp8_quantize_current(x, 0, 0, ws, q_row=qc, amax=am)
            stream.synchronize()
            out["qx"], out["sx"], out["qw"], out["sw"] = host(qx), host(sx), host(qw), host(sw)
            out["y"], out["qc"], out["amax"] = bf16_out_to_f64(y), host(qc), host(am)[0]
            results[seed] = (X, W, out)
    except Exception as e:  # reported by the main thread
        errors.append(e)


def test_concurrent_threads_and_streams():
    q = require_gpu()
    results, errors = {}, []
    threads = [threading.Thread(target=_work, args=(q, 100 + 10 * i, results, errors)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert len(results) == 4
    for seed, (X, W, out) in results.items():
        rx, rsx, _, _, _ = oracle.quantize_block(X, 0, oracle.MX_1x32)
        rw, rsw, _, _, _ = oracle.quantize_block(W, 0, oracle.MX_1x32)
        assert_codes_equal(out["qx"], rx, 0, "X")
        assert_codes_equal(out["qw"], rw, 0, "W")
        assert np.array_equal(out["sx"], rsx) and np.array_equal(out["sw"], rsw)
        y_ref, mag = oracle.gemm_full(rx, 0, oracle.MX_1x32, rsx, rw, 0, oracle.MX_1x32, rsw)
        assert_gemm_close(out["y"], y_ref, mag, True)
        a = oracle.amax(X)
        assert out["amax"] == a
        assert_codes_equal(out["qc"], oracle.quantize_tensor(X, 0, oracle.scale_triple(a, 0)[1])[0], 0, "current")
