"""The steady-state FP8 layer step (delayed-scaling casts, fprop / dgrad / wgrad, history updates)
captured in a CUDA graph and replayed gives the same bits as the same step run eagerly."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import dev_bf16, host, require_gpu

pytestmark = pytest.mark.gpu


def test_layer_step_replays_from_a_cuda_graph():
    require_gpu()
    from scaling_quantization_gemm_gb300.step import LinearFwdBwd
    X = dev_bf16(wl.random_bf16(31, 512, 256, "normal"))
    W = dev_bf16(wl.random_bf16(32, 384, 256, "normal", 0.02))
    dY = dev_bf16(wl.random_bf16(33, 512, 384, "laplace", 1e-5))
    eager, graphed = LinearFwdBwd(X, W, dY, history_len=8), LinearFwdBwd(X, W, dY, history_len=8)
    for f in (eager, graphed):  # step 0 (current scaling) and one delayed step, eagerly
        f.run()
        f.run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.run()  # recorded, not run
    for _ in range(3):
        eager.run()
        g.replay()
        torch.cuda.synchronize()
        for name in ("qx_row", "qx_col", "qw_row", "qw_col", "qg_row", "qg_col", "Y", "dX", "dW"):
            assert torch.equal(getattr(eager, name), getattr(graphed, name)), name
        for sa, sb in ((eager.sx, graphed.sx), (eager.sw, graphed.sw), (eager.sg, graphed.sg)):
            assert np.array_equal(host(sa.history), host(sb.history))
            assert host(sa.pos)[0] == host(sb.pos)[0] and host(sa.scale)[0] == host(sb.scale)[0]
