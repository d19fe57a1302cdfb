"""The sharded data-parallel layer on one GPU (one rank, no process group: the reductions are
identities) computes exactly what the unsharded layer computes, including its first step, which
takes the separate amax / compute_scale / cast path instead of the fused one."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import dev_bf16, host, require_gpu

pytestmark = pytest.mark.gpu


def test_one_rank_sharded_equals_unsharded():
    require_gpu()
    from scaling_quantization_gemm_gb300.sharded import ShardedLinearFwdBwd
    from scaling_quantization_gemm_gb300.step import LinearFwdBwd
    X = dev_bf16(wl.random_bf16(1, 512, 256, "normal"))
    W = dev_bf16(wl.random_bf16(2, 384, 256, "normal", 0.02))
    dY = dev_bf16(wl.random_bf16(3, 512, 384, "laplace", 1e-5))
    a, b = LinearFwdBwd(X, W, dY, history_len=8), ShardedLinearFwdBwd(X, W, dY, history_len=8)
    for _ in range(3):
        a.run()
        b.run()
        torch.cuda.synchronize()
        for name in ("qx_row", "qx_col", "qw_row", "qw_col", "qg_row", "qg_col", "Y", "dX", "dW"):
            assert torch.equal(getattr(a, name), getattr(b, name)), name
        for sa, sb in ((a.sx, b.sx), (a.sw, b.sw), (a.sg, b.sg)):
            assert np.array_equal(host(sa.history), host(sb.history))
            assert host(sa.scale)[0] == host(sb.scale)[0] and host(sa.pos)[0] == host(sb.pos)[0]
