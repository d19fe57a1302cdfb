"""The sharded data-parallel layer (scaling_quantization_gemm_gb300.sharded).

* One rank, no process group: the reductions are identities and the layer computes exactly what
  the unsharded layer computes, including its first step, which takes the separate amax /
  compute_scale / cast path instead of the fused one.
* Two ranks over gloo, each a process on cuda:0 with its half of the tokens (rows of X and dY) and
  the whole W: five delayed-scaling steps (history length 4, so the window wraps) through
  `ShardedLinearFwdBwd.run`, checked on both ranks against the oracle run on the WHOLE tensors --
  histories, positions, biases and scales bit-exact and identical on the ranks, every FP8 code of
  the rank's row- and column-wise copies bit-exact, Y and dX of the rank's rows and the summed dW
  within the GEMM tolerance.  An outlier planted in one rank's half at each step (alternating
  ranks) makes every step's scale depend on the MAX all-reduce.  The ranks' kernels never wait on
  one another: the exchanges are host-side gloo collectives between launches."""
import os
import socket

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import assert_codes_equal, assert_gemm_close, bf16_out_to_f64, dev_bf16, host, require_gpu

pytestmark = pytest.mark.gpu

M, K, N = 512, 256, 384  # tokens, in features, out features
HIST, STEPS, WORLD = 4, 5, 2
X_SCALES = (1.0, 4.0, 0.5, 0.25, 2.0)  # the activation's magnitude per step (non-monotone window max)


def step_inputs(t):
    """Whole X_t [M x K] and dY_t [M x N] (bf16 bits) for step t, each with one outlier planted in
    the half of rank t % 2; W [N x K] is the same every step."""
    X = wl.random_bf16(700 + t, M, K, "normal", X_SCALES[t])
    dY = wl.random_bf16(800 + t, M, N, "laplace", 1e-4 * (t + 1))
    r = t % 2
    X[r * (M // 2) + 17 + t, 5 + t] = wl.bf16_bits(np.array([[60.0 * X_SCALES[t]]]))[0, 0]
    dY[r * (M // 2) + 3 + t, 11 + t] = wl.bf16_bits(np.array([[-0.5 * (t + 1)]]))[0, 0]
    return X, dY


def weight():
    return wl.random_bf16(799, N, K, "normal", 0.02)


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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, out_q):
    """One rank: its token shard through STEPS steps of the sharded layer on cuda:0."""
    try:
        import torch.distributed as dist
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=WORLD)
        torch.cuda.set_device(0)
        import scaling_quantization_gemm_gb300 as q
        q.lib()
        from scaling_quantization_gemm_gb300.sharded import ShardedLinearFwdBwd
        rows = slice(rank * (M // WORLD), (rank + 1) * (M // WORLD))
        X0, dY0 = step_inputs(0)
        layer = ShardedLinearFwdBwd(dev_bf16(X0[rows]), dev_bf16(weight()), dev_bf16(dY0[rows]), history_len=HIST,
                                    grad_margin=1)
        steps = []
        for t in range(STEPS):
            Xt, dYt = step_inputs(t)
            layer.X.copy_(dev_bf16(Xt[rows]))
            layer.dY.copy_(dev_bf16(dYt[rows]))
            layer.run()
            torch.cuda.synchronize()
            rec = {k: host(getattr(layer, k)) for k in ("qx_row", "qx_col", "qw_row", "qw_col", "qg_row", "qg_col")}
            rec.update(Y=bf16_out_to_f64(layer.Y), dX=bf16_out_to_f64(layer.dX), dW=host(layer.dW).astype(np.float64))
            for k, st in (("x", layer.sx), ("w", layer.sw), ("g", layer.sg)):
                rec[f"hist_{k}"] = host(st.history).copy()
                rec[f"state_{k}"] = (int(host(st.pos)[0]), int(host(st.bias)[0]), float(host(st.scale)[0]),
                                     float(host(st.scale_inv)[0]), int(host(st.status)[0]))
            steps.append(rec)
        dist.barrier()
        dist.destroy_process_group()
        out_q.put((rank, steps, None))
    except Exception as e:  # report instead of hanging the parent on the queue
        import traceback
        out_q.put((rank, None, traceback.format_exc() + repr(e)))


def test_two_ranks_sharded_layer_against_oracle(oracle):
    require_gpu()
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, out_q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(WORLD):
        rank, steps, err = out_q.get(timeout=600)
        assert err is None, f"rank {rank}: {err}"
        res[rank] = steps
    for p in procs:
        p.join(60)
        assert p.exitcode == 0

    fmts, margins = {"x": 0, "w": 0, "g": 1}, {"x": 0, "w": 0, "g": 1}
    hist = {k: oracle.HistoryState(HIST) for k in "xwg"}
    W = weight()
    half = M // WORLD
    for t in range(STEPS):
        X, dY = step_inputs(t)
        whole = {"x": X, "w": W, "g": dY}
        amax = {k: oracle.amax(v) for k, v in whole.items()}
        # the scale of step t: the tensor's own amax on the first step (empty history), then the
        # scale the history chose at the end of step t - 1
        scale = {k: (oracle.scale_triple(amax[k], fmts[k], margins[k])[1:] if t == 0 else
                     (hist[k].scale[0], hist[k].scale_inv[0])) for k in "xwg"}
        codes = {k: oracle.quantize_tensor(whole[k], fmts[k], scale[k][0], row=True, col=True) for k in "xwg"}
        for k in "xwg":
            hist[k].update(float(amax[k]), fmts[k], margins[k])
        (qx_r, qx_c), (qw_r, qw_c), (qg_r, qg_c) = codes["x"], codes["w"], codes["g"]
        ix, iw, ig = scale["x"][1], scale["w"][1], scale["g"][1]
        dW_ref, dW_mag = oracle.gemm_full(qg_c, 1, 0, ig, qx_c, 0, 0, ix)
        for rank in range(WORLD):
            got = res[rank][t]
            rows = slice(rank * half, (rank + 1) * half)
            for k in "xwg":
                assert np.array_equal(got[f"hist_{k}"], hist[k].hist), (t, rank, k)
                pos, bias, s, si, status = got[f"state_{k}"]
                assert (pos, bias, status) == (t + 1, int(hist[k].bias[0]), 0), (t, rank, k)
                assert s == float(hist[k].scale[0]) and si == float(hist[k].scale_inv[0]), (t, rank, k)
            for name, ref, fmt in (("qx_row", qx_r[rows], 0), ("qx_col", qx_c[:, rows], 0), ("qw_row", qw_r, 0),
                                   ("qw_col", qw_c, 0), ("qg_row", qg_r[rows], 1), ("qg_col", qg_c[:, rows], 1)):
                assert_codes_equal(got[name], ref, fmt, f"step {t} rank {rank} {name}")
            y_ref, mag = oracle.gemm_full(qx_r[rows], 0, 0, ix, qw_r, 0, 0, iw)
            assert_gemm_close(got["Y"], y_ref, mag, True, f"step {t} rank {rank} Y")
            dx_ref, mag = oracle.gemm_full(qg_r[rows], 1, 0, ig, qw_c, 0, 0, iw)
            assert_gemm_close(got["dX"], dx_ref, mag, True, f"step {t} rank {rank} dX")
            assert_gemm_close(got["dW"], dW_ref, dW_mag, False, f"step {t} rank {rank} dW (summed over ranks)")
        # the planted outlier sits in one rank's half: that rank's local amax alone is the whole amax
        assert oracle.amax(X[(t % 2) * half:(t % 2 + 1) * half]) == amax["x"]
