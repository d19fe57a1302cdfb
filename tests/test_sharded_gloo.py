"""Host side of the data-parallel sharding (scaling_quantization_gemm_gb300.sharded), world size 2
over gloo on the CPU: the amax and weight-gradient reductions, and delayed scaling over token
shards keeping every rank's history identical to the history of the unsharded tensor."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import workloads as wl
    from scaling_quantization_gemm_gb300.sharded import allreduce_amax_, allreduce_sum_

    a = torch.tensor([1.5 if rank == 0 else 7.25])
    allreduce_amax_(a)
    # a non-finite amax on one rank reaches both, whichever rank holds it
    specials = []
    for bad_rank in (0, 1):
        for bad in (float("nan"), float("inf")):
            v = torch.tensor([bad if rank == bad_rank else 3.0])
            allreduce_amax_(v)
            specials.append(v.item())
    z = torch.tensor([0.0])
    allreduce_amax_(z)
    specials.append(z.item())
    s = torch.arange(6, dtype=torch.float32) * (rank + 1)
    allreduce_sum_(s)

    # delayed scaling over token shards: 6 steps, tensor rows split between the ranks
    L, hist = 4, oracle.HistoryState(4)
    for t in range(6):
        full = wl.random_bf16(900 + t, 256, 512, "laplace", 10.0 ** (t - 3))
        shard = full[rank * 128:(rank + 1) * 128]
        local = torch.tensor([float(oracle.amax(shard))])
        allreduce_amax_(local)
        hist.update(float(local[0]), 1, 1)
    q.put((rank, float(a[0]), s.tolist(), hist.hist.tolist(), int(hist.bias[0]), float(hist.scale[0]),
           [repr(v) for v in specials]))
    dist.destroy_process_group()


def test_sharded_reductions_and_delayed_scaling_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    res = dict((r[0], r[1:]) for r in (q.get(timeout=10) for _ in range(world)))
    assert res[0] == res[1]  # identical scaling state on every rank
    amax, s, hist, bias, scale, specials = res[0]
    assert amax == 7.25
    assert specials == ["nan", "inf", "nan", "inf", "0.0"]
    assert s == [3.0 * i for i in range(6)]
    # the unsharded reference: the same six tensors, whole
    import oracle
    import workloads as wl
    ref = oracle.HistoryState(4)
    for t in range(6):
        ref.update(float(oracle.amax(wl.random_bf16(900 + t, 256, 512, "laplace", 10.0 ** (t - 3)))), 1, 1)
    assert hist == ref.hist.tolist() and bias == int(ref.bias[0]) and scale == float(ref.scale[0])


def test_single_process_reductions_are_identity():
    from scaling_quantization_gemm_gb300.sharded import allreduce_amax_, allreduce_sum_
    a = torch.tensor([2.0])
    assert allreduce_amax_(a) is a and float(a[0]) == 2.0
    s = torch.ones(3)
    assert allreduce_sum_(s).tolist() == [1.0, 1.0, 1.0]
