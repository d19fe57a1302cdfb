"""Benchmark of the FP8 hot path on one GB300 (replicas across GPUs).

One step = one pass over every step of the path on synthetic inputs already
resident in HBM:
  * per-tensor current scaling linear forward (X 256x1024 with +-30 outliers,
    W 1024x1024): amax, compute_scale, cast, GEMM with fp32 output;
  * 13B-class FFN layer forward + backward with per-tensor delayed scaling
    (history 1024): X 16384x5120, W 20480x5120 (E4M3), dY 16384x20480 (E5M2),
    each cast row- and column-wise with fused amax; fprop, dgrad, wgrad GEMMs;
    three history updates;
  * MXFP8 forward (1x32 blocks, E8M0): X 16384x8192, W 28672x8192 cast row- and
    column-wise; block-scaled GEMM M=16384 N=28672 K=8192, bf16 output;
  * per-block forward (1x128 activations, 128x128 weights, fp32 scales), Llama-2-7B
    MLP up-projection: X 8192x4096, W 11008x4096; GEMM M=8192 N=11008 K=4096.

value = GEMM FLOPs of the step / step time (TFLOP/s, the quantisation time
included).  The quantiser's own GB/s and the per-kernel roofline fractions are
reported beside it.  `--impl reference` times the CPU oracle on a bounded
sample of the same step instead.

Run: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torchrun; every rank runs an independent replica.
"""
from __future__ import annotations

import argparse
import math
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantize GB/s and FP8 scaled-GEMM TFLOPS at 1 GB300, % of HBM/FP8 roofline"
WORKLOAD = ("fp8 training hot path step: per-tensor current-scaling fwd 256x1024x1024 + 13B FFN fwd+bwd "
            "16384x20480x5120 per-tensor delayed (L=1024, row+col casts) + MXFP8 fwd 16384x28672x8192 "
            "(row+col casts) + per-block 1x128/128x128 fwd 8192x11008x4096")
REFERENCE_BUDGET_S = 120.0  # wall time the reference arm aims for, warm-up and timed steps together
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio 4.5 / 2.25 PFLOP/s


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ---------------------------------------------------------------- inputs

def make_inputs():
    import workloads as wl
    X1, W1 = wl.linear_fwd_current()
    X5, W5, dY5 = wl.ffn_fwd_bwd()
    X4, W4 = wl.mxfp8_inputs()
    X3, W3 = wl.per_block_up_proj()
    return dict(X1=X1, W1=W1, X5=X5, W5=W5, dY5=dY5, X4=X4, W4=W4, X3=X3, W3=W3)


# ------------------------------------------------------------- GPU side

class Nvml:
    """The few NVML queries the clock record needs, through ctypes (no Python NVML package on the GPU
    hosts).  `handle(i)` is None where NVML cannot be loaded."""

    SM = 1  # NVML_CLOCK_SM

    def __init__(self):
        import ctypes
        self.c = ctypes
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            self.ok = self.lib.nvmlInit_v2() == 0
        except OSError:
            self.lib, self.ok = None, False

    def handle(self, cuda_index: int):
        """NVML handle of the CUDA device: by UUID where torch reports it, else the CUDA index mapped
        through CUDA_VISIBLE_DEVICES."""
        if not self.ok:
            return None
        c = self.c
        h = c.c_void_p()
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
            if self.lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), c.byref(h)) == 0:
                return h
        except (AttributeError, RuntimeError, AssertionError):
            pass
        idx = cuda_index
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
        if cuda_index < len(vis) and vis[cuda_index].strip().isdigit():
            idx = int(vis[cuda_index])
        return h if self.lib.nvmlDeviceGetHandleByIndex_v2(c.c_uint(idx), c.byref(h)) == 0 else None

    def sample_line(self, h, index: int) -> str:
        """One sample in the CSV fields of ClockSampler.FIELDS."""
        c = self.c
        clk, mx, mw, rs = c.c_uint(), c.c_uint(), c.c_uint(), c.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(h, self.SM, c.byref(clk))
        self.lib.nvmlDeviceGetMaxClockInfo(h, self.SM, c.byref(mx))
        self.lib.nvmlDeviceGetPowerUsage(h, c.byref(mw))
        self.lib.nvmlDeviceGetCurrentClocksEventReasons(h, c.byref(rs))
        act = lambda bit: "Active" if rs.value & bit else "Not Active"
        # reason bits: 0x4 sw power cap, 0x8 hw slowdown, 0x20 sw thermal, 0x40 hw thermal
        return (f"{index}, {clk.value}, {mx.value}, {mw.value / 1000.0:.2f}, 0x{rs.value:x}, {act(0x8)}, "
                f"{act(0x40)}, {act(0x20)}, {act(0x4)}")


class ClockSampler:
    """SM clock, power and throttle-reason samples during the timed region: NVML every 10 ms from a
    thread of this process (nvidia-smi every 50 ms where NVML cannot be loaded).  NVML refreshes the
    clock it reports only every few tens of ms, so a sample can lag the clock by that much."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.01

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.thread = None
        self.lines = []

    def __enter__(self):
        import threading
        self.lines = []
        nv = Nvml()
        h = nv.handle(self.gpu)
        if h is not None:
            self.stop = threading.Event()

            def run():
                while not self.stop.is_set():
                    self.lines.append(nv.sample_line(h, self.gpu))
                    self.stop.wait(self.PERIOD_S)

            self.thread = threading.Thread(target=run, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join()
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        loaded = [s for s, p in zip(sm, power) if p > 0.5 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def clock_suspect(summary) -> list:
    """Why a timed region's clock record makes its number invalid (empty if it is valid): hardware or
    thermal slowdown, or an SM clock far below its maximum with no reason reported (a clock lock left
    behind by another user).  The software power cap is normal under load and kept."""
    reasons = set(summary.get("reasons") or [])
    bad = sorted(reasons & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"})
    sm, sm_max = summary.get("sm_mhz"), summary.get("sm_max_mhz")
    if sm and sm_max and not reasons and sm < 0.75 * sm_max:
        bad.append("sm_clock_low_without_reason")
    return bad


def run_ours(args, rank, world):
    import torch

    import scaling_quantization_gemm_gb300 as q
    from scaling_quantization_gemm_gb300.step import BlockLinearFwd, LinearFwdBwd, PerTensorFwd

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    q.lib()

    t0 = time.time()
    host = make_inputs()
    gen_s = time.time() - t0

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    d = {k: to_dev(v) for k, v in host.items()}
    c1 = PerTensorFwd(d["X1"], d["W1"])
    c5 = LinearFwdBwd(d["X5"], d["W5"], d["dY5"], history_len=1024)
    c4 = BlockLinearFwd(d["X4"], d["W4"], mx=True, col=True)
    c3 = BlockLinearFwd(d["X3"], d["W3"], mx=False, col=False)

    ops = [  # (name, callable, kind, work per call, our kernel launches per call)
        ("c1_fwd", c1.run, "mixed", 0.0, 3),
        # the three casts (X, W E4M3; dY E5M2), row- and column-wise with the fused amax, one batched launch;
        # operands are looked up at call time (the end-to-end leg swaps the input buffers between steps)
        ("c5_quant", c5.quantize, "quant", float(c5.quant_bytes), 1),
        ("c5_fprop", lambda: q.fp8_scaled_gemm(q.FPROP, c5.qx_row, 0, 0, c5.sx.scale_inv, c5.qw_row, 0, 0,
                                               c5.sw.scale_inv, c5.Y), "gemm_tensor", c5.flops / 3, 1),
        ("c5_dgrad", lambda: q.fp8_scaled_gemm(q.DGRAD, c5.qg_row, 1, 0, c5.sg.scale_inv, c5.qw_col, 0, 0,
                                               c5.sw.scale_inv, c5.dX), "gemm_tensor", c5.flops / 3, 1),
        ("c5_wgrad", lambda: q.fp8_scaled_gemm(q.WGRAD, c5.qg_col, 1, 0, c5.sg.scale_inv, c5.qx_col, 0, 0,
                                               c5.sx.scale_inv, c5.dW), "gemm_tensor", c5.flops / 3, 1),
        ("c5_history", c5.advance, "other", 0.0, 1),
        ("c4_quant", c4.quantize, "quant", float(c4.quant_bytes), 1),
        ("c4_gemm_mx", c4.gemm, "gemm_blockscaled", c4.flops, 1),
        ("c3_quant", c3.quantize, "quant", float(c3.quant_bytes), 1),
        ("c3_gemm_block", c3.gemm, "gemm_blockscaled", c3.flops, 1),
    ]
    step_flops = c1.flops + c5.flops + c4.flops + c3.flops
    quant_bytes = sum(w for _, _, k, w, _ in ops if k == "quant")
    launches_per_step = sum(n for *_, n in ops)

    stream = torch.cuda.current_stream()

    def step():
        for _, f, *_ in ops:
            f()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # --- timed region: device-resident inputs, events around every op ---
    nops = len(ops)

    def timed():
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nops + 1)] for _ in range(args.steps)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        with ClockSampler(dev.index) as sampler:
            start.record(stream)
            for s in range(args.steps):
                evs[s][0].record(stream)
                for i, (_, f, *_) in enumerate(ops):
                    f()
                    evs[s][i + 1].record(stream)
            end.record(stream)
            torch.cuda.synchronize()
        barrier(world)
        total = max_over_ranks(start.elapsed_time(end), world)
        op_ms = lambda s, i: evs[s][i].elapsed_time(evs[s][i + 1])
        ops_ms = {ops[i][0]: statistics.mean(op_ms(s, i) for s in range(args.steps)) for i in range(nops)}
        # the software power cap lowers the SM clock once the GPU has drawn its limit for some tens of
        # ms: the first timed step runs before it bites, the last ones under it
        late = range(max(1, args.steps - 5), args.steps)
        cap = {"first_step_ms": {ops[i][0]: round(op_ms(0, i), 4) for i in range(nops) if ops[i][2] != "other"},
               "last_steps_ms": ({ops[i][0]: round(statistics.mean(op_ms(s, i) for s in late), 4)
                                  for i in range(nops) if ops[i][2] != "other"} if len(late) else None)}
        return total, ops_ms, sampler.summary(), cap

    total_ms, per_op, clock_summary, power_cap = timed()
    suspect = clock_suspect(clock_summary)
    if max_over_ranks(1.0 if suspect else 0.0, world) > 0:
        total_ms, per_op, clock_summary, power_cap = timed()
        clock_summary["remeasured_after"] = suspect or ["another rank"]
    ms_step = total_ms / args.steps

    # the same steps without the per-op events (they cost the step nothing measurable)
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    a_ev.record(stream)
    for _ in range(args.steps):
        step()
    b_ev.record(stream)
    torch.cuda.synchronize()
    power_cap["ms_per_step_without_op_events"] = round(max_over_ranks(a_ev.elapsed_time(b_ev), world) / args.steps, 3)
    # the same step for about a second: NVML's clock reading lags by tens of ms, so a short timed region
    # is mostly sampled before the cap bites; this record shows the clock once it has
    power_cap["sustained"] = sustained_load(ops, stream, ms_step, dev.index, world)
    status = [int(c4.status.item()), int(c3.status.item())] + [int(s.status.item()) for s in (c5.sx, c5.sw, c5.sg)]

    # --- end to end: pinned host inputs in, results out, every step ---
    e2e = run_e2e(args, d, host, ops, stream, c1, c5, c4, c3, step_flops, world)

    pk, pk_src = peaks()
    long_loop = total_ms > 1500.0
    bf16_peak = pk["bf16_tflops_sustained" if long_loop else "bf16_tflops"]
    fp8_peak = bf16_peak * FP8_OVER_BF16
    tensor_ms = statistics.mean(per_op[n] for n in ("c5_fprop", "c5_dgrad", "c5_wgrad"))
    tensor_tflops = (c5.flops / 3) / (tensor_ms * 1e-3) / 1e12
    mx_tflops = c4.flops / (per_op["c4_gemm_mx"] * 1e-3) / 1e12
    blk_tflops = c3.flops / (per_op["c3_gemm_block"] * 1e-3) / 1e12
    quant_ms = sum(per_op[n] for n, _, k, *_ in ops if k == "quant")
    quant_gbs = quant_bytes / (quant_ms * 1e-3) / 1e9
    value = step_flops * world / (ms_step * 1e-3) / 1e12
    traffic = load_traffic("gemm_tensor_pair_kernel")
    prof = load_profile_record("gemm_tensor_pair_kernel")
    peak_note = f"{'sustained' if long_loop else 'burst'} bf16 x {FP8_OVER_BF16:g} (nominal fp8/bf16), {pk_src}"

    nxt = measure_next_rows(args, dev, c5, pk, stream) if not args.no_next_rows else None
    # context for the FP8 peak (2 x the measured bf16 cuBLAS figure): the library FP8 GEMM on the fprop
    # operands, measured here, and the committed ncu tensor-pipe activity of the fprop launch
    lib_fp8 = cublaslt_fp8_tflops(c5.qx_row, c5.qw_row, c5.sx.scale_inv, c5.sw.scale_inv)

    cpu = cpu_baseline(host, step_flops) if (rank == 0 and not args.no_cpu_baseline) else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (about 2 GB read per step), no flush",
                   "step_gemm_tflop": round(step_flops / 1e12, 3), "input_gen_s": round(gen_s, 1)},
        "roofline": {"bound": "tensor", "kernel": "gemm_tensor_pair_kernel (13B FFN fprop/dgrad/wgrad)",
                     "achieved": round(tensor_tflops, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(tensor_tflops / fp8_peak, 4), "peak_source": peak_note,
                     "traffic": traffic,
                     # context: the step runs under the power cap, where the measured sustained bf16
                     # figure (a seconds-long cuBLAS loop) is the like-for-like denominator
                     "frac_of_sustained": round(
                         tensor_tflops / (pk["bf16_tflops_sustained"] * FP8_OVER_BF16), 4),
                     # the peak is not a measured FP8 figure: beside it, the kernel's tensor-pipe
                     # activity from ncu (standalone launch) and cuBLASLt FP8 on the same operands
                     "ncu_tensor_pipe_active": (float(prof["tensor_pipe_active"])
                                                if "tensor_pipe_active" in prof else None),
                     "cublaslt_fp8_tflops_same_shape": lib_fp8},
        "roofline_quantizer": {"bound": "hbm", "kernel": "quantize_tile_kernel (all casts of the step)",
                               "achieved": round(quant_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                               "frac": round(quant_gbs / pk["hbm_gbs"], 4), "peak_source": pk_src,
                               "algorithmic_bytes_per_step": int(quant_bytes)},
        "roofline_blockscaled": {"bound": "tensor", "mxfp8_tflops": round(mx_tflops, 1),
                                 "mxfp8_frac": round(mx_tflops / fp8_peak, 4),
                                 "per_block_tflops": round(blk_tflops, 1),
                                 "per_block_frac": round(blk_tflops / fp8_peak, 4)},
        "breakdown_ms": {k: round(v, 4) for k, v in per_op.items()},
        "power_cap": power_cap,
        "next_rows": nxt,
        "device_status": status,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clock_summary,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def sustained_load(ops, stream, ms_step: float, gpu_index: int, world: int, seconds: float = 1.0) -> dict:
    """The step repeated for about `seconds` with the clock sampler on (not part of the timed region):
    steps, mean ms per step, the clock record, and each op's mean time over the last five steps."""
    import torch
    n = max(20, int(seconds * 1000.0 / max(ms_step, 1e-3)))
    tail = 5
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(tail)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_index) as sampler:
        a.record(stream)
        for k in range(n):
            t = k - (n - tail)
            if t >= 0:
                evs[t][0].record(stream)
            for i, (_, f, *_) in enumerate(ops):
                f()
                if t >= 0:
                    evs[t][i + 1].record(stream)
        b.record(stream)
        torch.cuda.synchronize()
    total = max_over_ranks(a.elapsed_time(b), world)
    last = {ops[i][0]: round(statistics.mean(evs[t][i].elapsed_time(evs[t][i + 1]) for t in range(tail)), 4)
            for i in range(len(ops)) if ops[i][2] != "other"}
    return {"steps": n, "seconds": round(total / 1e3, 3), "ms_per_step": round(total / n, 3),
            "clocks": sampler.summary(), "last_steps_ms": last}


def _time_op(f, reps: int, stream, warmup: int = 3) -> float:
    """Mean device ms of f() over `reps` launches (events on the launching stream), after warm-up."""
    import torch
    for _ in range(warmup):
        f()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        f()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def measure_next_rows(args, dev, c5, pk, stream):
    """The rows beyond the training step, each on its own, outside the timed step: the fused
    current-scaling cast, the fixed-bias (FP8-CSCALE) sweep statistics, the 16-iteration delayed-scaling
    workload (activation and gradient casts with their history updates), and post-training-quantised
    inference through two FP8 linear layers with the hidden cast fused into GEMM 1's epilogue."""
    import torch

    import scaling_quantization_gemm_gb300 as q
    import workloads as wl
    from scaling_quantization_gemm_gb300.step import PTQStack, bias_sweep
    hbm = pk["hbm_gbs"]
    fp8_peak = pk["bf16_tflops"] * FP8_OVER_BF16
    out = {}

    # fused current scaling, row + column casts of X (16384 x 5120): 2 B amax read + 2 B read + 2 x 1 B
    x = c5.X
    qr, qc = torch.empty_like(c5.qx_row), torch.empty_like(c5.qx_col)
    ws = q.current_workspace(dev)
    o = [torch.zeros(1, device=dev) for _ in range(3)] + [torch.zeros(1, dtype=torch.int32, device=dev)]
    ms = _time_op(lambda: q.fp8_quantize_current(x, q.E4M3, 0, ws, q_row=qr, q_col=qc, amax=o[0], scale=o[1],
                                                 scale_inv=o[2], bias=o[3]), 20, stream)
    gbs = 6.0 * x.numel() / (ms * 1e-3) / 1e9
    out["current_scaling_fused"] = {"kernel": "quantize_current_kernel (E4M3, row+col)", "shape": list(x.shape),
                                    "ms": round(ms, 4), "achieved": round(gbs, 1), "unit": "GB/s",
                                    "peak": hbm, "frac": round(gbs / hbm, 4), "bytes_per_elem": 6}

    # fixed-bias sweep e in [-3, 3] over the E5M2 gradient dY (16384 x 20480): one pass, 2 B / element
    y = c5.dY
    scales = torch.empty(7, device=dev)
    for j, e in enumerate(range(-3, 4)):
        q.fp8_set_bias(e, scale=scales[j:j + 1])
    sat = torch.zeros(7, dtype=torch.int64, device=dev)
    und = torch.zeros(7, dtype=torch.int64, device=dev)
    ms = _time_op(lambda: q.fp8_cast_stats(y, q.E5M2, scales, sat, und), 20, stream)
    gbs = 2.0 * y.numel() / (ms * 1e-3) / 1e9
    sweep = bias_sweep(y, q.E5M2, range(-3, 4))
    out["cscale_sweep_stats"] = {"kernel": "cast_stats_kernel (7 fixed biases, E5M2)", "shape": list(y.shape),
                                 "ms": round(ms, 4), "achieved": round(gbs, 1), "unit": "GB/s", "peak": hbm,
                                 "frac": round(gbs / hbm, 4), "bytes_per_elem": 2,
                                 "underflow_frac_by_e": {r["e"]: round(r["underflow_frac"], 6) for r in sweep}}

    # delayed scaling over 16 iterations: a 4096 x 4096 activation N(0, 1) (1 + 0.1 t) in E4M3 (margin 0)
    # and a 4096 x 4096 gradient Laplace(0, 1e-4) in E5M2 (margin 1), history length 16.  Each iteration
    # casts both row-wise with the scale the history gives and the fused amax (one batched launch), then
    # updates both histories in one launch.  The 32 distinct inputs (1 GB) exceed L2, so a pass needs no flush;
    # 3 B per element and tensor (2 B read, 1 B written)
    from scaling_quantization_gemm_gb300.step import ScaleState, current_scaling
    to = lambda b: torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
    acts = [to(wl.delayed_activation(t)) for t in range(16)]
    grads = [to(wl.delayed_gradient(t)) for t in range(16)]
    sa, sg = ScaleState(q.E4M3, 0, 16, dev), ScaleState(q.E5M2, 1, 16, dev)
    qa = torch.empty(4096, 4096, dtype=torch.uint8, device=dev)
    qg = torch.empty_like(qa)
    current_scaling(acts[0], sa)  # the first iteration's scale comes from its own amax (empty history)
    current_scaling(grads[0], sg)

    def delayed_pass():
        for t in range(16):
            q.fp8_quantize_batch([dict(x=acts[t], fmt=q.E4M3, gran=q.TENSOR, scale=sa.scale, q_row=qa, amax=sa.amax),
                                  dict(x=grads[t], fmt=q.E5M2, gran=q.TENSOR, scale=sg.scale, q_row=qg, amax=sg.amax)])
            q.fp8_amax_history_update_batch((sa, sg))

    # 32 small launches: replayed from a CUDA graph, so the host's per-call cost does not starve the GPU
    for _ in range(2):
        delayed_pass()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        delayed_pass()
    ms_eager = _time_op(delayed_pass, 10, stream)
    ms = _time_op(graph.replay, 10, torch.cuda.current_stream())
    nbytes = 16 * 2 * 3.0 * 4096 * 4096
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["delayed_scaling_16_iterations"] = {
        "kernel": "quantize_batch_kernel (E4M3 activation + E5M2 gradient, row-wise, fused amax) + history_batch_kernel",
        "shape": [4096, 4096], "iterations": 16, "history_len": 16, "launches_per_pass": 32,
        "ms_per_pass": round(ms, 4), "achieved": round(gbs, 1), "unit": "GB/s", "peak": hbm,
        "frac": round(gbs / hbm, 4), "bytes_per_elem": 3, "launch": "CUDA graph replay",
        "ms_per_pass_eager_launches": round(ms_eager, 4),
        "status": [int(sa.status.item()), int(sg.status.item())]}
    del acts, grads

    # PTQ inference: 8192 tokens through 5120 -> 13824 -> 5120, hidden cast in GEMM 1's epilogue
    Xb, W1b, W2b = wl.ptq_ffn()
    Xd = to(Xb)
    stack = PTQStack(to(W1b), to(W2b), Xb.shape[0], act="current")
    stack.forward(Xd)  # first forward: no hidden history yet (bf16 GEMM 1 + current scaling)
    ms = _time_op(lambda: stack.forward(Xd), 20, stream)
    T, F = stack.T, stack.F
    g1 = lambda: q.fp8_scaled_gemm_quantize(q.FPROP, stack.qx, q.E4M3, stack.sx.scale_inv, stack.qw1, q.E4M3,
                                            stack.sw1.scale_inv, stack.qh, q.E4M3, stack.sh.scale, stack.sh.amax)
    ms_g1 = _time_op(g1, 20, stream)
    tf_g1 = 2.0 * T * F * stack.H / (ms_g1 * 1e-3) / 1e12
    out["ptq_ffn_inference"] = {
        "workload": "8192 tokens, 13B FFN 5120 -> 13824 -> 5120, PTQ weights, current-scaled input",
        "ms_per_forward": round(ms, 4), "tflops": round(stack.flops / (ms * 1e-3) / 1e12, 1),
        "fused_epilogue_gemm": {"kernel": "gemm_tensor_pair_kernel<E4M3 out> (GEMM 1 + hidden cast + amax)",
                                "ms": round(ms_g1, 4), "achieved": round(tf_g1, 1), "unit": "TFLOP/s",
                                "peak": round(fp8_peak, 1), "frac": round(tf_g1 / fp8_peak, 4)},
        "status": int(stack.sh.status.item())}
    return out


def run_e2e(args, d, host, ops, stream, c1, c5, c4, c3, step_flops, world):
    """The step through the public API with host data: every step copies its inputs from pinned host
    memory to the device and its results (all GEMM outputs) back to pinned host memory.  Like an
    input pipeline, copies overlap computation: inputs and outputs are double-buffered on the device,
    step i+1's inputs go up on one copy stream and step i-1's results come down on another while step
    i computes on the compute stream; events order every reuse of a buffer."""
    import torch
    pinned_in = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory() for k, v in host.items()}
    out_names = [(c1, "Y"), (c5, "Y"), (c5, "dX"), (c5, "dW"), (c4, "Y"), (c3, "Y")]
    in_names = {"X1": (c1, "X"), "W1": (c1, "W"), "X5": (c5, "X"), "W5": (c5, "W"), "dY5": (c5, "dY"),
                "X4": (c4, "X"), "W4": (c4, "W"), "X3": (c3, "X"), "W3": (c3, "W")}
    dev_in = [d, {k: torch.empty_like(v) for k, v in d.items()}]
    dev_out = [[getattr(o, a) for o, a in out_names], [torch.empty_like(getattr(o, a)) for o, a in out_names]]
    pinned_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out[0]]
    h2d = sum(t.numel() * t.element_size() for t in pinned_in.values())
    d2h = sum(t.numel() * t.element_size() for t in pinned_out)
    steps = max(2, args.e2e_steps)
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    h2d_done = [ev() for _ in range(steps)]
    g_done = [ev() for _ in range(steps)]
    d2h_done = [ev() for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def upload(i):
        with torch.cuda.stream(s_h2d):
            if i >= 2:
                s_h2d.wait_event(g_done[i - 2])  # step i-2 no longer reads this input set
            for k, t in pinned_in.items():
                dev_in[i % 2][k].copy_(t, non_blocking=True)
            h2d_done[i].record(s_h2d)

    barrier(world)
    torch.cuda.synchronize()
    start.record(s_h2d)
    upload(0)
    for i in range(steps):
        if i + 1 < steps:
            upload(i + 1)
        k = i % 2
        for name, (obj, attr) in in_names.items():
            setattr(obj, attr, dev_in[k][name])
        for (obj, attr), t in zip(out_names, dev_out[k]):
            setattr(obj, attr, t)
        stream.wait_event(h2d_done[i])
        if i >= 2:
            stream.wait_event(d2h_done[i - 2])  # step i-2's results have left this output set
        for _, f, *_ in ops:
            f()
        g_done[i].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(g_done[i])
            for t, p in zip(dev_out[k], pinned_out):
                p.copy_(t, non_blocking=True)
            d2h_done[i].record(s_d2h)
    s_d2h.wait_event(d2h_done[steps - 1])
    end.record(s_d2h)
    torch.cuda.synchronize()
    for name, (obj, attr) in in_names.items():  # restore the resident buffers
        setattr(obj, attr, dev_in[0][name])
    for (obj, attr), t in zip(out_names, dev_out[0]):
        setattr(obj, attr, t)
    ms = max_over_ranks(start.elapsed_time(end), world) / steps
    return {"value": round(step_flops * world / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 3),
            "steps": steps, "copies": "overlapped with compute (double-buffered, two copy streams)"}


def load_profile_record(kernel: str) -> dict:
    """The committed ncu record of `kernel` at the benchmark shape (profiles/traffic.txt): DRAM bytes per
    launch and tensor-pipe activity, as a dict, or {} when the kernel source has changed since the
    capture (the figures would describe other code)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return {}
    for line in open(p):
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("kernel") != kernel:
            continue
        src = os.path.join(ROOT, "scaling_quantization_gemm_gb300", "csrc", f.get("source", ""))
        if not os.path.exists(src) or hashlib.sha1(open(src, "rb").read()).hexdigest() != f.get("source_sha1"):
            return {}
        return f
    return {}


def load_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from its profile record, or None (no record, or a stale one)."""
    f = load_profile_record(kernel)
    return int(f["bytes_per_launch"]) if "bytes_per_launch" in f else None


def cublaslt_fp8_tflops(A8: "torch.Tensor", B8: "torch.Tensor", sa, sb, reps: int = 10):
    """TFLOP/s of the library FP8 GEMM (torch._scaled_mm, cuBLASLt) on the same E4M3 operands and bf16
    output, outside the timed step: a comparison for the per-tensor kernel, never part of the path.
    None where the installed torch cannot run it."""
    import torch
    try:
        a = A8.view(torch.float8_e4m3fn)
        b = B8.view(torch.float8_e4m3fn).t()
        f = lambda: torch._scaled_mm(a, b, scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)
        ms = _time_op(f, reps, torch.cuda.current_stream())
    except (RuntimeError, AttributeError, TypeError):
        return None
    return round(2.0 * A8.shape[0] * B8.shape[0] * A8.shape[1] / (ms * 1e-3) / 1e12, 1)


# ------------------------------------------------------------- CPU oracle

def ffn_scales(host):
    """Delayed-scaling state of the FFN layer for the oracle's sampled steps: the scales the history
    gives once it holds these tensors' amaxes (computed once, before any timed step)."""
    import oracle as o
    return {k: o.scale_triple(o.amax(host[k]), f) for k, f in (("X5", 0), ("W5", 0), ("dY5", 1))}


def oracle_step_sample(host, R: int, ffn):
    """The oracle on a bounded sample of the step: for each of the six GEMMs, quantise R operand rows of
    A and B and compute the R x R block of outputs in fp64.  Per-tensor current scaling takes the amax
    of the whole (small) tensors; the delayed-scaling FFN layer casts with the scales of its history
    (`ffn`) and records the amax of the rows it casts; block scales come from the sampled rows.
    Returns (flops, seconds)."""
    import oracle as o
    t0 = time.time()
    flops = 0.0

    def tens(x_bits, fmt, margin=0):
        return o.scale_triple(o.amax(x_bits), fmt, margin)

    def gemm(Aq, fa, ga, sa, Bq, fb, gb, sb):
        nonlocal flops
        y, _ = o.gemm_full(Aq, fa, ga, sa, Bq, fb, gb, sb)
        flops += 2.0 * Aq.shape[0] * Bq.shape[0] * Aq.shape[1]
        return y

    # per-tensor current scaling fwd
    X1, W1 = host["X1"], host["W1"]
    _, s1x, i1x = tens(X1, 0)
    _, s1w, i1w = tens(W1, 0)
    gemm(o.quantize_tensor(X1[:R], 0, s1x)[0], 0, 0, i1x, o.quantize_tensor(W1[:R], 0, s1w)[0], 0, 0, i1w)
    # FFN fwd + bwd, per-tensor delayed scaling: scales from the history, amax of the cast rows recorded
    X5, W5, dY5 = host["X5"], host["W5"], host["dY5"]
    (_, sx, ix), (_, sw, iw), (_, sg, ig) = ffn["X5"], ffn["W5"], ffn["dY5"]
    for x in (X5[:R], W5[:R], dY5[:R]):
        o.amax(x)
    qx = o.quantize_tensor(X5[:R], 0, sx)[0]
    qw = o.quantize_tensor(W5[:R], 0, sw)[0]
    gemm(qx, 0, 0, ix, qw, 0, 0, iw)
    qg = o.quantize_tensor(dY5[:R], 1, sg)[0]
    qwc = o.quantize_tensor(np.ascontiguousarray(W5[:, :R]), 0, sw, row=False, col=True)[1]
    gemm(qg, 1, 0, ig, qwc, 0, 0, iw)
    qgc = o.quantize_tensor(np.ascontiguousarray(dY5[:, :R]), 1, sg, row=False, col=True)[1]
    qxc = o.quantize_tensor(np.ascontiguousarray(X5[:, :R]), 0, sx, row=False, col=True)[1]
    gemm(qgc, 1, 0, ig, qxc, 0, 0, ix)
    # MXFP8
    qa, sa, _, _, _ = o.quantize_block(host["X4"][:R], 0, o.MX_1x32)
    qb, sb, _, _, _ = o.quantize_block(host["W4"][:R], 0, o.MX_1x32)
    gemm(qa, 0, 3, sa, qb, 0, 3, sb)
    # per-block
    qa, sa, _, _, _ = o.quantize_block(host["X3"][:R], 0, o.BLOCK_1x128)
    qb, sb, _, _, _ = o.quantize_block(host["W3"][:R], 0, o.BLOCK_128x128)
    gemm(qa, 0, 1, sa, qb, 0, 2, sb)
    return flops, time.time() - t0


def cpu_baseline(host, step_flops: float, R: int = 512):
    import oracle as o
    o.lib()
    flops, sec = oracle_step_sample(host, R, ffn_scales(host))
    cores = o.max_threads()
    # the oracle's casts in every mode (per-tensor, 1x128, 128x128, MX 1x32; row + column-wise) on one
    # thread and on all cores, over 1024 rows of the FFN gradient (21 M elements); GB/s of algorithmic
    # bytes as for the GPU casts (2 B read + 1 B per copy written + the scale bytes)
    xs = np.ascontiguousarray(host["dY5"][:1024])
    scale = o.scale_triple(o.amax(xs), 1, 1)[1]
    modes = (("tensor", None, 4.0), ("1x128", o.BLOCK_1x128, 4.0 + 8.0 / 128),
             ("128x128", o.BLOCK_128x128, 4.0 + 8.0 / 16384), ("mx_1x32", o.MX_1x32, 4.0 + 2.0 / 32))
    cast_rates, by_mode = {}, {}
    for nthreads in (1, cores):
        o.set_threads(nthreads)
        total_b, total_s = 0.0, 0.0
        for name, gran, bpe in modes:
            t0 = time.time()
            if gran is None:
                o.quantize_tensor(xs, 1, scale, row=True, col=True)
            else:
                o.quantize_block(xs, 1, gran, 0, row=True, col=True)
            dt = time.time() - t0
            by_mode.setdefault(name, {})[str(nthreads)] = round(bpe * xs.size / dt / 1e9, 3)
            total_b += bpe * xs.size
            total_s += dt
        cast_rates[nthreads] = total_b / total_s / 1e9
    o.set_threads(cores)
    value = flops / sec
    return {"value": round(value / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{R}x{R} output block of each of the 6 GEMMs of the step, its operand rows cast by the "
                      f"oracle (current scaling from whole-tensor amax, the FFN layer from its delayed-scaling "
                      f"history); {flops / 1e9:.2f} GFLOP in {sec:.1f} s",
            "extrapolated_full_step_s": round(step_flops / value, 1),
            "cast_gbs_1_thread": round(cast_rates[1], 3), "cast_gbs_all_cores": round(cast_rates[cores], 3),
            "cast_gbs_by_mode": by_mode,
            "cast_sample": "casts in every mode (per-tensor, 1x128, 128x128, MX 1x32), row + column-wise, of "
                           "1024 x 20480 bf16 (the FFN gradient); the keys of cast_gbs_by_mode are thread counts"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle as o
    o.lib()
    host = make_inputs()
    ffn = ffn_scales(host)
    R = args.reference_rows
    if R <= 0:
        # size the sample so that the warm-up and timed steps take about two minutes together: the
        # oracle's work per step grows about as R^2 (an R x R output block of each GEMM)
        f0, t0 = oracle_step_sample(host, 64, ffn)
        per_step = REFERENCE_BUDGET_S / (args.warmup + args.steps)
        R = int(64 * math.sqrt(per_step / max(t0, 1e-6)))
        R = max(16, min(512, R - R % 16))
    for _ in range(args.warmup):
        oracle_step_sample(host, R, ffn)
    tot_f, tot_s = 0.0, 0.0
    for _ in range(args.steps):
        f, s = oracle_step_sample(host, R, ffn)
        tot_f += f
        tot_s += s
    v = tot_f / tot_s / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_s / args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"{R}x{R} output block per GEMM"},
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": o.max_threads(), "kind": "oracle",
                         "sample": f"{R}x{R} output block of each of the 6 GEMMs per step"},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------- profiling cases

def run_case(name: str, launches: int = 3) -> None:
    """One kernel on inputs larger than L2 but a few hundred MB in total, `launches` times (for ncu)."""
    import torch

    import scaling_quantization_gemm_gb300 as q
    torch.cuda.set_device(0)
    g = torch.Generator(device="cuda").manual_seed(0)
    kind, shape = PROFILE_CASES[name]
    if kind == "gemm_quant":
        M, N, K = shape
        A = torch.randint(0, 0x7E, (M, K), dtype=torch.uint8, device="cuda", generator=g)
        B = torch.randint(0, 0x7E, (N, K), dtype=torch.uint8, device="cuda", generator=g)
        Dq = torch.empty(M, N, dtype=torch.uint8, device="cuda")
        s = torch.full((1,), 2.0 ** -8, device="cuda")
        amax = torch.zeros(1, device="cuda")
        for _ in range(launches):
            q.fp8_scaled_gemm_quantize(q.FPROP, A, 0, s, B, 0, s, Dq, 0, s, amax)
    elif kind == "quant_current":
        R, C = shape
        x = torch.randn(R, C, device="cuda", generator=g).to(torch.bfloat16)
        qr = torch.empty(R, C, dtype=torch.uint8, device="cuda")
        qc = torch.empty(C, R, dtype=torch.uint8, device="cuda")
        ws = q.current_workspace()
        for _ in range(launches):
            q.fp8_quantize_current(x, 0, 0, ws, q_row=qr, q_col=qc)
    elif kind == "quant_batch_block":
        # the per-block recipe's two casts in one launch: X 1x128, W 128x128 (shape = X rows, W rows, K)
        R1, R2, C = shape
        xs = [torch.randn(R, C, device="cuda", generator=g).to(torch.bfloat16) for R in (R1, R2)]
        casts = [dict(x=xs[0], fmt=0, gran=q.BLOCK_1x128, q_row=torch.empty(R1, C, dtype=torch.uint8, device="cuda"),
                      sf_row=torch.empty(R1, C // 128, device="cuda")),
                 dict(x=xs[1], fmt=0, gran=q.BLOCK_128x128,
                      q_row=torch.empty(R2, C, dtype=torch.uint8, device="cuda"),
                      sf_row=torch.empty((R2 + 127) // 128, C // 128, device="cuda"))]
        for _ in range(launches):
            q.fp8_quantize_batch(casts)
    elif kind == "cast_stats":
        R, C = shape
        x = torch.randn(R, C, device="cuda", generator=g).to(torch.bfloat16)
        sc = torch.exp2(torch.arange(-3, 4, device="cuda").float())
        sat = torch.zeros(7, dtype=torch.int64, device="cuda")
        und = torch.zeros(7, dtype=torch.int64, device="cuda")
        for _ in range(launches):
            q.fp8_cast_stats(x, 1, sc, sat, und)
    elif kind.startswith("gemm"):
        M, N, K = shape
        A = torch.randint(0, 0x7E, (M, K), dtype=torch.uint8, device="cuda", generator=g)
        B = torch.randint(0, 0x7E, (N, K), dtype=torch.uint8, device="cuda", generator=g)
        D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        if kind == "gemm_tensor":
            sa = sb = torch.ones(1, device="cuda")
            ga = gb = q.TENSOR
        elif kind == "gemm_block":
            e = torch.randint(-4, 5, (M, K // 128), device="cuda", generator=g).float()
            sa = torch.exp2(e)
            sb = torch.exp2(torch.randint(-4, 5, ((N + 127) // 128, K // 128), device="cuda", generator=g).float())
            ga, gb = q.BLOCK_1x128, q.BLOCK_128x128
        else:
            sa = torch.randint(120, 135, (M, K // 32), dtype=torch.uint8, device="cuda", generator=g)
            sb = torch.randint(120, 135, (N, K // 32), dtype=torch.uint8, device="cuda", generator=g)
            ga = gb = q.MX_1x32
        for _ in range(launches):
            q.fp8_scaled_gemm(q.FPROP, A, 0, ga, sa, B, 0, gb, sb, D)
    else:
        R, C = shape
        x = torch.randn(R, C, device="cuda", generator=g).to(torch.bfloat16)
        qr = torch.empty(R, C, dtype=torch.uint8, device="cuda")
        qc = torch.empty(C, R, dtype=torch.uint8, device="cuda")
        amax = torch.zeros(1, device="cuda")
        sr = torch.empty(R, C // 32, dtype=torch.uint8, device="cuda")
        sc = torch.empty(C, R // 32, dtype=torch.uint8, device="cuda")
        one = torch.ones(1, device="cuda")
        for _ in range(launches):
            if kind == "quant_tensor":
                q.fp8_quantize(x, 0, q.TENSOR, scale=one, q_row=qr, q_col=qc, amax=amax)
            else:
                q.fp8_quantize(x, 0, q.MX_1x32, q_row=qr, q_col=qc, sf_row=sr, sf_col=sc)
    torch.cuda.synchronize()
    print(f"case {name} ok")


PROFILE_CASES = {
    "gemm_tensor": ("gemm_tensor", (16384, 8192, 8192)),
    "gemm_mx": ("gemm_mx", (16384, 8192, 8192)),
    "gemm_block": ("gemm_block", (8192, 11008, 4096)),
    "gemm_ffn_fprop": ("gemm_tensor", (16384, 20480, 5120)),
    "quant_tensor": ("quant_tensor", (16384, 8192)),
    "quant_mx": ("quant_mx", (16384, 8192)),
    "gemm_fused_q": ("gemm_quant", (8192, 13824, 5120)),
    "quant_current": ("quant_current", (16384, 5120)),
    "cast_stats": ("cast_stats", (16384, 8192)),
    "quant_batch_block": ("quant_batch_block", (8192, 11008, 4096)),
}


# -------------------------------------------------------------- plumbing

def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--reference-rows", type=int, default=0,
                    help="rows of each GEMM's operands the reference arm samples (0: sized to the step count)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true", help="skip the rows measured beside the step")
    ap.add_argument("--case", choices=sorted(PROFILE_CASES), default=None,
                    help="run one kernel on a small (> L2) case for an ncu capture, then exit")
    args = ap.parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            dist.init_process_group("nccl")
    if args.case:
        run_case(args.case)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
