"""Host-side sequencing of the FP8 hot path over the C entry points.

Nothing here computes: each function enqueues library kernels on the current
CUDA stream in the method's order: scale, cast to FP8, multiply, unscale
("Training and inference of large language models using 8-bit floating
point", "Proposed method").  Device
buffers are torch tensors; torch is only the allocator.

* ``ScaleState`` holds one tensor's scaling state on the device: the amax
  accumulator, bias, scale 2^e and scale_inv 2^-e, plus the amax history ring
  and its position for delayed scaling.
* ``current_scaling`` runs amax -> compute_scale (the FP8-AMAX rule);
  ``quantize_current`` does that and the cast in one fused launch.
* ``LinearFwdBwd`` is one FP8 linear layer, forward and backward, with
  per-tensor delayed scaling: quantise X, W (E4M3) and dY (E5M2) row- and
  column-wise with the fused amax, run fprop / dgrad / wgrad, then advance
  the three histories.  On its first step a history is empty, so that step
  uses current scaling (the fused amax + scale + cast).
* ``BlockLinearFwd`` is the forward with per-block (1x128 activations,
  128x128 weights) or MXFP8 (1x32, E8M0) scales.
* ``bias_sweep`` casts a tensor at a range of fixed (FP8-CSCALE) biases and
  reports, per bias, how many elements saturate and how many flush to zero
  ("Training and inference of large language models using 8-bit floating
  point", "Key findings": the fixed-scaling sweep).
* ``PTQStack`` is post-training-quantised inference through two FP8 linear
  layers: weights cast once, the input cast per forward (current or delayed
  scaling), the hidden activation cast in the first GEMM's epilogue with its
  delayed scale ("Training and inference of large language models using 8-bit
  floating point", "Proposed method": inference with post-training
  quantization, scaling before and unscaling after each FP8 product).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import (BLOCK_1x128, BLOCK_128x128, DGRAD, E4M3, E5M2, FPROP, MX_1x32, MX_1x32_OCP, TENSOR, WGRAD,
               current_workspace, fp8_amax, fp8_amax_history_update, fp8_amax_history_update_batch, fp8_cast_stats,
               fp8_compute_scale, fp8_compute_scale_ratio, fp8_quantize, fp8_quantize_batch, fp8_quantize_current,
               fp8_scaled_gemm, fp8_scaled_gemm_quantize, fp8_set_bias)


class ScaleState:
    def __init__(self, fmt: int, margin: int, history_len: int = 0, device="cuda"):
        self.fmt, self.margin = fmt, margin
        self.amax = torch.zeros(1, dtype=torch.float32, device=device)
        self.bias = torch.zeros(1, dtype=torch.int32, device=device)
        self.scale = torch.ones(1, dtype=torch.float32, device=device)
        self.scale_inv = torch.ones(1, dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.history = torch.zeros(max(history_len, 1), dtype=torch.float32, device=device) if history_len else None
        self.pos = torch.zeros(1, dtype=torch.int64, device=device) if history_len else None
        self.steps = 0  # host-side count of completed delayed steps

    def advance(self) -> None:
        """One delayed-scaling update: record amax, next scale from the window max, reset amax."""
        fp8_amax_history_update(self.history, self.pos, self.amax, self.fmt, self.margin, self.bias, self.scale,
                                self.scale_inv, self.status)
        self.steps += 1


def current_scaling(x: torch.Tensor, st: ScaleState) -> None:
    """amax of x, then compute_bias -> (bias, scale, scale_inv) in st."""
    st.amax.zero_()
    fp8_amax(x, st.amax)
    fp8_compute_scale(st.amax, st.fmt, st.margin, st.bias, st.scale, st.scale_inv, st.status)
    st.amax.zero_()


def quantize_current(x: torch.Tensor, st: ScaleState, ws: torch.Tensor, q_row=None, q_col=None) -> None:
    """Current scaling and the cast in one launch: st.amax = max|x|, st.bias/scale/scale_inv from it."""
    fp8_quantize_current(x, st.fmt, st.margin, ws, q_row=q_row, q_col=q_col, amax=st.amax, bias=st.bias,
                         scale=st.scale, scale_inv=st.scale_inv, status=st.status)


def bias_sweep(x: torch.Tensor, fmt: int, biases=range(-3, 4)) -> list:
    """Fixed biases e (FP8-CSCALE) on tensor x: one pass over x per 8 biases.  Returns, per e, the
    number and fraction of elements the cast saturates and flushes to zero."""
    biases = list(biases)
    dev = x.device
    out = []
    for i in range(0, len(biases), 8):
        chunk = biases[i:i + 8]
        scales = torch.empty(len(chunk), dtype=torch.float32, device=dev)
        for j, e in enumerate(chunk):
            fp8_set_bias(e, scale=scales[j:j + 1])
        sat = torch.zeros(len(chunk), dtype=torch.int64, device=dev)
        und = torch.zeros(len(chunk), dtype=torch.int64, device=dev)
        fp8_cast_stats(x, fmt, scales, sat, und)
        for e, s_, u in zip(chunk, sat.tolist(), und.tolist()):
            out.append({"e": e, "saturated": s_, "underflow": u, "saturated_frac": s_ / max(x.numel(), 1),
                        "underflow_frac": u / max(x.numel(), 1)})
    return out


def gemm_flops(m: int, n: int, k: int) -> float:
    return 2.0 * m * n * k


@dataclass
class PerTensorFwd:
    """Per-tensor current-scaling forward: Y[M x N] fp32 = unscale(Q(X) Q(W)^T).  `scale_rule`
    "pow2" is the compute_bias rule (one fused launch per cast); "ratio" is the alternative
    s = fmax / amax (amax, ratio, cast: three launches)."""
    X: torch.Tensor
    W: torch.Tensor
    margin: int = 0
    scale_rule: str = "pow2"

    def __post_init__(self):
        dev = self.X.device
        M, K = self.X.shape
        N = self.W.shape[0]
        self.sx, self.sw = ScaleState(E4M3, self.margin, device=dev), ScaleState(E4M3, self.margin, device=dev)
        self.qx = torch.empty(M, K, dtype=torch.uint8, device=dev)
        self.qw = torch.empty(N, K, dtype=torch.uint8, device=dev)
        self.Y = torch.empty(M, N, dtype=torch.float32, device=dev)
        self.ws = current_workspace(dev)
        self.flops = gemm_flops(M, N, K)

    def run(self) -> None:
        for x, st, q in ((self.X, self.sx, self.qx), (self.W, self.sw, self.qw)):
            if self.scale_rule == "ratio":
                st.amax.zero_()
                fp8_amax(x, st.amax)
                fp8_compute_scale_ratio(st.amax, st.fmt, st.scale, st.scale_inv, st.status)
                fp8_quantize(x, st.fmt, TENSOR, scale=st.scale, q_row=q)
            else:
                quantize_current(x, st, self.ws, q_row=q)
        fp8_scaled_gemm(FPROP, self.qx, E4M3, TENSOR, self.sx.scale_inv, self.qw, E4M3, TENSOR, self.sw.scale_inv,
                        self.Y)


class LinearFwdBwd:
    """FP8 linear layer forward + backward with per-tensor delayed scaling.

    X [M x K] and W [N x K] in E4M3, dY [M x N] in E5M2 (margin `grad_margin`).
    Y  [M x N] bf16 = unscale(QX_row . QW_row^T)            (fprop)
    dX [M x K] bf16 = unscale(QdY_row . QW_col^T)           (dgrad)
    dW [N x K] fp32 = unscale(QdY_col . QX_col^T)           (wgrad)
    """

    def __init__(self, X: torch.Tensor, W: torch.Tensor, dY: torch.Tensor, history_len: int, margin: int = 0,
                 grad_margin: int = 0, dw_dtype=torch.float32, first_step: str = "current"):
        # first_step: the empty-history step scales from its own amax ("current"), or with the fixed
        # bias e = 0, scale 1 ("fixed", the alternative)
        assert first_step in ("current", "fixed")
        self.first_step = first_step
        dev = X.device
        M, K = X.shape
        N = W.shape[0]
        assert W.shape[1] == K and dY.shape == (M, N)
        self.X, self.W, self.dY = X, W, dY
        self.sx = ScaleState(E4M3, margin, history_len, dev)
        self.sw = ScaleState(E4M3, margin, history_len, dev)
        self.sg = ScaleState(E5M2, grad_margin, history_len, dev)
        u8 = dict(dtype=torch.uint8, device=dev)
        self.qx_row, self.qx_col = torch.empty(M, K, **u8), torch.empty(K, M, **u8)
        self.qw_row, self.qw_col = torch.empty(N, K, **u8), torch.empty(K, N, **u8)
        self.qg_row, self.qg_col = torch.empty(M, N, **u8), torch.empty(N, M, **u8)
        self.Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        self.dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty(N, K, dtype=dw_dtype, device=dev)
        self.ws = current_workspace(dev)
        self.flops = 3 * gemm_flops(M, N, K)
        self.quant_bytes = 4 * (M * K + N * K + M * N)  # 2 B read + 1 B row + 1 B col per element

    def quantize_one(self, i: int) -> None:
        x, st, qr, qc = ((self.X, self.sx, self.qx_row, self.qx_col), (self.W, self.sw, self.qw_row, self.qw_col),
                         (self.dY, self.sg, self.qg_row, self.qg_col))[i]
        if st.steps == 0 and self.first_step == "current":
            quantize_current(x, st, self.ws, q_row=qr, q_col=qc)  # empty history: scale from its own amax
        else:  # delayed scale (or the initial scale 1 for a fixed first step), amax recorded
            fp8_quantize(x, st.fmt, TENSOR, scale=st.scale, q_row=qr, q_col=qc, amax=st.amax)

    def quantize(self) -> None:
        """The three casts.  Once every history holds a scale (or with the fixed first step), they are
        one batched launch: each cast uses its delayed scale and records its amax."""
        states = (self.sx, self.sw, self.sg)
        if self.first_step == "fixed" or all(st.steps > 0 for st in states):
            fp8_quantize_batch(
                dict(x=x, fmt=st.fmt, gran=TENSOR, scale=st.scale, q_row=qr, q_col=qc, amax=st.amax)
                for x, st, qr, qc in ((self.X, self.sx, self.qx_row, self.qx_col),
                                      (self.W, self.sw, self.qw_row, self.qw_col),
                                      (self.dY, self.sg, self.qg_row, self.qg_col)))
        else:
            for i in range(3):
                self.quantize_one(i)

    def gemms(self) -> None:
        fp8_scaled_gemm(FPROP, self.qx_row, E4M3, TENSOR, self.sx.scale_inv, self.qw_row, E4M3, TENSOR,
                        self.sw.scale_inv, self.Y)
        fp8_scaled_gemm(DGRAD, self.qg_row, E5M2, TENSOR, self.sg.scale_inv, self.qw_col, E4M3, TENSOR,
                        self.sw.scale_inv, self.dX)
        fp8_scaled_gemm(WGRAD, self.qg_col, E5M2, TENSOR, self.sg.scale_inv, self.qx_col, E4M3, TENSOR,
                        self.sx.scale_inv, self.dW)

    def advance(self) -> None:
        """The three delayed-scaling updates in one launch."""
        states = (self.sx, self.sw, self.sg)
        fp8_amax_history_update_batch(states)
        for st in states:
            st.steps += 1

    def run(self) -> None:
        self.quantize()
        self.gemms()
        self.advance()


class BlockLinearFwd:
    """Forward with block scales: per-block (X 1x128, W 128x128, fp32 scales) or MXFP8 (1x32, E8M0).

    Y [M x N] bf16 = sum_k (QX sx)(QW sw).  With `col=True` the column-wise (transposed) copies and
    their scales are produced too, as the backward pass would need them."""

    def __init__(self, X: torch.Tensor, W: torch.Tensor, mx: bool, col: bool = False, margin: int = 0,
                 mx_rule: str = "compute_bias"):
        # mx_rule "ocp": MX blocks with the OCP MX bias rule (the alternative), same E8M0 storage
        dev = X.device
        M, K = X.shape
        N = W.shape[0]
        self.X, self.W, self.mx, self.col, self.margin = X, W, mx, col, margin
        mxg = MX_1x32_OCP if mx_rule == "ocp" else MX_1x32
        self.gx = mxg if mx else BLOCK_1x128
        self.gw = mxg if mx else BLOCK_128x128
        u8 = dict(dtype=torch.uint8, device=dev)
        sdt = dict(dtype=torch.uint8 if mx else torch.float32, device=dev)
        cd = lambda a, b: (a + b - 1) // b
        self.qx_row, self.qw_row = torch.empty(M, K, **u8), torch.empty(N, K, **u8)
        if mx:
            self.sx_row, self.sw_row = torch.empty(M, cd(K, 32), **sdt), torch.empty(N, cd(K, 32), **sdt)
        else:
            self.sx_row, self.sw_row = torch.empty(M, cd(K, 128), **sdt), torch.empty(cd(N, 128), cd(K, 128), **sdt)
        if col:
            self.qx_col, self.qw_col = torch.empty(K, M, **u8), torch.empty(K, N, **u8)
            if mx:
                self.sx_col, self.sw_col = torch.empty(K, cd(M, 32), **sdt), torch.empty(K, cd(N, 32), **sdt)
            else:
                self.sx_col = torch.empty(K, cd(M, 128), **sdt)
                self.sw_col = torch.empty(cd(K, 128), cd(N, 128), **sdt)
        else:
            self.qx_col = self.qw_col = self.sx_col = self.sw_col = None
        self.Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.flops = gemm_flops(M, N, K)
        ncopies = 2 if col else 1
        sbytes = lambda rows, cols, g: _scale_bytes(rows, cols, g)
        self.quant_bytes = 2 * (M * K + N * K) + ncopies * (M * K + N * K) + sbytes(M, K, self.gx) + \
            sbytes(N, K, self.gw) + (sbytes(K, M, self.gx) + sbytes(K, N, self.gw) if col else 0)

    def quantize(self) -> None:
        """Both casts in one batched launch."""
        fp8_quantize_batch([
            dict(x=self.X, fmt=E4M3, gran=self.gx, margin=self.margin, q_row=self.qx_row, q_col=self.qx_col,
                 sf_row=self.sx_row, sf_col=self.sx_col),
            dict(x=self.W, fmt=E4M3, gran=self.gw, margin=self.margin, q_row=self.qw_row, q_col=self.qw_col,
                 sf_row=self.sw_row, sf_col=self.sw_col)])

    def gemm(self) -> None:
        fp8_scaled_gemm(FPROP, self.qx_row, E4M3, self.gx, self.sx_row, self.qw_row, E4M3, self.gw, self.sw_row,
                        self.Y, status=self.status)

    def run(self) -> None:
        self.quantize()
        self.gemm()


class PTQStack:
    """Inference through two FP8 linear layers with post-training quantisation.

    W1 [F x H] and W2 [H x F] are cast to E4M3 once, with current scaling, when the stack is
    built.  Each forward on X [T x H]:
      QX = cast(X)                      current scaling (fused kernel), or delayed (`act="delayed"`)
      QH = cast(unscale(QX . QW1^T))    in GEMM 1's epilogue, with the hidden activation's delayed
                                        scale; its amax is folded in and recorded afterwards
      Y  = unscale(QH . QW2^T)          bf16 [T x H]
    The first forward has no hidden history: GEMM 1 writes bf16 and the hidden activation is cast
    from its own amax (current scaling); later forwards use the fused epilogue.  No nonlinearity
    sits between the layers (the method concerns the linear layers only)."""

    def __init__(self, W1: torch.Tensor, W2: torch.Tensor, tokens: int, act: str = "current",
                 history_len: int = 16):
        dev = W1.device
        F, H = W1.shape
        assert W2.shape == (H, F) and act in ("current", "delayed")
        self.act, self.T, self.H, self.F = act, tokens, H, F
        u8 = dict(dtype=torch.uint8, device=dev)
        self.ws = current_workspace(dev)
        self.sw1, self.sw2 = ScaleState(E4M3, 0, device=dev), ScaleState(E4M3, 0, device=dev)
        self.qw1, self.qw2 = torch.empty(F, H, **u8), torch.empty(H, F, **u8)
        quantize_current(W1, self.sw1, self.ws, q_row=self.qw1)  # once: post-training quantisation
        quantize_current(W2, self.sw2, self.ws, q_row=self.qw2)
        self.sx = ScaleState(E4M3, 0, history_len if act == "delayed" else 0, dev)
        self.sh = ScaleState(E4M3, 0, history_len, dev)
        self.qx, self.qh = torch.empty(tokens, H, **u8), torch.empty(tokens, F, **u8)
        self.h_bf16: Optional[torch.Tensor] = None  # first forward only
        self.Y = torch.empty(tokens, H, dtype=torch.bfloat16, device=dev)
        self.flops = gemm_flops(tokens, F, H) + gemm_flops(tokens, H, F)

    def forward(self, X: torch.Tensor) -> torch.Tensor:
        sx, sh = self.sx, self.sh
        if self.act == "current" or sx.steps == 0:
            quantize_current(X, sx, self.ws, q_row=self.qx)
        else:
            fp8_quantize(X, E4M3, TENSOR, scale=sx.scale, q_row=self.qx, amax=sx.amax)
        if sh.steps == 0:
            if self.h_bf16 is None:
                self.h_bf16 = torch.empty(self.T, self.F, dtype=torch.bfloat16, device=X.device)
            fp8_scaled_gemm(FPROP, self.qx, E4M3, TENSOR, sx.scale_inv, self.qw1, E4M3, TENSOR, self.sw1.scale_inv,
                            self.h_bf16)
            quantize_current(self.h_bf16, sh, self.ws, q_row=self.qh)
        else:
            fp8_scaled_gemm_quantize(FPROP, self.qx, E4M3, sx.scale_inv, self.qw1, E4M3, self.sw1.scale_inv, self.qh,
                                     E4M3, sh.scale, sh.amax, status=sh.status)
        fp8_scaled_gemm(FPROP, self.qh, E4M3, TENSOR, sh.scale_inv, self.qw2, E4M3, TENSOR, self.sw2.scale_inv,
                        self.Y)
        sh.advance()
        if self.act == "delayed":
            sx.advance()
        return self.Y


def _scale_bytes(rows: int, cols: int, gran: int) -> int:
    cd = lambda a, b: (a + b - 1) // b
    if gran in (MX_1x32, MX_1x32_OCP):
        return rows * cd(cols, 32)
    if gran == BLOCK_1x128:
        return 4 * rows * cd(cols, 128)
    if gran == BLOCK_128x128:
        return 4 * cd(rows, 128) * cd(cols, 128)
    return 0
