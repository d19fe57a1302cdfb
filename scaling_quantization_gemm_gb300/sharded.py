"""Data-parallel sharding of the FP8 linear layer over ranks (one GPU per rank).

Tokens (the rows of X and dY) are split over the ranks and W is replicated, as
in data-parallel training.  Two exchanges are real:

* per-tensor scaling needs the amax of the whole tensor, so every rank's amax
  is all-reduced with MAX before the scale is derived.  For delayed scaling
  this happens after the step's casts, off the critical path: the scale the
  next step uses is the same on every rank because the histories record the
  same reduced amax.  For current scaling (and the first delayed step, whose
  history is empty) the reduction sits between the amax pass and the cast.
* the weight gradient is a sum over all tokens, so the ranks' partial dW are
  all-reduced with SUM.

The collectives run on torch.distributed (NCCL between GPUs, gloo in the CPU
tests) on the caller's current stream, ordered with the library's kernels,
which run on the same stream.  Method: "Training and inference of large
language models using 8-bit floating point", "Proposed method" (per-tensor
scales from each tensor's amax; the scaled FP8 products of a linear layer).
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

from . import E4M3, E5M2, TENSOR, fp8_amax, fp8_amax_history_update_batch, fp8_compute_scale, fp8_quantize
from .step import LinearFwdBwd


def allreduce_amax_(amax: torch.Tensor, group: Optional[dist.ProcessGroup] = None) -> torch.Tensor:
    """In place: amax <- max over ranks (fp32).

    An amax is |x| of some element: a non-negative float, +Inf or a NaN with the sign bit clear, whose
    bit patterns, read as int32, order exactly as the values do, with every NaN above +Inf.  The
    reduction is a MAX over those integers, so a NaN on any rank reaches every rank (a floating-point
    MAX keeps or drops a NaN depending on the order of its operands)."""
    if dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(amax.view(torch.int32), op=dist.ReduceOp.MAX, group=group)
    return amax


def allreduce_sum_(t: torch.Tensor, group: Optional[dist.ProcessGroup] = None) -> torch.Tensor:
    """In place: t <- sum over ranks (the weight gradient's reduction over the data-parallel ranks)."""
    if dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return t


class ShardedLinearFwdBwd(LinearFwdBwd):
    """`LinearFwdBwd` on this rank's tokens: X [M_r x K] and dY [M_r x N] are the rank's rows, W
    [N x K] is replicated.  Scales are those of the whole (all-rank) tensors; dW is the sum over all
    ranks (fp32).  With one rank it computes exactly what `LinearFwdBwd` computes."""

    def __init__(self, X: torch.Tensor, W: torch.Tensor, dY: torch.Tensor, history_len: int,
                 group: Optional[dist.ProcessGroup] = None, **kw):
        super().__init__(X, W, dY, history_len, **kw)
        self.group = group

    def quantize_one(self, i: int) -> None:
        x, st, qr, qc = ((self.X, self.sx, self.qx_row, self.qx_col), (self.W, self.sw, self.qw_row, self.qw_col),
                         (self.dY, self.sg, self.qg_row, self.qg_col))[i]
        if st.steps == 0:
            # empty history: the scale of this step needs the whole tensor's amax before the cast
            st.amax.zero_()
            fp8_amax(x, st.amax)
            allreduce_amax_(st.amax, self.group)
            fp8_compute_scale(st.amax, st.fmt, st.margin, st.bias, st.scale, st.scale_inv, st.status)
            fp8_quantize(x, st.fmt, TENSOR, scale=st.scale, q_row=qr, q_col=qc)
        else:
            fp8_quantize(x, st.fmt, TENSOR, scale=st.scale, q_row=qr, q_col=qc, amax=st.amax)

    def gemms(self) -> None:
        super().gemms()
        allreduce_sum_(self.dW, self.group)

    def advance(self) -> None:
        # the first step's amax is already the reduced one; later steps reduce the fused local amax
        states = (self.sx, self.sw, self.sg)
        for st in states:
            if st.steps > 0:
                allreduce_amax_(st.amax, self.group)
        fp8_amax_history_update_batch(states)
        for st in states:
            st.steps += 1


__all__ = ["allreduce_amax_", "allreduce_sum_", "ShardedLinearFwdBwd", "E4M3", "E5M2"]
