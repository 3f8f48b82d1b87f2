"""The op interface of ROCm/mori's dispatch/combine over the library's
stateless calls.

ROCm/mori "Draft: cco + flydsl dispatch/combine #448" drives the path
through one op object (the op notes and the routing-handle note):

    out, total_recv, routing = op.dispatch(x, topk_w, topk_idx)
    y = experts(out, routing)                  # the caller's expert stage
    combined, combined_wts = op.combine(y, routing)

MoeOp gives that shape on one GPU with every expert local.  The routing
handle is the plan's buffers plus the weights, held by the caller: the op
keeps nothing between calls, so any number of dispatches may be in flight,
each with its own handle, and replaying a combine (or a second dispatch with
the same map) needs only the handle.  Every step runs in the library's
kernels; this module only chooses the calls and allocates their outputs.

Modes (fixed when the op is made):
  plain     moe_plan_dispatch (one launch for small batches); fp8 rows with
            per-block scales (x_scales) travel together
  quant     bf16 rows -> E4M3 codes + one f32 scale per `quant_block`
            elements (moe_plan, moe_dispatch_quant_fp8)
  capacity  padded buckets of `capacity` rows, entries past a bucket's
            capacity dropped in token order (moe_plan_capacity, then the
            plain or quantising dispatch)
  dedup     one copy per (token, virtual group of `group_size` experts),
            expanded per expert (moe_plan or moe_plan_capacity,
            moe_group_plan, moe_dispatch_dedup, moe_combine_dedup)

combine: weighted (sum_k w[s,k] * y[row]) or unweighted (the sum of the
copies: the op notes' identity round trip), both in f32 in increasing k;
combined_wts[s,i] is the sum of topk_w[s,i] over the token's valid copies
(the weight fold).  In dedup mode the weights are applied inside each group
row and the group rows are summed unweighted; the fold there takes a second
pass over the group rows.
"""
from __future__ import annotations

from typing import NamedTuple, Optional

import torch

from . import (GroupPlan, moe_combine_dedup, moe_combine_fold, moe_dispatch,
               moe_dispatch_dedup, moe_dispatch_quant_fp8, moe_group_plan, moe_plan,
               moe_plan_capacity, moe_plan_dispatch)

__all__ = ["MoeOp", "Routing"]


class Routing(NamedTuple):
    """The routing handle of one dispatch."""
    plan: object                 # Plan, or CapacityPlan in capacity mode
    topk_w: torch.Tensor         # f32 [S, K], as passed to dispatch
    group: Optional[GroupPlan]   # dedup mode only
    rows: int                    # rows of the dispatch output buffers


class MoeOp:
    def __init__(self, num_experts: int, *, capacity: int = 0, group_size: int = 0,
                 quant_block: int = 0, weighted: bool = True, fold: bool = True,
                 out_dtype: torch.dtype = torch.bfloat16):
        if not 1 <= num_experts <= 1024:
            raise ValueError("num_experts must be in 1..1024")
        if capacity < 0 or group_size < 0 or quant_block < 0:
            raise ValueError("capacity, group_size and quant_block must be >= 0")
        if group_size and num_experts % group_size:
            raise ValueError("group_size must divide num_experts")
        if quant_block and (quant_block & (quant_block - 1) or not 16 <= quant_block <= 256):
            raise ValueError("quant_block must be a power of two in 16..256")
        if quant_block and group_size:
            raise ValueError("the dedup path moves rows as they are: no quantising dispatch")
        if out_dtype not in (torch.bfloat16, torch.float32):
            raise ValueError("out_dtype must be bfloat16 or float32")
        self.E = num_experts
        self.capacity = capacity
        self.group_size = group_size
        self.quant_block = quant_block
        self.weighted = weighted
        self.fold = fold
        self.out_dtype = out_dtype

    def dispatch(self, x: torch.Tensor, topk_w: torch.Tensor, topk_idx: torch.Tensor, *,
                 x_scales: Optional[torch.Tensor] = None, stream=None):
        """Returns (out, total_recv, routing).  out is the packed rows, or
        (rows, scales) when scales travel or are made; total_recv is a
        one-element device tensor, off[E]: the rows the expert stage must
        process (the valid rows, or E * capacity padded rows in capacity
        mode, whose per-bucket fill is routing.plan.cnt)."""
        if topk_idx.dtype == torch.int64:
            topk_idx = topk_idx.to(torch.int32)   # expert ids below 1024
        if topk_idx.dtype != torch.int32 or topk_idx.dim() != 2:
            raise TypeError("topk_idx must be an integer [S, K] tensor")
        if topk_w.dtype != torch.float32 or tuple(topk_w.shape) != tuple(topk_idx.shape):
            raise TypeError("topk_w must be float32 with the shape of topk_idx")
        if (self.quant_block or self.group_size) and x_scales is not None:
            raise ValueError("x_scales travel with the plain or capacity dispatch only")
        E = self.E
        S, K = topk_idx.shape
        H = x.shape[1]
        dev = x.device
        scales = None
        group = None
        if self.capacity:
            plan = moe_plan_capacity(topk_idx, E, self.capacity, stream=stream)
            rows = E * self.capacity
        elif self.group_size or self.quant_block:
            plan = moe_plan(topk_idx, E, stream=stream)
            rows = max(S * K, 1)
        else:
            plan, packed, scales = moe_plan_dispatch(topk_idx, x, E, x_scales=x_scales,
                                                     stream=stream)
            rows = packed.shape[0]
        if self.group_size:
            group = moe_group_plan(topk_idx, plan.tok_map, E, self.group_size, stream=stream)
            packed = torch.empty(rows, H, dtype=x.dtype, device=dev)
            moe_dispatch_dedup(x, group, packed_x=packed, stream=stream)
        elif self.quant_block:
            packed = torch.empty(rows, H, dtype=torch.float8_e4m3fn, device=dev)
            scales = torch.empty(rows, H // self.quant_block, dtype=torch.float32, device=dev)
            moe_dispatch_quant_fp8(x, plan.tok_map, block=self.quant_block, packed_q=packed,
                                   packed_scales=scales, stream=stream)
        elif self.capacity:
            packed = torch.empty(rows, H, dtype=x.dtype, device=dev)
            if x_scales is not None:
                scales = torch.empty(rows, x_scales.shape[1], dtype=torch.float32, device=dev)
            moe_dispatch(x, plan.tok_map, packed_x=packed, x_scales=x_scales,
                         packed_scales=scales, stream=stream)
        out = packed if scales is None else (packed, scales)
        return out, plan.off[E:], Routing(plan, topk_w, group, rows)

    def combine(self, y: torch.Tensor, routing: Routing, *, stream=None):
        """Returns (combined [S, H] in out_dtype, combined_wts [S, K] f32 or
        None when the op was made with fold=False)."""
        if y.shape[0] < 1 or y.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("y must be bfloat16 or float32 rows")
        if routing.group is not None:
            gp = routing.group
            gtok, out = moe_combine_dedup(y, routing.topk_w, gp, out_dtype=self.out_dtype,
                                          stream=stream)
            if not self.fold:
                return out, None
            # the fold: the group rows summed once more, with the weights of
            # the copies; the same sums in the same order as the dedup
            # combine's second stage, so `out` is rewritten with equal bits
            return moe_combine_fold(gtok, routing.topk_w, gp.gtok_map, weighted=False,
                                    fold=True, out=out, stream=stream)
        return moe_combine_fold(y, routing.topk_w, routing.plan.tok_map,
                                weighted=self.weighted, fold=self.fold,
                                out_dtype=self.out_dtype, stream=stream)
