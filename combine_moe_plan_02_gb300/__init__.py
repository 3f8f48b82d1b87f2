"""Single-GPU MoE token dispatch and combine for GB300 (sm_103a).

Python binding of the C ABI in include/moe_plan.h: each function checks and
marshals torch tensors (device pointers, sizes, the current stream) into one
C call; all work runs in the library's CUDA kernels.  Output tensors are
allocated with torch when not passed in.

    plan  = moe_plan(topk_idx, E)                  # counts, offsets, maps
    px, _ = moe_dispatch(x, plan.tok_map)          # packed_x[off[e] + slot]
    y     = experts(px, plan)                      # caller's expert stage
    out   = moe_combine(y, topk_w, plan.tok_map)   # sum_k w * y[tok_map]
"""
from __future__ import annotations

from typing import NamedTuple, Optional

import torch

from . import _abi
from ._abi import MoeError, MOE_BF16, MOE_F32, MOE_FP8_E4M3  # noqa: F401

__all__ = [
    "moe_plan", "moe_group_plan", "moe_dispatch", "moe_plan_dispatch", "moe_dispatch_dedup", "moe_dispatch_quant_fp8",
    "moe_combine", "moe_combine_fold",
    "moe_combine_dedup", "moe_plan_workspace_size", "moe_group_plan_workspace_size",
    "moe_device_errors", "moe_plan_capacity", "Plan", "GroupPlan", "CapacityPlan", "MoeError",
    "MoeOp", "Routing", "lib",
]


def lib():
    return _abi.load()


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return MOE_FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


_TORCH_DT = {MOE_BF16: torch.bfloat16, MOE_F32: torch.float32}


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


# the raw handle of a device's current stream without building a Stream
# object (about 0.2 against 2.9 us per call on a Grace host)
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, like: torch.Tensor) -> int:
    """The stream to enqueue on: the given one, else the current stream of
    the device that holds `like`."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(like.get_device())
        return torch.cuda.current_stream(like.device).cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Plan(NamedTuple):
    cnt: torch.Tensor          # int32 [E]
    off: torch.Tensor          # int64 [E+1]
    packed_src: torch.Tensor   # int32 [S*K] (first off[E] valid)
    tok_map: torch.Tensor      # int64 [S, K]
    n_invalid: torch.Tensor    # int32 [1]


class GroupPlan(NamedTuple):
    gcnt: torch.Tensor         # int32 [G]
    goff: torch.Tensor         # int64 [G+1]
    gtok_map: torch.Tensor     # int64 [S, K]
    grp_src: torch.Tensor      # int32 [max_rows]
    grp_tok_map: torch.Tensor  # int64 [max_rows, K]
    group_size: int

    @property
    def G(self) -> int:
        return self.gcnt.numel()

    @property
    def max_rows(self) -> int:
        return self.grp_src.numel()


def moe_plan_workspace_size(S: int, K: int, E: int) -> int:
    return int(lib().moe_plan_workspace_size(S, K, E))


def moe_group_plan_workspace_size(S: int, K: int, E: int, group_size: int) -> int:
    return int(lib().moe_group_plan_workspace_size(S, K, E, group_size))


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]):
    if nbytes == 0:
        return ws
    if ws is None or ws.numel() * ws.element_size() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return ws


def moe_plan(topk_idx: torch.Tensor, E: int, *, out: Optional[Plan] = None,
             workspace: Optional[torch.Tensor] = None, stream=None) -> Plan:
    """Histogram, exclusive scan and stable (token, k)-order slot map."""
    if topk_idx.dtype != torch.int32 or topk_idx.dim() != 2:
        raise TypeError("topk_idx must be int32 [S, K]")
    S, K = topk_idx.shape
    dev = topk_idx.device
    if out is None:
        out = Plan(torch.empty(E, dtype=torch.int32, device=dev),
                   torch.empty(E + 1, dtype=torch.int64, device=dev),
                   torch.empty(max(S * K, 1), dtype=torch.int32, device=dev),
                   torch.empty(S, K, dtype=torch.int64, device=dev),
                   torch.empty(1, dtype=torch.int32, device=dev))
    L = lib()
    nws = int(L.moe_plan_workspace_size(S, K, E))
    ws = _workspace(nws, dev, workspace)
    _abi.check("moe_plan", L.moe_plan(
        _ptr(topk_idx), S, K, E, _ptr(out.cnt), _ptr(out.off), _ptr(out.packed_src),
        _ptr(out.tok_map), _ptr(out.n_invalid), _ptr(ws), nws, _stream(stream, topk_idx)))
    return out


class CapacityPlan(NamedTuple):
    cnt: torch.Tensor          # int32 [E] rows filled per bucket
    off: torch.Tensor          # int64 [E+1] = e * capacity
    packed_src: torch.Tensor   # int32 [E*capacity]
    tok_map: torch.Tensor      # int64 [S, K], -1 for dropped entries
    n_invalid: torch.Tensor    # int32 [1]
    n_dropped: torch.Tensor    # int32 [1]
    capacity: int


def moe_plan_capacity(topk_idx: torch.Tensor, E: int, capacity: int, *,
                      out: Optional[CapacityPlan] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> CapacityPlan:
    """Plan into padded buckets of `capacity` rows; entries past a bucket's
    capacity (later tokens first to go) are dropped to -1."""
    if topk_idx.dtype != torch.int32 or topk_idx.dim() != 2:
        raise TypeError("topk_idx must be int32 [S, K]")
    S, K = topk_idx.shape
    dev = topk_idx.device
    if out is None:
        out = CapacityPlan(torch.empty(E, dtype=torch.int32, device=dev),
                           torch.empty(E + 1, dtype=torch.int64, device=dev),
                           torch.empty(E * capacity, dtype=torch.int32, device=dev),
                           torch.empty(S, K, dtype=torch.int64, device=dev),
                           torch.empty(1, dtype=torch.int32, device=dev),
                           torch.empty(1, dtype=torch.int32, device=dev), capacity)
    L = lib()
    nws = int(L.moe_plan_workspace_size(S, K, E))
    ws = _workspace(nws, dev, workspace)
    _abi.check("moe_plan_capacity", L.moe_plan_capacity(
        _ptr(topk_idx), S, K, E, capacity, _ptr(out.cnt), _ptr(out.off), _ptr(out.packed_src),
        _ptr(out.tok_map), _ptr(out.n_invalid), _ptr(out.n_dropped), _ptr(ws), nws,
        _stream(stream, topk_idx)))
    return out


def moe_group_plan(topk_idx: torch.Tensor, tok_map: torch.Tensor, E: int, group_size: int, *,
                   out: Optional[GroupPlan] = None, workspace: Optional[torch.Tensor] = None,
                   stream=None) -> GroupPlan:
    """Dedup plan: one group row per (token, virtual group) it reaches."""
    S, K = topk_idx.shape
    G = E // group_size
    dev = topk_idx.device
    if out is None:
        rmax = max(S * min(K, G), 1)
        out = GroupPlan(torch.empty(G, dtype=torch.int32, device=dev),
                        torch.empty(G + 1, dtype=torch.int64, device=dev),
                        torch.empty(S, K, dtype=torch.int64, device=dev),
                        torch.empty(rmax, dtype=torch.int32, device=dev),
                        torch.empty(rmax, K, dtype=torch.int64, device=dev),
                        group_size)
    L = lib()
    nws = int(L.moe_group_plan_workspace_size(S, K, E, group_size))
    ws = _workspace(nws, dev, workspace)
    _abi.check("moe_group_plan", L.moe_group_plan(
        _ptr(topk_idx), _ptr(tok_map), S, K, E, group_size, _ptr(out.gcnt), _ptr(out.goff),
        _ptr(out.gtok_map), _ptr(out.grp_src), _ptr(out.grp_tok_map), _ptr(ws), nws,
        _stream(stream, topk_idx)))
    return out


def moe_dispatch(x: torch.Tensor, tok_map: torch.Tensor, *, packed_x: Optional[torch.Tensor] = None,
                 x_scales: Optional[torch.Tensor] = None,
                 packed_scales: Optional[torch.Tensor] = None, stream=None):
    """packed_x[tok_map[s,k]] = x[s] (and the scale rows with them).
    Returns (packed_x, packed_scales)."""
    S, H = x.shape
    K = tok_map.shape[1]
    if packed_x is None:
        packed_x = torch.empty(S * K, H, dtype=x.dtype, device=x.device)
    n_scales = 0
    if x_scales is not None:
        n_scales = x_scales.shape[1]
        if packed_scales is None:
            packed_scales = torch.empty(S * K, n_scales, dtype=torch.float32, device=x.device)
    if packed_scales is not None and packed_scales.shape[0] < packed_x.shape[0]:
        raise ValueError("packed_scales needs as many rows as packed_x")
    _abi.check("moe_dispatch", lib().moe_dispatch(
        _ptr(x), S, H, _dt(x), K, _ptr(tok_map), _ptr(packed_x), packed_x.shape[0],
        _ptr(x_scales), n_scales, _ptr(packed_scales), _stream(stream, x)))
    return packed_x, packed_scales


_fused_max_cache: list = []


def _fused_max(L) -> int:
    """Entries up to which moe_plan_dispatch runs as one launch (a constant
    of the loaded library)."""
    if not _fused_max_cache:
        _fused_max_cache.append(int(L.moe_plan_dispatch_fused_max()))
    return _fused_max_cache[0]


def moe_plan_dispatch(topk_idx: torch.Tensor, x: torch.Tensor, E: int, *,
                      x_scales: Optional[torch.Tensor] = None, out: Optional[Plan] = None,
                      packed_x: Optional[torch.Tensor] = None,
                      packed_scales: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None):
    """moe_plan followed by moe_dispatch, in one launch for small batches.
    Returns (plan, packed_x, packed_scales)."""
    if topk_idx.dtype != torch.int32 or topk_idx.dim() != 2:
        raise TypeError("topk_idx must be int32 [S, K]")
    S, K = topk_idx.shape
    H = x.shape[1]
    dev = topk_idx.device
    if out is None:
        out = Plan(torch.empty(E, dtype=torch.int32, device=dev),
                   torch.empty(E + 1, dtype=torch.int64, device=dev),
                   torch.empty(max(S * K, 1), dtype=torch.int32, device=dev),
                   torch.empty(S, K, dtype=torch.int64, device=dev),
                   torch.empty(1, dtype=torch.int32, device=dev))
    if packed_x is None:
        packed_x = torch.empty(max(S * K, 1), H, dtype=x.dtype, device=dev)
    n_scales = 0
    if x_scales is not None:
        n_scales = x_scales.shape[1]
        if packed_scales is None:
            packed_scales = torch.empty(packed_x.shape[0], n_scales, dtype=torch.float32,
                                        device=dev)
    if packed_scales is not None and packed_scales.shape[0] < packed_x.shape[0]:
        raise ValueError("packed_scales needs as many rows as packed_x")
    L = lib()
    nws = 0
    if S * K > _fused_max(L):
        nws = int(L.moe_plan_workspace_size(S, K, E))
    ws = _workspace(nws, dev, workspace)
    _abi.check("moe_plan_dispatch", L.moe_plan_dispatch(
        _ptr(topk_idx), _ptr(x), S, H, _dt(x), K, E, _ptr(x_scales), n_scales, _ptr(out.cnt),
        _ptr(out.off), _ptr(out.packed_src), _ptr(out.tok_map), _ptr(out.n_invalid),
        _ptr(packed_x), packed_x.shape[0], _ptr(packed_scales), _ptr(ws), nws,
        _stream(stream, topk_idx)))
    return out, packed_x, packed_scales


def moe_dispatch_quant_fp8(x: torch.Tensor, tok_map: torch.Tensor, *, block: int = 128,
                           packed_q: Optional[torch.Tensor] = None,
                           packed_scales: Optional[torch.Tensor] = None, stream=None):
    """bf16 rows -> blockwise E4M3 codes + f32 scales in the K packed rows of
    each token.  Returns (packed_q as float8_e4m3fn, packed_scales)."""
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16")
    S, H = x.shape
    K = tok_map.shape[1]
    if packed_q is None:
        packed_q = torch.empty(S * K, H, dtype=torch.float8_e4m3fn, device=x.device)
    if packed_scales is None:
        packed_scales = torch.empty(S * K, H // block, dtype=torch.float32, device=x.device)
    rows = min(packed_q.shape[0], packed_scales.shape[0])
    _abi.check("moe_dispatch_quant_fp8", lib().moe_dispatch_quant_fp8(
        _ptr(x), S, H, K, _ptr(tok_map), block, _ptr(packed_q), _ptr(packed_scales), rows,
        _stream(stream, x)))
    return packed_q, packed_scales


def moe_dispatch_dedup(x: torch.Tensor, gp: GroupPlan, *, packed_x: Optional[torch.Tensor] = None,
                       grp_x: Optional[torch.Tensor] = None, stream=None):
    """Copy each token once per group row, then expand per expert.
    Returns (grp_x, packed_x)."""
    S, H = x.shape
    K = gp.gtok_map.shape[1]
    if grp_x is None:
        grp_x = torch.empty(gp.max_rows, H, dtype=x.dtype, device=x.device)
    if packed_x is None:
        packed_x = torch.empty(S * K, H, dtype=x.dtype, device=x.device)
    _abi.check("moe_dispatch_dedup", lib().moe_dispatch_dedup(
        _ptr(x), S, H, _dt(x), K, gp.G, _ptr(gp.goff), _ptr(gp.grp_src), _ptr(gp.grp_tok_map),
        _ptr(gp.gtok_map), gp.max_rows, _ptr(grp_x), _ptr(packed_x), packed_x.shape[0],
        _stream(stream, x)))
    return grp_x, packed_x


def moe_combine(y: torch.Tensor, topk_w: torch.Tensor, tok_map: torch.Tensor, *,
                out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """out[s] = sum_k topk_w[s,k] * y[tok_map[s,k]] in f32, increasing k."""
    S, K = tok_map.shape
    H = y.shape[1]
    if out is None:
        out = torch.empty(S, H, dtype=out_dtype, device=y.device)
    _abi.check("moe_combine", lib().moe_combine(
        _ptr(y), y.shape[0], _dt(y), _ptr(topk_w), _ptr(tok_map), S, H, K, _ptr(out), _dt(out),
        _stream(stream, y)))
    return out


def moe_combine_dedup(y: torch.Tensor, topk_w: torch.Tensor, gp: GroupPlan, *,
                      out_dtype: torch.dtype = torch.float32, out: Optional[torch.Tensor] = None,
                      gtok: Optional[torch.Tensor] = None, stream=None):
    """Per group row weighted sum, then per token unweighted sum of its group
    rows.  Returns (gtok, out)."""
    S, K = gp.gtok_map.shape
    H = y.shape[1]
    if gtok is None:
        gtok = torch.empty(gp.max_rows, H, dtype=torch.float32, device=y.device)
    if out is None:
        out = torch.empty(S, H, dtype=out_dtype, device=y.device)
    _abi.check("moe_combine_dedup", lib().moe_combine_dedup(
        _ptr(y), y.shape[0], _dt(y), _ptr(topk_w), _ptr(gp.goff), gp.G, _ptr(gp.grp_src),
        _ptr(gp.grp_tok_map), _ptr(gp.gtok_map), S, H, K, gp.max_rows, _ptr(gtok), _ptr(out),
        _dt(out), _stream(stream, y)))
    return gtok, out


def moe_combine_fold(y: torch.Tensor, topk_w: Optional[torch.Tensor], token_map: torch.Tensor,
                     *, weighted: bool = False, fold: bool = True,
                     out_dtype: torch.dtype = torch.bfloat16, out: Optional[torch.Tensor] = None,
                     out_weights: Optional[torch.Tensor] = None, stream=None):
    """out[s] = sum over valid k of (topk_w[s,k] if weighted else 1) *
    y[token_map[s,k]]; out_weights[s,i] = sum over valid k of topk_w[s,i].
    token_map is tok_map (packed rows) or gtok_map (group rows).
    Returns (out, out_weights or None)."""
    S, K = token_map.shape
    H = y.shape[1]
    if out is None:
        out = torch.empty(S, H, dtype=out_dtype, device=y.device)
    if fold and out_weights is None:
        out_weights = torch.empty(S, K, dtype=torch.float32, device=y.device)
    if not fold:
        out_weights = None
    _abi.check("moe_combine_fold", lib().moe_combine_fold(
        _ptr(y), y.shape[0], _dt(y), _ptr(topk_w), int(weighted), _ptr(token_map), S, H, K,
        _ptr(out), _dt(out), _ptr(out_weights), _stream(stream, y)))
    return out, out_weights


def moe_device_errors() -> int:
    """Reads and clears the kernels' device error bits (synchronous): bit 0
    dispatch wait timeout, bit 1 dispatch row index out of range, bit 2
    combine row index out of range."""
    import ctypes
    v = ctypes.c_uint32(0)
    _abi.check("moe_device_errors", lib().moe_device_errors(ctypes.byref(v)))
    return int(v.value)


from .op import MoeOp, Routing  # noqa: E402  (the op interface over the calls above)
