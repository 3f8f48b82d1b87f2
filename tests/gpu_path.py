"""Runs one workload through the CUDA library (C ABI via the Python binding)
and returns every output as numpy, for comparison with the CPU oracle.

The synthetic expert stage between dispatch and combine is harness code (the
same definition the oracle uses, written with torch ops on the GPU).
"""
from __future__ import annotations

import numpy as np
import torch

import combine_moe_plan_02_gb300 as moe

POISON = 0xFF  # byte poured into every output before a run (bf16 0xFFFF is NaN)


def to_device(wl, device="cuda"):
    d = {}
    d["topk_idx"] = torch.from_numpy(np.ascontiguousarray(wl.topk_idx)).to(device)
    d["topk_w"] = torch.from_numpy(np.ascontiguousarray(wl.topk_w)).to(device)
    if wl.dtype == "bf16":
        d["x"] = torch.from_numpy(wl.x.view(np.int16)).to(device).view(torch.bfloat16)
    elif wl.dtype == "f32":
        d["x"] = torch.from_numpy(wl.x).to(device)
    else:
        d["x"] = torch.from_numpy(wl.x).to(device).view(torch.float8_e4m3fn)
        d["x_scales"] = torch.from_numpy(wl.x_scales).to(device)
    d["c"] = torch.from_numpy(wl.expert_scale).to(device)
    return d


def poisoned(shape, dtype, device="cuda"):
    t = torch.empty(shape, dtype=dtype, device=device)
    t.view(torch.uint8).fill_(POISON)
    return t


def expert_stage(wl, plan, packed_x, packed_scales):
    """y rows from packed rows: bf16 -> bf16(f32(x) * c_e); f32 identity;
    fp8 -> bf16(e4m3(q) * scale of its 128-block)."""
    V = int(plan.off[-1].item())
    if wl.dtype == "bf16":
        c_row = torch.repeat_interleave(torch.from_numpy(wl.expert_scale).cuda(), plan.cnt.long())
        y = torch.empty_like(packed_x)
        y[:V] = (packed_x[:V].float() * c_row[:, None]).to(torch.bfloat16)
        return y
    if wl.dtype == "f32":
        return packed_x
    y = torch.empty(packed_x.shape, dtype=torch.bfloat16, device=packed_x.device)
    sc = packed_scales[:V].repeat_interleave(wl.scale_block, dim=1)
    y[:V] = (packed_x[:V].float() * sc).to(torch.bfloat16)
    return y


def _np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def run(wl, dedup: bool = None):
    """Whole GPU path; outputs are poisoned first so that a skipped write
    cannot pass as a correct one."""
    dedup = bool(wl.group_size) if dedup is None else dedup
    d = to_device(wl)
    S, K, E, H = wl.S, wl.K, wl.E, wl.H
    plan = moe.Plan(poisoned((E,), torch.int32), poisoned((E + 1,), torch.int64),
                    poisoned((max(S * K, 1),), torch.int32), poisoned((S, K), torch.int64),
                    poisoned((1,), torch.int32))
    moe.moe_plan(d["topk_idx"], E, out=plan)
    packed = poisoned((S * K, H), d["x"].dtype)
    pscales = poisoned((S * K, d["x_scales"].shape[1]), torch.float32) if "x_scales" in d else None
    moe.moe_dispatch(d["x"], plan.tok_map, packed_x=packed, x_scales=d.get("x_scales"),
                     packed_scales=pscales)
    y = expert_stage(wl, plan, packed, pscales)
    out_dt = torch.bfloat16 if wl.out_dtype == "bf16" else torch.float32
    out = poisoned((S, H), out_dt)
    moe.moe_combine(y, d["topk_w"], plan.tok_map, out=out)
    torch.cuda.synchronize()
    V = int(plan.off[-1].item())
    res = dict(cnt=_np(plan.cnt), off=_np(plan.off), packed_src=_np(plan.packed_src)[:V],
               tok_map=_np(plan.tok_map), n_invalid=int(plan.n_invalid.item()),
               packed_x_full=_np(packed), packed_x=_np(packed)[:V], y=_np(y)[:V], out=_np(out))
    if pscales is not None:
        res["packed_scales"] = _np(pscales)[:V]
    if dedup:
        G = E // wl.group_size
        rmax = max(S * min(K, G), 1)
        gp = moe.GroupPlan(poisoned((G,), torch.int32), poisoned((G + 1,), torch.int64),
                           poisoned((S, K), torch.int64), poisoned((rmax,), torch.int32),
                           poisoned((rmax, K), torch.int64), wl.group_size)
        moe.moe_group_plan(d["topk_idx"], plan.tok_map, E, wl.group_size, out=gp)
        grp_x = poisoned((rmax, H), d["x"].dtype)
        packed_d = poisoned((S * K, H), d["x"].dtype)
        moe.moe_dispatch_dedup(d["x"], gp, grp_x=grp_x, packed_x=packed_d)
        y_d = expert_stage(wl, plan, packed_d, pscales)
        gtok = poisoned((rmax, H), torch.float32)
        out_d = poisoned((S, H), out_dt)
        moe.moe_combine_dedup(y_d, d["topk_w"], gp, out=out_d, gtok=gtok)
        torch.cuda.synchronize()
        R = int(gp.goff[-1].item())
        res.update(gcnt=_np(gp.gcnt), goff=_np(gp.goff), gtok_map=_np(gp.gtok_map),
                   grp_src=_np(gp.grp_src)[:R], grp_tok_map=_np(gp.grp_tok_map)[:R],
                   grp_x=_np(grp_x)[:R], packed_x_dedup=_np(packed_d)[:V], gtok=_np(gtok)[:R],
                   out_dedup=_np(out_d))
    return res
