"""Benchmark: single-GPU MoE plan -> dispatch -> combine.

One step = moe_plan + moe_dispatch + moe_combine over one batch of the
MoonEP-shaped workload (S=4096 tokens, H=7168, E=64 experts, K=8, bf16,
uniform top-8, softmax weights; the expert output rows y are produced once,
untimed, by the synthetic expert stage y = bf16(x * c_e)).  Before every
timed step L2 is flushed (a 512 MiB write, then a 512 MiB read of another
buffer, so that no dirty line of the flush is left to be written back inside
the step); step time is measured with CUDA events on the launching stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` = algorithmic bytes of plan + dispatch +
combine per step / mean step time, summed over ranks (replicas: every rank
runs its own batch; no data moves between GPUs).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "dispatch & combine GB/s and % HBM roofline at S=4096 H=7168 E=64 K=8; µs/call"
WORKLOAD = "moonep"
FALLBACK_HBM_GBS = 6800.0
SPEC_HBM_GBS = 8000.0     # GB300 HBM3e, nominal (~8 TB/s)
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------------------
# algorithmic bytes (what the method must move; scratch traffic not counted)
# ---------------------------------------------------------------------------

def algorithmic_bytes(S, H, E, K, V, elem=2, out_elem=2):
    plan = S * K * 4 + E * 4 + (E + 1) * 8 + V * 4 + S * K * 8 + 4
    dispatch = S * H * elem + S * K * 8 + V * H * elem
    combine = V * H * elem + S * K * (8 + 4) + S * H * out_elem
    return {"plan": plan, "dispatch": dispatch, "combine": combine}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        ent = t[kernel]
        src = os.path.join(ROOT, "combine_moe_plan_02_gb300", "csrc", ent["source"])
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if digest != ent["sha256"]:
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                "clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index: int, interval_ms: int = 100):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# multi-rank helpers (replicas; also exercised with gloo on CPU in the tests)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(elapsed_ms: float, local_bytes: float, world: int, device=None):
    """Max of the timed region over ranks and the sum of bytes processed."""
    if world == 1:
        return elapsed_ms, local_bytes
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    b = torch.tensor([local_bytes], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def pipelined_e2e(torch, moe, dev, stream, n, warmup, h_idx, h_w, h_x, plan, ws, packed, y, E,
                  S, H, step_bytes, world, idx0, w0, x16_0, out0):
    """Times n pipelined steps (see the caller); returns (max ms over ranks,
    bytes over ranks)."""
    s_h2d = torch.cuda.Stream(dev)
    s_d2h = torch.cuda.Stream(dev)
    bufs = [dict(idx=idx0, w=w0, x16=x16_0, out=out0,
                 h_out=torch.empty(S, H, dtype=torch.int16).pin_memory()),
            dict(idx=torch.empty_like(idx0), w=torch.empty_like(w0),
                 x16=torch.empty_like(x16_0), out=torch.empty_like(out0),
                 h_out=torch.empty(S, H, dtype=torch.int16).pin_memory())]
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def pipe_step(i):
        j = i & 1
        b = bufs[j]
        s_h2d.wait_event(comp_done[j])      # step i-2 has finished reading buffer j
        with torch.cuda.stream(s_h2d):
            b["idx"].copy_(h_idx, non_blocking=True)
            b["w"].copy_(h_w, non_blocking=True)
            b["x16"].copy_(h_x, non_blocking=True)
        h2d_done[j].record(s_h2d)
        stream.wait_event(h2d_done[j])
        stream.wait_event(d2h_done[j])      # step i-2's result has left out[j]
        moe.moe_plan_dispatch(b["idx"], b["x16"].view(torch.bfloat16), E, out=plan,
                              packed_x=packed, workspace=ws, stream=stream)
        moe.moe_combine(y, b["w"], plan.tok_map, out=b["out"], stream=stream)
        comp_done[j].record(stream)
        s_d2h.wait_event(comp_done[j])
        with torch.cuda.stream(s_d2h):
            b["h_out"].copy_(b["out"].view(torch.int16), non_blocking=True)
        d2h_done[j].record(s_d2h)

    for i in range(warmup):
        pipe_step(i)
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    start.record(stream)
    s_h2d.wait_event(start)
    s_d2h.wait_event(start)
    for i in range(n):
        pipe_step(i)
    stream.wait_event(d2h_done[(n - 1) & 1])
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    last = bufs[(n - 1) & 1]
    assert np.array_equal(last["h_out"].numpy(), last["out"].view(torch.int16).cpu().numpy())
    return aggregate(start.elapsed_time(end), step_bytes * n, world, dev)


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle leg (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

ORACLE_SAMPLE_TOKENS = 1024


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


class PinnedCore:
    """Pins the calling thread (where the oracle runs) to one logical CPU,
    the highest-numbered one it may use, and restores the old set on exit."""

    def __enter__(self):
        self.old = os.sched_getaffinity(0)
        self.core = max(self.old)
        os.sched_setaffinity(0, {self.core})
        try:
            with open(f"/sys/devices/system/cpu/cpu{self.core}/topology/thread_siblings_list") as f:
                self.siblings = f.read().strip()
        except Exception:
            self.siblings = None
        return self

    def __exit__(self, *exc):
        os.sched_setaffinity(0, self.old)
        return False


def _median_us(fn, reps: int = 3):
    """Median µs of `reps` calls after one untimed warm-up call."""
    fn()
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t0)
    return 1e6 * statistics.median(ts)


def _head(wl, n):
    """The first n tokens of a workload (a bounded sample of the batch)."""
    wl.S = n
    wl.topk_idx = np.ascontiguousarray(wl.topk_idx[:n])
    wl.topk_w = np.ascontiguousarray(wl.topk_w[:n])
    wl.x = np.ascontiguousarray(wl.x[:n])
    if wl.x_scales is not None:
        wl.x_scales = np.ascontiguousarray(wl.x_scales[:n])
    return wl


def _oracle_calls(wl):
    """Oracle calls of one workload, inputs prepared once (the expert output
    rows y of the harness's expert stage included, untimed): name ->
    (callable, algorithmic bytes)."""
    import oracle
    S, H, E, K = wl.S, wl.H, wl.E, wl.K
    p = oracle.plan(wl.topk_idx, wl.E)
    V = int(p["off"][-1])
    tm = p["tok_map"]
    calls = {}
    if wl.dtype == workloads.DT_FP8:
        nsc = wl.x_scales.shape[1]
        packed = oracle.dispatch(wl.x, tm, V)
        pscales = oracle.dispatch(wl.x_scales, tm, V)
        y = oracle.expert_dequant_fp8(packed, pscales, wl.scale_block)
        calls["plan"] = (lambda: oracle.plan(wl.topk_idx, E), algorithmic_bytes(S, H, E, K, V)["plan"])
        calls["dispatch"] = (lambda: (oracle.dispatch(wl.x, tm, V), oracle.dispatch(wl.x_scales, tm, V)),
                             S * H + S * K * 8 + V * H + (S + V) * nsc * 4)
        calls["combine"] = (lambda: oracle.combine(y, "bf16", wl.topk_w, tm, H, "bf16"),
                            algorithmic_bytes(S, H, E, K, V)["combine"])
        return calls
    b = 2 if wl.dtype == workloads.DT_BF16 else 4
    dt = "bf16" if wl.dtype == workloads.DT_BF16 else "f32"
    nby = algorithmic_bytes(S, H, E, K, V, elem=b, out_elem=b)
    packed = oracle.dispatch(wl.x, tm, V)
    if wl.dtype == workloads.DT_BF16:
        y = oracle.expert_scale_bf16(packed, p["off"], wl.expert_scale)
    else:
        y = packed                                   # identity experts
    calls["plan"] = (lambda: oracle.plan(wl.topk_idx, E), nby["plan"])
    calls["dispatch"] = (lambda: oracle.dispatch(wl.x, tm, V), nby["dispatch"])
    calls["combine"] = (lambda: oracle.combine(y, dt, wl.topk_w, tm, H, dt), nby["combine"])
    if wl.group_size:
        gs = wl.group_size
        gp = oracle.group_plan(wl.topk_idx, tm, E, gs)
        R = int(gp["goff"][-1])
        calls["group_plan"] = (lambda: oracle.group_plan(wl.topk_idx, tm, E, gs),
                               S * K * (4 + 8) + S * K * 8 + R * (4 + 8 * K) + (E // gs) * 12)
        calls["dispatch_dedup"] = (
            lambda: oracle.dispatch_dedup(wl.x, gp["grp_src"], gp["grp_tok_map"], K, V),
            S * H * b + R * H * b + V * H * b + R * (4 + 8 * K))
        calls["combine_dedup"] = (
            lambda: oracle.combine_dedup(y, dt, wl.topk_w, gp["grp_src"], gp["grp_tok_map"],
                                         gp["gtok_map"], H, dt),
            V * H * b + R * H * b + S * H * b + R * 8 * K + S * K * 16)
    return calls


def _time_calls(calls):
    res = {}
    for name, (fn, nbytes) in calls.items():
        us = _median_us(fn)
        res[name] = {"us": round(us, 1), "GB_per_s": round(nbytes / (us * 1e-6) / 1e9, 3),
                     "algorithmic_bytes": int(nbytes)}
    return res


def cpu_per_config():
    """µs per oracle call and GB/s for each of the five workloads: the tiny
    case, the dedup shape (with S=0 and S=1) and the small-token fp8 sweep
    at full size; the MoonEP and Zipf shapes on their first 1024 tokens."""
    per = {}
    per["tiny"] = {"sample": "full: S=128 H=256 E=8 K=2 bf16",
                   "calls": _time_calls(_oracle_calls(workloads.make("tiny", seed=0)))}
    for name in ("moonep", "zipf"):
        wl = workloads.make(name, seed=0)
        full = wl.S
        wl = _head(wl, ORACLE_SAMPLE_TOKENS)
        per[name] = {"sample": f"first {ORACLE_SAMPLE_TOKENS} of {full} tokens "
                               f"(H={wl.H} E={wl.E} K={wl.K} bf16)",
                     "calls": _time_calls(_oracle_calls(wl))}
    ded = {}
    for S in (4096, 0, 1):
        ded[f"S={S}"] = _time_calls(_oracle_calls(workloads.make("dedup", seed=0, S=S)))
    per["dedup"] = {"sample": "full: S=4096 H=4096 E=64 in 8 groups, K=8 f32; and S=0, S=1",
                    "calls": ded}
    fp8 = {}
    for S in workloads.FP8_SWEEP_TOKENS:
        fp8[f"S={S}"] = _time_calls(_oracle_calls(workloads.make("fp8small", seed=S, S=S)))
    per["fp8small"] = {"sample": "full: S in {4,8,16,32,128,1024}, H=6144 E=256 K=8, fp8 rows "
                                 "+ f32 scales, bf16 combine", "calls": fp8}
    return per


def oracle_sample(seed: int = 0):
    """A bounded sample of the workload: the first 1024 tokens of the batch,
    with the expert output rows prepared once."""
    import oracle
    wl = _head(workloads.make(WORKLOAD, seed=seed), ORACLE_SAMPLE_TOKENS)
    p = oracle.plan(wl.topk_idx, wl.E)
    V = int(p["off"][-1])
    packed = oracle.dispatch(wl.x, p["tok_map"], V)
    y = oracle.expert_scale_bf16(packed, p["off"], wl.expert_scale)
    return wl, y, V


def oracle_step(wl, y, V):
    import oracle
    p = oracle.plan(wl.topk_idx, wl.E)
    oracle.dispatch(wl.x, p["tok_map"], V)
    oracle.combine(y, "bf16", wl.topk_w, p["tok_map"], wl.H, "bf16")


def cpu_baseline():
    """The single-threaded C oracle on one pinned core: `value` is
    plan + dispatch + combine on the first 1024 tokens of the MoonEP batch
    (algorithmic bytes / summed median call times); `per_config` has every
    workload."""
    with PinnedCore() as pin:
        per = cpu_per_config()
    calls = per[WORKLOAD]["calls"]
    by = sum(c["algorithmic_bytes"] for c in calls.values())
    us = sum(c["us"] for c in calls.values())
    return {"value": by / (us * 1e-6) / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {ORACLE_SAMPLE_TOKENS} of the 4096 tokens (H=7168 E=64 K=8 bf16), "
                      "plan+dispatch+combine, median of 3 timed calls each after a warm-up, "
                      "single-threaded C oracle",
            "pinned_core": pin.core, "core_siblings": pin.siblings,
            "cpu_model": host_cpu_model(), "host_cpus": os.cpu_count(), "per_config": per}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    with PinnedCore() as pin:
        wl, y, V = oracle_sample()
        by = sum(algorithmic_bytes(wl.S, wl.H, wl.E, wl.K, V).values())
        for _ in range(args.warmup):
            oracle_step(wl, y, V)
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            oracle_step(wl, y, V)
            times.append(time.perf_counter() - t0)
        per = cpu_per_config()
    ms = 1e3 * sum(times) / len(times)
    value = by / (ms / 1e3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: first {ORACLE_SAMPLE_TOKENS} tokens of S=4096 "
                               "H=7168 E=64 K=8 bf16 per step (CPU oracle)",
                   "S": ORACLE_SAMPLE_TOKENS, "H": wl.H, "E": wl.E, "K": wl.K},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {ORACLE_SAMPLE_TOKENS} tokens per step",
                         "pinned_core": pin.core, "core_siblings": pin.siblings,
                         "cpu_model": host_cpu_model(), "host_cpus": os.cpu_count(),
                         "per_config": per},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# small-token latency (the mori EPv2 latency tables' shape: H=6144, top-8,
# 4..32 tokens; here on one GPU with fp8 rows and per-128 scales)
# ---------------------------------------------------------------------------

def _trimmed_mean(xs, cut: float = 0.1):
    """Mean of the values left after dropping the lowest and highest `cut`
    fraction."""
    v = sorted(xs)
    k = int(len(v) * cut)
    return statistics.mean(v[k:len(v) - k] if len(v) > 2 * k else v)


def small_token_latency(dev, reps: int = 50):
    """µs per plan + dispatch (fp8 rows + f32 scales) + combine (bf16) call
    sequence at small token counts, eager and replayed from a CUDA graph."""
    import torch

    import combine_moe_plan_02_gb300 as moe
    res = {"workload": "fp8small: H=6144 E=256 K=8, fp8 e4m3 rows + 48 f32 scales per row, "
                       "bf16 expert outputs, bf16 combine; inputs resident, y precomputed",
           "S": [], "eager_us": [], "graph_us": [], "plan_us": [], "dispatch_us": [],
           "combine_us": [], "fused_eager_us": [], "fused_graph_us": [],
           "plan_dispatch_us": [], "fused_max_entries": None}
    stream = torch.cuda.Stream(dev)  # graphs are captured on a non-default stream
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        _small_token_sweep(moe, torch, dev, stream, reps, res)
    torch.cuda.synchronize(dev)
    return res


def _small_token_sweep(moe, torch, dev, stream, reps, res):
    for S in workloads.FP8_SWEEP_TOKENS:
        wl = workloads.make("fp8small", seed=S, S=S)
        E, K, H = wl.E, wl.K, wl.H
        idx = torch.from_numpy(wl.topk_idx).to(dev)
        w = torch.from_numpy(wl.topk_w).to(dev)
        x = torch.from_numpy(wl.x).to(dev).view(torch.float8_e4m3fn)
        xs = torch.from_numpy(wl.x_scales).to(dev)
        plan = moe.moe_plan(idx, E)
        px, ps = moe.moe_dispatch(x, plan.tok_map, x_scales=xs)
        y = (px.float() * ps.repeat_interleave(wl.scale_block, dim=1)).to(torch.bfloat16)
        out = torch.empty(S, H, dtype=torch.bfloat16, device=dev)

        def calls():
            moe.moe_plan(idx, E, out=plan, stream=stream)
            moe.moe_dispatch(x, plan.tok_map, packed_x=px, x_scales=xs, packed_scales=ps,
                             stream=stream)
            moe.moe_combine(y, w, plan.tok_map, out=out, stream=stream)

        for _ in range(10):
            calls()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
        for e in ev:
            e[0].record(stream)
            moe.moe_plan(idx, E, out=plan, stream=stream)
            e[1].record(stream)
            moe.moe_dispatch(x, plan.tok_map, packed_x=px, x_scales=xs, packed_scales=ps,
                             stream=stream)
            e[2].record(stream)
            moe.moe_combine(y, w, plan.tok_map, out=out, stream=stream)
            e[3].record(stream)
        torch.cuda.synchronize()
        step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
        for a, b in step_ev:
            a.record(stream)
            calls()
            b.record(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            calls()
        for _ in range(5):
            g.replay()
        torch.cuda.synchronize()
        g_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(reps)]
        for a, b in g_ev:
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        # moe_plan_dispatch (one launch up to the crossover) + combine
        def calls_fused():
            moe.moe_plan_dispatch(idx, x, E, x_scales=xs, out=plan, packed_x=px,
                                  packed_scales=ps, stream=stream)
            moe.moe_combine(y, w, plan.tok_map, out=out, stream=stream)

        for _ in range(10):
            calls_fused()
        torch.cuda.synchronize()
        f_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
        for e in f_ev:
            e[0].record(stream)
            moe.moe_plan_dispatch(idx, x, E, x_scales=xs, out=plan, packed_x=px,
                                  packed_scales=ps, stream=stream)
            e[1].record(stream)
            moe.moe_combine(y, w, plan.tok_map, out=out, stream=stream)
            e[2].record(stream)
        torch.cuda.synchronize()
        fs_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(reps)]
        for a, b in fs_ev:
            a.record(stream)
            calls_fused()
            b.record(stream)
        torch.cuda.synchronize()
        gf = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gf, stream=stream):
            calls_fused()
        for _ in range(5):
            gf.replay()
        torch.cuda.synchronize()
        gf_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(reps)]
        for a, b in gf_ev:
            a.record(stream)
            gf.replay()
            b.record(stream)
        torch.cuda.synchronize()
        # means of the middle 80 %: CUDA event timestamps come in steps of
        # about 2 us on this part, so medians of short launches snap to those
        # steps, and a plain mean takes in the odd host-side stall of an
        # eager call (one 1 ms outlier moves a mean of 50 by 20 us)
        med = lambda xs_: round(1e3 * _trimmed_mean(xs_), 2)
        res["fused_eager_us"].append(med([a.elapsed_time(b) for a, b in fs_ev]))
        res["plan_dispatch_us"].append(med([e[0].elapsed_time(e[1]) for e in f_ev]))
        res["fused_graph_us"].append(med([a.elapsed_time(b) for a, b in gf_ev]))
        res["fused_max_entries"] = int(moe.lib().moe_plan_dispatch_fused_max())
        res["S"].append(S)
        res["eager_us"].append(med([a.elapsed_time(b) for a, b in step_ev]))
        res["graph_us"].append(med([a.elapsed_time(b) for a, b in g_ev]))
        res["plan_us"].append(med([e[0].elapsed_time(e[1]) for e in ev]))
        res["dispatch_us"].append(med([e[1].elapsed_time(e[2]) for e in ev]))
        res["combine_us"].append(med([e[2].elapsed_time(e[3]) for e in ev]))
    return res


# ---------------------------------------------------------------------------
# the step under contention (MoonEP "Drop cooperative launch from the
# CTA-independent local kernels": the local kernels timed alone and against a
# saturating GEMM stream, 100 launches)
# ---------------------------------------------------------------------------

def contended_step(torch, moe, dev, stream, idx, x, w, y, plan, packed, out, ws, E, n=100):
    """µs per call of the step's two calls, alone and while bf16 GEMMs
    (8192 x 8192 x 8192, torch.matmul) keep the GPU busy on another stream.
    The library's CTAs are independent (no cooperative launch, no grid-wide
    wait), so they share the SMs with the GEMM's instead of waiting for the
    whole GPU.  No L2 flush between steps in either run."""
    side = torch.cuda.Stream(dev)
    a = torch.randn(8192, 8192, device=dev).to(torch.bfloat16)
    b = torch.randn(8192, 8192, device=dev).to(torch.bfloat16)
    c = torch.empty(8192, 8192, device=dev, dtype=torch.bfloat16)

    def steps(evs, st=stream):
        for e in evs:
            e[0].record(st)
            moe.moe_plan_dispatch(idx, x, E, out=plan, packed_x=packed, workspace=ws, stream=st)
            e[1].record(st)
            moe.moe_combine(y, w, plan.tok_map, out=out, stream=st)
            e[2].record(st)

    def mk():
        return [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]

    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        torch.matmul(a, b, out=c)
    g0.record()
    for _ in range(5):
        torch.matmul(a, b, out=c)
    g1.record()
    torch.cuda.synchronize()
    one_gemm_ms = g0.elapsed_time(g1) / 5
    iso = mk()
    steps(iso)
    torch.cuda.synchronize()
    iso_ms = iso[0][0].elapsed_time(iso[-1][2])
    # GEMMs enqueued first, enough to outlast the steps even when the steps
    # run several times slower than alone
    n_gemm = int(8 * iso_ms / one_gemm_ms) + 1
    g0.record(side)
    with torch.cuda.stream(side):
        for _ in range(n_gemm):
            torch.matmul(a, b, out=c)
    g1.record(side)
    con = mk()
    steps(con)
    torch.cuda.synchronize()
    covered = g0.elapsed_time(g1) > g0.elapsed_time(con[-1][2])
    gemm_ms = g0.elapsed_time(g1)
    # the same with the step on a stream of the highest priority: its CTAs
    # go first whenever an SM frees up
    hp = torch.cuda.Stream(dev, priority=torch.cuda.Stream.priority_range()[1]
                           if hasattr(torch.cuda.Stream, "priority_range") else -1)
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    h0.record(side)
    with torch.cuda.stream(side):
        for _ in range(n_gemm):
            torch.matmul(a, b, out=c)
    h1.record(side)
    con_hp = mk()
    steps(con_hp, hp)
    torch.cuda.synchronize()
    covered_hp = h0.elapsed_time(h1) > h0.elapsed_time(con_hp[-1][2])
    gemm_hp_ms = h0.elapsed_time(h1)

    def m(evs, i, j):
        return round(1e3 * statistics.mean(e[i].elapsed_time(e[j]) for e in evs), 2)

    res = {"what": f"moe_plan_dispatch and moe_combine at the headline shape, {n} steps, "
                   f"alone and while {n_gemm} bf16 8192^3 GEMMs run on another stream",
           "alone_us": {"plan_dispatch": m(iso, 0, 1), "combine": m(iso, 1, 2)},
           "contended_us": {"plan_dispatch": m(con, 0, 1), "combine": m(con, 1, 2)},
           "gemm_stream_busy_throughout": bool(covered),
           "gemm_tflops_alone": round(2 * 8192 ** 3 / (one_gemm_ms * 1e-3) / 1e12, 1),
           "gemm_tflops_during": round(n_gemm * 2 * 8192 ** 3 / (gemm_ms * 1e-3) / 1e12, 1),
           "high_priority_stream": {
               "contended_us": {"plan_dispatch": m(con_hp, 0, 1), "combine": m(con_hp, 1, 2)},
               "gemm_stream_busy_throughout": bool(covered_hp),
               "gemm_tflops_during": round(n_gemm * 2 * 8192 ** 3 / (gemm_hp_ms * 1e-3) / 1e12,
                                           1)}}
    del a, b, c
    return res


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------

def _timed_calls(torch, stream, flush_l2, calls, n=10, warmup=3):
    """Mean µs of each call in `calls` (name -> fn), L2 flushed before each
    sequence, an event between the calls."""
    for _ in range(warmup):
        for fn in calls.values():
            fn()
    torch.cuda.synchronize()
    ts = {k: [] for k in calls}
    for i in range(n):
        flush_l2(i & 0xFF)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
        ev[0].record(stream)
        for j, fn in enumerate(calls.values()):
            fn()
            ev[j + 1].record(stream)
        torch.cuda.synchronize()
        for j, k in enumerate(calls):
            ts[k].append(ev[j].elapsed_time(ev[j + 1]))
    return {k: statistics.mean(v) * 1e3 for k, v in ts.items()}


def other_workloads(torch, moe, dev, stream, flush_l2, peak):
    """The skewed-routing and the dedup workloads through the same calls
    (identity experts: the combine gathers the dispatched rows), per call."""
    res = {}

    def entry(us, nbytes):
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"us": round(us, 2), "GB_per_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                "algorithmic_bytes": int(nbytes)}

    # Zipf(1.2) routing over 256 experts: buckets from ~S rows down to empty
    wl = workloads.make("zipf", seed=0)
    S, H, E, K = wl.S, wl.H, wl.E, wl.K
    idx = torch.from_numpy(wl.topk_idx).to(dev)
    w = torch.from_numpy(wl.topk_w).to(dev)
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev).view(torch.bfloat16)
    plan = moe.moe_plan(idx, E)
    packed = torch.empty(S * K, H, dtype=torch.bfloat16, device=dev)
    out = torch.empty(S, H, dtype=torch.bfloat16, device=dev)
    t = _timed_calls(torch, stream, flush_l2, {
        "plan": lambda: moe.moe_plan(idx, E, out=plan, stream=stream),
        "dispatch": lambda: moe.moe_dispatch(x, plan.tok_map, packed_x=packed, stream=stream),
        "combine": lambda: moe.moe_combine(packed, w, plan.tok_map, out=out, stream=stream)})
    V = int(plan.off[-1].item())
    nby = algorithmic_bytes(S, H, E, K, V)
    cnt = plan.cnt.cpu()
    res["zipf"] = {"workload": f"zipf: S={S} H={H} E={E} K={K} bf16, Zipf(1.2) routing",
                   "largest_bucket": int(cnt.max()), "empty_buckets": int((cnt == 0).sum()),
                   **{k: entry(t[k], nby[k]) for k in t}}
    del packed, out, x

    # dedup: 8 virtual groups of 8 experts, f32 rows
    wl = workloads.make("dedup", seed=0)
    S, H, E, K, gs = wl.S, wl.H, wl.E, wl.K, wl.group_size
    idx = torch.from_numpy(wl.topk_idx).to(dev)
    w = torch.from_numpy(wl.topk_w).to(dev)
    x = torch.from_numpy(wl.x).to(dev)
    plan = moe.moe_plan(idx, E)
    gp = moe.moe_group_plan(idx, plan.tok_map, E, gs)
    grp_x = torch.empty(gp.max_rows, H, dtype=torch.float32, device=dev)
    packed = torch.empty(S * K, H, dtype=torch.float32, device=dev)
    gtok = torch.empty(gp.max_rows, H, dtype=torch.float32, device=dev)
    out = torch.empty(S, H, dtype=torch.float32, device=dev)
    # the group plan's tile histograms: allocated once, as a caller's loop would
    gws = torch.empty(max(moe.moe_group_plan_workspace_size(S, K, E, gs), 256), dtype=torch.uint8,
                      device=dev)
    t = _timed_calls(torch, stream, flush_l2, {
        "plan": lambda: moe.moe_plan(idx, E, out=plan, stream=stream),
        "group_plan": lambda: moe.moe_group_plan(idx, plan.tok_map, E, gs, out=gp, workspace=gws,
                                                 stream=stream),
        "dispatch_dedup": lambda: moe.moe_dispatch_dedup(x, gp, grp_x=grp_x, packed_x=packed,
                                                         stream=stream),
        "combine_dedup": lambda: moe.moe_combine_dedup(packed, w, gp, gtok=gtok, out=out,
                                                       stream=stream)})
    V = int(plan.off[-1].item())
    R = int(gp.goff[-1].item())
    b = 4
    nby = {"plan": algorithmic_bytes(S, H, E, K, V)["plan"],
           "group_plan": S * K * (4 + 8) + S * K * 8 + R * (4 + 8 * K) + (E // gs) * 12,
           # x read once, group rows and packed rows written (one pass: the
           # group rows are not read back)
           "dispatch_dedup": S * H * b + R * H * b + V * H * b + R * (4 + 8 * K),
           # expert rows read, group-row sums and token sums written (one pass)
           "combine_dedup": V * H * b + R * H * b + S * H * b + R * 8 * K + S * K * 16}
    res["dedup"] = {"workload": f"dedup: S={S} H={H} E={E} in {E // gs} groups, K={K} f32",
                    "group_rows": R, **{k: entry(t[k], nby[k]) for k in t}}
    return res


def run_ours(args):
    import torch

    import combine_moe_plan_02_gb300 as moe

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    moe.lib()

    wl = workloads.make(WORKLOAD, seed=rank)
    S, H, E, K = wl.S, wl.H, wl.E, wl.K
    stream = torch.cuda.current_stream(dev)

    # device-resident inputs and preallocated outputs
    idx = torch.from_numpy(wl.topk_idx).to(dev)
    w = torch.from_numpy(wl.topk_w).to(dev)
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev).view(torch.bfloat16)
    plan = moe.Plan(torch.empty(E, dtype=torch.int32, device=dev),
                    torch.empty(E + 1, dtype=torch.int64, device=dev),
                    torch.empty(S * K, dtype=torch.int32, device=dev),
                    torch.empty(S, K, dtype=torch.int64, device=dev),
                    torch.empty(1, dtype=torch.int32, device=dev))
    ws = torch.empty(max(moe.moe_plan_workspace_size(S, K, E), 256), dtype=torch.uint8, device=dev)
    packed = torch.empty(S * K, H, dtype=torch.bfloat16, device=dev)
    out = torch.empty(S, H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2(v: int):
        flush.fill_(v)                 # evicts everything the step could reuse
        flush_r.sum()                  # writes the flush's dirty lines back, untimed

    # expert output rows, produced once (untimed): y = bf16(f32(x) * c_e)
    moe.moe_plan(idx, E, out=plan, workspace=ws)
    moe.moe_dispatch(x, plan.tok_map, packed_x=packed)
    c_row = torch.repeat_interleave(torch.from_numpy(wl.expert_scale).to(dev), plan.cnt.long())
    y = (packed.float() * c_row[:, None]).to(torch.bfloat16)
    torch.cuda.synchronize()
    V = int(plan.off[-1].item())
    nby = algorithmic_bytes(S, H, E, K, V)
    step_bytes = sum(nby.values())
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    # the rule moe_plan_dispatch applies: one launch up to 1024 entries, or
    # up to 131072 entries with at most 1024 per SM's token range and at most
    # 192 MiB of rows to copy; else moe_plan then moe_dispatch
    one_launch = (S * K <= int(moe.lib().moe_plan_dispatch_fused_max())
                  or (S * K <= 131072 and -(-S // n_sm) * K <= 1024
                      and S * K * H * 2 <= (192 << 20)))
    launches_per_step = (1 if one_launch else
                         (2 if moe.moe_plan_workspace_size(S, K, E) > 0 else 1) + 1) + 1

    def step():
        # plan + dispatch (moe_plan_dispatch: one launch or two), then combine
        moe.moe_plan_dispatch(idx, x, E, out=plan, packed_x=packed, workspace=ws, stream=stream)
        moe.moe_combine(y, w, plan.tok_map, out=out, stream=stream)

    sampler = ClockSampler(dev.index)
    for _ in range(args.warmup):
        flush_l2(1)
        step()
    torch.cuda.synchronize()

    n = args.steps
    # timed region 1 (the headline): whole steps, events only at step
    # boundaries, so the three launches chain as they do in use
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
    barrier(world, dev)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(n):
        flush_l2(i & 0xFF)
        ev_step[i][0].record(stream)
        step()
        ev_step[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world, dev)
    wall = time.perf_counter() - wall0

    # timed region 2 (per-call breakdown and the roofline): the same steps
    # with an event between the calls
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    barrier(world, dev)
    torch.cuda.synchronize()
    for i in range(n):
        flush_l2(i & 0xFF)
        e = ev[i]
        e[0].record(stream)
        moe.moe_plan(idx, E, out=plan, workspace=ws, stream=stream)
        e[1].record(stream)
        moe.moe_dispatch(x, plan.tok_map, packed_x=packed, stream=stream)
        e[2].record(stream)
        moe.moe_combine(y, w, plan.tok_map, out=out, stream=stream)
        e[3].record(stream)
    torch.cuda.synchronize()
    barrier(world, dev)

    # timed region 2b: the one-launch plan + dispatch of the step, per call
    ev_pd = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(n):
        flush_l2(i & 0xFF)
        e = ev_pd[i]
        e[0].record(stream)
        moe.moe_plan_dispatch(idx, x, E, out=plan, packed_x=packed, workspace=ws, stream=stream)
        e[1].record(stream)
        moe.moe_combine(y, w, plan.tok_map, out=out, stream=stream)
        e[2].record(stream)
    torch.cuda.synchronize()
    t_pd = [ev_pd[i][0].elapsed_time(ev_pd[i][1]) for i in range(n)]
    t_pd_comb = [ev_pd[i][1].elapsed_time(ev_pd[i][2]) for i in range(n)]

    # timed region 3: the same step captured once into a CUDA graph and
    # replayed (no host launch work between the calls), L2 flushed as above
    gstream = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gstream):
        def step_g():
            moe.moe_plan_dispatch(idx, x, E, out=plan, packed_x=packed, workspace=ws,
                                  stream=gstream)
            moe.moe_combine(y, w, plan.tok_map, out=out, stream=gstream)

        step_g()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=gstream):
            step_g()
        for _ in range(args.warmup):
            flush_l2(1)
            graph.replay()
        torch.cuda.synchronize()
        g_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n)]
        barrier(world, dev)
        for i in range(n):
            flush_l2(i & 0xFF)
            g_ev[i][0].record(gstream)
            graph.replay()
            g_ev[i][1].record(gstream)
        torch.cuda.synchronize()
    barrier(world, dev)
    g_max, g_bytes = aggregate(sum(a.elapsed_time(b) for a, b in g_ev), step_bytes * n, world, dev)
    clocks = sampler.stop()

    t_plan = [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]
    t_disp = [ev[i][1].elapsed_time(ev[i][2]) for i in range(n)]
    t_comb = [ev[i][2].elapsed_time(ev[i][3]) for i in range(n)]
    t_step = [a.elapsed_time(b) for a, b in ev_step]
    local_ms = sum(t_step)
    max_ms, tot_bytes = aggregate(local_ms, step_bytes * n, world, dev)
    ms_per_step = max_ms / n
    value = tot_bytes / (max_ms / 1e3) / 1e9

    # e2e: host (pinned) inputs -> GPU path -> host output, copies timed
    h_idx = torch.from_numpy(wl.topk_idx).pin_memory()
    h_w = torch.from_numpy(wl.topk_w).pin_memory()
    h_x = torch.from_numpy(wl.x.view(np.int16)).pin_memory()
    h_out = torch.empty(S, H, dtype=torch.int16).pin_memory()
    d_x16 = x.view(torch.int16)

    def e2e_step():
        idx.copy_(h_idx, non_blocking=True)
        w.copy_(h_w, non_blocking=True)
        d_x16.copy_(h_x, non_blocking=True)
        step()
        h_out.copy_(out.view(torch.int16), non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
    barrier(world, dev)
    for i in range(n):
        flush_l2(i & 0xFF)
        e2e_ev[i][0].record(stream)
        e2e_step()
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world, dev)
    e2e_local = sum(a.elapsed_time(b) for a, b in e2e_ev)
    e2e_max, e2e_bytes = aggregate(e2e_local, step_bytes * n, world, dev)
    assert np.array_equal(h_out.numpy(), out.view(torch.int16).cpu().numpy())

    # e2e, pipelined as a user would run a stream of batches: the inputs of
    # step i go host->device on one copy stream while step i-1 computes and
    # the result of step i-2 goes device->host on another; device inputs and
    # pinned host outputs are double-buffered.  Every step still copies its
    # own inputs in and its own result out inside the timed region.  The
    # step's working set (x, packed rows, y: about 1 GB) is larger than L2,
    # so no flush runs between these steps.
    e2e_pipe_ms, e2e_pipe_bytes = pipelined_e2e(torch, moe, dev, stream, n, args.warmup,
                                                h_idx, h_w, h_x, plan, ws, packed, y, E, S, H,
                                                step_bytes, world, idx, w, d_x16, out)

    peak, peak_kind = read_peaks()
    # the roofline kernel: the slowest of the step's launches, timed as they
    # run in the step -- the one-launch plan + dispatch and the combine
    # (timed region 2b), or plan, dispatch and combine (timed region 2)
    if one_launch:
        cand = {"plan_dispatch": (statistics.mean(t_pd), nby["plan"] + nby["dispatch"]),
                "combine": (statistics.mean(t_pd_comb), nby["combine"])}
    else:
        cand = {"plan": (statistics.mean(t_plan), nby["plan"]),
                "dispatch": (statistics.mean(t_disp), nby["dispatch"]),
                "combine": (statistics.mean(t_comb), nby["combine"])}
    dom = max(cand, key=lambda k_: cand[k_][0])
    dom_ms, dom_bytes = cand[dom]
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9

    def percall(name, ts, nbytes=None):
        nb = nby[name] if nbytes is None else nbytes
        m = statistics.mean(ts)
        gbs = nb / (m / 1e3) / 1e9
        return {"us": round(1e3 * m, 2), "us_median": round(1e3 * statistics.median(ts), 2),
                "us_min": round(1e3 * min(ts), 2), "us_std": round(1e3 * statistics.pstdev(ts), 2),
                "GB_per_s": round(gbs, 1),
                "frac_of_peak": round(gbs / peak, 4), "frac_of_spec": round(gbs / SPEC_HBM_GBS, 4),
                "algorithmic_bytes": nb}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": n,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "moonep: S=4096 H=7168 E=64 K=8 bf16, uniform distinct top-8, "
                               "softmax(N(0,1)) weights, per-expert scale c_e~U(0.5,1.5)",
                   "S": S, "H": H, "E": E, "K": K, "valid_rows": V,
                   "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write + "
                         f"{L2_FLUSH_BYTES >> 20} MiB read, untimed)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "step": "moe_plan_dispatch (plan + dispatch: " +
                           ("one launch" if one_launch else "moe_plan then moe_dispatch, two launches") +
                           ") + moe_combine"},
        "per_call": {"plan": percall("plan", t_plan), "dispatch": percall("dispatch", t_disp),
                     "combine": percall("combine", t_comb),
                     "plan_dispatch": percall("plan_dispatch", t_pd,
                                              nby["plan"] + nby["dispatch"]),
                     "combine_in_step": percall("combine", t_pd_comb),
                     "what": "plan, dispatch, combine: the three calls one after another; "
                             "plan_dispatch, combine_in_step: the step's two calls"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                     "algorithmic_bytes": dom_bytes, "us": round(1e3 * dom_ms, 2),
                     "peak": peak, "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "spec_peak": SPEC_HBM_GBS,
                     "frac_of_spec": round(achieved / SPEC_HBM_GBS, 4),
                     "traffic": kernel_traffic(dom)},
        "e2e": {"value": e2e_pipe_bytes / (e2e_pipe_ms / 1e3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_pipe_ms / n,
                "h2d_bytes_per_step": int(h_idx.numel() * 4 + h_w.numel() * 4 + h_x.numel() * 2),
                "d2h_bytes_per_step": int(h_out.numel() * 2),
                "mode": "pipelined: host->device copy of step i+1 and device->host copy of "
                        "step i-1 overlap step i (two copy streams, double buffers)",
                "serial": {"value": e2e_bytes / (e2e_max / 1e3) / 1e9,
                           "ms_per_step": e2e_max / n,
                           "mode": "copy in, step, copy out on one stream, L2 flushed "
                                   "between steps"}},
        "graph": {"value": g_bytes / (g_max / 1e3) / 1e9, "unit": "GB/s",
                  "ms_per_step": g_max / n,
                  "what": "the same step captured once into a CUDA graph and replayed"},
        "gpu_launches": launches_per_step * n,
        "wall_s_timed": round(wall, 4),
        "clocks": clocks,
    }
    if rank == 0:
        # the quantising dispatch on the same batch: bf16 rows in, E4M3 codes
        # and one f32 scale per 128 elements out (timed alone, L2 flushed)
        pq = torch.empty(S * K, H, dtype=torch.uint8, device=dev)
        psc = torch.empty(S * K, H // 128, dtype=torch.float32, device=dev)
        for _ in range(3):
            moe.moe_dispatch_quant_fp8(x, plan.tok_map, packed_q=pq, packed_scales=psc,
                                       stream=stream)
        qev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a_, b_ in qev:
            flush_l2(3)
            a_.record(stream)
            moe.moe_dispatch_quant_fp8(x, plan.tok_map, packed_q=pq, packed_scales=psc,
                                       stream=stream)
            b_.record(stream)
        torch.cuda.synchronize()
        tq = statistics.mean(a_.elapsed_time(b_) for a_, b_ in qev)
        qbytes = S * H * 2 + S * K * 8 + V * H + V * (H // 128) * 4
        line["dispatch_quant_fp8"] = {
            "us": round(1e3 * tq, 2), "GB_per_s": round(qbytes / (tq / 1e3) / 1e9, 1),
            "frac_of_peak": round(qbytes / (tq / 1e3) / 1e9 / peak, 4),
            "frac_of_spec": round(qbytes / (tq / 1e3) / 1e9 / SPEC_HBM_GBS, 4),
            "algorithmic_bytes": qbytes, "traffic": kernel_traffic("dispatch_quant_fp8"),
            "what": "bf16 rows -> E4M3 codes + f32 scale per 128 elements, K packed rows each"}
        del pq, psc
        # the weight fold (unweighted, with out_weights) and the capacity plan
        # on the same batch, each timed alone with L2 flushed before it
        ow = torch.empty(S, K, dtype=torch.float32, device=dev)
        cap = (S * K // E) * 5 // 4                  # 1.25 x the mean load per expert
        cplan = moe.moe_plan_capacity(idx, E, cap)
        tx = _timed_calls(torch, stream, flush_l2, {
            "combine_fold": lambda: moe.moe_combine_fold(y, w, plan.tok_map, weighted=False,
                                                         out=out, out_weights=ow, stream=stream),
            "plan_capacity": lambda: moe.moe_plan_capacity(idx, E, cap, out=cplan, workspace=ws,
                                                           stream=stream)}, n=n)
        kept = S * K - int(cplan.n_dropped.item())
        xb = {"combine_fold": V * H * 2 + S * K * (8 + 4 + 4) + S * H * 2,
              "plan_capacity": S * K * 4 + E * 4 + (E + 1) * 8 + kept * 4 + S * K * 8 + 8}
        for k_, us_ in tx.items():
            gbs = xb[k_] / (us_ * 1e-6) / 1e9
            line["per_call"][k_] = {"us": round(us_, 2), "GB_per_s": round(gbs, 1),
                                    "frac_of_peak": round(gbs / peak, 4),
                                    "frac_of_spec": round(gbs / SPEC_HBM_GBS, 4),
                                    "algorithmic_bytes": xb[k_]}
        line["per_call"]["combine_fold"]["what"] = "unweighted, with out_weights (weight fold)"
        line["per_call"]["plan_capacity"]["what"] = (f"capacity {cap} rows per expert "
                                                     f"(1.25 x mean load), {S * K - kept} dropped")
    if rank == 0 and not args.no_small_tokens:
        line["small_tokens"] = small_token_latency(dev)
    if rank == 0 and not args.no_other_workloads:
        line["other_workloads"] = other_workloads(torch, moe, dev, stream, flush_l2, peak)
        if not args.no_contended:
            line["contended"] = contended_step(torch, moe, dev, stream, idx, x, w, y, plan,
                                               packed, out, ws, E)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the Zipf and dedup per-call timings")
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the timed CPU oracle leg (profiling runs)")
    ap.add_argument("--no-small-tokens", action="store_true",
                    help="skip the small-token latency sweep (profiling runs)")
    ap.add_argument("--no-contended", action="store_true",
                    help="skip the step timed against a concurrent GEMM stream (it runs "
                         "with the other workloads)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
