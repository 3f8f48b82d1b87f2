"""Plan with a per-expert capacity (padded buckets, over-capacity entries
dropped to -1) and the dispatch / combine that run on its padded layout,
against the CPU oracle: maps, counts and rows bit-exact, combine bitwise."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from tests import gpu_path  # noqa: E402


def _run(wl, idx, cap):
    import combine_moe_plan_02_gb300 as moe
    S, K, E, H = wl.S, wl.K, wl.E, wl.H
    dev = torch.device("cuda")
    rows = E * cap
    out = moe.CapacityPlan(gpu_path.poisoned((E,), torch.int32),
                           gpu_path.poisoned((E + 1,), torch.int64),
                           gpu_path.poisoned((rows,), torch.int32),
                           gpu_path.poisoned((S, K), torch.int64),
                           gpu_path.poisoned((1,), torch.int32),
                           gpu_path.poisoned((1,), torch.int32), cap)
    t_idx = torch.from_numpy(np.ascontiguousarray(idx)).to(dev)
    moe.moe_plan_capacity(t_idx, E, cap, out=out)
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev).view(torch.bfloat16)
    packed = gpu_path.poisoned((rows, H), torch.bfloat16)
    moe.moe_dispatch(x, out.tok_map, packed_x=packed)
    w = torch.from_numpy(wl.topk_w).to(dev)
    comb = gpu_path.poisoned((S, H), torch.bfloat16)
    moe.moe_combine(packed, w, out.tok_map, out=comb)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    np_ = gpu_path._np
    return dict(cnt=np_(out.cnt), off=np_(out.off), packed_src=np_(out.packed_src),
                tok_map=np_(out.tok_map), n_invalid=int(out.n_invalid.item()),
                n_dropped=int(out.n_dropped.item()), packed=np_(packed), out=np_(comb))


def _check(wl, idx, cap):
    res = _run(wl, idx, cap)
    ref = oracle.plan_capacity(idx, wl.E, cap)
    for key in ("cnt", "off", "tok_map"):
        assert np.array_equal(res[key], ref[key]), key
    assert res["n_invalid"] == ref["n_invalid"] and res["n_dropped"] == ref["n_dropped"]
    rows = wl.E * cap
    kept = np.zeros(rows, bool)
    for e in range(wl.E):
        kept[e * cap: e * cap + ref["cnt"][e]] = True
    assert np.array_equal(res["packed_src"][kept], ref["packed_src"][kept])
    assert np.all(res["packed_src"][~kept].view(np.uint32) == 0xFFFFFFFF)   # untouched
    ref_packed = oracle.dispatch(wl.x, ref["tok_map"], rows)
    assert np.array_equal(res["packed"][kept], ref_packed[kept])
    assert np.all(res["packed"][~kept] == 0xFFFF)
    ref_out = oracle.combine(ref_packed, "bf16", wl.topk_w, ref["tok_map"], wl.H, "bf16")
    assert np.array_equal(res["out"], ref_out)
    return res, ref


@pytest.mark.timeout(600)
@pytest.mark.parametrize("S,E,K,cap", [
    (100, 8, 2, 1),          # single-tile plan, heavy dropping
    (700, 16, 4, 150),       # one launch, some drops
    (4096, 64, 8, 512),      # the MoonEP shape at its mean load: drops on busy experts
    (4096, 64, 8, 4096),     # capacity above every count: nothing dropped
    (20000, 64, 8, 1800),    # two-kernel plan
])
def test_capacity_uniform(S, E, K, cap):
    wl = workloads.make("moonep", seed=S + cap, S=S, H=64, E=E, K=K)
    res, ref = _check(wl, wl.topk_idx, cap)
    if cap >= S:
        assert ref["n_dropped"] == 0


@pytest.mark.timeout(600)
def test_capacity_zipf_drops_hot_experts():
    wl = workloads.make("zipf", seed=4, S=8192, H=64)
    cap = 8192 * 8 // 256 * 2          # twice the mean load
    res, ref = _check(wl, wl.topk_idx, cap)
    assert ref["n_dropped"] > 0 and (ref["cnt"] == cap).sum() >= 4


@pytest.mark.timeout(600)
def test_capacity_with_invalid_ids():
    wl = workloads.make("moonep", seed=9, S=900, H=32, E=32, K=4)
    idx = wl.topk_idx.copy()
    idx[::4, 1] = -1
    idx[::9, 3] = 99
    _check(wl, idx, 60)


def test_plan_replay_with_new_rows():
    """Routing-handle replay (mori #448, routing-handle note): one plan, then
    dispatch and combine of a second batch of rows with the same routing;
    both passes match the oracle run on their own rows."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("moonep", seed=71, S=333, H=1032, E=64, K=8)
    wl2 = workloads.make("moonep", seed=72, S=333, H=1032, E=64, K=8)
    dev = torch.device("cuda")
    plan = moe.moe_plan(torch.from_numpy(wl.topk_idx).to(dev), wl.E)
    w = torch.from_numpy(wl.topk_w).to(dev)
    p = oracle.plan(wl.topk_idx, wl.E)
    for rows in (wl.x, wl2.x, wl.x):
        x = torch.from_numpy(rows.view(np.int16)).to(dev).view(torch.bfloat16)
        packed = gpu_path.poisoned((wl.S * wl.K, wl.H), torch.bfloat16)
        moe.moe_dispatch(x, plan.tok_map, packed_x=packed)
        out = moe.moe_combine(packed, w, plan.tok_map)
        torch.cuda.synchronize()
        ref_packed = oracle.dispatch(rows, p["tok_map"], wl.S * wl.K)
        assert np.array_equal(gpu_path._np(packed), ref_packed)
        ref_out = oracle.combine(ref_packed, "bf16", wl.topk_w, p["tok_map"], wl.H, "bf16")
        assert np.array_equal(gpu_path._np(out), ref_out)
    assert moe.moe_device_errors() == 0


def test_quantising_dispatch_into_capacity_buckets():
    """Quantised rows into the padded buckets of a capacity plan: the kept
    rows hold the oracle's codes and scales, the rest keep the poison."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("moonep", seed=91, S=400, H=1024, E=16, K=4)
    cap = 60
    dev = torch.device("cuda")
    rows = wl.E * cap
    out = moe.moe_plan_capacity(torch.from_numpy(wl.topk_idx).to(dev), wl.E, cap)
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev).view(torch.bfloat16)
    q = gpu_path.poisoned((rows, wl.H), torch.uint8)
    sc = gpu_path.poisoned((rows, wl.H // 128), torch.float32)
    moe.moe_dispatch_quant_fp8(x, out.tok_map, packed_q=q, packed_scales=sc)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    ref = oracle.plan_capacity(wl.topk_idx, wl.E, cap)
    assert ref["n_dropped"] > 0
    q0, sc0 = oracle.quant_fp8(wl.x, 128)
    ref_q = oracle.dispatch(q0, ref["tok_map"], rows, fill=gpu_path.POISON)
    ref_s = oracle.dispatch(sc0, ref["tok_map"], rows, fill=gpu_path.POISON)
    assert np.array_equal(gpu_path._np(q), ref_q)
    assert np.array_equal(gpu_path._np(sc).view(np.uint32), ref_s.view(np.uint32))


def _dedup_over_capacity(wl, gs, cap):
    """GPU: capacity plan -> group plan -> dedup dispatch -> dedup combine
    (identity experts: y = the packed rows), every output poisoned first."""
    import combine_moe_plan_02_gb300 as moe
    S, K, E, H = wl.S, wl.K, wl.E, wl.H
    G = E // gs
    rows = E * cap
    rmax = max(S * min(K, G), 1)
    d = gpu_path.to_device(wl)
    xdt = d["x"].dtype
    cp = moe.moe_plan_capacity(d["topk_idx"], E, cap)
    gp = moe.GroupPlan(gpu_path.poisoned((G,), torch.int32), gpu_path.poisoned((G + 1,), torch.int64),
                       gpu_path.poisoned((S, K), torch.int64), gpu_path.poisoned((rmax,), torch.int32),
                       gpu_path.poisoned((rmax, K), torch.int64), gs)
    moe.moe_group_plan(d["topk_idx"], cp.tok_map, E, gs, out=gp)
    grp_x = gpu_path.poisoned((rmax, H), xdt)
    packed = gpu_path.poisoned((rows, H), xdt)
    moe.moe_dispatch_dedup(d["x"], gp, grp_x=grp_x, packed_x=packed)
    gtok = gpu_path.poisoned((rmax, H), torch.float32)
    out = gpu_path.poisoned((S, H), xdt)
    moe.moe_combine_dedup(packed, d["topk_w"], gp, gtok=gtok, out=out, out_dtype=xdt)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    R = int(gp.goff[-1].item())
    np_ = gpu_path._np
    return dict(tok_map=np_(cp.tok_map), n_dropped=int(cp.n_dropped.item()),
                gcnt=np_(gp.gcnt), goff=np_(gp.goff), gtok_map=np_(gp.gtok_map),
                grp_src=np_(gp.grp_src)[:R], grp_tok_map=np_(gp.grp_tok_map)[:R],
                grp_x=np_(grp_x)[:R], packed=np_(packed), gtok=np_(gtok)[:R], out=np_(out))


@pytest.mark.timeout(900)
@pytest.mark.parametrize("name,S,H,K,gs,cap", [
    # the dedup shape (f32, 8 groups of 8): E*cap = 34560 rows > S*K, and the
    # busiest experts drop entries
    ("dedup", 4096, 4096, 8, 8, 540),
    # heavy dropping: some group rows lose every expert they stood for
    ("dedup", 4096, 4096, 8, 8, 300),
    # bf16; K=12: one-pass dispatch by token, two-pass combine
    ("moonep", 600, 264, 12, 4, 120),
    # K=20: dispatch by group row, two-pass combine
    ("moonep", 500, 136, 20, 8, 170),
    # K=32: two-pass dispatch and combine
    ("moonep", 300, 136, 32, 2, 160),
])
def test_dedup_over_capacity_plan(name, S, H, K, gs, cap):
    """The dedup path over a capacity plan's padded rows, against the
    oracle's capacity plan -> group plan -> dedup dispatch -> dedup combine,
    bit-exact everywhere (mori #448: op-parity note, capped receive slots with
    a drop path that writes nothing out of bounds; StdMoE note)."""
    wl = workloads.make(name, seed=S + cap + K, S=S, H=H, E=64, K=K)
    rows = wl.E * cap
    res = _dedup_over_capacity(wl, gs, cap)
    cp = oracle.plan_capacity(wl.topk_idx, wl.E, cap)
    assert cp["n_dropped"] > 0 and cp["n_dropped"] == res["n_dropped"]
    assert np.array_equal(res["tok_map"], cp["tok_map"])
    assert int(cp["tok_map"].max()) >= S * K or cap * wl.E < S * K
    gp = oracle.group_plan(wl.topk_idx, cp["tok_map"], wl.E, gs)
    for key in ("gcnt", "goff", "gtok_map", "grp_src", "grp_tok_map"):
        assert np.array_equal(res[key], gp[key]), key
    ogx, opk = oracle.dispatch_dedup(wl.x, gp["grp_src"], gp["grp_tok_map"], K, rows,
                                     fill=gpu_path.POISON)
    # compared as bytes: poisoned f32 rows hold NaN patterns
    assert np.array_equal(res["grp_x"].view(np.uint8), ogx.view(np.uint8))
    assert np.array_equal(res["packed"].view(np.uint8), opk.view(np.uint8))  # rest poisoned
    dt = "f32" if wl.dtype == "f32" else "bf16"
    y = np.ascontiguousarray(opk)
    ogt, oout = oracle.combine_dedup(y, dt, wl.topk_w, gp["grp_src"], gp["grp_tok_map"],
                                     gp["gtok_map"], H, dt)
    assert np.array_equal(res["gtok"].view(np.uint32), ogt.view(np.uint32))
    assert np.array_equal(res["out"].view(np.uint16 if dt == "bf16" else np.uint32),
                          oout.view(np.uint16 if dt == "bf16" else np.uint32))
    if gs > 1 and cap <= 300:
        # group rows none of whose experts kept a slot: copied, summed to zero
        empty = np.all(gp["grp_tok_map"] < 0, axis=1)
        assert empty.any()
        assert np.all(res["gtok"][empty] == 0)
