"""MoeOp, the op interface of ROCm/mori's dispatch/combine (ROCm/mori "Draft:
cco + flydsl dispatch/combine #448", op notes: out, total_recv, routing =
op.dispatch(x, topk_w, topk_idx); combined, combined_wts = op.combine(y,
routing)), in every mode, against the CPU oracle: dispatch outputs,
total_recv, the combine and the weight fold, bitwise."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from tests import gpu_path  # noqa: E402

np_ = gpu_path._np


@pytest.mark.parametrize("weighted", [True, False])
def test_plain_mode(weighted):
    import combine_moe_plan_02_gb300 as moe
    for S in (16, 300, 2000):            # one launch, token ranges, token ranges
        wl = workloads.make("moonep", seed=S, S=S, H=1032)
        d = gpu_path.to_device(wl)
        op = moe.MoeOp(wl.E, weighted=weighted)
        out, total_recv, routing = op.dispatch(d["x"], d["topk_w"], d["topk_idx"].long())
        combined, wts = op.combine(out, routing)      # identity experts: y = out
        torch.cuda.synchronize()
        p = oracle.plan(wl.topk_idx, wl.E)
        V = int(p["off"][-1])
        assert int(total_recv.item()) == V
        opk = oracle.dispatch(wl.x, p["tok_map"], V)
        assert np.array_equal(np_(out)[:V], opk)
        ref, ref_w = oracle.combine_fold(opk, "bf16", wl.topk_w, p["tok_map"], wl.H, "bf16",
                                         weighted=weighted)
        assert np.array_equal(np_(combined), ref)
        assert np.array_equal(np_(wts).view(np.uint32), ref_w.view(np.uint32))
    assert moe.moe_device_errors() == 0


def test_fp8_rows_with_scales_and_f32_output():
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("fp8small", seed=3, S=64)
    d = gpu_path.to_device(wl)
    op = moe.MoeOp(wl.E, fold=False, out_dtype=torch.float32)
    (packed, scales), total_recv, routing = op.dispatch(d["x"], d["topk_w"], d["topk_idx"],
                                                        x_scales=d["x_scales"])
    y = gpu_path.expert_stage(wl, routing.plan, packed, scales)
    combined, wts = op.combine(y, routing)
    torch.cuda.synchronize()
    assert wts is None
    p = oracle.plan(wl.topk_idx, wl.E)
    V = int(p["off"][-1])
    assert int(total_recv.item()) == V
    assert np.array_equal(np_(packed)[:V], oracle.dispatch(wl.x, p["tok_map"], V))
    assert np.array_equal(np_(scales)[:V].view(np.uint32),
                          oracle.dispatch(wl.x_scales, p["tok_map"], V).view(np.uint32))
    ref = oracle.combine(np_(y)[:V], "bf16", wl.topk_w, p["tok_map"], wl.H, "f32")
    assert np.array_equal(np_(combined).view(np.uint32), ref.view(np.uint32))


def test_quant_mode():
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("moonep", seed=5, S=300, H=1024)
    d = gpu_path.to_device(wl)
    op = moe.MoeOp(wl.E, quant_block=128)
    (q, sc), total_recv, routing = op.dispatch(d["x"], d["topk_w"], d["topk_idx"])
    torch.cuda.synchronize()
    p = oracle.plan(wl.topk_idx, wl.E)
    V = int(p["off"][-1])
    assert int(total_recv.item()) == V
    q0, sc0 = oracle.quant_fp8(wl.x, 128)
    assert np.array_equal(np_(q)[:V], oracle.dispatch(q0, p["tok_map"], V))
    assert np.array_equal(np_(sc)[:V].view(np.uint32),
                          oracle.dispatch(sc0, p["tok_map"], V).view(np.uint32))


def test_capacity_mode():
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("moonep", seed=7, S=700, H=264)
    d = gpu_path.to_device(wl)
    cap = 80                                   # below the mean load: entries drop
    op = moe.MoeOp(wl.E, capacity=cap)
    out, total_recv, routing = op.dispatch(d["x"], d["topk_w"], d["topk_idx"])
    combined, wts = op.combine(out, routing)
    torch.cuda.synchronize()
    ref = oracle.plan_capacity(wl.topk_idx, wl.E, cap)
    assert ref["n_dropped"] > 0
    assert int(total_recv.item()) == wl.E * cap
    assert np.array_equal(np_(routing.plan.tok_map), ref["tok_map"])
    assert np.array_equal(np_(routing.plan.cnt), ref["cnt"])
    mapped = np.unique(ref["tok_map"][ref["tok_map"] >= 0])
    opk = oracle.dispatch(wl.x, ref["tok_map"], wl.E * cap)
    assert np.array_equal(np_(out)[mapped], opk[mapped])
    r_out, r_w = oracle.combine_fold(opk, "bf16", wl.topk_w, ref["tok_map"], wl.H, "bf16",
                                     weighted=True)
    assert np.array_equal(np_(combined), r_out)
    assert np.array_equal(np_(wts).view(np.uint32), r_w.view(np.uint32))


@pytest.mark.parametrize("fold", [True, False])
def test_dedup_mode(fold):
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("dedup", seed=9, S=300, H=264)
    gs = wl.group_size
    d = gpu_path.to_device(wl)
    op = moe.MoeOp(wl.E, group_size=gs, fold=fold, out_dtype=torch.float32)
    out, total_recv, routing = op.dispatch(d["x"], d["topk_w"], d["topk_idx"])
    combined, wts = op.combine(out, routing)
    torch.cuda.synchronize()
    p = oracle.plan(wl.topk_idx, wl.E)
    V = int(p["off"][-1])
    ogp = oracle.group_plan(wl.topk_idx, p["tok_map"], wl.E, gs)
    _, opk = oracle.dispatch_dedup(wl.x, ogp["grp_src"], ogp["grp_tok_map"], wl.K, V)
    r_gtok, r_out = oracle.combine_dedup(opk, "f32", wl.topk_w, ogp["grp_src"], ogp["grp_tok_map"],
                                         ogp["gtok_map"], wl.H, "f32")
    assert int(total_recv.item()) == V
    assert np.array_equal(np_(out)[:V].view(np.uint32), opk[:V].view(np.uint32))
    assert np.array_equal(np_(combined).view(np.uint32), r_out.view(np.uint32))
    if fold:
        R = ogp["grp_src"].shape[0]
        _, r_w = oracle.combine_fold(r_gtok[:R], "f32", wl.topk_w, ogp["gtok_map"], wl.H, "f32")
        assert np.array_equal(np_(wts).view(np.uint32), r_w.view(np.uint32))
        # the identity round trip: combined_wts == U * w, U = groups reached
        U = np.array([len(set((r // gs).tolist())) for r in wl.topk_idx], np.float64)
        gam = (U * 2.0 ** -24 / (1 - U * 2.0 ** -24))[:, None]
        ws = wl.topk_w.astype(np.float64)
        assert np.all(np.abs(np_(wts) - U[:, None] * ws) <= gam * U[:, None] * ws)
    else:
        assert wts is None
    assert moe.moe_device_errors() == 0
