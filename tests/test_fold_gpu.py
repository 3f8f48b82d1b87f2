"""Combine with the weight fold (unweighted or weighted rows over a token map,
plus out_weights = the sum of the forwarded weight vectors) against the CPU
oracle, bitwise, and against the closed forms U*x and U*w of the identity
round trip over group rows (ROCm/mori "Draft: cco + flydsl dispatch/combine
#448", combine-weight-fold and op notes)."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from tests import gpu_path  # noqa: E402

np_ = gpu_path._np


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _group_rows_gpu(wl, gs):
    """GPU plan -> group plan -> dedup dispatch; returns the group plan and
    the group rows grp_x (one copy of x[s] per (token, group))."""
    import combine_moe_plan_02_gb300 as moe
    d = gpu_path.to_device(wl)
    plan = moe.moe_plan(d["topk_idx"], wl.E)
    gp = moe.moe_group_plan(d["topk_idx"], plan.tok_map, wl.E, gs)
    grp_x = gpu_path.poisoned((gp.max_rows, wl.H), d["x"].dtype)
    packed = gpu_path.poisoned((max(wl.S * wl.K, 1), wl.H), d["x"].dtype)
    moe.moe_dispatch_dedup(d["x"], gp, grp_x=grp_x, packed_x=packed)
    return d, plan, gp, grp_x


@pytest.mark.parametrize("H", [8, 1032, 7168])
@pytest.mark.parametrize("gs", [1, 8, 64])
def test_fold_over_group_rows_is_U_times(H, gs):
    """Identity per-group stage: out == bf16(U*x) and out_weights ~ U*w;
    both bitwise equal to the oracle."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("moonep", seed=31 + gs, S=300, H=H)
    d, plan, gp, grp_x = _group_rows_gpu(wl, gs)
    out = gpu_path.poisoned((wl.S, H), torch.bfloat16)
    ow = gpu_path.poisoned((wl.S, wl.K), torch.float32)
    moe.moe_combine_fold(grp_x, d["topk_w"], gp.gtok_map, weighted=False, out=out,
                         out_weights=ow)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    p = oracle.plan(wl.topk_idx, wl.E)
    ogp = oracle.group_plan(wl.topk_idx, p["tok_map"], wl.E, gs)
    assert np.array_equal(np_(gp.gtok_map), ogp["gtok_map"])
    ogx, _ = oracle.dispatch_dedup(wl.x, ogp["grp_src"], ogp["grp_tok_map"], wl.K,
                                   int(p["off"][-1]))
    ref_out, ref_ow = oracle.combine_fold(ogx, "bf16", wl.topk_w, ogp["gtok_map"], H, "bf16")
    assert np.array_equal(np_(out), ref_out)
    assert np.array_equal(np_(ow).view(np.uint32), ref_ow.view(np.uint32))
    U = np.array([len(set((r // gs).tolist())) for r in wl.topk_idx], np.float64)
    xf = (wl.x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    want = torch.from_numpy((U[:, None] * xf).astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(out.cpu().float(), want.float())
    ws = wl.topk_w.astype(np.float64)
    gam = (U * 2.0 ** -24 / (1 - U * 2.0 ** -24))[:, None]
    assert np.all(np.abs(np_(ow) - U[:, None] * ws) <= gam * U[:, None] * ws)


@pytest.mark.parametrize("weighted", [False, True])
def test_fold_over_token_map_with_unused_entries(weighted):
    """Per-expert map with invalid ids: V copies per token; weighted mode is
    bitwise the plain combine."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("moonep", seed=41, S=257, H=1032)
    idx = wl.topk_idx.copy()
    idx[3, 0] = -1
    idx[10, :5] = wl.E
    idx[20, :] = -1
    dev = torch.device("cuda")
    plan = moe.moe_plan(torch.from_numpy(idx).to(dev), wl.E)
    x = _bf16_dev(wl.x)
    packed = gpu_path.poisoned((wl.S * wl.K, wl.H), torch.bfloat16)
    moe.moe_dispatch(x, plan.tok_map, packed_x=packed)
    w = torch.from_numpy(wl.topk_w).to(dev)
    out = gpu_path.poisoned((wl.S, wl.H), torch.float32)
    ow = gpu_path.poisoned((wl.S, wl.K), torch.float32)
    moe.moe_combine_fold(packed, w, plan.tok_map, weighted=weighted, out=out, out_weights=ow)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    p = oracle.plan(idx, wl.E)
    opk = oracle.dispatch(wl.x, p["tok_map"], wl.S * wl.K)
    ref_out, ref_ow = oracle.combine_fold(opk, "bf16", wl.topk_w, p["tok_map"], wl.H, "f32",
                                          weighted=weighted)
    assert np.array_equal(np_(out).view(np.uint32), ref_out.view(np.uint32))
    assert np.array_equal(np_(ow).view(np.uint32), ref_ow.view(np.uint32))
    assert np_(ow)[20].tolist() == [0.0] * wl.K
    if weighted:
        plain = moe.moe_combine(packed, w, plan.tok_map, out_dtype=torch.float32)
        assert torch.equal(plain.view(torch.int32), out.view(torch.int32))


def test_fold_f32_rows_no_weights():
    """f32 rows, unweighted, no fold and no weight pointer at all."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("dedup", seed=43, S=129, H=264)
    d, plan, gp, grp_x = _group_rows_gpu(wl, wl.group_size)
    out, ow = moe.moe_combine_fold(grp_x, None, gp.gtok_map, weighted=False, fold=False,
                                   out_dtype=torch.float32)
    assert ow is None
    torch.cuda.synchronize()
    p = oracle.plan(wl.topk_idx, wl.E)
    ogp = oracle.group_plan(wl.topk_idx, p["tok_map"], wl.E, wl.group_size)
    ogx, _ = oracle.dispatch_dedup(wl.x, ogp["grp_src"], ogp["grp_tok_map"], wl.K,
                                   int(p["off"][-1]))
    ref_out, _ = oracle.combine_fold(ogx, "f32", wl.topk_w, ogp["gtok_map"], wl.H, "f32",
                                     fold=False)
    assert np.array_equal(np_(out).view(np.uint32), ref_out.view(np.uint32))


def test_fold_K32_and_K1():
    import combine_moe_plan_02_gb300 as moe
    for K in (32, 1):
        wl = workloads.make("moonep", seed=44 + K, S=65, H=520, K=K)
        d = gpu_path.to_device(wl)
        plan = moe.moe_plan(d["topk_idx"], wl.E)
        packed = gpu_path.poisoned((wl.S * K, wl.H), torch.bfloat16)
        moe.moe_dispatch(d["x"], plan.tok_map, packed_x=packed)
        out, ow = moe.moe_combine_fold(packed, d["topk_w"], plan.tok_map, weighted=True)
        torch.cuda.synchronize()
        p = oracle.plan(wl.topk_idx, wl.E)
        opk = oracle.dispatch(wl.x, p["tok_map"], wl.S * K)
        ref_out, ref_ow = oracle.combine_fold(opk, "bf16", wl.topk_w, p["tok_map"], wl.H, "bf16",
                                              weighted=True)
        assert np.array_equal(np_(out), ref_out), K
        assert np.array_equal(np_(ow).view(np.uint32), ref_ow.view(np.uint32)), K


def test_fold_empty_batch():
    import combine_moe_plan_02_gb300 as moe
    y = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    tm = torch.zeros(0, 4, dtype=torch.int64, device="cuda")
    w = torch.zeros(0, 4, dtype=torch.float32, device="cuda")
    out, ow = moe.moe_combine_fold(y, w, tm)
    assert out.shape == (0, 64) and ow.shape == (0, 4)


def test_combine_alternating_K_in_one_process():
    """Calls whose shared-memory needs differ (K = 8, 1, 2, 8, 16, 2) in one
    process: a smaller call must not lower the limit a larger one relies on."""
    import combine_moe_plan_02_gb300 as moe
    for K in (8, 1, 2, 8, 16, 2):
        wl = workloads.make("moonep", seed=60 + K, S=40, H=264, K=K)
        d = gpu_path.to_device(wl)
        plan = moe.moe_plan(d["topk_idx"], wl.E)
        packed = gpu_path.poisoned((wl.S * K, wl.H), torch.bfloat16)
        moe.moe_dispatch(d["x"], plan.tok_map, packed_x=packed)
        out = moe.moe_combine(packed, d["topk_w"], plan.tok_map)
        torch.cuda.synchronize()
        p = oracle.plan(wl.topk_idx, wl.E)
        opk = oracle.dispatch(wl.x, p["tok_map"], wl.S * K)
        ref = oracle.combine(opk, "bf16", wl.topk_w, p["tok_map"], wl.H, "bf16")
        assert np.array_equal(np_(out), ref), K


@pytest.mark.timeout(900)
@pytest.mark.parametrize("weighted", [False, True])
def test_fold_headline_shape(weighted):
    """The MoonEP shape (S=4096 H=7168 E=64 K=8, bf16, per-expert scales
    between dispatch and combine), unweighted and weighted, with
    out_weights: every output element and every folded weight bitwise equal
    to the oracle's, whose plan, dispatch and expert stage run on their own."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("moonep", seed=0)
    d = gpu_path.to_device(wl)
    plan = moe.moe_plan(d["topk_idx"], wl.E)
    packed = gpu_path.poisoned((wl.S * wl.K, wl.H), torch.bfloat16)
    moe.moe_dispatch(d["x"], plan.tok_map, packed_x=packed)
    y = gpu_path.expert_stage(wl, plan, packed, None)
    out = gpu_path.poisoned((wl.S, wl.H), torch.bfloat16)
    ow = gpu_path.poisoned((wl.S, wl.K), torch.float32)
    moe.moe_combine_fold(y, d["topk_w"], plan.tok_map, weighted=weighted, out=out,
                         out_weights=ow)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    p = oracle.plan(wl.topk_idx, wl.E)
    V = int(p["off"][-1])
    opk = oracle.dispatch(wl.x, p["tok_map"], V)
    oy = oracle.expert_scale_bf16(opk, p["off"], wl.expert_scale)
    assert np.array_equal(np_(y)[:V], oy)
    ref_out, ref_ow = oracle.combine_fold(oy, "bf16", wl.topk_w, p["tok_map"], wl.H, "bf16",
                                          weighted=weighted)
    assert np.array_equal(np_(out), ref_out)
    assert np.array_equal(np_(ow).view(np.uint32), ref_ow.view(np.uint32))
