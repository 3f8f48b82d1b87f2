"""Calls captured once into a CUDA graph and replayed on new inputs copied
into the captured buffers: the dedup path (plan, group plan, dedup dispatch,
dedup combine), the capacity path (capacity plan, dispatch, combine, with
entries dropped) and the quantising dispatch.  Every replay must give the
oracle's bits, which it can only do if no call allocates, synchronises or
reads host state while it is captured.  The pages time their kernels
replayed from CUDA graphs (ROCm/mori "Draft: cco + flydsl dispatch/combine
#448", PR description); plan + dispatch + combine in a graph is covered in
tests/test_plan_dispatch_gpu.py."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from tests import gpu_path  # noqa: E402

np_ = gpu_path._np


def _load(dst: torch.Tensor, src: np.ndarray):
    """Copies a host array into a captured device buffer, bit for bit."""
    dst.view(torch.uint8).copy_(torch.from_numpy(np.ascontiguousarray(src)).view(torch.uint8)
                                .reshape(dst.view(torch.uint8).shape))


@pytest.mark.timeout(600)
def test_dedup_path_in_a_graph():
    import combine_moe_plan_02_gb300 as moe
    dev = torch.device("cuda")
    wls = [workloads.make("dedup", seed=90 + r, S=500, H=264) for r in range(3)]
    wl = wls[0]
    S, K, E, H, gs = wl.S, wl.K, wl.E, wl.H, wl.group_size
    idx = torch.from_numpy(wl.topk_idx).to(dev)
    w = torch.from_numpy(wl.topk_w).to(dev)
    x = torch.from_numpy(wl.x).to(dev)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        nws = max(moe.moe_plan_workspace_size(S, K, E),
                  moe.moe_group_plan_workspace_size(S, K, E, gs), 256)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)
        plan = moe.moe_plan(idx, E, workspace=ws, stream=stream)
        gp = moe.moe_group_plan(idx, plan.tok_map, E, gs, workspace=ws, stream=stream)
        grp_x, packed = moe.moe_dispatch_dedup(x, gp, stream=stream)
        gtok, out = moe.moe_combine_dedup(packed, w, gp, stream=stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            moe.moe_plan(idx, E, out=plan, workspace=ws, stream=stream)
            moe.moe_group_plan(idx, plan.tok_map, E, gs, out=gp, workspace=ws, stream=stream)
            moe.moe_dispatch_dedup(x, gp, grp_x=grp_x, packed_x=packed, stream=stream)
            moe.moe_combine_dedup(packed, w, gp, gtok=gtok, out=out, stream=stream)
    for v in wls[1:] + wls[:1]:
        _load(idx, v.topk_idx)
        _load(w, v.topk_w)
        _load(x, v.x)
        g.replay()
        torch.cuda.synchronize()
        p = oracle.plan(v.topk_idx, E)
        V = int(p["off"][-1])
        ogp = oracle.group_plan(v.topk_idx, p["tok_map"], E, gs)
        R = ogp["grp_src"].shape[0]
        ogx, opk = oracle.dispatch_dedup(v.x, ogp["grp_src"], ogp["grp_tok_map"], K, V)
        ref_gtok, ref_out = oracle.combine_dedup(opk, "f32", v.topk_w, ogp["grp_src"],
                                                 ogp["grp_tok_map"], ogp["gtok_map"], H, "f32")
        assert np.array_equal(np_(plan.tok_map), p["tok_map"])
        assert int(gp.goff[-1].item()) == R
        assert np.array_equal(np_(gp.gtok_map), ogp["gtok_map"])
        assert np.array_equal(np_(grp_x)[:R].view(np.uint32), ogx.view(np.uint32))
        assert np.array_equal(np_(packed)[:V].view(np.uint32), opk[:V].view(np.uint32))
        assert np.array_equal(np_(gtok)[:R].view(np.uint32), ref_gtok[:R].view(np.uint32))
        assert np.array_equal(np_(out).view(np.uint32), ref_out.view(np.uint32))
    assert moe.moe_device_errors() == 0


@pytest.mark.timeout(600)
def test_capacity_path_and_quantising_dispatch_in_a_graph():
    import combine_moe_plan_02_gb300 as moe
    dev = torch.device("cuda")
    wls = [workloads.make("moonep", seed=95 + r, S=700, H=1024) for r in range(3)]
    wl = wls[0]
    S, K, E, H = wl.S, wl.K, wl.E, wl.H
    cap = 80                         # below the mean load of 87.5: entries drop
    rows = E * cap
    idx = torch.from_numpy(wl.topk_idx).to(dev)
    w = torch.from_numpy(wl.topk_w).to(dev)
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev).view(torch.bfloat16)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        ws = torch.empty(max(moe.moe_plan_workspace_size(S, K, E), 256), dtype=torch.uint8,
                         device=dev)
        cp = moe.moe_plan_capacity(idx, E, cap, workspace=ws, stream=stream)
        packed = torch.empty(rows, H, dtype=torch.bfloat16, device=dev)
        q = torch.empty(rows, H, dtype=torch.float8_e4m3fn, device=dev)
        sc = torch.empty(rows, H // 128, dtype=torch.float32, device=dev)
        out = torch.empty(S, H, dtype=torch.bfloat16, device=dev)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            moe.moe_plan_capacity(idx, E, cap, out=cp, workspace=ws, stream=stream)
            moe.moe_dispatch(x, cp.tok_map, packed_x=packed, stream=stream)
            moe.moe_combine(packed, w, cp.tok_map, out=out, stream=stream)
            moe.moe_dispatch_quant_fp8(x, cp.tok_map, packed_q=q, packed_scales=sc,
                                       stream=stream)
    for v in wls[1:] + wls[:1]:
        _load(idx, v.topk_idx)
        _load(w, v.topk_w)
        _load(x, v.x)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.plan_capacity(v.topk_idx, E, cap)
        assert ref["n_dropped"] > 0
        assert int(cp.n_dropped.item()) == ref["n_dropped"]
        assert np.array_equal(np_(cp.tok_map), ref["tok_map"])
        # rows this replay maps (the others keep an earlier replay's bytes)
        mapped = np.unique(ref["tok_map"][ref["tok_map"] >= 0])
        opk = oracle.dispatch(v.x, ref["tok_map"], rows)
        assert np.array_equal(np_(packed)[mapped], opk[mapped])
        ref_out = oracle.combine(opk, "bf16", v.topk_w, ref["tok_map"], H, "bf16")
        assert np.array_equal(np_(out), ref_out)
        q0, sc0 = oracle.quant_fp8(v.x, 128)
        assert np.array_equal(np_(q)[mapped], oracle.dispatch(q0, ref["tok_map"], rows)[mapped])
        assert np.array_equal(np_(sc)[mapped].view(np.uint32),
                              oracle.dispatch(sc0, ref["tok_map"], rows)[mapped].view(np.uint32))
    assert moe.moe_device_errors() == 0
