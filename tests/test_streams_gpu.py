"""Independent batches on five streams at once: each stream runs its own plan +
dispatch + combine (and, on one of them, the dedup path) ten times over its
own buffers with no synchronisation between the streams, so kernels of
different calls overlap on the GPU.  Every stream's last results must be the
oracle's bits: the kernels keep no state between calls (no persistent
counters; MoonEP "Drop cooperative launch from the CTA-independent local
kernels": CTA-independent local kernels), and only moe_plan_static_scratch,
which is documented to share one array and is not used here, could race."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from tests import gpu_path  # noqa: E402

np_ = gpu_path._np

# (workload, S, H, E, K): one launch with every CTA ranking all entries (256-
# and 1024-thread CTAs), the token-range launch, plan then dispatch (two-
# kernel plan), and the token-range launch followed by the dedup path
CASES = [("moonep", 16, 1032, 64, 8), ("moonep", 40, 264, 1024, 8), ("moonep", 600, 520, 64, 8),
         ("moonep", 20000, 16, 64, 8), ("dedup", 900, 264, 64, 8)]


@pytest.mark.timeout(600)
def test_five_streams_at_once():
    import combine_moe_plan_02_gb300 as moe
    dev = torch.device("cuda")
    streams = [torch.cuda.Stream(dev) for _ in CASES]
    state = []
    for (name, S, H, E, K) in CASES:
        wl = workloads.make(name, seed=S + E, S=S, H=H, E=E, K=K)
        d = gpu_path.to_device(wl)
        state.append(dict(wl=wl, d=d))
    torch.cuda.synchronize()
    for _ in range(10):
        for st, s in zip(state, streams):
            wl, d = st["wl"], st["d"]
            with torch.cuda.stream(s):
                plan, px, _ = moe.moe_plan_dispatch(d["topk_idx"], d["x"], wl.E, stream=s)
                out = moe.moe_combine(px, d["topk_w"], plan.tok_map,
                                      out_dtype=d["x"].dtype, stream=s)
                st.update(plan=plan, px=px, out=out)
                if wl.group_size:
                    gp = moe.moe_group_plan(d["topk_idx"], plan.tok_map, wl.E, wl.group_size,
                                            stream=s)
                    grp_x, pk = moe.moe_dispatch_dedup(d["x"], gp, stream=s)
                    gtok, out_d = moe.moe_combine_dedup(pk, d["topk_w"], gp, stream=s)
                    st.update(gp=gp, grp_x=grp_x, gtok=gtok, out_d=out_d)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    for st in state:
        wl = st["wl"]
        p = oracle.plan(wl.topk_idx, wl.E)
        V = int(p["off"][-1])
        assert np.array_equal(np_(st["plan"].tok_map), p["tok_map"])
        opk = oracle.dispatch(wl.x, p["tok_map"], V)
        dt = "f32" if wl.x.dtype == np.float32 else "bf16"
        assert np.array_equal(np_(st["px"])[:V].view(np.uint8), opk.view(np.uint8))
        ref = oracle.combine(opk, dt, wl.topk_w, p["tok_map"], wl.H, dt)
        assert np.array_equal(np_(st["out"]).view(np.uint8), ref.view(np.uint8))
        if wl.group_size:
            ogp = oracle.group_plan(wl.topk_idx, p["tok_map"], wl.E, wl.group_size)
            R = ogp["grp_src"].shape[0]
            ogx, opd = oracle.dispatch_dedup(wl.x, ogp["grp_src"], ogp["grp_tok_map"], wl.K, V)
            rg, ro = oracle.combine_dedup(opd, dt, wl.topk_w, ogp["grp_src"], ogp["grp_tok_map"],
                                          ogp["gtok_map"], wl.H, dt)
            assert np.array_equal(np_(st["grp_x"])[:R].view(np.uint8), ogx.view(np.uint8))
            assert np.array_equal(np_(st["gtok"])[:R].view(np.uint32), rg[:R].view(np.uint32))
            assert np.array_equal(np_(st["out_d"]).view(np.uint8), ro.view(np.uint8))
