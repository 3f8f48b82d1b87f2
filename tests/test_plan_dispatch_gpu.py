"""Plan and dispatch in one call (one fused launch for small batches, plan
then dispatch above the crossover) against the CPU oracle's plan and
dispatch: every output bit-exact, unmapped rows untouched, and the same bits
as moe_plan followed by moe_dispatch."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from tests import gpu_path  # noqa: E402

np_ = gpu_path._np


def _fused_max():
    import combine_moe_plan_02_gb300 as moe
    return int(moe.lib().moe_plan_dispatch_fused_max())


def _run(wl, idx):
    import combine_moe_plan_02_gb300 as moe
    S, K, E, H = wl.S, wl.K, wl.E, wl.H
    d = gpu_path.to_device(wl)
    rows = max(S * K, 1)
    plan = moe.Plan(gpu_path.poisoned((E,), torch.int32), gpu_path.poisoned((E + 1,), torch.int64),
                    gpu_path.poisoned((rows,), torch.int32), gpu_path.poisoned((S, K), torch.int64),
                    gpu_path.poisoned((1,), torch.int32))
    px = gpu_path.poisoned((rows, H), d["x"].dtype)
    ps = gpu_path.poisoned((rows, d["x_scales"].shape[1]), torch.float32) \
        if "x_scales" in d else None
    t_idx = torch.from_numpy(np.ascontiguousarray(idx)).cuda()
    moe.moe_plan_dispatch(t_idx, d["x"], E, x_scales=d.get("x_scales"), out=plan, packed_x=px,
                          packed_scales=ps)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    return plan, px, ps, d, t_idx


def _check(wl, idx=None):
    idx = wl.topk_idx if idx is None else idx
    plan, px, ps, d, t_idx = _run(wl, idx)
    ref = oracle.plan(idx, wl.E)
    assert np.array_equal(np_(plan.cnt), ref["cnt"])
    assert np.array_equal(np_(plan.off), ref["off"])
    assert np.array_equal(np_(plan.tok_map), ref["tok_map"])
    assert int(plan.n_invalid.item()) == ref["n_invalid"]
    V = int(ref["off"][-1])
    assert np.array_equal(np_(plan.packed_src)[:V], ref["packed_src"][:V])
    rows = max(wl.S * wl.K, 1)
    want = oracle.dispatch(wl.x, ref["tok_map"], rows, fill=gpu_path.POISON)
    assert np.array_equal(np_(px), want)       # rows past off[E] keep the poison
    if ps is not None:
        want_s = oracle.dispatch(wl.x_scales, ref["tok_map"], rows, fill=gpu_path.POISON)
        assert np.array_equal(np_(ps).view(np.uint32), want_s.view(np.uint32))
    # the same bits as the two separate calls
    import combine_moe_plan_02_gb300 as moe
    p2 = moe.moe_plan(t_idx, wl.E)
    px2 = gpu_path.poisoned((rows, wl.H), d["x"].dtype)
    ps2 = gpu_path.poisoned(tuple(ps.shape), torch.float32) if ps is not None else None
    moe.moe_dispatch(d["x"], p2.tok_map, packed_x=px2, x_scales=d.get("x_scales"),
                     packed_scales=ps2)
    torch.cuda.synchronize()
    assert torch.equal(p2.tok_map, plan.tok_map)
    assert torch.equal(px2.view(torch.uint8), px.view(torch.uint8))
    if ps is not None:
        assert torch.equal(ps2.view(torch.int32), ps.view(torch.int32))


@pytest.mark.parametrize("S", [1, 4, 8, 31, 32, 127, 128, 129, 512, 1024])
def test_fp8_rows_and_scales(S):
    """fp8 rows + 48 scales per row (H=6144, E=256, K=8): S*K = 1024 is the
    last fused size, 1032 the first two-call size."""
    _check(workloads.make("fp8small", seed=100 + S, S=S))


@pytest.mark.parametrize("S,H,E,K", [(128, 7168, 64, 8), (3, 8, 1, 1), (32, 1032, 1024, 32),
                                     (33, 256, 1024, 31), (1000, 64, 7, 1), (17, 2056, 257, 5),
                                     (102, 264, 256, 10), (1, 64, 256, 8), (60, 520, 512, 16),
                                     (90, 136, 128, 11), (7, 1040, 129, 3), (40, 264, 513, 20)])
def test_bf16_shapes(S, H, E, K):
    _check(workloads.make("moonep", seed=S + E, S=S, H=H, E=E, K=K))


@pytest.mark.parametrize("S,H,E,K", [(1536, 7168, 64, 8), (2048, 7168, 64, 8), (4096, 7168, 64, 8),
                                     (3000, 264, 1024, 32), (5000, 136, 37, 5), (16000, 16, 64, 8),
                                     (200, 6144, 256, 8)])
def test_tiled_one_launch_shapes(S, H, E, K):
    """Above 1024 entries and up to 131072 entries and 192 MiB of rows, one
    launch whose CTAs own token ranges (1536 x 7168 is near the byte limit);
    2048 x 7168 and the benchmark shape (4096 x 7168, 470 MB of rows) take
    plan then dispatch; 19456 x 8 would exceed the entry range."""
    _check(workloads.make("moonep", seed=S + K, S=S, H=H, E=E, K=K))


def test_tiled_with_scales_invalid_and_unaligned_ids():
    """fp8 rows with scale rows, invalid ids, and a topk_idx that is not
    16-byte aligned (the counting pass then reads one id at a time)."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("fp8small", seed=11, S=700)
    idx = wl.topk_idx.copy()
    idx[::7, 3] = -1
    idx[5, :] = wl.E
    _check(wl, idx)
    wl2 = workloads.make("moonep", seed=12, S=777, H=64, E=16, K=5)
    big = torch.zeros(wl2.S * wl2.K + 1, dtype=torch.int32, device="cuda")
    big[1:] = torch.from_numpy(wl2.topk_idx.reshape(-1)).cuda()
    idx_view = big[1:].view(wl2.S, wl2.K)          # 4-byte aligned only
    assert idx_view.data_ptr() % 16 != 0
    x = gpu_path.to_device(wl2)["x"]
    plan, px, _ = moe.moe_plan_dispatch(idx_view, x, wl2.E)
    torch.cuda.synchronize()
    ref = oracle.plan(wl2.topk_idx, wl2.E)
    assert np.array_equal(np_(plan.tok_map), ref["tok_map"])
    assert np.array_equal(np_(plan.cnt), ref["cnt"])
    V = int(ref["off"][-1])
    assert np.array_equal(np_(px)[:V], oracle.dispatch(wl2.x, ref["tok_map"], V))
    assert moe.moe_device_errors() == 0


def test_invalid_ids_and_repeats():
    wl = workloads.make("fp8small", seed=7, S=100)
    idx = wl.topk_idx.copy()
    idx[0, :] = -1
    idx[1, 3] = wl.E
    idx[2, :] = 5           # one expert eight times
    idx[50, 2:] = -7
    _check(wl, idx)


def test_crossover_covers_the_small_token_sizes():
    assert _fused_max() >= 32 * 8


def test_short_packed_buffer_is_flagged_not_written():
    """packed_x with fewer rows than the plan fills: the rows past its end are
    skipped and bit 1 of moe_device_errors is set."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("fp8small", seed=9, S=16)
    d = gpu_path.to_device(wl)
    guard = gpu_path.poisoned((wl.S * wl.K + 64, wl.H), d["x"].dtype)
    px = guard[:100]
    moe.moe_plan_dispatch(d["topk_idx"], d["x"], wl.E, packed_x=px)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() & 2
    assert torch.all(guard[100:].view(torch.uint8) == gpu_path.POISON)
    assert moe.moe_device_errors() == 0


def test_empty_batch():
    import combine_moe_plan_02_gb300 as moe
    idx = torch.zeros(0, 8, dtype=torch.int32, device="cuda")
    x = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    plan, _, _ = moe.moe_plan_dispatch(idx, x, 16)
    torch.cuda.synchronize()
    assert plan.cnt.sum().item() == 0 and plan.off.sum().item() == 0


@pytest.mark.timeout(900)
@pytest.mark.parametrize("S,H", [(16, 1032), (600, 1032), (4096, 3200), (20000, 16)])
def test_cuda_graph_replay(S, H):
    """Plan, dispatch and combine captured once into a CUDA graph and
    replayed on new inputs copied into the captured buffers, for every form
    of moe_plan_dispatch: one fused launch (16 tokens), the token-range
    launch (600), plan then dispatch with the dispatch's early loads (4096 x
    3200: 210 MB of rows), and the two-kernel plan then dispatch (20000
    tokens); every replay matches the oracle."""
    import combine_moe_plan_02_gb300 as moe
    dev = torch.device("cuda")
    wls = [workloads.make("moonep", seed=80 + r, S=S, H=H, E=64, K=8) for r in range(3)]
    wl = wls[0]
    idx = torch.from_numpy(wl.topk_idx).to(dev)
    w = torch.from_numpy(wl.topk_w).to(dev)
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev).view(torch.bfloat16)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        plan, px, _ = moe.moe_plan_dispatch(idx, x, wl.E, stream=stream)
        out = moe.moe_combine(px, w, plan.tok_map, stream=stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            moe.moe_plan_dispatch(idx, x, wl.E, out=plan, packed_x=px, stream=stream)
            moe.moe_combine(px, w, plan.tok_map, out=out, stream=stream)
    for v in wls[1:] + wls[:1]:
        idx.copy_(torch.from_numpy(v.topk_idx))
        w.copy_(torch.from_numpy(v.topk_w))
        x.view(torch.int16).copy_(torch.from_numpy(v.x.view(np.int16)))
        g.replay()
        torch.cuda.synchronize()
        p = oracle.plan(v.topk_idx, v.E)
        assert np.array_equal(np_(plan.tok_map), p["tok_map"])
        opk = oracle.dispatch(v.x, p["tok_map"], v.S * v.K)
        ref = oracle.combine(opk, "bf16", v.topk_w, p["tok_map"], v.H, "bf16")
        assert np.array_equal(np_(out), ref)
    assert moe.moe_device_errors() == 0
