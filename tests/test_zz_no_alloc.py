"""moe_plan_static_scratch: the plan for callers that cannot allocate a
device workspace (a host linking only this library with no device allocator,
or a process whose device memory pool forbids further cudaMalloc calls).

It is called here through the C ABI (ctypes, no Python wrapper) and checked
against the CPU oracle and against moe_plan, which takes a caller-allocated
workspace, on two calls in a row: the plan is integer work, so the tolerance
is exact equality.  The second call uses different routing and a different
shape, so leftover histograms from the first call cannot pass as correct.
One case enqueues two such calls back to back on one stream with nothing in
between, the ordering that keeps the second call's histogram kernel from
overwriting the shared array while the first call's rank kernel reads it.
This file is named to be collected last.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _plan_buffers(S, K, E, dev):
    return (torch.full((E,), -7, dtype=torch.int32, device=dev),
            torch.full((E + 1,), -7, dtype=torch.int64, device=dev),
            torch.full((max(S * K, 1),), -7, dtype=torch.int32, device=dev),
            torch.full((S, K), -7, dtype=torch.int64, device=dev),
            torch.full((1,), -7, dtype=torch.int32, device=dev))


def _static_plan(L, idx, E):
    S, K = idx.shape
    cnt, off, src, tmap, ninv = _plan_buffers(S, K, E, idx.device)
    rc = L.moe_plan_static_scratch(idx.data_ptr(), S, K, E, cnt.data_ptr(), off.data_ptr(),
                                   src.data_ptr(), tmap.data_ptr(), ninv.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    return rc, (cnt, off, src, tmap, ninv)


@pytest.mark.timeout(300)
def test_static_scratch_plan_matches_moe_plan_twice():
    import combine_moe_plan_02_gb300 as moe
    L = moe.lib()
    dev = torch.device("cuda", 0)
    cases = [
        workloads.make("moonep", seed=11, S=20000, H=8),    # 160000 entries: 79 tiles
        workloads.make("zipf", seed=12, S=17000, H=8),      # 136000 entries, skewed, E=256
    ]
    for wl in cases:
        idx = torch.from_numpy(wl.topk_idx).to(dev)
        assert moe.moe_plan_workspace_size(wl.S, wl.K, wl.E) > 0   # the scratch is used
        ref = moe.moe_plan(idx, wl.E)
        rc, got = _static_plan(L, idx, wl.E)
        assert rc == 0, L.moe_status_string(rc)
        torch.cuda.synchronize()
        V = int(ref.off[-1])
        for a, b in zip(got, (ref.cnt, ref.off, ref.packed_src, ref.tok_map, ref.n_invalid)):
            if a.numel() == ref.packed_src.numel():
                a, b = a[:V], b[:V]
            assert torch.equal(a, b)
        _check_oracle(got, wl.topk_idx, wl.E)


def _check_oracle(got, topk_idx, E):
    """Every plan output equals the CPU oracle's (plain counting, prefix sum
    and the (token, k) cursor walk)."""
    ref = oracle.plan(topk_idx, E)
    cnt, off, src, tmap, ninv = (t.cpu().numpy() for t in got)
    V = int(ref["off"][-1])
    assert np.array_equal(cnt, ref["cnt"])
    assert np.array_equal(off, ref["off"])
    assert np.array_equal(src[:V], ref["packed_src"])
    assert np.array_equal(tmap, ref["tok_map"])
    assert int(ninv[0]) == ref["n_invalid"]


@pytest.mark.timeout(300)
def test_static_scratch_back_to_back_on_one_stream():
    """Two large plans of different shapes enqueued one after the other on
    the same stream, no synchronisation between them, then a third of the
    first shape: every result equals the oracle's."""
    import combine_moe_plan_02_gb300 as moe
    L = moe.lib()
    dev = torch.device("cuda", 0)
    wls = [workloads.make("zipf", seed=21, S=18000, H=8, E=256),     # 144000 entries, 71 tiles
           workloads.make("moonep", seed=22, S=40000, H=8, E=64),    # 320000 entries, 128 tiles
           workloads.make("zipf", seed=23, S=18000, H=8, E=256)]
    idxs = [torch.from_numpy(wl.topk_idx).to(dev) for wl in wls]
    torch.cuda.synchronize()
    results = []
    for wl, idx in zip(wls, idxs):
        rc, got = _static_plan(L, idx, wl.E)     # no synchronisation in between
        assert rc == 0, L.moe_status_string(rc)
        results.append(got)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    for wl, got in zip(wls, results):
        _check_oracle(got, wl.topk_idx, wl.E)


@pytest.mark.timeout(300)
def test_static_scratch_single_tile_and_empty():
    import combine_moe_plan_02_gb300 as moe
    L = moe.lib()
    dev = torch.device("cuda", 0)
    for S in (0, 5, 1024):
        wl = workloads.make("tiny", seed=S, S=S, H=8, E=8, K=2)
        idx = torch.from_numpy(np.ascontiguousarray(wl.topk_idx)).to(dev)
        ref = moe.moe_plan(idx, wl.E)
        rc, got = _static_plan(L, idx, wl.E)
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref.cnt) and torch.equal(got[1], ref.off)
        assert torch.equal(got[3], ref.tok_map) and torch.equal(got[4], ref.n_invalid)
        _check_oracle(got, wl.topk_idx, wl.E)


@pytest.mark.timeout(300)
def test_static_scratch_rejects_plans_beyond_its_size():
    import combine_moe_plan_02_gb300 as moe
    L = moe.lib()
    dev = torch.device("cuda", 0)
    S, K, E = 32768, 8, 1024     # 128 tiles x 1025 counters x 4 bytes > 256 KiB
    assert moe.moe_plan_workspace_size(S, K, E) > 256 * 1024
    idx = torch.zeros(S, K, dtype=torch.int32, device=dev)
    rc, got = _static_plan(L, idx, E)
    assert rc == 1                                       # MOE_EINVAL, nothing launched
    torch.cuda.synchronize()
    assert int(got[4].item()) == -7                      # outputs untouched
