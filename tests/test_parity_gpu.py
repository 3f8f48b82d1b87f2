"""GPU path (through the C ABI) against the CPU oracle on the same seeded inputs.

Bar: counts, offsets, maps and dispatched rows bit-exact; combine within
|gpu - ref| <= 2^-8 |ref| + 1e-6 (one bf16 unit roundoff of the reference
plus a floor), where ref is the oracle's output.  The kernels add the K
terms in the oracle's order with separately rounded f32 operations, so the
combine is also checked for bitwise equality.

Workloads: the pages' shapes (MoonEP S=4096 H=7168 K=8 E=64; Zipf-skewed
S=8192 E=256; dedup S=4096 H=4096 f32 with 8 groups of 8; fp8 H=6144 E=256 at
4..1024 tokens; the tiny case), plus ragged, empty and degenerate shapes.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from tests import gpu_path  # noqa: E402
from tests.pins import bf16_bits_to_f64  # noqa: E402

TOL_REL = 2.0 ** -8
TOL_ABS = 1e-6


def _as_f64(a: np.ndarray, dt: str) -> np.ndarray:
    return bf16_bits_to_f64(a) if dt == "bf16" else a.astype(np.float64)


def assert_combine_close(got, ref, dt, what="out"):
    g = _as_f64(got, dt)
    r = _as_f64(ref, dt)
    bad = np.abs(g - r) > TOL_REL * np.abs(r) + TOL_ABS
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside tolerance, first at " \
                          f"{np.argwhere(bad)[0]}: gpu {g[bad][0]} ref {r[bad][0]}"
    # same order of separately rounded f32 operations: identical bits
    assert np.array_equal(got, ref), f"{what}: within tolerance but not bitwise equal " \
                                     f"({int((got != ref).sum())} elements differ)"


def check_against_oracle(wl, res, ref):
    for key in ("cnt", "off", "packed_src", "tok_map"):
        assert np.array_equal(res[key], ref[key]), key
    assert res["n_invalid"] == ref["n_invalid"]
    assert np.array_equal(res["packed_x"].view(np.uint8), ref["packed_x"].view(np.uint8))
    # rows past off[E] keep the poison
    V = int(ref["off"][-1])
    assert np.all(res["packed_x_full"][V:].view(np.uint8) == gpu_path.POISON)
    if "packed_scales" in ref:
        assert np.array_equal(res["packed_scales"].view(np.uint8),
                              ref["packed_scales"].view(np.uint8))
    assert np.array_equal(res["y"].view(np.uint8), ref["y"].view(np.uint8))
    assert_combine_close(res["out"], ref["out"], wl.out_dtype)
    if "gcnt" in ref:
        for key in ("gcnt", "goff", "gtok_map", "grp_src", "grp_tok_map"):
            assert np.array_equal(res[key], ref[key]), key
        assert np.array_equal(res["grp_x"].view(np.uint8), ref["grp_x"].view(np.uint8))
        assert np.array_equal(res["packed_x_dedup"].view(np.uint8),
                              ref["packed_x_dedup"].view(np.uint8))
        assert_combine_close(res["gtok"], ref["gtok"], "f32", "gtok")
        assert_combine_close(res["out_dedup"], ref["out_dedup"], wl.out_dtype, "out_dedup")


def run_case(wl):
    ref = oracle.run_workload(wl)
    res = gpu_path.run(wl)
    check_against_oracle(wl, res, ref)
    return res, ref


# ---------------------------------------------------------------------------
# the pages' workloads at full size
# ---------------------------------------------------------------------------

@pytest.mark.timeout(600)
def test_tiny():
    run_case(workloads.make("tiny", seed=0))


@pytest.mark.timeout(600)
def test_moonep_full_size():
    """S=4096 H=7168 E=64 K=8 bf16 with per-expert scales: the benchmarked
    workload, at its full size and launch configuration."""
    run_case(workloads.make("moonep", seed=0))


@pytest.mark.timeout(600)
def test_zipf_full_size():
    res, ref = run_case(workloads.make("zipf", seed=0))
    assert ref["cnt"].max() > 20 * ref["cnt"].min()   # strong load imbalance reached


@pytest.mark.timeout(600)
def test_dedup_full_size():
    run_case(workloads.make("dedup", seed=0))


@pytest.mark.timeout(600)
@pytest.mark.parametrize("S", [0, 1])
def test_dedup_edge_tokens(S):
    run_case(workloads.make("dedup", seed=1, S=S))


@pytest.mark.parametrize("name,out_dt", [("dedup", "bf16"), ("dedup", "f32"), ("moonep", "f32"),
                                         ("moonep", "bf16")])
@pytest.mark.parametrize("H", [1032, 4096])
def test_dedup_combine_dtypes(name, out_dt, H):
    """The one-pass dedup combine for every (row, output) type pair, over
    rows whose last 256-element warp-step is ragged (H=1032) or not: group
    rows and outputs bitwise equal to the oracle's."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make(name, seed=5, S=300, H=H)
    gs = 8
    d = gpu_path.to_device(wl)
    plan = moe.moe_plan(d["topk_idx"], wl.E)
    gp = moe.moe_group_plan(d["topk_idx"], plan.tok_map, wl.E, gs)
    _, packed = moe.moe_dispatch_dedup(d["x"], gp)
    rmax = gp.grp_src.shape[0]
    gtok = gpu_path.poisoned((rmax, H), torch.float32)
    out = gpu_path.poisoned((wl.S, H), torch.float32 if out_dt == "f32" else torch.bfloat16)
    moe.moe_combine_dedup(packed, d["topk_w"], gp, gtok=gtok, out=out, out_dtype=out.dtype)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    p = oracle.plan(wl.topk_idx, wl.E)
    ogp = oracle.group_plan(wl.topk_idx, p["tok_map"], wl.E, gs)
    V = int(p["off"][-1])
    _, opk = oracle.dispatch_dedup(wl.x, ogp["grp_src"], ogp["grp_tok_map"], wl.K, V)
    in_dt = "f32" if wl.x.dtype == np.float32 else "bf16"
    ref_gtok, ref_out = oracle.combine_dedup(opk, in_dt, wl.topk_w, ogp["grp_src"],
                                             ogp["grp_tok_map"], ogp["gtok_map"], H, out_dt)
    R = int(gp.goff[-1].item())
    assert R == ogp["grp_src"].shape[0]
    assert np.array_equal(gpu_path._np(gtok)[:R].view(np.uint32), ref_gtok[:R].view(np.uint32))
    assert np.array_equal(gpu_path._np(out).view(np.uint8), ref_out.view(np.uint8))


@pytest.mark.timeout(600)
@pytest.mark.parametrize("S", workloads.FP8_SWEEP_TOKENS)
def test_fp8_small_token_sweep(S):
    run_case(workloads.make("fp8small", seed=2, S=S))


# ---------------------------------------------------------------------------
# ragged, degenerate and edge shapes
# ---------------------------------------------------------------------------

@pytest.mark.timeout(600)
@pytest.mark.parametrize("S,H,E,K", [
    (1, 8, 1, 1),          # smallest everything
    (3, 16, 4, 3),         # K not dividing 32
    (1023, 64, 8, 8),      # single tile, ragged
    (1024, 64, 8, 8),      # exactly 8192 entries: largest single-tile plan
    (1025, 64, 8, 8),      # first multi-tile plan, ragged last tile
    (16384, 8, 64, 8),     # largest one-launch multi-tile plan (131072 entries)
    (16385, 8, 64, 8),     # smallest two-kernel plan
    (2999, 136, 64, 6),    # K = 6, odd row of 17 vectors
    (777, 24, 1024, 32),   # E = 1024 (largest), K = 32
    (5000, 256, 37, 5),    # E not a power of two
    (40000, 16, 256, 8),   # many tiles (320000 entries)
    (524288, 8, 1024, 8),  # 4.2M entries: two-kernel plan over 128 tiles, E = 1024
    (131072, 8, 512, 32),  # K = 32 at 4.2M entries
])
def test_shapes(S, H, E, K):
    run_case(workloads.make("moonep", seed=S + H, S=S, H=H, E=E, K=K))


@pytest.mark.timeout(600)
def test_invalid_and_unused_entries():
    wl = workloads.make("moonep", seed=5, S=2000, H=64, E=32, K=4)
    idx = wl.topk_idx.copy()
    idx[::3, 1] = -1
    idx[::5, 2] = wl.E
    idx[7, :] = -1          # a token that goes nowhere: its output row is 0
    idx[::13, 0] = 1 << 30
    wl.topk_idx = idx
    res, ref = run_case(wl)
    assert res["n_invalid"] == int(((idx < 0) | (idx >= wl.E)).sum())
    assert np.all(res["out"][7] == 0)


@pytest.mark.timeout(600)
def test_repeated_expert_within_token():
    """Duplicate ids in one token each take their own slot, in k order."""
    wl = workloads.make("moonep", seed=6, S=500, H=32, E=16, K=4)
    idx = wl.topk_idx.copy()
    idx[:, 3] = idx[:, 0]
    wl.topk_idx = idx
    run_case(wl)


@pytest.mark.timeout(600)
@pytest.mark.parametrize("gs,K", [(1, 8), (2, 3), (16, 8), (64, 8), (4, 6), (2, 32), (8, 31)])
def test_dedup_group_sizes(gs, K):
    wl = workloads.make("dedup", seed=gs * 10 + K, S=700, H=64, K=K)
    wl.group_size = gs
    run_case(wl)


@pytest.mark.timeout(600)
def test_f32_output_of_bf16_combine():
    wl = workloads.make("moonep", seed=8, S=300, H=128)
    wl.out_dtype = "f32"
    run_case(wl)


# ---------------------------------------------------------------------------
# properties
# ---------------------------------------------------------------------------

@pytest.mark.timeout(900)
def test_bitwise_deterministic_100_launches():
    """100 launches of each step give the bits of the first (the method of
    TensorRT-LLM "cluster-scope acquire/release ... MoE GEMM scheduler",
    determinism check)."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("zipf", seed=3, S=2048, H=1024)
    d = gpu_path.to_device(wl)
    p0 = moe.moe_plan(d["topk_idx"], wl.E)
    px0, _ = moe.moe_dispatch(d["x"], p0.tok_map)
    o0 = moe.moe_combine(px0, d["topk_w"], p0.tok_map)
    V = int(p0.off[-1])
    for _ in range(100):
        p = moe.moe_plan(d["topk_idx"], wl.E)
        px, _ = moe.moe_dispatch(d["x"], p.tok_map)
        o = moe.moe_combine(px, d["topk_w"], p.tok_map)
        assert torch.equal(p.tok_map, p0.tok_map) and torch.equal(p.off, p0.off)
        assert torch.equal(p.packed_src[:V], p0.packed_src[:V])
        assert torch.equal(px[:V].view(torch.int16), px0[:V].view(torch.int16))
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16))


@pytest.mark.timeout(600)
def test_identity_experts_telescope_at_full_size():
    """With identity experts the combine returns (sum_k w) * x (mori #448,
    StdMoE note), checked on the GPU output directly."""
    wl = workloads.make("tiny", seed=0, S=4096, H=7168, E=64, K=8)
    res = gpu_path.run(wl)
    x = bf16_bits_to_f64(wl.x)
    ref = wl.topk_w.astype(np.float64).sum(axis=1)[:, None] * x
    got = bf16_bits_to_f64(res["out"])
    assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 8 * 2 ** -24 * np.abs(x) * 1.01)


@pytest.mark.timeout(600)
def test_no_device_errors_after_runs():
    import combine_moe_plan_02_gb300 as moe
    gpu_path.run(workloads.make("tiny", seed=0))
    assert moe.moe_device_errors() == 0


def test_bounded_wait_times_out_and_reports():
    """The dispatch kernels' mbarrier wait, run against a phase that nothing
    completes, gives up after its limit, sets the timeout bit and leaves the
    context usable (a plan runs right after and is checked)."""
    import combine_moe_plan_02_gb300 as moe
    L = moe.lib()
    assert moe.moe_device_errors() == 0
    assert L.moe_selftest_wait_timeout(2_000_000, None) == 0     # 2 ms
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 1
    assert moe.moe_device_errors() == 0                          # read clears
    assert L.moe_selftest_wait_timeout(10, None) == 1            # below 1 us: EINVAL
    wl = workloads.make("tiny", seed=5)
    d = gpu_path.to_device(wl)
    plan = moe.moe_plan(d["topk_idx"], wl.E)
    torch.cuda.synchronize()
    ref = oracle.plan(wl.topk_idx, wl.E)
    assert np.array_equal(plan.tok_map.cpu().numpy(), ref["tok_map"])


@pytest.mark.timeout(600)
def test_dispatch_several_chunks_per_warp():
    """A batch large enough that the dispatch grid (capped at a few resident
    waves) gives warps more than one chunk, so each warp's stage is reused:
    S=80000 rows of 4 KB, K=2.  Every packed row equals the oracle's."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("moonep", seed=77, S=80000, H=2048, E=64, K=2)
    d = gpu_path.to_device(wl)
    plan = moe.moe_plan(d["topk_idx"], wl.E)
    packed = gpu_path.poisoned((wl.S * wl.K, wl.H), torch.bfloat16)
    moe.moe_dispatch(d["x"], plan.tok_map, packed_x=packed)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    ref = oracle.plan(wl.topk_idx, wl.E)
    assert np.array_equal(gpu_path._np(plan.tok_map), ref["tok_map"])
    want = oracle.dispatch(wl.x, ref["tok_map"], wl.S * wl.K, fill=gpu_path.POISON)
    assert np.array_equal(gpu_path._np(packed), want)


@pytest.mark.timeout(600)
@pytest.mark.parametrize("S,E,gs,K", [(4096, 64, 8, 8), (3000, 256, 4, 6), (16384, 64, 2, 8)])
def test_group_plan_with_and_without_workspace(S, E, gs, K):
    """The group plan counts each tile once when given its workspace (two
    kernels) and lets every CTA count all entries without it (one launch):
    both give the oracle's group plan."""
    import combine_moe_plan_02_gb300 as moe
    L = moe.lib()
    wl = workloads.make("moonep", seed=S + gs, S=S, H=8, E=E, K=K)
    dev = torch.device("cuda")
    idx = torch.from_numpy(wl.topk_idx).to(dev)
    plan = moe.moe_plan(idx, E)
    G = E // gs
    rmax = S * min(K, G)
    need = int(L.moe_group_plan_workspace_size(S, K, E, gs))
    assert need > 0
    ref = oracle.group_plan(wl.topk_idx, oracle.plan(wl.topk_idx, E)["tok_map"], E, gs)
    R = int(ref["goff"][-1])
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    for ptr, nbytes in ((ws.data_ptr(), need), (None, 0)):
        out = [gpu_path.poisoned((G,), torch.int32), gpu_path.poisoned((G + 1,), torch.int64),
               gpu_path.poisoned((S, K), torch.int64), gpu_path.poisoned((rmax,), torch.int32),
               gpu_path.poisoned((rmax, K), torch.int64)]
        rc = L.moe_group_plan(idx.data_ptr(), plan.tok_map.data_ptr(), S, K, E, gs,
                              *[t.data_ptr() for t in out], ptr, nbytes,
                              torch.cuda.current_stream().cuda_stream)
        assert rc == 0, L.moe_status_string(rc)
        torch.cuda.synchronize()
        np_ = gpu_path._np
        assert np.array_equal(np_(out[0]), ref["gcnt"])
        assert np.array_equal(np_(out[1]), ref["goff"])
        assert np.array_equal(np_(out[2]), ref["gtok_map"])
        assert np.array_equal(np_(out[3])[:R], ref["grp_src"])
        assert np.array_equal(np_(out[4])[:R], ref["grp_tok_map"])
    assert moe.moe_device_errors() == 0
