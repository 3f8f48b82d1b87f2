"""Soak: thousands of rounds with a fresh token count and a randomly chosen
call path each round, over buffers reused from round to round, with every
64th round checked bit-exactly against the CPU oracle (ROCm/mori "EPv2
internode dispatch/combine over CCO/GDA", stress-soak section: many rounds
over a set of pre-generated datasets with random token counts).

What it hunts: state that survives a call and changes the next one -- the
per-device kernel caches (shared-memory limits, occupancy), the static
scratch array of moe_plan_static_scratch, the device error words, and output
buffers left holding an earlier round's data (each checked round poisons its
outputs first, so a skipped write cannot pass as a correct one).

Paths: plan + dispatch in one call (one fused launch, the token-range launch,
or the two calls, by size) with fp8 scale rows on some datasets; the
two-kernel plan; the static-scratch plan; the capacity plan; the dedup path;
the quantising dispatch.  Each path ends in the matching combine.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from tests import gpu_path  # noqa: E402

N_ROUNDS = 2048
CHECK_EVERY = 64
S_MAX = 20000          # two-kernel plans need more than 131072 entries
S_SMALL = 4096
H_MAX = 512
BIG_ARENA = 96 << 20     # rows: packed, outputs, group rows, codes
SMALL_ARENA = 8 << 20    # maps, counts, scales
BIG = {"packed", "out", "q", "grp_x", "gtok", "y"}
STATIC_SCRATCH_BYTES = 256 * 1024

np_ = gpu_path._np


class Arenas:
    """Flat device buffers reused by every round; each round takes
    contiguous views of the sizes it needs."""

    def __init__(self, dev):
        self.buf = {}
        self.dev = dev

    def view(self, name, shape, dtype, poison=False):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        size = BIG_ARENA if name in BIG else SMALL_ARENA
        if name not in self.buf:
            self.buf[name] = torch.empty(size, dtype=torch.uint8, device=self.dev)
        assert n <= size, (name, shape)
        t = self.buf[name][:max(n, 16)].view(dtype)[:int(np.prod(shape))].view(shape)
        if poison:
            t.view(torch.uint8).fill_(gpu_path.POISON)
        return t


def _datasets():
    """Pre-generated routing, weights and rows (bf16 unless noted); some
    datasets carry ids outside [0, E), one carries repeated experts."""
    out = []
    shapes = [(8, 2, 64), (64, 8, 144), (256, 8, 272), (37, 5, 16), (64, 1, 64),
              (1024, 8, 16), (64, 4, 144), (16, 8, 272), (256, 6, 64), (64, 8, 64),
              (8, 8, 16), (128, 3, 144)]
    for i, (E, K, H) in enumerate(shapes):
        wl = workloads.make("moonep", seed=7000 + i, S=S_MAX, H=H, E=E, K=K)
        idx = wl.topk_idx.copy()
        if i % 4 == 3:
            idx[::7, 0] = -1
            idx[::11, K - 1] = E + 3
        if i == 10:
            idx[::5, 1] = idx[::5, 0]           # the same expert twice in a token
        out.append(dict(kind="bf16", E=E, K=K, H=H, idx=idx, w=wl.topk_w, x=wl.x))
    for i, H in enumerate((512, 1024)):
        wl = workloads.make("fp8small", seed=7100 + i, S=S_SMALL, H=H)
        out.append(dict(kind="fp8", E=wl.E, K=wl.K, H=H, idx=wl.topk_idx, w=wl.topk_w, x=wl.x,
                        xs=wl.x_scales))
    return out


def _to_dev(ds, dev):
    d = dict(idx=torch.from_numpy(ds["idx"]).to(dev), w=torch.from_numpy(ds["w"]).to(dev))
    if ds["kind"] == "fp8":
        d["x"] = torch.from_numpy(ds["x"]).to(dev).view(torch.float8_e4m3fn)
        d["xs"] = torch.from_numpy(ds["xs"]).to(dev)
    else:
        d["x"] = torch.from_numpy(ds["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    return d


def _plan_views(A, S, K, E, poison, rows=None):
    import combine_moe_plan_02_gb300 as moe
    return moe.Plan(A.view("cnt", (E,), torch.int32, poison),
                    A.view("off", (E + 1,), torch.int64, poison),
                    A.view("src", (max(rows or S * K, 1),), torch.int32, poison),
                    A.view("tmap", (S, K), torch.int64, poison),
                    A.view("ninv", (1,), torch.int32, poison))


def _check_plan(plan, ref, S, K):
    V = int(ref["off"][-1])
    assert np.array_equal(np_(plan.cnt), ref["cnt"])
    assert np.array_equal(np_(plan.off), ref["off"])
    assert np.array_equal(np_(plan.tok_map), ref["tok_map"])
    assert np.array_equal(np_(plan.packed_src)[:V], ref["packed_src"][:V])
    assert int(plan.n_invalid.item()) == ref["n_invalid"]


def _round(moe, A, ds, d, path, S, rng, check):
    """One round; returns after checking against the oracle when `check`."""
    E, K, H = ds["E"], ds["K"], ds["H"]
    idx, w, x = d["idx"][:S], d["w"][:S], d["x"][:S]
    xdt = x.dtype
    if path == "quant":
        blocks = [b for b in (16, 32, 64, 128, 256) if H % b == 0]
        block = int(rng.choice(blocks))
        plan = moe.moe_plan(idx, E, out=_plan_views(A, S, K, E, check))
        q = A.view("q", (S * K, H), torch.uint8, check)
        sc = A.view("qs", (S * K, H // block), torch.float32, check)
        moe.moe_dispatch_quant_fp8(x, plan.tok_map, block=block, packed_q=q, packed_scales=sc)
        if check:
            torch.cuda.synchronize()
            ref = oracle.plan(ds["idx"][:S], E)
            _check_plan(plan, ref, S, K)
            q0, sc0 = oracle.quant_fp8(np.ascontiguousarray(ds["x"][:S]), block)
            assert np.array_equal(np_(q), oracle.dispatch(q0, ref["tok_map"], S * K,
                                                         fill=gpu_path.POISON))
            assert np.array_equal(np_(sc).view(np.uint32),
                                  oracle.dispatch(sc0, ref["tok_map"], S * K,
                                                  fill=gpu_path.POISON).view(np.uint32))
        return
    if path == "capacity":
        cap = int(rng.integers(1, 2 * S * K // E + 2))
        rows = E * cap
        cp = moe.CapacityPlan(*_plan_views(A, S, K, E, check, rows),
                              A.view("ndrop", (1,), torch.int32, check), cap)
        moe.moe_plan_capacity(idx, E, cap, out=cp)
        packed = A.view("packed", (rows, H), xdt, check)
        moe.moe_dispatch(x, cp.tok_map, packed_x=packed)
        out = A.view("out", (S, H), torch.bfloat16, check)
        moe.moe_combine(packed, w, cp.tok_map, out=out)
        if check:
            torch.cuda.synchronize()
            ref = oracle.plan_capacity(ds["idx"][:S], E, cap)
            for key in ("cnt", "off", "tok_map"):
                assert np.array_equal(np_(getattr(cp, key)), ref[key]), key
            assert int(cp.n_dropped.item()) == ref["n_dropped"]
            opk = oracle.dispatch(ds["x"][:S], ref["tok_map"], rows, fill=gpu_path.POISON)
            assert np.array_equal(np_(packed), opk)
            assert np.array_equal(np_(out), oracle.combine(opk, "bf16", ds["w"][:S],
                                                           ref["tok_map"], H, "bf16"))
        return
    if path == "dedup":
        gs = int(rng.choice([g for g in (1, 2, 4, 8, 16) if E % g == 0]))
        G = E // gs
        rmax = max(S * min(K, G), 1)
        plan = moe.moe_plan(idx, E, out=_plan_views(A, S, K, E, check))
        gp = moe.GroupPlan(A.view("gcnt", (G,), torch.int32, check),
                           A.view("goff", (G + 1,), torch.int64, check),
                           A.view("gtm", (S, K), torch.int64, check),
                           A.view("gsrc", (rmax,), torch.int32, check),
                           A.view("gtk", (rmax, K), torch.int64, check), gs)
        moe.moe_group_plan(idx, plan.tok_map, E, gs, out=gp)
        grp_x = A.view("grp_x", (rmax, H), xdt, check)
        packed = A.view("packed", (S * K, H), xdt, check)
        moe.moe_dispatch_dedup(x, gp, grp_x=grp_x, packed_x=packed)
        gtok = A.view("gtok", (rmax, H), torch.float32, check)
        out = A.view("out", (S, H), torch.bfloat16, check)
        moe.moe_combine_dedup(packed, w, gp, gtok=gtok, out=out)
        if check:
            torch.cuda.synchronize()
            ref = oracle.plan(ds["idx"][:S], E)
            _check_plan(plan, ref, S, K)
            ogp = oracle.group_plan(ds["idx"][:S], ref["tok_map"], E, gs)
            R = int(ogp["goff"][-1])
            for key in ("gcnt", "goff", "gtok_map"):
                assert np.array_equal(np_(getattr(gp, key)), ogp[key]), key
            assert np.array_equal(np_(gp.grp_src)[:R], ogp["grp_src"])
            assert np.array_equal(np_(gp.grp_tok_map)[:R], ogp["grp_tok_map"])
            ogx, opk = oracle.dispatch_dedup(ds["x"][:S], ogp["grp_src"], ogp["grp_tok_map"], K,
                                             S * K, fill=gpu_path.POISON)
            assert np.array_equal(np_(grp_x)[:R], ogx)
            assert np.array_equal(np_(packed), opk)
            ogt, oout = oracle.combine_dedup(opk, "bf16", ds["w"][:S], ogp["grp_src"],
                                             ogp["grp_tok_map"], ogp["gtok_map"], H, "bf16")
            assert np.array_equal(np_(gtok)[:R].view(np.uint32), ogt.view(np.uint32))
            assert np.array_equal(np_(out), oout)
        return
    # plan + dispatch (+ scales) + combine over the packed rows
    plan = _plan_views(A, S, K, E, check)
    packed = A.view("packed", (S * K, H), xdt, check)
    ps = A.view("pscales", (S * K, d["xs"].shape[1]), torch.float32, check) if "xs" in d else None
    xs = d["xs"][:S] if "xs" in d else None
    if path == "plan_dispatch":
        moe.moe_plan_dispatch(idx, x, E, x_scales=xs, out=plan, packed_x=packed,
                              packed_scales=ps)
    else:
        if path == "static":
            L = moe.lib()
            rc = L.moe_plan_static_scratch(idx.data_ptr(), S, K, E, plan.cnt.data_ptr(),
                                           plan.off.data_ptr(), plan.packed_src.data_ptr(),
                                           plan.tok_map.data_ptr(), plan.n_invalid.data_ptr(),
                                           torch.cuda.current_stream().cuda_stream)
            assert rc == 0
        else:
            moe.moe_plan(idx, E, out=plan)
        moe.moe_dispatch(x, plan.tok_map, packed_x=packed, x_scales=xs, packed_scales=ps)
    if ds["kind"] == "bf16":
        y = packed
    else:
        y = A.view("y", (S * K, H), torch.bfloat16)
        block = H // d["xs"].shape[1]
        y.copy_((packed.float() * ps.repeat_interleave(block, dim=1)).to(torch.bfloat16))
    out = A.view("out", (S, H), torch.bfloat16, check)
    moe.moe_combine(y, w, plan.tok_map, out=out)
    if check:
        torch.cuda.synchronize()
        ref = oracle.plan(ds["idx"][:S], E)
        _check_plan(plan, ref, S, K)
        opk = oracle.dispatch(ds["x"][:S], ref["tok_map"], S * K, fill=gpu_path.POISON)
        assert np.array_equal(np_(packed), opk)
        if ds["kind"] == "bf16":
            oy = opk
        else:
            ops = oracle.dispatch(ds["xs"][:S], ref["tok_map"], S * K, fill=gpu_path.POISON)
            assert np.array_equal(np_(ps).view(np.uint32), ops.view(np.uint32))
            V = int(ref["off"][-1])
            oy = oracle.expert_dequant_fp8(opk[:V], ops[:V], H // ds["xs"].shape[1])
        assert np.array_equal(np_(out), oracle.combine(oy, "bf16", ds["w"][:S],
                                                       ref["tok_map"], H, "bf16"))


@pytest.mark.timeout(1800)
def test_soak_random_token_counts_and_paths():
    import combine_moe_plan_02_gb300 as moe
    dev = torch.device("cuda", 0)
    sets = _datasets()
    dsets = [_to_dev(ds, dev) for ds in sets]
    A = Arenas(dev)
    rng = np.random.default_rng(2024)
    assert moe.moe_device_errors() == 0
    seen = {}
    for rnd in range(N_ROUNDS):
        i = int(rng.integers(len(sets)))
        ds, d = sets[i], dsets[i]
        paths = ["plan_dispatch", "static", "capacity", "dedup"]
        if ds["kind"] == "bf16":
            paths.append("quant")
            if ds["K"] * (S_SMALL + 1) <= 131072 < ds["K"] * S_MAX:
                paths.append("two_kernel")
        else:
            paths = ["plan_dispatch", "static", "plan_dispatch"]
        path = paths[int(rng.integers(len(paths)))]
        if path in ("two_kernel",):
            S = int(rng.integers(131072 // ds["K"] + 1, S_MAX + 1))
        elif path == "static" and ds["kind"] == "bf16":
            S = int(rng.integers(1, S_MAX + 1))
            # the static array holds the tile histograms of every plan with
            # E <= 511; larger plans with more experts take moe_plan
            if moe.moe_plan_workspace_size(S, ds["K"], ds["E"]) > STATIC_SCRATCH_BYTES:
                path = "two_kernel"
        else:
            S = int(rng.integers(1, S_SMALL + 1))
        check = (rnd + 1) % CHECK_EVERY == 0
        _round(moe, A, ds, d, path, S, rng, check)
        seen[path] = seen.get(path, 0) + 1
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    assert set(seen) == {"plan_dispatch", "static", "capacity", "dedup", "quant", "two_kernel"}
