"""Pins that tie the CPU oracle to facts fixed outside it.

Each pin takes an oracle library handle so that the mutation tests can run
the same pins against deliberately broken copies of the oracle and check that
at least one pin catches each planted mistake.

Sources of the facts:
  * definitions checked a second, different way (sorting instead of cursor
    walking; numpy scatter instead of the byte-copy loop);
  * closed forms printed on the pages: with identity experts the combine
    telescopes to (sum_k w[s,k]) * x[s] (ROCm/mori "cco + flydsl
    dispatch/combine #448", StdMoE note), and the unweighted cross-group sum
    gives U[s] * x[s] with U the number of distinct destinations (same page,
    op-parity note; ROCm/mori "EPv2 internode dispatch/combine", v2-native op
    note);
  * the exact value from rational arithmetic, within the error bound of f32
    accumulation followed by one bf16 rounding;
  * library routines: torch's CPU bf16 and float8_e4m3fn conversions.
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np

import oracle

U_BF16 = 2.0 ** -8    # unit roundoff of bfloat16 (8 significant bits)
U_F32 = 2.0 ** -24    # unit roundoff of binary32


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# plan
# ---------------------------------------------------------------------------

def plan_by_sorting(idx: np.ndarray, E: int):
    """The plan computed a second way: stable-sort the valid entries by expert
    and read each entry's packed row off its sorted position."""
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    ids = np.nonzero(valid)[0]
    order = ids[np.argsort(flat[ids], kind="stable")]
    tok_map = np.full(flat.shape, -1, np.int64)
    tok_map[order] = np.arange(order.size)
    cnt = np.bincount(flat[ids], minlength=E).astype(np.int32)
    off = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int64)
    return cnt, off, tok_map.reshape(idx.shape), order.astype(np.int32), int((~valid).sum())


def pin_plan_bruteforce(lib, S=2, K=2, E=3):
    """Every topk_idx tuple over {-1, 0..E} (E itself is out of range), with
    repeats allowed, on a tiny shape."""
    vals = list(range(-1, E + 1))
    for combo in itertools.product(vals, repeat=S * K):
        idx = np.array(combo, np.int32).reshape(S, K)
        p = oracle.plan(idx, E, lib=lib)
        cnt, off, tmap, src, ninv = plan_by_sorting(idx, E)
        assert np.array_equal(p["cnt"], cnt), (combo, p["cnt"], cnt)
        assert np.array_equal(p["off"], off), (combo, p["off"], off)
        assert np.array_equal(p["tok_map"], tmap), (combo, p["tok_map"], tmap)
        assert np.array_equal(p["packed_src"], src), (combo, p["packed_src"], src)
        assert p["n_invalid"] == ninv


def pin_plan_hand_example(lib):
    """Worked by hand from the definition.  S=3, K=2, E=3:
        token 0 -> experts (2, 0); token 1 -> (0, 2); token 2 -> (1, -1)
    counts (2, 1, 2), offsets (0, 2, 3, 5); bucket 0 receives (0,1) then
    (1,0) -> rows 0, 1; bucket 1 receives (2,0) -> row 2; bucket 2 receives
    (0,0) then (1,1) -> rows 3, 4; (2,1) is unused -> -1."""
    idx = np.array([[2, 0], [0, 2], [1, -1]], np.int32)
    p = oracle.plan(idx, 3, lib=lib)
    assert p["cnt"].tolist() == [2, 1, 2]
    assert p["off"].tolist() == [0, 2, 3, 5]
    assert p["tok_map"].tolist() == [[3, 0], [1, 4], [2, -1]]
    assert p["packed_src"].tolist() == [1, 2, 4, 0, 3]
    assert p["n_invalid"] == 1


def check_plan_invariants(idx: np.ndarray, E: int, p: dict):
    """Invariants the pages fix for the StdMoE repack: counts add up to the
    number of valid entries (S*K when all valid), packed_src inverts the
    token map, unused entries hold -1, and slots are stable."""
    S, K = idx.shape
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    V = int(valid.sum())
    assert int(p["cnt"].sum()) == V
    assert int(p["off"][E]) == V
    assert np.array_equal(np.diff(p["off"]), p["cnt"].astype(np.int64))
    tm = p["tok_map"].reshape(-1)
    assert np.all(tm[~valid] == -1)
    rows = tm[valid]
    assert np.array_equal(np.sort(rows), np.arange(V))
    src = p["packed_src"]
    assert np.array_equal(src[rows], np.nonzero(valid)[0])            # src o map = id
    assert np.array_equal(tm[src], np.arange(V))                       # map o src = id
    e_of_row = np.repeat(np.arange(E), p["cnt"])
    assert np.array_equal(flat[src], e_of_row)                         # right bucket
    for e in range(E):
        seg = src[p["off"][e]:p["off"][e + 1]]
        assert np.all(np.diff(seg) > 0)                                # stable order


def pin_plan_invariants(lib):
    import workloads
    for name, kw in [("tiny", {}), ("zipf", dict(S=300, H=16)), ("moonep", dict(S=77, H=16))]:
        wl = workloads.make(name, seed=3, **kw)
        idx = wl.topk_idx.copy()
        idx[::7, -1] = -1            # some unused entries
        idx[::11, 0] = wl.E + 5      # some out-of-range entries
        p = oracle.plan(idx, wl.E, lib=lib)
        check_plan_invariants(idx, wl.E, p)
        assert p["n_invalid"] == int(((idx < 0) | (idx >= wl.E)).sum())


# ---------------------------------------------------------------------------
# group plan (dedup)
# ---------------------------------------------------------------------------

def group_plan_by_sets(idx: np.ndarray, tok_map: np.ndarray, E: int, gs: int):
    """Second method: for every token the set of groups it reaches (as a
    Python dict keyed by group, first k wins), then rows per group listed by
    increasing token."""
    S, K = idx.shape
    G = E // gs
    reps = []   # (g, s, k)
    for s in range(S):
        seen = {}
        for k in range(K):
            e = int(idx[s, k])
            if 0 <= e < E and (e // gs) not in seen:
                seen[e // gs] = k
        for g, k in seen.items():
            reps.append((g, s, k))
    reps.sort()
    gcnt = np.zeros(G, np.int32)
    for g, _, _ in reps:
        gcnt[g] += 1
    goff = np.concatenate([[0], np.cumsum(gcnt)]).astype(np.int64)
    gtok_map = np.full((S, K), -1, np.int64)
    grp_src = np.zeros(len(reps), np.int32)
    grp_tok_map = np.full((len(reps), K), -1, np.int64)
    for r, (g, s, k) in enumerate(reps):
        gtok_map[s, k] = r
        grp_src[r] = s * K + k
        for k2 in range(K):
            e2 = int(idx[s, k2])
            if 0 <= e2 < E and e2 // gs == g:
                grp_tok_map[r, k2] = tok_map[s, k2]
    return gcnt, goff, gtok_map, grp_src, grp_tok_map


def pin_group_plan_bruteforce(lib, S=2, K=3, E=4, gs=2):
    vals = list(range(-1, E + 1))
    for combo in itertools.product(vals, repeat=S * K):
        idx = np.array(combo, np.int32).reshape(S, K)
        p = oracle.plan(idx, E, lib=lib)
        gp = oracle.group_plan(idx, p["tok_map"], E, gs, lib=lib)
        ref = group_plan_by_sets(idx, p["tok_map"], E, gs)
        for name, a, b in zip(("gcnt", "goff", "gtok_map", "grp_src", "grp_tok_map"),
                              (gp["gcnt"], gp["goff"], gp["gtok_map"], gp["grp_src"],
                               gp["grp_tok_map"]), ref):
            assert np.array_equal(a, b), (combo, name, a, b)


def pin_group_plan_invariants(lib):
    import workloads
    wl = workloads.make("dedup", seed=5, S=200, H=8)
    p = oracle.plan(wl.topk_idx, wl.E, lib=lib)
    gp = oracle.group_plan(wl.topk_idx, p["tok_map"], wl.E, wl.group_size, lib=lib)
    groups = wl.topk_idx // wl.group_size
    U = np.array([len(set(row.tolist())) for row in groups])
    R = int(gp["goff"][-1])
    assert R == int(U.sum())                                 # one row per (token, group)
    # every valid (s,k) appears in exactly one group row, at its packed row
    vals = gp["grp_tok_map"][gp["grp_tok_map"] >= 0]
    assert np.array_equal(np.sort(vals), np.arange(wl.S * wl.K))
    # representatives: exactly U[s] per token, and grp_src inverts gtok_map
    assert np.array_equal((gp["gtok_map"] >= 0).sum(axis=1), U)
    rows = gp["gtok_map"][gp["gtok_map"] >= 0]
    assert np.array_equal(gp["gtok_map"].reshape(-1)[gp["grp_src"]], np.arange(R))
    assert np.array_equal(np.sort(rows), np.arange(R))


# ---------------------------------------------------------------------------
# dispatch
# ---------------------------------------------------------------------------

def pin_dispatch_scatter(lib):
    """Dispatch equals numpy's fancy-index scatter of the repeated rows;
    rows beyond the valid count keep the poison byte."""
    import workloads
    wl = workloads.make("tiny", seed=1)
    idx = wl.topk_idx.copy()
    idx[5, 1] = -1
    p = oracle.plan(idx, wl.E, lib=lib)
    V = int(p["off"][-1])
    n_out = V + 3
    packed = oracle.dispatch(wl.x, p["tok_map"], n_out, fill=0xA5, lib=lib)
    ref = np.empty_like(packed)
    ref.view(np.uint8)[:] = 0xA5
    tm = p["tok_map"].reshape(-1)
    src_tok = np.repeat(np.arange(wl.S), wl.K)
    ok = tm >= 0
    ref[tm[ok]] = wl.x[src_tok[ok]]
    assert np.array_equal(packed.view(np.uint8), ref.view(np.uint8))


def pin_dispatch_dedup(lib):
    """The dedup dispatch lands every expert row exactly where the direct
    dispatch puts it, and each group row is a copy of its token's row."""
    import workloads
    wl = workloads.make("dedup", seed=2, S=40, H=8)
    p = oracle.plan(wl.topk_idx, wl.E, lib=lib)
    gp = oracle.group_plan(wl.topk_idx, p["tok_map"], wl.E, wl.group_size, lib=lib)
    V = int(p["off"][-1])
    direct = oracle.dispatch(wl.x, p["tok_map"], V, lib=lib)
    grp_x, packed = oracle.dispatch_dedup(wl.x, gp["grp_src"], gp["grp_tok_map"], wl.K, V,
                                          lib=lib)
    assert np.array_equal(direct.view(np.uint8), packed.view(np.uint8))
    assert np.array_equal(grp_x, wl.x[gp["grp_src"] // wl.K])


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------

def combine_error_bound(terms_abs_sum: np.ndarray, exact: np.ndarray, K: int, out_bf16: bool):
    """|computed - exact| for f32 accumulation of K terms (each product
    rounded once) followed by one rounding to the output format:
    gamma_{K} * sum|terms| for the f32 part (Higham, Accuracy and Stability
    of Numerical Algorithms, 2nd ed., eq. (3.5)); then u_out * |value| for the
    final rounding, where value is the f32 result."""
    gam = K * U_F32 / (1 - K * U_F32)
    f32_err = gam * terms_abs_sum
    if not out_bf16:
        return f32_err + 1e-45
    return f32_err * (1 + U_BF16) + U_BF16 * np.abs(exact)


def pin_combine_exact_rational(lib, seed=11):
    """Against the exact rational value of sum_k w*y, within the error bound
    of the f32-accumulate, bf16-store rule."""
    import workloads
    S, H, K = 6, 16, 4
    rows = S * K
    y_f = workloads.normal(seed, 50, rows * H).astype(np.float32).reshape(rows, H)
    y = workloads.to_bf16_bits(y_f)
    w = workloads.softmax_weights(seed, S, K)
    perm = np.argsort(workloads.uniform01(seed, 51, rows), kind="stable")
    tm = perm.reshape(S, K).astype(np.int64)
    tm[2, 1] = -1
    out = oracle.combine(y, "bf16", w, tm, H, "bf16", lib=lib)
    yv = bf16_bits_to_f64(y)
    got = bf16_bits_to_f64(out)
    for s in range(S):
        for j in range(H):
            ex = Fraction(0)
            mag = 0.0
            for k in range(K):
                r = tm[s, k]
                if r < 0:
                    continue
                t = Fraction(float(w[s, k])) * Fraction(float(yv[r, j]))
                ex += t
                mag += abs(float(t))
            exf = float(ex)
            bound = combine_error_bound(np.array(mag), np.array(exf), K, True)
            assert abs(got[s, j] - exf) <= bound, (s, j, got[s, j], exf, bound)


def pin_combine_identity_telescopes(lib):
    """Identity experts: out[s] == (sum_k w[s,k]) * x[s] up to the rounding
    bound (mori #448 StdMoE note).  Unused entries drop out of the sum."""
    import workloads
    wl = workloads.make("tiny", seed=4)
    idx = wl.topk_idx.copy()
    idx[3, 0] = -1
    p = oracle.plan(idx, wl.E, lib=lib)
    packed = oracle.dispatch(wl.x, p["tok_map"], int(p["off"][-1]), lib=lib)
    out = oracle.combine(packed, "bf16", wl.topk_w, p["tok_map"], wl.H, "bf16", lib=lib)
    xs = bf16_bits_to_f64(wl.x)
    wsum = np.where(p["tok_map"] >= 0, wl.topk_w.astype(np.float64), 0.0).sum(axis=1)
    exact = wsum[:, None] * xs
    mag = np.where(p["tok_map"] >= 0, wl.topk_w.astype(np.float64), 0.0).sum(axis=1)[:, None] \
        * np.abs(xs)
    bound = combine_error_bound(mag, exact, wl.K, True)
    assert np.all(np.abs(bf16_bits_to_f64(out) - exact) <= bound)


def pin_combine_expert_scale_closed_form(lib):
    """Per-expert scale c_e between dispatch and combine:
    out[s] ~= (sum_k w[s,k] c_{e(s,k)}) x[s]."""
    import workloads
    wl = workloads.make("moonep", seed=6, S=64, H=64)
    p = oracle.plan(wl.topk_idx, wl.E, lib=lib)
    packed = oracle.dispatch(wl.x, p["tok_map"], int(p["off"][-1]), lib=lib)
    y = oracle.expert_scale_bf16(packed, p["off"], wl.expert_scale, lib=lib)
    out = oracle.combine(y, "bf16", wl.topk_w, p["tok_map"], wl.H, "bf16", lib=lib)
    xs = bf16_bits_to_f64(wl.x)
    coef = (wl.topk_w.astype(np.float64) * wl.expert_scale[wl.topk_idx].astype(np.float64))
    exact = coef.sum(axis=1)[:, None] * xs
    # the expert stage rounds each row to bf16 once more: widen by u_bf16 per term
    mag = coef.sum(axis=1)[:, None] * np.abs(xs) * (1 + U_BF16)
    bound = combine_error_bound(mag, exact, wl.K, True) + U_BF16 * mag
    assert np.all(np.abs(bf16_bits_to_f64(out) - exact) <= bound)


def pin_combine_single_k_is_copy(lib):
    """K = 1 with weight 1: the combine returns the gathered row unchanged."""
    import workloads
    wl = workloads.make("tiny", seed=7, K=1)
    p = oracle.plan(wl.topk_idx, wl.E, lib=lib)
    packed = oracle.dispatch(wl.x, p["tok_map"], int(p["off"][-1]), lib=lib)
    out = oracle.combine(packed, "bf16", np.ones((wl.S, 1), np.float32), p["tok_map"], wl.H,
                         "bf16", lib=lib)
    assert np.array_equal(out, wl.x)


def pin_combine_k_order(lib):
    """Hand-worked: f32 terms (1, 2^-24, 2^-24) with unit weights.  Added in
    increasing k, each 2^-24 is half an ulp of 1 and rounds away (ties to
    even): the result is exactly 1.  Any other order gives 1 + 2^-23."""
    y = np.array([[1.0], [2.0 ** -24], [2.0 ** -24]], np.float32)
    tm = np.array([[0, 1, 2]], np.int64)
    out = oracle.combine(y, "f32", np.ones((1, 3), np.float32), tm, 1, "f32", lib=lib)
    assert out[0, 0] == np.float32(1.0)
    tm2 = np.array([[2, 1, 0]], np.int64)
    out2 = oracle.combine(y, "f32", np.ones((1, 3), np.float32), tm2, 1, "f32", lib=lib)
    assert out2[0, 0] == np.float32(1.0 + 2.0 ** -23)


def pin_combine_dedup_closed_forms(lib):
    """Dedup combine: (a) with the softmax weights and identity experts the
    result still telescopes to (sum_k w) x; (b) with weights 1/n_g inside each
    group (n_g = the token's experts in group g) each group row returns ~x[s]
    and the unweighted cross-group sum gives U[s] x[s]."""
    import workloads
    wl = workloads.make("dedup", seed=8, S=50, H=32)
    p = oracle.plan(wl.topk_idx, wl.E, lib=lib)
    gp = oracle.group_plan(wl.topk_idx, p["tok_map"], wl.E, wl.group_size, lib=lib)
    V = int(p["off"][-1])
    packed = oracle.dispatch(wl.x, p["tok_map"], V, lib=lib)
    xs = wl.x.astype(np.float64)
    _, out = oracle.combine_dedup(packed, "f32", wl.topk_w, gp["grp_src"], gp["grp_tok_map"],
                                  gp["gtok_map"], wl.H, "f32", lib=lib)
    exact = wl.topk_w.astype(np.float64).sum(axis=1)[:, None] * xs
    mag = wl.topk_w.astype(np.float64).sum(axis=1)[:, None] * np.abs(xs)
    assert np.all(np.abs(out - exact) <= 2 * combine_error_bound(mag, exact, wl.K, False))
    groups = wl.topk_idx // wl.group_size
    n_g = np.array([[np.count_nonzero(row == g) for g in row] for row in groups], np.float32)
    w1 = (1.0 / n_g).astype(np.float32)
    _, out1 = oracle.combine_dedup(packed, "f32", w1, gp["grp_src"], gp["grp_tok_map"],
                                   gp["gtok_map"], wl.H, "f32", lib=lib)
    U = np.array([len(set(r.tolist())) for r in groups], np.float64)
    exact1 = U[:, None] * xs
    assert np.all(np.abs(out1 - exact1) <= 4 * wl.K * U_F32 * (U[:, None] * np.abs(xs)) + 1e-30)


def _group_rows_setup(lib, seed, S, H, E=64, K=8, gs=8):
    """bf16 MoonEP-like routing, its group plan, and the group-row copies of x."""
    import workloads
    wl = workloads.make("moonep", seed=seed, S=S, H=H, E=E, K=K)
    p = oracle.plan(wl.topk_idx, wl.E, lib=lib)
    gp = oracle.group_plan(wl.topk_idx, p["tok_map"], wl.E, gs, lib=lib)
    grp_x, _ = oracle.dispatch_dedup(wl.x, gp["grp_src"], gp["grp_tok_map"], wl.K,
                                     int(p["off"][-1]), lib=lib)
    U = np.array([len(set((r // gs).tolist())) for r in wl.topk_idx], np.float64)
    return wl, p, gp, grp_x, U


def _dyadic_weights(seed, S, K):
    """Weights m/256 with m in 1..255: at most 8 significant bits, so that up
    to 8 repeated f32 additions stay exact."""
    import workloads
    m = np.floor(workloads.uniform01(seed, 60, S * K) * 255.0) + 1.0
    return (m / 256.0).astype(np.float32).reshape(S, K)


def pin_combine_fold_group_rows(lib):
    """Unweighted combine over group rows with the weight fold (mori #448
    op note: an identity round trip gives comb == U*input and
    out_weights == U*wts, U = the token's distinct destinations).  With bf16
    x and U <= 8 the f32 sum U*x is exact, so out == bf16(U*x) exactly
    (bf16 rounding by torch's CPU cast); with 8-bit weights U*w is exact."""
    import torch
    wl, p, gp, grp_x, U = _group_rows_setup(lib, seed=21, S=48, H=32)
    w = _dyadic_weights(21, wl.S, wl.K)
    out, ow = oracle.combine_fold(grp_x, "bf16", w, gp["gtok_map"], wl.H, "bf16",
                                  weighted=False, lib=lib)
    ux = (U[:, None] * bf16_bits_to_f64(wl.x)).astype(np.float32)
    want = torch.from_numpy(ux).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_bits_to_f64(out), bf16_bits_to_f64(want))
    assert np.array_equal(ow.astype(np.float64), U[:, None] * w.astype(np.float64))
    # softmax weights: U*w up to the rounding of U-1 additions
    ws = wl.topk_w.astype(np.float64)
    _, ow2 = oracle.combine_fold(grp_x, "bf16", wl.topk_w, gp["gtok_map"], wl.H, "bf16",
                                 weighted=False, lib=lib)
    gam = (U * U_F32 / (1 - U * U_F32))[:, None]
    assert np.all(np.abs(ow2 - U[:, None] * ws) <= gam * U[:, None] * ws)


def pin_combine_fold_direct_map(lib):
    """Fold over the per-expert token map: every valid entry forwards the
    token's whole weight vector, so out_weights[s] == V[s] * w[s] with V the
    valid entries (unused entries drop out); the unweighted rows give V*x."""
    import workloads
    wl = workloads.make("tiny", seed=22, K=4)
    idx = wl.topk_idx.copy()
    idx[1, 0] = -1
    idx[5, :3] = wl.E
    idx[9, :] = -1
    p = oracle.plan(idx, wl.E, lib=lib)
    packed = oracle.dispatch(wl.x, p["tok_map"], max(int(p["off"][-1]), 1), lib=lib)
    w = _dyadic_weights(22, wl.S, wl.K)
    out, ow = oracle.combine_fold(packed, "bf16", w, p["tok_map"], wl.H, "f32",
                                  weighted=False, lib=lib)
    V = (p["tok_map"] >= 0).sum(axis=1).astype(np.float64)
    assert V[9] == 0 and V[5] == 1 and V[1] == 3
    assert np.array_equal(ow.astype(np.float64), V[:, None] * w.astype(np.float64))
    assert np.array_equal(out.astype(np.float64), V[:, None] * bf16_bits_to_f64(wl.x))


def pin_combine_fold_weighted_telescopes(lib):
    """Weighted mode of the fold combine is the StdMoE combine: identity
    experts give (sum over valid k of w) * x within the rounding bound."""
    import workloads
    wl = workloads.make("tiny", seed=23)
    p = oracle.plan(wl.topk_idx, wl.E, lib=lib)
    packed = oracle.dispatch(wl.x, p["tok_map"], int(p["off"][-1]), lib=lib)
    out, ow = oracle.combine_fold(packed, "bf16", wl.topk_w, p["tok_map"], wl.H, "bf16",
                                  weighted=True, fold=False, lib=lib)
    assert ow is None
    xs = bf16_bits_to_f64(wl.x)
    wsum = wl.topk_w.astype(np.float64).sum(axis=1)
    exact = wsum[:, None] * xs
    bound = combine_error_bound(wsum[:, None] * np.abs(xs), exact, wl.K, True)
    assert np.all(np.abs(bf16_bits_to_f64(out) - exact) <= bound)


# ---------------------------------------------------------------------------
# number formats and expert stages, against torch's CPU conversions
# ---------------------------------------------------------------------------

def pin_bf16_rounding(lib):
    """oracle f32->bf16 (used through a K=1, w=1, f32-in / bf16-out combine,
    which is the identity before rounding) against torch's CPU cast, over
    every upper half-word with low halves at and around the rounding ties."""
    import torch
    hi = np.arange(1 << 16, dtype=np.uint32)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], np.uint32)
    bits = ((hi[:, None] << 16) | lows[None, :]).reshape(-1)
    f = bits.view(np.float32)
    # zeros excluded: the combine starts from +0, so 0 + (-0) is +0 by IEEE rules
    keep = np.isfinite(f) & (np.abs(f) < 3.3e38) & (f != 0)
    f = np.ascontiguousarray(f[keep]).reshape(-1, 1)
    n = f.shape[0]
    tm = np.arange(n, dtype=np.int64).reshape(n, 1)
    out = oracle.combine(f, "f32", np.ones((n, 1), np.float32), tm, 1, "bf16", lib=lib)
    ref = torch.from_numpy(f.reshape(-1)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(out.reshape(-1), ref.view(np.uint16))


def pin_e4m3_table(lib):
    """All 256 E4M3 codes decode as torch's float8_e4m3fn does."""
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle.e4m3_to_f32(int(c), lib=lib) for c in range(256)], np.float32)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def pin_expert_stages(lib):
    import torch
    import workloads
    wl = workloads.make("moonep", seed=9, S=16, H=32)
    p = oracle.plan(wl.topk_idx, wl.E, lib=lib)
    packed = oracle.dispatch(wl.x, p["tok_map"], int(p["off"][-1]), lib=lib)
    y = oracle.expert_scale_bf16(packed, p["off"], wl.expert_scale, lib=lib)
    c_row = torch.from_numpy(np.repeat(wl.expert_scale, p["cnt"]))
    t = torch.from_numpy(packed.view(np.int16)).view(torch.bfloat16).float() * c_row[:, None]
    assert np.array_equal(y, t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    wl8 = workloads.make("fp8small", seed=9, S=8)
    p8 = oracle.plan(wl8.topk_idx, wl8.E, lib=lib)
    V = int(p8["off"][-1])
    q = oracle.dispatch(wl8.x, p8["tok_map"], V, lib=lib)
    sc = oracle.dispatch(wl8.x_scales, p8["tok_map"], V, lib=lib)
    y8 = oracle.expert_dequant_fp8(q, sc, 128, lib=lib)
    tq = torch.from_numpy(q).view(torch.float8_e4m3fn).float()
    ts = torch.from_numpy(sc).repeat_interleave(128, dim=1)
    ref = (tq * ts).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y8, ref)


def plan_capacity_by_sorting(idx: np.ndarray, E: int, cap: int):
    """Second method: stable-sort the valid entries by expert; an entry's
    rank in its expert is its sorted position minus the expert's first
    position; ranks below cap keep row e*cap + rank."""
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    ids = np.nonzero(valid)[0]
    order = ids[np.argsort(flat[ids], kind="stable")]
    ex = flat[order]
    first = np.searchsorted(ex, ex, side="left")
    rank = np.arange(order.size) - first
    keep = rank < cap
    tok_map = np.full(flat.shape, -1, np.int64)
    tok_map[order[keep]] = ex[keep].astype(np.int64) * cap + rank[keep]
    src = np.full(E * cap, -7, np.int32)
    src[ex[keep].astype(np.int64) * cap + rank[keep]] = order[keep]
    counts = np.bincount(flat[ids], minlength=E)
    cnt = np.minimum(counts, cap).astype(np.int32)
    off = (np.arange(E + 1) * cap).astype(np.int64)
    return cnt, off, tok_map.reshape(idx.shape), src, int((~valid).sum()), int((counts - cnt).sum())


def pin_plan_capacity_bruteforce(lib, S=2, K=2, E=3):
    vals = list(range(-1, E + 1))
    for cap in (1, 2, 3):
        for combo in itertools.product(vals, repeat=S * K):
            idx = np.array(combo, np.int32).reshape(S, K)
            p = oracle.plan_capacity(idx, E, cap, lib=lib)
            cnt, off, tmap, src, ninv, ndrop = plan_capacity_by_sorting(idx, E, cap)
            assert np.array_equal(p["cnt"], cnt), (cap, combo)
            assert np.array_equal(p["off"], off), (cap, combo)
            assert np.array_equal(p["tok_map"], tmap), (cap, combo, p["tok_map"], tmap)
            assert np.array_equal(p["packed_src"], src), (cap, combo)
            assert p["n_invalid"] == ninv and p["n_dropped"] == ndrop, (cap, combo)


def pin_plan_capacity_hand_example(lib):
    """Worked by hand.  S=3, K=2, E=3, capacity 1:
        token 0 -> (2, 0); token 1 -> (0, 2); token 2 -> (1, -1)
    expert 0 keeps (0,1), drops (1,0); expert 1 keeps (2,0); expert 2 keeps
    (0,0), drops (1,1).  Rows are e*1 + 0."""
    idx = np.array([[2, 0], [0, 2], [1, -1]], np.int32)
    p = oracle.plan_capacity(idx, 3, 1, lib=lib)
    assert p["cnt"].tolist() == [1, 1, 1]
    assert p["off"].tolist() == [0, 1, 2, 3]
    assert p["tok_map"].tolist() == [[2, 0], [-1, -1], [1, -1]]
    assert p["packed_src"].tolist() == [1, 4, 0]
    assert p["n_invalid"] == 1 and p["n_dropped"] == 2


def _e4m3_torch(vals: np.ndarray) -> np.ndarray:
    import torch
    return torch.from_numpy(np.ascontiguousarray(vals, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_e4m3_encode(lib):
    """The oracle's E4M3 encoder against torch's CPU float8_e4m3fn cast
    (round to nearest, ties to even) wherever torch does not overflow
    (|v| < 464): every bf16 value, every midpoint between neighbouring codes
    and its f32 neighbours, and random f32 values; plus saturation and NaN,
    where the oracle follows the satfinite rule."""
    import workloads
    hi = np.arange(1 << 16, dtype=np.uint32)
    bf = (hi << 16).view(np.float32)
    bf = bf[np.isfinite(bf) & (np.abs(bf) < 464)]
    codes = np.arange(0x7f, dtype=np.uint8)
    import torch
    mags = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    near = np.concatenate([near, -near])
    rnd = (np.exp(workloads.uniform01(7, 60, 20000) * 18 - 12) *
           np.where(workloads.uniform01(7, 61, 20000) < 0.5, -1, 1)).astype(np.float32)
    rnd = rnd[np.abs(rnd) < 464]
    vals = np.concatenate([bf, near, rnd]).astype(np.float32)
    got = np.array([oracle.f32_to_e4m3(float(v), lib=lib) for v in vals], np.uint8)
    assert np.array_equal(got, _e4m3_torch(vals))
    assert oracle.f32_to_e4m3(450.0, lib=lib) == 0x7E
    assert oracle.f32_to_e4m3(1e30, lib=lib) == 0x7E
    assert oracle.f32_to_e4m3(-1e30, lib=lib) == 0xFE
    assert oracle.f32_to_e4m3(float("nan"), lib=lib) & 0x7F == 0x7F


def pin_quant_fp8_rule(lib):
    """Blockwise quantisation: equals the same rule applied with numpy f32
    division and torch's cast (a library cross-check); the largest element of
    every block maps to +-448; an all-zero block has scale 1 and zero codes;
    dequantised values are within E4M3's rounding error of the input."""
    import workloads
    S, H, block = 24, 512, 128
    xf = workloads.activations_f32(9, S, H)
    xf[3, :128] = 0.0                              # an all-zero block
    xf[5, 128:256] *= 1e-6                         # a tiny block (subnormal codes)
    x = workloads.to_bf16_bits(xf)
    q, sc = oracle.quant_fp8(x, block, lib=lib)
    xv = bf16_bits_to_f64(x).astype(np.float32).reshape(S, H // block, block)
    amax = np.abs(xv).max(axis=2)
    ref_sc = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    assert np.array_equal(sc, ref_sc)
    ref_q = _e4m3_torch((xv / ref_sc[:, :, None]).astype(np.float32).reshape(S, H))
    assert np.array_equal(q, ref_q)
    assert np.all(sc[3, 0] == 1.0) and np.all(q[3, :128] == 0)
    import torch
    deq = torch.from_numpy(q).view(torch.float8_e4m3fn).float().numpy().reshape(S, H // block, block)
    top = np.abs(deq).max(axis=2)
    assert np.all((top == 448.0) | (amax == 0))
    back = deq * sc[:, :, None]
    err = np.abs(back - xv)
    assert np.all(err <= np.abs(xv) * 2.0 ** -4 + sc[:, :, None] * 2.0 ** -10 * 1.0001)


ALL_PINS = [
    pin_plan_bruteforce, pin_plan_hand_example, pin_plan_invariants,
    pin_plan_capacity_bruteforce, pin_plan_capacity_hand_example,
    pin_group_plan_bruteforce, pin_group_plan_invariants,
    pin_dispatch_scatter, pin_dispatch_dedup,
    pin_combine_exact_rational, pin_combine_identity_telescopes,
    pin_combine_expert_scale_closed_form, pin_combine_single_k_is_copy, pin_combine_k_order,
    pin_combine_dedup_closed_forms,
    pin_combine_fold_group_rows, pin_combine_fold_direct_map, pin_combine_fold_weighted_telescopes,
    pin_bf16_rounding, pin_e4m3_table, pin_expert_stages, pin_e4m3_encode, pin_quant_fp8_rule,
]
