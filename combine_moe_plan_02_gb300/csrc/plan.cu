// Plan: per-expert histogram, exclusive scan and stable slot assignment.
//
// Sources: ROCm/mori "Draft: cco + flydsl dispatch/combine #448", StdMoE note
// (packed_cnt / packed_src / i64 slot map with -1) and routing-handle note
// (local_expert_count); the same page's PR description (ballot dedup per
// destination) for the group plan.  The pages hand out slots with atomics;
// here the slot of entry (s,k) is its rank among earlier entries of the same
// expert in (token, k) order, so the map is a pure function of topk_idx.
//
// Design (no inter-CTA spin waits and no cooperative launch: every CTA is
// independent, as MoonEP "Drop cooperative launch from the CTA-independent
// local kernels" argues for local kernels):
//   the flat entry list i = s*K + k is cut into T tiles of `tile` entries;
//   a tile is cut into 32 warp sub-tiles of `sub` entries, walked in chunks
//   of 32 consecutive entries (one per lane).
//   kernel 1 (large plans only): per-tile key histograms -> workspace
//     [T][nkeys + 1] (last column: invalid entries).
//   kernel 2, one CTA per tile:
//     (a) per-warp key counts: lanes holding the same key find each other
//         with __match_any_sync and the lowest lane adds the group size;
//     (b) the global counts and the counts of earlier tiles: from (a) when
//         there is one tile (up to 1024 entries); else, for plans of up to
//         128K entries, every CTA counts all entries itself (shared-memory
//         atomics over 16-byte loads; the redundant pass costs less than a
//         second launch, and for the direct plan it also yields the per-warp
//         counts of (a)); else after a programmatic-dependent-launch wait,
//         from kernel 1's tile histograms;
//     (c) a block scan over keys gives off[];
//     (d) a scan over the 32 warps per key (thread e walks key e's
//         column) gives each warp's base;
//     (e) the warps walk their chunks again: rank = warp base + running
//         count + popc(match mask & lanemask_lt).
// The group plan (dedup) runs the same two kernels on the key "group of
// the entry, if it is its token's first entry in that group".

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int64_t kSingleTileMax = 1024;   // entries handled by one CTA alone
#ifndef MOE_PLAN_FUSED_MAX
#define MOE_PLAN_FUSED_MAX 131072
#endif
#ifndef MOE_PLAN_TWO_KERNEL_MIN_TILE
#define MOE_PLAN_TWO_KERNEL_MIN_TILE 2048
#endif
constexpr int64_t kFusedMax = MOE_PLAN_FUSED_MAX;  // entries every CTA can count by itself
constexpr int64_t kMaxTiles = 128;

// How the counts reach each tile:
//   kModeSingle    one tile: its own per-warp counts are the global counts;
//   kModeFused     every tile's CTA counts all n entries itself (one launch,
//                  no workspace; n <= kFusedMax keeps that redundant pass short);
//   kModeTwoKernel a histogram kernel writes per-tile counts to the workspace.
enum PlanMode { kModeSingle = 0, kModeFused = 1, kModeTwoKernel = 2 };

struct PlanGeom {
    int64_t n;      // entries S*K
    int64_t tile;   // entries per tile (multiple of kThreads)
    int64_t sub;    // entries per warp sub-tile (multiple of 32)
    int T;          // tiles
    int mode;       // PlanMode
};

// split_counting: use the two-kernel mode above one tile, so that every
// tile is counted once (by kernel 1) instead of by every CTA.  The group plan
// asks for it: its key (is this entry its token's first in its group?) costs
// far more per entry than the plain plan's, and at S=4096 K=8 with 8 groups
// the two kernels take 12.3 us against 26.6 us for the one launch in which
// every CTA counts all entries (the plain plan: 12.3 us either way).
PlanGeom plan_geom(int64_t S, int K, bool split_counting = false)
{
    PlanGeom g;
    g.n = S * (int64_t)K;
    int64_t tile;
    if (g.n <= kSingleTileMax) {
        tile = (g.n + kThreads - 1) / kThreads * kThreads;
        if (tile == 0) tile = kThreads;
        g.mode = kModeSingle;
    } else {
        const int64_t want = (g.n + kMaxTiles - 1) / kMaxTiles;
        tile = (want + kThreads - 1) / kThreads * kThreads;
        if (g.n <= kFusedMax && !split_counting) {
            g.mode = kModeFused;
        } else {
            if (g.n > kFusedMax && tile < MOE_PLAN_TWO_KERNEL_MIN_TILE)
                tile = MOE_PLAN_TWO_KERNEL_MIN_TILE;
            g.mode = kModeTwoKernel;
        }
    }
    g.tile = tile;
    g.sub = tile / kWarps;
    g.T = (int)((g.n + tile - 1) / tile);
    if (g.T == 0) g.T = 1;
    return g;
}

size_t hist_ws_bytes(const PlanGeom &g, int nkeys)
{
    if (g.mode != kModeTwoKernel) return 0;
    size_t b = (size_t)g.T * (size_t)(nkeys + 1) * sizeof(int32_t);
    return (b + 255) / 256 * 256;
}

struct RankOut {
    int32_t *cnt;          // [nkeys]
    int64_t *off;          // [nkeys + 1]
    int64_t *map;          // [n]
    int32_t *src;          // [n]
    int32_t *n_invalid;    // [1] (direct plan) or null
    const int64_t *tok_map;  // group plan: tok_map of the direct plan
    int64_t *grp_tok_map;    // group plan: [rows, K]
    int64_t cap;             // > 0: padded buckets of cap rows, later entries dropped
    int32_t *n_dropped;      // [1] with cap > 0
};

// Key of the 32 entries [c, c+32) of a chunk, one per lane: the slot key, -1
// for an entry that takes no slot, -2 for a lane past the end.  All lanes of
// the warp call it together.
struct DirectKey {
    const int32_t *idx;
    int E;
    static constexpr bool kCountsInvalid = true;
    __device__ __forceinline__ int chunk_key(int64_t i, bool in_range) const
    {
        if (!in_range) return -2;
        int e = __ldg(idx + i);
        return (e >= 0 && e < E) ? e : -1;
    }
    __device__ __forceinline__ void emit_chunk(int64_t, bool, int64_t, int, const RankOut &) const
    {
    }

    static constexpr bool kMergesWarpCounts = true;

    // One entry of the all-entries pass: before this tile -> s_bef, else
    // s_aft; inside this tile also the count of its warp sub-tile (wc row).
    __device__ __forceinline__ void add(int e, bool before, int32_t *wc, int32_t *s_aft,
                                        int32_t *s_bef, int &invalid) const
    {
        if (e >= 0 && e < E) {
            atomicAdd(before ? &s_bef[e] : &s_aft[e], 1);
            if (wc) atomicAdd(&wc[e], 1);
        } else {
            ++invalid;
        }
    }

    // The first kPre 16-byte groups of this thread in the all-entries pass,
    // loaded at kernel start so that their latency overlaps the set-up.
    static constexpr int kPre = 8;
    struct Pre {
        int4 v[kPre];
    };
    __device__ __forceinline__ void prefetch(int64_t n, Pre &pre) const
    {
        if ((reinterpret_cast<uintptr_t>(idx) & 15u) != 0) return;
        const int4 *p = reinterpret_cast<const int4 *>(idx);
        const int64_t n4 = n / 4;
#pragma unroll
        for (int u = 0; u < kPre; ++u) {
            const int64_t q = threadIdx.x + (int64_t)u * kThreads;
            if (q < n4) pre.v[u] = __ldg(p + q);
        }
    }

    // Counts all n entries: those before `tile_begin` (a multiple of 1024)
    // into s_bef, the others into s_aft, and those of this tile [tile_begin,
    // tile_end) also into their warp sub-tile's row of s_wc.  Returns this
    // thread's invalid entries.  Each thread takes 16-byte groups of 4
    // entries (always inside one sub-tile): first the kPre prefetched ones,
    // then the rest four in flight.
    __device__ __forceinline__ int count_all(int64_t n, int64_t tile_begin, int64_t tile_end,
                                             int64_t sub, int wstride, int32_t *s_aft,
                                             int32_t *s_bef, int32_t *s_wc, const Pre &pre) const
    {
        auto wc_row = [&](int64_t j) -> int32_t * {
            return (j >= tile_begin && j < tile_end) ? s_wc + ((j - tile_begin) / sub) * wstride
                                                     : nullptr;
        };
        int invalid = 0;
        int64_t done = 0;
        if ((reinterpret_cast<uintptr_t>(idx) & 15u) == 0) {
            const int4 *p = reinterpret_cast<const int4 *>(idx);
            const int64_t n4 = n / 4;
#pragma unroll
            for (int u = 0; u < kPre; ++u) {
                const int64_t q = threadIdx.x + (int64_t)u * kThreads;
                if (q < n4) {
                    const bool before = q * 4 < tile_begin;
                    int32_t *wc = wc_row(q * 4);
                    add(pre.v[u].x, before, wc, s_aft, s_bef, invalid);
                    add(pre.v[u].y, before, wc, s_aft, s_bef, invalid);
                    add(pre.v[u].z, before, wc, s_aft, s_bef, invalid);
                    add(pre.v[u].w, before, wc, s_aft, s_bef, invalid);
                }
            }
            for (int64_t q0 = threadIdx.x + (int64_t)kPre * kThreads; q0 < n4;
                 q0 += 4 * kThreads) {
                int4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (q0 + u * kThreads < n4) v[u] = __ldg(p + q0 + u * kThreads);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t q = q0 + u * kThreads;
                    if (q < n4) {
                        const bool before = q * 4 < tile_begin;
                        int32_t *wc = wc_row(q * 4);
                        add(v[u].x, before, wc, s_aft, s_bef, invalid);
                        add(v[u].y, before, wc, s_aft, s_bef, invalid);
                        add(v[u].z, before, wc, s_aft, s_bef, invalid);
                        add(v[u].w, before, wc, s_aft, s_bef, invalid);
                    }
                }
            }
            done = n4 * 4;
        }
        for (int64_t j = done + threadIdx.x; j < n; j += kThreads)
            add(__ldg(idx + j), j < tile_begin, wc_row(j), s_aft, s_bef, invalid);
        return invalid;
    }
};

struct GroupKey {
    const int32_t *idx;
    int E, K, gs;
    static constexpr bool kCountsInvalid = false;
    __device__ __forceinline__ int group(int64_t i) const
    {
        int e = __ldg(idx + i);
        return (e >= 0 && e < E) ? e / gs : -1;
    }
    __device__ __forceinline__ int chunk_key(int64_t i, bool in_range) const
    {
        return chunk_key_g(i, in_range, in_range ? group(i) : -1);
    }
    // chunk_key with the entry's group already loaded (g = -1 when i is past
    // the end or its expert is invalid)
    __device__ __forceinline__ int chunk_key_g(int64_t i, bool in_range, int g) const
    {
        const int lane = threadIdx.x & 31;
        if ((32 % K) == 0) {
            // Chunks start at multiples of 32, so a token's K entries sit in
            // one chunk: an entry represents its group unless an earlier lane
            // of the same token holds the same group (K - 1 shuffles)
            const int base = lane - lane % K;
            bool rep = g >= 0;
            for (int kk = 0; kk < K - 1; ++kk) {
                const int v = __shfl_sync(0xffffffffu, g, base + kk);
                if (kk < lane - base && v == g) rep = false;
            }
            if (!in_range) return -2;
            return rep ? g : -1;
        }
        if (!in_range) return -2;
        if (g < 0) return -1;
        const int64_t s0 = i - i % K;
        for (int64_t j = s0; j < i; ++j)
            if (group(j) == g) return -1;
        return g;
    }
    // Each representative row lists its token's experts that fall in its
    // group (the direct plan's row, else -1).  Called by all lanes of a chunk
    // together; `row` >= 0 marks a representative.  When tokens sit whole in
    // a chunk (32 % K == 0) the lanes of a token fill the rows together:
    // lane j writes column j of every representative row of its token, from
    // its own entry.  Otherwise each representative walks its token.
    __device__ __forceinline__ void emit_chunk(int64_t i, bool in_range, int64_t row, int g,
                                               const RankOut &o) const
    {
        if ((32 % K) == 0) {
            const int lane = threadIdx.x & 31;
            const int base = lane - lane % K;
            const int gj = in_range ? group(i) : -1;
            const int64_t tm = in_range ? o.tok_map[i] : -1;
            for (int kk = 0; kk < K; ++kk) {
                const int64_t rq = __shfl_sync(0xffffffffu, row, base + kk);
                const int gq = __shfl_sync(0xffffffffu, g, base + kk);
                if (rq >= 0 && in_range)
                    o.grp_tok_map[rq * K + (lane - base)] = (gj == gq) ? tm : -1;
            }
            return;
        }
        if (row < 0 || !in_range) return;
        const int64_t s0 = i - i % K;
        for (int kk = 0; kk < K; ++kk)
            o.grp_tok_map[row * K + kk] = (group(s0 + kk) == g) ? o.tok_map[s0 + kk] : -1;
    }

    static constexpr bool kMergesWarpCounts = false;

    struct Pre {};
    __device__ __forceinline__ void prefetch(int64_t, Pre &) const {}

    // Counts the representatives among all n entries (warp chunks of 32, so
    // that the ballot dedup sees whole tokens); chunks lie wholly before or
    // wholly after `tile_begin`, a multiple of 1024.  Per-warp counts of the
    // own tile come from step (a) instead.
    __device__ __forceinline__ int count_all(int64_t n, int64_t tile_begin, int64_t, int64_t,
                                             int, int32_t *s_tot, int32_t *s_bef, int32_t *,
                                             const Pre &) const
    {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const int G = E / gs;
        if (G <= 8) {
            // one token per thread: its representatives are found by comparing
            // its K groups, and counted in 8-bit fields of two registers (a
            // thread sees at most n / K / kThreads < 256 tokens here), then
            // summed over the warp and added once per group
            uint64_t pb = 0, pa = 0;
            const int64_t ntok = n / K;
            for (int64_t t = threadIdx.x; t < ntok; t += kThreads) {
                int gv[32];
#pragma unroll
                for (int kk = 0; kk < 32; ++kk)
                    if (kk < K) gv[kk] = group(t * K + kk);
#pragma unroll
                for (int kk = 0; kk < 32; ++kk) {
                    if (kk >= K) break;
                    bool rep = gv[kk] >= 0;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        if (jj < kk && gv[jj] == gv[kk]) rep = false;
                    if (rep) {
                        const uint64_t one = 1ull << (8 * gv[kk]);
                        if (t * K + kk < tile_begin)
                            pb += one;
                        else
                            pa += one;
                    }
                }
            }
            for (int gg = 0; gg < G; ++gg) {
                int b = (int)((pb >> (8 * gg)) & 0xff), f = (int)((pa >> (8 * gg)) & 0xff);
                for (int o = 16; o; o >>= 1) {
                    b += __shfl_xor_sync(0xffffffffu, b, o);
                    f += __shfl_xor_sync(0xffffffffu, f, o);
                }
                if (lane == 0) {
                    if (b) atomicAdd(&s_bef[gg], b);
                    if (f) atomicAdd(&s_tot[gg], f);
                }
            }
            return 0;
        }
        // the groups of kPre chunks are loaded before any of them is keyed,
        // so the loads of a warp overlap instead of queueing one by one
        constexpr int kPre = 8;
        const int64_t cstride = (int64_t)kWarps * 32;
        if (G <= 32) {
            // lane g tallies group g in registers (one ballot per group and
            // chunk), then adds once: no contended shared-memory atomics
            int bef = 0, aft = 0;
            for (int64_t c0 = (int64_t)warp * 32; c0 < n; c0 += cstride * kPre) {
                int gv[kPre];
#pragma unroll
                for (int q = 0; q < kPre; ++q) {
                    const int64_t i = c0 + q * cstride + lane;
                    gv[q] = i < n ? group(i) : -1;
                }
#pragma unroll
                for (int q = 0; q < kPre; ++q) {
                    const int64_t c = c0 + q * cstride;
                    if (c >= n) break;  // the same for every lane
                    const int64_t i = c + lane;
                    const int k = chunk_key_g(i, i < n, gv[q]);
                    const bool before = c < tile_begin;
                    for (int gg = 0; gg < G; ++gg) {
                        const int cnt = __popc(__ballot_sync(0xffffffffu, k == gg));
                        if (lane == gg) {
                            if (before)
                                bef += cnt;
                            else
                                aft += cnt;
                        }
                    }
                }
            }
            if (lane < G) {
                if (bef) atomicAdd(&s_bef[lane], bef);
                if (aft) atomicAdd(&s_tot[lane], aft);
            }
            return 0;
        }
        for (int64_t c0 = (int64_t)warp * 32; c0 < n; c0 += cstride * kPre) {
            int gv[kPre];
#pragma unroll
            for (int q = 0; q < kPre; ++q) {
                const int64_t i = c0 + q * cstride + lane;
                gv[q] = i < n ? group(i) : -1;
            }
#pragma unroll
            for (int q = 0; q < kPre; ++q) {
                const int64_t c = c0 + q * cstride;
                if (c >= n) break;  // the same for every lane
                const int64_t i = c + lane;
                const int k = chunk_key_g(i, i < n, gv[q]);
                const unsigned peers = __match_any_sync(0xffffffffu, k);
                if (k >= 0 && lane == __ffs(peers) - 1)
                    atomicAdd(c < tile_begin ? &s_bef[k] : &s_tot[k], __popc(peers));
            }
        }
        return 0;
    }
};

// Kernel 1: histogram of tile t into ws[t * (nkeys + 1) + key]; invalid
// entries into ws[t * (nkeys + 1) + nkeys].
template <typename Key>
__global__ void __launch_bounds__(kThreads, 1) plan_hist_kernel(Key key, int nkeys, PlanGeom g,
                                                             int32_t *__restrict__ ws)
{
    extern __shared__ int32_t s_hist[];  // [nkeys + 1]
    griddep_launch_dependents();
    for (int e = threadIdx.x; e <= nkeys; e += kThreads) s_hist[e] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x;
    const int64_t wbegin = (int64_t)t * g.tile + (int64_t)warp * g.sub;
    const int64_t wend = min(wbegin + g.sub, g.n);
    int invalid = 0;
    for (int64_t c = wbegin; c < wend; c += 32) {
        const int64_t i = c + lane;
        int k = key.chunk_key(i, i < wend);
        if (k == -1) ++invalid;
        unsigned peers = __match_any_sync(0xffffffffu, k);
        if (k >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[k], __popc(peers));
    }
    if (Key::kCountsInvalid) {
        for (int o = 16; o; o >>= 1) invalid += __shfl_xor_sync(0xffffffffu, invalid, o);
        if (lane == 0 && invalid) atomicAdd(&s_hist[nkeys], invalid);
    }
    __syncthreads();
    int32_t *row = ws + (int64_t)t * (nkeys + 1);
    for (int e = threadIdx.x; e <= nkeys; e += kThreads) row[e] = s_hist[e];
}

// Exclusive scan of v over the block; returns this thread's exclusive
// prefix and sets `total`.
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t *s_warp, int64_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t x = v;
    for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t w = s_warp[lane];
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    total = s_warp[kWarps - 1];
    const int64_t before = warp ? s_warp[warp - 1] : 0;
    return before + x - v;
}

// Kernel 2: stable ranks of one tile (steps (a)-(e) of the file comment).
template <typename Key>
__global__ void __launch_bounds__(kThreads, 1) plan_rank_kernel(Key key, int nkeys, PlanGeom g,
                                                             const int32_t *__restrict__ ws,
                                                             RankOut o)
{
    extern __shared__ int32_t smem[];
    // per-warp counts, one row of nkeys | 1 ints per warp
    const int wstride = nkeys | 1;
    int32_t *s_wc = smem;                               // [kWarps][wstride]
    int64_t *s_base = reinterpret_cast<int64_t *>(s_wc + ((kWarps * wstride + 1) & ~1));  // [nkeys]
    int32_t *s_tot = reinterpret_cast<int32_t *>(s_base + nkeys);                     // [nkeys]
    int32_t *s_bef = s_tot + nkeys;                                                   // [nkeys]
    __shared__ int64_t s_scan[kWarps];
    __shared__ int32_t s_inval;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x;
    const bool single = (g.mode == kModeSingle);

    // Unless kernel 1 ran first, nothing of this plan ran before: wait for
    // whatever wrote topk_idx, and only then let the next kernel launch, so
    // that everything before this plan is complete when the next kernel
    // starts (the dispatch of moe_plan_dispatch loads x before its own wait).
    // In two-kernel mode kernel 1 was launched without the attribute, so it
    // (and this kernel) began only after earlier stream work finished:
    // topk_idx may be read before the wait, and the dependents may launch at
    // once.
    if (g.mode != kModeTwoKernel) griddep_wait();
    griddep_launch_dependents();

    const int64_t wbegin = (int64_t)t * g.tile + (int64_t)warp * g.sub;
    const int64_t wend = min(wbegin + g.sub, g.n);
    int32_t *my_wc = s_wc + warp * wstride;

    // first loads before anything else, so that their latency overlaps the
    // clearing of shared memory: the keys of the warp's first chunk ((a) and
    // (e) reuse them) and, in one-launch mode, the first groups of the
    // all-entries pass
    const int k_first = key.chunk_key(wbegin + lane, wbegin + lane < wend);
    typename Key::Pre pre;
    if (g.mode == kModeFused) key.prefetch(g.n, pre);

    for (int i = threadIdx.x; i < kWarps * wstride; i += kThreads) s_wc[i] = 0;
    for (int i = threadIdx.x; i < nkeys; i += kThreads) s_tot[i] = s_bef[i] = 0;
    if (threadIdx.x == 0) s_inval = 0;
    __syncthreads();
    // in the one-launch mode the direct plan takes the per-warp counts of
    // its own tile from the all-entries pass in (b)
    const bool merged = g.mode == kModeFused && Key::kMergesWarpCounts;

    // (a) per-warp counts
    int invalid = 0;
    if (!merged) {
        for (int64_t c = wbegin; c < wend; c += 32) {
            const int64_t i = c + lane;
            const int k = (c == wbegin) ? k_first : key.chunk_key(i, i < wend);
            if (k == -1) ++invalid;
            const unsigned peers = __match_any_sync(0xffffffffu, k);
            if (k >= 0 && lane == __ffs(peers) - 1) my_wc[k] += __popc(peers);
            __syncwarp();
        }
    }
    if (Key::kCountsInvalid && single) {
        for (int sh = 16; sh; sh >>= 1) invalid += __shfl_xor_sync(0xffffffffu, invalid, sh);
        if (lane == 0 && invalid) atomicAdd(&s_inval, invalid);
    }

    // (b) global counts and counts of earlier tiles
    if (single) {
        // totals; the same walk leaves each key's exclusive prefixes over
        // the warps in place of its counts, which is step (d) (32 tokens at
        // E=1024, per plan back to back in a graph: 5.5 -> 5.1 us)
        __syncthreads();
        for (int e = threadIdx.x; e < nkeys; e += kThreads) {
            int32_t run = 0;
#pragma unroll 8
            for (int w = 0; w < kWarps; ++w) {
                const int32_t c = s_wc[w * wstride + e];
                s_wc[w * wstride + e] = run;
                run += c;
            }
            s_tot[e] = run;
        }
    } else if (g.mode == kModeFused) {
        // s_tot collects the entries from this tile on, s_bef those before
        const int64_t tile_begin = (int64_t)t * g.tile;
        int inv = key.count_all(g.n, tile_begin, min(tile_begin + g.tile, g.n), g.sub, wstride,
                                s_tot, s_bef, s_wc, pre);
        if (Key::kCountsInvalid && t == 0) {
            for (int sh = 16; sh; sh >>= 1) inv += __shfl_xor_sync(0xffffffffu, inv, sh);
            if (lane == 0 && inv) atomicAdd(&s_inval, inv);
        }
        __syncthreads();
        for (int k = threadIdx.x; k < nkeys; k += kThreads) s_tot[k] += s_bef[k];
    } else {
        griddep_wait();  // tile histograms of kernel 1 are complete and visible
        const int stride = nkeys + 1;
        const int64_t nws = (int64_t)g.T * stride;
#pragma unroll 4
        for (int64_t j = threadIdx.x; j < nws; j += kThreads) {
            const int tt = (int)(j / stride);
            const int e = (int)(j - (int64_t)tt * stride);
            const int32_t h = ws[j];
            if (e < nkeys) {
                atomicAdd(&s_tot[e], h);
                if (tt < t) atomicAdd(&s_bef[e], h);
            } else if (Key::kCountsInvalid && t == 0) {
                atomicAdd(&s_inval, h);
            }
        }
    }
    __syncthreads();

    // (c) exclusive scan over keys (nkeys <= kThreads: one key per thread).
    // s_base holds the first rank of this tile in each key; with a capacity
    // the bucket of key e starts at e * cap instead of at the scan.
    const int e = threadIdx.x;
    const int64_t tot = (e < nkeys) ? s_tot[e] : 0;
    int64_t total;
    const int64_t offe = block_exclusive_scan(tot, s_scan, total);
    if (e < nkeys) {
        s_base[e] = (o.cap > 0 ? 0 : offe) + s_bef[e];
        if (t == 0) {
            o.cnt[e] = (int32_t)(o.cap > 0 ? min(tot, o.cap) : tot);
            o.off[e] = o.cap > 0 ? (int64_t)e * o.cap : offe;
        }
    }
    if (t == 0 && threadIdx.x == 0) {
        o.off[nkeys] = o.cap > 0 ? (int64_t)nkeys * o.cap : total;
        if (o.n_invalid) *o.n_invalid = s_inval;
    }
    if (o.cap > 0 && t == 0) {
        // entries that do not fit: sum over keys of max(0, count - cap)
        __syncthreads();  // every thread has read the first scan's s_scan
        int64_t dropped_total;
        (void)block_exclusive_scan(e < nkeys ? max((int64_t)0, tot - o.cap) : 0, s_scan,
                                   dropped_total);
        if (threadIdx.x == 0) *o.n_dropped = (int32_t)dropped_total;
    }

    // (d) exclusive scan over the 32 warps, per key, relative to the tile
    // base: thread e walks key e's column (16 counts loaded before any is
    // rewritten).  Per plan back to back in a graph, against one warp per
    // key scanning the column with shuffles: 7.17 -> 7.0 us at S=4096 K=8
    // E=64, 10.57 -> 9.87 us for the Zipf batch (S=8192, E=256), 11.53 ->
    // 8.93 us at E=1024.
    if (!single && e < nkeys) {
        int32_t run = 0;
#pragma unroll
        for (int w0 = 0; w0 < kWarps; w0 += 16) {
            int32_t c[16];
#pragma unroll
            for (int w = 0; w < 16; ++w) c[w] = s_wc[(w0 + w) * wstride + e];
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                s_wc[(w0 + w) * wstride + e] = run;
                run += c[w];
            }
        }
    }
    __syncthreads();

    // (e) assign ranks
    for (int64_t c = wbegin; c < wend; c += 32) {
        const int64_t i = c + lane;
        const int k = (c == wbegin) ? k_first : key.chunk_key(i, i < wend);
        const unsigned peers = __match_any_sync(0xffffffffu, k);
        int64_t row = -1;
        if (k >= 0) {
            row = s_base[k] + my_wc[k] + __popc(peers & lanemask_lt());
            if (o.cap > 0) row = row < o.cap ? (int64_t)k * o.cap + row : -1;
        }
        __syncwarp();
        if (k >= 0 && lane == __ffs(peers) - 1) my_wc[k] += __popc(peers);
        __syncwarp();
        if (i < wend) {
            o.map[i] = row;
            if (row >= 0) o.src[row] = (int32_t)i;
        }
        key.emit_chunk(i, i < wend, row, k, o);
    }
}

template <typename Key>
int run_plan(Key key, int nkeys, const PlanGeom &g, const RankOut &o, void *ws,
             size_t ws_bytes, cudaStream_t stream)
{
    const size_t need = hist_ws_bytes(g, nkeys);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) return MOE_EINVAL;
    if (need > 0 && (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_EALIGN;
    if (g.mode == kModeTwoKernel) {
        const size_t smem1 = (size_t)(nkeys + 1) * sizeof(int32_t);
        static KernelCache hcache;  // one per Key instantiation
        if (cudaError_t e = prepare_kernel(plan_hist_kernel<Key>, smem1, kThreads, hcache, nullptr)) {
            set_cuda_error(e);
            return MOE_ECUDA;
        }
        // A plain launch, not a programmatic dependent one: it starts only
        // after everything before it on the stream has finished, including
        // the rank kernel of an earlier plan that may still be reading the
        // same workspace.  moe_plan_static_scratch depends on this: all its
        // calls share one array, and a launch_pdl here would let this kernel
        // overwrite the histograms of the previous call while its rank
        // kernel (which allows dependents at entry) still reads them.
        plan_hist_kernel<Key><<<g.T, kThreads, smem1, stream>>>(key, nkeys, g,
                                                                 static_cast<int32_t *>(ws));
        if (int rc = check_launch()) return rc;
    }
    const size_t smem2 = (size_t)((kWarps * (nkeys | 1) + 1) & ~1) * sizeof(int32_t) +
                         (size_t)nkeys * (sizeof(int64_t) + 2 * sizeof(int32_t));
    static KernelCache cache;  // one per Key instantiation
    cudaError_t err = prepare_kernel(plan_rank_kernel<Key>, smem2, kThreads, cache, nullptr);
    if (err == cudaSuccess)
        err = launch_pdl(plan_rank_kernel<Key>, dim3(g.T), dim3(kThreads), smem2, stream, key,
                         nkeys, g, static_cast<const int32_t *>(ws), o);
    if (err != cudaSuccess) {
        set_cuda_error(err);
        return MOE_ECUDA;
    }
    return check_launch();
}

int check_plan_args(int64_t S, int K, int E)
{
    if (S < 0 || K < 1 || K > 32 || E < 1 || E > 1024) return MOE_EINVAL;
    if (S * (int64_t)K >= ((int64_t)1 << 31)) return MOE_EINVAL;
    return MOE_OK;
}

} // namespace
} // namespace moe

using namespace moe;

MOE_EXPORT size_t moe_plan_workspace_size(int64_t S, int K, int E)
{
    if (check_plan_args(S, K, E)) return 0;
    return hist_ws_bytes(plan_geom(S, K), E);
}

MOE_EXPORT int moe_plan(const int32_t *topk_idx, int64_t S, int K, int E, int32_t *cnt,
                        int64_t *off, int32_t *packed_src, int64_t *tok_map,
                        int32_t *n_invalid, void *workspace, size_t workspace_bytes,
                        moe_stream_t stream)
{
    MOE_TRACE("moe_plan");
    if (int rc = check_plan_args(S, K, E)) return rc;
    if (!cnt || !off || !n_invalid) return MOE_EINVAL;
    if (S > 0 && (!topk_idx || !packed_src || !tok_map)) return MOE_EINVAL;
    const PlanGeom g = plan_geom(S, K);
    const DirectKey key{topk_idx, E};
    const RankOut o{cnt, off, tok_map, packed_src, n_invalid, nullptr, nullptr, 0, nullptr};
    return run_plan(key, E, g, o, workspace, workspace_bytes, (cudaStream_t)stream);
}

MOE_EXPORT int moe_plan_capacity(const int32_t *topk_idx, int64_t S, int K, int E,
                                 int64_t capacity, int32_t *cnt, int64_t *off,
                                 int32_t *packed_src, int64_t *tok_map, int32_t *n_invalid,
                                 int32_t *n_dropped, void *workspace, size_t workspace_bytes,
                                 moe_stream_t stream)
{
    MOE_TRACE("moe_plan_capacity");
    if (int rc = check_plan_args(S, K, E)) return rc;
    if (capacity < 1 || capacity * (int64_t)E >= ((int64_t)1 << 31)) return MOE_EINVAL;
    if (!cnt || !off || !n_invalid || !n_dropped) return MOE_EINVAL;
    if (S > 0 && (!topk_idx || !packed_src || !tok_map)) return MOE_EINVAL;
    const PlanGeom g = plan_geom(S, K);
    const DirectKey key{topk_idx, E};
    const RankOut o{cnt, off, tok_map, packed_src, n_invalid, nullptr, nullptr, capacity,
                    n_dropped};
    return run_plan(key, E, g, o, workspace, workspace_bytes, (cudaStream_t)stream);
}

MOE_EXPORT size_t moe_group_plan_workspace_size(int64_t S, int K, int E, int group_size)
{
    if (check_plan_args(S, K, E) || group_size < 1 || E % group_size) return 0;
    return hist_ws_bytes(plan_geom(S, K, true), E / group_size);
}

MOE_EXPORT int moe_group_plan(const int32_t *topk_idx, const int64_t *tok_map, int64_t S, int K,
                              int E, int group_size, int32_t *gcnt, int64_t *goff,
                              int64_t *gtok_map, int32_t *grp_src, int64_t *grp_tok_map,
                              void *workspace, size_t workspace_bytes, moe_stream_t stream)
{
    MOE_TRACE("moe_group_plan");
    if (int rc = check_plan_args(S, K, E)) return rc;
    if (group_size < 1 || E % group_size) return MOE_EINVAL;
    if (!gcnt || !goff) return MOE_EINVAL;
    if (S > 0 && (!topk_idx || !tok_map || !gtok_map || !grp_src || !grp_tok_map))
        return MOE_EINVAL;
    PlanGeom g = plan_geom(S, K, true);
    // without the workspace for the tile histograms, plans of up to kFusedMax
    // entries run in one launch whose CTAs count all entries themselves
    if (g.n <= kFusedMax && (workspace == nullptr || workspace_bytes < hist_ws_bytes(g, E / group_size)))
        g = plan_geom(S, K, false);
    const GroupKey key{topk_idx, E, K, group_size};
    const RankOut o{gcnt, goff, gtok_map, grp_src, nullptr, tok_map, grp_tok_map, 0, nullptr};
    return run_plan(key, E / group_size, g, o, workspace, workspace_bytes, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------
// moe_plan_static_scratch: moe_plan without a caller-supplied workspace.
//
// Some callers cannot hand this library a device workspace: a C or C++ host
// that links only this library and owns no device allocator, or a process
// whose device memory belongs to a pool that forbids further cudaMalloc calls
// (a cudaMalloc may synchronise the device and fragment a packed heap).  For
// them the tile histograms live in the file-scope array below, which is part
// of the library image: every GPU that loads the library holds it until the
// process exits, and this entry point allocates nothing.
//
// The array is shared by every call.  Each call overwrites every histogram
// entry it later reads, so leftover contents from an earlier call need no
// clearing; but two calls whose plans overlap on the GPU (for example on two
// streams) race on it and must not be issued.
// ---------------------------------------------------------------------------

#include <mutex>

// Stated maximum: 256 KiB, enough for the tile histograms of every plan with
// E <= 511 experts (at most 128 tiles); plans of up to 131,072 entries use no
// scratch at all.  Larger plans are rejected with MOE_EINVAL.
#define MOE_STATIC_PLAN_SCRATCH_BYTES (256u * 1024u)

static __device__ __align__(256) unsigned char g_plan_static_scratch[MOE_STATIC_PLAN_SCRATCH_BYTES];

namespace moe {
namespace {

constexpr size_t kStaticPlanScratchBytes = MOE_STATIC_PLAN_SCRATCH_BYTES;
constexpr int kMaxStaticDevices = 64;
std::mutex g_static_scratch_mu;
void *g_static_scratch_ptr[kMaxStaticDevices];  // device address per device, once known

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in; the real address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
// The address stays valid for the life of the device's primary context; a
// cudaDeviceReset after the first call would leave a stale address behind,
// so resetting a device this library has planned on is not supported.
int static_scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return MOE_ECUDA;
    }
    if (dev < 0 || dev >= kMaxStaticDevices) return MOE_EINVAL;
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    if (g_static_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_plan_static_scratch);
        if (e != cudaSuccess || p == nullptr) {
            set_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
            return MOE_ECUDA;
        }
        g_static_scratch_ptr[dev] = p;
    }
    *out = g_static_scratch_ptr[dev];
    return MOE_OK;
}

} // namespace
} // namespace moe

MOE_EXPORT int moe_plan_static_scratch(const int32_t *topk_idx, int64_t S, int K, int E,
                                       int32_t *cnt, int64_t *off, int32_t *packed_src,
                                       int64_t *tok_map, int32_t *n_invalid,
                                       moe_stream_t stream)
{
    MOE_TRACE("moe_plan_static_scratch");
    if (int rc = check_plan_args(S, K, E)) return rc;
    if (!cnt || !off || !n_invalid) return MOE_EINVAL;
    if (S > 0 && (!topk_idx || !packed_src || !tok_map)) return MOE_EINVAL;
    const PlanGeom g = plan_geom(S, K);
    const size_t need = hist_ws_bytes(g, E);
    if (need > kStaticPlanScratchBytes) return MOE_EINVAL;  // plan too large for the array
    void *ws = nullptr;
    if (int rc = static_scratch_address(&ws)) return rc;
    const DirectKey key{topk_idx, E};
    const RankOut o{cnt, off, tok_map, packed_src, n_invalid, nullptr, nullptr, 0, nullptr};
    return run_plan(key, E, g, o, ws, kStaticPlanScratchBytes, (cudaStream_t)stream);
}
