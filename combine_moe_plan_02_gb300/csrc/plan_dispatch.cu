// Plan and dispatch in one launch.
//
// Sources: ROCm/mori "EPv2 internode dispatch/combine over CCO/GDA": the
// page keeps two kernel families, a throughput one and a low-latency one,
// and picks per call by token count (its automatic crossover sits at 512
// tokens); ROCm/mori "Draft: cco + flydsl dispatch/combine #448", StdMoE note
// (the plan outputs: per-expert counts, packed_src, the i64 slot map with -1)
// and PR description (each token row is written once per destination).
//
// GB300 design: at small batch sizes a step is a chain of short kernels
// whose cost is launch and tail latency, not bytes, so plan and dispatch are
// fused.  Below the crossover the flat entry list holds at most
// kFusedMaxEntries entries, few enough that every CTA of the launch ranks all
// of them itself in shared memory -- the same stable (token, k) ranks as
// moe_plan: per-warp counts by __match_any_sync, then thread e walks expert
// e's warp counts (its total, and the exclusive prefix over warps left in
// place), an exclusive scan over experts, then rank = expert offset + warp
// base + running count + popc(peers below the lane).  CTA 0 also writes the
// plan outputs.  Then every warp of the grid copies 512-byte segments of
// token rows (32 lanes x 16 bytes) to the token's destinations, read from
// the CTA's own copy of the map.  No CTA waits for another CTA.
//
// Larger batches (up to kTiledMaxEntries entries and MOE_PD_TILED_MAX_BYTES
// of rows) take plan_dispatch_tiles_kernel, whose CTAs own token ranges
// instead (see there): a kernel boundary between a separate plan and dispatch
// costs several microseconds on this part, more than the redundant counting
// does, until the copy is long enough for the balanced dispatch to win.

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;  // one expert per thread in the scan: E <= 1024
constexpr int kWarps = kThreads / 32;
constexpr int kSeg = 512;       // bytes of a row segment copied by one warp
#ifndef MOE_PLAN_DISPATCH_FUSED_MAX
#define MOE_PLAN_DISPATCH_FUSED_MAX 1024
#endif
constexpr int64_t kFusedMaxEntries = MOE_PLAN_DISPATCH_FUSED_MAX;
// CTAs of the smallest of 256, 512 or 1024 threads that gives every expert
// a thread: the per-warp count table then has as many rows as the CTA has
// warps.  fp8 rows, H=6144 E=256 K=8,
// per call back to back in a graph: 6.54 -> 4.57 us at 4..16 tokens with 256
// threads instead of 1024, 8.60 -> 7.58 us at 128, 12.93 us at 1024 either
// way; two or four such CTAs per SM made 128 tokens slower (9.2 us).  At
// E=512, 512 threads: 4.5 against 6.3 us for 1024.  At E=64, 128 threads
// gained 0.2 us at 4..16 tokens and lost 2 us at 128 (fewer warps rank and
// copy), hence the floor of 256.

__device__ uint32_t g_pd_error;  // kErrDispatchIndex

struct PDArgs {
    const int32_t *idx;   // [S, K]
    int64_t S;
    int K, E;
    int64_t n;            // S * K
    const uint8_t *x;     // [S, row_bytes]
    int64_t row_bytes;
    const uint8_t *xs;    // [S, scale_bytes] or null
    int64_t scale_bytes;
    int64_t segs, ssegs;  // 512-byte segments of a row / of a scale row
    int32_t *cnt;         // [E]
    int64_t *off;         // [E + 1]
    int32_t *src;         // [n]
    int64_t *map;         // [n]
    int32_t *n_invalid;   // [1]
    uint8_t *px;          // [packed_rows, row_bytes]
    uint8_t *ps;          // [packed_rows, scale_bytes] or null
    int64_t packed_rows;
};

// Exclusive scan of v over a block of kW warps; sets `total`.
template <int kW = kWarps>
__device__ __forceinline__ int32_t block_scan(int32_t v, int32_t *s_warp, int32_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t x = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < kW ? s_warp[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kW) s_warp[lane] = w;
    }
    __syncthreads();
    total = s_warp[kW - 1];
    return (warp ? s_warp[warp - 1] : 0) + x - v;
}

// The same scan with one block barrier: every warp sums the kW warp totals
// itself instead of warp 0 scanning them for the others.
template <int kW>
__device__ __forceinline__ int32_t block_scan_1(int32_t v, int32_t *s_warp, int32_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t x = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    int32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
        const int32_t t = s_warp[w];
        before += w < warp ? t : 0;
        all += t;
    }
    total = all;
    return before + x - v;
}

// Expert of entry i, -1 if it takes no slot, -2 past the warp's range.
__device__ __forceinline__ int entry_key(const PDArgs &a, int64_t i, bool in_range)
{
    if (!in_range) return -2;
    const int e = __ldg(a.idx + i);
    return (e >= 0 && e < a.E) ? e : -1;
}

// kT threads per CTA, at least E (one expert per thread in the totals).
template <int kT>
__global__ void __launch_bounds__(kT, 1) plan_dispatch_kernel(PDArgs a)
{
    constexpr int kW = kT / 32;
    extern __shared__ int32_t smem[];
    const int wstride = a.E | 1;                 // odd: the column walks hit 32 banks
    int32_t *s_wc = smem;                        // [kW][wstride] per-warp counts
    int32_t *s_off = s_wc + kW * wstride;        // [E] bucket offsets
    int32_t *s_row = s_off + a.E;                // [n] packed row of each entry
    __shared__ int32_t s_scan[kW];
    __shared__ int32_t s_winv[kW];  // invalid entries counted by each warp

    griddep_wait();  // topk_idx and x come from earlier stream work
    griddep_launch_dependents();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool writer = blockIdx.x == 0;

    // The rows do not depend on the plan: each warp loads the segment of its
    // first (token, segment) unit now, so that the load overlaps the ranking.
    const int64_t per_tok = a.segs + a.ssegs;
    const int64_t units = a.S * per_tok;
    const int64_t u0 = (int64_t)blockIdx.x * kW + warp;
    uint4 v0 = make_uint4(0, 0, 0, 0);
    {
        const int64_t s = u0 / per_tok;
        const int64_t g = u0 - s * per_tok;
        const bool is_row = g < a.segs;
        const int64_t len = is_row ? a.row_bytes : a.scale_bytes;
        const int64_t ob = (is_row ? g : g - a.segs) * kSeg + lane * 16;
        if (u0 < units && ob < len) v0 = ld_stream16((is_row ? a.x : a.xs) + s * len + ob);
    }

    // each warp owns `sub` consecutive entries (a multiple of 32)
    const int64_t sub = (a.n + kT - 1) / kT * 32;
    const int64_t wbegin = (int64_t)warp * sub;
    const int64_t wend = min(wbegin + sub, a.n);
    int32_t *my_wc = s_wc + warp * wstride;
    // each warp clears its own row: no block barrier before the counting
    for (int i = lane; i < wstride; i += 32) my_wc[i] = 0;
    __syncwarp();

    // per-warp counts
    int invalid = 0;
    for (int64_t c = wbegin; c < wend; c += 32) {
        const int64_t i = c + lane;
        const int k = entry_key(a, i, i < wend);
        if (k == -1) ++invalid;
        const unsigned peers = __match_any_sync(0xffffffffu, k);
        if (k >= 0 && lane == __ffs(peers) - 1) my_wc[k] += __popc(peers);
        __syncwarp();
    }
    for (int sh = 16; sh; sh >>= 1) invalid += __shfl_xor_sync(0xffffffffu, invalid, sh);
    if (lane == 0) s_winv[warp] = invalid;
    __syncthreads();

    // totals and bucket offsets (thread e owns expert e); the same walk
    // turns expert e's warp counts into their exclusive prefixes over warps
    const int e = threadIdx.x;
    int32_t tot = 0;
    if (e < a.E) {
#pragma unroll
        for (int w = 0; w < kW; ++w) {
            const int32_t c = s_wc[w * wstride + e];
            s_wc[w * wstride + e] = tot;
            tot += c;
        }
    }
    int32_t total;
    // one barrier when every warp can sum the few warp totals itself (fp8
    // rows, E=256, per call back to back in a graph: 6.66 -> 6.55 us at 128
    // tokens, 3.6 -> 3.5 us at 4; with 32 warps it was slower, 7.7 against
    // 7.0 us at E=1024)
    const int32_t offe = kW <= 8 ? block_scan_1<kW>(tot, s_scan, total)
                                 : block_scan<kW>(tot, s_scan, total);
    if (e < a.E) {
        s_off[e] = offe;
        if (writer) {
            a.cnt[e] = tot;
            a.off[e] = offe;
        }
    }
    if (writer && threadIdx.x == 0) {
        a.off[a.E] = total;
        int32_t inv = 0;
        for (int w = 0; w < kW; ++w) inv += s_winv[w];
        *a.n_invalid = inv;
    }

    __syncthreads();

    // ranks
    for (int64_t c = wbegin; c < wend; c += 32) {
        const int64_t i = c + lane;
        const int k = entry_key(a, i, i < wend);
        const unsigned peers = __match_any_sync(0xffffffffu, k);
        const int below = __popc(peers & lanemask_lt()), total = __popc(peers);
        int32_t row = -1;
        if (k >= 0) row = s_off[k] + my_wc[k] + below;
        __syncwarp();
        if (k >= 0 && below == 0) my_wc[k] += total;
        __syncwarp();
        if (i < wend) {
            s_row[i] = row;
            if (writer) {
                a.map[i] = row;
                if (row >= 0) a.src[row] = (int32_t)i;
            }
        }
    }
    __syncthreads();

    // rows: unit = (token, segment); scale rows follow the row's segments
    for (int64_t u = u0; u < units; u += (int64_t)gridDim.x * kW) {
        const int64_t s = u / per_tok;
        const int64_t g = u - s * per_tok;
        const bool is_row = g < a.segs;
        const int64_t len = is_row ? a.row_bytes : a.scale_bytes;
        const int64_t ob = (is_row ? g : g - a.segs) * kSeg + lane * 16;
        if (ob >= len) continue;
        const uint8_t *srow = (is_row ? a.x : a.xs) + s * len;
        uint8_t *dst = is_row ? a.px : a.ps;
        const uint4 v = (u == u0) ? v0 : ld_stream16(srow + ob);
        for (int k = 0; k < a.K; ++k) {
            const int32_t r = s_row[s * a.K + k];
            if (r < 0) continue;
            if (r < a.packed_rows)
                st16(dst + (int64_t)r * len + ob, v);
            else
                atomicOr(&g_pd_error, kErrDispatchIndex);
        }
    }
}

// ---------------------------------------------------------------------------
// Larger batches: one launch with CTAs that own token ranges.  CTA c owns
// the tpc tokens [c*tpc, (c+1)*tpc) (at most 1024 entries).  It counts all n
// entries itself -- those before its range and the rest, per expert (16-byte
// loads, shared-memory atomics) -- which gives the bucket offsets and the
// counts of earlier tokens; ranks its own entries (one 32-entry chunk per
// warp: __match_any_sync, a scan over warps per expert); writes their map and
// packed_src entries; and then copies its own token rows to their packed
// rows.  The copies of a CTA start as soon as its ranks are known, without a
// kernel boundary between plan and dispatch; no CTA waits for another.
// ---------------------------------------------------------------------------

// packed rows are written with streaming stores: fewer of them are still
// dirty in L2 when the combine that follows starts reading (step 190.2 ->
// 189.3 us at the MoonEP shape)
#ifndef MOE_PD_STORE_CS
#define MOE_PD_STORE_CS 1
#endif
#ifndef MOE_PD_PREFETCH
#define MOE_PD_PREFETCH 1
#endif
#ifndef MOE_PD_PREFETCH_CHUNK
#define MOE_PD_PREFETCH_CHUNK 65536
#endif
constexpr int64_t kPrefetchChunk = MOE_PD_PREFETCH_CHUNK;  // bytes per L2 prefetch request
constexpr int kTilePre = 8;     // 16-byte index groups per thread loaded up front
constexpr int kCopyUnroll = 4;  // row segments per warp with loads in flight

__global__ void __launch_bounds__(kThreads, 1) plan_dispatch_tiles_kernel(PDArgs a, int64_t tpc)
{
    extern __shared__ int32_t smem[];
    const int wstride = a.E | 1;
    int32_t *s_wc = smem;                        // [kWarps][wstride] own-range per-warp counts
    int32_t *s_bef = s_wc + kWarps * wstride;    // [E] entries before the range
    int32_t *s_aft = s_bef + a.E;                // [E] the others
    int32_t *s_base = s_aft + a.E;               // [E] first rank of the range per expert
    int32_t *s_row = s_base + a.E;               // [tpc*K] packed row of each own entry
    __shared__ int32_t s_scan[kWarps];
    __shared__ int32_t s_inval;

    griddep_wait();  // topk_idx and x come from earlier stream work
    griddep_launch_dependents();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool writer = blockIdx.x == 0;
    const int64_t t0 = (int64_t)blockIdx.x * tpc;
    const int64_t t1 = min(t0 + tpc, a.S);
    const int64_t b0 = t0 * a.K, b1 = t1 * a.K;   // own entries [b0, b1)

#if MOE_PD_PREFETCH
    // The range's token rows (one contiguous span of x, and of the scales)
    // are pulled into L2 while the CTA plans, when DRAM has little else to
    // do, so that the copies afterwards mostly hit L2 (plan + dispatch 95.8
    // -> 93.0 us at the MoonEP shape).  An evict-last priority on these lines,
    // set back to normal as each is read, measured slower (93.5-95.6 us).
    {
        const int64_t hi = (t1 - t0) * a.row_bytes, shi = (t1 - t0) * a.scale_bytes;
        const uint8_t *xr = a.x + t0 * a.row_bytes;
        for (int64_t p = (int64_t)threadIdx.x * kPrefetchChunk; p < hi;
             p += (int64_t)kThreads * kPrefetchChunk)
            prefetch_l2_bulk(xr + p, (uint32_t)min(kPrefetchChunk, hi - p));
        if (shi > 0 && threadIdx.x == kThreads - 1)
            prefetch_l2_bulk(a.xs + t0 * a.scale_bytes, (uint32_t)shi);
    }
#endif

    // first loads: this warp's own chunk and the first index groups of the
    // all-entries pass, so that their latency overlaps the set-up
    const int64_t ci = b0 + warp * 32 + lane;
    const int k_own = entry_key(a, ci, ci < b1);
    const bool vec = (reinterpret_cast<uintptr_t>(a.idx) & 15u) == 0;
    const int64_t n4 = vec ? a.n / 4 : 0;
    const int4 *p4 = reinterpret_cast<const int4 *>(a.idx);
    int4 pre[kTilePre];
#pragma unroll
    for (int u = 0; u < kTilePre; ++u) {
        const int64_t q = threadIdx.x + (int64_t)u * kThreads;
        if (q < n4) pre[u] = __ldg(p4 + q);
    }

    for (int i = threadIdx.x; i < kWarps * wstride; i += kThreads) s_wc[i] = 0;
    for (int i = threadIdx.x; i < a.E; i += kThreads) s_bef[i] = s_aft[i] = 0;
    if (threadIdx.x == 0) s_inval = 0;
    __syncthreads();

    // own-range per-warp counts (one chunk per warp)
    {
        const unsigned peers = __match_any_sync(0xffffffffu, k_own);
        if (k_own >= 0 && lane == __ffs(peers) - 1) s_wc[warp * wstride + k_own] = __popc(peers);
    }

    // all entries: before the range -> s_bef, the rest -> s_aft
    int invalid = 0;
    auto add = [&](int e, int64_t i) {
        if (e >= 0 && e < a.E)
            atomicAdd(i < b0 ? &s_bef[e] : &s_aft[e], 1);
        else
            ++invalid;
    };
#pragma unroll
    for (int u = 0; u < kTilePre; ++u) {
        const int64_t q = threadIdx.x + (int64_t)u * kThreads;
        if (q < n4) {
            add(pre[u].x, 4 * q); add(pre[u].y, 4 * q + 1);
            add(pre[u].z, 4 * q + 2); add(pre[u].w, 4 * q + 3);
        }
    }
    for (int64_t q0 = threadIdx.x + (int64_t)kTilePre * kThreads; q0 < n4; q0 += 4 * kThreads) {
        int4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (q0 + u * kThreads < n4) v[u] = __ldg(p4 + q0 + u * kThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t q = q0 + u * kThreads;
            if (q < n4) {
                add(v[u].x, 4 * q); add(v[u].y, 4 * q + 1);
                add(v[u].z, 4 * q + 2); add(v[u].w, 4 * q + 3);
            }
        }
    }
    for (int64_t i = n4 * 4 + threadIdx.x; i < a.n; i += kThreads) add(__ldg(a.idx + i), i);
    if (writer) {
        for (int sh = 16; sh; sh >>= 1) invalid += __shfl_xor_sync(0xffffffffu, invalid, sh);
        if (lane == 0 && invalid) atomicAdd(&s_inval, invalid);
    }
    __syncthreads();

    // totals, bucket offsets, the range's first rank per expert
    const int e = threadIdx.x;
    const int32_t bef = (e < a.E) ? s_bef[e] : 0;
    const int32_t tot = (e < a.E) ? bef + s_aft[e] : 0;
    int32_t total;
    const int32_t offe = block_scan(tot, s_scan, total);
    if (e < a.E) {
        s_base[e] = offe + bef;
        if (writer) {
            a.cnt[e] = tot;
            a.off[e] = offe;
        }
    }
    if (writer && threadIdx.x == 0) {
        a.off[a.E] = total;
        *a.n_invalid = s_inval;
    }
    // per expert, exclusive scan over the warps of the range: thread e walks
    // expert e's column (16 counts loaded before any is rewritten; against
    // one warp per expert scanning it with shuffles, back to back in a
    // graph: 13.27 -> 12.44 us for 1024 fp8 tokens at E=256, 28.8 -> 26.1 us
    // for 3000 tokens at E=1024 K=32)
    if (e < a.E) {
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

    // ranks of the own entries
    {
        const unsigned peers = __match_any_sync(0xffffffffu, k_own);
        if (ci < b1) {
            int32_t row = -1;
            if (k_own >= 0)
                row = s_base[k_own] + s_wc[warp * wstride + k_own] + __popc(peers & lanemask_lt());
            s_row[ci - b0] = row;
            a.map[ci] = row;
            if (row >= 0) a.src[row] = (int32_t)ci;
        }
    }
    __syncthreads();

    // rows: unit = (own token, 512-byte segment), kCopyUnroll units per warp
    // with their loads issued first
    const int64_t per_tok = a.segs + a.ssegs;
    const int64_t units = (t1 - t0) * per_tok;
    for (int64_t u0 = (int64_t)warp * kCopyUnroll; u0 < units; u0 += (int64_t)kWarps * kCopyUnroll) {
        uint4 v[kCopyUnroll];
        int64_t tok[kCopyUnroll], obs[kCopyUnroll], len[kCopyUnroll];
        bool is_row[kCopyUnroll], act[kCopyUnroll];
#pragma unroll
        for (int j = 0; j < kCopyUnroll; ++j) {
            const int64_t u = u0 + j;
            const int64_t tl = u / per_tok;
            const int64_t g = u - tl * per_tok;
            is_row[j] = g < a.segs;
            len[j] = is_row[j] ? a.row_bytes : a.scale_bytes;
            obs[j] = (is_row[j] ? g : g - a.segs) * kSeg + lane * 16;
            tok[j] = tl;
            act[j] = u < units && obs[j] < len[j];
            if (act[j])
                v[j] = ld_stream16((is_row[j] ? a.x : a.xs) + (t0 + tl) * len[j] + obs[j]);
        }
#pragma unroll
        for (int j = 0; j < kCopyUnroll; ++j) {
            if (!act[j]) continue;
            uint8_t *dst = is_row[j] ? a.px : a.ps;
            for (int k = 0; k < a.K; ++k) {
                const int32_t r = s_row[tok[j] * a.K + k];
                if (r < 0) continue;
                if (r < a.packed_rows) {
#if MOE_PD_STORE_CS
                    st16_cs(dst + (int64_t)r * len[j] + obs[j], v[j]);
#else
                    st16(dst + (int64_t)r * len[j] + obs[j], v[j]);
#endif
                } else {
                    atomicOr(&g_pd_error, kErrDispatchIndex);
                }
            }
        }
    }
}

#ifndef MOE_PD_TILED
#define MOE_PD_TILED 1
#endif
constexpr int64_t kTiledMaxEntries = 131072;
// Copy bytes up to which the token-range kernel is used.  Its CTAs split the
// copy statically, one range each, and SMs of this part copy at different
// rates, so its time grows with the slowest SM's share; moe_plan followed by
// the multi-wave dispatch pays a second launch but balances the copy (and
// overlaps its first loads with the plan).  Measured on GB300 (plan +
// dispatch alone, and followed by the combine): H=7168 bf16, K=8: the one
// launch ahead at 1536 tokens (176 MB of packed rows: 37.3 against 40.1 us),
// the two calls ahead from 2048 tokens (235 MB: 48.8 against 50.8 us; with
// the combine 87.2 against 90.3 us) and by 2-40 us beyond; H=6144 fp8 rows
// with scales, K=8: the one launch ahead or level up to 4096 tokens (207 MB).
#ifndef MOE_PD_TILED_MAX_BYTES
#define MOE_PD_TILED_MAX_BYTES (192ll << 20)
#endif

int launch_tiles(const int32_t *topk_idx, const void *x, int64_t S, int K, int E,
                 int64_t row_bytes, const float *x_scales, int64_t n_scales, int32_t *cnt,
                 int64_t *off, int32_t *packed_src, int64_t *tok_map, int32_t *n_invalid,
                 void *packed_x, int64_t packed_rows, float *packed_scales, int64_t tpc,
                 cudaStream_t stream)
{
    PDArgs a = {};
    a.idx = topk_idx;
    a.S = S;
    a.K = K;
    a.E = E;
    a.n = S * (int64_t)K;
    a.x = static_cast<const uint8_t *>(x);
    a.row_bytes = row_bytes;
    a.xs = reinterpret_cast<const uint8_t *>(x_scales);
    a.scale_bytes = n_scales > 0 ? n_scales * 4 : 0;
    a.segs = (row_bytes + kSeg - 1) / kSeg;
    a.ssegs = (a.scale_bytes + kSeg - 1) / kSeg;
    a.cnt = cnt;
    a.off = off;
    a.src = packed_src;
    a.map = tok_map;
    a.n_invalid = n_invalid;
    a.px = static_cast<uint8_t *>(packed_x);
    a.ps = reinterpret_cast<uint8_t *>(packed_scales);
    a.packed_rows = packed_rows;
    const size_t smem =
        ((size_t)kWarps * (E | 1) + 3 * (size_t)E + (size_t)(tpc * K)) * sizeof(int32_t);
    static KernelCache cache;
    cudaError_t err = prepare_kernel(plan_dispatch_tiles_kernel, smem, kThreads, cache, nullptr);
    if (err == cudaSuccess) {
        const unsigned blocks = (unsigned)((S + tpc - 1) / tpc);
        err = launch_pdl(plan_dispatch_tiles_kernel, dim3(blocks), dim3(kThreads), smem, stream,
                         a, tpc);
    }
    if (err != cudaSuccess) {
        set_cuda_error(err);
        return MOE_ECUDA;
    }
    return check_launch();
}

} // namespace
} // namespace moe

using namespace moe;

MOE_EXPORT int64_t moe_plan_dispatch_fused_max(void) { return kFusedMaxEntries; }

MOE_EXPORT int moe_plan_dispatch(const int32_t *topk_idx, const void *x, int64_t S, int64_t H,
                                 int dtype, int K, int E, const float *x_scales,
                                 int64_t n_scales, int32_t *cnt, int64_t *off,
                                 int32_t *packed_src, int64_t *tok_map, int32_t *n_invalid,
                                 void *packed_x, int64_t packed_rows, float *packed_scales,
                                 void *workspace, size_t workspace_bytes, moe_stream_t stream)
{
    MOE_TRACE("moe_plan_dispatch");
    const int es = elem_size(dtype);
    if (es == 0 || S < 0 || H < 1 || K < 1 || K > 32 || E < 1 || E > 1024 || n_scales < 0 ||
        n_scales > 256)
        return MOE_EINVAL;
    if (S * (int64_t)K >= ((int64_t)1 << 31)) return MOE_EINVAL;
    if (!cnt || !off || !n_invalid) return MOE_EINVAL;
    if (S > 0 && (!topk_idx || !x || !packed_src || !tok_map || !packed_x || packed_rows < 1))
        return MOE_EINVAL;
    if (S > 0 && n_scales > 0 && (!x_scales || !packed_scales)) return MOE_EINVAL;
    const int64_t row_bytes = H * es;
    if (S > 0) {
        if (row_bytes % 16 || !aligned16(x) || !aligned16(packed_x)) return MOE_EALIGN;
        if (n_scales > 0 &&
            ((n_scales * 4) % 16 || !aligned16(x_scales) || !aligned16(packed_scales)))
            return MOE_EALIGN;
    }
    const int64_t n = S * (int64_t)K;
    // larger batches: CTAs own token ranges of at most 1024 entries, one CTA
    // per SM; each counts all n entries itself, so this stops at kTiledMax;
    // and above MOE_PD_TILED_MAX_BYTES of rows to copy the two calls win
    const int64_t tpc = (S + sm_count() - 1) / sm_count();
    const int64_t copy_bytes = n * (row_bytes + n_scales * 4);
    if (MOE_PD_TILED && n > kFusedMaxEntries && n <= kTiledMaxEntries && tpc * K <= kThreads &&
        copy_bytes <= MOE_PD_TILED_MAX_BYTES)
        return launch_tiles(topk_idx, x, S, K, E, row_bytes, x_scales, n_scales, cnt, off,
                            packed_src, tok_map, n_invalid, packed_x, packed_rows, packed_scales,
                            tpc, (cudaStream_t)stream);
    if (n == 0 || n > kFusedMaxEntries) {
        // throughput path: the two calls it fuses, back to back; the plan's
        // kernel lets the dispatch launch only once everything before the
        // plan is complete, so the dispatch may load x before it waits
        if (int rc = moe_plan(topk_idx, S, K, E, cnt, off, packed_src, tok_map, n_invalid,
                              workspace, workspace_bytes, stream))
            return rc;
        return dispatch_rows(x, S, H, dtype, K, tok_map, packed_x, packed_rows, x_scales,
                             n_scales, packed_scales, true, (cudaStream_t)stream);
    }
    PDArgs a = {};
    a.idx = topk_idx;
    a.S = S;
    a.K = K;
    a.E = E;
    a.n = n;
    a.x = static_cast<const uint8_t *>(x);
    a.row_bytes = row_bytes;
    a.xs = reinterpret_cast<const uint8_t *>(x_scales);
    a.scale_bytes = n_scales > 0 ? n_scales * 4 : 0;
    a.segs = (row_bytes + kSeg - 1) / kSeg;
    a.ssegs = (a.scale_bytes + kSeg - 1) / kSeg;
    a.cnt = cnt;
    a.off = off;
    a.src = packed_src;
    a.map = tok_map;
    a.n_invalid = n_invalid;
    a.px = static_cast<uint8_t *>(packed_x);
    a.ps = reinterpret_cast<uint8_t *>(packed_scales);
    a.packed_rows = packed_rows;

    // one warp per (token, segment) unit, at most one CTA per SM
    int ti = 0;  // 256 << ti threads
    while ((256 << ti) < E) ++ti;
    static void (*const kFns[3])(PDArgs) = {plan_dispatch_kernel<256>, plan_dispatch_kernel<512>,
                                           plan_dispatch_kernel<1024>};
    static_assert(kThreads == 1024, "the largest CTA gives every expert of E <= 1024 a thread");
    const int threads = 256 << ti;
    void (*fn)(PDArgs) = kFns[ti];
    const size_t smem =
        ((size_t)(threads / 32) * (E | 1) + (size_t)E + (size_t)n) * sizeof(int32_t);
    static KernelCache caches[3];
    int per_sm = 0;
    cudaError_t err = prepare_kernel(fn, smem, threads, caches[ti], &per_sm);
    if (err != cudaSuccess || per_sm < 1) {
        set_cuda_error(err != cudaSuccess ? err : cudaErrorInvalidConfiguration);
        return MOE_ECUDA;
    }
    const int64_t units = S * (a.segs + a.ssegs);
    int64_t blocks = (units + threads / 32 - 1) / (threads / 32);
    if (blocks > sm_count()) blocks = sm_count();
    if (blocks < 1) blocks = 1;
    err = launch_pdl(fn, dim3((unsigned)blocks), dim3(threads), smem, (cudaStream_t)stream, a);
    if (err != cudaSuccess) {
        set_cuda_error(err);
        return MOE_ECUDA;
    }
    return check_launch();
}

namespace moe {
// Reads and clears this file's device error bits.
cudaError_t read_plan_dispatch_errors(uint32_t *flags)
{
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_pd_error, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_pd_error, &zero, sizeof(uint32_t));
    return e;
}
} // namespace moe
