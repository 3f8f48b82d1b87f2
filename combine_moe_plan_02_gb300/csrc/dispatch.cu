// Dispatch: scatter token rows into per-expert packed buckets with bulk TMA.
//
// Sources: ROCm/mori "Draft: cco + flydsl dispatch/combine #448": PR
// description (16-byte scatter of each token row, a byte-generic copy),
// StdMoE note (packed_x[expert, slot] repack, per (received token, k)),
// scale_dim note (each token's scale block forwarded verbatim with the row);
// MoonEP "Drop cooperative launch ...": the local dispatch epilogue stages
// rows through shared memory with TMA and mbarriers, CTAs independent.
//
// GB300 design: each warp runs its own ring of kStages shared-memory stages.
// Lane 0 pulls one chunk of a source row into a stage with
// cp.async.bulk (global -> shared, completion counted on an mbarrier); once
// it lands, lanes 0..K-1 each push that stage to their destination row with
// cp.async.bulk (shared -> global).  The row is read from HBM once and
// written K times, and the SM issues two instructions per 16 B * chunk/16 of
// traffic instead of one load/store pair per 16 bytes.  A stage is refilled
// only after the stores that read it have drained (bulk wait_group.read).
// Every mbarrier wait is bounded; on expiry the kernel records an error bit,
// drains what it issued, and returns.

#include "common.cuh"

#include <cuda_fp8.h>

namespace moe {
namespace {

#ifndef MOE_DISPATCH_WARPS
#define MOE_DISPATCH_WARPS 4
#endif
// One stage per warp: with a grid of several resident waves a warp mostly
// moves a single chunk, and small CTAs (14 KB of shared memory at 3.5 KB
// chunks) let many of them wait ready while the plan before them finishes:
// plan + dispatch 91.8 -> 89.4 us and the step 176.9 -> 174.7 us at the
// MoonEP shape, against four stages.
#ifndef MOE_DISPATCH_STAGES
#define MOE_DISPATCH_STAGES 1
#endif
#ifndef MOE_DISPATCH_CHUNK
#define MOE_DISPATCH_CHUNK 4096
#endif
// Grid size in resident waves.  With one wave (a persistent grid) every warp
// owns a fixed share of the chunks and the slowest SMs set the pace; with
// eight, the block scheduler keeps handing CTAs to the SMs that finish
// first: 89.0 -> 81.9 us at S=4096 H=7168 K=8 (each warp then mostly moves
// one chunk through its ring).
#ifndef MOE_DISPATCH_GRID_WAVES
#define MOE_DISPATCH_GRID_WAVES 8
#endif
constexpr int kWarpsPerCta = MOE_DISPATCH_WARPS;
constexpr int kStages = MOE_DISPATCH_STAGES;
constexpr int kMaxChunk = MOE_DISPATCH_CHUNK;  // bytes of a row moved per stage
constexpr int kMaxScaleBytes = 1024;   // scale row bytes that travel with a row
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per mbarrier wait

__device__ uint32_t g_dispatch_error;  // kErrDispatchTimeout | kErrDispatchIndex

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for phase `parity` of `bar`; false after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Self-test of the timeout path: one warp waits, through the same bounded
// wait as the dispatch kernels, on an mbarrier phase that nothing completes
// (no copy is issued and nothing arrives), records the dispatch timeout bit
// when the limit expires, and returns.  Nothing else is touched.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const bool landed = mbar_wait_bounded(&bar, 0, limit_ns);
    if (!__all_sync(0xffffffffu, landed) && lane == 0)
        atomicOr(&g_dispatch_error, kErrDispatchTimeout);
}

struct CopyArgs {
    const uint8_t *src;        // source rows, row_bytes apart
    uint8_t *dst;              // destination rows, row_bytes apart
    int64_t row_bytes;         // multiple of 16
    int chunk;                 // bytes per stage (multiple of 16)
    int n_chunks;              // chunks per row
    int K;                     // destinations per source row (dst_map) or 1
    const int64_t *dst_map;    // [rows, K] destination row or -1; null: dst row = item row
    const int32_t *src_map;    // null: source row = item row; else src_map[item] / src_div
    int src_div;
    int64_t rows;              // item rows (host bound)
    const int64_t *rows_dev;   // if set, item rows = min(*rows_dev, rows)
    int64_t src_rows;          // rows of the source buffer (bounds check)
    int64_t dst_rows;          // rows the destination buffer may hold (bounds check)
    const uint8_t *ssrc;       // scale rows travelling with chunk 0 (or null)
    uint8_t *sdst;
    int scale_bytes;           // multiple of 16 (0 = none)
    int stage_bytes;           // chunk + scale area, multiple of 128
    uint8_t *dst2;             // with dst_map and K < 32: lane K also stores item row r here
    int64_t dst2_rows;         // rows of dst2 (bounds check)
    // dedup by token (2K <= 32): item row r is token r; lanes K..2K-1 store
    // to its group rows gtok_map[r, k] in dst2, lanes 0..K-1 to the packed
    // rows read from grp_map (the group rows' expert maps)
    const int64_t *gtok_map;   // [rows, K] or null
    const int64_t *grp_map;    // [dst2_rows, K]
    // the source rows were complete before the previous kernel of the stream
    // started waiting for its own predecessors (the plan of moe_plan_dispatch
    // lets its dependents launch only after that), so the first loads may be
    // issued before this kernel waits; with src_map or rows_dev: ignored
    bool early_src;
};

__global__ void __launch_bounds__(kWarpsPerCta * 32) dispatch_bulk_kernel(CopyArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kWarpsPerCta][kStages];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *ring = smem + (size_t)warp * kStages * a.stage_bytes;
    uint64_t *bar = bars[warp];

    if (lane == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(&bar[st], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // Everything that reads the maps or writes packed rows waits for earlier
    // stream work (the plan; readers of packed_x).  With early_src the first
    // source loads go out before that wait, while the plan finishes.
    const bool early = a.early_src && a.src_map == nullptr && a.rows_dev == nullptr;
    if (!early) {
        griddep_wait();
        griddep_launch_dependents();
    }

    const int64_t rows = a.rows_dev ? min(*a.rows_dev, a.rows) : a.rows;
    const int64_t n_items = rows * a.n_chunks;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerCta + warp;
    const int64_t W = (int64_t)gridDim.x * kWarpsPerCta;
    if (gw >= n_items) return;
    // items of this warp: gw + j*W, j = 0 .. n_mine-1
    const int64_t n_mine = (n_items - gw + W - 1) / W;

    int64_t dst_row[kStages];  // this lane's destination row per stage
    int64_t issued = 0;        // items whose load has been issued

    // the source chunk of item j into stage st; returns whether the source
    // row lies inside its buffer
    auto issue_load = [&](int64_t j, int st) -> bool {
        issued = j + 1;
        const int64_t it = gw + j * W;
        const int64_t r = it / a.n_chunks;
        const int c = (int)(it - r * a.n_chunks);
        const int64_t off = (int64_t)c * a.chunk;
        const uint32_t bytes = (uint32_t)min((int64_t)a.chunk, a.row_bytes - off);
        int64_t sr = a.src_map ? (int64_t)(__ldg(a.src_map + r) / a.src_div) : r;
        const bool src_ok = sr >= 0 && sr < a.src_rows;
        const bool with_scales = a.scale_bytes > 0 && c == 0;
        if (lane == 0) {
            uint8_t *stage = ring + (size_t)st * a.stage_bytes;
            if (src_ok) {
                mbar_arrive_expect_tx(&bar[st], bytes + (with_scales ? a.scale_bytes : 0));
                bulk_g2s(stage, a.src + sr * a.row_bytes + off, bytes, &bar[st]);
                if (with_scales)
                    bulk_g2s(stage + a.chunk, a.ssrc + sr * a.scale_bytes, a.scale_bytes,
                             &bar[st]);
            } else {
                // a source row outside the buffer: move nothing, complete the
                // phase with a plain arrive, and report it
                mbar_arrive(&bar[st]);
                atomicOr(&g_dispatch_error, kErrDispatchIndex);
            }
        }
        return src_ok;
    };

    // this lane's destination row of item j, from the maps
    auto issue_dst = [&](int64_t j, int st, bool src_ok) {
        const int64_t it = gw + j * W;
        const int64_t r = it / a.n_chunks;
        int64_t d = -1;
        bool second;  // this lane stores to dst2
        if (a.gtok_map) {
            second = lane >= a.K && lane < 2 * a.K;
            int64_t gk = -1;  // lane k < K: the token's group row through entry k
            if (lane < a.K) {
                gk = __ldg(a.gtok_map + r * a.K + lane);
                if (gk < -1 || gk >= a.dst2_rows) {
                    atomicOr(&g_dispatch_error, kErrDispatchIndex);
                    gk = -1;
                }
            }
            // lane k < K: its packed row, from the map of the group row that
            // holds entry k (one load per group row of the token)
            for (unsigned m = __ballot_sync(0xffffffffu, gk >= 0); m; m &= m - 1) {
                const int64_t rq = __shfl_sync(0xffffffffu, gk, __ffs(m) - 1);
                if (lane < a.K) {
                    const int64_t e = __ldg(a.grp_map + rq * a.K + lane);
                    if (e != -1) d = e;
                }
            }
            const int64_t g2 = __shfl_sync(0xffffffffu, gk, (lane - a.K) & 31);
            if (second) d = g2;
        } else {
            second = a.dst2 != nullptr && lane == a.K;  // the item's own copy
            if (a.dst_map) {
                if (lane < a.K) d = __ldg(a.dst_map + r * a.K + lane);
                else if (second) d = r;
            } else if (lane == 0) {
                d = r;
            }
        }
        const int64_t lim = second ? a.dst2_rows : a.dst_rows;
        if (d >= lim || d < -1 || (d >= 0 && !src_ok)) {
            if (d >= lim || d < -1) atomicOr(&g_dispatch_error, kErrDispatchIndex);
            d = -1;
        }
        dst_row[st] = d;
    };

    auto issue = [&](int64_t j, int st) { issue_dst(j, st, issue_load(j, st)); };

    // prologue: fill the ring
    if (early) {
        bool ok_src[kStages];
#pragma unroll
        for (int st = 0; st < kStages; ++st)
            if (st < n_mine) ok_src[st] = issue_load(st, st);
        griddep_wait();
        griddep_launch_dependents();
#pragma unroll
        for (int st = 0; st < kStages; ++st)
            if (st < n_mine) issue_dst(st, st, ok_src[st]);
    } else {
#pragma unroll
        for (int st = 0; st < kStages; ++st)
            if (st < n_mine) issue(st, st);
    }

    bool ok = true;
    int64_t consumed = 0;   // items whose load has been waited for
    for (int64_t j0 = 0; j0 < n_mine && ok; j0 += kStages) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) {
            const int64_t j = j0 + st;
            if (j >= n_mine || !ok) break;
            // every lane that stores waits on the barrier itself; the outcome
            // is made warp-uniform so the warp never splits around __syncwarp
            const bool landed = mbar_wait_bounded(&bar[st], (uint32_t)((j / kStages) & 1));
            if (!__all_sync(0xffffffffu, landed)) {
                ok = false;
                break;
            }
            consumed = j + 1;
            const int64_t it = gw + j * W;
            const int64_t r = it / a.n_chunks;
            const int c = (int)(it - r * a.n_chunks);
            const int64_t off = (int64_t)c * a.chunk;
            const uint32_t bytes = (uint32_t)min((int64_t)a.chunk, a.row_bytes - off);
            const uint8_t *stage = ring + (size_t)st * a.stage_bytes;
            const int64_t d = dst_row[st];
            if (d >= 0) {
                if (a.gtok_map ? lane >= a.K : (a.dst2 != nullptr && lane == a.K)) {
                    bulk_s2g(a.dst2 + d * a.row_bytes + off, stage, bytes);
                } else {
                    bulk_s2g(a.dst + d * a.row_bytes + off, stage, bytes);
                    if (a.scale_bytes > 0 && c == 0)
                        bulk_s2g(a.sdst + d * a.scale_bytes, stage + a.chunk, a.scale_bytes);
                }
            }
            bulk_commit();
            if constexpr (kStages == 1) {
                // one stage: the next item waits until this item's stores
                // have read the stage
                if (j + 1 < n_mine) {
                    bulk_wait_read<0>();
                    __syncwarp();
                    issue(j + 1, 0);
                }
            } else {
                // refill the stage of item j-1 with item j-1+kStages once
                // the stores reading it have drained
                const int prev = (st + kStages - 1) % kStages;
                const int64_t jn = j - 1 + kStages;
                if (j >= 1 && jn < n_mine) {
                    bulk_wait_read<1>();
                    __syncwarp();
                    issue(jn, prev);
                }
            }
        }
    }

    bulk_wait_all();
    if (!ok) {
        if (lane == 0) atomicOr(&g_dispatch_error, kErrDispatchTimeout);
        // loads already issued but not consumed: items consumed .. issued-1
        for (int64_t j = consumed; j < issued; ++j)
            (void)mbar_wait_bounded(&bar[j % kStages], (uint32_t)((j / kStages) & 1));
    }
}

// ---------------------------------------------------------------------------
// Quantising dispatch: bf16 rows in, blockwise E4M3 codes and f32 scales out,
// each written to the token's K packed rows.  Sources: ROCm/mori "Draft: cco +
// flydsl dispatch/combine #448", Fp8BlockwiseQuant notes (per-block amax and
// f32 scale, then the fp8 cast; the coalesced version reduces the block amax
// across lanes with a butterfly) and scale_dim note (scale rows travel with
// the token).  The rule: scale = amax / 448 (1 for an all-zero block),
// code = E4M3(v / scale), both divisions IEEE f32, the cast to nearest even
// and saturating.
//
// Two kernels compute the same bits: the wide kernel further down takes the
// common case (H a multiple of 4 * block, 16-byte aligned scales); the
// register kernel here takes every other shape.  It gives a warp (token,
// slice) units: each lane holds 8 consecutive elements (one 16-byte load), a
// block of `block` elements spans block/8 lanes, and its amax is an
// xor-shuffle reduction inside that lane group.  All of a unit's loads are
// issued first.  Each lane then stores its 8 codes (8 bytes; a warp writes
// 256 contiguous bytes) to every destination row, and the first lane of each
// block stores the block's scale.
// ---------------------------------------------------------------------------

constexpr int kQThreads = 256;
constexpr int kQMaxIters = 8;  // 256-element steps per lane group per unit

struct QuantArgs {
    const uint8_t *x;         // bf16 [S, H]
    int64_t S, H;
    int K;
    const int64_t *tok_map;   // [S, K]
    int64_t dst_rows;         // rows of the packed buffers (bounds check)
    int block;                // elements per scale (16..256, power of two)
    int iters;                // 256-element steps per row
    int R;                    // steps per unit
    int slices;               // units per row
    uint8_t *q;               // [dst_rows, H] E4M3 codes
    float *scales;            // [dst_rows, H / block]
};

// IEEE division, kept out of line: only blocks of tiny values take it, and
// inlined it would crowd the registers of the common path.
__device__ __noinline__ float div_rn_out_of_line(float a, float b) { return __fdiv_rn(a, b); }

// The scale of one block and the correctly rounded quotient of an element
// by it.  Divisions, correctly rounded, by Markstein's correction step
// (P. Markstein, IBM J. Res. Dev. 34(1), 1990): with y = RN(1/b) and
// q = RN(a*y), the residual a - q*b is exact under FMA and RN(q + residual*y)
// = RN(a/b).  The residual is exact only while a is at least 2^-102 (24 bits
// above the subnormal range); a block whose amax is below 2^-83 can hold
// elements that small with quotients that still reach an E4M3 code, so such
// blocks take full divisions instead.
struct BlockScale {
    float scale;  // amax / 448, or 1 for an all-zero block
    float y;      // RN(1 / scale): one reciprocal per block
    bool slow;    // a block of tiny values: full divisions
};

__device__ __forceinline__ BlockScale block_scale(float amax)
{
    constexpr float kInv448 = 1.0f / 448.0f;  // RN(1/448)
    const bool exact_fast = amax >= 0x1p-83f;
    BlockScale b;
    b.scale = 1.0f;
    if (exact_fast) {
        const float q0 = __fmul_rn(amax, kInv448);
        b.scale = __fmaf_rn(__fmaf_rn(-q0, 448.0f, amax), kInv448, q0);
    } else if (amax > 0.0f) {
        b.scale = div_rn_out_of_line(amax, 448.0f);
    }
    b.y = __frcp_rn(b.scale);
    b.slow = amax > 0.0f && !exact_fast;
    return b;
}

// RN(x / scale).  A zero residual means q0 is the exact quotient, and
// returning it keeps the sign of -0.
__device__ __forceinline__ float quot_rn(float x, const BlockScale &b)
{
    if (b.slow) return div_rn_out_of_line(x, b.scale);
    const float q0 = __fmul_rn(x, b.y);
    const float r = __fmaf_rn(-q0, b.scale, x);
    return r == 0.0f ? q0 : __fmaf_rn(r, b.y, q0);
}

// Four E4M3 codes (nearest even, saturating), little-endian in one word.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE,
                                                             __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE,
                                                             __NV_E4M3);
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// The 8 bf16 values of a 16-byte word, widened to f32 in element order.
__device__ __forceinline__ void widen8(const uint4 v, float *f)
{
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        f[2 * q] = __uint_as_float(w4[q] << 16);
        f[2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u);
    }
}

// Quantises the 8 bf16 values of one lane (one 16-byte word) for a block of
// GL lanes: returns the 8 E4M3 codes (little-endian in two words) and the
// block's scale.  All 32 lanes must call it together (block amax shuffle).
template <int GL>
__device__ __forceinline__ uint2 quant8(const uint4 v, bool active, float &scale_out)
{
    float f[8];
    widen8(v, f);
    float amax = 0.0f;
    if (active) {
#pragma unroll
        for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(f[q]));
    }
#pragma unroll
    for (int o = GL / 2; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const BlockScale b = block_scale(amax);
    uint32_t packed[2];
#pragma unroll
    for (int q = 0; q < 2; ++q)
        packed[q] = e4m3x4(quot_rn(f[4 * q], b), quot_rn(f[4 * q + 1], b),
                           quot_rn(f[4 * q + 2], b), quot_rn(f[4 * q + 3], b));
    scale_out = b.scale;
    return make_uint2(packed[0], packed[1]);
}

// The same for the 16 bf16 values of two consecutive 16-byte words (a block
// spans GL lanes of 16 elements): 16 codes in one 16-byte word.
template <int GL>
__device__ __forceinline__ uint4 quant16(const uint4 v0, const uint4 v1, bool active,
                                         float &scale_out)
{
    float f[16];
    widen8(v0, f);
    widen8(v1, f + 8);
    float amax = 0.0f;
    if (active) {
#pragma unroll
        for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(f[q]));
    }
#pragma unroll
    for (int o = GL / 2; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const BlockScale b = block_scale(amax);
    uint32_t packed[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        packed[q] = e4m3x4(quot_rn(f[4 * q], b), quot_rn(f[4 * q + 1], b),
                           quot_rn(f[4 * q + 2], b), quot_rn(f[4 * q + 3], b));
    scale_out = b.scale;
    return make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

template <int GL>  // lanes per block (block / 8)
__global__ void __launch_bounds__(kQThreads, 2) dispatch_quant_kernel(QuantArgs a)
{
    griddep_wait();
    griddep_launch_dependents();

    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * kQThreads + threadIdx.x) >> 5;
    const int64_t W = ((int64_t)gridDim.x * kQThreads) >> 5;
    const int64_t units = a.S * a.slices;
    const int K = a.K;
    const int64_t nb = a.H / a.block;

    for (int64_t u = gw; u < units; u += W) {
        const int64_t s = u / a.slices;
        const int sl = (int)(u - s * a.slices);
        int32_t my_row = -1;
        if (lane < K) {
            const int64_t r = __ldg(a.tok_map + s * K + lane);
            if (r >= 0 && r < a.dst_rows) {
                my_row = (int32_t)r;
            } else if (r != -1) {
                atomicOr(&g_dispatch_error, kErrDispatchIndex);
            }
        }
        // load first: every 16-byte load of the unit is in flight
        uint4 v[kQMaxIters];
        const int it0 = sl * a.R;
#pragma unroll
        for (int r = 0; r < kQMaxIters; ++r) {
            const int64_t e = ((int64_t)(it0 + r) * 32 + lane) * 8;  // first element
            if (r < a.R && it0 + r < a.iters && e < a.H)
                v[r] = ld_stream16(a.x + (s * a.H + e) * 2);
        }
#pragma unroll
        for (int r = 0; r < kQMaxIters; ++r) {
            if (r >= a.R || it0 + r >= a.iters) break;  // uniform across the warp
            const int64_t e = ((int64_t)(it0 + r) * 32 + lane) * 8;
            const bool active = e < a.H;
            float scale;
            const uint2 codes = quant8<GL>(v[r], active, scale);
            const uint32_t packed[2] = {codes.x, codes.y};
            const bool block_lead = (lane % GL) == 0;
            const int64_t b = e / a.block;
            for (int k = 0; k < K; ++k) {
                const int32_t d = __shfl_sync(0xffffffffu, my_row, k);
                if (d < 0 || !active) continue;
                uint8_t *dst = a.q + (int64_t)d * a.H + e;
                asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(dst), "r"(packed[0]),
                             "r"(packed[1])
                             : "memory");
                if (block_lead) a.scales[(int64_t)d * nb + b] = scale;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Quantising dispatch, wide form (the common case: every chunk's scale run is
// a whole number of 16-byte words, H a multiple of 4 * block, and the scale
// buffer 16-byte aligned).  A warp owns (token, 1024-element chunk) units;
// each lane quantises 16 consecutive elements per 512-element step, so that
// its 16 codes leave as ONE 16-byte store per destination row (a warp store
// covers 512 contiguous bytes), and the chunk's scale run (4 to 64 floats) is
// collected in shared memory and leaves as 16-byte stores of whole words.
// All of a unit's loads (4 x 16 bytes per lane) are issued first.  No
// mbarrier, no bulk-copy engine: the stores go straight from registers, and
// at 48 registers per thread 40 warps fit on an SM.
// ---------------------------------------------------------------------------

#ifndef MOE_QW_STORE_CS
#define MOE_QW_STORE_CS 1
#endif
// Grid size in resident waves, as MOE_DISPATCH_GRID_WAVES: 55.0 -> 51.2 us
// at S=4096 H=7168 K=8 with four waves instead of one.
#ifndef MOE_QW_GRID_WAVES
#define MOE_QW_GRID_WAVES 4
#endif
constexpr int kQWThreads = 256;
constexpr int kQWWarps = kQWThreads / 32;
constexpr int kQWChunk = 1024;            // elements per unit (2 steps of 512)

struct QWideArgs {
    const uint8_t *x;         // bf16 [S, H]
    int64_t S, H;
    int K;
    const int64_t *tok_map;   // [S, K]
    int64_t dst_rows;
    int block;
    int64_t nb;               // scales per row, H / block (a multiple of 4)
    int n_chunks;             // units per row
    uint8_t *q;               // [dst_rows, H]
    float *sc;                // [dst_rows, nb], 16-byte aligned
};

__device__ __forceinline__ void st16_q(void *p, uint4 v)
{
#if MOE_QW_STORE_CS
    st16_cs(p, v);
#else
    st16(p, v);
#endif
}

// Five 256-thread CTAs per SM (48 registers): 49.1 us at the MoonEP shape
// against 50.6 us for four (60 registers).
template <int GL>  // lanes per block (block / 16)
__global__ void __launch_bounds__(kQWThreads, 5) dispatch_quant_wide_kernel(QWideArgs a)
{
    __shared__ __align__(16) float s_sc[kQWWarps][kQWChunk / 16];  // a unit's scale run

    griddep_wait();  // the plan and earlier readers of the packed buffers are done
    griddep_launch_dependents();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * kQWWarps + warp;
    const int64_t W = (int64_t)gridDim.x * kQWWarps;
    const int64_t units = a.S * a.n_chunks;
    const int K = a.K;
    float *my_sc = s_sc[warp];

    for (int64_t u = gw; u < units; u += W) {
        const int64_t s = u / a.n_chunks;
        const int c = (int)(u - s * a.n_chunks);
        const int64_t e0 = (int64_t)c * kQWChunk;
        const int elems = (int)min((int64_t)kQWChunk, a.H - e0);  // a multiple of 4 * block
        int32_t my_row = -1;
        if (lane < K) {
            const int64_t r = __ldg(a.tok_map + s * K + lane);
            if (r >= 0 && r < a.dst_rows)
                my_row = (int32_t)r;
            else if (r != -1)
                atomicOr(&g_dispatch_error, kErrDispatchIndex);
        }
        // load first: both steps' 32 bytes per lane are in flight together
        const uint8_t *src = a.x + (s * a.H + e0) * 2;
        uint4 v[2][2];
        bool act[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int e = t * 512 + lane * 16;
            act[t] = e < elems;
            if (act[t]) {
                v[t][0] = ld_stream16(src + e * 2);
                v[t][1] = ld_stream16(src + e * 2 + 16);
            } else {
                v[t][0] = v[t][1] = make_uint4(0, 0, 0, 0);
            }
        }
        uint4 codes[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            float scale;
            codes[t] = quant16<GL>(v[t][0], v[t][1], act[t], scale);
            const int e = t * 512 + lane * 16;
            if (act[t] && (lane % GL) == 0) my_sc[e / a.block] = scale;
        }
        __syncwarp();
        const int nsc = elems / a.block;            // scales of this unit
        const bool sc_lane = lane * 4 < nsc;
        uint4 scw = make_uint4(0, 0, 0, 0);
        if (sc_lane) scw = *reinterpret_cast<const uint4 *>(my_sc + lane * 4);
        __syncwarp();                                // my_sc is rewritten by the next unit
        for (int k = 0; k < K; ++k) {
            const int32_t d = __shfl_sync(0xffffffffu, my_row, k);
            if (d < 0) continue;                     // the same for every lane
            uint8_t *dq = a.q + (int64_t)d * a.H + e0;
#pragma unroll
            for (int t = 0; t < 2; ++t)
                if (act[t]) st16_q(dq + t * 512 + lane * 16, codes[t]);
            if (sc_lane) st16_q(a.sc + (int64_t)d * a.nb + e0 / a.block + lane * 4, scw);
        }
    }
}

int pick_chunk(int64_t row_bytes, int *n_chunks)
{
    // split the row into m equal chunks of at most kMaxChunk bytes when the
    // 16-byte units divide evenly, else kMaxChunk-sized chunks and a short tail
    const int64_t units = row_bytes / 16;
    int64_t m = (row_bytes + kMaxChunk - 1) / kMaxChunk;
    for (int64_t mm = m; mm <= m + 8; ++mm) {
        if (units % mm == 0) {
            *n_chunks = (int)mm;
            return (int)(row_bytes / mm);
        }
    }
    *n_chunks = (int)m;
    return kMaxChunk;
}

int launch_copy(CopyArgs &a, cudaStream_t stream)
{
    a.stage_bytes = (a.chunk + a.scale_bytes + 127) / 128 * 128;
    const size_t smem = (size_t)kWarpsPerCta * kStages * a.stage_bytes;
    static KernelCache cache;
    int per_sm = 0;
    cudaError_t err = prepare_kernel(dispatch_bulk_kernel, smem, kWarpsPerCta * 32, cache, &per_sm);
    if (err != cudaSuccess || per_sm < 1) {
        set_cuda_error(err != cudaSuccess ? err : cudaErrorInvalidConfiguration);
        return MOE_ECUDA;
    }
    const int64_t items = a.rows * a.n_chunks;
    int64_t blocks = (items + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t cap = (int64_t)sm_count() * per_sm * MOE_DISPATCH_GRID_WAVES;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    err = launch_pdl(dispatch_bulk_kernel, dim3((unsigned)blocks), dim3(kWarpsPerCta * 32), smem,
                     stream, a);
    if (err != cudaSuccess) {
        set_cuda_error(err);
        return MOE_ECUDA;
    }
    return check_launch();
}

} // namespace
} // namespace moe

using namespace moe;

MOE_EXPORT int moe_dispatch(const void *x, int64_t S, int64_t H, int dtype, int K,
                            const int64_t *tok_map, void *packed_x, int64_t packed_rows,
                            const float *x_scales, int64_t n_scales, float *packed_scales,
                            moe_stream_t stream)
{
    MOE_TRACE("moe_dispatch");
    return dispatch_rows(x, S, H, dtype, K, tok_map, packed_x, packed_rows, x_scales, n_scales,
                         packed_scales, false, (cudaStream_t)stream);
}

// moe_dispatch; with early_src (moe_plan_dispatch, right after its plan) the
// first source loads may precede the wait for the plan
int moe::dispatch_rows(const void *x, int64_t S, int64_t H, int dtype, int K,
                       const int64_t *tok_map, void *packed_x, int64_t packed_rows,
                       const float *x_scales, int64_t n_scales, float *packed_scales,
                       bool early_src, cudaStream_t stream)
{
    const int es = elem_size(dtype);
    if (es == 0 || S < 0 || H < 1 || K < 1 || K > 32 || n_scales < 0) return MOE_EINVAL;
    if (S == 0) return MOE_OK;
    if (!x || !tok_map || !packed_x || packed_rows < 1) return MOE_EINVAL;
    if (n_scales > 0 && (!x_scales || !packed_scales)) return MOE_EINVAL;
    const int64_t row_bytes = H * es;
    if (row_bytes % 16 || !aligned16(x) || !aligned16(packed_x)) return MOE_EALIGN;
    if (n_scales > 0 && ((n_scales * 4) % 16 || !aligned16(x_scales) || !aligned16(packed_scales)))
        return MOE_EALIGN;
    if (n_scales * 4 > kMaxScaleBytes) return MOE_EINVAL;
    CopyArgs a = {};
    a.src = static_cast<const uint8_t *>(x);
    a.dst = static_cast<uint8_t *>(packed_x);
    a.row_bytes = row_bytes;
    a.chunk = pick_chunk(row_bytes, &a.n_chunks);
    a.K = K;
    a.dst_map = tok_map;
    a.src_div = 1;
    a.rows = S;
    a.src_rows = S;
    a.dst_rows = packed_rows;
    a.ssrc = reinterpret_cast<const uint8_t *>(x_scales);
    a.sdst = reinterpret_cast<uint8_t *>(packed_scales);
    a.scale_bytes = (int)(n_scales * 4);
    a.early_src = early_src;
    return launch_copy(a, stream);
}

MOE_EXPORT int moe_dispatch_dedup(const void *x, int64_t S, int64_t H, int dtype, int K, int G,
                                  const int64_t *goff, const int32_t *grp_src,
                                  const int64_t *grp_tok_map, const int64_t *gtok_map,
                                  int64_t max_rows, void *grp_x, void *packed_x,
                                  int64_t packed_rows, moe_stream_t stream)
{
    MOE_TRACE("moe_dispatch_dedup");
    const int es = elem_size(dtype);
    if (es == 0 || S < 0 || H < 1 || K < 1 || K > 32 || G < 1 || G > 1024) return MOE_EINVAL;
    if (S == 0) return MOE_OK;
    if (!x || !goff || !grp_src || !grp_tok_map || !gtok_map || !grp_x || !packed_x ||
        packed_rows < 1)
        return MOE_EINVAL;
    if (max_rows < S * (int64_t)(K < G ? K : G)) return MOE_EINVAL;
    const int64_t row_bytes = H * es;
    if (row_bytes % 16 || !aligned16(x) || !aligned16(grp_x) || !aligned16(packed_x))
        return MOE_EALIGN;
    CopyArgs a = {};
    a.row_bytes = row_bytes;
    a.chunk = pick_chunk(row_bytes, &a.n_chunks);
    if (2 * K <= 32) {
        // by token: each chunk of x[s] is staged once and stored to the
        // token's group rows and to its experts' packed rows
        a.src = static_cast<const uint8_t *>(x);
        a.rows = S;
        a.src_rows = S;
        a.src_div = 1;
        a.dst = static_cast<uint8_t *>(packed_x);
        a.K = K;
        a.dst_rows = packed_rows;
        a.dst2 = static_cast<uint8_t *>(grp_x);
        a.dst2_rows = max_rows;
        a.gtok_map = gtok_map;
        a.grp_map = grp_tok_map;
        return launch_copy(a, (cudaStream_t)stream);
    }
    a.rows = max_rows;
    a.rows_dev = goff + G;
    if (K < 32) {
        // one pass: each chunk of x[grp_src[r] / K] is staged once and stored
        // to the group row r and to the packed rows of its experts
        a.src = static_cast<const uint8_t *>(x);
        a.src_map = grp_src;
        a.src_div = K;
        a.src_rows = S;
        a.dst = static_cast<uint8_t *>(packed_x);
        a.dst_map = grp_tok_map;
        a.K = K;
        a.dst_rows = packed_rows;
        a.dst2 = static_cast<uint8_t *>(grp_x);
        a.dst2_rows = max_rows;
        return launch_copy(a, (cudaStream_t)stream);
    }
    // K = 32 leaves no lane for the group row: two passes
    // stage 1: one copy of the token per group row
    a.src = static_cast<const uint8_t *>(x);
    a.dst = static_cast<uint8_t *>(grp_x);
    a.K = 1;
    a.src_map = grp_src;
    a.src_div = K;
    a.src_rows = S;
    a.dst_rows = max_rows;
    if (int rc = launch_copy(a, (cudaStream_t)stream)) return rc;
    // stage 2: per-expert expansion out of the group rows
    a.src = static_cast<const uint8_t *>(grp_x);
    a.dst = static_cast<uint8_t *>(packed_x);
    a.K = K;
    a.dst_map = grp_tok_map;
    a.src_map = nullptr;
    a.src_div = 1;
    a.src_rows = max_rows;
    a.dst_rows = packed_rows;
    return launch_copy(a, (cudaStream_t)stream);
}

namespace moe {
namespace {
int launch_quant_wide(const void *x, int64_t S, int64_t H, int K, const int64_t *tok_map,
                      int block, void *packed_q, float *packed_scales, int64_t packed_rows,
                      cudaStream_t stream)
{
    QWideArgs a = {};
    a.x = static_cast<const uint8_t *>(x);
    a.S = S;
    a.H = H;
    a.K = K;
    a.tok_map = tok_map;
    a.dst_rows = packed_rows;
    a.block = block;
    a.nb = H / block;
    a.n_chunks = (int)((H + kQWChunk - 1) / kQWChunk);
    a.q = static_cast<uint8_t *>(packed_q);
    a.sc = packed_scales;
    void (*fn)(QWideArgs) = nullptr;
    static KernelCache caches[5];
    KernelCache *cache = nullptr;
    switch (block) {
    case 16: fn = dispatch_quant_wide_kernel<1>; cache = &caches[0]; break;
    case 32: fn = dispatch_quant_wide_kernel<2>; cache = &caches[1]; break;
    case 64: fn = dispatch_quant_wide_kernel<4>; cache = &caches[2]; break;
    case 128: fn = dispatch_quant_wide_kernel<8>; cache = &caches[3]; break;
    default: fn = dispatch_quant_wide_kernel<16>; cache = &caches[4]; break;
    }
    int per_sm = 0;
    cudaError_t err = prepare_kernel(fn, 0, kQWThreads, *cache, &per_sm);
    if (err != cudaSuccess || per_sm < 1) {
        set_cuda_error(err != cudaSuccess ? err : cudaErrorInvalidConfiguration);
        return MOE_ECUDA;
    }
    const int64_t units = S * a.n_chunks;
    int64_t blocks = (units + kQWWarps - 1) / kQWWarps;
    const int64_t cap = (int64_t)sm_count() * per_sm * MOE_QW_GRID_WAVES;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    err = launch_pdl(fn, dim3((unsigned)blocks), dim3(kQWThreads), 0, stream, a);
    if (err != cudaSuccess) {
        set_cuda_error(err);
        return MOE_ECUDA;
    }
    return check_launch();
}
} // namespace
} // namespace moe

MOE_EXPORT int moe_dispatch_quant_fp8(const void *x, int64_t S, int64_t H, int K,
                                      const int64_t *tok_map, int block, void *packed_q,
                                      float *packed_scales, int64_t packed_rows,
                                      moe_stream_t stream)
{
    MOE_TRACE("moe_dispatch_quant_fp8");
    if (S < 0 || H < 1 || K < 1 || K > 32) return MOE_EINVAL;
    if (block != 16 && block != 32 && block != 64 && block != 128 && block != 256)
        return MOE_EINVAL;
    if (H % block) return MOE_EINVAL;
    if (S == 0) return MOE_OK;
    if (!x || !tok_map || !packed_q || !packed_scales || packed_rows < 1) return MOE_EINVAL;
    if (!aligned16(x) || !aligned16(packed_q) || (reinterpret_cast<uintptr_t>(packed_scales) & 3u))
        return MOE_EALIGN;
    if (H % (4 * block) == 0 && aligned16(packed_scales))
        return launch_quant_wide(x, S, H, K, tok_map, block, packed_q, packed_scales,
                                 packed_rows, (cudaStream_t)stream);
    QuantArgs a = {};
    a.x = static_cast<const uint8_t *>(x);
    a.S = S;
    a.H = H;
    a.K = K;
    a.tok_map = tok_map;
    a.dst_rows = packed_rows;
    a.block = block;
    a.iters = (int)((H + 255) / 256);
    a.slices = (a.iters + kQMaxIters - 1) / kQMaxIters;
    a.R = (a.iters + a.slices - 1) / a.slices;
    a.q = static_cast<uint8_t *>(packed_q);
    a.scales = packed_scales;
    void (*fn)(QuantArgs) = nullptr;
    static KernelCache caches[5];
    KernelCache *cache = nullptr;
    switch (block) {
    case 16: fn = dispatch_quant_kernel<2>; cache = &caches[0]; break;
    case 32: fn = dispatch_quant_kernel<4>; cache = &caches[1]; break;
    case 64: fn = dispatch_quant_kernel<8>; cache = &caches[2]; break;
    case 128: fn = dispatch_quant_kernel<16>; cache = &caches[3]; break;
    default: fn = dispatch_quant_kernel<32>; cache = &caches[4]; break;
    }
    int per_sm = 0;
    cudaError_t err = prepare_kernel(fn, 0, kQThreads, *cache, &per_sm);
    if (err != cudaSuccess || per_sm < 1) {
        set_cuda_error(err != cudaSuccess ? err : cudaErrorInvalidConfiguration);
        return MOE_ECUDA;
    }
    const int64_t units = S * a.slices;
    int64_t blocks = (units + kQThreads / 32 - 1) / (kQThreads / 32);
    const int64_t cap = (int64_t)sm_count() * per_sm;
    if (blocks > cap) blocks = cap;
    err = launch_pdl(fn, dim3((unsigned)blocks), dim3(kQThreads), 0, (cudaStream_t)stream, a);
    if (err != cudaSuccess) {
        set_cuda_error(err);
        return MOE_ECUDA;
    }
    return check_launch();
}

MOE_EXPORT int moe_selftest_wait_timeout(int64_t limit_ns, moe_stream_t stream)
{
    MOE_TRACE("moe_selftest_wait_timeout");
    if (limit_ns < 1000 || limit_ns > 100000000) return MOE_EINVAL;  // 1 us .. 100 ms
    wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_ns);
    return check_launch();
}

namespace moe {
// Reads and clears this file's device error bits.
cudaError_t read_dispatch_errors(uint32_t *flags)
{
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_dispatch_error, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_dispatch_error, &zero, sizeof(uint32_t));
    return e;
}
} // namespace moe
