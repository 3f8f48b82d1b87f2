// Combine: gather each token's K expert-output rows, weighted f32 sum.
//
// Sources: ROCm/mori "Draft: cco + flydsl dispatch/combine #448": PR
// description (gather each token's k expert outputs and reduce in f32),
// StdMoE note (convert_combine_input = sum_k wts[k]*packed_x[slot_k]; the
// gather combine then sums over destinations), accumulator note (bf16 and
// f32 inputs widened to f32).  ROCm/mori "EPv2 internode dispatch/combine
// over CCO/GDA", combine note: 16-byte load-first gathers, and warp slices
// sized to whole vector steps so that no warp runs a scalar tail.
//
// GB300 design: the work unit is (output row, slice); a slice is 32 lanes x
// R steps of 8 elements (16 bytes of bf16 or 32 bytes of f32 per k).  A warp
// reads the row's K map entries and weights once (lane k holds entry k,
// shuffled to all lanes), then per step issues all K 16-byte gathers before
// the first add (load first), accumulates in f32 in increasing k with a
// separately rounded multiply and add, and stores the rounded result with
// one 16-byte store.  The grid holds several resident waves of CTAs whose
// warps stride over units (see MOE_COMBINE_GRID_WAVES).  There is no shared
// memory, no atomics and no inter-CTA wait.
//
// Weight fold (mori #448, the note on reducing the K forwarded per-token
// weight vectors into out_weights, folded into the gather at part 0): the
// warp that owns slice 0 of a row also writes out_weights[row, j], the sum of
// w[row, j] over the row's valid copies, from the map entries it already
// holds.

#include "common.cuh"

#include <cuda_bf16.h>

namespace moe {
namespace {

#ifndef MOE_COMBINE_THREADS
#define MOE_COMBINE_THREADS 128
#endif
constexpr int kThreads = MOE_COMBINE_THREADS;
constexpr int kKChunk = 8;   // map entries held in registers at a time
#ifndef MOE_COMBINE_LANE_STEPS
#define MOE_COMBINE_LANE_STEPS 4
#endif
constexpr int kMaxLaneSteps = MOE_COMBINE_LANE_STEPS;  // 8-element steps per lane per unit
// Grid size in resident waves (CTAs per SM x SMs x waves).  SMs of this part
// do not move data at the same rate (per-SM times of one equal share measured
// 51 to 82 us in the dispatch, the same SMs slow on every launch), so a grid
// of several waves of short CTAs, which the block scheduler hands to
// whichever SM frees up, beats a persistent grid whose warps stride over a
// fixed share: at S=4096 H=7168 K=8 the combine inside the step (after the
// dispatch) went 92.9 -> 90.1 us and the step 181.8 -> 179.4 us, for 74.7 ->
// 77.9 us when timed alone.  Handing the units out through a global counter
// instead measured slower (atomic latency under the write traffic).
#ifndef MOE_COMBINE_GRID_WAVES
#define MOE_COMBINE_GRID_WAVES 8
#endif

enum WMode { kWeightDirect = 0, kWeightViaSrc = 1, kUnweighted = 2 };

__device__ uint32_t g_combine_error;  // kErrCombineIndex

struct CombineArgs {
    const uint8_t *y;          // input rows
    const float *w;            // [*, K] weights (unless unweighted)
    const int32_t *wsrc;       // kWeightViaSrc: weight row = wsrc[i] / K
    const int64_t *map;        // [rows, K] input row or -1
    int64_t rows;              // output rows (host bound)
    const int64_t *rows_dev;   // if set: rows = min(*rows_dev, rows)
    int64_t y_rows;            // rows of y (bounds check)
    int64_t w_rows;            // rows of w (bounds check, kWeightViaSrc)
    int K;
    int64_t H;                 // elements per row (multiple of 8)
    int64_t steps;             // H / 8
    int R;                     // steps per lane per unit
    int slices;                // units per row
    uint8_t *out;
    float *out_w;              // if set: [rows, K] weight fold (reads w[i, *])
};

// Element layout of a lane-step.  A warp-step covers 256 consecutive
// elements (32 lanes x 8).  Contiguous layout: lane l owns elements
// 8l..8l+7.  Quad layout (used when a row holds f32, input or output, and the
// warp-step is whole): lane l owns 4l..4l+3 and 128+4l..128+4l+3, so that
// each 16-byte f32 access of the warp covers 512 contiguous bytes and no
// 32-byte sector is split between two instructions.  p is the lane-step
// index (warp-step p >> 5, lane p & 31); f[0..3] and f[4..7] are the two
// halves in element order.
template <typename T> struct Io;

template <> struct Io<__nv_bfloat16> {
    static constexpr int kVec = 1;  // 16-byte vectors per 8 elements
    __device__ __forceinline__ static void load(uint4 (&v)[1], const uint8_t *row, int64_t p,
                                                bool quad)
    {
        if (!quad) {
            v[0] = ld_stream16(row + p * 16);
        } else {
            const int64_t base = (p >> 5) * 512 + (p & 31) * 8;
            const uint2 a = ld_stream8(row + base);
            const uint2 b = ld_stream8(row + base + 256);
            v[0] = make_uint4(a.x, a.y, b.x, b.y);
        }
    }
    __device__ __forceinline__ static void widen(const uint4 (&v)[1], float (&f)[8])
    {
        const uint32_t u[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            f[2 * q] = __uint_as_float(u[q] << 16);
            f[2 * q + 1] = __uint_as_float(u[q] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static void store(uint8_t *out_row, int64_t p, const float (&f)[8],
                                                 bool quad)
    {
        uint32_t u[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * q], f[2 * q + 1]);  // RNE
            u[q] = *reinterpret_cast<uint32_t *>(&b);
        }
        if (!quad) {
            st16(out_row + p * 16, make_uint4(u[0], u[1], u[2], u[3]));
        } else {
            const int64_t base = (p >> 5) * 512 + (p & 31) * 8;
            st8(out_row + base, make_uint2(u[0], u[1]));
            st8(out_row + base + 256, make_uint2(u[2], u[3]));
        }
    }
};

template <> struct Io<float> {
    static constexpr int kVec = 2;
    __device__ __forceinline__ static void load(uint4 (&v)[2], const uint8_t *row, int64_t p,
                                                bool quad)
    {
        if (!quad) {
            v[0] = ld_stream16(row + p * 32);
            v[1] = ld_stream16(row + p * 32 + 16);
        } else {
            const int64_t base = (p >> 5) * 1024 + (p & 31) * 16;
            v[0] = ld_stream16(row + base);
            v[1] = ld_stream16(row + base + 512);
        }
    }
    __device__ __forceinline__ static void widen(const uint4 (&v)[2], float (&f)[8])
    {
        f[0] = __uint_as_float(v[0].x); f[1] = __uint_as_float(v[0].y);
        f[2] = __uint_as_float(v[0].z); f[3] = __uint_as_float(v[0].w);
        f[4] = __uint_as_float(v[1].x); f[5] = __uint_as_float(v[1].y);
        f[6] = __uint_as_float(v[1].z); f[7] = __uint_as_float(v[1].w);
    }
    __device__ __forceinline__ static void store(uint8_t *out_row, int64_t p, const float (&f)[8],
                                                 bool quad)
    {
        const uint4 a = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                                   __float_as_uint(f[2]), __float_as_uint(f[3]));
        const uint4 b = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]),
                                   __float_as_uint(f[6]), __float_as_uint(f[7]));
        if (!quad) {
            st16(out_row + p * 32, a);
            st16(out_row + p * 32 + 16, b);
        } else {
            const int64_t base = (p >> 5) * 1024 + (p & 31) * 16;
            st16(out_row + base, a);
            st16(out_row + base + 512, b);
        }
    }
};

// Register budgets are set as resident threads per SM, whatever the CTA
// size: 512 for the general kernel (<= 128 registers), 640 for the lean one
// (<= 102); the dedup kernel's are set by input type, below.  128-thread CTAs fit more warps per SM than
// 256-thread ones at the same budget: the combine at the MoonEP shape went
// 77.8 -> 75.7 us alone and 90.2 -> 89.3 us inside the step with seven lean
// CTAs of 72 registers (28 warps) against three of 256 threads.
#ifndef MOE_COMBINE_MIN_BLOCKS
#define MOE_COMBINE_MIN_BLOCKS (512 / MOE_COMBINE_THREADS)
#endif
template <typename Tin, typename Tout, int WM>
__global__ void __launch_bounds__(kThreads, MOE_COMBINE_MIN_BLOCKS) combine_kernel(CombineArgs a)
{
    griddep_wait();  // y, map, weights come from earlier stream work
    griddep_launch_dependents();

    constexpr bool kQuad = sizeof(Tin) == 4 || sizeof(Tout) == 4;
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t W = ((int64_t)gridDim.x * kThreads) >> 5;
    const int64_t rows = a.rows_dev ? min(*a.rows_dev, a.rows) : a.rows;
    const int64_t units = rows * a.slices;
    const int K = a.K;
    constexpr int kInBytes = (int)sizeof(Tin) * 8;    // bytes of 8 input elements
    constexpr int kOutBytes = (int)sizeof(Tout) * 8;
    const int64_t in_row_bytes = a.steps * kInBytes;
    const int64_t out_row_bytes = a.steps * kOutBytes;

    for (int64_t u = gw; u < units; u += W) {
        const int64_t i = u / a.slices;
        const int sl = (int)(u - i * a.slices);
        // this lane's map entry and weight (lane k <-> entry k)
        int32_t my_row = -1;  // rows of y are below 2^31 (S*K < 2^31)
        float my_w = 1.0f;
        if (lane < K) {
            const int64_t r = __ldg(a.map + i * K + lane);
            my_row = (r >= 0 && r < a.y_rows) ? (int32_t)r : (r == -1 ? -1 : -2);
            int64_t wr = i;
            if (WM == kWeightViaSrc) wr = (int64_t)(__ldg(a.wsrc + i) / K);
            const bool ok = my_row >= -1 && (WM != kWeightViaSrc || (wr >= 0 && wr < a.w_rows));
            if (!ok) {
                // never gather outside the buffers: drop the term and report
                atomicOr(&g_combine_error, kErrCombineIndex);
                my_row = -1;
            } else if (WM != kUnweighted && my_row >= 0) {
                my_w = __ldg(a.w + wr * K + lane);
            }
        }
        if (a.out_w != nullptr && sl == 0) {
            // weight fold: the token's weight vector travels with each of its
            // valid copies, so entry j accumulates w[i, j] once per copy
            const unsigned valid = __ballot_sync(0xffffffffu, lane < K && my_row >= 0);
            if (lane < K) {
                const float fw = __ldg(a.w + i * K + lane);
                float acc = 0.0f;
                for (int c = __popc(valid); c > 0; --c) acc = __fadd_rn(acc, fw);
                a.out_w[i * K + lane] = acc;
            }
        }
        const int64_t pbase = (int64_t)sl * 32 * a.R;
        uint8_t *out_row = a.out + i * out_row_bytes;

        // the trip count is the same for every lane (shuffles below need the
        // whole warp); lanes past the end of the row are predicated off
        for (int r = 0; r < a.R; ++r) {
            const int64_t p = pbase + (int64_t)r * 32 + lane;
            const bool active = p < a.steps;
            // quad layout when f32 is involved and the warp-step is whole
            // (the same for every lane: pbase is a multiple of 32)
            const bool quad = kQuad && (((p >> 5) + 1) << 5) <= a.steps;
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
            for (int k0 = 0; k0 < K; k0 += kKChunk) {
                // load first: every gather of this chunk of k is in flight
                // before the first add
                uint4 v[kKChunk][Io<Tin>::kVec];
                int32_t rk[kKChunk];
#pragma unroll
                for (int kk = 0; kk < kKChunk; ++kk) {
                    rk[kk] = __shfl_sync(0xffffffffu, my_row, (k0 + kk) & 31);
                    if (active && k0 + kk < K && rk[kk] >= 0)
                        Io<Tin>::load(v[kk], a.y + (int64_t)rk[kk] * in_row_bytes, p, quad);
                }
#pragma unroll
                for (int kk = 0; kk < kKChunk; ++kk) {
                    const float wk = __shfl_sync(0xffffffffu, my_w, (k0 + kk) & 31);
                    if (active && k0 + kk < K && rk[kk] >= 0) {
                        float f[8];
                        Io<Tin>::widen(v[kk], f);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            if (WM == kUnweighted)
                                acc[q] = __fadd_rn(acc[q], f[q]);
                            else
                                acc[q] = __fadd_rn(acc[q], __fmul_rn(wk, f[q]));
                        }
                    }
                }
            }
            if (active) Io<Tout>::store(out_row, p, acc, quad);
        }
    }
}

// ---------------------------------------------------------------------------
// The same sum for the common case -- bf16 rows in and out, weights per
// output row or none, K <= 8, with or without the weight fold -- written so
// that more gathers are in flight per SM: per unit the lanes keep one row
// pointer each (shuffled to the warp when a step issues its loads) and one
// ballot of the valid entries instead of K row indices, and each 32-bit word
// of a gathered vector is widened and added in place.  A lane gathers two
// steps at once (2 x K 16-byte loads in flight before the first add), which
// costs 96 registers; five 128-thread CTAs (20 warps) then hold 160 KB of
// gathers per SM, against 112 KB for one step at a time with 28 warps of 72
// registers.  The combine of 4096 rows of 7168 bf16 from K = 8 gathered
// rows: 90 us on the general kernel, 75.5 us one step at a time, 71.9 us
// two steps at a time (85.0 against 89.1 us inside the step).  The order of
// operations on every element is the kernel's above, for every mode.
// ---------------------------------------------------------------------------

#ifndef MOE_COMBINE_LEAN
#define MOE_COMBINE_LEAN 1
#endif
#ifndef MOE_COMBINE_LEAN_MIN_BLOCKS
#define MOE_COMBINE_LEAN_MIN_BLOCKS (640 / MOE_COMBINE_THREADS)
#endif

template <bool kWeighted, bool kFold>
__global__ void __launch_bounds__(kThreads, MOE_COMBINE_LEAN_MIN_BLOCKS)
combine_lean_kernel(CombineArgs a)
{
    griddep_wait();  // y, map, weights come from earlier stream work
    griddep_launch_dependents();

    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t W = ((int64_t)gridDim.x * kThreads) >> 5;
    const int64_t units = a.rows * a.slices;
    const int K = a.K;
    const int64_t row_bytes = a.steps * 16;  // bf16 rows, in and out

    for (int64_t u = gw; u < units; u += W) {
        const int64_t i = u / a.slices;
        const int sl = (int)(u - i * a.slices);
        const uint8_t *base = a.y;  // this lane's y row (lane k <-> entry k)
        float w = 0.0f;
        bool valid = false;
        if (lane < K) {
            const int64_t r = __ldg(a.map + i * K + lane);
            if (r >= 0 && r < a.y_rows) {
                valid = true;
                base = a.y + r * row_bytes;
                if (kWeighted) w = __ldg(a.w + i * K + lane);
            } else if (r != -1) {
                atomicOr(&g_combine_error, kErrCombineIndex);  // dropped, never gathered
            }
        }
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        if (kFold && sl == 0 && lane < K) {
            // weight fold: the token's weight vector travels with each of its
            // valid copies, so entry j accumulates w[i, j] once per copy
            const float fw = __ldg(a.w + i * K + lane);
            float acc = 0.0f;
            for (int c = __popc(vmask); c > 0; --c) acc = __fadd_rn(acc, fw);
            a.out_w[i * K + lane] = acc;
        }
        const int64_t pbase = (int64_t)sl * 32 * a.R;
        uint8_t *out_row = a.out + i * row_bytes;
        for (int r = 0; r < a.R; r += 2) {
            const int64_t p0 = pbase + (int64_t)r * 32 + lane;
            const int64_t p1 = p0 + 32;
            const bool act0 = p0 < a.steps;
            const bool act1 = r + 1 < a.R && p1 < a.steps;
            uint4 v0[kKChunk], v1[kKChunk];
#pragma unroll
            for (int k = 0; k < kKChunk; ++k) {
                const uint8_t *bk = reinterpret_cast<const uint8_t *>(
                    __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(base), k));
                if ((vmask >> k) & 1u) {
                    if (act0) v0[k] = ld_stream16(bk + p0 * 16);
                    if (act1) v1[k] = ld_stream16(bk + p1 * 16);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const bool active = h ? act1 : act0;
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
                for (int k = 0; k < kKChunk; ++k) {
                    const float wk = kWeighted ? __shfl_sync(0xffffffffu, w, k) : 1.0f;
                    if (active && ((vmask >> k) & 1u)) {
                        const uint4 vk = h ? v1[k] : v0[k];
                        const uint32_t q[4] = {vk.x, vk.y, vk.z, vk.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float lo = __uint_as_float(q[e] << 16);
                            const float hi = __uint_as_float(q[e] & 0xffff0000u);
                            if (kWeighted) {
                                acc[2 * e] = __fadd_rn(acc[2 * e], __fmul_rn(wk, lo));
                                acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], __fmul_rn(wk, hi));
                            } else {
                                acc[2 * e] = __fadd_rn(acc[2 * e], lo);
                                acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], hi);
                            }
                        }
                    }
                }
                if (active) Io<__nv_bfloat16>::store(out_row, h ? p1 : p0, acc, false);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Dedup combine in one pass (K <= kKChunk).  The work unit is (token s,
// slice).  Lane k holds the token's group-row entry gtok_map[s,k] (set for the
// first entry of each group: the representatives, in increasing k) and, after
// one load per representative, the y row of its own entry and the index of
// the representative whose group it is in.  Per step all of the token's
// gathers are issued first; then, representative by representative in k
// order, the group row's weighted sum is formed in increasing k (exactly the
// first stage), stored to gtok, and added to the token's sum (exactly the
// second stage), so gtok is written but never read back.  The weights come
// from the token's own row, which is grp_src[r] / K for every group row r of
// the token in a plan from moe_group_plan.
// ---------------------------------------------------------------------------

struct DedupArgs {
    const uint8_t *y;          // expert outputs [y_rows, H]
    int64_t y_rows;
    const float *w;            // [S, K]
    const int64_t *gtok_map;   // [S, K]
    const int64_t *grp_tok_map;  // [max_rows, K]
    int64_t max_rows;
    int64_t S;
    int K;
    int64_t steps;             // H / 8
    int R, slices;
    float *gtok;               // [max_rows, H] f32
    uint8_t *out;              // [S, H]
};

// Register budgets of the dedup kernel as resident threads per SM, by input
// type.  Each entry's row, representative and weight stay in its lane and
// are shuffled out where used instead of being held per lane for all K
// entries (117 -> 96 registers with f32 rows, 121 -> 72 with bf16 rows): at
// S=4096 K=8 in 8 groups, f32 rows of 4096 154.5 -> 153.3 us (five CTAs per
// SM; six spill, 171.7 us), bf16 rows of 7168 with f32 group rows 207.6 ->
// 178.5 us (six or seven CTAs per SM, 72 registers either way).
#ifndef MOE_DEDUP_THREADS_F32
#define MOE_DEDUP_THREADS_F32 640
#endif
#ifndef MOE_DEDUP_THREADS_BF16
#define MOE_DEDUP_THREADS_BF16 768
#endif

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads, (sizeof(Tin) == 4 ? MOE_DEDUP_THREADS_F32
                                                               : MOE_DEDUP_THREADS_BF16) / kThreads)
combine_dedup_kernel(DedupArgs a)
{
    griddep_wait();
    griddep_launch_dependents();

    constexpr bool kQuad = sizeof(Tin) == 4 || sizeof(Tout) == 4;
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t W = ((int64_t)gridDim.x * kThreads) >> 5;
    const int64_t units = a.S * a.slices;
    const int K = a.K;
    constexpr int kInBytes = (int)sizeof(Tin) * 8;
    constexpr int kOutBytes = (int)sizeof(Tout) * 8;
    const int64_t in_row_bytes = a.steps * kInBytes;
    const int64_t out_row_bytes = a.steps * kOutBytes;
    const int64_t g_row_bytes = a.steps * 32;  // gtok rows are f32

    for (int64_t u = gw; u < units; u += W) {
        const int64_t s = u / a.slices;
        const int sl = (int)(u - s * a.slices);
        // lane k: the token's group-row entry (representatives only)
        int64_t gk = -1;
        if (lane < K) {
            gk = __ldg(a.gtok_map + s * K + lane);
            if (gk < -1 || gk >= a.max_rows) {
                atomicOr(&g_combine_error, kErrCombineIndex);
                gk = -1;
            }
        }
        const unsigned reps = __ballot_sync(0xffffffffu, gk >= 0);
        // lane k: its y row and the rank of its representative (k order)
        int32_t my_row = -1;
        int my_rep = -1;
        {
            unsigned m = reps;
            for (int j = 0; m; ++j, m &= m - 1) {
                const int q = __ffs(m) - 1;
                const int64_t rq = __shfl_sync(0xffffffffu, gk, q);
                if (lane < K) {
                    const int64_t e = __ldg(a.grp_tok_map + rq * K + lane);
                    if (e >= 0 && e < a.y_rows) {
                        my_row = (int32_t)e;
                        my_rep = j;
                    } else if (e != -1) {
                        atomicOr(&g_combine_error, kErrCombineIndex);
                    }
                }
            }
        }
        const float my_w = (lane < K && my_row >= 0) ? __ldg(a.w + s * K + lane) : 0.0f;
        // entry k's representative rank in nibble k (15: entry unused); its
        // row and weight stay in lane k and are shuffled out where used
        uint32_t jmask = 0;
#pragma unroll
        for (int kk = 0; kk < kKChunk; ++kk) {
            const int j = __shfl_sync(0xffffffffu, my_rep, kk);
            jmask |= (uint32_t)((kk < K && j >= 0) ? j : 15) << (4 * kk);
        }
        const int n_reps = __popc(reps);
        const int64_t pbase = (int64_t)sl * 32 * a.R;
        uint8_t *out_row = a.out + s * out_row_bytes;

        for (int r = 0; r < a.R; ++r) {
            const int64_t p = pbase + (int64_t)r * 32 + lane;
            const bool active = p < a.steps;
            const bool quad = kQuad && (((p >> 5) + 1) << 5) <= a.steps;
            uint4 v[kKChunk][Io<Tin>::kVec];
#pragma unroll
            for (int kk = 0; kk < kKChunk; ++kk) {
                const int32_t rr = __shfl_sync(0xffffffffu, my_row, kk);
                if (active && ((jmask >> (4 * kk)) & 15u) != 15u)
                    Io<Tin>::load(v[kk], a.y + (int64_t)rr * in_row_bytes, p, quad);
            }
            float tot[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) tot[q] = 0.0f;
            unsigned m = reps;
            for (int j = 0; j < n_reps; ++j, m &= m - 1) {
                const int64_t rq = __shfl_sync(0xffffffffu, gk, __ffs(m) - 1);
                float acc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
                for (int kk = 0; kk < kKChunk; ++kk) {
                    if (((jmask >> (4 * kk)) & 15u) == (uint32_t)j) {  // warp-uniform
                        const float wk = __shfl_sync(0xffffffffu, my_w, kk);
                        if (active) {
                            float f[8];
                            Io<Tin>::widen(v[kk], f);
#pragma unroll
                            for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], __fmul_rn(wk, f[q]));
                        }
                    }
                }
                if (active) {
                    Io<float>::store(reinterpret_cast<uint8_t *>(a.gtok) + rq * g_row_bytes, p, acc,
                                     quad);
#pragma unroll
                    for (int q = 0; q < 8; ++q) tot[q] = __fadd_rn(tot[q], acc[q]);
                }
            }
            if (active) Io<Tout>::store(out_row, p, tot, quad);
        }
    }
}

template <typename Tin, typename Tout>
void (*pick_kernel(int wm))(CombineArgs)
{
    switch (wm) {
    case kWeightDirect: return combine_kernel<Tin, Tout, kWeightDirect>;
    case kWeightViaSrc: return combine_kernel<Tin, Tout, kWeightViaSrc>;
    default: return combine_kernel<Tin, Tout, kUnweighted>;
    }
}

void (*select_kernel(int in_dt, int out_dt, int wm))(CombineArgs)
{
    if (in_dt == MOE_BF16 && out_dt == MOE_BF16) return pick_kernel<__nv_bfloat16, __nv_bfloat16>(wm);
    if (in_dt == MOE_BF16 && out_dt == MOE_F32) return pick_kernel<__nv_bfloat16, float>(wm);
    if (in_dt == MOE_F32 && out_dt == MOE_BF16) return pick_kernel<float, __nv_bfloat16>(wm);
    if (in_dt == MOE_F32 && out_dt == MOE_F32) return pick_kernel<float, float>(wm);
    return nullptr;
}

// Slices per row and steps per lane for a grid of `warp_slots` warps.
void set_slices(CombineArgs &a, int64_t warp_slots)
{
    // slices: at most kMaxLaneSteps steps per lane per unit, slices of equal
    // size; finer units even out the work of the warps.  When the
    // rows cannot fill every warp of the grid (small batches), rows are cut
    // finer, down to one step per lane, so that more gathers are in flight
    // at once; the summation order of an element never depends on this.
    const int64_t lane_steps = (a.steps + 31) / 32;
    int64_t slices = (lane_steps + kMaxLaneSteps - 1) / kMaxLaneSteps;
    if (a.rows * slices < warp_slots) {
        const int64_t want = (warp_slots + a.rows - 1) / a.rows;
        slices = want < lane_steps ? want : lane_steps;
    }
    a.R = (int)((lane_steps + slices - 1) / slices);
    a.slices = (int)((lane_steps + a.R - 1) / a.R);
}

int launch_combine(CombineArgs &a, int in_dt, int out_dt, int wm, cudaStream_t stream)
{
    void (*fn)(CombineArgs) = select_kernel(in_dt, out_dt, wm);
    if (!fn) return MOE_EINVAL;
    // one cache per (input, output, weight-mode) kernel, one per lean one
    static KernelCache caches[2][2][3];
    static KernelCache lean_cache[2][2];
    KernelCache *cp = &caches[in_dt == MOE_F32][out_dt == MOE_F32][wm];
    if (MOE_COMBINE_LEAN && in_dt == MOE_BF16 && out_dt == MOE_BF16 &&
        (wm == kWeightDirect || wm == kUnweighted) && a.K <= kKChunk && !a.rows_dev) {
        const bool weighted = wm == kWeightDirect, fold = a.out_w != nullptr;
        fn = weighted ? (fold ? combine_lean_kernel<true, true> : combine_lean_kernel<true, false>)
                      : (fold ? combine_lean_kernel<false, true> : combine_lean_kernel<false, false>);
        cp = &lean_cache[weighted][fold];
    }
    KernelCache &cache = *cp;
    int per_sm = 0;
    cudaError_t err = prepare_kernel(fn, 0, kThreads, cache, &per_sm);
    if (err != cudaSuccess || per_sm < 1) {
        set_cuda_error(err != cudaSuccess ? err : cudaErrorInvalidConfiguration);
        return MOE_ECUDA;
    }
    set_slices(a, (int64_t)sm_count() * per_sm * (kThreads / 32));
    const int64_t units = a.rows * a.slices;
    int64_t blocks = (units + kThreads / 32 - 1) / (kThreads / 32);
    const int64_t cap = (int64_t)sm_count() * per_sm * MOE_COMBINE_GRID_WAVES;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    err = launch_pdl(fn, dim3((unsigned)blocks), dim3(kThreads), 0, stream, a);
    if (err != cudaSuccess) {
        set_cuda_error(err);
        return MOE_ECUDA;
    }
    return check_launch();
}

bool combine_dtype_ok(int dt) { return dt == MOE_BF16 || dt == MOE_F32; }

int launch_dedup(DedupArgs &d, int in_dt, int out_dt, cudaStream_t stream)
{
    void (*fn)(DedupArgs) = nullptr;
    if (in_dt == MOE_BF16 && out_dt == MOE_BF16) fn = combine_dedup_kernel<__nv_bfloat16, __nv_bfloat16>;
    if (in_dt == MOE_BF16 && out_dt == MOE_F32) fn = combine_dedup_kernel<__nv_bfloat16, float>;
    if (in_dt == MOE_F32 && out_dt == MOE_BF16) fn = combine_dedup_kernel<float, __nv_bfloat16>;
    if (in_dt == MOE_F32 && out_dt == MOE_F32) fn = combine_dedup_kernel<float, float>;
    if (!fn) return MOE_EINVAL;
    static KernelCache caches[2][2];
    KernelCache &cache = caches[in_dt == MOE_F32][out_dt == MOE_F32];
    int per_sm = 0;
    cudaError_t err = prepare_kernel(fn, 0, kThreads, cache, &per_sm);
    if (err != cudaSuccess || per_sm < 1) {
        set_cuda_error(err != cudaSuccess ? err : cudaErrorInvalidConfiguration);
        return MOE_ECUDA;
    }
    CombineArgs geo = {};
    geo.rows = d.S;
    geo.steps = d.steps;
    set_slices(geo, (int64_t)sm_count() * per_sm * (kThreads / 32));
    d.R = geo.R;
    d.slices = geo.slices;
    const int64_t units = d.S * d.slices;
    int64_t blocks = (units + kThreads / 32 - 1) / (kThreads / 32);
    const int64_t cap = (int64_t)sm_count() * per_sm * MOE_COMBINE_GRID_WAVES;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    err = launch_pdl(fn, dim3((unsigned)blocks), dim3(kThreads), 0, stream, d);
    if (err != cudaSuccess) {
        set_cuda_error(err);
        return MOE_ECUDA;
    }
    return check_launch();
}

} // namespace
} // namespace moe

using namespace moe;

MOE_EXPORT int moe_combine(const void *y, int64_t y_rows, int in_dtype, const float *topk_w,
                           const int64_t *tok_map, int64_t S, int64_t H, int K, void *out,
                           int out_dtype, moe_stream_t stream)
{
    MOE_TRACE("moe_combine");
    if (!combine_dtype_ok(in_dtype) || !combine_dtype_ok(out_dtype)) return MOE_EINVAL;
    if (S < 0 || H < 1 || K < 1 || K > 32) return MOE_EINVAL;
    if (S == 0) return MOE_OK;
    if (!y || !topk_w || !tok_map || !out || y_rows < 1 || y_rows >= ((int64_t)1 << 31))
        return MOE_EINVAL;
    if (H % 8 || !aligned16(y) || !aligned16(out)) return MOE_EALIGN;
    CombineArgs a = {};
    a.y = static_cast<const uint8_t *>(y);
    a.w = topk_w;
    a.map = tok_map;
    a.rows = S;
    a.y_rows = y_rows;
    a.K = K;
    a.H = H;
    a.steps = H / 8;
    a.out = static_cast<uint8_t *>(out);
    return launch_combine(a, in_dtype, out_dtype, kWeightDirect, (cudaStream_t)stream);
}

MOE_EXPORT int moe_combine_dedup(const void *y, int64_t y_rows, int in_dtype,
                                 const float *topk_w, const int64_t *goff, int G,
                                 const int32_t *grp_src, const int64_t *grp_tok_map,
                                 const int64_t *gtok_map, int64_t S, int64_t H, int K,
                                 int64_t max_rows, float *gtok, void *out, int out_dtype,
                                 moe_stream_t stream)
{
    MOE_TRACE("moe_combine_dedup");
    if (!combine_dtype_ok(in_dtype) || !combine_dtype_ok(out_dtype)) return MOE_EINVAL;
    if (S < 0 || H < 1 || K < 1 || K > 32 || G < 1 || G > 1024) return MOE_EINVAL;
    if (S == 0) return MOE_OK;
    if (!y || !topk_w || !goff || !grp_src || !grp_tok_map || !gtok_map || !gtok || !out ||
        y_rows < 1 || y_rows >= ((int64_t)1 << 31))
        return MOE_EINVAL;
    if (max_rows < S * (int64_t)(K < G ? K : G)) return MOE_EINVAL;
    if (H % 8 || !aligned16(y) || !aligned16(out) || !aligned16(gtok)) return MOE_EALIGN;
    if (K <= kKChunk) {
        DedupArgs d = {};
        d.y = static_cast<const uint8_t *>(y);
        d.y_rows = y_rows;
        d.w = topk_w;
        d.gtok_map = gtok_map;
        d.grp_tok_map = grp_tok_map;
        d.max_rows = max_rows;
        d.S = S;
        d.K = K;
        d.steps = H / 8;
        d.gtok = gtok;
        d.out = static_cast<uint8_t *>(out);
        return launch_dedup(d, in_dtype, out_dtype, (cudaStream_t)stream);
    }
    // K > kKChunk: two passes
    // stage 1: per group row, weighted sum of its experts' outputs (f32)
    CombineArgs a = {};
    a.y = static_cast<const uint8_t *>(y);
    a.w = topk_w;
    a.wsrc = grp_src;
    a.map = grp_tok_map;
    a.rows = max_rows;
    a.rows_dev = goff + G;
    a.y_rows = y_rows;
    a.w_rows = S;
    a.K = K;
    a.H = H;
    a.steps = H / 8;
    a.out = reinterpret_cast<uint8_t *>(gtok);
    if (int rc = launch_combine(a, in_dtype, MOE_F32, kWeightViaSrc, (cudaStream_t)stream))
        return rc;
    // stage 2: per token, unweighted sum of its group rows
    CombineArgs b = {};
    b.y = reinterpret_cast<const uint8_t *>(gtok);
    b.map = gtok_map;
    b.rows = S;
    b.y_rows = max_rows;
    b.K = K;
    b.H = H;
    b.steps = H / 8;
    b.out = static_cast<uint8_t *>(out);
    return launch_combine(b, MOE_F32, out_dtype, kUnweighted, (cudaStream_t)stream);
}

MOE_EXPORT int moe_combine_fold(const void *y, int64_t y_rows, int in_dtype,
                                const float *topk_w, int weighted, const int64_t *map, int64_t S,
                                int64_t H, int K, void *out, int out_dtype, float *out_weights,
                                moe_stream_t stream)
{
    MOE_TRACE("moe_combine_fold");
    if (!combine_dtype_ok(in_dtype) || !combine_dtype_ok(out_dtype)) return MOE_EINVAL;
    if (S < 0 || H < 1 || K < 1 || K > 32 || (weighted != 0 && weighted != 1)) return MOE_EINVAL;
    if (S == 0) return MOE_OK;
    if (!y || !map || !out || y_rows < 1 || y_rows >= ((int64_t)1 << 31)) return MOE_EINVAL;
    if ((weighted || out_weights) && !topk_w) return MOE_EINVAL;
    if (H % 8 || !aligned16(y) || !aligned16(out)) return MOE_EALIGN;
    if (out_weights && (reinterpret_cast<uintptr_t>(out_weights) & 3)) return MOE_EALIGN;
    CombineArgs a = {};
    a.y = static_cast<const uint8_t *>(y);
    a.w = topk_w;
    a.map = map;
    a.rows = S;
    a.y_rows = y_rows;
    a.K = K;
    a.H = H;
    a.steps = H / 8;
    a.out = static_cast<uint8_t *>(out);
    a.out_w = out_weights;
    return launch_combine(a, in_dtype, out_dtype, weighted ? kWeightDirect : kUnweighted,
                          (cudaStream_t)stream);
}

namespace moe {
// Reads and clears this file's device error bits.
cudaError_t read_combine_errors(uint32_t *flags)
{
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_combine_error, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_combine_error, &zero, sizeof(uint32_t));
    return e;
}
} // namespace moe
