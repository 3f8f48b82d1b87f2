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

namespace moe {
namespace {

#ifndef MOE_DISPATCH_WARPS
#define MOE_DISPATCH_WARPS 4
#endif
#ifndef MOE_DISPATCH_STAGES
#define MOE_DISPATCH_STAGES 4
#endif
#ifndef MOE_DISPATCH_CHUNK
#define MOE_DISPATCH_CHUNK 4096
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

// Bounded wait for phase `parity` of `bar`; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
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

    griddep_wait();  // earlier stream work (the plan; readers of packed_x) is done
    griddep_launch_dependents();

    const int64_t rows = a.rows_dev ? min(*a.rows_dev, a.rows) : a.rows;
    const int64_t n_items = rows * a.n_chunks;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerCta + warp;
    const int64_t W = (int64_t)gridDim.x * kWarpsPerCta;
    if (gw >= n_items) return;
    // items of this warp: gw + j*W, j = 0 .. n_mine-1
    const int64_t n_mine = (n_items - gw + W - 1) / W;

    int64_t dst_row[kStages];  // this lane's destination row per stage
    int64_t issued = 0;        // items whose load has been issued

    auto issue = [&](int64_t j, int st) {
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
        int64_t d = -1;
        if (a.dst_map) {
            if (lane < a.K) d = __ldg(a.dst_map + r * a.K + lane);
        } else if (lane == 0) {
            d = r;
        }
        if (d >= a.dst_rows || d < -1 || (d >= 0 && !src_ok)) {
            if (d >= a.dst_rows || d < -1) atomicOr(&g_dispatch_error, kErrDispatchIndex);
            d = -1;
        }
        dst_row[st] = d;
    };

    // prologue: fill the ring
#pragma unroll
    for (int st = 0; st < kStages; ++st)
        if (st < n_mine) issue(st, st);

    bool ok = true;
    int64_t consumed = 0;   // items whose load has been waited for
    for (int64_t j0 = 0; j0 < n_mine && ok; j0 += kStages) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) {
            const int64_t j = j0 + st;
            if (j >= n_mine || !ok) break;
            // every lane that stores waits on the barrier itself; the verdict
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
                bulk_s2g(a.dst + d * a.row_bytes + off, stage, bytes);
                if (a.scale_bytes > 0 && c == 0)
                    bulk_s2g(a.sdst + d * a.scale_bytes, stage + a.chunk, a.scale_bytes);
            }
            bulk_commit();
            // refill the stage of item j-1 with item j-1+kStages once the
            // stores reading it have drained
            const int prev = (st + kStages - 1) % kStages;
            const int64_t jn = j - 1 + kStages;
            if (j >= 1 && jn < n_mine) {
                bulk_wait_read<1>();
                __syncwarp();
                issue(jn, prev);
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
    const int64_t cap = (int64_t)sm_count() * per_sm;
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
                            const int64_t *tok_map, void *packed_x, const float *x_scales,
                            int64_t n_scales, float *packed_scales, moe_stream_t stream)
{
    const int es = elem_size(dtype);
    if (es == 0 || S < 0 || H < 1 || K < 1 || K > 32 || n_scales < 0) return MOE_EINVAL;
    if (S == 0) return MOE_OK;
    if (!x || !tok_map || !packed_x) return MOE_EINVAL;
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
    a.dst_rows = S * (int64_t)K;
    a.ssrc = reinterpret_cast<const uint8_t *>(x_scales);
    a.sdst = reinterpret_cast<uint8_t *>(packed_scales);
    a.scale_bytes = (int)(n_scales * 4);
    return launch_copy(a, (cudaStream_t)stream);
}

MOE_EXPORT int moe_dispatch_dedup(const void *x, int64_t S, int64_t H, int dtype, int K, int G,
                                  const int64_t *goff, const int32_t *grp_src,
                                  const int64_t *grp_tok_map, int64_t max_rows, void *grp_x,
                                  void *packed_x, moe_stream_t stream)
{
    const int es = elem_size(dtype);
    if (es == 0 || S < 0 || H < 1 || K < 1 || K > 32 || G < 1 || G > 1024) return MOE_EINVAL;
    if (S == 0) return MOE_OK;
    if (!x || !goff || !grp_src || !grp_tok_map || !grp_x || !packed_x) return MOE_EINVAL;
    if (max_rows < S * (int64_t)(K < G ? K : G)) return MOE_EINVAL;
    const int64_t row_bytes = H * es;
    if (row_bytes % 16 || !aligned16(x) || !aligned16(grp_x) || !aligned16(packed_x))
        return MOE_EALIGN;
    CopyArgs a = {};
    a.row_bytes = row_bytes;
    a.chunk = pick_chunk(row_bytes, &a.n_chunks);
    a.rows = max_rows;
    a.rows_dev = goff + G;
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
    a.dst_rows = S * (int64_t)K;
    return launch_copy(a, (cudaStream_t)stream);
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
