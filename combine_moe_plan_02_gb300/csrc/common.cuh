// Shared device and host helpers of the sm_103a MoE dispatch/combine library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_plan.h"

#ifndef MOE_NVTX
#define MOE_NVTX 1
#endif
#if MOE_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

#define MOE_EXPORT extern "C" __attribute__((visibility("default")))

namespace moe {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Remembers the CUDA error behind the last MOE_ECUDA on this host thread.
void set_cuda_error(cudaError_t e);

// A host-side NVTX range around one ABI call, named after the call, so that
// profilers can attribute the kernels it enqueues (nsys timelines, ncu
// --nvtx filters).  Header-only NVTX: without a tool attached, a push and a
// pop cost a few nanoseconds and load nothing.
struct TraceRange {
    explicit TraceRange(const char *name)
    {
#if MOE_NVTX
        nvtxRangePushA(name);
#else
        (void)name;
#endif
    }
    ~TraceRange()
    {
#if MOE_NVTX
        nvtxRangePop();
#endif
    }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};
#define MOE_TRACE(name) ::moe::TraceRange moe_trace_range_(name)

// Returns MOE_ECUDA (recording the error) if the last launch failed.
inline int check_launch()
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return MOE_ECUDA;
    }
    return MOE_OK;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int elem_size(int dtype)
{
    switch (dtype) {
    case MOE_BF16: return 2;
    case MOE_F32: return 4;
    case MOE_FP8_E4M3: return 1;
    default: return 0;
    }
}

// Device error bits, reported by moe_device_errors().
enum : uint32_t {
    kErrDispatchTimeout = 1u,  // a bounded wait for a staged row ran out of time
    kErrDispatchIndex = 2u,    // dispatch met a row index outside its buffers
    kErrCombineIndex = 4u,     // combine met a row index outside its buffers
    kErrCombineTimeout = 8u,   // a bounded wait for staged rows in combine ran out of time
};
cudaError_t read_dispatch_errors(uint32_t *flags);
cudaError_t read_combine_errors(uint32_t *flags);
cudaError_t read_plan_dispatch_errors(uint32_t *flags);

// moe_dispatch's body; early_src: the source rows were complete before the
// previous kernel of the stream started waiting (see CopyArgs::early_src).
int dispatch_rows(const void *x, int64_t S, int64_t H, int dtype, int K, const int64_t *tok_map,
                  void *packed_x, int64_t packed_rows, const float *x_scales, int64_t n_scales,
                  float *packed_scales, bool early_src, cudaStream_t stream);

// Number of SMs of the current device (cached per device ordinal).
int sm_count();

// Per-device launch facts of one kernel, filled on first use.  Raising a
// kernel's dynamic shared-memory limit can wait for the device, so it is done
// once per device and size, never per launch; the occupancy query is cached
// by size too.  Races between host threads only repeat a query.
constexpr int kMaxCachedDevices = 64;
struct KernelCache {
    int smem_limit[kMaxCachedDevices];  // dynamic smem limit already set
    int occ_smem[kMaxCachedDevices];    // smem of the cached occupancy + 1 (0 = none)
    int occ[kMaxCachedDevices];         // resident CTAs per SM at occ_smem - 1
};

// Makes `fn` launchable with `smem` bytes of dynamic shared memory and, if
// per_sm is given, returns its resident CTAs per SM at that size.
template <typename F>
cudaError_t prepare_kernel(F fn, size_t smem, int threads, KernelCache &kc, int *per_sm)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < kMaxCachedDevices;
    // set whenever dynamic memory is used: static shared memory counts
    // against the same 48 KB default
    if (smem > 0 && (!cached || kc.smem_limit[dev] < (int)smem)) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (cached) kc.smem_limit[dev] = (int)smem;
    }

    if (per_sm) {
        if (cached && kc.occ_smem[dev] == (int)smem + 1) {
            *per_sm = kc.occ[dev];
        } else {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, fn, threads, smem);
            if (e != cudaSuccess) return e;
            if (cached) {
                kc.occ[dev] = *per_sm;
                kc.occ_smem[dev] = (int)smem + 1;
            }
        }
    }
    return cudaSuccess;
}

#ifndef MOE_USE_PDL
#define MOE_USE_PDL 1
#endif

// Launch with programmatic dependent launch allowed: the kernel may start
// while its predecessor in the stream is finishing, and must execute
// griddep_wait() before touching memory that earlier work reads or writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = MOE_USE_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// device side: PTX wrappers (sm_90+ forms, valid on sm_103a)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// mbarrier ------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One bounded probe of the barrier phase; true once phase `parity` completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk (non-tensor) TMA copies ------------------------------------------------

// global -> shared, completion signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                         uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// shared -> global, tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void *gmem_dst, const void *smem_src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(gmem_dst), "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups completed (writes visible).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Streaming 16-byte global load that bypasses L1 (read-only data).
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_stream8(const void *p)
{
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ void st8(void *p, uint2 v)
{
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// 16-byte store marked streaming (evict first)
__device__ __forceinline__ void st16_cs(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Asks the bulk-copy engine to bring [p, p + bytes) into L2 (no completion
// to wait for).  p 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void st16(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

} // namespace moe
