// Status codes, error bookkeeping and device queries of the C ABI.
#include "common.cuh"

namespace moe {

namespace {
thread_local int t_last_cuda_error = 0;
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];  // 0 = not queried yet
} // namespace

// Records the error for moe_last_cuda_error() and consumes the runtime's
// pending copy, so that a failure reported here does not resurface at the
// caller's next, unrelated CUDA call.
void set_cuda_error(cudaError_t e)
{
    t_last_cuda_error = (int)e;
    (void)cudaGetLastError();
}

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev < kMaxDevices && g_sm_count[dev] > 0) return g_sm_count[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 1;
    if (dev < kMaxDevices) g_sm_count[dev] = n;
    return n;
}

} // namespace moe

MOE_EXPORT int moe_version(void) { return 2; }

MOE_EXPORT const char *moe_status_string(int status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_EINVAL: return "invalid argument (null pointer, size out of range, bad dtype or group size)";
    case MOE_EALIGN: return "misaligned: row pointers and row sizes must be multiples of 16 bytes";
    case MOE_ECUDA: return "CUDA launch or attribute call failed (see moe_last_cuda_error)";
    default: return "unknown status";
    }
}

MOE_EXPORT int moe_last_cuda_error(void) { return moe::t_last_cuda_error; }

MOE_EXPORT int moe_device_errors(uint32_t *flags)
{
    if (!flags) return MOE_EINVAL;
    uint32_t a = 0, b = 0, c = 0;
    cudaError_t e = moe::read_dispatch_errors(&a);
    if (e == cudaSuccess) e = moe::read_combine_errors(&b);
    if (e == cudaSuccess) e = moe::read_plan_dispatch_errors(&c);
    if (e != cudaSuccess) {
        moe::set_cuda_error(e);
        return MOE_ECUDA;
    }
    *flags = a | b | c;
    return MOE_OK;
}
