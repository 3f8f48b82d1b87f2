// Self-test of the number-format conversions the kernels use, over any range
// of binary32 bit patterns (the whole 2^32 included): the E4M3 cast of the
// quantising dispatch (OCP 8-bit Floating Point Specification v1.0, E4M3:
// round to nearest even, saturated to +-448 -- the cast `e4m3x4` applies,
// __nv_cvt_float2_to_fp8x2 with __NV_SATFINITE and __NV_E4M3) and the
// bfloat16 store of the combines (round to nearest even, the
// __floats2bfloat162_rn of `Io<__nv_bfloat16>::store`).  Sources: ROCm/mori
// "Draft: cco + flydsl dispatch/combine #448", Fp8BlockwiseQuant notes (the
// fp8 cast of each scaled element) and accumulator note (bf16 rows widened
// to f32, summed, stored back).

#include "common.cuh"

#include <cuda_fp8.h>

namespace moe {
namespace {

// thread g converts patterns first + 4g .. first + 4g + 3
__global__ void selftest_convert_kernel(uint32_t first, int64_t groups, uint8_t *e4m3_out,
                                        uint16_t *bf16_out)
{
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups;
         g += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t b0 = first + (uint32_t)(4 * g);  // wraps only past 2^32, never reached
        float f[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(b0 + (uint32_t)i);
        if (e4m3_out) {
            const __nv_fp8x2_storage_t lo =
                __nv_cvt_float2_to_fp8x2(make_float2(f[0], f[1]), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi =
                __nv_cvt_float2_to_fp8x2(make_float2(f[2], f[3]), __NV_SATFINITE, __NV_E4M3);
            reinterpret_cast<uint32_t *>(e4m3_out)[g] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        if (bf16_out) {
            const __nv_bfloat162 p = __floats2bfloat162_rn(f[0], f[1]);
            const __nv_bfloat162 q = __floats2bfloat162_rn(f[2], f[3]);
            reinterpret_cast<uint2 *>(bf16_out)[g] =
                make_uint2(*reinterpret_cast<const uint32_t *>(&p),
                           *reinterpret_cast<const uint32_t *>(&q));
        }
    }
}

} // namespace
} // namespace moe

using namespace moe;

MOE_EXPORT int moe_selftest_convert(uint32_t first, int64_t count, uint8_t *e4m3_out,
                                    uint16_t *bf16_out, moe_stream_t stream)
{
    MOE_TRACE("moe_selftest_convert");
    if (count < 0 || (first & 3u) || (count & 3) || (int64_t)first + count > ((int64_t)1 << 32))
        return MOE_EINVAL;
    if (!e4m3_out && !bf16_out) return MOE_EINVAL;
    if ((e4m3_out && !aligned16(e4m3_out)) || (bf16_out && !aligned16(bf16_out)))
        return MOE_EALIGN;
    if (count == 0) return MOE_OK;
    const int64_t groups = count / 4;
    int64_t blocks = (groups + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    selftest_convert_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(first, groups,
                                                                                 e4m3_out, bf16_out);
    return check_launch();
}
