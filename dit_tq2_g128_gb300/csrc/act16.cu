// Conversions between f32 activations and the library's binary16 activation
// layout: row-major [m][k], element i of every 16-element group stored at
// position 2i (i < 8) or 2(i-8)+1 (i >= 8).  That is the k order in which the
// tensor-core kernel decodes weights (weights i and i+8 of a code word share
// one half2), so activations in this layout feed the kernel's MMA tiles with a
// plain tensor copy and no conversion pass.  Conversion to binary16 rounds to
// nearest even (|x| >= 65520 becomes Inf); the way back is exact.
#include <algorithm>

#include "tq2_internal.cuh"

namespace tq2 {
namespace {

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);  // lo in the low 16 bits
    return *reinterpret_cast<const uint32_t *>(&h);
}

// One thread per 16-element group: word j of the group holds elements j and j+8.
__global__ void __launch_bounds__(256) act16_from_f32_kernel(const float *__restrict__ x, uint4 *__restrict__ y,
                                                             int64_t groups) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; g < groups; g += stride) {
        const float4 *src = reinterpret_cast<const float4 *>(x + g * 16);
        const float4 a = __ldcs(src), b = __ldcs(src + 1), c = __ldcs(src + 2), d = __ldcs(src + 3);
        // elements 0..7 = a, b; 8..15 = c, d
        y[2 * g] = make_uint4(pack_half2(a.x, c.x), pack_half2(a.y, c.y), pack_half2(a.z, c.z),
                              pack_half2(a.w, c.w));
        y[2 * g + 1] = make_uint4(pack_half2(b.x, d.x), pack_half2(b.y, d.y), pack_half2(b.z, d.z),
                                  pack_half2(b.w, d.w));
    }
}

__global__ void __launch_bounds__(256) act16_to_f32_kernel(const uint4 *__restrict__ y, float *__restrict__ x,
                                                           int64_t groups) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; g < groups; g += stride) {
        const uint4 p = y[2 * g], q = y[2 * g + 1];
        const uint32_t w[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
        float lo[8], hi[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const __half2 h = *reinterpret_cast<const __half2 *>(&w[j]);
            lo[j] = __low2float(h);
            hi[j] = __high2float(h);
        }
        float4 *dst = reinterpret_cast<float4 *>(x + g * 16);
        dst[0] = make_float4(lo[0], lo[1], lo[2], lo[3]);
        dst[1] = make_float4(lo[4], lo[5], lo[6], lo[7]);
        dst[2] = make_float4(hi[0], hi[1], hi[2], hi[3]);
        dst[3] = make_float4(hi[4], hi[5], hi[6], hi[7]);
    }
}

}  // namespace

cudaError_t launch_act16_from_f32(const float *x, __half *x16, int64_t m, int64_t k, const LaunchCtx &ctx) {
    const int64_t groups = m * (k / 16);
    if (groups == 0) return cudaSuccess;
    const int64_t grid = std::min<int64_t>((groups + 255) / 256, int64_t(ctx.num_sms) * 8);
    act16_from_f32_kernel<<<unsigned(grid), 256, 0, ctx.stream>>>(x, reinterpret_cast<uint4 *>(x16), groups);
    return cudaPeekAtLastError();
}

cudaError_t launch_act16_to_f32(const __half *x16, float *x, int64_t m, int64_t k, const LaunchCtx &ctx) {
    const int64_t groups = m * (k / 16);
    if (groups == 0) return cudaSuccess;
    const int64_t grid = std::min<int64_t>((groups + 255) / 256, int64_t(ctx.num_sms) * 8);
    act16_to_f32_kernel<<<unsigned(grid), 256, 0, ctx.stream>>>(reinterpret_cast<const uint4 *>(x16), x, groups);
    return cudaPeekAtLastError();
}

}  // namespace tq2
