// Encoder: f32 weights [n][k] -> TQ2_0_g128 AoS blocks [n][k/128] (34 bytes).
//
// The pages never show how the blocks are produced (they are read from a GGUF
// file); this library's reading is the absmean rule of ternary weights, with
// every floating-point step that decides a code fixed so that the result is
// reproducible bit for bit:
//   gamma = (sum_{j=0..127} |w_j|) / 128, the sum in double in index order;
//   d     = binary16(gamma), round to nearest even;
//   q_j   = rint(w_j / (float)d) in binary32 (IEEE division, ties to even),
//           clamped to [-1, 1]; code c_j = q_j + 1 at bits 2*(j%4) of qs[j/4].
// A zero or non-finite d gives code 1 (weight 0) everywhere.
//
// A CTA takes 32 consecutive blocks (16 KB of the row-major weights, one
// contiguous range): coalesced 16-byte loads into shared memory, one thread per
// block for the sequential double sum, four threads per block for the codes,
// and the 32 x 34 output bytes staged in shared memory and written out
// contiguously.  A block is stored as four 32-float parts 40 floats apart and
// blocks 161 floats apart: word (t + 8 part + j) mod 32 is the bank, so both the
// per-block sum (32 threads, one block each) and the code phase (8 blocks x 4
// parts per warp) read without bank conflicts.
#include <cuda_fp16.h>

#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int kQBlocks = 32;   // blocks per CTA
constexpr int kQThreads = 128;
constexpr int kQPart = 40;     // float stride of a staged 32-weight part
constexpr int kQBlk = 161;     // float stride of a staged block (4 parts + 1)

// double -> binary16 bits, round to nearest even: |v| >= 65520 -> Inf (halfway
// past the largest finite 65504), subnormals on the 2^-24 grid.
__device__ __forceinline__ uint16_t to_half_rne(double v) {
    const uint16_t sign = signbit(v) ? 0x8000 : 0;
    const double a = fabs(v);
    if (isnan(v)) return 0x7e00;
    if (a >= 65520.0) return uint16_t(sign | 0x7c00);
    if (a < 6.103515625e-05) {  // 2^-14: subnormal grid of 2^-24 (1024 carries into the exponent)
        return uint16_t(sign | uint16_t(rint(a * 16777216.0)));
    }
    int ex;
    frexp(a, &ex);  // a = m * 2^ex, m in [0.5, 1)
    int e = ex - 1;
    double r = rint(ldexp(a, 10 - e));  // in [1024, 2048]
    if (r >= 2048.0) {
        r = 1024.0;
        e += 1;
    }
    if (e > 15) return uint16_t(sign | 0x7c00);
    return uint16_t(sign | uint16_t((e + 15) << 10) | uint16_t(r - 1024.0));
}

__global__ void __launch_bounds__(kQThreads)
quantize_kernel(const float *__restrict__ w, uint8_t *__restrict__ aos, int64_t nblk) {
    __shared__ float sw[kQBlocks * kQBlk];
    __shared__ uint16_t sd[kQBlocks];
    __shared__ __align__(16) uint8_t so[kQBlocks * kBlockBytes];
    const int64_t b0 = int64_t(blockIdx.x) * kQBlocks;
    const int nb = nblk - b0 < kQBlocks ? int(nblk - b0) : kQBlocks;
    const float4 *src = reinterpret_cast<const float4 *>(w + b0 * kBlockW);
    for (int i = threadIdx.x; i < nb * 32; i += kQThreads) {  // 32 float4 per block
        const float4 v = __ldcs(src + i);
        const int blk = i >> 5, j = (i & 31) * 4;
        float *d = sw + blk * kQBlk + (j >> 5) * kQPart + (j & 31);
        d[0] = v.x;
        d[1] = v.y;
        d[2] = v.z;
        d[3] = v.w;
    }
    __syncthreads();
    if (int(threadIdx.x) < nb) {
        const float *b = sw + threadIdx.x * kQBlk;
        double s = 0.0;
        for (int j = 0; j < kBlockW; ++j) s += fabs(double(b[(j >> 5) * kQPart + (j & 31)]));
        sd[threadIdx.x] = to_half_rne(s * 0.0078125);  // / 128, exact
    }
    __syncthreads();
    {
        const int blk = threadIdx.x >> 2, part = threadIdx.x & 3;  // 32 weights each
        if (blk < nb) {
            const uint16_t dh = sd[blk];
            const float df = __half2float(__ushort_as_half(dh));
            const bool live = df > 0.f && isfinite(df);
            const float *p = sw + blk * kQBlk + part * kQPart;
            uint8_t *ob = so + blk * kBlockBytes + part * 8;
#pragma unroll
            for (int by = 0; by < 8; ++by) {
                uint32_t byte = 0;
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    int c = 1;
                    if (live) {
                        const float q = rintf(__fdiv_rn(p[by * 4 + f], df));
                        c = q >= 1.f ? 2 : (q <= -1.f ? 0 : 1);
                    }
                    byte |= uint32_t(c) << (2 * f);
                }
                ob[by] = uint8_t(byte);
            }
            if (part == 0) {
                so[blk * kBlockBytes + 32] = uint8_t(dh & 0xff);
                so[blk * kBlockBytes + 33] = uint8_t(dh >> 8);
            }
        }
    }
    __syncthreads();
    // nb * 34 bytes, contiguous from block b0 (even offsets: 16-bit stores)
    const uint16_t *s16 = reinterpret_cast<const uint16_t *>(so);
    uint16_t *d16 = reinterpret_cast<uint16_t *>(aos + b0 * kBlockBytes);
    for (int i = threadIdx.x; i < nb * (kBlockBytes / 2); i += kQThreads) d16[i] = s16[i];
}

}  // namespace

cudaError_t launch_quantize(const float *w, void *w_aos, int64_t n, int64_t k, const LaunchCtx &ctx) {
    const int64_t nblk = n * (k / kBlockW);
    if (nblk == 0) return cudaSuccess;
    const int64_t grid = (nblk + kQBlocks - 1) / kQBlocks;
    if (grid > int64_t(INT32_MAX)) return cudaErrorInvalidValue;
    quantize_kernel<<<unsigned(grid), kQThreads, 0, ctx.stream>>>(w, static_cast<uint8_t *>(w_aos), nblk);
    return cudaPeekAtLastError();
}

}  // namespace tq2
