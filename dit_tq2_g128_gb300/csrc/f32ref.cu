// Exact-f32 CUDA-core tiled GEMM (tq2_gemm_f32ref).
//
// The role of the pages' `gemm_tq2_g128_v8_tiled` ("oxibonsai-kernels 0.1.5
// src/gpu_backend/metal_graph/pipelines.rs": a 2-D grid over N and M,
// register-blocked micro-tiles, each weight block decoded once per M-tile):
// a plain, numerically conservative kernel kept for tolerance checks.
//
// One CTA computes a 64 (M) x 64 (N) tile; each of its 256 threads a 4x4
// micro-tile.  K advances in 32-wide slices: the x slice is copied to shared
// memory and the code slice is decoded to (c - 1) as f32 in shared memory.
// Products are exact; sums run per 128-weight block into a partial that is
// then scaled by the block's d and added to the accumulator (blocked
// summation keeps the rounding error at about (128 + K/128) ulps worst case).
#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int kBM = 64, kBN = 64, kBK = 32, kThreads = 256;

__global__ void __launch_bounds__(kThreads)
f32ref_kernel(const uint8_t *__restrict__ qs, const __half *__restrict__ dpl,
              const float *__restrict__ x, const float *residual, float *out, int m, int n,
              int k) {
    __shared__ float xs[kBK][kBM + 4];  // [k][m]
    __shared__ float ws[kBK][kBN + 4];  // [k][n], (c - 1)
    const int tid = threadIdx.x;
    const int tm = tid / 16, tn = tid % 16;  // 16 x 16 threads, 4 x 4 each
    const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
    const int64_t kq = k / 4, kb = k / kBlockW;

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int64_t b = 0; b < kb; ++b) {
        float p[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) p[i][j] = 0.f;
        for (int s = 0; s < kBlockW / kBK; ++s) {
            const int64_t k0 = b * kBlockW + s * kBK;
            __syncthreads();
            // x slice: 64 rows x 32 k, two float4 per thread
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int e = tid + h * kThreads;  // 0..511 float4 slots
                const int row = e / 8, q = e % 8;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (m0 + row < m)
                    v = __ldg(reinterpret_cast<const float4 *>(x + int64_t(m0 + row) * k + k0) + q);
                xs[4 * q + 0][row] = v.x;
                xs[4 * q + 1][row] = v.y;
                xs[4 * q + 2][row] = v.z;
                xs[4 * q + 3][row] = v.w;
            }
            // codes: 64 rows x 8 bytes; threads 0..127 decode one 32-bit word each
            if (tid < 128) {
                const int row = tid / 2, half = tid % 2;
                uint32_t w = 0x55555555u;  // all-zero weights beyond N
                if (n0 + row < n)
                    w = __ldg(reinterpret_cast<const unsigned int *>(qs + int64_t(n0 + row) * kq +
                                                                      k0 / 4) + half);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    ws[16 * half + i][row] = float(int((w >> (2 * i)) & 3u) - 1);
            }
            __syncthreads();
#pragma unroll 8
            for (int kk = 0; kk < kBK; ++kk) {
                float a[4], bb[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = xs[kk][tm * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) bb[j] = ws[kk][tn * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) p[i][j] = fmaf(a[i], bb[j], p[i][j]);
            }
        }
        float dj[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = n0 + tn * 4 + j;
            dj[j] = col < n ? __half2float(dpl[int64_t(col) * kb + b]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(p[i][j], dj[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = m0 + tm * 4 + i;
        if (row >= m) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = n0 + tn * 4 + j;
            if (col >= n) continue;
            const int64_t o = int64_t(row) * n + col;
            float v = acc[i][j];
            if (residual) v += residual[o];
            out[o] = v;
        }
    }
}

}  // namespace

cudaError_t launch_f32ref(const void *w_soa, const float *x, const float *residual, float *out,
                          int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx) {
    if (m > INT32_MAX || n > INT32_MAX || k > INT32_MAX) return cudaErrorInvalidValue;
    const SoaView v = soa_view(w_soa, n, k);
    dim3 grid(static_cast<unsigned>((n + kBN - 1) / kBN), static_cast<unsigned>((m + kBM - 1) / kBM));
    if (grid.y > 65535) return cudaErrorInvalidValue;
    f32ref_kernel<<<grid, kThreads, 0, ctx.stream>>>(v.qs, v.d, x, residual, out, int(m), int(n),
                                                     int(k));
    return cudaPeekAtLastError();
}

}  // namespace tq2
