// AoS -> SoA weight relayout (a byte permutation, bit-exact).
//
// The pages upload the raw 34-byte `BlockTQ2_0_g128` records and convert them
// on the GPU with `reformat_tq2_aos_to_soa` ("oxibonsai-image 0.2.2
// src/gpu.rs", doc of `blocks_as_bytes`).  Because blocks are stored in
// row-major (n, b) order in both layouts, the relayout de-interleaves one
// stream of 34-byte records into a 32-byte stream (qs plane) and a 2-byte
// stream (d plane).
//
// One CTA moves a tile of 256 blocks (8704 bytes): coalesced 16-byte loads
// into shared memory, then coalesced 16-byte stores of the 8192 qs bytes and
// the 512 d bytes.  HBM-bound: 34 bytes read + 34 bytes written per block.
#include <algorithm>

#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int kTileBlocks = 256;
constexpr int kTileBytes = kTileBlocks * kBlockBytes;  // 8704 = 544 * 16
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
reformat_kernel(const uint8_t *__restrict__ aos, uint8_t *__restrict__ qs_plane,
                uint8_t *__restrict__ d_plane, int64_t nblk) {
    __shared__ __align__(16) uint8_t tile[kTileBytes];
    const bool vec = (reinterpret_cast<uintptr_t>(aos) & 15u) == 0;
    const int64_t ntiles = (nblk + kTileBlocks - 1) / kTileBlocks;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int64_t b0 = t * kTileBlocks;
        const int nb = static_cast<int>(nblk - b0 < kTileBlocks ? nblk - b0 : kTileBlocks);
        const int bytes = nb * kBlockBytes;
        const uint8_t *src = aos + b0 * kBlockBytes;
        __syncthreads();  // previous tile fully consumed
        if (vec) {
            const int nvec = bytes / 16;
            for (int i = threadIdx.x; i < nvec; i += kThreads)
                reinterpret_cast<uint4 *>(tile)[i] = __ldg(reinterpret_cast<const uint4 *>(src) + i);
            for (int i = nvec * 16 + threadIdx.x; i < bytes; i += kThreads) tile[i] = src[i];
        } else {
            for (int i = threadIdx.x; i < bytes; i += kThreads) tile[i] = src[i];
        }
        __syncthreads();
        // qs: 2 * nb output 16-byte words, word u = half (u & 1) of block u >> 1.
        uint8_t *qdst = qs_plane + b0 * kQsBytes;
        for (int u = threadIdx.x; u < 2 * nb; u += kThreads) {
            const uint16_t *s16 =
                reinterpret_cast<const uint16_t *>(tile + (u >> 1) * kBlockBytes + (u & 1) * 16);
            uint4 v;
            v.x = uint32_t(s16[0]) | (uint32_t(s16[1]) << 16);
            v.y = uint32_t(s16[2]) | (uint32_t(s16[3]) << 16);
            v.z = uint32_t(s16[4]) | (uint32_t(s16[5]) << 16);
            v.w = uint32_t(s16[6]) | (uint32_t(s16[7]) << 16);
            reinterpret_cast<uint4 *>(qdst)[u] = v;
        }
        // d: 8 blocks per 16-byte output word; a ragged tail is written per block.
        uint8_t *ddst = d_plane + b0 * 2;
        const int nfull = nb / 8;
        for (int u = threadIdx.x; u < nfull; u += kThreads) {
            uint32_t h[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                h[j] = *reinterpret_cast<const uint16_t *>(tile + (8 * u + j) * kBlockBytes + kQsBytes);
            uint4 v = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                                 h[6] | (h[7] << 16));
            reinterpret_cast<uint4 *>(ddst)[u] = v;
        }
        for (int b = nfull * 8 + threadIdx.x; b < nb; b += kThreads) {
            reinterpret_cast<uint16_t *>(ddst)[b] =
                *reinterpret_cast<const uint16_t *>(tile + b * kBlockBytes + kQsBytes);
        }
    }
}

}  // namespace

cudaError_t launch_reformat(const void *w_aos, void *w_soa, int64_t n, int64_t k,
                            const LaunchCtx &ctx) {
    const int64_t nblk = n * (k / kBlockW);
    const int64_t ntiles = (nblk + kTileBlocks - 1) / kTileBlocks;
    const int64_t grid = std::min<int64_t>(ntiles, int64_t(ctx.num_sms) * 8);
    uint8_t *soa = static_cast<uint8_t *>(w_soa);
    reformat_kernel<<<static_cast<unsigned>(grid), kThreads, 0, ctx.stream>>>(
        static_cast<const uint8_t *>(w_aos), soa, soa + nblk * kQsBytes, nblk);
    return cudaPeekAtLastError();
}

}  // namespace tq2
