// Skinny-M tensor-core kernel (2 <= M <= 32): one launch, no workspace.
//
// Computes the contract of "oxibonsai-image 0.2.2 src/gpu.rs" (module doc
// "Correctness contract"), out[m, n] = sum_k x[m, k] * dequant(W)[n, k]
// (+ residual), for the few-row batches that the pages' `gemm_tq2_g128_v7`
// serves ("oxibonsai-kernels 0.1.5 src/gpu_backend/metal_graph/pipelines.rs",
// TQ2 pipeline fields: any batch size).  With M this small the product is
// bound by streaming and decoding the weights, not by multiply throughput, so
// the design keeps decoded weights out of shared memory altogether:
//
//  * Warp-level MMAs (m16n8k16, f16 operands, f32 accumulation) take their A
//    operand from registers.  A = 16 weight rows x 16 k, decoded straight into
//    the fragment registers; B = the x rows (8 per n-tile) from shared memory.
//    (The tcgen05 MMAs read A from shared memory or tensor memory only; for
//    N <= 32 their decoded-operand traffic, 2 bytes per weight through shared
//    memory, would cost more than the whole multiply.)
//  * Decode without bias removal.  A code c at mantissa bits 2p of a binary16
//    whose exponent is chosen for that position reads as 2^(10-2p) + c exactly
//    (one AND-OR for two weights), so the MMA computes sum_k (B_k + c_k) x_k.
//    The weight-independent part sum_k (B_k + 1) x_k of each 128-weight block
//    (the "+1" gives c - 1) is computed once per CTA from the same binary16 x
//    and subtracted per block before the block's scale d is applied in f32.
//  * K order.  Within a 16-weight code word, MMA columns (2q, 2q+1) hold
//    weights (q, q+8) and columns (2q+8, 2q+9) hold (q+4, q+12): the first
//    pair comes from one mask of the word, the second from one mask of the word
//    shifted by 2q.  x is staged in the matching order (the library's binary16
//    activation layout: element i of a 16-group at position 2i, or 2(i-8)+1).
//  * Work split.  A CTA (8 warps x 16 rows) owns 128 weight rows and a K slice;
//    the S CTAs that share a row tile form a cluster, and after the contraction
//    each CTA sums a share of the tile's rows over the S partials in rank order
//    (distributed shared memory): deterministic, one launch, nothing in global
//    memory but the result.  The CTA's codes arrive by tensor copies
//    (128 rows x 128 bytes per box, 128-byte swizzle: conflict-free 16-byte
//    reads), its x slice and block scales by plain loads.
#include <algorithm>
#include <climits>
#include <cstring>

#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int SK_WARPS = 8;
constexpr int SK_THREADS = 32 * SK_WARPS;
constexpr int SK_ROWS = 16 * SK_WARPS;     // weight rows per CTA
constexpr int SK_BOX_W = 512;              // weights per code box (128 bytes per row)
constexpr int SK_BOX_BYTES = SK_ROWS * 128;
constexpr int SK_PART_PAD = 4;             // floats of padding per partial row
constexpr size_t SK_SMEM_BUDGET = 200 * 1024;

struct SkParams {
    int M, N, K;
    int S;              // K slices = CTAs per cluster
    int nb;             // 128-weight blocks per row (K / 128)
    int mpad;           // M rounded up to a multiple of 8
    int xstride;        // halves per staged x row
    int nbs_max;        // most blocks any slice holds
    uint32_t off_x, off_d, off_bias, off_part, off_bar;  // shared-memory offsets from the 1024-aligned base
};

__device__ __forceinline__ void sk_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void sk_tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void sk_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t sk_mapa(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// D += A * B, m16n8k16, f16 inputs, f32 accumulation.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Bias of staged x position p (0..15) of a 16-group: 2^(10 - 2(p/2)) for p < 8, else 4.
__device__ __forceinline__ float sk_pos_bias(int p) {
    return p < 8 ? float(1 << (10 - 2 * (p >> 1))) : 4.0f;
}

template <int NT>
__global__ void __launch_bounds__(SK_THREADS, 1)
skinny_mma_kernel(const __grid_constant__ CUtensorMap qmap, const __half *__restrict__ dpl,
                  const float *__restrict__ x, const float *residual, float *out, SkParams P,
                  unsigned int *status, uint64_t wait_ns) {
    extern __shared__ __align__(1024) uint8_t sk_raw[];
    uint8_t *base = sk_raw + ((1024u - (smem_u32(sk_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = P.S;
    const int rank = int(blockIdx.x) % S, tile = int(blockIdx.x) / S;
    const int b0 = int(int64_t(rank) * P.nb / S), b1 = int(int64_t(rank + 1) * P.nb / S);
    const int nbs = b1 - b0;                      // blocks of this slice
    const int kslice = nbs * kBlockW;
    const int nbox = (nbs + 3) / 4;               // 512-weight code boxes
    const int row0 = tile * SK_ROWS;

    __half *xs = reinterpret_cast<__half *>(base + P.off_x);     // [mpad][xstride] binary16, activation order
    float *dsm = reinterpret_cast<float *>(base + P.off_d);      // [SK_ROWS][nbs_max] block scales
    float *bsm = reinterpret_cast<float *>(base + P.off_bias);   // [nbs_max][mpad] bias sums
    float *part = reinterpret_cast<float *>(base + P.off_part);  // receive buffer [S][mpad][SK_ROWS / S]
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + P.off_bar);

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_proxy_async_smem();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&qmap)) : "memory");
        // the CTA's code boxes and block scales go to L2 before the dependency
        // wait (L2 is the point of coherence: a prefetch cannot leave stale data)
        for (int j = 0; j < nbox; ++j)
            asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                             reinterpret_cast<uint64_t>(&qmap)),
                         "r"((b0 * kBlockW + j * SK_BOX_W) / 4), "r"(row0)
                         : "memory");
    }
    if (tid < SK_ROWS && row0 + tid < P.N)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(dpl + int64_t(row0 + tid) * P.nb + b0) : "memory");
    __syncthreads();
    // Programmatic dependent launch: x, the weights, the residual and out are
    // touched only after the preceding kernel of the stream has completed; the
    // next kernel may start its own set-up now.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0 && nbox > 0) {
        sk_expect_tx(bar, uint32_t(nbox) * SK_BOX_BYTES);
        for (int j = 0; j < nbox; ++j)
            sk_tma_2d(smem_u32(base) + uint32_t(j) * SK_BOX_BYTES, &qmap, (b0 * kBlockW + j * SK_BOX_W) / 4, row0,
                      bar);
    }
    // x slice -> binary16 in the activation order (rows past M are zero), and
    // the block scales of the tile's rows (rows past N: 0).  Every load of a
    // round is issued before any of it is used: the loads' latency is paid once
    // per round, not once per item.
    {
        const int groups = kslice / 16;
        const int k0 = b0 * kBlockW;
        const int kb = P.nb;
        const int nx = P.mpad * groups, nd = SK_ROWS * nbs;
        // x items (one 16-element group of one row) two per thread and round,
        // block scales four per thread and round; the item count of x is a
        // multiple of 64, so every round is warp-uniform for the shuffles below
        for (int r0 = 0; r0 < nx || r0 < nd; r0 += 4 * SK_THREADS) {
            unsigned short dv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int it = r0 + j * SK_THREADS + tid;
                const int r = it / nbs, b = it - r * nbs;
                dv[j] = (it < nd && row0 + r < P.N) ? ldg_u16(dpl + int64_t(row0 + r) * kb + b0 + b) : 0;
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int xb = r0 + half * 2 * SK_THREADS;
                if (xb >= nx) break;  // warp-uniform (nx % 64 == 0)
                float f[2][16];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int it = xb + j * SK_THREADS + tid;
                    const int nrow = it / groups, gi = it - nrow * groups;
                    if (it < nx && nrow < P.M) {
                        const float4 *src = reinterpret_cast<const float4 *>(x + int64_t(nrow) * P.K + k0 + 16 * gi);
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            const float4 v = __ldg(src + qq);
                            f[j][4 * qq] = v.x; f[j][4 * qq + 1] = v.y; f[j][4 * qq + 2] = v.z; f[j][4 * qq + 3] = v.w;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) f[j][i] = 0.f;
                    }
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int it = xb + j * SK_THREADS + tid;
                    if (it >= nx) break;  // warp-uniform
                    const int nrow = it / groups, gi = it - nrow * groups;
                    uint32_t h[8];
                    float bsum = 0.f;  // this group's share of sum (bias + 1) * x16 over its block
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const __half2 v = __floats2half2_rn(f[j][i], f[j][i + 8]);  // positions 2i, 2i+1
                        h[i] = *reinterpret_cast<const uint32_t *>(&v);
                        const float2 rr = __half22float2(v);
                        bsum = fmaf(sk_pos_bias(2 * i) + 1.0f, rr.x + rr.y, bsum);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(xs + int64_t(nrow) * P.xstride + 16 * gi);
                    dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
                    dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
                    // the 8 groups of a block sit in 8 consecutive lanes (groups per
                    // row and the thread stride are multiples of 8): a fixed-order sum
                    bsum += __shfl_xor_sync(0xffffffffu, bsum, 1);
                    bsum += __shfl_xor_sync(0xffffffffu, bsum, 2);
                    bsum += __shfl_xor_sync(0xffffffffu, bsum, 4);
                    if ((gi & 7) == 0) bsm[(gi >> 3) * P.mpad + nrow] = bsum;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int it = r0 + j * SK_THREADS + tid;
                if (it < nd) {
                    const int r = it / nbs, b = it - r * nbs;
                    dsm[r * P.nbs_max + b] = __half2float(__ushort_as_half(dv[j]));
                }
            }
        }
    }
    __syncthreads();

    // ---- contraction: warp w owns weight rows 16w + g and 16w + g + 8 of the tile
    const int g = lane >> 2, q = lane & 3;
    const int ra = warp * 16 + g, rb = ra + 8;  // tile-relative rows of this thread's fragment
    const uint32_t mask_lo = 0x00030003u << (2 * q);
    const uint32_t mag_lo = uint32_t(25 - 2 * q) << 10 | (uint32_t(25 - 2 * q) << 26);
    const uint32_t sh = uint32_t(2 * q);
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[t][j] = 0.f;
    const bool ok = mbar_wait_spin(bar, 0, wait_ns, status);
    if (ok) {
        const uint8_t *codes = base;
        const __half *xrow[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) xrow[t] = xs + int64_t(t * 8 + g) * P.xstride + 2 * q;
        // independent accumulator chains per n-tile (k16-step mod CH) hide the
        // MMA latency: four when there are one or two n-tiles, else two
        constexpr int CH = NT <= 2 ? 4 : 2;
        for (int b = 0; b < nbs; ++b) {
            float cc[CH][NT][4];
#pragma unroll
            for (int h = 0; h < CH; ++h)
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int j = 0; j < 4; ++j) cc[h][t][j] = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // 16 bytes (four code words) of rows ra and rb: chunk c of box j
                const int s4 = b * 8 + h * 4;  // first k16-step of the chunk within the slice
                const int j = s4 >> 5, c = (s4 & 31) >> 2;
                const uint8_t *bx = codes + j * SK_BOX_BYTES;
                const uint4 wa = *reinterpret_cast<const uint4 *>(bx + ra * 128 + ((c ^ (ra & 7)) << 4));
                const uint4 wb = *reinterpret_cast<const uint4 *>(bx + rb * 128 + ((c ^ (rb & 7)) << 4));
                const uint32_t wav[4] = {wa.x, wa.y, wa.z, wa.w}, wbv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint32_t a[4];
                    a[0] = (wav[u] & mask_lo) | mag_lo;
                    a[1] = (wbv[u] & mask_lo) | mag_lo;
                    a[2] = ((wav[u] >> sh) & 0x03000300u) | 0x44004400u;
                    a[3] = ((wbv[u] >> sh) & 0x03000300u) | 0x44004400u;
                    const int kx = (s4 + u) * 16;  // staged x offset of this k16-step
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const uint32_t bb0 = *reinterpret_cast<const uint32_t *>(xrow[t] + kx);
                        const uint32_t bb1 = *reinterpret_cast<const uint32_t *>(xrow[t] + kx + 8);
                        mma16816(cc[(h * 4 + u) % CH][t], a, bb0, bb1);
                    }
                }
            }
            // block fixup: acc += d_row * (sum - bias sum of the x row)
            const float da = dsm[ra * P.nbs_max + b], db = dsm[rb * P.nbs_max + b];
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float sm[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    float v = cc[0][t][jj];
#pragma unroll
                    for (int hh = 1; hh < CH; ++hh) v += cc[hh][t][jj];
                    sm[jj] = v;
                }
                const float2 bs = *reinterpret_cast<const float2 *>(bsm + b * P.mpad + t * 8 + 2 * q);
                acc[t][0] = fmaf(da, sm[0] - bs.x, acc[t][0]);
                acc[t][1] = fmaf(da, sm[1] - bs.y, acc[t][1]);
                acc[t][2] = fmaf(db, sm[2] - bs.x, acc[t][2]);
                acc[t][3] = fmaf(db, sm[3] - bs.y, acc[t][3]);
            }
        }
    }
    // Reduction over the S CTAs of the tile.  CTA r finishes tile rows
    // [r * rpr, (r + 1) * rpr): every CTA pushes its partial sums of those
    // rows into CTA r's receive buffer (slot = the sender's rank) with
    // distributed-shared-memory stores, one cluster barrier makes them
    // visible, and each CTA sums its slots in rank order (+ residual).  Nothing
    // is read from another CTA after the barrier, so no second one is needed.
    const int rpr = SK_ROWS / S;
    const uint32_t part_addr = smem_u32(part);
    auto push = [&](int row, int n, float v) {
        const int o = row / rpr, rl = row - o * rpr;
        const uint32_t off = uint32_t(((rank * P.mpad + n) * rpr + rl) * 4);
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(sk_mapa(part_addr + off, uint32_t(o))), "f"(v)
                     : "memory");
    };
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int n0 = t * 8 + 2 * q;
        push(ra, n0, acc[t][0]);
        push(ra, n0 + 1, acc[t][1]);
        push(rb, n0, acc[t][2]);
        push(rb, n0 + 1, acc[t][3]);
    }
    sk_cluster_sync();
    for (int it = tid; it < P.M * rpr; it += SK_THREADS) {
        const int nrow = it / rpr, rl = it - nrow * rpr;
        const int grow = row0 + rank * rpr + rl;
        if (grow >= P.N) continue;
        float sum = 0.f;
        for (int sr = 0; sr < S; ++sr) sum += part[(sr * P.mpad + nrow) * rpr + rl];
        const int64_t o = int64_t(nrow) * P.N + grow;
        if (residual) sum += residual[o];
        out[o] = sum;
    }
    if (!ok && tid == 0) {
        // the code copies never completed: give them a fixed 200 us to land
        // before the CTA's shared memory goes away
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
    }
}

size_t sk_smem_bytes(int mpad, int xstride, int nbs_max) {
    const size_t codes = size_t((nbs_max + 3) / 4) * SK_BOX_BYTES;
    const size_t xb = size_t(mpad) * xstride * 2;
    const size_t db = size_t(SK_ROWS) * nbs_max * 4;
    const size_t bb = size_t(nbs_max) * mpad * 4;
    const size_t pb = size_t(mpad) * (SK_ROWS + SK_PART_PAD) * 4;
    return 1024 + codes + ((xb + 15) & ~size_t(15)) + db + bb + pb + 16;
}

}  // namespace

bool skinny_mma_fits(int64_t m, int64_t n, int64_t k) {
    if (m < 2 || m > 32 || n > INT32_MAX || k > INT32_MAX || k % kBlockW) return false;
    const int nb = int(k / kBlockW);
    const int mpad = int((m + 7) / 8) * 8;
    const int s = std::min(8, nb);  // the most slices a launch can use
    const int nbs_max = (nb + s - 1) / s;
    return sk_smem_bytes(mpad, nbs_max * kBlockW + 8, nbs_max) <= SK_SMEM_BUDGET;
}

cudaError_t launch_skinny_mma(const void *w_soa, const float *x, const float *residual, float *out,
                              int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx) {
    if (!skinny_mma_fits(m, n, k)) return cudaErrorNotSupported;
    const int nb = int(k / kBlockW);
    const int64_t tiles = (n + SK_ROWS - 1) / SK_ROWS;
    if (tiles > INT32_MAX / 8) return cudaErrorNotSupported;
    const int mpad = int((m + 7) / 8) * 8;
    // K slices: as many as keep the grid within one wave (1 CTA per SM), at
    // most 8 (cluster size) and at most one per block; more if shared memory
    // needs it
    auto smem_for = [&](int s) {
        const int nbs_max = (nb + s - 1) / s;
        const int xstride = nbs_max * kBlockW + 8;  // 16 bytes of padding: conflict-free x rows
        return sk_smem_bytes(mpad, xstride, nbs_max);
    };
    int S = 1;
    while (S < 8 && 2 * S <= nb && tiles * 2 * S <= ctx.num_sms) S *= 2;
    while (S < 8 && 2 * S <= nb && smem_for(S) > SK_SMEM_BUDGET) S *= 2;
    if (smem_for(S) > SK_SMEM_BUDGET) return cudaErrorNotSupported;

    SkParams P;
    P.M = int(m);
    P.N = int(n);
    P.K = int(k);
    P.S = S;
    P.nb = nb;
    P.mpad = mpad;
    P.nbs_max = (nb + S - 1) / S;
    P.xstride = P.nbs_max * kBlockW + 8;
    const size_t codes = size_t((P.nbs_max + 3) / 4) * SK_BOX_BYTES;
    const size_t xb = (size_t(mpad) * P.xstride * 2 + 15) & ~size_t(15);
    P.off_x = uint32_t(codes);
    P.off_d = uint32_t(codes + xb);
    P.off_bias = P.off_d + uint32_t(SK_ROWS * P.nbs_max * 4);
    P.off_part = P.off_bias + uint32_t(P.nbs_max * mpad * 4);
    P.off_bar = P.off_part + uint32_t(mpad * (SK_ROWS + SK_PART_PAD) * 4);
    const size_t smem = 1024 + size_t(P.off_bar) + 16;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const SoaView v = soa_view(w_soa, n, k);
    CUtensorMap qmap;
    {
        const cuuint64_t gdim[2] = {cuuint64_t(k / 4), cuuint64_t(n)};
        const cuuint64_t gstride[1] = {cuuint64_t(k / 4)};
        const cuuint32_t box[2] = {128, SK_ROWS};
        const cuuint32_t estride[2] = {1, 1};
        if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(v.qs), gdim, gstride, box, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    void (*kern)(const CUtensorMap, const __half *, const float *, const float *, float *, SkParams, unsigned int *,
                 uint64_t) = nullptr;
    switch (mpad / 8) {
        case 1: kern = skinny_mma_kernel<1>; break;
        case 2: kern = skinny_mma_kernel<2>; break;
        case 3: kern = skinny_mma_kernel<3>; break;
        default: kern = skinny_mma_kernel<4>; break;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(tiles * S));
    cfg.blockDim = dim3(SK_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, qmap, v.d, x, residual, out, P, ctx.status, ctx.wait_ns);
}

}  // namespace tq2
