// Small-M CUDA-core kernels: the M = 1 decode GEMV and the skinny GEMM
// (M up to a few rows), exact f32 products with f32 accumulation.
//
// The pages' decode path is `gemv_tq2_g128_v1` and the skinny prefill path
// `gemm_tq2_g128_v7` ("oxibonsai-kernels 0.1.5
// src/gpu_backend/metal_graph/pipelines.rs", the TQ2_0_g128 pipeline fields);
// both compute the contract of "oxibonsai-image 0.2.2 src/gpu.rs" (module doc
// "Correctness contract").  This kernel is designed for sm_103a:
//
//  * Work split.  A weight row's codes are cut into chunks of 32*WL weights;
//    within a chunk, lane l of a warp owns weights [l*WL, l*WL+WL).  A warp is
//    pinned to one chunk at a time and walks a set of rows, so that one
//    coalesced load per row fetches 32*WL/4 contiguous code bytes, and the
//    lane's slice of x (pre-scaled, see below) stays in registers for all of
//    those rows.  Per-(row, chunk) partial sums go to shared memory and are
//    summed per row at the end (plus the residual).
//  * Decode.  For a 32-bit code word (16 weights, code i at bits 2i), weight
//    i's code is placed into the mantissa of 2^23 by one AND-OR:
//    as_float((w & (3 << 2i)) | 0x4B000000) = 2^23 + c * 4^i (i <= 10; codes
//    11..15 first move down by 22 bits).  Subtracting 2^23 + 4^i gives
//    (c - 1) * 4^i exactly, and multiplying by x * 4^-i (the register copy of
//    x is pre-scaled by that power of two) gives (c - 1) * x exactly, so the
//    only roundings are the f32 additions.  The subtract and the fused
//    multiply-add run as packed f32x2 operations.
//  * Scale.  A lane's WL <= 32 weights sit inside one 128-weight block, so its
//    partial is multiplied by that block's d once.
//  * Reduction.  U = 4 rows (times MR x-rows) are reduced across the warp with
//    a halving butterfly (V/2 + V/4 + ... shuffles instead of 5 per value).
#include <algorithm>
#include <climits>

#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kU = 4;  // rows per unrolled group

__device__ __forceinline__ float pos_scale(int i) {
    // 4^-i for code positions 0..10, 4^-(i-11) for 11..15
    const int e = i <= 10 ? i : i - 11;
    return __int_as_float((127 - 2 * e) << 23);
}

__device__ __forceinline__ constexpr float pos_bias(int i) {
    // 2^23 + 4^i (i <= 10) or 2^23 + 4^(i-11)
    return 8388608.0f + float(1u << (2 * (i <= 10 ? i : i - 11)));
}

// acc += sum_i (c_i - 1) * x_i over the 16 weights of code word w; xs holds
// x_i * 4^-pos(i).
__device__ __forceinline__ float2 dot16(uint32_t w, const float *xs, float2 acc) {
    const uint32_t w2 = w >> 22;
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t src = i <= 10 ? w : w2;
        const int sh = 2 * (i <= 10 ? i : i - 11);
        t[i] = __uint_as_float((src & (3u << sh)) | 0x4B000000u);
    }
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const float2 tt = __fadd2_rn(make_float2(t[2 * p], t[2 * p + 1]),
                                     make_float2(-pos_bias(2 * p), -pos_bias(2 * p + 1)));
        acc = __ffma2_rn(tt, make_float2(xs[2 * p], xs[2 * p + 1]), acc);
    }
    return acc;
}

// Reduce V values per lane across the warp; afterwards lane L (with
// L % (32/V) == 0) holds the total of value L / (32/V) in v[0].
template <int V>
__device__ __forceinline__ void butterfly(float (&v)[V], int lane) {
    int cnt = V;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (cnt > 1) {
            const int half = cnt / 2;
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < half) {
                    const float give = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
                }
            }
            cnt = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
}

template <int MR, int WPL>
__global__ void __launch_bounds__(kThreads, 2)
smallm_kernel(const uint8_t *__restrict__ qs, const __half *__restrict__ dpl,
              const float *__restrict__ x, const float *residual, float *out, int m, int n,
              int k, int C, int Cw, int S, int rps) {
    constexpr int WL = WPL * 16;  // weights per lane per row
    constexpr int CH = 32 * WL;   // weights per chunk
    constexpr int V = kU * MR;
    static_assert(V <= 32 && (V & (V - 1)) == 0, "V must be a power of two <= 32");
    extern __shared__ float partial[];  // [R][C][MR]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = S * rps;
    const int row0 = blockIdx.x * R;
    const int m0 = blockIdx.y * MR;
    const int rows_here = min(R, n - row0);
    const int64_t kq = k / 4, kb = k / kBlockW;

    if (warp < Cw * S) {
        const int cw = warp % Cw, s = warp / Cw;
        for (int c = cw; c < C; c += Cw) {
            const int kw0 = c * CH + lane * WL;
            const bool active = kw0 < k;
            float xs[MR][WL];
#pragma unroll
            for (int mm = 0; mm < MR; ++mm) {
                const bool ok = active && (m0 + mm) < m;
                const float4 *xp = reinterpret_cast<const float4 *>(x + int64_t(m0 + mm) * k + kw0);
#pragma unroll
                for (int q = 0; q < WL / 4; ++q) {
                    const float4 v = ok ? __ldg(xp + q) : make_float4(0.f, 0.f, 0.f, 0.f);
                    xs[mm][4 * q + 0] = v.x * pos_scale((4 * q + 0) & 15);
                    xs[mm][4 * q + 1] = v.y * pos_scale((4 * q + 1) & 15);
                    xs[mm][4 * q + 2] = v.z * pos_scale((4 * q + 2) & 15);
                    xs[mm][4 * q + 3] = v.w * pos_scale((4 * q + 3) & 15);
                }
            }
            const uint8_t *qrow = qs + int64_t(row0) * kq + kw0 / 4;
            const __half *drow = dpl + int64_t(row0) * kb + kw0 / kBlockW;
            for (int r = s; r < rows_here; r += S * kU) {
                uint32_t w[kU][WPL];
                float d[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int rr = r + u * S;
                    if (active && rr < rows_here) {
                        const uint8_t *p = qrow + int64_t(rr) * kq;
                        if constexpr (WPL == 2) {
                            const uint2 v = ldg_stream_u2(p);
                            w[u][0] = v.x;
                            w[u][1] = v.y;
                        } else {
                            w[u][0] = __ldg(reinterpret_cast<const unsigned int *>(p));
                        }
                        d[u] = __half2float(__ushort_as_half(ldg_u16(drow + int64_t(rr) * kb)));
                    } else {
#pragma unroll
                        for (int j = 0; j < WPL; ++j) w[u][j] = 0x55555555u;  // all-zero weights
                        d[u] = 0.f;
                    }
                }
                float v[V];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
#pragma unroll
                    for (int mm = 0; mm < MR; ++mm) {
                        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                        for (int j = 0; j < WPL; ++j) acc = dot16(w[u][j], &xs[mm][16 * j], acc);
                        v[u * MR + mm] = (acc.x + acc.y) * d[u];
                    }
                }
                butterfly<V>(v, lane);
                constexpr int G = 32 / V;
                if (lane % G == 0) {
                    const int idx = lane / G;
                    const int u = idx / MR, mm = idx % MR;
                    const int rr = r + u * S;
                    if (rr < rows_here) partial[(int64_t(rr) * C + c) * MR + mm] = v[0];
                }
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < rows_here * MR; i += kThreads) {
        const int mm = i / rows_here, rr = i % rows_here;
        const int row = m0 + mm;
        if (row >= m) continue;
        float sum = 0.f;
        for (int c = 0; c < C; ++c) sum += partial[(int64_t(rr) * C + c) * MR + mm];
        const int64_t o = int64_t(row) * n + row0 + rr;
        if (residual) sum += residual[o];
        out[o] = sum;
    }
}

template <int MR, int WPL>
cudaError_t launch_tpl(const void *w_soa, const float *x, const float *residual, float *out,
                       int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx) {
    constexpr int CH = 32 * 16 * WPL;
    const int C = static_cast<int>((k + CH - 1) / CH);
    // Chunk-parallel warps Cw (a divisor of C, at most 8) and row streams S
    // = 8 / Cw, choosing the split that keeps the most warps busy.
    int Cw = 1, best = 0;
    for (int cand = 1; cand <= kWarps; ++cand) {
        if (C % cand) continue;
        const int busy = cand * (kWarps / cand);
        if (busy >= best) best = busy, Cw = cand;
    }
    const int S = kWarps / Cw;
    // Rows per stream: aim at ~3 resident CTAs per SM in one wave.
    const int64_t target_ctas = int64_t(ctx.num_sms) * 3;
    int64_t rps = (n + S * target_ctas - 1) / (S * target_ctas);
    rps = std::max<int64_t>(1, std::min<int64_t>(rps, 16));
    const int64_t max_smem = 200 * 1024;
    while (rps > 1 && S * rps * C * MR * 4 > max_smem) --rps;
    const int64_t R = S * rps;
    const size_t smem = size_t(R) * C * MR * 4;
    if (smem > size_t(max_smem)) return cudaErrorInvalidValue;  // K beyond ~1.6M (MR=1)
    if (int64_t(k) > INT32_MAX || n > INT32_MAX || m > INT32_MAX) return cudaErrorInvalidValue;
    auto kern = smallm_kernel<MR, WPL>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const SoaView v = soa_view(w_soa, n, k);
    dim3 grid(static_cast<unsigned>((n + R - 1) / R), static_cast<unsigned>((m + MR - 1) / MR));
    if (grid.y > 65535) return cudaErrorInvalidValue;
    kern<<<grid, kThreads, smem, ctx.stream>>>(v.qs, v.d, x, residual, out, int(m), int(n), int(k),
                                              C, Cw, S, int(rps));
    return cudaPeekAtLastError();
}


constexpr int kGvChunk = 2048;  // weights per warp-chunk (32 lanes x 64)

// ---------------------------------------------------------------------------
// M = 1 decode GEMV (K <= 16384): bulk-copy streaming + integer dot products.
//
// Memory side.  One CTA per SM owns a contiguous row range, i.e. a contiguous
// range of the qs plane.  One producer thread streams it into a shared-memory
// ring with cp.async.bulk (four rows per stage, completion counted on an
// mbarrier), so the bytes in flight do not depend on per-thread load slots.
//
// Arithmetic.  x is quantised once per CTA, per 64-weight segment, to a signed
// fixed-point integer X = rint(x * 2^22 / s) with s = max |x| of the segment
// (|X| <= 2^22), held as three 8-bit limbs (top limb signed).  For one 32-bit
// code word (16 weights, code i at bits 2i), (w >> 2t) & 0x03030303 gathers
// the codes of weights t, t+4, t+8, t+12 into four bytes, and dp4a multiplies
// them with the matching limb bytes and accumulates exactly in int32.  Per row
// and segment, sum_i (c_i - 1) X_i = sum c*X - sum X is exact; one conversion
// to f32 and one multiply by s * 2^-22 * d finish the segment.  Per weight this
// is 3/4 dp4a + 7/16 shift/logic operations instead of the 2 operations of an
// exact-f32 decode.  The only error is the quantisation of x: per element at
// most 2^-22 * s (s the segment's max |x|: half a step of 2^-22 * s plus the
// rounding of the reciprocal); all sums are exact until the final f32 sum over
// segments.
// Consumer warps take (row, 2048-weight chunk) items round-robin: each lane
// owns one 64-weight segment of the chunk, reads its 16 code bytes from the
// ring and its segment's limbs from shared memory, and the row's 32 lane
// partials are reduced with shuffles.  Per-(row, chunk) partials meet in
// shared memory and are summed per row at the end (plus the residual).

constexpr int kSegWords = 52;  // 48 limb words per segment, padded (conflict-free 16-byte reads)
constexpr int kGvThreads = 512;    // two CTAs per SM (registers, threads and shared memory)
constexpr int kGvMaxSegs = 256;    // 64-weight segments of x: K <= 16384

__device__ __forceinline__ void bulk_g2s_gv(uint32_t dst, const void *src, uint32_t bytes,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx_gv(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

struct GvsParams {
    int n, k, C;       // rows, K, 2048-weight chunks per row
    int rbase, rextra; // CTA b owns rbase (+1 if b < rextra) rows starting at b*rbase + min(b, rextra)
    // shared-memory offsets (bytes), computed on the host
    uint32_t off_limbs, off_scale, off_sum, off_d, off_partial, off_bar;
    int rs;            // rows per stage
    int ns;            // ring slots
    int consumers;     // consumer warps = groups * C
    int groups;        // consumer warp groups; group g owns the ring slots s with s % groups == g
    int rows_cta;      // max rows of a CTA (partial buffer size)
};

template <int RS>  // rows per stage
__global__ void __launch_bounds__(kGvThreads, 2)
gemv_stream_kernel(const uint8_t *__restrict__ qs, const __half *__restrict__ dpl,
                   const float *__restrict__ x, const float *residual, float *out, GvsParams P,
                   unsigned int *status, uint64_t wait_ns) {
    extern __shared__ __align__(128) uint8_t gvs_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = P.k, C = P.C;
    const int64_t kq = k / 4, kb = k / kBlockW;
    const int nseg = C * 32;                 // 64-weight segments incl. padding past K
    const int consumers = P.consumers;       // warps 0 .. consumers-1
    const int pwarp = int(blockDim.x >> 5) - 1;  // the producer: the last warp
    const int b = int(blockIdx.x);
    const int R0 = b * P.rbase + min(b, P.rextra);
    const int rows = P.rbase + (b < P.rextra ? 1 : 0);
    const int nstages = (rows + P.rs - 1) / P.rs;
    const bool dbulk = (kb % 8) == 0;  // row scales travel with their stage (16-byte multiples)
    const uint32_t code_bytes = uint32_t(P.rs * kq);
    const uint32_t stage_bytes = code_bytes + (dbulk ? uint32_t(P.rs * kb * 2) : 0u);

    // shared memory: [ring][limbs][seg scale][seg sum X][d rows][partials][barriers]
    uint8_t *ring = gvs_smem;
    uint32_t *limbs = reinterpret_cast<uint32_t *>(gvs_smem + P.off_limbs);
    float *sscale = reinterpret_cast<float *>(gvs_smem + P.off_scale);
    int *ssum = reinterpret_cast<int *>(gvs_smem + P.off_sum);
    __half *dsm = reinterpret_cast<__half *>(gvs_smem + P.off_d);
    float *partial = reinterpret_cast<float *>(gvs_smem + P.off_partial);
    uint64_t *full = reinterpret_cast<uint64_t *>(gvs_smem + P.off_bar);
    uint64_t *empty = full + P.ns;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + P.ns);
    const uint32_t ring_addr = smem_u32(ring);

    // barriers: the lanes of warp 0 initialise them in parallel
    if (warp == 0) {
        for (int i = lane; i < P.ns; i += 32) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 32 * C);
        }
        if (lane == 0) *abort_flag = 0;
        fence_proxy_async_smem();   // the inits are visible to the copy engine
    }
    __syncthreads();
    // ---- producer warp, part 1: the first ring-full of stages needs no slot to
    // free up; its 32 lanes issue those copies in parallel
    const bool producer = warp == pwarp && lane == 0;
    const uint8_t *src = qs + int64_t(R0) * kq;
    const __half *dsrc_rows = dpl + int64_t(R0) * kb;
    auto issue = [&](int st) {
        const int slot = st % P.ns;
        const int r = min(P.rs, rows - st * P.rs);
        const uint32_t bytes = uint32_t(r * kq);
        const uint32_t dbytes = dbulk ? uint32_t(r * kb * 2) : 0u;
        const uint32_t dst = ring_addr + uint32_t(slot) * stage_bytes;
        mbar_expect_tx_gv(&full[slot], bytes + dbytes);
        bulk_g2s_gv(dst, src + int64_t(st) * code_bytes, bytes, &full[slot]);
        if (dbytes)
            bulk_g2s_gv(dst + code_bytes, dsrc_rows + int64_t(st) * P.rs * kb, dbytes, &full[slot]);
    };
    // The weights go to L2 before waiting for the preceding kernel.  A
    // prefetch cannot leave stale data behind (L2 is the point of coherence,
    // and the copies below read through it after the wait).
    if (warp == pwarp) {
        for (int st = lane; st < nstages; st += 32) {
            const int r = min(P.rs, rows - st * P.rs);
            bulk_prefetch_l2(src + int64_t(st) * code_bytes, uint32_t(r * kq));
            if (dbulk) bulk_prefetch_l2(dsrc_rows + int64_t(st) * P.rs * kb, uint32_t(r * kb * 2));
        }
    }
    // Everything a preceding kernel may have written (x, the weights, out and
    // the residual) is touched only after this.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int first = min(nstages, P.ns);
    if (warp == pwarp)
        for (int st = lane; st < first; st += 32) issue(st);
    // ---- everyone: quantise x per 64-weight segment.  Item (segment, word q,
    // group t) loads the four consecutive elements 16q + 4t + m (m = 0..3) in
    // one 16-byte read; 16 items per segment find its max |x| with shuffles.
    // A 4 x 4 byte transpose among the four items of word q then leaves item
    // (q, t) with the limb words whose byte m holds weight 16q + 4m + t, the
    // order in which the dot products unpack the codes.  Items are taken three
    // passes at a time, loads first.  The producer warp takes no items (it is
    // busy issuing the copies).
    const int nthr = nseg * 16;  // a multiple of 512: warp-uniform bounds
    const int nq = int(blockDim.x) - 32;  // item threads (a multiple of 32)
#pragma unroll 1
    for (int p0 = 0; warp != pwarp && p0 * nq < nthr; p0 += 3) {  // warp-uniform
        float4 xv[3];
#pragma unroll
        for (int pp = 0; pp < 3; ++pp) {
            const int qi = int(threadIdx.x) + (p0 + pp) * nq;
            const int kk = (qi >> 4) * 64 + 16 * ((qi >> 2) & 3) + 4 * (qi & 3);
            xv[pp] = (qi < nthr && kk < k) ? __ldg(reinterpret_cast<const float4 *>(x + kk))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // the three items' shuffle chains are interleaved step by step
        float m[3], xe[3][4];
#pragma unroll
        for (int pp = 0; pp < 3; ++pp) {
            xe[pp][0] = xv[pp].x; xe[pp][1] = xv[pp].y; xe[pp][2] = xv[pp].z; xe[pp][3] = xv[pp].w;
            m[pp] = fmaxf(fmaxf(fabsf(xe[pp][0]), fabsf(xe[pp][1])), fmaxf(fabsf(xe[pp][2]), fabsf(xe[pp][3])));
        }
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1)
#pragma unroll
            for (int pp = 0; pp < 3; ++pp) m[pp] = fmaxf(m[pp], __shfl_xor_sync(0xffffffffu, m[pp], o));
        uint32_t r[3][3];  // item pp, limb l: weight 16q + 4t + mm in byte mm
        int sx[3];
#pragma unroll
        for (int pp = 0; pp < 3; ++pp) {
            // 2^22 / s: the correctly rounded reciprocal times 2^22 (exact
            // scaling), i.e. the correctly rounded quotient
            const float inv = m[pp] > 0.f ? __frcp_rn(m[pp]) * 4194304.0f : 0.f;
            r[pp][0] = r[pp][1] = r[pp][2] = 0;
            sx[pp] = 0;
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
                // |X| <= 2^22 (the rounded reciprocal may overshoot by half an ulp)
                const int X = max(-4194304, min(4194304, __float2int_rn(xe[pp][mm] * inv)));
                sx[pp] += X;
                r[pp][0] |= uint32_t(X & 0xFF) << (8 * mm);
                r[pp][1] |= uint32_t((X >> 8) & 0xFF) << (8 * mm);
                r[pp][2] |= uint32_t((X >> 16) & 0xFF) << (8 * mm);
            }
        }
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1)
#pragma unroll
            for (int pp = 0; pp < 3; ++pp) sx[pp] += __shfl_xor_sync(0xffffffffu, sx[pp], o);
        // transpose: item t gathers byte t of the four items' words of word q
        const int qt = int(threadIdx.x) & 3;
        uint32_t h[3][3];
#pragma unroll
        for (int pp = 0; pp < 3; ++pp)
#pragma unroll
            for (int l = 0; l < 3; ++l) {
                const uint32_t o1 = __shfl_xor_sync(0xffffffffu, r[pp][l], 1);
                h[pp][l] = (qt & 1) ? __byte_perm(r[pp][l], o1, 0x3715) : __byte_perm(r[pp][l], o1, 0x6240);
            }
#pragma unroll
        for (int pp = 0; pp < 3; ++pp)
#pragma unroll
            for (int l = 0; l < 3; ++l) {
                const uint32_t o2 = __shfl_xor_sync(0xffffffffu, h[pp][l], 2);
                r[pp][l] = (qt & 2) ? __byte_perm(h[pp][l], o2, 0x3276) : __byte_perm(h[pp][l], o2, 0x5410);
            }
#pragma unroll
        for (int pp = 0; pp < 3; ++pp) {
            const int qi = int(threadIdx.x) + (p0 + pp) * nq;
            if (qi < nthr) {
                const int qseg = qi >> 4, qq = (qi >> 2) & 3;
                uint32_t *lw = limbs + qseg * kSegWords + (qq * 4 + qt) * 3;
                lw[0] = r[pp][0];
                lw[1] = r[pp][1];
                lw[2] = r[pp][2];
                if ((qi & 15) == 0) {
                    sscale[qseg] = m[pp] * (1.0f / 4194304.0f);  // s * 2^-22
                    ssum[qseg] = sx[pp];
                }
            }
        }
    }
    if (!dbulk) {
        const unsigned short *dsrc = reinterpret_cast<const unsigned short *>(dpl + int64_t(R0) * kb);
        unsigned short *ddst = reinterpret_cast<unsigned short *>(dsm);
        for (int64_t i = threadIdx.x; i < int64_t(rows) * kb; i += blockDim.x) ddst[i] = dsrc[i];
    }
    __syncthreads();

    // Programmatic dependent launch: once this CTA holds x and has its
    // weight copies in flight, the next kernel of the stream may start
    // launching.  Two CTAs of this kernel fit on one SM, so the next call's
    // set-up and weight prefetch overlap this call's arithmetic (which needs
    // no memory bandwidth); the next call reads nothing a predecessor may
    // write before its own griddepcontrol.wait.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (producer) {
        // ---- producer, part 2: refill slots as the consumers release them
        for (int st = P.ns; st < nstages; ++st) {
            const int slot = st % P.ns, u = st / P.ns;
            if (!mbar_wait_bounded(&empty[slot], (u - 1) & 1, wait_ns, status)) {
                *abort_flag = 1;
                break;
            }
            if (*abort_flag) break;
            issue(st);
        }
        // every copy issued must land before the CTA exits: the last round of each slot
        const uint64_t drain = wait_ns > 1000000000ull ? wait_ns : 1000000000ull;
        for (int st = max(0, nstages - P.ns); st < nstages; ++st)
            mbar_wait_bounded(&full[st % P.ns], (st / P.ns) & 1, drain, status);
    }
    if (warp < consumers) {
        // Warp w takes chunk w % C of the stages st = g, g + groups, ... (g = w / C).
        // The ring size is a multiple of `groups`, so every slot is only ever
        // touched by one group, in stage order: no warp can wait on a slot's
        // next round before the group released the current one.
        const int g = warp / C, c = warp % C;
        const int seg = c * 32 + lane;
        const int kw0 = seg * 64;
        const bool active = kw0 < k;
        const int kw_rd = active ? kw0 : 0;
        for (int st = g; st < nstages; st += P.groups) {
            const int slot = st % P.ns, u = st / P.ns;
            if (!mbar_wait_bounded(&full[slot], u & 1, wait_ns, status)) {
                *abort_flag = 1;
                break;
            }
            if (*abort_flag) break;
            const int r0 = st * P.rs;                 // first row (CTA-relative) of the stage
            const int nv = min(P.rs, rows - r0);      // warp-uniform, >= 1
            const uint8_t *base = ring + size_t(slot) * stage_bytes + kw_rd / 4;
            const __half *sd = dbulk ? reinterpret_cast<const __half *>(ring + size_t(slot) * stage_bytes + code_bytes)
                                     : dsm + int64_t(r0) * kb;  // this stage's row scales
            // each lane's 16 code bytes of a row in one conflict-free 16-byte read
            uint4 cw[RS];
#pragma unroll
            for (int uu = 0; uu < RS; ++uu)
                cw[uu] = *reinterpret_cast<const uint4 *>(base + size_t(uu < nv ? uu : nv - 1) * kq);
            int a0[RS], a1[RS], a2[RS];
#pragma unroll
            for (int uu = 0; uu < RS; ++uu) a0[uu] = a1[uu] = a2[uu] = 0;
            const uint4 *lw = reinterpret_cast<const uint4 *>(limbs + seg * kSegWords);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                // limb words (q, t, l) for t = 0..3, l = 0..2: 12 words
                const uint4 L0 = lw[3 * q + 0], L1 = lw[3 * q + 1], L2 = lw[3 * q + 2];
                const uint32_t lv[12] = {L0.x, L0.y, L0.z, L0.w, L1.x, L1.y, L1.z, L1.w,
                                         L2.x, L2.y, L2.z, L2.w};
#pragma unroll
                for (int uu = 0; uu < RS; ++uu) {
                    const uint32_t wq = q == 0 ? cw[uu].x : q == 1 ? cw[uu].y : q == 2 ? cw[uu].z : cw[uu].w;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const uint32_t v = (wq >> (2 * t)) & 0x03030303u;
                        a0[uu] = dp4a_uu(v, lv[3 * t + 0], a0[uu]);
                        a1[uu] = dp4a_uu(v, lv[3 * t + 1], a1[uu]);
                        a2[uu] = dp4a_us(v, lv[3 * t + 2], a2[uu]);
                    }
                }
            }
            // every lane has read its codes: release this chunk's share of the slot
            mbar_arrive(&empty[slot]);
            const float sc = active ? sscale[seg] : 0.f;
            const int sx = active ? ssum[seg] : 0;
            float v[RS];
#pragma unroll
            for (int uu = 0; uu < RS; ++uu) {
                const int ur = uu < nv ? uu : nv - 1;
                const int tot = a2[uu] * 65536 + a1[uu] * 256 + a0[uu] - sx;
                const float d = __half2float(sd[int64_t(ur) * kb + kw_rd / kBlockW]);
                v[uu] = float(tot) * (sc * d);
            }
            butterfly<RS>(v, lane);
            constexpr int G = 32 / RS;
            if (lane % G == 0) {
                const int uu = lane / G;
                if (uu < nv) partial[(r0 + uu) * C + c] = v[0];
            }
        }
    }
    __syncthreads();
    if (*abort_flag) return;
    for (int i = threadIdx.x; i < rows; i += blockDim.x) {
        float sum = 0.f;
        for (int cc = 0; cc < C; ++cc) sum += partial[i * C + cc];
        if (residual) sum += residual[R0 + i];
        out[R0 + i] = sum;
    }
}

}  // namespace

cudaError_t launch_gemv_stream(const void *w_soa, const float *x, const float *residual,
                               float *out, int64_t n, int64_t k, const LaunchCtx &ctx) {
    const int C = int((k + kGvChunk - 1) / kGvChunk);
    const int64_t kq = k / 4, kb = k / kBlockW;
    if (C > 30) return cudaErrorNotSupported;
    GvsParams P;
    P.n = int(n);
    P.k = int(k);
    P.C = C;
    P.rs = 4;
    const int threads = kGvThreads;  // consumer warps, the producer warp, one spare
    P.groups = std::max(1, (threads / 32 - 2) / C);  // consumer warp groups of C warps (one per chunk)
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(ctx.num_sms, (n + P.rs - 1) / P.rs));
    P.rbase = int(n / grid);
    P.rextra = int(n % grid);
    P.rows_cta = P.rbase + (P.rextra ? 1 : 0);
    const int nseg = C * 32;
    const bool dbulk = (kb % 8) == 0;  // scales travel with their stage in the ring
    const size_t stage_bytes = size_t(P.rs) * kq + (dbulk ? size_t(P.rs) * kb * 2 : 0);
    const size_t dsm_bytes = dbulk ? 0 : size_t((int64_t(P.rows_cta) * kb + 7) & ~int64_t(7)) * 2;
    const size_t lwords = size_t(nseg) * kSegWords;
    if (nseg > kGvMaxSegs) return cudaErrorNotSupported;
    const size_t fixed = lwords * 4 + size_t(nseg) * 8 + dsm_bytes +
                         size_t((P.rows_cta * C + 1) & ~1) * 4;
    const size_t budget = 108 * 1024;  // two CTAs per SM
    if (fixed + stage_bytes + 64 * 16 + 32 > budget) return cudaErrorNotSupported;
    // ring: enough slots for all of a CTA's stages if shared memory allows (no
    // refill round trips), as a multiple of the group count
    const int nst = (P.rows_cta + P.rs - 1) / P.rs;
    const int max_slots = int(std::min<size_t>(64, (budget - fixed - 64 * 16 - 32) / stage_bytes));
    int ns = std::min(max_slots, ((nst + P.groups - 1) / P.groups) * P.groups);
    ns = (ns / P.groups) * P.groups;
    if (ns < P.groups) {  // fewer slots than groups: shrink the groups
        P.groups = std::max(1, max_slots);
        ns = P.groups;
    }
    P.ns = ns;
    P.consumers = P.groups * C;
    P.off_limbs = uint32_t(size_t(ns) * stage_bytes);
    P.off_scale = uint32_t(P.off_limbs + lwords * 4);
    P.off_sum = uint32_t(P.off_scale + size_t(nseg) * 4);
    P.off_d = uint32_t(P.off_sum + size_t(nseg) * 4);
    P.off_partial = uint32_t(P.off_d + dsm_bytes);
    P.off_bar = uint32_t(P.off_partial + size_t((P.rows_cta * C + 1) & ~1) * 4);
    const size_t smem = size_t(P.off_bar) + size_t(2 * ns) * 8 + 16;
    cudaError_t e = cudaFuncSetAttribute(gemv_stream_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // the largest shared-memory carve-out, so that two CTAs fit on an SM
    e = cudaFuncSetAttribute(gemv_stream_kernel<4>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    const SoaView v = soa_view(w_soa, n, k);
    // programmatic dependent launch (see the kernel): the launch may begin
    // before the preceding kernel of the stream has finished
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_stream_kernel<4>, v.qs, v.d, x, residual, out, P, ctx.status,
                              ctx.wait_ns);
}

cudaError_t launch_gemv(const void *w_soa, const float *x, const float *residual, float *out,
                        int64_t n, int64_t k, const LaunchCtx &ctx) {
    if (k <= 16384 && n <= INT32_MAX) {
        cudaError_t e = launch_gemv_stream(w_soa, x, residual, out, n, k, ctx);
        if (e != cudaErrorNotSupported) return e;
        (void)cudaGetLastError();
    }
    // very long rows: the chunk-looping small-M kernel (exact f32)
    return launch_tpl<1, 2>(w_soa, x, residual, out, 1, n, k, ctx);
}

cudaError_t launch_skinny(const void *w_soa, const float *x, const float *residual, float *out,
                          int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx) {
    if (m == 1) return launch_tpl<1, 2>(w_soa, x, residual, out, m, n, k, ctx);
    if (m == 2) return launch_tpl<2, 1>(w_soa, x, residual, out, m, n, k, ctx);
    return launch_tpl<4, 1>(w_soa, x, residual, out, m, n, k, ctx);
}

}  // namespace tq2
