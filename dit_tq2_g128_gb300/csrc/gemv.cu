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


// ---------------------------------------------------------------------------
// M = 1 decode GEMV.
//
// Lane l of a warp owns 64 consecutive weights (one 16-byte code load, half
// a block) of a 2048-weight chunk; a CTA holds C chunk-warps per row stream
// (C = ceil(K / 2048)) and S = max(1, 8 / C) row streams.  Rows are split
// into contiguous, near-equal ranges over all streams of the grid.  Per
// batch of kP rows a warp issues all code and scale loads before decoding
// (the next batch's loads are issued before the current batch is decoded),
// so that a large part of the weight is in flight from the start.  x is
// copied once per CTA into shared memory, pre-scaled per code position, in
// 64-float segments padded to 68 floats (conflict-free 16-byte reads, zeros
// past K).  The inner loop is branch-free: rows past a stream's range and
// lanes past K read clamped, valid addresses and contribute zero.  The kP
// row partials are reduced across the warp with one halving butterfly; the
// per-(row, chunk) partials meet in shared memory.
constexpr int kP = 4;           // rows per load batch
constexpr int kGvChunk = 2048;  // weights per warp-chunk (32 lanes x 64)
constexpr int kSeg = 68;        // padded floats per 64-weight segment

// (w & MASK) | magic in one LOP3, the magic constant in a register.
template <uint32_t MASK>
__device__ __forceinline__ float mag(uint32_t w, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "n"(MASK), "r"(magic));
    return __uint_as_float(r);
}

// Loop-invariant constants kept in registers (pinned through an opaque move
// so the compiler does not rematerialise them at every use).
struct GvConst {
    uint32_t magic;
    float2 nb[8];  // -(2^23 + 4^pos) for positions (2p, 2p+1)
};

__device__ __forceinline__ float pin(float v) {
    float r;
    asm volatile("mov.b32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ void gv_const_init(GvConst &c) {
    uint32_t m;
    asm volatile("mov.b32 %0, 0x4B000000;" : "=r"(m));
    c.magic = m;
#pragma unroll
    for (int p = 0; p < 8; ++p) c.nb[p] = make_float2(pin(-pos_bias(2 * p)), pin(-pos_bias(2 * p + 1)));
}

// acc += sum_i (c_i - 1) * x_i over one 16-weight code word; xs pre-scaled.
__device__ __forceinline__ float2 dot16c(uint32_t w, const float4 (&xs)[4], const GvConst &k,
                                         float2 acc) {
    const uint32_t w2 = w >> 22;
    const uint32_t mg = k.magic;
    float2 t;
#define TQ2_STEP(P, A, B, XA, XB)                                              \
    t = __fadd2_rn(make_float2(A, B), k.nb[P]);                                \
    acc = __ffma2_rn(t, make_float2(XA, XB), acc);
    TQ2_STEP(0, mag<0x3u>(w, mg), mag<0xCu>(w, mg), xs[0].x, xs[0].y)
    TQ2_STEP(1, mag<0x30u>(w, mg), mag<0xC0u>(w, mg), xs[0].z, xs[0].w)
    TQ2_STEP(2, mag<0x300u>(w, mg), mag<0xC00u>(w, mg), xs[1].x, xs[1].y)
    TQ2_STEP(3, mag<0x3000u>(w, mg), mag<0xC000u>(w, mg), xs[1].z, xs[1].w)
    TQ2_STEP(4, mag<0x30000u>(w, mg), mag<0xC0000u>(w, mg), xs[2].x, xs[2].y)
    TQ2_STEP(5, mag<0x300000u>(w, mg), mag<0x3u>(w2, mg), xs[2].z, xs[2].w)
    TQ2_STEP(6, mag<0xCu>(w2, mg), mag<0x30u>(w2, mg), xs[3].x, xs[3].y)
    TQ2_STEP(7, mag<0xC0u>(w2, mg), mag<0x300u>(w2, mg), xs[3].z, xs[3].w)
#undef TQ2_STEP
    return acc;
}

// Up to kR rows of one warp's stream are loaded at once (all of them, for
// the row counts the launcher picks), then decoded in groups of kP.
template <int kR, int kMaxThreads>
__global__ void __launch_bounds__(kMaxThreads, 1)
gemv_kernel(const uint8_t *__restrict__ qs, const __half *__restrict__ dpl,
            const float *__restrict__ x, const float *residual, float *out, int n, int k, int C,
            int S) {
    extern __shared__ float4 gv_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = warp % C, s = warp / C;
    // contiguous row range of this CTA, then of this stream inside it
    const int R0 = int(int64_t(n) * blockIdx.x / gridDim.x);
    const int R1 = int(int64_t(n) * (blockIdx.x + 1) / gridDim.x);
    const int ra = R0 + (R1 - R0) * s / S, rb = R0 + (R1 - R0) * (s + 1) / S;
    const int kw0 = c * kGvChunk + lane * 64;
    const bool active = kw0 < k;
    const int64_t kq = k / 4, kb = k / kBlockW;
    const int nseg = C * 32;                       // 64-weight segments incl. padding past K
    float *xsm = reinterpret_cast<float *>(gv_smem);
    float *partial = xsm + nseg * kSeg;            // [R1 - R0][C]

    const int kw_ld = active ? kw0 : 0;           // inactive lanes read a valid address
    const uint8_t *qbase = qs + kw_ld / 4;
    const __half *dbase = dpl + kw_ld / kBlockW;
    uint4 w[kR];
    unsigned short dh[kR];
    // rows r .. r+kR-1; rows at or past rb re-read row rb-1 (never used)
    auto load = [&](int r) {
        const uint8_t *q = qbase + int64_t(r) * kq;
        const __half *dd = dbase + int64_t(r) * kb;
        const int last = rb - 1 - r;
#pragma unroll
        for (int u = 0; u < kR; ++u) {
            const int uu = u < last ? u : last;
            w[u] = ldg_stream_u4(q + uu * kq);
            dh[u] = ldg_u16(dd + uu * kb);
        }
    };
    if (ra < rb) load(ra);

    // x -> shared memory, pre-scaled per code position, zero past K.
    for (int i = threadIdx.x; i < nseg * 16; i += blockDim.x) {
        const int seg = i >> 4, q = i & 15;
        const int kk = seg * 64 + 4 * q;
        float4 v = kk < k ? __ldg(reinterpret_cast<const float4 *>(x + kk)) : make_float4(0.f, 0.f, 0.f, 0.f);
        v.x *= pos_scale((4 * q + 0) & 15);
        v.y *= pos_scale((4 * q + 1) & 15);
        v.z *= pos_scale((4 * q + 2) & 15);
        v.w *= pos_scale((4 * q + 3) & 15);
        *reinterpret_cast<float4 *>(xsm + seg * kSeg + 4 * q) = v;
    }
    GvConst kc;
    gv_const_init(kc);
    __syncthreads();

    const float4 *xl = reinterpret_cast<const float4 *>(xsm + (c * 32 + lane) * kSeg);
    for (int r = ra; r < rb; r += kR) {
        if (r != ra) load(r);
#pragma unroll
        for (int g0 = 0; g0 < kR; g0 += kP) {
            const int nv = min(kP, rb - (r + g0));  // warp-uniform
            if (nv <= 0) break;
            float2 acc[kP];
#pragma unroll
            for (int u = 0; u < kP; ++u) acc[u] = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float4 xs[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) xs[j] = xl[4 * q + j];
#pragma unroll
                for (int u = 0; u < kP; ++u) {
                    const uint4 &wu = w[g0 + u];
                    const uint32_t wq = q == 0 ? wu.x : q == 1 ? wu.y : q == 2 ? wu.z : wu.w;
                    if (u < nv) acc[u] = dot16c(wq, xs, kc, acc[u]);
                }
            }
            float v[kP];
#pragma unroll
            for (int u = 0; u < kP; ++u)
                v[u] = (acc[u].x + acc[u].y) *
                       (active ? __half2float(__ushort_as_half(dh[g0 + u])) : 0.f);
            butterfly<kP>(v, lane);
            constexpr int G = 32 / kP;
            if (lane % G == 0) {
                const int u = lane / G;
                if (u < nv) partial[(r + g0 + u - R0) * C + c] = v[0];
            }
        }
    }
    __syncthreads();
    for (int i = R0 + threadIdx.x; i < R1; i += blockDim.x) {
        float sum = 0.f;
        for (int cc = 0; cc < C; ++cc) sum += partial[(i - R0) * C + cc];
        if (residual) sum += residual[i];
        out[i] = sum;
    }
}

}  // namespace

cudaError_t launch_gemv(const void *w_soa, const float *x, const float *residual, float *out,
                        int64_t n, int64_t k, const LaunchCtx &ctx) {
    const int64_t C = (k + kGvChunk - 1) / kGvChunk;
    if (C > 16 || n > INT32_MAX)  // K > 32768: the chunk-looping small-M kernel
        return launch_tpl<1, 2>(w_soa, x, residual, out, 1, n, k, ctx);
    // One CTA per SM, up to 16 warps: C chunk-warps per row stream, S streams.
    const int S = std::max<int>(1, 16 / int(C));
    const int threads = 32 * int(C) * S;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(ctx.num_sms, (n + kP - 1) / kP));
    const int64_t rows_cta = (n + grid - 1) / grid;
    const size_t smem = size_t(C) * 32 * kSeg * 4 + size_t(rows_cta) * size_t(C) * 4;
    if (smem > 200 * 1024) return launch_tpl<1, 2>(w_soa, x, residual, out, 1, n, k, ctx);
    const int64_t rows_stream = (rows_cta + S - 1) / S;
    // deeper register batches when the CTA is small enough to afford them
    auto kern = (threads <= 384 && rows_stream > 12) ? gemv_kernel<16, 384> : gemv_kernel<12, 512>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(std::max<size_t>(smem, 48 * 1024)));
    if (e != cudaSuccess) return e;
    const SoaView v = soa_view(w_soa, n, k);
    kern<<<static_cast<unsigned>(grid), threads, smem, ctx.stream>>>(v.qs, v.d, x, residual, out,
                                                                     int(n), int(k), int(C), S);
    return cudaPeekAtLastError();
}

cudaError_t launch_skinny(const void *w_soa, const float *x, const float *residual, float *out,
                          int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx) {
    if (m == 1) return launch_tpl<1, 2>(w_soa, x, residual, out, m, n, k, ctx);
    if (m == 2) return launch_tpl<2, 1>(w_soa, x, residual, out, m, n, k, ctx);
    return launch_tpl<4, 1>(w_soa, x, residual, out, m, n, k, ctx);
}

}  // namespace tq2
