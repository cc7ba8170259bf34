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


constexpr int kGvLaneW = 32;                 // weights per lane: a quarter of a 128-weight block
constexpr int kGvChunk = 32 * kGvLaneW;      // weights per warp-chunk (1024)
// Consumer warps per CTA: up to 12 (three per scheduler, up to 72 registers
// per thread with two CTAs per SM).  With 16 (56 registers) the per-row code
// spends more instructions on register moves: 6.67 vs 6.51 us at K=4096,
// N=12288.
constexpr int kGvMaxConsumers = 12;

// ---------------------------------------------------------------------------
// M = 1 decode GEMV (K <= 12288): bulk-copy streaming + integer dot products.
//
// Memory side.  One CTA per SM owns a contiguous row range, i.e. a contiguous
// range of the qs plane (with swiglu: a feature range, whose gate rows and up
// rows are two ranges).  The producer warp streams it into a shared-memory
// ring with cp.async.bulk (RS rows per stage with their block scales, RS in
// 2..8 chosen per shape so that the stages balance across the consumer groups;
// completion counted on an mbarrier), so the bytes in flight do not depend on
// per-thread load slots.  Before waiting for the preceding kernel of the
// stream it prefetches all of it into L2.  x arrives once per CTA by a 2-D
// tensor copy with the 128-byte swizzle.
//
// Arithmetic.  A row is cut into 1024-weight chunks; consumer warp w owns chunk
// w % C of every row of the stages it takes, and lane l of it the 32 weights
// [1024 c + 32 l, +32), i.e. a fixed slice of x, inside 128-weight block l / 4.
// Each lane quantises its own slice once, to a signed fixed-point integer
// X = rint(x * 2^22 / s) with s = max |x| over the slice's 128-weight block
// (the four lanes 4j .. 4j+3 agree on it by two shuffles; |X| <= 2^22), held in
// registers as three 8-bit limbs (top limb signed): no shared-memory table and
// no block-wide barrier between the quantisation and the dot products.  For one
// 32-bit code word (16 weights, code i at bits 2i), (w >> 2t) & 0x03030303
// gathers the codes of weights t, t+4, t+8, t+12 into four bytes, and dp4a
// multiplies them with the matching limb bytes and accumulates exactly in
// int32.  Per row and lane, T = sum_i (c_i - 1) X_i = sum c*X - sum X is exact
// (|T| <= 2^28).  The rows of a stage are then reduced over the warp by a
// halving butterfly: its first two levels add the four lanes of one block,
// which share s, as integers (exact, |sum| <= 2^30); each value left is
// converted once to f32 and multiplied by s * 2^-22 * d of its block; float
// levels finish the sum over the chunk.  Per weight this is 3/4 dp4a + 7/16
// shift/logic operations instead of the 2 operations of an exact-f32 decode.
// The error is the quantisation of x (per element at most 2^-22 * s: half a
// step plus the rounding of the reciprocal), the rounding of each block's
// integer sum to f32 and the f32 sums over blocks.  Per-(row, chunk) partials
// meet in shared memory and are summed per row at the end (plus the residual).

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

__device__ __forceinline__ void tma_load_2d_gv(uint32_t dst, const CUtensorMap *map, int cx, int cy,
                                               uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cx), "r"(cy), "r"(smem_u32(bar))
        : "memory");
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
    int n, k, C;       // rows, K, 1024-weight chunks per row
    int rbase, rextra; // CTA b owns rbase (+1 if b < rextra) rows (features, with swiglu)
                       // starting at b*rbase + min(b, rextra)
    int swiglu, f;     // fused gate/up: rows [0, f) gate, [f, 2f) up; out[i] = silu(g_i) * u_i
    int xbox_rows, nxbox;  // x arrives as nxbox tensor boxes of xbox_rows 128-byte rows
    // shared-memory offsets (bytes, from the 1024-aligned base), computed on the host
    uint32_t off_ring, off_partial, off_bar;
    int rs;            // rows per stage
    int ns;            // ring slots
    int consumers;     // consumer warps = groups * C
    int groups;        // consumer warp groups; group g owns the ring slots s with s % groups == g
    int rows_cta;      // max rows of a CTA (partial buffer size)
    int early;         // resident weights (wide-lane kernel): the first ring of stages is
                       // copied before the dependency wait (no unfinished work writes them)
};

// RS: rows per stage; DBULK: the rows' block scales travel with their stage in
// the ring (K a multiple of 1024: 16-byte multiples), else they are read from
// global memory
template <int RS, bool DBULK, int MAXC>
__global__ void __launch_bounds__(32 * (MAXC + 1), 2)
gemv_stream_kernel(const __grid_constant__ CUtensorMap xmap, const uint8_t *__restrict__ qs,
                   const __half *__restrict__ dpl, const float *residual, float *out, GvsParams P,
                   unsigned int *status, uint64_t wait_ns) {
    extern __shared__ __align__(128) uint8_t gvs_raw[];
    // the 128-byte swizzle of the x tile repeats every 1024 bytes: align the base
    uint8_t *gvs_smem = gvs_raw + ((1024u - (smem_u32(gvs_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = P.k, C = P.C;
    const int64_t kq = k / 4, kb = k / kBlockW;
    const int consumers = P.consumers;           // warps 0 .. consumers-1
    const int pwarp = int(blockDim.x >> 5) - 1;  // the producer: the last warp
    const int b = int(blockIdx.x);
    const int R0 = b * P.rbase + min(b, P.rextra);  // first row (first feature, with swiglu)
    const int nf = P.rbase + (b < P.rextra ? 1 : 0);
    // The CTA's row list: rows R0 .. R0+nf-1, or with swiglu the gate rows
    // R0 .. R0+nf-1 followed by the matching up rows f+R0 .. f+R0+nf-1.
    const int rows = P.swiglu ? 2 * nf : nf;
    auto real_row = [&](int i) { return (P.swiglu && i >= nf) ? P.f + R0 + (i - nf) : R0 + i; };
    const int nstages = (rows + RS - 1) / RS;
    constexpr bool dbulk = DBULK;
    const uint32_t code_bytes = uint32_t(RS * kq);
    const uint32_t stage_bytes = code_bytes + (dbulk ? uint32_t(RS * kb * 2) : 0u);

    // shared memory: [x][ring][partials][barriers][abort flag]
    const float *xs = reinterpret_cast<const float *>(gvs_smem);
    uint8_t *ring = gvs_smem + P.off_ring;
    float *partial = reinterpret_cast<float *>(gvs_smem + P.off_partial);
    uint64_t *full = reinterpret_cast<uint64_t *>(gvs_smem + P.off_bar);
    uint64_t *empty = full + P.ns;
    uint64_t *xbar = empty + P.ns;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(xbar + 1);
    const uint32_t ring_addr = smem_u32(ring);

    // barriers: the lanes of warp 0 initialise them in parallel
    if (warp == 0) {
        for (int i = lane; i < P.ns; i += 32) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 32 * C);
        }
        if (lane == 0) {
            mbar_init(xbar, 1);
            *abort_flag = 0;
        }
        fence_proxy_async_smem();   // the inits are visible to the copy engine
    }
    __syncthreads();
    const bool producer = warp == pwarp && lane == 0;
    // A stage's rows are consecutive in the list; they are consecutive weight
    // rows except where a swiglu stage crosses from the gate to the up rows:
    // there the stage is copied (or prefetched) as two pieces.
    auto pieces = [&](int st, auto &&fn) {
        const int lo = st * RS, hi = min(lo + RS, rows);
        if (P.swiglu && lo < nf && hi > nf) {
            fn(lo, nf - lo, 0);
            fn(nf, hi - nf, nf - lo);
        } else {
            fn(lo, hi - lo, 0);
        }
    };
    auto issue = [&](int st) {
        const int slot = st % P.ns;
        const int r = min(RS, rows - st * RS);
        const uint32_t dst = ring_addr + uint32_t(slot) * stage_bytes;
        mbar_expect_tx_gv(&full[slot], uint32_t(r) * (uint32_t(kq) + (dbulk ? uint32_t(kb * 2) : 0u)));
        pieces(st, [&](int i0, int cnt, int off) {
            const int64_t row = real_row(i0);
            bulk_g2s_gv(dst + uint32_t(off) * uint32_t(kq), qs + row * kq, uint32_t(cnt * kq), &full[slot]);
            if (dbulk)
                bulk_g2s_gv(dst + code_bytes + uint32_t(off) * uint32_t(kb * 2), dpl + row * kb,
                            uint32_t(cnt * kb * 2), &full[slot]);
        });
    };
    // The weights go to L2 before waiting for the preceding kernel.  A
    // prefetch cannot leave stale data behind (L2 is the point of coherence,
    // and the copies below read through it after the wait).
    if (warp == pwarp) {
        for (int st = lane; st < nstages; st += 32) {
            pieces(st, [&](int i0, int cnt, int) {
                const int64_t row = real_row(i0);
                bulk_prefetch_l2(qs + row * kq, uint32_t(cnt * kq));
                if (dbulk) bulk_prefetch_l2(dpl + row * kb, uint32_t(cnt * kb * 2));
            });
        }
    }
    // Everything a preceding kernel may have written (x, the weights, out and
    // the residual) is touched only after this.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Programmatic dependent launch: the next kernel of the stream may start
    // launching once every thread of this CTA has passed its trigger below
    // (the producer after issuing x and the first stages, consumers after
    // quantising x, idle warps at once).  Two CTAs of this kernel fit on one
    // SM, so the next call's set-up and weight prefetch overlap this call's
    // arithmetic without competing with this call's x; the next call reads
    // nothing a predecessor may write before its own griddepcontrol.wait.
    if (warp != pwarp && warp >= consumers) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == pwarp) {
        // x first: one tensor copy per box of 128-byte rows (32 elements), each
        // row's 16-byte pieces permuted by the 128-byte swizzle (piece i of row
        // r lands at piece i ^ (r % 8)), so that the consumers' reads below are
        // free of bank conflicts.  Rows past K arrive as zeros.
        if (lane == 0) {
            mbar_expect_tx_gv(xbar, uint32_t(P.nxbox * P.xbox_rows * 128));
            for (int bx = 0; bx < P.nxbox; ++bx)
                tma_load_2d_gv(smem_u32(gvs_smem) + uint32_t(bx * P.xbox_rows * 128), &xmap, 0,
                               bx * P.xbox_rows, xbar);
        }
        // the first ring-full of stages needs no slot to free up: the 32 lanes
        // issue those copies in parallel; lane 0 then refills slots as the
        // consumers release them
        const int first = min(nstages, P.ns);
        for (int st = lane; st < first; st += 32) issue(st);
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (producer) {
            for (int st = P.ns; st < nstages; ++st) {
                const int slot = st % P.ns, u = st / P.ns;
                if (!mbar_wait_spin(&empty[slot], (u - 1) & 1, wait_ns, status)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                issue(st);
            }
            // every copy issued must land before the CTA exits: the last round of each slot
            const uint64_t drain = wait_ns > 1000000000ull ? wait_ns : 1000000000ull;
            for (int st = max(0, nstages - P.ns); st < nstages; ++st)
                mbar_wait_spin(&full[st % P.ns], (st / P.ns) & 1, drain, status);
        }
    } else if (warp < consumers) {
        // Warp w takes chunk c = w % C of the stages st = g, g + groups, ...
        // (g = w / C).  The ring size is a multiple of `groups`, so every slot
        // is only ever touched by one group, in stage order: no warp can wait
        // on a slot's next round before the group released the current one.
        const int g = warp / C, c = warp % C;
        const int kw0 = c * kGvChunk + lane * kGvLaneW;
        const bool active = kw0 < k;
        const int kw_rd = active ? kw0 : 0;
        // ---- quantise this lane's 32 elements of x into three limbs.
        // L[q][t][l] holds in byte i limb l of X[16q + t + 4i], the order in
        // which a code word unpacks (bytes of (w >> 2t) & 0x03030303).
        uint32_t L[2][4][3];
        int sx = 0;
        float sc;
        if (!mbar_wait_spin(xbar, 0, wait_ns, status)) *abort_flag = 1;
        {
            float xv[kGvLaneW];
            const int xrow = kw_rd / kGvLaneW;  // this lane's 128-byte row of the x tile
#pragma unroll
            for (int i = 0; i < kGvLaneW / 4; ++i) {
                const float4 v = active ? *reinterpret_cast<const float4 *>(xs + xrow * 32 + ((i ^ (xrow & 7)) << 2))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                xv[4 * i + 0] = v.x;
                xv[4 * i + 1] = v.y;
                xv[4 * i + 2] = v.z;
                xv[4 * i + 3] = v.w;
            }
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < kGvLaneW; ++j) s = fmaxf(s, fabsf(xv[j]));
            // one scale per 128-weight block: the largest |x| over the block's
            // four lanes (lanes 4j .. 4j+3), so that the block's four integer
            // sums share it and can be added exactly before any scaling
            s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 1));
            s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 2));
            // 2^22 / s: the correctly rounded reciprocal times 2^22 (exact scaling)
            const float inv = s > 0.f ? __frcp_rn(s) * 4194304.0f : 0.f;
            // X = x * inv rounded to the nearest integer (ties to even) by one
            // fused multiply-add onto 1.5 * 2^23: the sum lies in [2^23, 2^24),
            // where the binary32 spacing is 1, so the low mantissa bits hold
            // X + 2^22.  |x * inv| <= 2^22 + 2^-2 (the reciprocal is within half
            // an ulp), so |X| <= 2^22 without a clamp.
            // B = the bits of that sum = 0x4B400000 + X: bytes 0 and 1 are those
            // of X, byte 2 of X is byte 2 of B minus 0x40 (two values per
            // subtraction, byte 3 = 0x4B absorbing the borrow), and
            // sum X = sum B - 32 * 0x4B400000 (mod 2^32; |sum X| <= 2^27)
            uint32_t B[kGvLaneW];
            uint32_t bs = 0;
#pragma unroll
            for (int j = 0; j < kGvLaneW; ++j) {
                B[j] = __float_as_uint(__fmaf_rn(xv[j], inv, 12582912.0f));
                bs += B[j];
            }
            sx = -int(bs - 32u * 0x4B400000u);  // the first accumulator of every row starts at -sum X
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t x0 = B[16 * q + t], x1 = B[16 * q + t + 4];
                    const uint32_t x2 = B[16 * q + t + 8], x3 = B[16 * q + t + 12];
                    const uint32_t p01 = __byte_perm(x0, x1, 0x5140);  // x0.b0 x1.b0 x0.b1 x1.b1
                    const uint32_t p23 = __byte_perm(x2, x3, 0x5140);
                    L[q][t][0] = __byte_perm(p01, p23, 0x5410);        // byte 0 of X0..X3
                    L[q][t][1] = __byte_perm(p01, p23, 0x7632);        // byte 1
                    const uint32_t h01 = __byte_perm(x0, x1, 0x7632) - 0x00400040u;
                    const uint32_t h23 = __byte_perm(x2, x3, 0x7632) - 0x00400040u;
                    L[q][t][2] = __byte_perm(h01, h23, 0x6420);        // byte 2 of X0..X3 (signed)
                }
            sc = s * (1.0f / 4194304.0f);  // s * 2^-22
        }
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // loop-invariant 32-bit shared-memory offsets of this lane's data in a
        // slot: code bytes of row u at code_off + u * kq, the row's block scale
        // at d_off + u * kb * 2
        const uint32_t kq32 = uint32_t(kq), kb2 = uint32_t(kb) * 2;
        const uint32_t code_off = uint32_t(kw_rd / 4);
        const uint32_t d_off = code_bytes + uint32_t(kw_rd / kBlockW) * 2;
        const int64_t dcol = kw_rd / kBlockW;
        int slot = g, ph = 0;  // ring slot and phase of stage st, advanced incrementally
        for (int st = g; st < nstages; st += P.groups) {
            if (!mbar_wait_spin(&full[slot], uint32_t(ph), wait_ns, status)) {
                *abort_flag = 1;
                break;
            }
            if (*abort_flag) break;
            const int r0 = st * RS;             // first row (CTA-relative) of the stage
            const int nv = min(RS, rows - r0);  // warp-uniform, >= 1
            const uint8_t *sb = ring + uint32_t(slot) * stage_bytes;
            // Each lane's 8 code bytes of a row in one 8-byte read (a warp reads
            // 256 contiguous bytes: conflict-free) and the row's block scale.
            // All RS rows of the slot are read: rows past nv (the CTA's last
            // stage) hold stale bytes of the slot and their results are dropped.
            uint2 cw[RS];
#pragma unroll
            for (int uu = 0; uu < RS; ++uu)
                cw[uu] = *reinterpret_cast<const uint2 *>(sb + code_off + uint32_t(uu) * kq32);
            // Release this chunk's share of the slot once all its reads are
            // done: right here when the block scales come from global memory,
            // after the scale reads below when they travel in the slot.
            if (!dbulk) mbar_arrive(&empty[slot]);
            // Per row: T = sum_i (c_i - 1) X_i over the lane's 32 weights, exact
            // in int32 (|T| <= 2^28).  Codes of weights t, t+4, t+8, t+12 of a
            // word are the bytes of (w >> 2t) & 0x03030303; each dp4a multiplies
            // them with one 8-bit limb of the matching X values.
            constexpr int V = RS <= 2 ? 2 : RS <= 4 ? 4 : 8;  // reduction width (power of two)
            int tv[V];
#pragma unroll
            for (int uu = 0; uu < V; ++uu) tv[uu] = 0;
#pragma unroll
            for (int uu = 0; uu < RS; ++uu) {
                int a0 = sx, a1 = 0, a2 = 0;
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const uint32_t wq = q == 0 ? cw[uu].x : cw[uu].y;
                        const uint32_t cv = (wq >> (2 * t)) & 0x03030303u;
                        a0 = dp4a_uu(cv, L[q][t][0], a0);
                        a1 = dp4a_uu(cv, L[q][t][1], a1);
                        a2 = dp4a_us(cv, L[q][t][2], a2);
                    }
                tv[uu] = a0 + (a1 << 8) + (a2 << 16);
            }
            // Reduction over the 32 lanes, one row per value (halving
            // butterfly: at each level a lane keeps half of its rows and adds the
            // partner's share of them).  The first two levels pair the four
            // lanes of one 128-weight block, which share the x scale: exact
            // integer adds (|sum| <= 2^30).  Then each remaining value (row) is
            // scaled once by s_b * 2^-22 * d of its block and the float levels
            // follow.
            constexpr int NI = V >= 4 ? 2 : 1;  // integer halving levels
#pragma unroll
            for (int lv = 0; lv < NI; ++lv) {
                const int o = 1 << lv, half = V >> (lv + 1);
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < V / 2; ++i)
                    if (i < half) {
                        const int give = upper ? tv[i] : tv[i + half];
                        const int keep = upper ? tv[i + half] : tv[i];
                        tv[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
                    }
            }
            if (V == 2) tv[0] += __shfl_xor_sync(0xffffffffu, tv[0], 2);  // the block's other lane pair
            // rows held now: lane bits 0 (and 1) select which part of the stage
            constexpr int VH = V >> NI;  // values per lane after the integer levels
            const int sel = NI == 2 ? ((lane & 1) << 1) | ((lane >> 1) & 1) : (lane & 1);
            float fv[VH];
#pragma unroll
            for (int i = 0; i < VH; ++i) {
                const int uu = sel * VH + i;  // stage row of value i
                float dd = 0.f;
                if (uu < nv)
                    dd = dbulk ? __half2float(*reinterpret_cast<const __half *>(sb + d_off + uint32_t(uu) * kb2))
                               : __half2float(__ushort_as_half(ldg_u16(dpl + int64_t(real_row(r0 + uu)) * kb + dcol)));
                fv[i] = active ? float(tv[i]) * (sc * dd) : 0.f;
            }
            if (dbulk) mbar_arrive(&empty[slot]);
            // float halving levels at offsets 4, 8, ... until one value is left, then full levels
#pragma unroll
            for (int lv = 0; (VH >> lv) > 1; ++lv) {
                const int o = 4 << lv, half = VH >> (lv + 1);
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < VH / 2; ++i)
                    if (i < half) {
                        const float give = upper ? fv[i] : fv[i + half];
                        const float keep = upper ? fv[i + half] : fv[i];
                        fv[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
                    }
            }
            constexpr int LV = V == 8 ? 3 : 2;  // levels done so far (offsets 1 .. 2^(LV-1))
#pragma unroll
            for (int o = 1 << LV; o < 32; o <<= 1) fv[0] += __shfl_xor_sync(0xffffffffu, fv[0], o);
            // lane l (l < 2^LV) holds the row whose index bits are lane bits 0, 1(, 2), most significant first
            if (lane < V) {
                const int uu = V == 8 ? ((lane & 1) << 2) | (((lane >> 1) & 1) << 1) | ((lane >> 2) & 1)
                                      : V == 4 ? ((lane & 1) << 1) | ((lane >> 1) & 1) : (lane & 1);
                if (uu < RS && uu < nv) partial[(r0 + uu) * C + c] = fv[0];
            }
            slot += P.groups;
            if (slot >= P.ns) slot -= P.ns, ph ^= 1;
        }
    }
    __syncthreads();
    if (*abort_flag) return;
    if (P.swiglu) {
        for (int i = threadIdx.x; i < nf; i += blockDim.x) {
            float g = 0.f, u = 0.f;
            for (int cc = 0; cc < C; ++cc) g += partial[i * C + cc];
            for (int cc = 0; cc < C; ++cc) u += partial[(nf + i) * C + cc];
            out[R0 + i] = g / (1.0f + expf(-g)) * u;  // silu(g) * u
        }
        return;
    }
    for (int i = threadIdx.x; i < rows; i += blockDim.x) {
        float sum = 0.f;
        for (int cc = 0; cc < C; ++cc) sum += partial[i * C + cc];
        if (residual) sum += residual[R0 + i];
        out[R0 + i] = sum;
    }
}


// ---------------------------------------------------------------------------
// M = 1 decode GEMV with wide lanes (K a multiple of 2048, at most 8192).
//
// The same streaming and the same exact integer arithmetic as above, but lane
// l of a chunk warp owns 64 weights, [2048 c + 64 l, +64) = half of 128-weight
// block 32 c + l / 2.  A row then costs one 16-byte shared-memory read per
// lane, and the per-row work outside the dot products (the address, the limb
// combination, the butterfly) is spread over twice the weights.  The 48 limb
// registers need up to 112 registers per thread: eight consumer warps (two
// per scheduler) and the producer, two CTAs per SM.
//
// x arrives as two tensor copies of 128-byte rows: the first 32 elements of
// every lane slice, then the last 32 (a 3-D view [K/64][2][32] of x), so that
// lane l of chunk c reads row 32 c + l of each half.  With the 128-byte
// swizzle the eight lanes of one shared-memory wavefront then hit eight
// different 16-byte bank groups.
constexpr int kGwLaneW = 64;               // weights per lane: half a 128-weight block
constexpr int kGwChunk = 32 * kGwLaneW;    // weights per warp-chunk (2048)
constexpr int kGwConsumers = 8;            // consumer warps (groups x chunks)
constexpr int kGwMaxK = 4 * kGwChunk;      // at least two groups of chunk warps

template <int RS, bool DBULK>
__global__ void __launch_bounds__(32 * (kGwConsumers + 1), 2)
gemv_wide_kernel(const __grid_constant__ CUtensorMap xmap, const uint8_t *__restrict__ qs,
                 const __half *__restrict__ dpl, const float *residual, float *out, GvsParams P,
                 unsigned int *status, uint64_t wait_ns) {
    extern __shared__ __align__(128) uint8_t gvw_raw[];
    uint8_t *gvs_smem = gvw_raw + ((1024u - (smem_u32(gvw_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = P.k, C = P.C;
    const int64_t kq = k / 4, kb = k / kBlockW;
    const int consumers = P.consumers;
    const int pwarp = int(blockDim.x >> 5) - 1;
    const int b = int(blockIdx.x);
    const int R0 = b * P.rbase + min(b, P.rextra);
    const int nf = P.rbase + (b < P.rextra ? 1 : 0);
    const int rows = P.swiglu ? 2 * nf : nf;
    auto real_row = [&](int i) { return (P.swiglu && i >= nf) ? P.f + R0 + (i - nf) : R0 + i; };
    const int nstages = (rows + RS - 1) / RS;
    constexpr bool dbulk = DBULK;
    const uint32_t code_bytes = uint32_t(RS * kq);
    const uint32_t stage_bytes = code_bytes + (dbulk ? uint32_t(RS * kb * 2) : 0u);
    const int xr = k / kGwLaneW;  // 128-byte rows per half of the x tile

    // shared memory: [x: two halves][ring][partials][barriers][abort flag]
    const float *xs = reinterpret_cast<const float *>(gvs_smem);
    uint8_t *ring = gvs_smem + P.off_ring;
    float *partial = reinterpret_cast<float *>(gvs_smem + P.off_partial);
    uint64_t *full = reinterpret_cast<uint64_t *>(gvs_smem + P.off_bar);
    uint64_t *empty = full + P.ns;
    uint64_t *xbar = empty + P.ns;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(xbar + 1);
    const uint32_t ring_addr = smem_u32(ring);

    if (warp == 0) {
        for (int i = lane; i < P.ns; i += 32) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 32 * C);
        }
        if (lane == 0) {
            mbar_init(xbar, 1);
            *abort_flag = 0;
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    const bool producer = warp == pwarp && lane == 0;
    auto pieces = [&](int st, auto &&fn) {
        const int lo = st * RS, hi = min(lo + RS, rows);
        if (P.swiglu && lo < nf && hi > nf) {
            fn(lo, nf - lo, 0);
            fn(nf, hi - nf, nf - lo);
        } else {
            fn(lo, hi - lo, 0);
        }
    };
    auto issue = [&](int st) {
        const int slot = st % P.ns;
        const int r = min(RS, rows - st * RS);
        const uint32_t dst = ring_addr + uint32_t(slot) * stage_bytes;
        mbar_expect_tx_gv(&full[slot], uint32_t(r) * (uint32_t(kq) + (dbulk ? uint32_t(kb * 2) : 0u)));
        pieces(st, [&](int i0, int cnt, int off) {
            const int64_t row = real_row(i0);
            bulk_g2s_gv(dst + uint32_t(off) * uint32_t(kq), qs + row * kq, uint32_t(cnt * kq), &full[slot]);
            if (dbulk)
                bulk_g2s_gv(dst + code_bytes + uint32_t(off) * uint32_t(kb * 2), dpl + row * kb,
                            uint32_t(cnt * kb * 2), &full[slot]);
        });
    };
    // weights to L2 before the dependency wait (see gemv_stream_kernel)
    // With resident weights the first ring of stages goes straight to shared
    // memory here, during the preceding kernel; only the stages beyond the
    // ring are prefetched into L2.
    const int first = min(nstages, P.ns);
    if (warp == pwarp) {
        if (P.early)
            for (int st = lane; st < first; st += 32) issue(st);
        for (int st = (P.early ? first : 0) + lane; st < nstages; st += 32) {
            pieces(st, [&](int i0, int cnt, int) {
                const int64_t row = real_row(i0);
                bulk_prefetch_l2(qs + row * kq, uint32_t(cnt * kq));
                if (dbulk) bulk_prefetch_l2(dpl + row * kb, uint32_t(cnt * kb * 2));
            });
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The next kernel of the stream may launch once every thread has passed
    // this point: at once with resident weights (its early weight copies need
    // the time), else after this CTA's x has been issued and quantised, so that
    // the next call's set-up and prefetch do not compete with this call's x.
    if (P.early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == pwarp) {
        if (lane == 0) {
            // half h: elements [64 j + 32 h, +32) of every j, as xr rows of 128 bytes
            mbar_expect_tx_gv(xbar, uint32_t(2 * xr * 128));
            for (int h = 0; h < 2; ++h)
                asm volatile(
                    "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                    "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(gvs_smem) + uint32_t(h * xr * 128)),
                    "l"(reinterpret_cast<uint64_t>(&xmap)), "r"(0), "r"(h), "r"(0), "r"(smem_u32(xbar))
                    : "memory");
        }
        if (!P.early) {
            for (int st = lane; st < first; st += 32) issue(st);
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        }
        if (producer) {
            for (int st = P.ns; st < nstages; ++st) {
                const int slot = st % P.ns, u = st / P.ns;
                if (!mbar_wait_spin(&empty[slot], (u - 1) & 1, wait_ns, status)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                issue(st);
            }
            const uint64_t drain = wait_ns > 1000000000ull ? wait_ns : 1000000000ull;
            for (int st = max(0, nstages - P.ns); st < nstages; ++st)
                mbar_wait_spin(&full[st % P.ns], (st / P.ns) & 1, drain, status);
        }
    } else if (warp < consumers) {
        const int g = warp / C, c = warp % C;
        const int kw0 = c * kGwChunk + lane * kGwLaneW;
        // ---- quantise this lane's 64 elements of x (one scale per 128-weight
        // block, shared with the neighbouring lane) into three limbs.
        // L[q][t][l] holds in byte i limb l of X[16q + t + 4i].
        uint32_t L[4][4][3];
        int sx;
        float sc;
        if (!mbar_wait_spin(xbar, 0, wait_ns, status)) *abort_flag = 1;
        {
            float xv[kGwLaneW];
            const int xrow = c * 32 + lane;  // this lane's row in each half
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 v =
                        *reinterpret_cast<const float4 *>(xs + (h * xr + xrow) * 32 + ((i ^ (xrow & 7)) << 2));
                    xv[32 * h + 4 * i + 0] = v.x;
                    xv[32 * h + 4 * i + 1] = v.y;
                    xv[32 * h + 4 * i + 2] = v.z;
                    xv[32 * h + 4 * i + 3] = v.w;
                }
            // max |x| as a balanced tree (short dependency chain)
            float m[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) m[j] = fmaxf(fabsf(xv[2 * j]), fabsf(xv[2 * j + 1]));
#pragma unroll
            for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j) m[j] = fmaxf(m[j], m[j + w]);
            float s = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], 1));  // the block's other half
            // 2^22 / s (correctly rounded reciprocal, exact scaling)
            const float inv = s > 0.f ? __frcp_rn(s) * 4194304.0f : 0.f;
            // X = rint(x * inv) by one fused multiply-add onto 1.5 * 2^23 (|X| <= 2^22)
            // B = the bits of that sum = 0x4B400000 + X.  Bytes 0 and 1 of B are
            // those of X (the offset's low half is zero); byte 2 of X is byte 2
            // of B minus 0x40, subtracted for two values at once with byte 3
            // (0x4B) of each absorbing the borrow; sum X = sum B - 64 * 0x4B400000.
            uint32_t B[kGwLaneW];
#pragma unroll
            for (int j = 0; j < kGwLaneW; ++j) B[j] = __float_as_uint(__fmaf_rn(xv[j], inv, 12582912.0f));
            uint32_t ps[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) ps[j] = (B[4 * j] + B[4 * j + 1]) + (B[4 * j + 2] + B[4 * j + 3]);
#pragma unroll
            for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j) ps[j] += ps[j + w];
            // the first accumulator of every row starts at -sum X (|sum X| <= 2^28: exact mod 2^32)
            sx = -int(ps[0] - 64u * 0x4B400000u);
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t x0 = B[16 * q + t], x1 = B[16 * q + t + 4];
                    const uint32_t x2 = B[16 * q + t + 8], x3 = B[16 * q + t + 12];
                    const uint32_t p01 = __byte_perm(x0, x1, 0x5140);  // x0.b0 x1.b0 x0.b1 x1.b1
                    const uint32_t p23 = __byte_perm(x2, x3, 0x5140);
                    L[q][t][0] = __byte_perm(p01, p23, 0x5410);        // byte 0 of X0..X3
                    L[q][t][1] = __byte_perm(p01, p23, 0x7632);        // byte 1
                    const uint32_t h01 = __byte_perm(x0, x1, 0x7632) - 0x00400040u;  // x0.b2 x0.b3 x1.b2 x1.b3
                    const uint32_t h23 = __byte_perm(x2, x3, 0x7632) - 0x00400040u;
                    L[q][t][2] = __byte_perm(h01, h23, 0x6420);        // byte 2 of X0..X3 (signed)
                }
            sc = s * (1.0f / 4194304.0f);
        }
        if (!P.early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        const uint32_t kq32 = uint32_t(kq), kb2 = uint32_t(kb) * 2;
        const uint32_t code_off = uint32_t(kw0 / 4);
        const uint32_t d_off = code_bytes + uint32_t(kw0 / kBlockW) * 2;
        const int64_t dcol = kw0 / kBlockW;
        int slot = g, ph = 0;
        for (int st = g; st < nstages; st += P.groups) {
            if (!mbar_wait_spin(&full[slot], uint32_t(ph), wait_ns, status)) {
                *abort_flag = 1;
                break;
            }
            if (*abort_flag) break;
            const int r0 = st * RS;
            const int nv = min(RS, rows - r0);
            const uint8_t *sb = ring + uint32_t(slot) * stage_bytes;
            // one 16-byte read per row and lane (a warp reads 512 contiguous bytes)
            uint4 cw[RS];
#pragma unroll
            for (int uu = 0; uu < RS; ++uu)
                cw[uu] = *reinterpret_cast<const uint4 *>(sb + code_off + uint32_t(uu) * kq32);
            if (!dbulk) mbar_arrive(&empty[slot]);
            constexpr int V = RS <= 2 ? 2 : RS <= 4 ? 4 : 8;
            int tv[V];
#pragma unroll
            for (int uu = 0; uu < V; ++uu) tv[uu] = 0;
#pragma unroll
            for (int uu = 0; uu < RS; ++uu) {
                int a0 = sx, a1 = 0, a2 = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t wq = q == 0 ? cw[uu].x : q == 1 ? cw[uu].y : q == 2 ? cw[uu].z : cw[uu].w;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const uint32_t cv = (wq >> (2 * t)) & 0x03030303u;
                        a0 = dp4a_uu(cv, L[q][t][0], a0);
                        a1 = dp4a_uu(cv, L[q][t][1], a1);
                        a2 = dp4a_us(cv, L[q][t][2], a2);
                    }
                }
                tv[uu] = a0 + (a1 << 8) + (a2 << 16);  // |T| <= 64 * 2^22
            }
            // butterfly level 1 (lanes 2j, 2j+1: one block, one x scale):
            // exact integer adds (|sum| <= 2^29)
            constexpr int VH = V / 2;
            {
                const bool upper = (lane & 1) != 0;
#pragma unroll
                for (int i = 0; i < VH; ++i) {
                    const int give = upper ? tv[i] : tv[i + VH];
                    const int keep = upper ? tv[i + VH] : tv[i];
                    tv[i] = keep + __shfl_xor_sync(0xffffffffu, give, 1);
                }
            }
            const int sel = lane & 1;
            float fv[VH];
#pragma unroll
            for (int i = 0; i < VH; ++i) {
                const int uu = sel * VH + i;
                float dd = 0.f;
                if (uu < nv)
                    dd = dbulk ? __half2float(*reinterpret_cast<const __half *>(sb + d_off + uint32_t(uu) * kb2))
                               : __half2float(__ushort_as_half(ldg_u16(dpl + int64_t(real_row(r0 + uu)) * kb + dcol)));
                fv[i] = float(tv[i]) * (sc * dd);
            }
            if (dbulk) mbar_arrive(&empty[slot]);
            // float halving levels at offsets 2, 4, ... until one value is left
#pragma unroll
            for (int lv = 0; (VH >> lv) > 1; ++lv) {
                const int o = 2 << lv, half = VH >> (lv + 1);
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < VH / 2; ++i)
                    if (i < half) {
                        const float give = upper ? fv[i] : fv[i + half];
                        const float keep = upper ? fv[i + half] : fv[i];
                        fv[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
                    }
            }
            constexpr int LV = V == 8 ? 3 : V == 4 ? 2 : 1;
#pragma unroll
            for (int o = 1 << LV; o < 32; o <<= 1) fv[0] += __shfl_xor_sync(0xffffffffu, fv[0], o);
            if (lane < V) {
                const int uu = V == 8 ? ((lane & 1) << 2) | (((lane >> 1) & 1) << 1) | ((lane >> 2) & 1)
                                      : V == 4 ? ((lane & 1) << 1) | ((lane >> 1) & 1) : (lane & 1);
                if (uu < RS && uu < nv) partial[(r0 + uu) * C + c] = fv[0];
            }
            slot += P.groups;
            if (slot >= P.ns) slot -= P.ns, ph ^= 1;
        }
    }
    __syncthreads();
    if (*abort_flag) return;
    if (P.swiglu) {
        for (int i = threadIdx.x; i < nf; i += blockDim.x) {
            float g = 0.f, u = 0.f;
            for (int cc = 0; cc < C; ++cc) g += partial[i * C + cc];
            for (int cc = 0; cc < C; ++cc) u += partial[(nf + i) * C + cc];
            out[R0 + i] = g / (1.0f + expf(-g)) * u;
        }
        return;
    }
    for (int i = threadIdx.x; i < rows; i += blockDim.x) {
        float sum = 0.f;
        for (int cc = 0; cc < C; ++cc) sum += partial[i * C + cc];
        if (residual) sum += residual[R0 + i];
        out[R0 + i] = sum;
    }
}

}  // namespace

// swiglu: n = 2f weight rows (gate then up), out has f elements, no residual.
cudaError_t launch_gemv_stream(const void *w_soa, const float *x, const float *residual,
                               float *out, int64_t n, int64_t k, bool swiglu, bool resident,
                               const LaunchCtx &ctx) {
    // wide lanes (64 weights) where K splits into at most four 2048-weight chunks
    const bool wide = k % kGwChunk == 0 && k <= kGwMaxK;
    const int C = wide ? int(k / kGwChunk) : int((k + kGvChunk - 1) / kGvChunk);
    const int64_t kq = k / 4, kb = k / kBlockW;
    if (C > kGvMaxConsumers) return cudaErrorNotSupported;
    GvsParams P;
    P.n = int(n);
    P.k = int(k);
    P.C = C;
    P.swiglu = swiglu ? 1 : 0;
    P.early = 0;  // set below, once the ring size is known
    P.f = int(n / 2);
    P.groups = std::max(1, (wide ? kGwConsumers : kGvMaxConsumers) / C);  // groups of C warps (one per chunk)
    // the CTAs split the rows (with swiglu: the features, two rows each)
    const int64_t units = swiglu ? n / 2 : n;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(ctx.num_sms, (n + 7) / 8));
    P.rbase = int(units / grid);
    P.rextra = int(units % grid);
    P.rows_cta = (P.rbase + (P.rextra ? 1 : 0)) * (swiglu ? 2 : 1);
    // Rows per stage: a group's time is (its stages) x (RS rows + a per-stage
    // cost of about two rows); pick the RS in [2, 8] that minimises it for the
    // CTA's row count (ties: more rows per stage).
    {
        int best = 8;
        long best_cost = LONG_MAX;
        for (int rs = 8; rs >= 2; --rs) {
            const long nst_rs = (P.rows_cta + rs - 1) / rs;
            const long cost = ((nst_rs + P.groups - 1) / P.groups) * (rs + 2);
            if (cost < best_cost) best_cost = cost, best = rs;
        }
        P.rs = best;
    }
    const bool dbulk = (kb % 8) == 0;  // scales travel with their stage in the ring
    const size_t stage_bytes = size_t(P.rs) * kq + (dbulk ? size_t(P.rs) * kb * 2 : 0);
    const size_t partial_bytes = size_t((P.rows_cta * C + 1) & ~1) * 4;
    // x as a tensor of K/32 rows of 128 bytes, in boxes of at most 256 rows
    // (a multiple of 8 rows: every box starts on a 1024-byte swizzle atom);
    // wide lanes: two halves of K/64 rows (K/64 <= 128, a multiple of 32)
    const int xrows = int(k / kGvLaneW);
    P.nxbox = wide ? 2 : (xrows + 255) / 256;
    P.xbox_rows = wide ? int(k / kGwLaneW) : (((xrows + P.nxbox - 1) / P.nxbox) + 7) & ~7;
    const size_t x_bytes = size_t(P.nxbox) * P.xbox_rows * 128;
    // two CTAs per SM: 2 * (this + 1 KB reserved per CTA) within 228 KB
    const size_t budget = 112 * 1024;
    const size_t fixed = 1024 + x_bytes + partial_bytes + 64 * 16 + 32;
    if (fixed + stage_bytes > budget) return cudaErrorNotSupported;
    // ring: enough slots for all of a CTA's stages if shared memory allows (no
    // refill round trips), as a multiple of the group count
    const int nst = (P.rows_cta + P.rs - 1) / P.rs;
    const int max_slots = int(std::min<size_t>(64, (budget - fixed) / stage_bytes));
    int ns = std::min(max_slots, ((nst + P.groups - 1) / P.groups) * P.groups);
    ns = (ns / P.groups) * P.groups;
    if (ns < P.groups) {  // fewer slots than groups: shrink the groups
        P.groups = std::max(1, max_slots);
        ns = P.groups;
    }
    P.ns = ns;
    P.consumers = P.groups * C;
    // Resident weights: copy early only when the ring holds all of a CTA's
    // stages (measured slower otherwise: 7.6 against 6.9 us at K=N=8192, and
    // 6.50 against 6.21 us with the 32-weight lanes at K=12288, N=4096).
    P.early = resident && wide && ns >= nst ? 1 : 0;
    P.off_ring = uint32_t(x_bytes);
    P.off_partial = uint32_t(x_bytes + size_t(ns) * stage_bytes);
    P.off_bar = uint32_t((P.off_partial + partial_bytes + 7) & ~size_t(7));
    const size_t smem = 1024 + size_t(P.off_bar) + size_t(2 * ns + 1) * 8 + 16;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap xmap;
    if (wide) {
        // [K/64][2][32] view of x: element (e, h, j) = x[64 j + 32 h + e]
        const cuuint64_t gdim[3] = {32, 2, cuuint64_t(k / kGwLaneW)};
        const cuuint64_t gstride[2] = {128, 256};
        const cuuint32_t box[3] = {32, 1, cuuint32_t(k / kGwLaneW)};
        const cuuint32_t estride[3] = {1, 1, 1};
        if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(x), gdim, gstride, box,
                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        const cuuint64_t gdim[2] = {cuuint64_t(kGvLaneW), cuuint64_t(xrows)};
        const cuuint64_t gstride[1] = {cuuint64_t(kGvLaneW) * 4};
        const cuuint32_t box[2] = {cuuint32_t(kGvLaneW), cuuint32_t(P.xbox_rows)};
        const cuuint32_t estride[2] = {1, 1};
        if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(x), gdim, gstride, box,
                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int threads = 32 * (P.consumers + 1);  // consumer warps and the producer warp
    void (*kern)(const CUtensorMap, const uint8_t *, const __half *, const float *, float *, GvsParams,
                 unsigned int *, uint64_t) = nullptr;
#define TQ2_GV_KERN(RSV)                                                                                    \
    kern = wide ? (dbulk ? gemv_wide_kernel<RSV, true> : gemv_wide_kernel<RSV, false>)                      \
                : (dbulk ? gemv_stream_kernel<RSV, true, kGvMaxConsumers> : gemv_stream_kernel<RSV, false, kGvMaxConsumers>)
    switch (P.rs) {
        case 2: TQ2_GV_KERN(2); break;
        case 3: TQ2_GV_KERN(3); break;
        case 4: TQ2_GV_KERN(4); break;
        case 5: TQ2_GV_KERN(5); break;
        case 6: TQ2_GV_KERN(6); break;
        case 7: TQ2_GV_KERN(7); break;
        default: TQ2_GV_KERN(8); break;
    }
#undef TQ2_GV_KERN
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // the largest shared-memory carve-out, so that two CTAs fit on an SM
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
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
    return cudaLaunchKernelEx(&cfg, kern, xmap, v.qs, v.d, residual, out, P, ctx.status,
                              ctx.wait_ns);
}

cudaError_t launch_gemv_swiglu(const void *w_soa, const float *x, float *out, int64_t f, int64_t k,
                               const LaunchCtx &ctx, bool resident) {
    if (k > int64_t(kGvMaxConsumers) * kGvChunk || 2 * f > INT32_MAX) return cudaErrorNotSupported;
    return launch_gemv_stream(w_soa, x, nullptr, out, 2 * f, k, true, resident, ctx);
}

cudaError_t launch_gemv(const void *w_soa, const float *x, const float *residual, float *out,
                        int64_t n, int64_t k, const LaunchCtx &ctx, bool resident) {
    if (k <= int64_t(kGvMaxConsumers) * kGvChunk && n <= INT32_MAX) {
        cudaError_t e = launch_gemv_stream(w_soa, x, residual, out, n, k, false, resident, ctx);
        if (e != cudaErrorNotSupported) return e;
        (void)cudaGetLastError();
    }
    // very long rows: the chunk-looping small-M kernel (exact f32)
    return launch_tpl<1, 2>(w_soa, x, residual, out, 1, n, k, ctx);
}

namespace {
__global__ void __launch_bounds__(256) swiglu_rows_kernel(const float *__restrict__ gu, float *__restrict__ out,
                                                          int64_t m, int64_t f) {
    const int64_t total = m * f, stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t r = i / f, j = i - r * f;
        const float g = gu[r * 2 * f + j], u = gu[r * 2 * f + f + j];
        out[i] = g / (1.0f + expf(-g)) * u;
    }
}
}  // namespace

cudaError_t launch_swiglu_rows(const float *gu, float *out, int64_t m, int64_t f, const LaunchCtx &ctx) {
    const int64_t total = m * f;
    if (total == 0) return cudaSuccess;
    const int64_t grid = std::min<int64_t>((total + 255) / 256, int64_t(ctx.num_sms) * 8);
    swiglu_rows_kernel<<<unsigned(grid), 256, 0, ctx.stream>>>(gu, out, m, f);
    return cudaPeekAtLastError();
}

cudaError_t launch_skinny(const void *w_soa, const float *x, const float *residual, float *out,
                          int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx) {
    if (m == 1) return launch_tpl<1, 2>(w_soa, x, residual, out, m, n, k, ctx);
    if (m == 2) return launch_tpl<2, 1>(w_soa, x, residual, out, m, n, k, ctx);
    return launch_tpl<4, 1>(w_soa, x, residual, out, m, n, k, ctx);
}

}  // namespace tq2
