// Large-M tensor-core kernel: tcgen05 MMA (kind::f16, f32 accumulation in
// TMEM) with the ternary codes decoded once per tile into binary16 shared
// memory.
//
// The pages' large-M TQ2 kernels (`gemm_tq2_g128_v9_simdgroup` and
// `gemm_tq2_g128_v10_simdgroup`, "oxibonsai-kernels 0.1.5
// src/gpu_backend/metal_graph/pipelines.rs") dequantise the weight into
// threadgroup memory, stage it as half ("exact for ternary code x scale"),
// stage f16 activations and accumulate in f32 on the matrix units, with the
// K-tile staging double-buffered.  On sm_103a the same contraction becomes:
//
//  * CTA tile 128 (M) x 256 (N), K advancing 64 per pipeline stage, a
//    STAGES-deep ring of shared-memory stages guarded by mbarriers.
//  * 8 producer warps.  Each thread decodes one weight row's 64 codes per
//    stage (one 16-byte load), and converts 4 x 8 activations f32 -> f16
//    (round to nearest even).  Both operands are written in the canonical
//    K-major SWIZZLE_128B layout (8-row x 128-byte atoms, 16-byte chunks
//    XOR-ed with the row index) that the MMA reads through shared-memory
//    descriptors.  Registers hold the next stage's loads while the current
//    stage is written.
//  * Decode: the two codes of weights i and i+8 of a 16-weight word are masked
//    into the mantissas of a half2 of 1024 (0x6400) in one AND-OR, giving
//    1024 + c*2^s; one half2 FMA with 2^-s and -(1024*2^-s + 1) gives c - 1,
//    one half2 multiply by d gives the weight.  All three steps are exact in
//    binary16.  The pairing (i, i+8) permutes K inside every 16-wide group;
//    the activations are written with the same permutation, which leaves the
//    contraction unchanged.
//  * One thread issues the MMAs (4 x K=16 per stage) and commits each stage's
//    completion to that stage's "empty" barrier; a final commit signals the
//    accumulator to the epilogue.
//  * 4 epilogue warps read the 128 x 256 f32 accumulator from TMEM
//    (tcgen05.ld 32x32b), add the residual and store f32 rows.
//  * Every mbarrier wait is bounded (%globaltimer); a timeout records
//    TQ2_ERR_TIMEOUT, stops the other roles through a shared flag, lets the
//    issued MMAs drain and frees TMEM before the CTA exits.
#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BYTES = BN * BK * 2;             // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 48 KB
constexpr int NUM_EPI_WARPS = 4;
constexpr int MMA_WARP = 4;
constexpr int PROD_WARP0 = 5;
constexpr int NUM_PROD_WARPS = 8;
constexpr int NUM_PROD = NUM_PROD_WARPS * 32;    // 256 = BN
constexpr int THREADS = (PROD_WARP0 + NUM_PROD_WARPS) * 32;  // 416
constexpr uint32_t TMEM_COLS = 256;
constexpr int A_TASKS = BM * 8 / NUM_PROD;       // 16-byte A chunks per producer thread
static_assert(NUM_PROD == BN, "one weight row per producer thread");
static_assert(A_TASKS == 4, "");

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B f16
// (format 0), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t IDESC = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

struct Ctl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t accum_full;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t SMEM_BYTES = size_t(STAGES) * STAGE_BYTES + sizeof(Ctl) + 1024;

// Shared-memory matrix descriptor for a K-major SWIZZLE_128B tile whose 8-row
// atoms are 1024 bytes apart: start address >> 4 (bits 0-13), leading byte
// offset (unused for this layout, 16 B), stride byte offset 1024 >> 4
// (bits 32-45), descriptor version 1 (bits 46-47), swizzle mode 2 =
// 128-byte swizzle (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Byte offset of 16-byte chunk j (0..7) of row r inside a SW128 K-major tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int j) {
    return uint32_t((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) {
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Decode one 16-weight code word into 8 half2 (weights (i, i+8), i = 0..7),
// each (c - 1) * d exactly.
__device__ __forceinline__ void decode_word(uint32_t w, __half2 d2, uint32_t (&o)[8]) {
    const uint32_t w6 = w >> 6;
    const uint32_t base = 0x64006400u;
    // position s of pair i: i<=4 -> 2i in w; i>=5 -> 2(i-3) in w >> 6
    const uint32_t v0 = (w & 0x00030003u) | base;
    const uint32_t v1 = (w & 0x000C000Cu) | base;
    const uint32_t v2 = (w & 0x00300030u) | base;
    const uint32_t v3 = (w & 0x00C000C0u) | base;
    const uint32_t v4 = (w & 0x03000300u) | base;
    const uint32_t v5 = (w6 & 0x00300030u) | base;
    const uint32_t v6 = (w6 & 0x00C000C0u) | base;
    const uint32_t v7 = (w6 & 0x03000300u) | base;
    const __half2 s0 = __float2half2_rn(1.0f), b0 = __float2half2_rn(-1025.0f);
    const __half2 s2 = __float2half2_rn(0.25f), b2 = __float2half2_rn(-257.0f);
    const __half2 s4 = __float2half2_rn(0.0625f), b4 = __float2half2_rn(-65.0f);
    const __half2 s6 = __float2half2_rn(0.015625f), b6 = __float2half2_rn(-17.0f);
    const __half2 s8 = __float2half2_rn(0.00390625f), b8 = __float2half2_rn(-5.0f);
    o[0] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(v0), s0, b0), d2));
    o[1] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(v1), s2, b2), d2));
    o[2] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(v2), s4, b4), d2));
    o[3] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(v3), s6, b6), d2));
    o[4] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(v4), s8, b8), d2));
    o[5] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(v5), s4, b4), d2));
    o[6] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(v6), s6, b6), d2));
    o[7] = h2_as_u32(__hmul2(__hfma2(u32_as_h2(v7), s8, b8), d2));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

struct ProdRegs {
    uint4 code;        // 64 codes of this thread's weight row
    uint32_t dbits;    // binary16 scale bits
    float4 xa[A_TASKS][2];
};

__global__ void __launch_bounds__(THREADS, 1)
tc_kernel(const uint8_t *__restrict__ qs, const __half *__restrict__ dpl,
          const float *__restrict__ x, const float *residual, float *out, int M, int N, int K,
          unsigned int *status, uint64_t wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t smem_base = raw_addr + pad;
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + size_t(STAGES) * STAGE_BYTES);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
    const int KT = K / BK;
    const int64_t kq = K / 4, kb = K / kBlockW;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&ctl->full[s], NUM_PROD);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->accum_full, 1);
        ctl->abort = 0;
        fence_mbarrier_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(&ctl->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort;

    if (warp >= PROD_WARP0) {
        // ---------------- producers ----------------
        const int pt = tid - PROD_WARP0 * 32;
        const int nrow = n0 + pt;
        const bool bvalid = nrow < N;
        const uint8_t *bq = qs + int64_t(bvalid ? nrow : 0) * kq;
        const __half *bd = dpl + int64_t(bvalid ? nrow : 0) * kb;
        int arow[A_TASKS], aj[A_TASKS];
        bool avalid[A_TASKS];
        const float *ax[A_TASKS];
#pragma unroll
        for (int i = 0; i < A_TASKS; ++i) {
            const int t = pt + NUM_PROD * i;
            arow[i] = t >> 3;
            aj[i] = t & 7;
            avalid[i] = (m0 + arow[i]) < M;
            // chunk j = (word q = j/2, half h = j%2): x[16q + 4h .. +3] and x[16q + 8 + 4h .. +3]
            ax[i] = x + int64_t(avalid[i] ? m0 + arow[i] : 0) * K + 16 * (aj[i] >> 1) + 4 * (aj[i] & 1);
        }
        auto load = [&](int it, ProdRegs &r) {
            const int k0 = it * BK;
            if (bvalid) {
                r.code = ldg_stream_u4(bq + k0 / 4);
                r.dbits = ldg_u16(bd + k0 / kBlockW);
            } else {
                r.code = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
                r.dbits = 0;
            }
#pragma unroll
            for (int i = 0; i < A_TASKS; ++i) {
                if (avalid[i]) {
                    r.xa[i][0] = __ldg(reinterpret_cast<const float4 *>(ax[i] + k0));
                    r.xa[i][1] = __ldg(reinterpret_cast<const float4 *>(ax[i] + k0 + 8));
                } else {
                    r.xa[i][0] = make_float4(0.f, 0.f, 0.f, 0.f);
                    r.xa[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        };
        // Returns false when the pipeline was aborted.
        auto produce = [&](int it, const ProdRegs &cur) -> bool {
            const int s = it % STAGES;
            if (it >= STAGES) {
                if (!mbar_wait_bounded(&ctl->empty[s], ((it / STAGES) - 1) & 1, wait_ns, status)) {
                    *abort_flag = 1;
                    return false;
                }
            }
            if (*abort_flag) return false;
            const uint32_t a_base = smem_base + s * STAGE_BYTES;
            const uint32_t b_base = a_base + A_BYTES;
            // activations: f32 -> f16 (RNE), pairs (i, i+8)
#pragma unroll
            for (int i = 0; i < A_TASKS; ++i) {
                const float4 lo = cur.xa[i][0], hi = cur.xa[i][1];
                st_shared_v4(a_base + sw128_off(arow[i], aj[i]),
                             h2_as_u32(__floats2half2_rn(lo.x, hi.x)),
                             h2_as_u32(__floats2half2_rn(lo.y, hi.y)),
                             h2_as_u32(__floats2half2_rn(lo.z, hi.z)),
                             h2_as_u32(__floats2half2_rn(lo.w, hi.w)));
            }
            // weights: decode 4 words -> 8 chunks
            const __half d = __ushort_as_half(static_cast<unsigned short>(cur.dbits));
            const __half2 d2 = __half2half2(d);
            const uint32_t words[4] = {cur.code.x, cur.code.y, cur.code.z, cur.code.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t o[8];
                decode_word(words[q], d2, o);
                st_shared_v4(b_base + sw128_off(pt, 2 * q), o[0], o[1], o[2], o[3]);
                st_shared_v4(b_base + sw128_off(pt, 2 * q + 1), o[4], o[5], o[6], o[7]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&ctl->full[s]);
            return true;
        };
        // Two register stages in flight: the loads of stage it+2 are issued as
        // soon as stage it has been written.
        ProdRegs ra, rb;
        if (KT > 0) load(0, ra);
        if (KT > 1) load(1, rb);
        for (int it = 0; it < KT; it += 2) {
            if (!produce(it, ra)) break;
            if (it + 2 < KT) load(it + 2, ra);
            if (it + 1 >= KT) break;
            if (!produce(it + 1, rb)) break;
            if (it + 3 < KT) load(it + 3, rb);
        }
    } else if (warp == MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            for (int it = 0; it < KT; ++it) {
                const int s = it % STAGES;
                if (!mbar_wait_bounded(&ctl->full[s], (it / STAGES) & 1, wait_ns, status)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                tc_fence_after();
                const uint32_t a_base = smem_base + s * STAGE_BYTES;
                const uint64_t adesc = sw128_desc(a_base);
                const uint64_t bdesc = sw128_desc(a_base + A_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    // +32 bytes along K inside the 128-byte swizzle row = +2 in the address field
                    tc_mma_f16(tmem, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (it | kk) != 0);
                }
                tc_commit(&ctl->empty[s]);
            }
            tc_commit(&ctl->accum_full);  // fires once every issued MMA has completed
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 0..3) ----------------
        const bool ok = mbar_wait_bounded(&ctl->accum_full, 0, wait_ns, status);
        if (!ok) *abort_flag = 1;
        if (ok && !*abort_flag && KT > 0) {
            tc_fence_after();
            const int row = m0 + warp * 32 + lane;
            const bool rvalid = row < M;
            const bool vec = (N % 4) == 0;
            for (int c = 0; c < BN / 16; ++c) {
                uint32_t r[16];
                tmem_ld16(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c * 16), r);
                tc_wait_ld();
                const int col0 = n0 + c * 16;
                if (!rvalid || col0 >= N) continue;
                float *op = out + int64_t(row) * N + col0;
                const float *rp = residual ? residual + int64_t(row) * N + col0 : nullptr;
                if (vec && col0 + 16 <= N) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float4 v = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                               __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                        if (rp) {
                            const float4 rr = *reinterpret_cast<const float4 *>(rp + 4 * q);
                            v.x += rr.x; v.y += rr.y; v.z += rr.z; v.w += rr.w;
                        }
                        *reinterpret_cast<float4 *>(op + 4 * q) = v;
                    }
                } else {
                    for (int j = 0; j < 16 && col0 + j < N; ++j) {
                        float v = __uint_as_float(r[j]);
                        if (rp) v += rp[j];
                        op[j] = v;
                    }
                }
            }
        }
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        if (lane == 0) {
            // Every issued MMA must be complete before TMEM is released.
            const uint64_t drain = wait_ns > 1000000000ull ? wait_ns : 1000000000ull;
            mbar_wait_bounded(&ctl->accum_full, 0, drain, status);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_tc(const void *w_soa, const float *x, const float *residual, float *out,
                      int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx) {
    if (m > INT32_MAX || n > INT32_MAX || k > INT32_MAX) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    const SoaView v = soa_view(w_soa, n, k);
    dim3 grid(static_cast<unsigned>((n + BN - 1) / BN), static_cast<unsigned>((m + BM - 1) / BM));
    if (grid.y > 65535) return cudaErrorInvalidValue;
    tc_kernel<<<grid, THREADS, SMEM_BYTES, ctx.stream>>>(v.qs, v.d, x, residual, out, int(m), int(n),
                                                         int(k), ctx.status, ctx.wait_ns);
    return cudaPeekAtLastError();
}

}  // namespace tq2
