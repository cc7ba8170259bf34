// DiT joint attention on the tcgen05 tensor cores (flash attention, one pass
// over the keys with an online softmax).
//
// Contract of the pages' `joint_attention_gpu` ("oxibonsai-image 0.2.2
// src/gpu.rs"; kernel `joint_attention_flash_f32` of "oxibonsai-kernels 0.1.5
// src/gpu_backend/metal_graph/pipelines.rs", FLUX.2 DiT joint attention):
// q, k, v head-major f32 [H, S, D]; out token-major f32 [S, H*D] (heads
// concatenated along the features); scale 1/sqrt(D); non-causal softmax over
// all S keys.
//
// Design (sm_103a):
//  * Pre-pass: q -> binary16 pre-scaled by log2(e)/sqrt(D) (scores come out in
//    log2 units for ex2), k -> binary16, v -> binary16 transposed per head
//    ([H, D, Sp]); Sp = S rounded up to 128, padding zero.  All three are
//    then K-major MMA operands loaded by tensor copies with the 128-byte
//    swizzle.
//  * One CTA per (head, 256 queries) = two query tiles of 128 that share every
//    K and V^T tile they copy (each copied tile feeds twice the MMA work of a
//    one-tile CTA: the SM's L2 -> shared-memory bandwidth, not the tensor
//    core, paced the one-tile form).  Warp 0 copies Q once and K, V^T through
//    two-stage rings; warp 1 issues the MMAs (the whole warp waits and
//    computes the descriptors, lane 0 issues); warps 4-7 run the softmax of
//    tile 0 and warps 8-11 that of tile 1 (one thread per query row = TMEM
//    lane).
//  * Tensor memory: the scores S_t of tile t at columns 128 t, its output O_t
//    at 256 + 128 t.  The softmax reads S_t and writes P_t = 2^(S_t - m) as
//    binary16 over the first 64 columns of S_t; P_t V is then an MMA whose A
//    operand is read from tensor memory (lane = query, column c = keys 2c,
//    2c + 1), so P never passes through shared memory.
//  * MMA order per key block j: P_0 V_j, S_0 of block j + 1, P_1 V_j, S_1 of
//    block j + 1.  Tile 0's softmax of block j + 1 overlaps P_1 V_j and S_1;
//    tile 1's overlaps the next P_0 V and S_0.  MMAs of one thread execute in
//    issue order, so S_t of block j + 1 overwrites P_t only after P_t V_j has
//    read it.
//  * Softmax per block: the row maximum over the valid keys first, then
//    P = 2^(s - mu).  Lazy rescale: the running maximum mu changes (and O and
//    l are rescaled by 2^(m_old - m_new)) only when a block's maximum exceeds
//    it by more than 8, so P <= 2^8 always fits binary16 and the rescale is
//    rare.  (Measured alternatives: two threads per row, one pass with P held
//    in registers, part of the exponentials by a polynomial on the FMA pipe:
//    all slower at the DiT shape.)
//  * Epilogue: out = O / l, f32.
// Every wait is bounded; a timeout sets the device status word and the CTA
// drains and exits.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int AQ = 128;        // queries per tile (MMA M)
constexpr int AQT = 2;         // query tiles per CTA
constexpr int AKB = 128;       // keys per block
constexpr int ATHREADS = 384;  // warp 0 copies, warp 1 MMA + TMEM, warps 4-7 / 8-11 softmax of tile 0 / 1
constexpr int A_SMT = AQ;      // softmax threads per tile (one per query row)
constexpr int A_TMA = 0, A_MMA = 1, A_SM0 = 4;
constexpr float kLazyLog2 = 8.0f;
constexpr uint32_t ATMEM_COLS = 512;  // S/P of tile t at 128 t, O of tile t at 256 + 128 t
constexpr uint32_t A_OCOL = 256;

template <int D>
struct AttnLayout {
    static constexpr int SUB = 128 * 128;            // one swizzled 128-row x 64-element sub-tile
    static constexpr int QB = AQ * D * 2;            // one Q tile
    static constexpr int KB = AKB * D * 2;           // one K tile
    static constexpr int VB = D * AKB * 2;           // one V^T tile (D rows x 128 keys)
    static constexpr int OFF_K = AQT * QB, OFF_V = OFF_K + 2 * KB;
    static constexpr int OFF_CTL = OFF_V + 2 * VB;
    static constexpr int BYTES = OFF_CTL + 256 + 1024;  // barriers + alignment slack
    // f32 accumulator D, binary16 A and B, both K-major; N >> 3 at bit 17, M >> 4 at bit 24
    static constexpr uint32_t IDESC_S = (1u << 4) | (uint32_t(AKB >> 3) << 17) | (uint32_t(AQ >> 4) << 24);
    static constexpr uint32_t IDESC_O = (1u << 4) | (uint32_t(D >> 3) << 17) | (uint32_t(AQ >> 4) << 24);
};

static_assert(AttnLayout<128>::BYTES <= 232448, "shared memory budget");

struct AttnCtl {
    uint64_t q_full, k_full[2], k_empty[2], v_full[2], v_empty[2];
    uint64_t s_full[AQT], p_full[AQT], o_done[AQT], drain;  // per query tile
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(AttnCtl) <= 256, "control block");

// Shared-memory matrix descriptor of a K-major operand with the 128-byte
// swizzle: rows 128 B apart, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t att_desc(uint32_t saddr) {
    return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

__device__ __forceinline__ void att_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void att_tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16: A is read from tensor memory
// (128 lanes = rows, 32-bit column c = elements 2c, 2c + 1 of the row).
__device__ __forceinline__ void att_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void att_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void att_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void att_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x by the hardware approximation (relative error about 2^-22; 2^-inf = 0)
__device__ __forceinline__ float att_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


// max(a, b, c) in one instruction (a NaN operand is ignored, as by fmaxf)
__device__ __forceinline__ float att_max3(float a, float b, float c) {
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

// Two f32 lanes in one 64-bit register, and their lane-wise sum (each lane
// rounded as a scalar add).
__device__ __forceinline__ uint64_t att_pack2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void att_unpack2(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t att_add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

template <int D>
__global__ void __launch_bounds__(ATHREADS, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap, float *__restrict__ out, int H, int S, int Sp, int Dout,
                unsigned int *status, uint64_t wait_ns) {
    using Lay = AttnLayout<D>;
    extern __shared__ uint8_t att_raw[];
    const uint32_t raw_addr = smem_u32(att_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    const uint32_t sbase = raw_addr + pad;
    AttnCtl *ctl = reinterpret_cast<AttnCtl *>(att_raw + pad + Lay::OFF_CTL);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qp = blockIdx.x, h = blockIdx.y;  // queries AQT * AQ * qp .. + AQT * AQ - 1 of head h
    const int nb = (S + AKB - 1) / AKB;         // key blocks
    const uint32_t sQ = sbase, sK = sbase + Lay::OFF_K, sV = sbase + Lay::OFF_V;

    if (threadIdx.x == 0) {
        mbar_init(&ctl->q_full, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->k_full[b], 1);
            mbar_init(&ctl->k_empty[b], 1);
            mbar_init(&ctl->v_full[b], 1);
            mbar_init(&ctl->v_empty[b], 1);
        }
        for (int t = 0; t < AQT; ++t) {
            mbar_init(&ctl->s_full[t], 1);
            mbar_init(&ctl->p_full[t], A_SMT);
            mbar_init(&ctl->o_done[t], 1);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_proxy_async_smem();
    }
    if (warp == A_MMA) {
        tmem_alloc(&ctl->tmem_base, ATMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort;

    if (warp == A_TMA) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&qmap)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
            // Launched right behind the binary16 pre-pass (programmatic
            // dependent launch): the set-up above overlapped its tail; its
            // output is read only from here on.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            // both query tiles (a tile past the end of the head reads other
            // rows or the fill value: its rows are computed, never written)
            att_expect_tx(&ctl->q_full, AQT * Lay::QB);
            for (int t = 0; t < AQT; ++t)
                for (int sub = 0; sub < D / 64; ++sub)
                    att_tma_2d(sQ + t * Lay::QB + sub * Lay::SUB, &qmap, sub * 64, h * Sp + (AQT * qp + t) * AQ,
                               &ctl->q_full);
            int issued = 0;
            for (int j = 0; j < nb; ++j, ++issued) {
                const int b = j & 1, u = j >> 1;
                if (u > 0 && !mbar_wait_spin(&ctl->k_empty[b], (u - 1) & 1, wait_ns, status)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                att_expect_tx(&ctl->k_full[b], Lay::KB);
                for (int sub = 0; sub < D / 64; ++sub)
                    att_tma_2d(sK + b * Lay::KB + sub * Lay::SUB, &kmap, sub * 64, h * Sp + j * AKB, &ctl->k_full[b]);
                if (u > 0 && !mbar_wait_spin(&ctl->v_empty[b], (u - 1) & 1, wait_ns, status)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                att_expect_tx(&ctl->v_full[b], Lay::VB);
                for (int sub = 0; sub < AKB / 64; ++sub)
                    att_tma_2d(sV + b * Lay::VB + sub * (D * 128), &vmap, j * AKB + sub * 64, h * D, &ctl->v_full[b]);
            }
            // every copy issued must land before the CTA exits: the last round of each slot
            const uint64_t drain = wait_ns > 1000000000ull ? wait_ns : 1000000000ull;
            mbar_wait_bounded(&ctl->q_full, 0, drain, status);
            for (int j = max(0, issued - 2); j < issued; ++j) {
                mbar_wait_bounded(&ctl->k_full[j & 1], (j >> 1) & 1, drain, status);
                mbar_wait_bounded(&ctl->v_full[j & 1], (j >> 1) & 1, drain, status);
            }
        }
        __syncwarp();
    } else if (warp == A_MMA) {
        // The whole warp runs the loop (waits, descriptors); lane 0 issues.
        // Descriptor of a shared-memory operand + byte offset d: the 16-byte
        // address field is the low 14 bits and never carries out here.
        const uint64_t dq0 = att_desc(sQ), dq1 = att_desc(sQ + Lay::QB);
        const uint64_t dk0 = att_desc(sK), dk1 = att_desc(sK + Lay::KB);
        const uint64_t dv0 = att_desc(sV), dv1 = att_desc(sV + Lay::VB);
        const bool leader = lane == 0;
        // waits by the whole warp, with one outcome for all lanes
        auto wait_all = [&](uint64_t *bar, uint32_t parity) {
            const bool got = mbar_wait_spin(bar, parity, wait_ns, status);
            return __all_sync(0xffffffffu, got && *abort_flag == 0);
        };
        // S_t of block j into columns 128 t (A = Q_t, B = K_j from shared memory)
        auto issue_s = [&](int t, int j) {
            const uint64_t a0 = t ? dq1 : dq0, b0 = (j & 1) ? dk1 : dk0;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = uint64_t((((kk >> 2) * Lay::SUB) >> 4) + 2 * (kk & 3));
                    tc_mma_f16(tmem + uint32_t(t * AKB), a0 + off, b0 + off, Lay::IDESC_S, kk > 0);
                }
                tc_commit(&ctl->s_full[t]);
            }
            __syncwarp();
        };
        // O_t += P_t V_j (A = P_t from tensor memory, B = V_j^T from shared memory)
        auto issue_pv = [&](int t, int j) {
            const uint64_t b0 = (j & 1) ? dv1 : dv0;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < AKB / 16; ++kk)
                    att_mma_ts(tmem + A_OCOL + uint32_t(t * AKB), tmem + uint32_t(t * AKB + 8 * kk),
                               b0 + uint64_t((((kk >> 2) * (D * 128)) >> 4) + 2 * (kk & 3)), Lay::IDESC_O,
                               (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&ctl->o_done[t]);
            }
            __syncwarp();
        };
        auto commit = [&](uint64_t *bar) {
            if (leader) tc_commit(bar);
            __syncwarp();
        };
        bool ok = wait_all(&ctl->q_full, 0) && wait_all(&ctl->k_full[0], 0);
        if (ok) {
            tc_fence_after();
            issue_s(0, 0);
            issue_s(1, 0);
            commit(&ctl->k_empty[0]);
        }
        for (int j = 0; j < nb && ok; ++j) {
            const bool next = j + 1 < nb;
            if (!wait_all(&ctl->v_full[j & 1], (j >> 1) & 1)) { ok = false; break; }
            for (int t = 0; t < AQT && ok; ++t) {
                // P_t of block j written by the softmax (which has also read S_t)
                if (!wait_all(&ctl->p_full[t], j & 1)) { ok = false; break; }
                tc_fence_after();
                issue_pv(t, j);
                if (t == AQT - 1) commit(&ctl->v_empty[j & 1]);
                if (next) {
                    if (t == 0 && !wait_all(&ctl->k_full[(j + 1) & 1], ((j + 1) >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(t, j + 1);
                    if (t == AQT - 1) commit(&ctl->k_empty[(j + 1) & 1]);
                }
            }
        }
        if (!ok && leader) *abort_flag = 1;
        __syncwarp();
    } else if (warp >= A_SM0) {
        const int t = (warp - A_SM0) >> 2;             // query tile
        const int quarter = warp & 3;                  // TMEM lanes 32 quarter .. + 31
        const int r = quarter * 32 + lane;             // query row in the tile = TMEM lane
        const uint32_t tl = uint32_t(quarter * 32) << 16;
        const uint32_t ts = tmem + tl + uint32_t(t * AKB);          // this row's S / P
        const uint32_t to = tmem + tl + A_OCOL + uint32_t(t * AKB); // this row's O
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nb; ++j) {
            if (!mbar_wait_spin(&ctl->s_full[t], j & 1, wait_ns, status)) *abort_flag = 1;
            if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
            tc_fence_after();
            const int kvalid = S - j * AKB;  // keys of this block below S
            // the row maximum over the valid keys
            float mx = -INFINITY;
#pragma unroll
            for (int cp = 0; cp < AKB / 64; ++cp) {
                uint32_t va[32], vb[32];
                att_ld32(ts + uint32_t(cp * 64), va);
                att_ld32(ts + uint32_t(cp * 64 + 32), vb);
                tc_wait_ld();
                if (kvalid >= AKB) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx = att_max3(mx, __uint_as_float(va[i]), __uint_as_float(vb[i]));
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (cp * 64 + i < kvalid) mx = fmaxf(mx, __uint_as_float(va[i]));
                        if (cp * 64 + 32 + i < kvalid) mx = fmaxf(mx, __uint_as_float(vb[i]));
                    }
                }
            }
            // lazy rescale: keep the running maximum unless this block's exceeds it by more than 8
            const bool grow = j == 0 || mx > m + kLazyLog2;
            const float mu = grow ? mx : m;
            const float alpha = (j > 0 && grow) ? att_ex2(m - mu) : 1.f;
            // P = 2^(s - mu) as binary16 over the first 64 columns of S (keys
            // 64 cp .. 64 cp + 63 -> columns 32 cp .. 32 cp + 31, read before written)
            // (key pairs in packed f32x2 arithmetic: s - mu and the row sum)
            const uint64_t negmu2 = att_pack2(-mu, -mu);
            uint64_t lsum2 = att_pack2(0.f, 0.f);
#pragma unroll
            for (int cp = 0; cp < AKB / 64; ++cp) {
                uint32_t va[32], vb[32], w[32];
                att_ld32(ts + uint32_t(cp * 64), va);
                att_ld32(ts + uint32_t(cp * 64 + 32), vb);
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int i = 2 * e;  // keys 64 cp + i, + i + 1
                    float s0 = __uint_as_float(i < 32 ? va[i] : vb[i - 32]);
                    float s1 = __uint_as_float(i < 32 ? va[i + 1] : vb[i - 31]);
                    if (kvalid < AKB) {
                        if (cp * 64 + i >= kvalid) s0 = -INFINITY;
                        if (cp * 64 + i + 1 >= kvalid) s1 = -INFINITY;
                    }
                    float d0, d1;
                    att_unpack2(att_add2(att_pack2(s0, s1), negmu2), d0, d1);
                    const float p0 = att_ex2(d0), p1 = att_ex2(d1);
                    lsum2 = att_add2(lsum2, att_pack2(p0, p1));
                    const __half2 hp = __floats2half2_rn(p0, p1);
                    w[e] = *reinterpret_cast<const uint32_t *>(&hp);
                }
                att_st32(ts + uint32_t(cp * 32), w);
            }
            float lsum0, lsum1;
            att_unpack2(lsum2, lsum0, lsum1);
            const float lsum = lsum0 + lsum1;
            if (j > 0 && __any_sync(0xffffffffu, grow)) {
                // rescale this row of O (rows that keep m scale by 1) once
                // P V of block j - 1 has accumulated into it
                if (!mbar_wait_spin(&ctl->o_done[t], (j - 1) & 1, wait_ns, status)) *abort_flag = 1;
                if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    att_ld32(to + uint32_t(c * 32), o);
                    tc_wait_ld();
#pragma unroll
                    for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
                    att_st32(to + uint32_t(c * 32), o);
                }
            }
            l = l * alpha + lsum;
            m = mu;
            att_wait_st();
            tc_fence_before();
            mbar_arrive(&ctl->p_full[t]);
        }
        if (ok) {
            if (!mbar_wait_spin(&ctl->o_done[t], (nb - 1) & 1, wait_ns, status)) *abort_flag = 1;
            if (!__any_sync(0xffffffffu, *abort_flag != 0)) {
                tc_fence_after();
                const float inv = 1.0f / l;
                const int tok = (AQT * qp + t) * AQ + r;
                // the head's Dout real features (the staged operands pad D to
                // the kernel's width with zeros; those columns are not written)
                float *orow = out + int64_t(tok) * H * Dout + int64_t(h) * Dout;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    if (c * 32 >= Dout) break;
                    uint32_t o[32];
                    att_ld32(to + uint32_t(c * 32), o);
                    tc_wait_ld();
                    if (tok < S) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            if (c * 32 + i < Dout)
                                *reinterpret_cast<float4 *>(orow + c * 32 + i) =
                                    make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                                                __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == A_MMA) {
        if (lane == 0) {
            // every issued MMA must be complete before TMEM is released
            tc_commit(&ctl->drain);
            const uint64_t drain = wait_ns > 1000000000ull ? wait_ns : 1000000000ull;
            mbar_wait_bounded(&ctl->drain, 0, drain, status);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, ATMEM_COLS);
    }
}

// The binary16 pre-pass in one launch, grid (nvt + nqk, H), head h = blockIdx.y:
//  * blocks x < nvt (nvt = Sp/64 * D/64): v [H][S][Din] -> binary16 v^T
//    [H][D][Sp], one 64-key x 64-feature tile through shared memory, 16-byte
//    reads and writes;
//  * the other blocks: q and k [H][S][Din] -> binary16 [H][Sp][D], 256 items of
//    8 elements per block (q times `qscale`).
// Keys past S and features past Din are zero.
__global__ void __launch_bounds__(256)
attn_prep_kernel(const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
                 __half *__restrict__ qh, __half *__restrict__ kh, __half *__restrict__ vt, int S, int Sp, int D,
                 int Din, float qscale) {
    // the attention kernel behind this one may launch now: it waits for this
    // kernel's completion before it reads any staged operand
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ __align__(16) __half tile[64][72];  // [feature][key], 8 halves of padding
    const int h = blockIdx.y;
    const int nst = Sp / 64, nvt = nst * (D / 64);
    const int t = threadIdx.x;
    if (int(blockIdx.x) < nvt) {
        const int s0 = (int(blockIdx.x) % nst) * 64, d0 = (int(blockIdx.x) / nst) * 64;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = t + 256 * i;           // 0..1023: key idx / 16, features 4 (idx % 16) .. +3
            const int key = idx >> 4, f4 = idx & 15;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s0 + key < S && d0 + 4 * f4 < Din)
                x = __ldcs(reinterpret_cast<const float4 *>(v + (int64_t(h) * S + s0 + key) * Din + d0) + f4);
            tile[4 * f4 + 0][key] = __float2half_rn(x.x);
            tile[4 * f4 + 1][key] = __float2half_rn(x.y);
            tile[4 * f4 + 2][key] = __float2half_rn(x.z);
            tile[4 * f4 + 3][key] = __float2half_rn(x.w);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int idx = t + 256 * i;           // 0..511: feature idx / 8, keys 8 (idx % 8) .. +7
            const int f = idx >> 3, c = idx & 7;
            *reinterpret_cast<uint4 *>(vt + (int64_t(h) * D + d0 + f) * Sp + s0 + 8 * c) =
                *reinterpret_cast<const uint4 *>(&tile[f][8 * c]);
        }
        return;
    }
    const int64_t per = int64_t(Sp) * (D / 8);  // items of q (or k) of one head
    const int64_t it = int64_t(int(blockIdx.x) - nvt) * 256 + t;
    if (it >= 2 * per) return;
    const bool isk = it >= per;
    const int64_t idx = isk ? it - per : it;
    const int s = int(idx / (D / 8)), g = int(idx % (D / 8));
    const float *src = isk ? k : q;
    __half *dst = isk ? kh : qh;
    const float scale = isk ? 1.0f : qscale;
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (s < S && g * 8 < Din) {
        const float4 *p = reinterpret_cast<const float4 *>(src + (int64_t(h) * S + s) * Din + g * 8);
        const float4 a = __ldcs(p), c = __ldcs(p + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
    }
    uint4 o;
    __half2 t0 = __floats2half2_rn(f[0] * scale, f[1] * scale), t1 = __floats2half2_rn(f[2] * scale, f[3] * scale);
    __half2 t2 = __floats2half2_rn(f[4] * scale, f[5] * scale), t3 = __floats2half2_rn(f[6] * scale, f[7] * scale);
    o.x = *reinterpret_cast<uint32_t *>(&t0);
    o.y = *reinterpret_cast<uint32_t *>(&t1);
    o.z = *reinterpret_cast<uint32_t *>(&t2);
    o.w = *reinterpret_cast<uint32_t *>(&t3);
    *reinterpret_cast<uint4 *>(dst + (int64_t(h) * Sp + s) * D + g * 8) = o;
}

// D: the kernel's head width (64 or 128); Din <= D the caller's (a multiple of 8)
template <int D>
cudaError_t launch_attention_d(const float *q, const float *k, const float *v, float *out, int64_t H, int64_t S,
                               int Din, void *ws, const LaunchCtx &ctx) {
    using Lay = AttnLayout<D>;
    const int64_t Sp = (S + 127) / 128 * 128;
    __half *qh = static_cast<__half *>(ws);
    __half *kh = qh + H * Sp * D;
    __half *vt = kh + H * Sp * D;
    const float qscale = 1.4426950408889634f / sqrtf(float(Din));  // log2(e) / sqrt(head dim)
    const int64_t nvt = (Sp / 64) * (D / 64), nqk = (2 * Sp * (D / 8) + 255) / 256;  // blocks per head
    attn_prep_kernel<<<dim3(unsigned(nvt + nqk), unsigned(H)), 256, 0, ctx.stream>>>(q, k, v, qh, kh, vt, int(S),
                                                                                      int(Sp), D, Din, qscale);
    cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap qmap, kmap, vmap;
    const cuuint32_t estride[2] = {1, 1};
    const cuuint64_t qkdim[2] = {cuuint64_t(D), cuuint64_t(H * Sp)};
    const cuuint64_t qkstride[1] = {cuuint64_t(D) * 2};
    const cuuint32_t qkbox[2] = {64, 128};
    const cuuint64_t vdim[2] = {cuuint64_t(Sp), cuuint64_t(H * D)};
    const cuuint64_t vstride[1] = {cuuint64_t(Sp) * 2};
    const cuuint32_t vbox[2] = {64, cuuint32_t(D)};
    if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, qh, qkdim, qkstride, qkbox, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, kh, qkdim, qkstride, qkbox, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&vmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, vt, vdim, vstride, vbox, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned((Sp / AQ + AQT - 1) / AQT), unsigned(H));
    cfg.blockDim = dim3(ATHREADS);
    cfg.dynamicSmemBytes = Lay::BYTES;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attn_fwd_kernel<D>, qmap, kmap, vmap, out, int(H), int(S), int(Sp), Din,
                           ctx.status, ctx.wait_ns);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

}  // namespace

// Head width of the kernel that serves head dim D (a multiple of 8, <= 128).
static int64_t attn_width(int64_t D) { return D <= 64 ? 64 : 128; }

size_t attention_ws_bytes(int64_t H, int64_t S, int64_t D) {
    const int64_t Sp = (S + 127) / 128 * 128;
    return size_t(3) * size_t(H) * size_t(Sp) * size_t(attn_width(D)) * 2;
}

cudaError_t launch_attention(const float *q, const float *k, const float *v, float *out, int64_t H, int64_t S,
                             int64_t D, void *ws, const LaunchCtx &ctx) {
    if (H > 65535 || S > (int64_t(1) << 24) || H * ((S + 127) / 128 * 128) > INT32_MAX) return cudaErrorInvalidValue;
    if (D < 8 || D > 128 || D % 8) return cudaErrorInvalidValue;
    if (attn_width(D) == 64) return launch_attention_d<64>(q, k, v, out, H, S, int(D), ws, ctx);
    return launch_attention_d<128>(q, k, v, out, H, S, int(D), ws, ctx);
}

}  // namespace tq2
