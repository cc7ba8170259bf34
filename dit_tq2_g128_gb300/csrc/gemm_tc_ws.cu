// Large-M tensor-core kernel, workspace variant: the activations are
// converted once to binary16 tiles in a caller-provided workspace, then the
// persistent tcgen05 kernel streams them with bulk copies.
//
// Same contraction as the in-kernel-conversion kernel (the role of the
// pages' `gemm_tq2_g128_v10_simdgroup`: weights dequantised on chip as half,
// f16 operands, f32 accumulation, staging overlapped with the matrix units;
// "oxibonsai-kernels 0.1.5 src/gpu_backend/metal_graph/pipelines.rs").  On
// sm_103a it is computed transposed, out^T = W . x^T:
//
//  * Pre-pass: x f32 [M,K] -> f16 tiles of 128 rows x 64 k (16 KB each), laid
//    out exactly as the MMA's K-major SWIZZLE_128B shared-memory image, with
//    the K permutation that matches the weight decode (pairs (i, i+8) of every
//    16-wide group).  Rows past M are zero.  Two tiles (256 x rows) form the
//    MMA's B operand of a pipeline stage.  CTAs run in clusters of two that
//    work on neighbouring weight tiles of the same x rows: each CTA copies
//    one of the two tiles with a multicast cp.async.bulk into both CTAs'
//    shared memory, which halves the L2 traffic for x.
//  * Weight codes: a 2-D TMA load of the qs plane (128 rows x 16 bytes per
//    stage).  Decoder threads each turn one row's 64 codes into (c - 1) * d
//    in f16 registers and store them as the A operand (128 rows x 64 k, the
//    same swizzled image) in shared memory.
//  * tcgen05.mma kind::f16, M = 128 weight rows, N = 256 x rows, K = 16, both
//    operands in shared memory (the tensor core's full rate), f32
//    accumulation in tensor memory.  TMEM holds two 256-column accumulators,
//    so the epilogue of one output tile (256 x rows x 128 weight rows)
//    overlaps the MMAs of the next.  Persistent clusters walk pairs of tiles.
//  * Epilogue: TMEM lane = output column, so each tcgen05.ld gives a warp 32
//    consecutive output columns of 32 output rows.  The warp stages that
//    32 x 32 block in shared memory and hands it to a TMA tensor store (or a
//    TMA reduce-add when the residual is the output itself), so the
//    global writes are issued asynchronously.  When N is not a multiple of 4 (no
//    16-byte row pitch for a tensor map) or the residual is a separate array,
//    the warp stores directly (each store still 128-byte coalesced).
//  * Roles: warp 0 issues the code TMA loads, warp 1 the MMAs (and owns TMEM),
//    warp 2 the x-tile bulk copies, warps 4-7 run the epilogue, warps 8-23
//    decode (four sets of four warps; set j fills ring slot j, i.e. the
//    stages g = j mod 4).  All mbarrier
//    waits are bounded; on a timeout the roles stop, the issued copies and
//    MMAs drain, and TMEM is freed before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <mutex>

#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int BM = 128;                  // pre-converted x tile height (rows)
constexpr int BX = 256;                  // x rows per output tile (MMA N)
constexpr int BW = 128;                  // weight rows per output tile (MMA M)
constexpr int BK = 64, STAGES = 4, CSTAGES = 4;
constexpr int A_BYTES = BM * BK * 2;     // 16 KB: one pre-converted x tile
constexpr int X_BYTES = BX * BK * 2;     // 32 KB: the B operand of one stage
constexpr int W_BYTES = BW * BK * 2;     // 16 KB: the decoded A operand of one stage
constexpr int C_BYTES = BW * BK / 4;     // 2 KB of raw codes
constexpr int NUM_THREADS = 768;
// warp 0: code TMA issuer, warp 1: MMA issuer + TMEM owner, warp 2: x-tile
// issuer, warps 4-7: epilogue, warps 8-23: decoders (four sets of four warps,
// one set per ring slot)
constexpr int TMA_WARP = 0, MMA_WARP = 1, X_WARP = 2, EPI_WARP0 = 4, DEC_WARP0 = 8;
constexpr int DEC_SETS = 4;
constexpr int NUM_DEC = 128;             // per stage: one decoder thread per weight row (64 codes)
constexpr int NUM_EPI = 128;
constexpr int EPI_NB = 1;                // staging buffers per epilogue warp
constexpr int EPI_BYTES = 32 * 32 * 4;   // one 32 x 32 f32 block
// Epilogue modes chosen by the host.
// EPI_SWIGLU: fused gate/up projection.  The N = 2F weight rows hold the gate
// projection in rows [0, F) and the up projection in rows [F, 2F); weight tile
// nw is assembled from features 64 nw .. 64 nw + 63 as four groups of 16 gate
// rows each followed by the matching 16 up rows (tile row 32 q + r: gate of
// feature 64 nw + 16 q + r for r < 16, its up row for r >= 16).  Each epilogue
// warp then holds g and u of 16 features in its lanes r and r + 16 and writes
// out[m, f] = silu(g) * u (out has F columns).
// EPI_ACT16: binary16 activations in and out (the library's activation
// layout: row-major, element i of every 16-element group stored at position
// 2i for i < 8 and 2(i-8)+1 for i >= 8, the k order of the decoded weights).
// x tiles then arrive by tensor copy with no pre-pass, and the output, in the
// same layout, is the next layer's input.
constexpr int EPI_DIRECT = 0, EPI_TMA_STORE = 1, EPI_TMA_ADD = 2, EPI_SWIGLU = 3, EPI_ACT16 = 4;

// Position of element i (0..15) of a 16-element group in the activation layout.
__host__ __device__ __forceinline__ constexpr int act16_pos(int i) { return i < 8 ? 2 * i : 2 * (i - 8) + 1; }
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;          // two f32 accumulators of BX columns
// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B f16, both
// K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t IDESC = (1u << 4) | (uint32_t(BX >> 3) << 17) | (uint32_t(BW >> 4) << 24);

struct Ctl {
    uint64_t full[STAGES];   // x tile landed (tx bytes + issuer arrival) and A decoded (decoder arrivals)
    uint64_t empty[STAGES];
    uint64_t codes_full[CSTAGES];
    uint64_t codes_empty[CSTAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t EPI_TOTAL = size_t(4) * EPI_NB * EPI_BYTES;
constexpr size_t SMEM_BYTES = size_t(STAGES) * (X_BYTES + W_BYTES) + size_t(CSTAGES) * C_BYTES +
                              EPI_TOTAL + sizeof(Ctl) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
// Decoder set j takes the stages g = j (mod 4); with ring depths that are
// multiples of 4 every ring slot is always visited by the same set, which
// keeps each set's barrier phases in step (no parity aliasing).
static_assert(STAGES % DEC_SETS == 0 && CSTAGES % DEC_SETS == 0, "ring depths vs decoder sets");
static_assert(ACC_COL + 2 * BX <= TMEM_COLS, "TMEM budget");

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

__device__ __forceinline__ uint32_t sw128_off(int r, int j) {
    return uint32_t((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Bulk copy into the same shared-memory offset of every CTA in `mask`; each
// destination's mbarrier at `bar`'s offset receives the byte count.
__device__ __forceinline__ void bulk_g2s_mc(uint32_t dst, const void *src, uint32_t bytes,
                                            uint64_t *bar, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "h"(mask)
        : "memory");
}

// Arrive on the mbarrier at `bar`'s offset in every CTA of `mask` once all
// prior tcgen05 operations of this thread have completed.
__device__ __forceinline__ void tc_commit_mc(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void tma_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                       int c3, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

// Tensor copy delivered to the same offset in every CTA of `mask`.
__device__ __forceinline__ void tma_2d_mc(uint32_t dst, const CUtensorMap *map, int x, int y,
                                          uint64_t *bar, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(mask)
        : "memory");
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                       uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Tensor store (or reduce-add) of one staged box; completion tracked by bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void tma_add_2d(const CUtensorMap *map, int x, int y, uint32_t src) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(src)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// At most EPI_NB - 1 of this thread's bulk groups may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read_nb() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(EPI_NB - 1) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Decode one 16-weight code word into 8 half2 (weights (i, i+8)), each (c-1)*d.
__device__ __forceinline__ void decode_word(uint32_t w, __half2 d2, uint32_t (&o)[8]) {
    const uint32_t w6 = w >> 6;
    const uint32_t base = 0x64006400u;
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
    o[0] = h2u(__hmul2(__hfma2(u2h(v0), s0, b0), d2));
    o[1] = h2u(__hmul2(__hfma2(u2h(v1), s2, b2), d2));
    o[2] = h2u(__hmul2(__hfma2(u2h(v2), s4, b4), d2));
    o[3] = h2u(__hmul2(__hfma2(u2h(v3), s6, b6), d2));
    o[4] = h2u(__hmul2(__hfma2(u2h(v4), s8, b8), d2));
    o[5] = h2u(__hmul2(__hfma2(u2h(v5), s4, b4), d2));
    o[6] = h2u(__hmul2(__hfma2(u2h(v6), s6, b6), d2));
    o[7] = h2u(__hmul2(__hfma2(u2h(v7), s8, b8), d2));
}

// --------------------------------------------------------------------------
// Pre-pass: x f32 [M,K] -> f16 MMA tiles.  Item = (row, 16-float group).  A
// thread converts kPrepassItems items, all loaded before any is stored; the
// grid is sized so that its blocks are resident together.  Block b also asks
// L2 for slice b of the weight planes, which the tensor kernel behind this one
// reads from its first stage on.
constexpr int kPrepassItems = 2;
constexpr int kPrepassThreads = 256;

__global__ void __launch_bounds__(kPrepassThreads)
x_to_tiles_kernel(const float *__restrict__ x, uint8_t *__restrict__ ws, int M, int K, int MT,
                  const uint8_t *__restrict__ w, int64_t wbytes) {
    // the tensor-core kernel behind this one may launch now: it waits for this
    // kernel's completion before it reads a tile
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        // L2 is the point of coherence: a prefetch cannot leave stale data behind
        const int64_t chunk = ((wbytes + gridDim.x - 1) / gridDim.x + 15) & ~int64_t(15);
        const int64_t b0 = int64_t(blockIdx.x) * chunk;
        const int64_t len = (b0 < wbytes ? (wbytes - b0 < chunk ? wbytes - b0 : chunk) : 0) & ~int64_t(15);
        if (len > 0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(w + b0), "r"(uint32_t(len)) : "memory");
    }
    const int groups = K / 16;                 // 16-float groups per row
    const int KT = K / BK;
    const int64_t items = int64_t(MT) * BM * groups;
    const int64_t nth = int64_t(gridDim.x) * blockDim.x;
    for (int64_t it0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; it0 < items; it0 += kPrepassItems * nth) {
        float f[kPrepassItems][16];
#pragma unroll
        for (int u = 0; u < kPrepassItems; ++u) {
            const int64_t it = it0 + u * nth;
            const int row = int(it / groups), g = int(it % groups);
            if (it < items && row < M) {
                const float4 *src = reinterpret_cast<const float4 *>(x + int64_t(row) * K + 16 * g);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 v = __ldg(src + q);
                    f[u][4 * q] = v.x; f[u][4 * q + 1] = v.y; f[u][4 * q + 2] = v.z; f[u][4 * q + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) f[u][i] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kPrepassItems; ++u) {
            const int64_t it = it0 + u * nth;
            if (it >= items) break;
            const int row = int(it / groups), g = int(it % groups);
            const int mt = row / BM, r = row % BM, kt = g / 4, q = g % 4;
            uint8_t *tile = ws + (int64_t(mt) * KT + kt) * A_BYTES;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint4 v;
                v.x = h2u(__floats2half2_rn(f[u][4 * h + 0], f[u][8 + 4 * h + 0]));
                v.y = h2u(__floats2half2_rn(f[u][4 * h + 1], f[u][8 + 4 * h + 1]));
                v.z = h2u(__floats2half2_rn(f[u][4 * h + 2], f[u][8 + 4 * h + 2]));
                v.w = h2u(__floats2half2_rn(f[u][4 * h + 3], f[u][8 + 4 * h + 3]));
                *reinterpret_cast<uint4 *>(tile + sw128_off(r, 2 * q + h)) = v;
            }
        }
    }
}

// --------------------------------------------------------------------------
// Main kernel.

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
tc_ws_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
             const __grid_constant__ CUtensorMap xmap, const __half *__restrict__ dpl,
             const uint8_t *__restrict__ xtiles, const float *residual, float *out, const __half *res16,
             __half *out16, int M, int N, int K, int epi_mode, int ksplit, float *partial, int after_prepass,
             unsigned int *status, uint64_t wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    const uint32_t sbase = raw_addr + pad;
    Ctl *ctl = reinterpret_cast<Ctl *>(smem_raw + pad + size_t(STAGES) * (X_BYTES + W_BYTES) +
                                       size_t(CSTAGES) * C_BYTES + EPI_TOTAL);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KT = K / BK;
    const int MT = (M + BM - 1) / BM;           // 128-row x tiles in the workspace
    const int MX = (M + BX - 1) / BX;           // 256-row output tiles
    const int NW = (N + BW - 1) / BW;
    // Tiles are walked in pairs (mx, 2*nwp + rank) by clusters of two CTAs.
    const int rank = int(cluster_rank());
    const int cl = int(blockIdx.x) >> 1, ncl = int(gridDim.x) >> 1;
    const int ntiles = MX * ((NW + 1) / 2);
    const uint16_t pair_mask = 0x3;
    // Work item t: output tile pair t / ksplit, K slice t % ksplit (split-K for
    // shapes with fewer tile pairs than clusters; slices go to `partial`).
    const int nitems = ntiles * ksplit;
    struct Item {
        int mx, nw, ks, kbeg, nk;
    };
    auto item = [&](int t) {
        Item it;
        const int tile = t / ksplit;
        it.ks = t % ksplit;
        it.mx = tile % MX;
        it.nw = 2 * (tile / MX) + rank;
        it.kbeg = int(int64_t(it.ks) * KT / ksplit);
        it.nk = int(int64_t(it.ks + 1) * KT / ksplit) - it.kbeg;
        return it;
    };
    const int64_t kb = K / kBlockW;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&ctl->full[s], NUM_DEC + 1);
            mbar_init(&ctl->empty[s], 2);  // released by the MMAs of both CTAs of the pair
        }
        for (int s = 0; s < CSTAGES; ++s) {
            mbar_init(&ctl->codes_full[s], 1);
            mbar_init(&ctl->codes_empty[s], NUM_DEC);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&ctl->tmem_full[a], 1);
            mbar_init(&ctl->tmem_empty[a], NUM_EPI);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_mbarrier_init();  // visible to the peer's multicast copies and commits
        fence_proxy_async_smem();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(&ctl->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    // the peer multicasts into this CTA's barriers: both must be initialised
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort;

    // shared memory: x ring | decoded-weight ring | code ring | epilogue staging | Ctl
    auto stage_x = [&](int s) { return sbase + uint32_t(s) * X_BYTES; };
    auto stage_w = [&](int s) { return sbase + uint32_t(STAGES) * X_BYTES + uint32_t(s) * W_BYTES; };
    auto stage_c = [&](int s) {
        return sbase + uint32_t(STAGES) * (X_BYTES + W_BYTES) + uint32_t(s) * C_BYTES;
    };
    const uint32_t ebase = sbase + uint32_t(STAGES) * (X_BYTES + W_BYTES) + uint32_t(CSTAGES) * C_BYTES;

    if (warp == TMA_WARP || warp == X_WARP) {
        // Two independent copy streams: weight codes into their own ring
        // (warp 0), this CTA's half of the x tiles into both CTAs' operand
        // rings (warp 2).
        const bool codes = warp == TMA_WARP;
        const int depth = codes ? CSTAGES : STAGES;
        if (lane == 0) {
            if (codes)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&qmap)) : "memory");
            // Launched right behind the x pre-pass (programmatic dependent
            // launch): the pre-pass writes only the x tiles, so only their
            // issuer waits for it; weight codes stream and decode meanwhile.
            // (Everything before the pre-pass completed before it started.)
            if (!codes && after_prepass) asm volatile("griddepcontrol.wait;" ::: "memory");
            int64_t g = 0;
            int last_round[STAGES > CSTAGES ? STAGES : CSTAGES];
            for (int s = 0; s < depth; ++s) last_round[s] = -1;
            bool ok = true;
            for (int t = cl; t < nitems && ok; t += ncl) {
                const Item it = item(t);
                const int mx = it.mx, nw = it.nw;
                const int mt0 = 2 * mx, nmt = min(2, MT - mt0);  // 128-row x tiles of this output tile
                for (int j = 0; j < it.nk; ++j, ++g) {
                    const int kt = it.kbeg + j;
                    const int s = int(g % depth);
                    const int u = int(g / depth);
                    uint64_t *freed = codes ? &ctl->codes_empty[s] : &ctl->empty[s];
                    if (u > 0 && !mbar_wait_spin(freed, (u - 1) & 1, wait_ns, status)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    if (*abort_flag) { ok = false; break; }
                    if (codes) {
                        mbar_expect_tx(&ctl->codes_full[s], C_BYTES);
                        if (epi_mode == EPI_SWIGLU)  // 4 feature groups x {gate, up} x 16 rows
                            tma_4d(stage_c(s), &qmap, kt * (BK / 4), 0, 0, nw * 4, &ctl->codes_full[s]);
                        else
                            tma_2d(stage_c(s), &qmap, kt * (BK / 4), nw * BW, &ctl->codes_full[s]);
                    } else {
                        // lane 0 arrives with the byte count of both halves; the
                        // CTA of rank h copies half h into both CTAs.  A half
                        // may land before that arrival (the transaction count
                        // goes transiently negative; the phase cannot complete
                        // without the arrival).
                        if (lane == 0) {
                            mbar_expect_tx(&ctl->full[s], uint32_t(nmt) * A_BYTES);
                            if (rank < nmt) {
                                if (epi_mode == EPI_ACT16)  // 128 rows x 64 k of the activation tensor
                                    tma_2d_mc(stage_x(s) + uint32_t(rank) * A_BYTES, &xmap, kt * BK,
                                              (mt0 + rank) * BM, &ctl->full[s], pair_mask);
                                else
                                    bulk_g2s_mc(stage_x(s) + uint32_t(rank) * A_BYTES,
                                                xtiles + (int64_t(mt0 + rank) * KT + kt) * A_BYTES, A_BYTES,
                                                &ctl->full[s], pair_mask);
                            }
                        }
                    }
                    last_round[s] = u;
                }
            }
            // Drain: every copy issued into shared memory must land before the
            // CTAs exit.  Code copies are awaited on their own barriers.  On
            // the normal path every x stage was consumed by both CTAs' MMAs,
            // so all x copies have landed; after an abort the stages may never
            // complete, so the issuer gives its copies in flight (a few
            // microseconds each) a fixed 200 us.  Both CTAs leave through a
            // cluster barrier, so the peer's copies into this CTA are covered
            // by the peer's own drain.
            if (codes) {
                const uint64_t drain = wait_ns > 1000000000ull ? wait_ns : 1000000000ull;
                for (int s = 0; s < depth; ++s) {
                    if (last_round[s] < 0) continue;
                    mbar_wait_bounded(&ctl->codes_full[s], last_round[s] & 1, drain, status);
                }
            } else if (!ok || *abort_flag) {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // The single-thread roles (this issuer and the two copy issuers) wait
        // by spinning: the suspend-hinted wait wakes them measurably late
        // (0.5 us per call at M=1536, N=3072; 1.4 us at N=12288).
        if (lane == 0) {
            int64_t g = 0;
            int i = 0;
            bool ok = true;
            for (int t = cl; t < nitems && ok; t += ncl, ++i) {
                const int nk = item(t).nk;
                const int a = i & 1;
                // accumulator a was last used by tile i - 2: wait for its epilogue
                if (i >= 2 && !mbar_wait_spin(&ctl->tmem_empty[a], ((i >> 1) - 1) & 1, wait_ns, status)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t dcol = tmem + ACC_COL + uint32_t(a) * BX;
                for (int j = 0; j < nk; ++j, ++g) {
                    const int s = int(g % STAGES);
                    const uint32_t par = uint32_t(g / STAGES) & 1;
                    if (!mbar_wait_spin(&ctl->full[s], par, wait_ns, status)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    if (*abort_flag) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t adesc = sw128_desc(stage_w(s));
                    const uint64_t bdesc = sw128_desc(stage_x(s));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma_f16(dcol, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (j | kk) != 0);
                    tc_commit_mc(&ctl->empty[s], pair_mask);
                }
                if (ok) tc_commit(&ctl->tmem_full[a]);
            }
        }
        __syncwarp();
    } else if (warp >= DEC_WARP0) {
        const int dset = (warp - DEC_WARP0) >> 2;  // stages g = dset (mod 4), i.e. ring slot dset
        const int pr = (warp & 3) * 32 + lane;     // weight row in the tile
        const uint32_t rsw = uint32_t(pr & 7);     // SWIZZLE_128B phase of this row
        const uint32_t rbase = uint32_t(pr >> 3) * 1024 + rsw * 128;
        int64_t gbase = 0;
        for (int t = cl; t < nitems; t += ncl) {
            const Item it = item(t);
            const int nw = it.nw;
            int row = nw * BW + pr;
            bool rvalid = row < N;
            if (epi_mode == EPI_SWIGLU) {  // tile row pr: feature 64 nw + 16 (pr / 32) + pr % 16
                const int feat = nw * (BW / 2) + (pr >> 5) * 16 + (pr & 15);
                rvalid = feat < N / 2;
                row = feat + ((pr >> 4) & 1) * (N / 2);
            }
            const __half *drow = dpl + int64_t(rvalid ? row : 0) * kb;
            const int j0 = int(((dset - gbase) % DEC_SETS + DEC_SETS) % DEC_SETS);
            // the scale of this thread's next stage, loaded one stage ahead
            uint32_t dnext = (rvalid && j0 < it.nk) ? ldg_u16(drow + ((it.kbeg + j0) >> 1)) : 0u;
            bool stop = false;
            for (int j = j0; j < it.nk; j += DEC_SETS) {
                const int kt = it.kbeg + j;
                const int64_t g = gbase + j;
                const int cs = int(g % CSTAGES);
                const int s = int(g % STAGES);
                const uint32_t dbits = dnext;
                if (rvalid && j + DEC_SETS < it.nk) dnext = ldg_u16(drow + ((kt + DEC_SETS) >> 1));
                if (!mbar_wait_bounded(&ctl->codes_full[cs], uint32_t(g / CSTAGES) & 1, wait_ns,
                                       status)) {
                    *abort_flag = 1;
                    stop = true;
                }
                uint4 code = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
                if (!stop)
                    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(code.x), "=r"(code.y), "=r"(code.z), "=r"(code.w)
                                 : "r"(stage_c(cs) + uint32_t(pr) * 16)
                                 : "memory");
                mbar_arrive(&ctl->codes_empty[cs]);
                // decode into registers first, then wait for the slot
                const __half2 d2 =
                    __half2half2(__ushort_as_half(static_cast<unsigned short>(rvalid ? dbits : 0u)));
                uint32_t o[4][8];
                decode_word(code.x, d2, o[0]);
                decode_word(code.y, d2, o[1]);
                decode_word(code.z, d2, o[2]);
                decode_word(code.w, d2, o[3]);
                // the A slot is free once the MMAs of its previous round completed
                const int u = int(g / STAGES);
                if (!stop && u > 0 && !mbar_wait_bounded(&ctl->empty[s], (u - 1) & 1, wait_ns, status)) {
                    *abort_flag = 1;
                    stop = true;
                }
                if (stop || *abort_flag) break;
                // word w (k 16w..16w+15 of the stage) -> 16-byte chunks 2w, 2w+1 of the row
                const uint32_t wbase = stage_w(s) + rbase;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(wbase + (((2 * w) ^ rsw) << 4)),
                                 "r"(o[w][0]), "r"(o[w][1]), "r"(o[w][2]), "r"(o[w][3])
                                 : "memory");
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(wbase + (((2 * w + 1) ^ rsw) << 4)),
                                 "r"(o[w][4]), "r"(o[w][5]), "r"(o[w][6]), "r"(o[w][7])
                                 : "memory");
                }
                // make the generic-proxy stores visible to the tensor core
                fence_proxy_async_smem();
                mbar_arrive(&ctl->full[s]);
            }
            gbase += it.nk;
            if (__any_sync(0xffffffffu, stop || *abort_flag)) break;
        }
        // The decoders then join the epilogue of the CTA's last tile (plain f32
        // output): 20 warps instead of 4 drain its accumulator, five per TMEM
        // lane quarter, chunk c of 32 columns to worker c % 5 (worker 0 is the
        // epilogue warp).  With one tile per CTA (M=1536, N=3072) the epilogue
        // is otherwise exposed: 4.0 -> 2.5 us.
        {
            const int cnt = cl < nitems ? (nitems - 1 - cl) / ncl + 1 : 0;
            const bool wide = cnt > 0 && ksplit == 1 && (epi_mode == EPI_DIRECT || epi_mode == EPI_TMA_STORE);
            if (wide && !__any_sync(0xffffffffu, *abort_flag != 0)) {
                const int il = cnt - 1;
                const Item it = item(cl + il * ncl);
                const int a = il & 1;
                const int quarter = warp & 3, worker = 1 + ((warp - DEC_WARP0) >> 2);
                if (!mbar_wait_bounded(&ctl->tmem_full[a], (il >> 1) & 1, wait_ns, status)) *abort_flag = 1;
                if (!__any_sync(0xffffffffu, *abort_flag != 0)) {
                    tc_fence_after();
                    const int col = it.nw * BW + quarter * 32 + lane;
                    for (int c = worker; c < BX / 32; c += 5) {
                        uint32_t r[32];
                        tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + ACC_COL + uint32_t(a) * BX +
                                      uint32_t(c * 32),
                                  r);
                        tc_wait_ld();
                        const int row0 = it.mx * BX + c * 32;
                        if (row0 < M && col < N) {
                            const int nr = min(32, M - row0);  // rows of this block inside the output
                            float *op = out + int64_t(row0) * N + col;
                            const float *rp = residual ? residual + int64_t(row0) * N + col : nullptr;
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < nr) op[int64_t(j) * N] = __uint_as_float(r[j]) + (rp ? rp[int64_t(j) * N] : 0.f);
                        }
                    }
                }
            }
        }
    } else if (warp >= EPI_WARP0) {
        const int quarter = warp - EPI_WARP0;  // TMEM lanes 32*quarter .. +31 = output columns
        const uint32_t ebuf = ebase + uint32_t(quarter) * EPI_NB * EPI_BYTES;
        int i = 0, e = 0;
        for (int t = cl; t < nitems; t += ncl, ++i) {
            const Item it = item(t);
            const int mx = it.mx, nw = it.nw;
            // a K slice of a split problem writes its partial sums, plainly
            float *const dst = ksplit > 1 ? partial + int64_t(it.ks) * M * N : out;
            const float *const res = ksplit > 1 ? nullptr : residual;
            const int mode = ksplit > 1 ? EPI_DIRECT : epi_mode;  // (never split with swiglu)
            const int a = i & 1;
            {
                // The residual this warp adds (its 32 columns of the tile's 256
                // rows) goes to L2 while the tile's MMAs run: the epilogue's
                // loads then wait on L2, not on DRAM.
                const int pcol = nw * BW + quarter * 32;
                if (pcol < N && (mode == EPI_DIRECT || mode == EPI_ACT16)) {
                    const bool h16 = mode == EPI_ACT16;
                    const char *rb = h16 ? reinterpret_cast<const char *>(res16) : reinterpret_cast<const char *>(res);
                    if (rb) {
                        const int esz = h16 ? 2 : 4;
                        const int ncol = min(32, N - pcol);
                        for (int rr = lane; rr < BX; rr += 32) {
                            const int row = mx * BX + rr;
                            if (row >= M) break;
                            const char *p0 = rb + (int64_t(row) * N + pcol) * esz;
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(p0));
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(p0 + ncol * esz - 1));
                        }
                    }
                }
            }
            if (!mbar_wait_bounded(&ctl->tmem_full[a], (i >> 1) & 1, wait_ns, status)) *abort_flag = 1;
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            tc_fence_after();
            const int col0 = nw * BW + quarter * 32;
            const int col = col0 + lane;
            // the last tile's chunks are shared with the decoder warps (above)
            const int cnt = cl < nitems ? (nitems - 1 - cl) / ncl + 1 : 0;
            const bool wide = i == cnt - 1 && ksplit == 1 && (epi_mode == EPI_DIRECT || epi_mode == EPI_TMA_STORE);
            for (int c = 0; c < BX / 32; c += wide ? 5 : 1) {
                uint32_t r[32];
                tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + ACC_COL + uint32_t(a) * BX +
                              uint32_t(c * 32),
                          r);
                tc_wait_ld();
                if (c == BX / 32 - 1) {
                    tc_fence_before();
                    mbar_arrive(&ctl->tmem_empty[a]);
                }
                const int row0 = mx * BX + c * 32;
                if (mode == EPI_SWIGLU) {
                    // lanes r and r + 16 hold g and u of feature 64 nw + 16 quarter + r
                    const int F = N / 2;
                    const int feat = nw * (BW / 2) + quarter * 16 + (lane & 15);
                    const int nr = row0 < M ? min(32, M - row0) : 0;
                    float *op = out + int64_t(row0) * F + feat;
                    // the pair splits the block's 32 rows: lane r takes rows 0..15,
                    // lane r + 16 rows 16..31 (each swaps the other half with its
                    // partner), so that each lane evaluates 16 activations.
                    // Fast exp and division here (relative error ~1e-6, far inside
                    // the f16 path's bound): the activation shares the issue slots
                    // of the SM with the weight decoders.
                    const bool lo = lane < 16;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float a0 = __shfl_xor_sync(0xffffffffu, __uint_as_float(r[jj]), 16);
                        const float a1 = __shfl_xor_sync(0xffffffffu, __uint_as_float(r[jj + 16]), 16);
                        const float g = lo ? __uint_as_float(r[jj]) : a1;
                        const float u = lo ? a0 : __uint_as_float(r[jj + 16]);
                        const int j = lo ? jj : jj + 16;
                        if (feat < F && j < nr) op[int64_t(j) * F] = __fdividef(g, 1.0f + __expf(-g)) * u;
                    }
                    continue;
                }
                if (row0 >= M || col0 >= N) continue;  // block wholly outside the output
                if (mode == EPI_ACT16) {
                    // binary16 out (and residual) at the activation-layout position of col
                    if (col >= N) continue;
                    const int nr = min(32, M - row0);
                    const int64_t pc = (col & ~15) | act16_pos(col & 15);
                    __half *op = out16 + int64_t(row0) * N + pc;
                    const __half *rp = res16 ? res16 + int64_t(row0) * N + pc : nullptr;
                    if (rp) {
                        // eight residual loads in flight before their first use
#pragma unroll
                        for (int h = 0; h < 32; h += 8) {
                            float rv[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                rv[j] = h + j < nr ? __half2float(rp[int64_t(h + j) * N]) : 0.f;
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (h + j < nr)
                                    op[int64_t(h + j) * N] = __float2half_rn(__uint_as_float(r[h + j]) + rv[j]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nr) op[int64_t(j) * N] = __float2half_rn(__uint_as_float(r[j]));
                    }
                    continue;
                }
                if (mode == EPI_DIRECT) {
                    if (col >= N) continue;
                    const int nr = min(32, M - row0);  // rows of this block inside the output
                    float *op = dst + int64_t(row0) * N + col;
                    if (res) {
                        // 16 residual loads in flight before their first use
                        const float *rp = res + int64_t(row0) * N + col;
#pragma unroll
                        for (int h = 0; h < 32; h += 16) {
                            float rv[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                rv[j] = h + j < nr ? __ldcs(rp + int64_t(h + j) * N) : 0.f;
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (h + j < nr) op[int64_t(h + j) * N] = __uint_as_float(r[h + j]) + rv[j];
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nr) op[int64_t(j) * N] = __uint_as_float(r[j]);
                    }
                } else {
                    // Stage the 32 x 32 block (row j, column lane) and hand it
                    // to the tensor engine; rows >= M and columns >= N of the
                    // box are clipped by the tensor map.
                    const uint32_t buf = ebuf + uint32_t(e % EPI_NB) * EPI_BYTES;
                    if (lane == 0) bulk_wait_read_nb();  // the store that last used buf has read it
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        asm volatile("st.shared.b32 [%0], %1;" ::"r"(buf + uint32_t(j) * 128 + uint32_t(lane) * 4),
                                     "r"(r[j])
                                     : "memory");
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (mode == EPI_TMA_ADD)
                            tma_add_2d(&omap, col0, row0, buf);
                        else
                            tma_store_2d(&omap, col0, row0, buf);
                        bulk_commit();
                    }
                    ++e;
                }
            }
        }
        // every tensor store must have finished before the CTA's shared memory goes away
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        if (lane == 0) {
            // Every issued MMA must be complete before TMEM is released: one
            // more commit arrives once all of them have finished.
            tc_commit(&ctl->drain);
            const uint64_t drain = wait_ns > 1000000000ull ? wait_ns : 1000000000ull;
            mbar_wait_bounded(&ctl->drain, 0, drain, status);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    // The peer may still arrive on this CTA's barriers until its own MMAs
    // have drained: leave together.
    cluster_sync();
}

// Activation-layout variant of the reduction: binary16 out (and residual) at
// the layout position of each column.
__global__ void __launch_bounds__(256)
ksplit_reduce_act16_kernel(const float *__restrict__ part, int S, int64_t m, int64_t n,
                           const __half *res16, __half *out16) {
    const int64_t mn = m * n, stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < mn; i += stride) {
        float acc = part[i];
        for (int s = 1; s < S; ++s) acc += part[int64_t(s) * mn + i];
        const int64_t r = i / n, c = i - r * n;
        const int64_t o = r * n + ((c & ~int64_t(15)) | act16_pos(int(c & 15)));
        if (res16) acc += __half2float(res16[o]);
        out16[o] = __float2half_rn(acc);
    }
}

// out = sum of the K-slice partials in slice order (+ residual): deterministic.
__global__ void __launch_bounds__(256)
ksplit_reduce_kernel(const float *__restrict__ part, int S, int64_t mn, const float *residual,
                     float *out) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    const int64_t i0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if ((mn & 3) == 0) {
        const int64_t n4 = mn / 4;
        const float4 *p4 = reinterpret_cast<const float4 *>(part);
        for (int64_t i = i0; i < n4; i += stride) {
            float4 acc = __ldcs(p4 + i);
            for (int s = 1; s < S; ++s) {
                const float4 v = __ldcs(p4 + int64_t(s) * n4 + i);
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
            if (residual) {
                const float4 r = reinterpret_cast<const float4 *>(residual)[i];
                acc.x += r.x; acc.y += r.y; acc.z += r.z; acc.w += r.w;
            }
            reinterpret_cast<float4 *>(out)[i] = acc;
        }
    } else {
        for (int64_t i = i0; i < mn; i += stride) {
            float acc = part[i];
            for (int s = 1; s < S; ++s) acc += part[int64_t(s) * mn + i];
            if (residual) acc += residual[i];
            out[i] = acc;
        }
    }
}

std::mutex g_noalloc_mu;
uint8_t *g_noalloc_ptr[64];  // device address of the scratch array, per device

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Fixed scratch of the allocation-free entry point (tq2_gemm_noalloc): the
// binary16 activation tiles live here instead of in a caller workspace.  Being
// a file-scope device array, it is reserved on every device that loads this
// library and stays reserved until the process exits.  All calls share it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

cudaError_t launch_tc_noalloc(const void *w_soa, const float *x, const float *residual, float *out,
                              int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx) {
    // (the API layer has checked the shape against the scratch size)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    uint8_t *scratch = nullptr;
    {
        // One-time set-up per device, with that device current: the host-side
        // name of the array is not a device address, so ask the runtime for it.
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return e;
            g_noalloc_ptr[dev] = static_cast<uint8_t *>(p);
        }
        scratch = g_noalloc_ptr[dev];
    }
    return launch_tc_ws(w_soa, x, residual, out, m, n, k, scratch, ctx);
}

// K slices per output tile pair when `pairs` CTA pairs are available: enough
// work items for all of them when the shape has fewer tile pairs, at least 4
// stages per slice, at most 16 slices.
static int ksplit_for(int64_t m, int64_t n, int64_t k, int64_t pairs) {
    const int64_t tiles = ((m + BX - 1) / BX) * ((((n + BW - 1) / BW) + 1) / 2);
    int64_t s = tiles < pairs ? pairs / tiles : 1;
    s = std::min<int64_t>(s, (k / BK) / 4);
    s = std::min<int64_t>(s, 16);
    return int(std::max<int64_t>(s, 1));
}

// The split the workspace is sized for: a function of the shape only (callers
// size workspaces without a device), computed for the 76 CTA pairs of a
// 152-SM GB300.  A launch uses the split of the device it runs on, capped by
// this one (what the workspace holds).
constexpr int64_t kWsPairs = 76;
int tc_ksplit(int64_t m, int64_t n, int64_t k) { return ksplit_for(m, n, k, kWsPairs); }

static size_t x_tile_bytes(int64_t m, int64_t k) {
    const int64_t mt = (m + BM - 1) / BM;
    return size_t(mt) * BM * size_t(k) * 2;
}

size_t tc_ws_bytes(int64_t m, int64_t n, int64_t k) {
    const size_t xb = x_tile_bytes(m, k);
    const int s = tc_ksplit(m, n, k);
    if (s == 1) return xb;
    return ((xb + 255) & ~size_t(255)) + size_t(s) * size_t(m) * size_t(n) * 4;
}

size_t tc_swiglu_ws_bytes(int64_t m, int64_t k) { return x_tile_bytes(m, k); }

// Activation-layout GEMM: the workspace holds only split-K partials (x needs no tiles).
size_t tc_act16_ws_bytes(int64_t m, int64_t n, int64_t k) {
    const int s = tc_ksplit(m, n, k);
    return s == 1 ? 0 : size_t(s) * size_t(m) * size_t(n) * 4;
}

cudaError_t launch_tc_ws(const void *w_soa, const float *x, const float *residual, float *out,
                         int64_t m, int64_t n, int64_t k, void *ws, const LaunchCtx &ctx) {
    TcIo io{x, residual, out, nullptr, nullptr, nullptr};
    return launch_tc_ws_mode(w_soa, io, m, n, k, ws, TC_PLAIN, ctx);
}

cudaError_t launch_tc_swiglu(const void *w_soa, const float *x, float *out, int64_t m, int64_t f,
                             int64_t k, void *ws, const LaunchCtx &ctx) {
    if (f % 16) return cudaErrorNotSupported;  // whole 16-row groups in the 4-D view
    TcIo io{x, nullptr, out, nullptr, nullptr, nullptr};
    return launch_tc_ws_mode(w_soa, io, m, 2 * f, k, ws, TC_SWIGLU, ctx);
}

cudaError_t launch_tc_act16(const void *w_soa, const __half *x16, const __half *res16, __half *out16,
                            int64_t m, int64_t n, int64_t k, void *ws, const LaunchCtx &ctx) {
    if (n % 16) return cudaErrorInvalidValue;  // whole 16-element groups in the output layout
    TcIo io{nullptr, nullptr, nullptr, x16, res16, out16};
    return launch_tc_ws_mode(w_soa, io, m, n, k, ws, TC_ACT16, ctx);
}

cudaError_t launch_tc_ws_mode(const void *w_soa, const TcIo &io, int64_t m, int64_t n, int64_t k,
                              void *ws, int variant, const LaunchCtx &ctx) {
    if (m > INT32_MAX || n > INT32_MAX || k > INT32_MAX) return cudaErrorInvalidValue;
    const bool swiglu = variant == TC_SWIGLU, act16 = variant == TC_ACT16;
    const SoaView v = soa_view(w_soa, n, k);
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap qmap;
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    if (swiglu) {
        // codes viewed as [F/16 groups][2: gate, up][16 rows][K/4 bytes]
        // (innermost first below); one box = 4 groups x 2 halves x 16 rows x 16 bytes
        const int64_t f = n / 2;
        const cuuint64_t gdim[4] = {cuuint64_t(k / 4), 16, 2, cuuint64_t(f / 16)};
        const cuuint64_t gstride[3] = {cuuint64_t(k / 4), cuuint64_t(f) * cuuint64_t(k / 4),
                                       16 * cuuint64_t(k / 4)};
        const cuuint32_t box[4] = {BK / 4, 16, 2, 4};
        if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t *>(v.qs), gdim, gstride, box,
                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        const cuuint64_t gdim[2] = {cuuint64_t(k / 4), cuuint64_t(n)};
        const cuuint64_t gstride[1] = {cuuint64_t(k / 4)};
        const cuuint32_t box[2] = {BK / 4, BW};
        if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(v.qs), gdim, gstride, box,
                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // binary16 activations: 128-row x 64-k boxes of x with the 128-byte swizzle,
    // the layout of the MMA's B operand (rows past m arrive as zeros)
    CUtensorMap xmap;
    std::memset(&xmap, 0, sizeof(xmap));
    if (act16) {
        const cuuint64_t xdim[2] = {cuuint64_t(k), cuuint64_t(m)};
        const cuuint64_t xstride[1] = {cuuint64_t(k) * 2};
        const cuuint32_t xbox[2] = {BK, BM};
        if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(io.x16), xdim, xstride, xbox,
                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // Output tensor map for the TMA epilogue: needs a 16-byte row pitch (n % 4
    // == 0; the base is 16-byte aligned by the API's checks) and either no
    // residual or an in-place residual (reduce-add into out).
    int epi_mode = swiglu ? EPI_SWIGLU : act16 ? EPI_ACT16 : EPI_DIRECT;
    CUtensorMap omap;
    std::memset(&omap, 0, sizeof(omap));
    if (variant == TC_PLAIN && n % 4 == 0 && (io.residual == nullptr || io.residual == io.out)) {
        const cuuint64_t odim[2] = {cuuint64_t(n), cuuint64_t(m)};
        const cuuint64_t ostride[1] = {cuuint64_t(n) * 4};
        const cuuint32_t obox[2] = {32, 32};
        if (enc(&omap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, io.out, odim, ostride, obox, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
            epi_mode = io.residual ? EPI_TMA_ADD : EPI_TMA_STORE;
    }
    cudaError_t e;
    if (!act16) {
        // pre-pass: f32 x -> binary16 MMA tiles in the workspace
        const int MT = int((m + BM - 1) / BM);
        const int64_t items = int64_t(MT) * BM * (k / 16);
        const int64_t per_block = int64_t(kPrepassThreads) * kPrepassItems;
        const int64_t pgrid = std::min<int64_t>((items + per_block - 1) / per_block, int64_t(ctx.num_sms) * 4);
        const int64_t wbytes = n * (k / kBlockW) * (kQsBytes + 2);  // code and scale planes
        x_to_tiles_kernel<<<unsigned(pgrid), kPrepassThreads, 0, ctx.stream>>>(
            io.x, static_cast<uint8_t *>(ws), int(m), int(k), MT, static_cast<const uint8_t *>(w_soa), wbytes);
        e = cudaPeekAtLastError();
        if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(tc_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    // clusters of two CTAs, each cluster a pair of neighbouring weight tiles
    // (times the K slices of a split problem)
    const int ksplit =
        swiglu ? 1 : std::min(tc_ksplit(m, n, k), ksplit_for(m, n, k, std::max(1, ctx.num_sms / 2)));
    float *partial = nullptr;
    if (ksplit > 1)
        partial = act16 ? static_cast<float *>(ws)
                        : reinterpret_cast<float *>(static_cast<uint8_t *>(ws) +
                                                    ((x_tile_bytes(m, k) + 255) & ~size_t(255)));
    const int64_t nitems = ((m + BX - 1) / BX) * ((((n + BW - 1) / BW) + 1) / 2) * ksplit;
    const int64_t grid = 2 * std::min<int64_t>(nitems, ctx.num_sms / 2);
    {
        // behind the pre-pass: programmatic dependent launch (see the x issuer)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(grid));
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cfg.stream = ctx.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = act16 ? 0 : 1;
        const int after_prepass = act16 ? 0 : 1;
        e = cudaLaunchKernelEx(&cfg, tc_ws_kernel, qmap, omap, xmap, v.d, static_cast<const uint8_t *>(ws),
                               io.residual, io.out, io.res16, io.out16, int(m), int(n), int(k), epi_mode, ksplit,
                               partial, after_prepass, ctx.status, ctx.wait_ns);
    }
    if (e == cudaSuccess) e = cudaPeekAtLastError();
    if (e != cudaSuccess || ksplit == 1) return e;
    const int64_t mn = m * n;
    const int64_t rgrid = std::min<int64_t>((mn / 4 + 255) / 256 + 1, int64_t(ctx.num_sms) * 8);
    if (act16)
        ksplit_reduce_act16_kernel<<<unsigned(rgrid), 256, 0, ctx.stream>>>(partial, ksplit, m, n, io.res16,
                                                                            io.out16);
    else
        ksplit_reduce_kernel<<<unsigned(rgrid), 256, 0, ctx.stream>>>(partial, ksplit, mn, io.residual, io.out);
    return cudaPeekAtLastError();
}

}  // namespace tq2
