// Internal declarations and device helpers of the TQ2_0_g128 CUDA library.
// Everything here is sm_103a code written against the public PTX ISA
// (mbarrier, tcgen05, fences); nothing is shared with the CPU oracle.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tq2.h"

namespace tq2 {

constexpr int kBlockW = 128;    // weights per block
constexpr int kQsBytes = 32;    // code bytes per block
constexpr int kBlockBytes = 34; // qs[32] + binary16 d

// Per-launch context the API layer hands every kernel launcher.
struct LaunchCtx {
    cudaStream_t stream;
    unsigned int *status;  // device status word (TQ2_ERR_TIMEOUT is OR-ed in)
    uint64_t wait_ns;      // limit of every bounded device-side wait
    int num_sms;
};

// Views of the SoA weight buffer.
struct SoaView {
    const uint8_t *qs;   // [N][K/4]
    const __half *d;     // [N][K/128]
};

inline SoaView soa_view(const void *w_soa, int64_t n, int64_t k) {
    const uint8_t *base = static_cast<const uint8_t *>(w_soa);
    int64_t nblk = n * (k / kBlockW);
    return SoaView{base, reinterpret_cast<const __half *>(base + nblk * kQsBytes)};
}

// ---------------------------------------------------------------------------
// Kernel launchers (one per .cu file).  All return cudaError_t of the launch.
cudaError_t launch_quantize(const float *w, void *w_aos, int64_t n, int64_t k, const LaunchCtx &ctx);
cudaError_t launch_reformat(const void *w_aos, void *w_soa, int64_t n, int64_t k,
                            const LaunchCtx &ctx);
// resident: the weights are written by no work still unfinished when the call
// is enqueued, so their copies into shared memory may precede the dependency
// wait (same arithmetic and result either way).
cudaError_t launch_gemv(const void *w_soa, const float *x, const float *residual, float *out,
                        int64_t n, int64_t k, const LaunchCtx &ctx, bool resident = false);
// Fused gate/up + SwiGLU (weight rows [0, f) gate, [f, 2f) up; out [m, f]).
// cudaErrorNotSupported: shape outside the fused kernels (the caller falls back).
cudaError_t launch_gemv_swiglu(const void *w_soa, const float *x, float *out, int64_t f, int64_t k,
                               const LaunchCtx &ctx, bool resident = false);
cudaError_t launch_tc_swiglu(const void *w_soa, const float *x, float *out, int64_t m, int64_t f,
                             int64_t k, void *ws, const LaunchCtx &ctx);
size_t tc_swiglu_ws_bytes(int64_t m, int64_t k);
// out[i, j] = silu(gu[i, j]) * gu[i, f + j] for a row-major gu [m, 2f].
cudaError_t launch_swiglu_rows(const float *gu, float *out, int64_t m, int64_t f, const LaunchCtx &ctx);
cudaError_t launch_skinny(const void *w_soa, const float *x, const float *residual, float *out,
                          int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx);
cudaError_t launch_f32ref(const void *w_soa, const float *x, const float *residual, float *out,
                          int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx);
cudaError_t launch_tc(const void *w_soa, const float *x, const float *residual, float *out,
                      int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx);
// Workspace variant of the tensor-core kernel (x pre-converted to f16 tiles).
size_t tc_ws_bytes(int64_t m, int64_t n, int64_t k);  // x tiles (+ split-K partials)
int tc_ksplit(int64_t m, int64_t n, int64_t k);
cudaError_t launch_tc_ws(const void *w_soa, const float *x, const float *residual, float *out,
                         int64_t m, int64_t n, int64_t k, void *ws, const LaunchCtx &ctx);
// Operands of the tensor-core kernel: f32 x/residual/out, or binary16
// activations in the library's activation layout (x16/res16/out16).
struct TcIo {
    const float *x;
    const float *residual;
    float *out;
    const __half *x16;
    const __half *res16;
    __half *out16;
};
constexpr int TC_PLAIN = 0, TC_SWIGLU = 1, TC_ACT16 = 2;
cudaError_t launch_tc_ws_mode(const void *w_soa, const TcIo &io, int64_t m, int64_t n, int64_t k,
                              void *ws, int variant, const LaunchCtx &ctx);
// Binary16 activations in and out (out n % 16 == 0); ws: tc_act16_ws_bytes (may be 0).
size_t tc_act16_ws_bytes(int64_t m, int64_t n, int64_t k);
cudaError_t launch_tc_act16(const void *w_soa, const __half *x16, const __half *res16, __half *out16,
                            int64_t m, int64_t n, int64_t k, void *ws, const LaunchCtx &ctx);
// f32 [m, k] <-> binary16 activation layout (k % 16 == 0)
cudaError_t launch_act16_from_f32(const float *x, __half *x16, int64_t m, int64_t k, const LaunchCtx &ctx);
cudaError_t launch_act16_to_f32(const __half *x16, float *x, int64_t m, int64_t k, const LaunchCtx &ctx);
// Same kernel pair with the library's fixed device scratch (no allocation).
constexpr size_t kNoAllocScratchBytes = size_t(TQ2_NOALLOC_SCRATCH_BYTES);
cudaError_t launch_tc_noalloc(const void *w_soa, const float *x, const float *residual, float *out,
                              int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx);

// The driver's cuTensorMapEncodeTiled (null if the driver lacks it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// DiT joint attention: q, k, v head-major f32 [H, S, D] -> out token-major
// f32 [S, H*D]; D a multiple of 8 up to 128; ws: attention_ws_bytes (binary16 copies).
size_t attention_ws_bytes(int64_t H, int64_t S, int64_t D);
cudaError_t launch_attention(const float *q, const float *k, const float *v, float *out, int64_t H, int64_t S,
                             int64_t D, void *ws, const LaunchCtx &ctx);

// Skinny-M tensor-core kernel (2 <= m <= 32, k up to the shared-memory limit
// of its K slices): one launch, no workspace.  cudaErrorNotSupported outside.
bool skinny_mma_fits(int64_t m, int64_t n, int64_t k);
cudaError_t launch_skinny_mma(const void *w_soa, const float *x, const float *residual, float *out,
                              int64_t m, int64_t n, int64_t k, const LaunchCtx &ctx);

// Largest M the small-M CUDA-core kernel handles.
constexpr int64_t kSkinnyMaxM = 16;

// ---------------------------------------------------------------------------
// Device helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// One try_wait: the thread may sleep (without using issue slots) until the
// phase completes or about `hint_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity,
                                              uint32_t hint_ns = 1000000u) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false (and records
// TQ2_ERR_TIMEOUT in *status) if the phase did not complete within
// `limit_ns` of %globaltimer time.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns, unsigned int *status) {
    const uint32_t hint = limit_ns < 1000000ull ? uint32_t(limit_ns) : 1000000u;
    if (mbar_try_wait(bar, parity, hint)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity, hint)) return true;
        if (globaltimer_ns() - t0 >= limit_ns) {
            atomicOr(status, static_cast<unsigned int>(TQ2_ERR_TIMEOUT));
            return false;
        }
    }
}

// Bounded wait that spins without a suspend hint (no sleeping between polls:
// the phase is seen as soon as it completes), reading the timer only every 64
// polls.  For waits that are usually short (data that is about to land).
__device__ __forceinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                               unsigned int *status) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((it & 63u) == 0) {
            const uint64_t t = globaltimer_ns();
            if (it == 0) t0 = t;
            // (a zero limit gives up at the first poll that finds the phase open)
            if (t - t0 >= limit_ns) {
                atomicOr(status, static_cast<unsigned int>(TQ2_ERR_TIMEOUT));
                return false;
            }
        }
    }
}

// Make generic-proxy shared-memory writes visible to the async proxy
// (the tensor core reads operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --- tcgen05 ---------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, one CTA.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on an mbarrier when all previously issued tcgen05 ops of this
// thread have completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// --- streaming global loads -------------------------------------------------

__device__ __forceinline__ uint2 ldg_stream_u2(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_stream_u4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned short ldg_u16(const void *p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

}  // namespace tq2
