// C-ABI entry points: host-side validation, kernel choice by shape, launch.
//
// The contract follows "oxibonsai-image 0.2.2 src/gpu.rs" (`ternary_matmul_gpu`
// and its module doc "Correctness contract"): row-major f32 input[M,K],
// out-major TQ2_0_g128 weight blocks [N, K/128], f32 out[M,N] written in full,
// K a multiple of 128.  Unlike the page, every failure is a returned status
// and there is no CPU fallback.
#include <atomic>
#include <initializer_list>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "tq2_internal.cuh"

namespace {

// Device status word: kernels OR TQ2_ERR_TIMEOUT into it when a bounded wait
// gives up.  Static device memory of this module (one word per device).
__device__ unsigned int g_device_status;

std::atomic<uint64_t> g_wait_ns{2000000000ull};

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    int checked = 0;    // 0 = not yet, 1 = supported, -1 = unsupported
    int num_sms = 0;
    unsigned int *status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Looks up (once per device) whether the current device is sm_103 and where
// its status word lives.
int current_device(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ2_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TQ2_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    if (d.checked == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TQ2_ERR_CUDA;
        if (major != 10 || minor != 3) {
            d.checked = -1;
        } else {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return TQ2_ERR_CUDA;
            d.status = static_cast<unsigned int *>(p);
            d.num_sms = sms;
            d.checked = 1;
        }
    }
    if (d.checked < 0) return TQ2_ERR_UNSUPPORTED_DEVICE;
    *out = d;
    return TQ2_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every operand a kernel reads or writes (through plain accesses, tensor maps,
// bulk copies or the tensor kernels' cluster-multicast copies) must be device
// memory of the current device: host memory, managed memory and another
// GPU's memory (peer or imported mappings) are refused before any launch.
// NULL pointers pass (the callers check them where they are required).
bool on_current_device(const void *p, int dev) {
    if (!p) return true;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // not a pointer the runtime knows: not device memory
        return false;
    }
    return a.type == cudaMemoryTypeDevice && a.device == dev;
}

int check_local(std::initializer_list<const void *> ptrs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ2_ERR_CUDA;
    for (const void *p : ptrs)
        if (!on_current_device(p, dev)) return TQ2_ERR_INVALID_ARG;
    return TQ2_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na && nb && x < y + nb && y < x + na;
}

// Shape-only checks.  Returns TQ2_OK and sets *noop when there is nothing
// to compute.
int check_shape(int64_t m, int64_t n, int64_t k, bool *noop) {
    *noop = false;
    if (k <= 0 || k % tq2::kBlockW) return TQ2_ERR_BAD_K;
    if (m < 0 || n < 0) return TQ2_ERR_INVALID_ARG;
    const int64_t lim = int64_t(1) << 40;  // element counts beyond this are rejected
    if (k > lim || m > lim || n > lim || (m && k > lim / m) || (n && k > lim / n) ||
        (m && n > lim / m))
        return TQ2_ERR_INVALID_ARG;
    if (m == 0 || n == 0) *noop = true;
    return TQ2_OK;
}

// Shape and pointer checks shared by every matmul entry point.
int check_matmul(const void *w, const float *x, const float *residual, const float *out,
                 int64_t m, int64_t n, int64_t k, bool *noop) {
    int st = check_shape(m, n, k, noop);
    if (st != TQ2_OK || *noop) return st;
    if (!w || !x || !out) return TQ2_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(x) || !aligned16(out) || (residual && !aligned16(residual)))
        return TQ2_ERR_MISALIGNED;
    const size_t wb = size_t(n) * size_t(k / tq2::kBlockW) * tq2::kBlockBytes;
    const size_t xb = size_t(m) * size_t(k) * 4, ob = size_t(m) * size_t(n) * 4;
    if (overlaps(out, ob, x, xb) || overlaps(out, ob, w, wb)) return TQ2_ERR_INVALID_ARG;
    if (residual && residual != out && overlaps(out, ob, residual, ob)) return TQ2_ERR_INVALID_ARG;
    return TQ2_OK;
}

int make_ctx(cudaStream_t stream, tq2::LaunchCtx *ctx) {
    DeviceInfo d;
    int st = current_device(&d);
    if (st != TQ2_OK) return st;
    ctx->stream = stream;
    ctx->status = d.status;
    ctx->wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    ctx->num_sms = d.num_sms;
    return TQ2_OK;
}

// Launch context for the current device, then the residency check of every
// operand the call's kernels touch (see on_current_device).
int prepare(void *stream, tq2::LaunchCtx *ctx, std::initializer_list<const void *> ptrs) {
    int st = make_ctx(static_cast<cudaStream_t>(stream), ctx);
    if (st != TQ2_OK) return st;
    return check_local(ptrs);
}

int finish(cudaError_t e) { return e == cudaSuccess ? TQ2_OK : TQ2_ERR_CUDA; }

// M at and above which the tcgen05 kernel beats the f32 CUDA-core small-M kernel.
// (measured at K = N = 4096: M=2 15.4 vs 17.6 us, M=3 20.8 vs 17.6 us)
constexpr int64_t kTcMinM = 3;
// Largest M that tq2_gemm sends to the one-launch skinny tensor-core kernel.
constexpr int64_t kSkinnyMmaMaxM = 32;

}  // namespace

extern "C" {

size_t tq2_soa_bytes(int64_t n, int64_t k) {
    if (n < 0 || k <= 0 || k % tq2::kBlockW) return 0;
    return size_t(n) * size_t(k / tq2::kBlockW) * tq2::kBlockBytes;
}

const char *tq2_status_string(int status) {
    switch (status) {
        case TQ2_OK: return "TQ2_OK";
        case TQ2_ERR_INVALID_ARG: return "TQ2_ERR_INVALID_ARG: null pointer, negative size, overlap or size overflow";
        case TQ2_ERR_BAD_K: return "TQ2_ERR_BAD_K: k must be a positive multiple of 128";
        case TQ2_ERR_MISALIGNED: return "TQ2_ERR_MISALIGNED: device pointers must be 16-byte aligned";
        case TQ2_ERR_UNSUPPORTED_DEVICE: return "TQ2_ERR_UNSUPPORTED_DEVICE: needs compute capability 10.3 (sm_103a)";
        case TQ2_ERR_CUDA: return "TQ2_ERR_CUDA: CUDA launch or runtime error";
        case TQ2_ERR_TIMEOUT: return "TQ2_ERR_TIMEOUT: a bounded device-side wait expired";
        case TQ2_ERR_TOO_LARGE: return "TQ2_ERR_TOO_LARGE: the shape needs more scratch than tq2_gemm_noalloc has";
        default: return "unknown tq2 status";
    }
}

int tq2_version(void) { return 0x000100; }

uint64_t tq2_set_wait_timeout_ns(uint64_t ns) { return g_wait_ns.exchange(ns); }

int tq2_device_status(void *stream) {
    DeviceInfo d;
    int st = current_device(&d);
    if (st != TQ2_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TQ2_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpy(&v, d.status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return TQ2_ERR_CUDA;
    if (cudaMemcpy(d.status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return TQ2_ERR_CUDA;
    return (v & TQ2_ERR_TIMEOUT) == TQ2_ERR_TIMEOUT ? TQ2_ERR_TIMEOUT : TQ2_OK;
}

int tq2_select_kernel(int64_t m, int64_t n, int64_t k) {
    if (m == 1) return TQ2_KERNEL_GEMV;
    if (m <= kSkinnyMmaMaxM && tq2::skinny_mma_fits(m, n, k)) return TQ2_KERNEL_SKINNY_MMA;
    if (m < kTcMinM && m <= tq2::kSkinnyMaxM) return TQ2_KERNEL_SKINNY;
    return TQ2_KERNEL_TC;
}

int tq2_reformat_aos_to_soa(const void *w_aos, void *w_soa, int64_t n, int64_t k, void *stream) {
    if (k <= 0 || k % tq2::kBlockW) return TQ2_ERR_BAD_K;
    if (n < 0 || n > (int64_t(1) << 40) / (k / tq2::kBlockW)) return TQ2_ERR_INVALID_ARG;
    if (n == 0) return TQ2_OK;
    if (!w_aos || !w_soa) return TQ2_ERR_INVALID_ARG;
    if (!aligned16(w_soa)) return TQ2_ERR_MISALIGNED;
    if (overlaps(w_aos, tq2_soa_bytes(n, k), w_soa, tq2_soa_bytes(n, k))) return TQ2_ERR_INVALID_ARG;
    tq2::LaunchCtx ctx;
    int st = prepare(stream, &ctx, {w_aos, w_soa});
    if (st != TQ2_OK) return st;
    return finish(tq2::launch_reformat(w_aos, w_soa, n, k, ctx));
}

int tq2_quantize_f32(const float *w, void *w_aos, int64_t n, int64_t k, void *stream) {
    if (k <= 0 || k % tq2::kBlockW) return TQ2_ERR_BAD_K;
    if (n < 0 || n > (int64_t(1) << 40) / k) return TQ2_ERR_INVALID_ARG;
    if (n == 0) return TQ2_OK;
    if (!w || !w_aos) return TQ2_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(w_aos)) return TQ2_ERR_MISALIGNED;
    if (overlaps(w, size_t(n) * size_t(k) * 4, w_aos, tq2_soa_bytes(n, k))) return TQ2_ERR_INVALID_ARG;
    tq2::LaunchCtx ctx;
    int st = prepare(stream, &ctx, {w, w_aos});
    if (st != TQ2_OK) return st;
    return finish(tq2::launch_quantize(w, w_aos, n, k, ctx));
}

int tq2_gemm_with(int kernel, const void *w_soa, const float *x, const float *residual,
                  float *out, int64_t m, int64_t n, int64_t k, void *stream) {
    bool noop = false;
    int st = check_matmul(w_soa, x, residual, out, m, n, k, &noop);
    if (st != TQ2_OK || noop) return st;
    if (kernel == TQ2_KERNEL_AUTO) kernel = tq2_select_kernel(m, n, k);
    if (kernel == TQ2_KERNEL_GEMV && m != 1) return TQ2_ERR_INVALID_ARG;
    if (kernel == TQ2_KERNEL_SKINNY && m > tq2::kSkinnyMaxM) return TQ2_ERR_INVALID_ARG;
    if (kernel == TQ2_KERNEL_SKINNY_MMA && !tq2::skinny_mma_fits(m, n, k)) return TQ2_ERR_INVALID_ARG;
    if (kernel < TQ2_KERNEL_GEMV || kernel > TQ2_KERNEL_SKINNY_MMA) return TQ2_ERR_INVALID_ARG;
    tq2::LaunchCtx ctx;
    st = prepare(stream, &ctx, {w_soa, x, residual, out});
    if (st != TQ2_OK) return st;
    switch (kernel) {
        case TQ2_KERNEL_GEMV: return finish(tq2::launch_gemv(w_soa, x, residual, out, n, k, ctx));
        case TQ2_KERNEL_SKINNY:
            return finish(tq2::launch_skinny(w_soa, x, residual, out, m, n, k, ctx));
        case TQ2_KERNEL_TC: {
            // x -> f16 tiles in a stream-ordered temporary, then the clustered
            // kernel.  A failed allocation is reported (TQ2_ERR_CUDA, the
            // CUDA error left for the caller), never replaced by another kernel.
            void *ws = nullptr;
            if (cudaMallocAsync(&ws, tq2::tc_ws_bytes(m, n, k), ctx.stream) != cudaSuccess)
                return TQ2_ERR_CUDA;
            const cudaError_t e = tq2::launch_tc_ws(w_soa, x, residual, out, m, n, k, ws, ctx);
            const cudaError_t f = cudaFreeAsync(ws, ctx.stream);
            return finish(e != cudaSuccess ? e : f);
        }
        case TQ2_KERNEL_TC_DIRECT:
            return finish(tq2::launch_tc(w_soa, x, residual, out, m, n, k, ctx));
        case TQ2_KERNEL_SKINNY_MMA:
            return finish(tq2::launch_skinny_mma(w_soa, x, residual, out, m, n, k, ctx));
        default: return finish(tq2::launch_f32ref(w_soa, x, residual, out, m, n, k, ctx));
    }
}

size_t tq2_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k) {
    bool noop = false;
    if (check_shape(m, n, k, &noop) != TQ2_OK || noop) return 0;
    if (tq2_select_kernel(m, n, k) != TQ2_KERNEL_TC) return 0;
    return tq2::tc_ws_bytes(m, n, k);
}

int tq2_gemm_ws(const void *w_soa, const float *x, const float *residual, float *out, int64_t m,
                int64_t n, int64_t k, void *workspace, size_t workspace_bytes, void *stream) {
    bool noop = false;
    int st = check_matmul(w_soa, x, residual, out, m, n, k, &noop);
    if (st != TQ2_OK || noop) return st;
    if (tq2_select_kernel(m, n, k) != TQ2_KERNEL_TC)
        return tq2_gemm_with(TQ2_KERNEL_AUTO, w_soa, x, residual, out, m, n, k, stream);
    const size_t need = tq2::tc_ws_bytes(m, n, k);
    if (!workspace || workspace_bytes < need) return TQ2_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 127u) != 0) return TQ2_ERR_MISALIGNED;
    const size_t wb = size_t(n) * size_t(k / tq2::kBlockW) * tq2::kBlockBytes;
    const size_t xb = size_t(m) * size_t(k) * 4, ob = size_t(m) * size_t(n) * 4;
    if (overlaps(workspace, need, x, xb) || overlaps(workspace, need, w_soa, wb) ||
        overlaps(workspace, need, out, ob) || (residual && overlaps(workspace, need, residual, ob)))
        return TQ2_ERR_INVALID_ARG;
    tq2::LaunchCtx ctx;
    st = prepare(stream, &ctx, {w_soa, x, residual, out, workspace});
    if (st != TQ2_OK) return st;
    return finish(tq2::launch_tc_ws(w_soa, x, residual, out, m, n, k, workspace, ctx));
}

int tq2_gemm_noalloc(const void *w_soa, const float *x, const float *residual, float *out,
                     int64_t m, int64_t n, int64_t k, void *stream) {
    bool noop = false;
    int st = check_matmul(w_soa, x, residual, out, m, n, k, &noop);
    if (st != TQ2_OK || noop) return st;
    if (tq2_select_kernel(m, n, k) != TQ2_KERNEL_TC)  // these kernels use no scratch
        return tq2_gemm_with(TQ2_KERNEL_AUTO, w_soa, x, residual, out, m, n, k, stream);
    // the one place that checks the shape against the fixed scratch; it comes
    // before the device is looked up (a host-only decision, like the other
    // argument checks)
    if (tq2::tc_ws_bytes(m, n, k) > tq2::kNoAllocScratchBytes) return TQ2_ERR_TOO_LARGE;
    tq2::LaunchCtx ctx;
    st = prepare(stream, &ctx, {w_soa, x, residual, out});
    if (st != TQ2_OK) return st;
    return finish(tq2::launch_tc_noalloc(w_soa, x, residual, out, m, n, k, ctx));
}

int tq2_gemm(const void *w_soa, const float *x, const float *residual, float *out, int64_t m,
             int64_t n, int64_t k, void *stream) {
    return tq2_gemm_with(TQ2_KERNEL_AUTO, w_soa, x, residual, out, m, n, k, stream);
}

static int gate_up_swiglu(const void *w_soa, const float *x, float *out, int64_t m, int64_t f,
                          int64_t k, void *stream, bool resident) {
    if (k <= 0 || k % tq2::kBlockW) return TQ2_ERR_BAD_K;
    if (f < 0 || f > (int64_t(1) << 39)) return TQ2_ERR_INVALID_ARG;
    bool noop = false;
    int st = check_shape(m, 2 * f, k, &noop);
    if (st != TQ2_OK || noop) return st;
    if (!w_soa || !x || !out) return TQ2_ERR_INVALID_ARG;
    if (!aligned16(w_soa) || !aligned16(x) || !aligned16(out)) return TQ2_ERR_MISALIGNED;
    const size_t wb = size_t(2 * f) * size_t(k / tq2::kBlockW) * tq2::kBlockBytes;
    const size_t xb = size_t(m) * size_t(k) * 4, ob = size_t(m) * size_t(f) * 4;
    if (overlaps(out, ob, x, xb) || overlaps(out, ob, w_soa, wb)) return TQ2_ERR_INVALID_ARG;
    tq2::LaunchCtx ctx;
    st = prepare(stream, &ctx, {w_soa, x, out});
    if (st != TQ2_OK) return st;
    cudaError_t e = cudaErrorNotSupported;
    if (m == 1) {
        e = tq2::launch_gemv_swiglu(w_soa, x, out, f, k, ctx, resident);
    } else if (f % 16 == 0) {
        void *ws = nullptr;
        if (cudaMallocAsync(&ws, tq2::tc_swiglu_ws_bytes(m, k), ctx.stream) != cudaSuccess) {
            (void)cudaGetLastError();
            return TQ2_ERR_CUDA;
        }
        e = tq2::launch_tc_swiglu(w_soa, x, out, m, f, k, ws, ctx);
        const cudaError_t fr = cudaFreeAsync(ws, ctx.stream);
        if (e == cudaSuccess) e = fr;
    }
    if (e != cudaErrorNotSupported) return finish(e);
    (void)cudaGetLastError();
    // Shapes outside the fused kernels: the plain product into a stream-ordered
    // temporary [m, 2f], then the element-wise activation.
    void *gu = nullptr;
    if (cudaMallocAsync(&gu, size_t(m) * size_t(2 * f) * 4, ctx.stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return TQ2_ERR_CUDA;
    }
    st = tq2_gemm_with(TQ2_KERNEL_AUTO, w_soa, x, nullptr, static_cast<float *>(gu), m, 2 * f, k, stream);
    if (st == TQ2_OK) st = finish(tq2::launch_swiglu_rows(static_cast<const float *>(gu), out, m, f, ctx));
    const cudaError_t fr = cudaFreeAsync(gu, ctx.stream);
    return st != TQ2_OK ? st : finish(fr);
}

int tq2_gate_up_swiglu(const void *w_soa, const float *x, float *out, int64_t m, int64_t f,
                       int64_t k, void *stream) {
    return gate_up_swiglu(w_soa, x, out, m, f, k, stream, false);
}

int tq2_gate_up_swiglu_resident(const void *w_soa, const float *x, float *out, int64_t m, int64_t f,
                                int64_t k, void *stream) {
    return gate_up_swiglu(w_soa, x, out, m, f, k, stream, true);
}

int tq2_act16_from_f32(const float *x, void *x16, int64_t m, int64_t k, void *stream) {
    if (k <= 0 || k % 16 || m < 0 || (m && k > (int64_t(1) << 40) / m)) return TQ2_ERR_INVALID_ARG;
    if (m == 0) return TQ2_OK;
    if (!x || !x16) return TQ2_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(x16)) return TQ2_ERR_MISALIGNED;
    if (overlaps(x, size_t(m) * size_t(k) * 4, x16, size_t(m) * size_t(k) * 2)) return TQ2_ERR_INVALID_ARG;
    tq2::LaunchCtx ctx;
    int st = prepare(stream, &ctx, {x, x16});
    if (st != TQ2_OK) return st;
    return finish(tq2::launch_act16_from_f32(x, static_cast<__half *>(x16), m, k, ctx));
}

int tq2_act16_to_f32(const void *x16, float *x, int64_t m, int64_t k, void *stream) {
    if (k <= 0 || k % 16 || m < 0 || (m && k > (int64_t(1) << 40) / m)) return TQ2_ERR_INVALID_ARG;
    if (m == 0) return TQ2_OK;
    if (!x || !x16) return TQ2_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(x16)) return TQ2_ERR_MISALIGNED;
    if (overlaps(x, size_t(m) * size_t(k) * 4, x16, size_t(m) * size_t(k) * 2)) return TQ2_ERR_INVALID_ARG;
    tq2::LaunchCtx ctx;
    int st = prepare(stream, &ctx, {x16, x});
    if (st != TQ2_OK) return st;
    return finish(tq2::launch_act16_to_f32(static_cast<const __half *>(x16), x, m, k, ctx));
}

int tq2_gemm_act16(const void *w_soa, const void *x16, const void *residual16, void *out16, int64_t m,
                   int64_t n, int64_t k, void *stream) {
    bool noop = false;
    int st = check_shape(m, n, k, &noop);
    if (st != TQ2_OK || noop) return st;
    if (n % 16) return TQ2_ERR_INVALID_ARG;
    if (!w_soa || !x16 || !out16) return TQ2_ERR_INVALID_ARG;
    if (!aligned16(w_soa) || !aligned16(x16) || !aligned16(out16) || (residual16 && !aligned16(residual16)))
        return TQ2_ERR_MISALIGNED;
    const size_t wb = size_t(n) * size_t(k / tq2::kBlockW) * tq2::kBlockBytes;
    const size_t xb = size_t(m) * size_t(k) * 2, ob = size_t(m) * size_t(n) * 2;
    if (overlaps(out16, ob, x16, xb) || overlaps(out16, ob, w_soa, wb)) return TQ2_ERR_INVALID_ARG;
    if (residual16 && residual16 != out16 && overlaps(out16, ob, residual16, ob)) return TQ2_ERR_INVALID_ARG;
    tq2::LaunchCtx ctx;
    st = prepare(stream, &ctx, {w_soa, x16, residual16, out16});
    if (st != TQ2_OK) return st;
    const size_t need = tq2::tc_act16_ws_bytes(m, n, k);
    void *ws = nullptr;
    if (need && cudaMallocAsync(&ws, need, ctx.stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return TQ2_ERR_CUDA;
    }
    cudaError_t e = tq2::launch_tc_act16(w_soa, static_cast<const __half *>(x16),
                                         static_cast<const __half *>(residual16), static_cast<__half *>(out16),
                                         m, n, k, ws, ctx);
    if (ws) {
        const cudaError_t f = cudaFreeAsync(ws, ctx.stream);
        if (e == cudaSuccess) e = f;
    }
    return finish(e);
}

int tq2_attention_f32(const float *q, const float *k, const float *v, float *out, int64_t heads,
                      int64_t seq, int64_t dim, void *stream) {
    if (heads < 0 || seq < 0 || dim < 8 || dim > 128 || dim % 8) return TQ2_ERR_INVALID_ARG;
    if (heads > 65535 || seq > (int64_t(1) << 24) || heads * ((seq + 127) / 128 * 128) > INT32_MAX)
        return TQ2_ERR_INVALID_ARG;
    if (heads == 0 || seq == 0) return TQ2_OK;
    if (!q || !k || !v || !out) return TQ2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return TQ2_ERR_MISALIGNED;
    const size_t nb = size_t(heads) * size_t(seq) * size_t(dim) * 4;
    if (overlaps(out, nb, q, nb) || overlaps(out, nb, k, nb) || overlaps(out, nb, v, nb))
        return TQ2_ERR_INVALID_ARG;
    tq2::LaunchCtx ctx;
    int st = prepare(stream, &ctx, {q, k, v, out});
    if (st != TQ2_OK) return st;
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, tq2::attention_ws_bytes(heads, seq, dim), ctx.stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return TQ2_ERR_CUDA;
    }
    cudaError_t e = tq2::launch_attention(q, k, v, out, heads, seq, dim, ws, ctx);
    const cudaError_t f = cudaFreeAsync(ws, ctx.stream);
    return finish(e != cudaSuccess ? e : f);
}

int tq2_gemv(const void *w_soa, const float *x, const float *residual, float *out, int64_t n,
             int64_t k, void *stream) {
    return tq2_gemm_with(TQ2_KERNEL_GEMV, w_soa, x, residual, out, 1, n, k, stream);
}

int tq2_gemv_resident(const void *w_soa, const float *x, const float *residual, float *out,
                      int64_t n, int64_t k, void *stream) {
    bool noop = false;
    int st = check_matmul(w_soa, x, residual, out, 1, n, k, &noop);
    if (st != TQ2_OK || noop) return st;
    tq2::LaunchCtx ctx;
    st = prepare(stream, &ctx, {w_soa, x, residual, out});
    if (st != TQ2_OK) return st;
    return finish(tq2::launch_gemv(w_soa, x, residual, out, n, k, ctx, true));
}

int tq2_gemm_f32ref(const void *w_soa, const float *x, const float *residual, float *out,
                    int64_t m, int64_t n, int64_t k, void *stream) {
    return tq2_gemm_with(TQ2_KERNEL_F32REF, w_soa, x, residual, out, m, n, k, stream);
}

}  // extern "C"
