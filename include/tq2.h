/*
 * tq2.h -- C ABI of the GB300 (sm_103a) TQ2_0_g128 ternary matmul library.
 *
 * Operation ("oxibonsai-image 0.2.2 src/gpu.rs", module doc "Correctness
 * contract", and the doc of `ternary_matmul_gpu`):
 *
 *     out[m, n] = sum_k input[m, k] * dequant(W)[n, k]   (+ residual[m, n])
 *
 * with row-major f32 input[M, K], out-major weight blocks [N, K/128] and
 * row-major f32 out[M, N], written in full.  K must be a positive multiple of
 * 128 (the page rejects `k % 128 != 0`).
 *
 * Weight block ("BlockTQ2_0_g128", same page, doc of `blocks_as_bytes` and
 * test `block_is_thirty_four_bytes`): 34 bytes, no padding, little endian:
 *
 *     struct { uint8_t qs[32]; uint16_t d; }   // d: IEEE binary16 scale
 *
 * Code convention of this library (the pages do not print it): weight j
 * (0..127) of a block has the 2-bit code c = (qs[j/4] >> 2*(j%4)) & 3, and
 * its value is (c - 1) * d, i.e. c in {0,1,2} -> {-1, 0, +1} * d.  Code 3 is
 * never produced by an encoder; every entry point decodes it arithmetically
 * as c - 1 = +2.
 *
 * Device weight layout (SoA; the "SoA weight buffer" that the TQ2 kernels
 * read, named on the "oxibonsai-kernels 0.1.5
 * src/gpu_backend/metal_graph/pipelines.rs" page; the layout itself is this
 * library's definition).  For B = N*(K/128) blocks in row-major (n, b) order:
 *
 *     bytes [0, 32*B)          qs plane: block (n,b)'s qs[32] at (n*(K/128)+b)*32
 *     bytes [32*B, 34*B)       d plane : block (n,b)'s d (2 bytes) at 32*B + (n*(K/128)+b)*2
 *
 * The total size equals the AoS size, tq2_soa_bytes(n, k) = N*(K/128)*34.
 *
 * Conventions shared by every entry point below:
 *  - Pointers are DEVICE pointers of the current device, owned by the caller.
 *    Before any launch every operand is checked (cudaPointerGetAttributes):
 *    memory that is not device memory of the current device (pageable or
 *    pinned host memory, managed memory, another GPU's memory reached through
 *    a peer or imported mapping) gives TQ2_ERR_INVALID_ARG.  Every call runs
 *    on one GPU.
 *  - Memory: the library keeps no cache of weights (the pages' pointer-keyed
 *    upload cache is the caller's job here) and frees only what it took.  The
 *    entry points whose doc has a "Memory:" paragraph take a temporary from
 *    the device's default stream-ordered pool (cudaMallocAsync, released by
 *    cudaFreeAsync on the same stream; both are legal inside stream capture)
 *    and return TQ2_ERR_CUDA if it cannot be had; all others allocate nothing
 *    (tq2_gemm_ws and tq2_gemm_noalloc are the allocation-free forms of the
 *    tensor-core path).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *    is asynchronous on it and never synchronises the host.
 *  - Errors are returned as a tq2_status; nothing aborts and there is no CPU
 *    fallback.  Argument errors are detected on the host before any launch.
 *    TQ2_ERR_CUDA means a launch or runtime error (the CUDA error is left for
 *    the caller to inspect with cudaGetLastError/cudaPeekAtLastError).
 *  - m == 0 or n == 0 is a successful no-op (nothing is launched, nothing is
 *    read).  m, n must be >= 0; k must be a positive multiple of 128.
 *  - Alignment: w_soa, x, residual and out must be 16-byte aligned (128-bit
 *    loads and stores).  w_aos needs no alignment.
 *  - Aliasing: `residual` may equal `out` exactly (in-place out += x.W^T);
 *    otherwise no output may overlap an input.
 *  - Device: compute capability 10.3 (sm_103a) only; any other device gives
 *    TQ2_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef TQ2_H_
#define TQ2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TQ2_OK = 0,
    TQ2_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad aliasing, size overflow */
    TQ2_ERR_BAD_K = 2,              /* k <= 0 or k % 128 != 0 */
    TQ2_ERR_MISALIGNED = 3,         /* a pointer that must be 16-byte aligned is not */
    TQ2_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not sm_103 */
    TQ2_ERR_CUDA = 5,               /* launch or runtime error */
    TQ2_ERR_TIMEOUT = 6,            /* a bounded device-side wait expired (see tq2_device_status) */
    TQ2_ERR_TOO_LARGE = 7           /* tq2_gemm_noalloc: the shape needs more than its fixed scratch */
} tq2_status;

/* Size of the fixed device scratch behind tq2_gemm_noalloc (32 MiB). */
#define TQ2_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* Kernel choice for tq2_gemm_with().  TQ2_KERNEL_AUTO is what tq2_gemm uses. */
typedef enum {
    TQ2_KERNEL_AUTO = 0,
    TQ2_KERNEL_GEMV = 1,   /* M == 1 only: f32 CUDA-core decode GEMV */
    TQ2_KERNEL_SKINNY = 2, /* small M: f32 CUDA-core kernel, weights decoded once per M rows */
    TQ2_KERNEL_TC = 3,     /* tcgen05 tensor-core path: x converted once to f16 tiles in a
                              stream-ordered temporary, then the clustered kernel; f16
                              operands, f32 accumulation in TMEM */
    TQ2_KERNEL_F32REF = 4, /* exact-f32 CUDA-core tiled kernel */
    TQ2_KERNEL_TC_DIRECT = 5, /* tcgen05 kernel that converts x itself (no temporary memory);
                                 same arithmetic as TQ2_KERNEL_TC */
    TQ2_KERNEL_SKINNY_MMA = 6 /* 2 <= M <= 32: one-launch tensor-core kernel for few rows (x
                                 rounded to binary16, f32 accumulation; no temporary memory) */
} tq2_kernel;

/* Bytes of a weight of n rows and k columns in either layout: n*(k/128)*34.
 * Returns 0 for n < 0 or a k that is not a positive multiple of 128. */
size_t tq2_soa_bytes(int64_t n, int64_t k);

/* Human-readable name of a tq2_status value (static string, never NULL). */
const char *tq2_status_string(int status);

/* Relayout AoS weight blocks into the SoA layout above, bit-exactly.
 * The pages convert the uploaded AoS bytes with a `reformat_tq2_aos_to_soa`
 * kernel ("oxibonsai-image 0.2.2 src/gpu.rs", doc of `blocks_as_bytes`).
 *   w_aos : device, n*(k/128)*34 bytes, AoS [N][K/128] blocks, any alignment
 *   w_soa : device, same size, 16-byte aligned, must not overlap w_aos
 */
int tq2_reformat_aos_to_soa(const void *w_aos, void *w_soa, int64_t n, int64_t k, void *stream);

/* Encoder: f32 weights -> TQ2_0_g128 blocks.  (No counterpart on the pages:
 * their blocks come ready-made from a GGUF file, and they never show how
 * blocks are produced.  This library reads it as the absmean rule of ternary
 * weights, with every step that decides a code fixed, so that the bytes are
 * reproducible exactly.)  For each block of 128 weights of a row:
 *   gamma = (sum_j |w_j|) / 128, summed in double in index order;
 *   d     = binary16(gamma), round to nearest even (Inf above 65504);
 *   code  = clamp(rint(w_j / d), -1, 1) + 1, the quotient in binary32 (IEEE
 *           division, ties to even); a zero or non-finite d gives code 1.
 *   w     : device f32 [n, k] row-major, 16-byte aligned, finite
 *   w_aos : device, n*(k/128)*34 bytes, AoS [N][K/128] blocks, 16-byte
 *           aligned, must not overlap w (relayout with
 *           tq2_reformat_aos_to_soa for the matmul entry points)
 * Errors: TQ2_ERR_BAD_K, TQ2_ERR_INVALID_ARG, TQ2_ERR_MISALIGNED. */
int tq2_quantize_f32(const float *w, void *w_aos, int64_t n, int64_t k, void *stream);

/* M = 1 decode GEMV: out[n] = sum_k x[k] * dequant(W)[n,k] (+ residual[n]).
 * The decode-path GEMV `gemv_tq2_g128_v1` of the "oxibonsai-kernels 0.1.5 ...
 * pipelines.rs" page; the operation is the contract above with M = 1.
 *   w_soa    : device SoA weight (tq2_soa_bytes(n,k) bytes)
 *   x        : device f32 [k], finite
 *   residual : device f32 [n], or NULL
 *   out      : device f32 [n]
 * Arithmetic (k <= 12288): x is quantised per 128-weight block to a signed
 * fixed-point integer relative to the block's largest |x| (23 bits:
 * |x - xq| <= 2^-22 * max|x_block|); the ternary dot products are then exact
 * integer sums per block, scaled by max|x_block| * 2^-22 * d and summed in f32.
 * Per element: |error| <= sum over blocks of 2^-22 * max|x_block| * sum_block |w|
 * plus f32 rounding of the block sums and of the final sum.  For k > 12288:
 * exact f32 products and f32 accumulation. */
int tq2_gemv(const void *w_soa, const float *x, const float *residual, float *out,
             int64_t n, int64_t k, void *stream);

/* tq2_gemv for weights that stay resident across calls (decoding with a
 * weight set uploaded once): the same arguments, arithmetic and result, bit
 * for bit.  Contract: no work that is still unfinished when this call is
 * enqueued writes w_soa (write the weights, then synchronise the stream or the
 * device before the decode loop).  Under it the call copies its weight rows
 * into shared memory before it waits for the preceding kernel of the stream,
 * i.e. while that kernel runs; x, residual and out are still read and written
 * only after that kernel has finished.  Breaking the contract gives results
 * from stale weights (no fault).  Errors as tq2_gemv. */
int tq2_gemv_resident(const void *w_soa, const float *x, const float *residual, float *out,
                      int64_t n, int64_t k, void *stream);

/* Any-M matmul with optional residual epilogue, dispatching on M (and N, K)
 * between the GEMV (m = 1), the one-launch skinny tensor-core kernel
 * (2 <= m <= 32, TQ2_KERNEL_SKINNY_MMA below) and the tcgen05 tensor-core
 * kernel ("oxibonsai-image 0.2.2 src/gpu.rs", `ternary_matmul_gpu`;
 * the batched TQ2 GEMMs of the "oxibonsai-kernels 0.1.5 ... pipelines.rs"
 * page).
 *   w_soa    : device SoA weight
 *   x        : device f32 [m, k] row-major
 *   residual : device f32 [m, n] row-major, or NULL
 *   out      : device f32 [m, n] row-major
 * Arithmetic: the tensor-core kernel rounds x to binary16 (round to nearest
 * even; |x| must stay below 65504) and multiplies by the exactly representable
 * binary16 weights (c-1)*d with f32 accumulation; the CUDA-core kernels use
 * exact f32 products and f32 accumulation.
 * Memory: on the tensor-core path the call takes a temporary of
 * tq2_gemm_workspace_bytes(m,n,k) bytes from the device's default memory pool,
 * ordered on `stream`; if it cannot be had the call returns TQ2_ERR_CUDA
 * without launching anything (no silent change of kernel).  Callers that
 * manage memory themselves use tq2_gemm_ws or tq2_gemm_noalloc, or
 * tq2_gemm_with(TQ2_KERNEL_TC_DIRECT), which converts x inside the kernel and
 * needs no temporary (about half the speed). */
int tq2_gemm(const void *w_soa, const float *x, const float *residual, float *out,
             int64_t m, int64_t n, int64_t k, void *stream);

/* Fused gate/up projection with the SwiGLU activation: the TQ2 analogue of
 * the pages' `fused_gate_up_swiglu_q1` (decode) and
 * `fused_gate_up_swiglu_gemm_q1` (prefill) pipelines ("oxibonsai-kernels
 * 0.1.5 src/gpu_backend/metal_graph/pipelines.rs", fused-kernel fields), which
 * the pages name without a listing.  The weight holds 2f rows: the gate
 * projection in rows [0, f), the up projection in rows [f, 2f).  For each
 * input row i and feature j:
 *   g = sum_k x[i,k] W[j,k],  u = sum_k x[i,k] W[f+j,k],
 *   out[i,j] = silu(g) * u,  silu(z) = z / (1 + exp(-z)).
 *   w_soa : device SoA weight of n = 2f rows (from tq2_reformat_aos_to_soa)
 *   x     : device f32 [m, k] row-major
 *   out   : device f32 [m, f] row-major (may not overlap x or w_soa)
 * Arithmetic: m = 1 runs the GEMV (x quantised per 128-weight block, exact
 * integer dot products; see tq2_gemv) for k <= 12288; m >= 2 runs the
 * tensor-core kernel (x rounded to binary16; see tq2_gemm) with the activation
 * in its epilogue when f % 16 == 0.  Other shapes compute the plain product
 * into a temporary [m, 2f] and apply the activation in a second kernel.  g and
 * u are never written to memory on the fused paths.  The activation is
 * evaluated in f32: with expf and IEEE division on the GEMV and unfused paths,
 * with the fast exp2-based exponential and division (relative error about
 * 1e-6) in the tensor-core epilogue.
 * Memory: m >= 2 (and the unfused shapes) take a temporary from the device's
 * default memory pool, ordered on `stream` (as tq2_gemm).
 * Errors: TQ2_ERR_BAD_K, TQ2_ERR_INVALID_ARG (negative m or f, NULL pointers,
 * out overlapping x or w_soa), TQ2_ERR_MISALIGNED (pointers not 16-byte
 * aligned), TQ2_ERR_CUDA (launch or temporary allocation failure).  m = 0 or
 * f = 0 is a no-op. */
int tq2_gate_up_swiglu(const void *w_soa, const float *x, float *out, int64_t m, int64_t f,
                       int64_t k, void *stream);

/* tq2_gate_up_swiglu for weights that stay resident across calls: the same
 * arguments, arithmetic and result, bit for bit.  Contract (as
 * tq2_gemv_resident): no work that is still unfinished when this call is
 * enqueued writes w_soa.  At m = 1 the call may then copy its weight rows into
 * shared memory before it waits for the preceding kernel of the stream;
 * other m are computed exactly as tq2_gate_up_swiglu.  Errors as
 * tq2_gate_up_swiglu. */
int tq2_gate_up_swiglu_resident(const void *w_soa, const float *x, float *out, int64_t m, int64_t f,
                                int64_t k, void *stream);

/* Binary16 activation layout (activation-resident chaining of layers): a
 * row-major [m][k] array of binary16 in which element i (0..15) of every
 * 16-element group of a row is stored at position 2i for i < 8 and 2(i-8)+1
 * for i >= 8 (the k order in which the tensor-core kernel decodes weights).
 * tq2_gemm_act16 reads x and writes out in this layout, so the output of one
 * layer is the next layer's input with no f32 round trip and no conversion
 * pass.  Converters (k % 16 == 0; pointers 16-byte aligned, not overlapping):
 * from f32 rounds to nearest even (|x| >= 65520 becomes Inf), to f32 is exact.
 * Errors: TQ2_ERR_INVALID_ARG (k not a positive multiple of 16, m < 0, NULL,
 * overlap), TQ2_ERR_MISALIGNED, TQ2_ERR_CUDA. */
int tq2_act16_from_f32(const float *x, void *x16, int64_t m, int64_t k, void *stream);
int tq2_act16_to_f32(const void *x16, float *x, int64_t m, int64_t k, void *stream);

/* out16[m, n] = x16[m, k] . dequant(W)^T (+ residual16), binary16 activations
 * in the layout above (the pages' DiT linears, "oxibonsai-image 0.2.2
 * src/gpu.rs" contract, with the activations kept in binary16 between layers:
 * only activations cross between kernels).  The tensor-core kernel multiplies
 * the exactly representable binary16 weights with x16 (no rounding of x),
 * accumulates in f32, adds the residual in f32 and rounds the result once to
 * binary16 (nearest even).  x tiles arrive by tensor copy: no pre-pass.
 *   n must be a multiple of 16 (the output layout's groups); residual16 may be
 *   NULL or equal to out16 (in place).
 * Memory: shapes with too few output tiles for the GPU split K and take a
 * temporary of S*m*n f32 from the device's default memory pool on `stream`.
 * Errors: TQ2_ERR_BAD_K, TQ2_ERR_INVALID_ARG (n % 16 != 0, negative sizes,
 * NULL, overlaps), TQ2_ERR_MISALIGNED, TQ2_ERR_CUDA.  m = 0 or n = 0: no-op. */
int tq2_gemm_act16(const void *w_soa, const void *x16, const void *residual16, void *out16,
                   int64_t m, int64_t n, int64_t k, void *stream);

/* DiT joint multi-head attention (the pages' `joint_attention_gpu`,
 * "oxibonsai-image 0.2.2 src/gpu.rs", and its kernel
 * `joint_attention_flash_f32`, "oxibonsai-kernels 0.1.5
 * src/gpu_backend/metal_graph/pipelines.rs"):
 *   out[t, h*dim + d] = sum_j softmax_j(q[h,t] . k[h,j] / sqrt(dim)) v[h,j,d]
 * over all seq keys (non-causal).
 *   q, k, v : device f32 [heads, seq, dim], head-major (RoPE already applied)
 *   out     : device f32 [seq, heads*dim], token-major (may not overlap q, k, v)
 *   dim     : head dimension, a multiple of 8 from 8 to 128 (the page's
 *             range); the kernel runs 64 (dim <= 64) or 128 features wide
 *             with the extra features zero in its staged copies, which
 *             changes no result
 * Arithmetic: q (times log2(e)/sqrt(dim)), k and v are rounded to binary16
 * (nearest even; their magnitudes must stay below 65504) and multiplied on the
 * tensor cores with f32 accumulation; the softmax runs in f32 with the
 * hardware 2^x, its weights rounded to binary16 for the second product; the
 * normalisation by the weight sum is the last step (flash attention: one pass
 * over the keys, no [seq, seq] matrix in memory).
 * Memory: a temporary of 3*heads*ceil(seq/128)*128*w*2 bytes (w = 64 for
 * dim <= 64, else 128) from the device's default memory pool, ordered on
 * `stream`.
 * Errors: TQ2_ERR_INVALID_ARG (dim not a multiple of 8 in [8, 128], negative or too large sizes
 * (heads <= 65535, seq <= 2^24), NULL, overlap), TQ2_ERR_MISALIGNED (pointers
 * not 16-byte aligned), TQ2_ERR_TIMEOUT via tq2_device_status, TQ2_ERR_CUDA.
 * heads = 0 or seq = 0: no-op. */
int tq2_attention_f32(const float *q, const float *k, const float *v, float *out, int64_t heads,
                      int64_t seq, int64_t dim, void *stream);

/* Same operation as tq2_gemm, computed by the exact-f32 CUDA-core tiled
 * kernel (the role of the pages' non-matrix-unit `gemm_tq2_g128_v8_tiled`,
 * kept for tolerance checks). */
int tq2_gemm_f32ref(const void *w_soa, const float *x, const float *residual, float *out,
                    int64_t m, int64_t n, int64_t k, void *stream);

/* Workspace bytes that tq2_gemm_ws needs for this shape when it selects the
 * tensor-core kernel, else 0: the binary16 copy of x, padded to a multiple of
 * 128 rows (ceil(m/128)*128*k*2 bytes), plus, for shapes with too few output
 * tiles to occupy the GPU, S f32 partial results of m*n elements (S K slices,
 * a function of the shape only, summed afterwards in slice order).  Host only.
 * Returns 0 for invalid shapes. */
size_t tq2_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k);

/* tq2_gemm with a caller-owned device workspace (the library still
 * allocates nothing).  When the shape selects the tensor-core kernel, x is
 * first converted to binary16 MMA tiles in the workspace by a pre-pass and the
 * tensor-core kernel streams those tiles with bulk copies instead of
 * converting x itself; results are those of the tensor-core kernel.  Other
 * shapes ignore the workspace and behave exactly like tq2_gemm.
 *   workspace       : device, >= tq2_gemm_workspace_bytes(m,n,k) bytes,
 *                     128-byte aligned, overlapping no other argument; may be
 *                     NULL when that size is 0.  Its contents on return are
 *                     unspecified; the call only reads what it wrote.
 *   workspace_bytes : its size; a smaller size gives TQ2_ERR_INVALID_ARG.
 * Two calls that share a workspace must be ordered (same stream). */
int tq2_gemm_ws(const void *w_soa, const float *x, const float *residual, float *out, int64_t m,
                int64_t n, int64_t k, void *workspace, size_t workspace_bytes, void *stream);

/* tq2_gemm for callers that cannot allocate device memory.  (No counterpart
 * on the pages; this is an addition of this library.)
 *
 * Some callers may not call cudaMalloc or any allocating routine at all: a
 * host application that owns every byte of device memory and gives its
 * plugins no allocator, a real-time loop that must never allocate after
 * start-up, or code that runs where an allocation could fail or block.
 * tq2_gemm_ws needs such a caller to provide a workspace; this entry point
 * needs none.  For shapes that select the tensor-core kernel it converts x
 * into a fixed scratch array that is part of the library's device image
 * (TQ2_NOALLOC_SCRATCH_BYTES, reserved on every device that loads the library
 * until the process exits) and then runs the same kernel as tq2_gemm_ws, with
 * the same results.  Other shapes use no scratch and behave like tq2_gemm.
 *   - Limit: shapes with tq2_gemm_workspace_bytes(m,n,k) >
 *     TQ2_NOALLOC_SCRATCH_BYTES return TQ2_ERR_TOO_LARGE before any work
 *     (e.g. m = 4096 with k up to 4096 fits; k = 12288 does not).  Like the
 *     other argument checks this is decided on the host before the device is
 *     looked up, so it precedes TQ2_ERR_UNSUPPORTED_DEVICE.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - The first call on a device looks up the scratch array's device address
 *     (one-time set-up, with that device current); make that first call before
 *     any stream capture.
 *   - Every call shares the one scratch array, which keeps the last call's
 *     contents (each call writes all of the scratch it reads, so nothing needs
 *     clearing).  Calls whose GPU work overlaps in time race on it: issue them
 *     on one stream or otherwise order them.
 * Arguments, layouts and other errors as tq2_gemm. */
int tq2_gemm_noalloc(const void *w_soa, const float *x, const float *residual, float *out,
                     int64_t m, int64_t n, int64_t k, void *stream);

/* tq2_gemm with an explicit kernel choice (a tq2_kernel value), for
 * benchmarks and tests.  TQ2_KERNEL_GEMV requires m == 1, TQ2_KERNEL_SKINNY
 * m <= 16 and TQ2_KERNEL_SKINNY_MMA 2 <= m <= 32 with k small enough for its
 * K slices' shared memory (k <= 12288 at m = 32) (else TQ2_ERR_INVALID_ARG).
 * TQ2_KERNEL_TC allocates as tq2_gemm does.
 *
 * TQ2_KERNEL_SKINNY_MMA ("the few-row batches" of the pages' TQ2 GEMMs, any
 * batch size): one launch.  CTAs of 128 weight rows each take a K slice; the
 * CTAs of one row tile form a thread-block cluster and sum their partial
 * results through distributed shared memory in a fixed order (results are
 * the same bits on every call).  Warp-level tensor-core MMAs take the weight
 * codes decoded in registers as the A operand and x rounded to binary16
 * (nearest even; |x| < 65504) as the B operand, with f32 accumulation per
 * 128-weight block, then the block's d applied in f32: the tensor-core
 * path's arithmetic. */
int tq2_gemm_with(int kernel, const void *w_soa, const float *x, const float *residual,
                  float *out, int64_t m, int64_t n, int64_t k, void *stream);

/* The kernel that tq2_gemm picks for this shape (a tq2_kernel value).  Host
 * only; needs no device. */
int tq2_select_kernel(int64_t m, int64_t n, int64_t k);

/* Bounded device-side waits.  Every spin-wait inside a kernel (on an mbarrier)
 * gives up after `ns` nanoseconds of %globaltimer time, records
 * TQ2_ERR_TIMEOUT in a device status word and lets the kernel exit cleanly
 * (draining its own in-flight work first).  Default 2e9 (2 s).  Applies to
 * launches issued after the call.  Returns the previous value. */
uint64_t tq2_set_wait_timeout_ns(uint64_t ns);

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device: TQ2_OK, or TQ2_ERR_TIMEOUT if any kernel since the last
 * check gave up on a wait; TQ2_ERR_CUDA if the synchronisation itself failed. */
int tq2_device_status(void *stream);

/* Library version, e.g. 0x000100 for 0.1.0. */
int tq2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TQ2_H_ */
