// Encoder: f32 weights [n][k] -> TQ2_0_g128 AoS blocks [n][k/128] (34 bytes).
//
// The pages never show how the blocks are produced (they are read from a GGUF
// file); this library's reading is the absmean rule of ternary weights, with
// every floating-point step that decides a code fixed so that the result is
// reproducible bit for bit:
//   gamma = (sum_{j=0..127} |w_j|) / 128, the sum in double in index order;
//   d     = binary16(gamma), round to nearest even;
//   q_j   = rint(w_j / (float)d) in binary32 (IEEE division, ties to even),
//           clamped to [-1, 1]; code c_j = q_j + 1 at bits 2*(j%4) of qs[j/4].
// A zero or non-finite d gives code 1 (weight 0) everywhere.
//
// One warp per 128-weight block: lane l loads weights 4l .. 4l+3 with one
// coalesced 16-byte load, decides the codes of exactly those four weights and
// so produces qs[l].  The block's double sum in index order is exact whenever
// every partial sum fits a double's 53-bit significand: with the nonzero
// magnitudes m_j * 2^(e_j - 150) (24-bit m_j) and e_max - e_min <= 22 the total
// is below 2^53 units of 2^(e_min - 150), so the sequential sum equals the exact
// one, which the warp forms in any order as an integer of aligned significands
// (FP32 and integer instructions only), and d is that integer times
// 2^(e_min - 157) rounded to binary16.  Blocks with a wider exponent span,
// magnitudes below 2^-104, or an Inf or NaN take the literal route: lane 0
// adds the 128 magnitudes in double in index order.  Both give the same bytes;
// the FP64 pipe, a small fraction of the FP32 one on this part, is used only
// for those blocks.  The codes need no division (see the code step below).
#include <algorithm>

#include <cuda_fp16.h>

#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int kQThreads = 256;

// double -> binary16 bits, round to nearest even: |v| >= 65520 -> Inf (halfway
// past the largest finite 65504), subnormals on the 2^-24 grid.
__device__ __forceinline__ uint16_t to_half_rne(double v) {
    const uint16_t sign = signbit(v) ? 0x8000 : 0;
    const double a = fabs(v);
    if (isnan(v)) return 0x7e00;
    if (a >= 65520.0) return uint16_t(sign | 0x7c00);
    if (a < 6.103515625e-05) {  // 2^-14: subnormal grid of 2^-24 (1024 carries into the exponent)
        return uint16_t(sign | uint16_t(rint(a * 16777216.0)));
    }
    int ex;
    frexp(a, &ex);  // a = m * 2^ex, m in [0.5, 1)
    int e = ex - 1;
    double r = rint(ldexp(a, 10 - e));  // in [1024, 2048]
    if (r >= 2048.0) {
        r = 1024.0;
        e += 1;
    }
    if (e > 15) return uint16_t(sign | 0x7c00);
    return uint16_t(sign | uint16_t((e + 15) << 10) | uint16_t(r - 1024.0));
}

// binary16 bits of S * 2^E, round to nearest even (S < 2^53): S is first
// rounded to 24 bits with round-to-odd (the truncation's lost bits folded into
// the last bit), which the binary16 conversion's round-to-nearest then rounds
// exactly as it would round S itself (the intermediate keeps at least two more
// bits than binary16 has, also on the subnormal grid); the power-of-two scale
// is exact wherever the result can be nonzero.
__device__ __forceinline__ uint16_t half_of_scaled(uint64_t S, int E) {
    if (S == 0 || E < -126) return 0;  // S * 2^E < 2^-73: rounds to zero
    const int p = 63 - __clzll(static_cast<long long>(S));
    uint32_t m;
    int k = E;
    if (p > 23) {
        const int sh = p - 23;
        m = uint32_t(S >> sh) | uint32_t((S & ((uint64_t(1) << sh) - 1)) != 0);
        k += sh;  // <= 97 + 29: a finite power of two
    } else {
        m = uint32_t(S);
    }
    const float y = float(m) * __int_as_float((k + 127) << 23);  // m < 2^24: exact conversion
    return __half_as_ushort(__float2half_rn(y));
}

constexpr int kQWarps = kQThreads / 32;

__global__ void __launch_bounds__(kQThreads, 5)
quantize_kernel(const float *__restrict__ w, uint8_t *__restrict__ aos, int64_t nblk) {
    __shared__ float fb[kQWarps][kBlockW];  // the literal route's staging, per warp
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    const int64_t nw = int64_t(gridDim.x) * kQWarps;
    auto one = [&](int64_t b, const float4 v) {
        const float x[4] = {v.x, v.y, v.z, v.w};
        uint32_t a[4];
#pragma unroll
        for (int f = 0; f < 4; ++f) a[f] = __float_as_uint(x[f]) & 0x7fffffffu;
        // largest magnitude, and smallest nonzero one (a - 1 wraps zero to the top)
        const uint32_t amax = __reduce_max_sync(0xffffffffu, max(max(a[0], a[1]), max(a[2], a[3])));
        const uint32_t amin1 =
            __reduce_min_sync(0xffffffffu, min(min(a[0] - 1u, a[1] - 1u), min(a[2] - 1u, a[3] - 1u)));
        const int emax = int(amax >> 23), emin = int((amin1 + 1u) >> 23);
        // integer route: finite, every nonzero magnitude at least 2^-104 and
        // within 22 binades of the largest (or all zero)
        const bool fast = amax < 0x7f800000u && (amax == 0 || (emin >= 23 && emax - emin <= 22));
        uint16_t dh;
        if (fast) {
            // v = |w| * 2^(150 - emin): an integer below 2^46, exact in binary32,
            // split as vh * 2^23 + vl with both parts below 2^23, each read off
            // the bits of a sum onto 2^23 (vh by a round-down add): FP32 and
            // integer pipes only.  Per lane the biased bits add without overflow.
            const float scale = __int_as_float((150 - emin + 127) << 23);
            uint32_t hs = 0, ls = 0;
#pragma unroll
            for (int f = 0; f < 4; ++f) {
                const float v = __uint_as_float(a[f]) * scale;
                const float rh = __fadd_rd(v * 1.1920928955078125e-7f, 8388608.0f);  // 2^23 + floor(v / 2^23)
                const float vl = __fmaf_rn(rh - 8388608.0f, -8388608.0f, v);         // v mod 2^23, exact
                hs += __float_as_uint(rh);
                ls += __float_as_uint(vl + 8388608.0f);
            }
            const uint32_t hi = __reduce_add_sync(0xffffffffu, hs - 4u * 0x4B000000u);  // < 2^30
            const uint32_t lo = __reduce_add_sync(0xffffffffu, ls - 4u * 0x4B000000u);
            const uint64_t S = (uint64_t(hi) << 23) + uint64_t(lo);
            dh = half_of_scaled(S, emin - 157);  // (sum / 128) = S * 2^(emin - 150 - 7)
        } else {
#pragma unroll
            for (int f = 0; f < 4; ++f) fb[wi][4 * lane + f] = x[f];
            __syncwarp();
            uint32_t d32 = 0;
            if (lane == 0) {
                double s = 0.0;
                for (int j = 0; j < kBlockW; ++j) s += fabs(double(fb[wi][j]));
                d32 = to_half_rne(s * 0.0078125);  // / 128, exact
            }
            dh = uint16_t(__shfl_sync(0xffffffffu, d32, 0));
            __syncwarp();
        }
        // code: rint(w / d) in binary32 is >= 1 in magnitude exactly when the
        // rounded quotient exceeds 1/2, i.e. when |w| / d > 1/2 + 2^-25 (a tie
        // goes to the even 1/2), i.e. when |w| exceeds T, the largest binary32 not
        // above d/2 + d * 2^-25: one round-toward-zero FMA per block (T = +Inf
        // when d is zero or not finite: every code 1).  Per weight, on the FP32
        // pipe: g = saturate((|w| - T) * 2^127) is exactly 1 when |w| > T (the
        // smallest positive difference, 2^-48 or more, times 2^127 exceeds 1) and
        // 0 otherwise (NaN saturates to 0), the code is g * sign(w) + 1, and its
        // bits are read off a sum onto 2^23.  No division.
        const float df = __half2float(__ushort_as_half(dh));
        const bool live = df > 0.f && isfinite(df);
        const float tf = live ? __fmaf_rz(df, 2.98023223876953125e-8f, 0.5f * df) : __int_as_float(0x7f800000);
        uint32_t cb[4];
#pragma unroll
        for (int f = 0; f < 4; ++f) {
            const float g = __saturatef((__uint_as_float(a[f]) - tf) * 1.7014118346046923e38f);  // 2^127
            const float sgn = __uint_as_float((__float_as_uint(x[f]) & 0x80000000u) | 0x3f800000u);  // +-1
            cb[f] = __float_as_uint(__fmaf_rn(g, sgn, 1.0f) + 8388608.0f);  // 0x4B000000 + code
        }
        // the offsets of the four sums vanish from the low byte after the shifts
        const uint32_t byte = (cb[0] + (cb[1] << 2) + (cb[2] << 4) + (cb[3] << 6)) & 0xffu;
        // qs[l] is this lane's byte: lanes 2i and 2i+1 store one 16-bit word
        // (a block starts on an even byte); lane 0 also stores d
        const uint32_t hi8 = __shfl_down_sync(0xffffffffu, byte, 1);
        uint8_t *ob = aos + b * kBlockBytes;
        if ((lane & 1) == 0) *reinterpret_cast<uint16_t *>(ob + lane) = uint16_t(byte | (hi8 << 8));
        if (lane == 0) *reinterpret_cast<uint16_t *>(ob + 32) = dh;
    };
    // grid-stride over blocks, two at a time; the next two blocks' loads are
    // issued before the current two are encoded (four per warp in flight)
    auto load = [&](int64_t blk) {
        return blk < nblk ? __ldcs(reinterpret_cast<const float4 *>(w + blk * kBlockW) + lane)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    int64_t b = int64_t(blockIdx.x) * kQWarps + wi;
    float4 n0 = load(b), n1 = load(b + nw);
    for (; b < nblk; b += 2 * nw) {
        const float4 v0 = n0, v1 = n1;
        n0 = load(b + 2 * nw);
        n1 = load(b + 3 * nw);
        one(b, v0);
        if (b + nw < nblk) one(b + nw, v1);
    }
}

}  // namespace

cudaError_t launch_quantize(const float *w, void *w_aos, int64_t n, int64_t k, const LaunchCtx &ctx) {
    const int64_t nblk = n * (k / kBlockW);
    if (nblk == 0) return cudaSuccess;
    // resident CTAs, a grid-stride loop over the blocks
    const int64_t grid = std::min<int64_t>((nblk + kQWarps - 1) / kQWarps, int64_t(ctx.num_sms) * 5);
    quantize_kernel<<<unsigned(grid), kQThreads, 0, ctx.stream>>>(w, static_cast<uint8_t *>(w_aos), nblk);
    return cudaPeekAtLastError();
}

}  // namespace tq2
