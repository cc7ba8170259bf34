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
// one, which the warp forms in any order as a 64-bit integer of aligned
// significands, and d is that integer times 2^(e_min - 157) rounded to binary16
// with integer operations.  Blocks with a wider exponent span, or with an Inf
// or NaN, take the literal route: lane 0 adds the 128 magnitudes in double in
// index order.  Both give the same bytes; the FP64 pipe, a small fraction of
// the FP32 one on this part, is used only for the rare wide blocks.
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

// binary16 bits of S * 2^E, round to nearest even (S < 2^53): overflow to Inf
// from 65520 up, subnormals on the 2^-24 grid (1024 carries into the exponent).
__device__ __forceinline__ uint16_t half_of_scaled(uint64_t S, int E) {
    if (S == 0) return 0;
    const int p = 63 - __clzll(static_cast<long long>(S));  // leading bit
    int e = p + E;                                          // unbiased exponent of the value
    // bits to drop: to 11 significant bits (normal) or to the 2^-24 grid (subnormal)
    const int shift = e >= -14 ? p - 10 : -(E + 24);
    uint64_t m;
    if (shift <= 0) {
        m = S << (-shift);
    } else if (shift >= 64) {
        m = 0;  // below half of the smallest subnormal
    } else {
        m = S >> shift;
        const uint64_t rem = S & ((uint64_t(1) << shift) - 1), half = uint64_t(1) << (shift - 1);
        if (rem > half || (rem == half && (m & 1))) ++m;
    }
    if (e < -14) return uint16_t(m);  // subnormal (m == 1024 is the smallest normal's encoding)
    if (m == 2048) m = 1024, ++e;
    if (e > 15) return 0x7c00;
    return uint16_t(((e + 15) << 10) | int(m - 1024));
}

constexpr int kQWarps = kQThreads / 32;

__global__ void __launch_bounds__(kQThreads)
quantize_kernel(const float *__restrict__ w, uint8_t *__restrict__ aos, int64_t nblk) {
    __shared__ float fb[kQWarps][kBlockW];  // the literal route's staging, per warp
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    const int64_t nw = int64_t(gridDim.x) * kQWarps;
    auto one = [&](int64_t b, const float4 v) {
        const float x[4] = {v.x, v.y, v.z, v.w};
        uint32_t a[4];
        int ex_lo = 255, ex_hi = 0;
        bool wide = false;
#pragma unroll
        for (int f = 0; f < 4; ++f) {
            a[f] = __float_as_uint(x[f]) & 0x7fffffffu;
            const int E = int(a[f] >> 23);
            wide |= E == 255;  // Inf or NaN
            if (a[f] != 0) {
                const int ex = E > 0 ? E : 1;
                ex_lo = min(ex_lo, ex);
                ex_hi = max(ex_hi, ex);
            }
        }
        const int emin = int(__reduce_min_sync(0xffffffffu, uint32_t(ex_lo)));
        const int emax = int(__reduce_max_sync(0xffffffffu, uint32_t(ex_hi)));
        wide = __any_sync(0xffffffffu, wide) || (emax >= emin && emax - emin > 22);
        uint16_t dh;
        if (!wide) {
            uint64_t t = 0;
            if (emax >= emin) {  // some nonzero weight
#pragma unroll
                for (int f = 0; f < 4; ++f)
                    if (a[f] != 0) {
                        const int E = int(a[f] >> 23);
                        const uint64_t mant = (a[f] & 0x7fffffu) | (E > 0 ? 0x800000u : 0u);
                        t += mant << ((E > 0 ? E : 1) - emin);
                    }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            }
            dh = half_of_scaled(t, emin - 157);  // (sum / 128) = t * 2^(emin - 150 - 7)
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
        const float df = __half2float(__ushort_as_half(dh));
        const bool live = df > 0.f && isfinite(df);
        uint32_t byte = 0;
#pragma unroll
        for (int f = 0; f < 4; ++f) {
            int c = 1;
            if (live) {
                const float q = rintf(__fdiv_rn(x[f], df));
                c = q >= 1.f ? 2 : (q <= -1.f ? 0 : 1);
            }
            byte |= uint32_t(c) << (2 * f);
        }
        // qs[l] is this lane's byte: lanes 2i and 2i+1 store one 16-bit word
        // (a block starts on an even byte); lane 0 also stores d
        const uint32_t hi = __shfl_down_sync(0xffffffffu, byte, 1);
        uint8_t *ob = aos + b * kBlockBytes;
        if ((lane & 1) == 0) *reinterpret_cast<uint16_t *>(ob + lane) = uint16_t(byte | (hi << 8));
        if (lane == 0) *reinterpret_cast<uint16_t *>(ob + 32) = dh;
    };
    // grid-stride over blocks, two loads in flight per warp
    for (int64_t b = int64_t(blockIdx.x) * kQWarps + wi; b < nblk; b += 2 * nw) {
        const float4 v0 = __ldcs(reinterpret_cast<const float4 *>(w + b * kBlockW) + lane);
        const bool two = b + nw < nblk;
        float4 v1 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (two) v1 = __ldcs(reinterpret_cast<const float4 *>(w + (b + nw) * kBlockW) + lane);
        one(b, v0);
        if (two) one(b + nw, v1);
    }
}

}  // namespace

cudaError_t launch_quantize(const float *w, void *w_aos, int64_t n, int64_t k, const LaunchCtx &ctx) {
    const int64_t nblk = n * (k / kBlockW);
    if (nblk == 0) return cudaSuccess;
    // resident CTAs, a grid-stride loop over the blocks
    const int64_t grid = std::min<int64_t>((nblk + kQWarps - 1) / kQWarps, int64_t(ctx.num_sms) * 4);
    quantize_kernel<<<unsigned(grid), kQThreads, 0, ctx.stream>>>(w, static_cast<uint8_t *>(w_aos), nblk);
    return cudaPeekAtLastError();
}

}  // namespace tq2
