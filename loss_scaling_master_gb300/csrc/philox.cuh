// philox.cuh - Philox4x32-10 counter-based generator (Salmon, Moraes, Dror,
// Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011), and the
// stochastic bf16 rounding it feeds ("第20章 量化与混合精度训练" §20.5.14).
#pragma once

#include "common.cuh"

namespace amp {

// Ten rounds on a 4 x 32-bit counter with a 2 x 32-bit key: two 32x32->64
// products per round (multipliers 0xD2511F53, 0xCD9E8D57), key bumped by the
// Weyl constants 0x9E3779B9 and 0xBB67AE85 between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

// 16 random bits per element: element k of tensor `tensor` at optimizer step
// `step` takes half (k%8)%2 (low first) of word (k%8)/2 of the generator's
// output for counter {k/8 low, k/8 high, step, tensor} under key = seed.
__device__ __forceinline__ uint4 sr_random8(uint64_t seed, int32_t step, int32_t tensor,
                                            int64_t group) {
    return philox4x32_10(make_uint4(uint32_t(group), uint32_t(uint64_t(group) >> 32),
                                    uint32_t(step), uint32_t(tensor)),
                         make_uint2(uint32_t(seed), uint32_t(seed >> 32)));
}

// Round p to bf16 away from zero with probability (dropped 16 bits) / 2^16,
// toward zero otherwise; NaN -> canonical 0x7FC0.
__device__ __forceinline__ uint32_t bf16_stochastic(float p, uint32_t u16) {
    const uint32_t bits = __float_as_uint(p);
    const uint32_t mag = bits & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return kBf16NaN;
    const uint32_t r = (mag >> 16) + ((u16 & 0xFFFFu) < (mag & 0xFFFFu) ? 1u : 0u);
    return ((bits >> 16) & 0x8000u) | r;
}

}  // namespace amp

namespace amp {

// Tensor word of the FP8 copies' random stream: 16 bits per element in
// sr_random8's layout, at tensor word tensor | 2^31 - apart from the bf16
// copy's stream, whose tensor words stay below 2^31.
constexpr uint32_t kSr8Stream = 0x80000000u;

// Stochastic rounding of the fp32 value y (already scaled) to FP8 format FT
// with 16 random bits u ("第20章 量化与混合精度训练" §20.5.14): |y| is clamped
// to fp8_max; between the FP8 magnitudes lo <= |y| < lo + quantum the result
// is the upper one exactly when u < floor(2^16 * (|y| - lo) / quantum), else
// lo, with y's sign; NaN gives the canonical NaN byte.  The probability is
// the distance ratio truncated to a multiple of 2^-16.
//   - FP8 normal range (|y| >= 2^EMIN): the quantum is 2^(e - M) for |y|'s
//     binade e, so lo is |y| with its low 23 - M fraction bits cleared, and
//     the top 16 of those bits are the threshold; one quantum added to lo's
//     bit pattern carries into the exponent at a binade edge.  Integer
//     operations only.
//   - below it the quantum is 2^(EMIN - M): |y| / quantum, its integer part
//     and fraction are exact in fp32, so the threshold is the fraction times
//     2^16, truncated.
// The result, on the FP8 grid and not above fp8_max, converts exactly.
template <int FT>
__device__ __forceinline__ uint32_t fp8_stochastic(float y, uint32_t u16) {
    constexpr int M = FT == kE4M3 ? 3 : 2;       // fraction bits
    constexpr int EMIN = FT == kE4M3 ? -6 : -14;  // exponent of the smallest normal
    constexpr uint32_t kDrop = 23 - M;            // fp32 fraction bits below an FP8 quantum
    const uint32_t yb = __float_as_uint(y);
    const uint32_t ab = min(yb & 0x7FFFFFFFu, __float_as_uint(fp8_max<FT>()));
    uint32_t rb;
    if (ab >= uint32_t(127 + EMIN) << 23) {
        const uint32_t num = (ab >> (kDrop - 16)) & 0xFFFFu;
        rb = (ab & ~((1u << kDrop) - 1u)) + (u16 < num ? (1u << kDrop) : 0u);
    } else {
        const float s =
            __fmul_rn(__uint_as_float(ab), __uint_as_float(uint32_t(127 + M - EMIN) << 23));
        const float n = truncf(s);
        const uint32_t num = __float2uint_rz(__fmul_rn(__fsub_rn(s, n), 65536.0f));
        rb = __float_as_uint(__fmul_rn(u16 < num ? __fadd_rn(n, 1.0f) : n,
                                       __uint_as_float(uint32_t(127 - M + EMIN) << 23)));
    }
    const uint32_t q =
        f32x2_to_fp8x2_raw<FT>(__uint_as_float(rb | (yb & 0x80000000u)), 0.0f) & 0xFFu;
    return (yb & 0x7FFFFFFFu) > 0x7F800000u ? uint32_t(FT == kE4M3 ? kE4M3NaN : kE5M2NaN) : q;
}

// Eight fp32 values (already scaled) of consecutive elements k0 .. k0+7 (k0 a
// multiple of 8) of FP8 tensor `tensor` -> eight stochastically rounded fp8
// bytes, one generator call.
template <int FT>
__device__ __forceinline__ uint2 fp8x8_stochastic(const float (&y)[8], uint64_t seed, int32_t step,
                                                  int32_t tensor, int64_t k0) {
    const uint4 r = sr_random8(seed, step, int32_t(uint32_t(tensor) | kSr8Stream), k0 >> 3);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint32_t b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        b[j] = fp8_stochastic<FT>(y[j], (w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
    return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                      b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// The 16 random bits of one element k of FP8 tensor `tensor` (element paths).
__device__ __forceinline__ uint32_t sr8_word(uint64_t seed, int32_t step, int32_t tensor,
                                             int64_t k) {
    const uint4 r = sr_random8(seed, step, int32_t(uint32_t(tensor) | kSr8Stream), k >> 3);
    const int lane = int(k & 7);
    const uint32_t w = (lane >> 1) == 0 ? r.x : (lane >> 1) == 1 ? r.y : (lane >> 1) == 2 ? r.z : r.w;
    return (lane & 1) ? (w >> 16) : (w & 0xFFFFu);
}

}  // namespace amp
