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
// toward zero otherwise, with 16 random bits u: away exactly when u < the
// dropped bits.  As an addition: p's bit pattern plus 2^16 - 1 - u carries
// into bit 16 exactly then, and for a non-NaN p never into the sign bit, so
// bits 16..31 of the sum are the bf16 result.  NaN is left to the caller.
__device__ __forceinline__ uint32_t bf16_sr_top(float p, uint32_t u16) {
    return __float_as_uint(p) + (0xFFFFu - u16);
}

// One element: NaN -> canonical 0x7FC0.
__device__ __forceinline__ uint32_t bf16_stochastic(float p, uint32_t u16) {
    return p != p ? kBf16NaN : bf16_sr_top(p, u16 & 0xFFFFu) >> 16;
}

// max with NaN propagation (a NaN in either operand gives NaN).
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// True when any of eight values is NaN.
__device__ __forceinline__ bool any_nan8(const float (&v)[8]) {
    const float m = fmax_nan(fmax_nan(fmax_nan(v[0], v[1]), fmax_nan(v[2], v[3])),
                             fmax_nan(fmax_nan(v[4], v[5]), fmax_nan(v[6], v[7])));
    return m != m;
}

// Eight fp32 values -> four bf16x2 words, stochastically rounded with the
// 16-bit halves of the four random words (low half for the even element).
__device__ __forceinline__ uint4 bf16x8_stochastic(const float (&p)[8], const uint4 &rnd) {
    const uint32_t w[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        h[j] = __byte_perm(bf16_sr_top(p[2 * j], w[j] & 0xFFFFu),
                           bf16_sr_top(p[2 * j + 1], w[j] >> 16), 0x7632);
    if (any_nan8(p)) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (p[j] != p[j])
                h[j >> 1] = (j & 1) ? (h[j >> 1] & 0xFFFFu) | (kBf16NaN << 16)
                                    : (h[j >> 1] & 0xFFFF0000u) | kBf16NaN;
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
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
// One integer path reads lo's code and the threshold off an fp32 bit
// pattern z whose fraction field starts with M bits of lo and 16 bits of the
// threshold:
//   - FP8 normal range (|y| >= 2^EMIN): z = |y|; the quantum is 2^(e - M) for
//     |y|'s binade e, and z >> (23 - M) is lo's code plus (127 - bias) << M.
//   - below it the quantum is 2^(EMIN - M), the spacing of the M-bit grid on
//     [2^EMIN, 2^(EMIN+1)): z = (|y| + 2^EMIN) / 2 rounded toward zero (one
//     fused multiply-add), whose fraction field is floor(|y| * 2^(23 - EMIN))
//     - truncation, so its top bits are the floors of |y| / quantum and of
//     2^16 |y| / quantum - and whose exponent is the normal range's offset.
//   That z is the larger of the two patterns: (|y| + 2^EMIN) / 2 is below |y|
//   exactly when |y| > 2^EMIN, and equal at 2^EMIN.
// The decision is an addition: (2^16 - 1 - u) placed under the threshold's
// 16 bits carries into lo's code exactly when u < threshold (the 4 or 5 bits
// below the threshold cannot carry); adding one quantum to the code carries
// into the exponent at a binade edge and from the largest subnormal code into
// the smallest normal one.  Everything is shifted left by M + 1, so that the
// code lands in bits 24..30: (z - (127 - bias) << 23 + addend) << (M + 1),
// modulo 2^32, is z * 2^(M+1) + (2^16 - 1 - u) * 2^8 + 2^30 in both formats.
// Bit 31 takes y's sign; NaN is left to the caller.
template <int FT>
__device__ __forceinline__ uint32_t fp8_sr_top(float y, uint32_t c) {
    constexpr int M = FT == kE4M3 ? 3 : 2;       // fraction bits
    constexpr int EMIN = FT == kE4M3 ? -6 : -14;  // exponent of the smallest normal
    constexpr uint32_t kBias = uint32_t(127 + EMIN - 1) << 23;
    static_assert(0u - (kBias << (M + 1)) == 0x40000000u, "addend constant");
    const float a = fminf(fabsf(y), fp8_max<FT>());
    const uint32_t z = max(__float_as_uint(a),
                           __float_as_uint(__fmaf_rz(a, 0.5f, __uint_as_float(kBias))));
    return (z * (1u << (M + 1)) + c) | (__float_as_uint(y) & 0x80000000u);
}

// The addend of fp8_sr_top for 16 random bits u.
__device__ __forceinline__ uint32_t fp8_sr_addend(uint32_t u16) {
    return (0xFFFFu - u16) * 256u + 0x40000000u;
}

template <int FT>
__device__ __forceinline__ uint32_t fp8_stochastic(float y, uint32_t u16) {
    return y != y ? uint32_t(FT == kE4M3 ? kE4M3NaN : kE5M2NaN)
                  : fp8_sr_top<FT>(y, fp8_sr_addend(u16 & 0xFFFFu)) >> 24;
}

// Eight fp32 values (already scaled) of consecutive elements k0 .. k0+7 (k0 a
// multiple of 8) of FP8 tensor `tensor` -> eight stochastically rounded fp8
// bytes, one generator call; the codes are gathered from the top bytes.
template <int FT>
__device__ __forceinline__ uint2 fp8x8_stochastic(const float (&y)[8], uint64_t seed, int32_t step,
                                                  int32_t tensor, int64_t k0) {
    const uint4 r = sr_random8(seed, step, int32_t(uint32_t(tensor) | kSr8Stream), k0 >> 3);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint32_t t[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        t[2 * j] = fp8_sr_top<FT>(y[2 * j], fp8_sr_addend(w[j] & 0xFFFFu));
        t[2 * j + 1] = fp8_sr_top<FT>(y[2 * j + 1], fp8_sr_addend(w[j] >> 16));
    }
    uint2 q = make_uint2(
        __byte_perm(__byte_perm(t[0], t[1], 0x0073), __byte_perm(t[2], t[3], 0x0073), 0x5410),
        __byte_perm(__byte_perm(t[4], t[5], 0x0073), __byte_perm(t[6], t[7], 0x0073), 0x5410));
    if (any_nan8(y)) {
        constexpr uint32_t kNaN = FT == kE4M3 ? kE4M3NaN : kE5M2NaN;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (y[j] != y[j]) {
                uint32_t &word = j < 4 ? q.x : q.y;
                const int sh = 8 * (j & 3);
                word = (word & ~(0xFFu << sh)) | (kNaN << sh);
            }
    }
    return q;
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
