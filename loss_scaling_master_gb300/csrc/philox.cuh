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
