// unscale_check.cu - A1: non-finite check of the scaled gradients, and the
// optional in-place unscale ("第20章 量化与混合精度训练" §20.2.2; "从 AMP 到
// Mixed Precision" section "Gradient 和 Loss Scaling").
//
// Read-only check.  For a finite input g and the fp32 factor r = 1/S the
// product g*r is non-finite exactly when |g|*|r| overflows, and rounding is
// monotone, so a block of gradients holds a non-finite g*r iff
//     max|g| is inf/NaN, or max|g| * r is non-finite
// (this also covers r = inf, where 0*inf = NaN, and r = NaN).  The kernel
// therefore keeps a running max of |g| bit patterns - one SIMD integer max per
// two 16-bit gradients - and does one multiply per warp at the end.  Bytes
// moved: 2 per 16-bit gradient.
#include "internal.h"

namespace amp {
namespace {

template <int ET>
struct GradTraits;
template <>
struct GradTraits<kF32> {
    static constexpr uint32_t kAbsMask = 0x7FFFFFFFu;
    static constexpr uint32_t kInf = 0x7F800000u;
    static constexpr int kPerVec = 4;
};
template <>
struct GradTraits<kF16> {
    static constexpr uint32_t kAbsMask = 0x7FFF7FFFu;
    static constexpr uint32_t kInf = 0x7C00u;
    static constexpr int kPerVec = 8;
};
template <>
struct GradTraits<kBF16> {
    static constexpr uint32_t kAbsMask = 0x7FFF7FFFu;
    static constexpr uint32_t kInf = 0x7F80u;
    static constexpr int kPerVec = 8;
};

template <int ET>
__device__ __forceinline__ uint32_t abs_bits(const void *base, int64_t k) {
    if (ET == kF32) return reinterpret_cast<const uint32_t *>(base)[k] & 0x7FFFFFFFu;
    return reinterpret_cast<const uint16_t *>(base)[k] & 0x7FFFu;
}

template <int ET>
__device__ __forceinline__ float abs_bits_to_f32(uint32_t b) {
    if (ET == kF32) return __uint_as_float(b);
    return lowp_to_f32<ET>(b);
}

template <int ET>
__global__ void __launch_bounds__(kThreads) check_kernel(ListView g, const float *scale,
                                                         int32_t *found_inf) {
    using T = GradTraits<ET>;
    constexpr int esz = ET == kF32 ? 4 : 2;
    const uint2 ch = g.chunks[blockIdx.x];
    const int64_t start = int64_t(ch.y) * kChunk;
    const int64_t n = min(int64_t(kChunk), g.numel[ch.x] - start);
    const char *base = static_cast<const char *>(g.ptrs[ch.x]) + start * esz;

    uint32_t mx = 0;  // packed per-lane maxima of |g| bit patterns
    if (aligned16(base)) {
        const int64_t nv = n / T::kPerVec;
        for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
            uint4 w = ld_cs(base + i * 16);
            if (ET == kF32) {
                mx = max(mx, max(max(w.x & T::kAbsMask, w.y & T::kAbsMask),
                                 max(w.z & T::kAbsMask, w.w & T::kAbsMask)));
            } else {
                mx = __vmaxu2(mx, __vmaxu2(__vmaxu2(w.x & T::kAbsMask, w.y & T::kAbsMask),
                                           __vmaxu2(w.z & T::kAbsMask, w.w & T::kAbsMask)));
            }
        }
        if (ET != kF32) mx = max(mx & 0xFFFFu, mx >> 16);
        for (int64_t k = nv * T::kPerVec + threadIdx.x; k < n; k += kThreads)
            mx = max(mx, abs_bits<ET>(base, k));
    } else {
        for (int64_t k = threadIdx.x; k < n; k += kThreads) mx = max(mx, abs_bits<ET>(base, k));
    }
    // A warp whose lanes saw no element tests max|g| = 0, and 0 * r is
    // non-finite only for r = inf or NaN - and then every element of this
    // (non-empty) chunk gives a non-finite product too, so the flag is right.
    mx = warp_max_u32(mx);
    if ((threadIdx.x & 31) == 0) {
        const float r = scale ? __fdiv_rn(1.0f, *scale) : 1.0f;
        const bool bad = mx >= T::kInf || !isfinite(__fmul_rn(abs_bits_to_f32<ET>(mx), r));
        if (bad) atomicOr(found_inf, 1);
    }
}

// In place: every element is multiplied, checked and stored back.
template <int ET>
__global__ void __launch_bounds__(kThreads) unscale_inplace_kernel(ListView g, const float *scale,
                                                                   int32_t *found_inf) {
    const uint2 ch = g.chunks[blockIdx.x];
    const int64_t start = int64_t(ch.y) * kChunk;
    const int64_t n = min(int64_t(kChunk), g.numel[ch.x] - start);
    const float r = scale ? __fdiv_rn(1.0f, *scale) : 1.0f;
    bool bad = false;
    if (ET == kF32) {
        float *p = static_cast<float *>(g.ptrs[ch.x]) + start;
        for (int64_t k = threadIdx.x; k < n; k += kThreads) {
            const float y = __fmul_rn(p[k], r);
            bad |= !isfinite(y);
            p[k] = y;
        }
    } else {
        uint16_t *p = static_cast<uint16_t *>(g.ptrs[ch.x]) + start;
        for (int64_t k = threadIdx.x; k < n; k += kThreads) {
            const float y = __fmul_rn(lowp_to_f32<ET>(p[k]), r);
            bad |= !isfinite(y);
            p[k] = ET == kBF16 ? f32_to_bf16(y) : f32_to_f16(y);
        }
    }
    if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) atomicOr(found_inf, 1);
}

}  // namespace

cudaError_t launch_unscale_check(const ListView &g, int64_t n_chunks, int elem, const float *scale,
                                 int32_t *found_inf, int inplace, cudaStream_t s) {
    if (n_chunks == 0) return cudaSuccess;
    const dim3 grid((unsigned)n_chunks), block(kThreads);
    if (inplace) {
        if (elem == kF32) unscale_inplace_kernel<kF32><<<grid, block, 0, s>>>(g, scale, found_inf);
        else if (elem == kF16) unscale_inplace_kernel<kF16><<<grid, block, 0, s>>>(g, scale, found_inf);
        else unscale_inplace_kernel<kBF16><<<grid, block, 0, s>>>(g, scale, found_inf);
    } else {
        if (elem == kF32) check_kernel<kF32><<<grid, block, 0, s>>>(g, scale, found_inf);
        else if (elem == kF16) check_kernel<kF16><<<grid, block, 0, s>>>(g, scale, found_inf);
        else check_kernel<kBF16><<<grid, block, 0, s>>>(g, scale, found_inf);
    }
    return cudaGetLastError();
}

}  // namespace amp
