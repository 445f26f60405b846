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
#include "pdl.cuh"

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

// Compensated (Kahan) fp32 running sum, one per thread.
struct SqSum {
    float sum = 0.0f, comp = 0.0f;
    __device__ __forceinline__ void add_value(float x) {
        const float y = __fsub_rn(x, comp);
        const float t = __fadd_rn(sum, y);
        comp = __fsub_rn(__fsub_rn(t, sum), y);
        sum = t;
    }
    __device__ __forceinline__ void add(float x) { add_value(__fmul_rn(x, x)); }
    __device__ __forceinline__ double value() const { return double(sum) - double(comp); }
};

// The two 16-bit values of a word as fp32, exactly.  bf16: a shift.  fp16:
// the 15 magnitude bits moved into an fp32 pattern read as v * 2^-112 (the
// exponent bias differs by 112; fp16 subnormals land on fp32 subnormals), then
// rescaled by 2^112 - integer and FMA-pipe work instead of a conversion per
// element.  Signs are dropped (only squares are needed); inf/NaN inputs are
// not represented, the caller flags them.
template <int ET>
__device__ __forceinline__ void widen_abs2(uint32_t w, float &lo, float &hi) {
    if (ET == kBF16) {
        lo = __uint_as_float((w << 16) & 0x7FFF0000u);
        hi = __uint_as_float(w & 0x7FFF0000u);
    } else {
        lo = __fmul_rn(__uint_as_float((w & 0x7FFFu) << 13), 0x1p112f);
        hi = __fmul_rn(__uint_as_float((w >> 3) & 0x0FFFE000u), 0x1p112f);
    }
}

// Sum of squares of one 16-byte vector: two fused multiply-add chains (the
// products of 16-bit values are exact in fp32), then one compensated add.
template <int ET>
__device__ __forceinline__ void sq_add_vec(SqSum &q, const uint4 &w) {
    if (ET == kF32) {
        const float x0 = __uint_as_float(w.x), x1 = __uint_as_float(w.y);
        const float x2 = __uint_as_float(w.z), x3 = __uint_as_float(w.w);
        float a = __fmul_rn(x0, x0);
        a = __fmaf_rn(x1, x1, a);
        a = __fmaf_rn(x2, x2, a);
        a = __fmaf_rn(x3, x3, a);
        q.add_value(a);
    } else {
        float x[8];
        widen_abs2<ET>(w.x, x[0], x[1]);
        widen_abs2<ET>(w.y, x[2], x[3]);
        widen_abs2<ET>(w.z, x[4], x[5]);
        widen_abs2<ET>(w.w, x[6], x[7]);
        float a = __fmul_rn(x[0], x[0]), b = __fmul_rn(x[4], x[4]);
        a = __fmaf_rn(x[1], x[1], a);
        b = __fmaf_rn(x[5], x[5], b);
        a = __fmaf_rn(x[2], x[2], a);
        b = __fmaf_rn(x[6], x[6], b);
        a = __fmaf_rn(x[3], x[3], a);
        b = __fmaf_rn(x[7], x[7], b);
        q.add_value(__fadd_rn(a, b));
    }
}

// NORM: also the chunk's sum of squared unscaled gradients, written to
// g.partials[chunk] in fp64.  Each thread keeps a compensated fp32 sum of the
// squared stored values (exact for 16-bit inputs), the CTA adds the threads'
// sums in fp64 in a fixed tree, and the chunk total is multiplied by (1/S)^2
// - the same per-element value as squaring the fp32 unscaled gradient when
// 1/S is a power of two, as the scale state machine keeps it.  The fixed
// order makes the result independent of scheduling.
template <int ET, bool NORM>
__global__ void __launch_bounds__(kThreads) check_kernel(ListView g, const float *scale,
                                                         int32_t *found_inf) {
    pdl_wait();
    pdl_trigger();
    using T = GradTraits<ET>;
    constexpr int esz = ET == kF32 ? 4 : 2;
    const uint2 ch = g.chunks[blockIdx.x];
    const int64_t start = int64_t(ch.y) * kChunk;
    const int64_t n = min(int64_t(kChunk), g.numel[ch.x] - start);
    const char *base = static_cast<const char *>(g.ptrs[ch.x]) + start * esz;

    uint32_t mx = 0;  // packed per-lane maxima of |g| bit patterns
    SqSum q;
    if (aligned16(base)) {
        const int64_t nv = n / T::kPerVec;
        // four independent 16-byte loads in flight per thread before any use
        constexpr int U = 4;
        for (int64_t i = threadIdx.x; i < nv; i += U * kThreads) {
            uint4 w[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t j = i + int64_t(u) * kThreads;
                w[u] = j < nv ? ld16(base + j * 16) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (ET == kF32) {
                    mx = max(mx, max(max(w[u].x & T::kAbsMask, w[u].y & T::kAbsMask),
                                     max(w[u].z & T::kAbsMask, w[u].w & T::kAbsMask)));
                } else {
                    mx = __vmaxu2(mx, __vmaxu2(__vmaxu2(w[u].x & T::kAbsMask, w[u].y & T::kAbsMask),
                                               __vmaxu2(w[u].z & T::kAbsMask, w[u].w & T::kAbsMask)));
                }
                if constexpr (NORM) sq_add_vec<ET>(q, w[u]);
            }
        }
        if (ET != kF32) mx = max(mx & 0xFFFFu, mx >> 16);
        for (int64_t k = nv * T::kPerVec + threadIdx.x; k < n; k += kThreads) {
            mx = max(mx, abs_bits<ET>(base, k));
            if constexpr (NORM) q.add(abs_bits_to_f32<ET>(abs_bits<ET>(base, k)));
        }
    } else {
        for (int64_t k = threadIdx.x; k < n; k += kThreads) {
            mx = max(mx, abs_bits<ET>(base, k));
            if constexpr (NORM) q.add(abs_bits_to_f32<ET>(abs_bits<ET>(base, k)));
        }
    }
    if constexpr (NORM) {
        __shared__ double part[kThreads / 32];
        double v = q.value();
        for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xFFFFFFFFu, v, off);
        if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
        const int part_bad = __syncthreads_or(mx >= T::kInf);
        if (threadIdx.x == 0) {
            double t = 0.0;
            for (int w = 0; w < kThreads / 32; ++w) t += part[w];
            const double r = double(scale ? __fdiv_rn(1.0f, *scale) : 1.0f);
            // a non-finite gradient makes the sum NaN (the step is skipped then)
            g.partials[blockIdx.x] = part_bad ? __longlong_as_double(0x7FF8000000000000ll)
                                              : t * (r * r);
        }
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
__device__ __forceinline__ uint16_t narrow16(float y) {
    return ET == kBF16 ? f32_to_bf16(y) : f32_to_f16(y);
}

// One 16-byte word of gradients unscaled in place: 4 fp32 or 8 16-bit values,
// each multiplied by r and rounded back exactly as the element path does.
template <int ET>
__device__ __forceinline__ uint4 unscale_word(uint4 w, float r, bool &bad) {
    uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (ET == kF32) {
            const float y = __fmul_rn(__uint_as_float(v[j]), r);
            bad |= !isfinite(y);
            v[j] = __float_as_uint(y);
        } else {
            const float lo = __fmul_rn(lowp_to_f32<ET>(v[j] & 0xFFFFu), r);
            const float hi = __fmul_rn(lowp_to_f32<ET>(v[j] >> 16), r);
            bad |= !isfinite(lo) || !isfinite(hi);
            v[j] = uint32_t(narrow16<ET>(lo)) | (uint32_t(narrow16<ET>(hi)) << 16);
        }
    }
    return make_uint4(v[0], v[1], v[2], v[3]);
}

// 16-byte loads and stores, four words in flight per thread, when the chunk
// is 16-byte aligned; the tail and misaligned chunks go element by element.
// 2 bytes read + 2 written per 16-bit gradient.
template <int ET>
__global__ void __launch_bounds__(kThreads) unscale_inplace_kernel(ListView g, const float *scale,
                                                                   int32_t *found_inf) {
    pdl_wait();
    pdl_trigger();
    using T = GradTraits<ET>;
    constexpr int esz = ET == kF32 ? 4 : 2;
    const uint2 ch = g.chunks[blockIdx.x];
    const int64_t start = int64_t(ch.y) * kChunk;
    const int64_t n = min(int64_t(kChunk), g.numel[ch.x] - start);
    char *base = static_cast<char *>(g.ptrs[ch.x]) + start * esz;
    const float r = scale ? __fdiv_rn(1.0f, *scale) : 1.0f;
    bool bad = false;
    int64_t done = 0;
    if (aligned16(base)) {
        const int64_t nv = n / T::kPerVec;
        constexpr int U = 4;
        for (int64_t i = threadIdx.x; i < nv; i += U * kThreads) {
            uint4 w[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t j = i + int64_t(u) * kThreads;
                if (j < nv) w[u] = ld16(base + j * 16);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t j = i + int64_t(u) * kThreads;
                if (j < nv)
                    *reinterpret_cast<uint4 *>(base + j * 16) = unscale_word<ET>(w[u], r, bad);
            }
        }
        done = nv * T::kPerVec;
    }
    if (ET == kF32) {
        float *p = reinterpret_cast<float *>(base);
        for (int64_t k = done + threadIdx.x; k < n; k += kThreads) {
            const float y = __fmul_rn(p[k], r);
            bad |= !isfinite(y);
            p[k] = y;
        }
    } else {
        uint16_t *p = reinterpret_cast<uint16_t *>(base);
        for (int64_t k = done + threadIdx.x; k < n; k += kThreads) {
            const float y = __fmul_rn(lowp_to_f32<ET>(p[k]), r);
            bad |= !isfinite(y);
            p[k] = narrow16<ET>(y);
        }
    }
    if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) atomicOr(found_inf, 1);
}

// Sum of the per-chunk partials in a fixed order: each thread a fixed
// strided subset, then a fixed shared-memory tree.
__global__ void __launch_bounds__(1024) norm_reduce_kernel(const double *partials, int64_t n,
                                                           double *out) {
    pdl_wait();
    pdl_trigger();
    __shared__ double sm[1024];
    double v = 0.0;
    for (int64_t i = threadIdx.x; i < n; i += 1024) v += partials[i];
    sm[threadIdx.x] = v;
    __syncthreads();
    for (int s = 512; s > 0; s >>= 1) {
        if (threadIdx.x < s) sm[threadIdx.x] += sm[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) *out = sm[0];
}

}  // namespace

cudaError_t launch_check_norm(const ListView &g, int64_t n_chunks, int elem, const float *scale,
                              int32_t *found_inf, double *sumsq, cudaStream_t s) {
    if (n_chunks > 0) {
        const dim3 grid((unsigned)n_chunks), block(kThreads);
        if (elem == kF32) launch_pdl(check_kernel<kF32, true>, dim3(grid), dim3(block), 0, s, g,
                                     scale, found_inf);
        else if (elem == kF16) launch_pdl(check_kernel<kF16, true>, dim3(grid), dim3(block), 0, s,
                                          g, scale, found_inf);
        else launch_pdl(check_kernel<kBF16, true>, dim3(grid), dim3(block), 0, s, g, scale,
                        found_inf);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    launch_pdl(norm_reduce_kernel, dim3(1), dim3(1024), 0, s, g.partials, n_chunks, sumsq);
    return cudaGetLastError();
}

cudaError_t launch_unscale_check(const ListView &g, int64_t n_chunks, int elem, const float *scale,
                                 int32_t *found_inf, int inplace, cudaStream_t s) {
    if (n_chunks == 0) return cudaSuccess;
    const dim3 grid((unsigned)n_chunks), block(kThreads);
    if (inplace) {
        if (elem == kF32) launch_pdl(unscale_inplace_kernel<kF32>, dim3(grid), dim3(block), 0, s, g,
                                     scale, found_inf);
        else if (elem == kF16) launch_pdl(unscale_inplace_kernel<kF16>, dim3(grid), dim3(block), 0,
                                          s, g, scale, found_inf);
        else launch_pdl(unscale_inplace_kernel<kBF16>, dim3(grid), dim3(block), 0, s, g, scale,
                        found_inf);
    } else {
        if (elem == kF32) launch_pdl(check_kernel<kF32, false>, dim3(grid), dim3(block), 0, s, g,
                                     scale, found_inf);
        else if (elem == kF16) launch_pdl(check_kernel<kF16, false>, dim3(grid), dim3(block), 0, s,
                                          g, scale, found_inf);
        else launch_pdl(check_kernel<kBF16, false>, dim3(grid), dim3(block), 0, s, g, scale,
                        found_inf);
    }
    return cudaGetLastError();
}

}  // namespace amp
