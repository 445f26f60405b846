// fp8_quant.cu - A6..A9: tensorwise dynamic FP8 quantization with the
// transposed (column-major) copy.
//
//   "FP8训练：量化、自动微分、Torchao" §2: amax = max|x| (fp32), scale =
//   fp8_max / max(double(amax), EPS) in fp64, q = clamp(x*scale, +-fp8_max)
//   cast to fp8, inv_scale = 1/scale; §3: e4m3fn (448) for weights and
//   activations, e5m2 (57344) for gradients; §4: the backward GEMMs need
//   column-major copies, i.e. the same bytes laid out [cols, rows].
//
// amax pass (single tensor, when not given): grid-stride 16-byte loads, four
//   in flight per thread, SIMD integer max of |x| bit patterns, a block-level
//   max and one atomicMax per CTA - 2 bytes read per bf16 element.
// quant pass: one CTA per 128x128 tile.  Each thread loads 8 rows x 8
//   columns with 16-byte coalesced loads, converts pairs with the hardware
//   RNE+satfinite cvt, stores its 8 row-major bytes, and parks them in a
//   16 KB shared tile whose 4-byte words are XOR-swizzled by row band.  The
//   transposed copy is then read back 16 words per thread (conflict-free),
//   transposed 4x4 bytes at a time with byte permutes, and written as 16-byte
//   stores in which 8 lanes cover one 128-byte segment of a transposed row.
//   Bytes: 2 read + 1 + 1 written per element.
// Tiles on a ragged edge, or with sizes/addresses that break 16-byte access,
// take an element-wise path with the same arithmetic.
// The list cast has a stochastic-rounding form for the FP8 weight copies
// ("第20章 量化与混合精度训练" §20.5.14): the same scaled fp32 values, each
// rounded by fp8_stochastic (philox.cuh) with 16 random bits drawn per
// element from its row-major index, so the transposed copy holds the same
// bytes.
#include <algorithm>

#include "fp8_tile.cuh"
#include "internal.h"
#include "pdl.cuh"
#include "philox.cuh"

namespace amp {
namespace {

template <int XT>
__device__ __forceinline__ float x_at(const void *x, int64_t k) {
    if (XT == kF32) return static_cast<const float *>(x)[k];
    return lowp_to_f32<XT>(static_cast<const uint16_t *>(x)[k]);
}

// Random-bit source of the stochastic cast: element k of this tensor rounds
// with sr8 bits of (seed, step, tensor, k).
struct SrArgs {
    uint64_t seed;
    int32_t step;
    int32_t tensor;
};

template <int XT, int FT, bool SR = false>
__device__ __forceinline__ void quant_tile(const void *x, int64_t rows, int64_t cols, uint8_t *out,
                                           uint8_t *out_t, int64_t r0, int64_t c0,
                                           const float *s_scale, uint32_t *sm,
                                           SrArgs sr = SrArgs{}) {
    constexpr int esz = XT == kF32 ? 4 : 2;
    constexpr int nv = XT == kF32 ? 2 : 1;  // 16-byte loads per 8 elements
    const bool fast = r0 + kTile <= rows && c0 + kTile <= cols && (cols & 7) == 0 &&
                      aligned16(x) && (reinterpret_cast<uintptr_t>(out) & 7) == 0 &&
                      (out_t == nullptr || ((rows & 15) == 0 && aligned16(out_t)));
    if (fast) {
        const int c8 = threadIdx.x & 15, rb = threadIdx.x >> 4;
        uint4 raw[8][nv];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t e = (r0 + rb + 16 * k) * cols + c0 + 8 * c8;
            const char *src = static_cast<const char *>(x) + e * esz;
#pragma unroll
            for (int u = 0; u < nv; ++u) raw[k][u] = ld16(src + 16 * u);
        }
        __syncthreads();  // s_scale is ready
        const float s32 = *s_scale;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float y[8];
            if constexpr (XT == kF32) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    y[4 * u + 0] = __uint_as_float(raw[k][u].x);
                    y[4 * u + 1] = __uint_as_float(raw[k][u].y);
                    y[4 * u + 2] = __uint_as_float(raw[k][u].z);
                    y[4 * u + 3] = __uint_as_float(raw[k][u].w);
                }
            } else {
                const uint32_t w[4] = {raw[k][0].x, raw[k][0].y, raw[k][0].z, raw[k][0].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    y[2 * j] = lowp_to_f32<XT>(w[j] & 0xFFFFu);
                    y[2 * j + 1] = lowp_to_f32<XT>(w[j] >> 16);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; j += 2) mul2_rn(y[j], y[j + 1], s32, s32, y[j], y[j + 1]);
            const int r = rb + 16 * k;
            uint2 q;
            if constexpr (SR) {
                q = fp8x8_stochastic<FT>(y, sr.seed, sr.step, sr.tensor,
                                         (r0 + r) * cols + c0 + 8 * c8);
            } else {
                q.x = fp8x4_canonical_nan<FT>(f32x2_to_fp8x2_raw<FT>(y[0], y[1]) |
                                              (f32x2_to_fp8x2_raw<FT>(y[2], y[3]) << 16));
                q.y = fp8x4_canonical_nan<FT>(f32x2_to_fp8x2_raw<FT>(y[4], y[5]) |
                                              (f32x2_to_fp8x2_raw<FT>(y[6], y[7]) << 16));
            }
            *reinterpret_cast<uint2 *>(out + (r0 + r) * cols + c0 + 8 * c8) = q;
            if (out_t) *reinterpret_cast<uint2 *>(sm + swz(r, 2 * c8)) = q;
        }
        if (out_t == nullptr) return;
        __syncthreads();
        store_transposed_tile(sm, out_t, rows, r0, c0);
    } else {
        __syncthreads();
        const float s32 = *s_scale;
        for (int idx = threadIdx.x; idx < kTile * kTile; idx += kThreads) {
            const int64_t i = r0 + (idx >> 7), j = c0 + (idx & (kTile - 1));
            if (i < rows && j < cols) {
                const int64_t k = i * cols + j;
                uint8_t q;
                if constexpr (SR)
                    q = uint8_t(fp8_stochastic<FT>(__fmul_rn(x_at<XT>(x, k), s32),
                                                   sr8_word(sr.seed, sr.step, sr.tensor, k)));
                else
                    q = quant1<FT>(x_at<XT>(x, k), s32);
                out[k] = q;
                if (out_t) out_t[j * rows + i] = q;
            }
        }
    }
}

template <int XT, int FT>
__global__ void __launch_bounds__(kThreads) quant_single_kernel(const void *x, int64_t rows,
                                                                int64_t cols, uint8_t *out,
                                                                uint8_t *out_t, const float *amax,
                                                                float *inv_scale, EpsFloor ef,
                                                                const int32_t *skip_if) {
    pdl_wait();
    pdl_trigger();
    if (skip_if && *skip_if) return;
    __shared__ __align__(16) uint32_t sm[kTile * 32];
    __shared__ float s_scale;
    // Tiles in reverse row-major order: the maxima pass sweeps x from its
    // start, so its last reads, still in L2, are the first ones here.
    const int64_t tiles_c = (cols + kTile - 1) / kTile;
    const int64_t tile = int64_t(gridDim.x) - 1 - blockIdx.x;
    const int64_t tr = tile / tiles_c, tc = tile % tiles_c;
    if (threadIdx.x == 0) {
        float s32, inv;
        tensor_scale(*amax, ef, fp8_max<FT>(), s32, inv);
        s_scale = s32;
        if (blockIdx.x == 0) *inv_scale = inv;
    }
    quant_tile<XT, FT>(x, rows, cols, out, out_t, tr * kTile, tc * kTile, &s_scale, sm);
}

// Tensor t of the list takes amax[a] and writes inv_scale[a] with a = its
// slot in X (use_slots; the slots the bf16 list folded the amax into) or t.
template <int XT, int FT, bool SR>
__device__ __forceinline__ void quant_list_body(const ListView &X, const ListView &O,
                                                const ListView &OT, int has_t, int use_slots,
                                                const float *amax, float *inv_scale,
                                                const EpsFloor &ef, const int32_t *skip_if,
                                                uint64_t sr_seed, const int32_t *sr_step) {
    pdl_wait();
    pdl_trigger();
    if (skip_if && *skip_if) return;
    __shared__ __align__(16) uint32_t sm[kTile * 32];
    __shared__ float s_scale;
    const uint2 tl = X.tiles[blockIdx.x];
    const int t = int(tl.x);
    const int64_t rows = X.rows[t], cols = X.cols[t];
    const int64_t tiles_c = (cols + kTile - 1) / kTile;
    const int64_t tr = tl.y / tiles_c, tc = tl.y % tiles_c;
    const int a = use_slots ? X.slots[t] : t;
    if (threadIdx.x == 0) {
        float s32, inv;
        tensor_scale(amax[a], ef, fp8_max<FT>(), s32, inv);
        s_scale = s32;
        if (tl.y == 0) inv_scale[a] = inv;
    }
    uint8_t *ot = has_t ? static_cast<uint8_t *>(OT.ptrs[t]) : nullptr;
    SrArgs sr{};
    if constexpr (SR) sr = SrArgs{sr_seed, *sr_step, a};
    quant_tile<XT, FT, SR>(X.ptrs[t], rows, cols, static_cast<uint8_t *>(O.ptrs[t]), ot,
                           tr * kTile, tc * kTile, &s_scale, sm, sr);
}

template <int XT, int FT>
__global__ void __launch_bounds__(kThreads) quant_list_kernel(ListView X, ListView O, ListView OT,
                                                              int has_t, int use_slots,
                                                              const float *amax,
                                                              float *inv_scale, EpsFloor ef,
                                                              const int32_t *skip_if) {
    quant_list_body<XT, FT, false>(X, O, OT, has_t, use_slots, amax, inv_scale, ef, skip_if, 0,
                                   nullptr);
}

// The stochastic cast: the same tile walk with the rounding of philox.cuh.
template <int XT, int FT>
__global__ void __launch_bounds__(kThreads) quant_list_sr_kernel(
    ListView X, ListView O, ListView OT, int has_t, int use_slots, const float *amax,
    float *inv_scale, EpsFloor ef, const int32_t *skip_if, uint64_t sr_seed,
    const int32_t *sr_step) {
    quant_list_body<XT, FT, true>(X, O, OT, has_t, use_slots, amax, inv_scale, ef, skip_if,
                                  sr_seed, sr_step);
}

// Tensors of a list with no elements have no tiles, so quant_list_kernel never
// visits them; their inv_scale still follows from their amax like any other's.
template <int FT>
__global__ void quant_list_empty_kernel(ListView X, int use_slots, const float *amax,
                                        float *inv_scale, EpsFloor ef, const int32_t *skip_if) {
    pdl_wait();
    pdl_trigger();
    if (skip_if && *skip_if) return;
    for (int t = threadIdx.x; t < X.n; t += blockDim.x) {
        if (X.numel[t] != 0) continue;
        const int a = use_slots ? X.slots[t] : t;
        float s32, inv;
        tensor_scale(amax[a], ef, fp8_max<FT>(), s32, inv);
        inv_scale[a] = inv;
    }
}

// amax is an output: it starts from +0 (unless the call is skipped).
__global__ void amax_zero_kernel(float *amax, const int32_t *skip_if) {
    pdl_wait();
    pdl_trigger();
    if (!(skip_if && *skip_if)) *amax = 0.0f;
}

template <int XT>
__global__ void __launch_bounds__(kThreads) amax_kernel(const void *x, int64_t n,
                                                        unsigned int *amax_bits,
                                                        const int32_t *skip_if) {
    pdl_wait();
    pdl_trigger();
    if (skip_if && *skip_if) return;
    const int64_t gtid = int64_t(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t gstride = int64_t(gridDim.x) * kThreads;
    uint32_t mx = 0;
    if (aligned16(x)) {
        constexpr int per = XT == kF32 ? 4 : 8;
        const int64_t nv = n / per;
        const char *b = static_cast<const char *>(x);
        auto fold = [&](const uint4 &w) {
            if (XT == kF32) {
                mx = max(mx, max(max(w.x & 0x7FFFFFFFu, w.y & 0x7FFFFFFFu),
                                 max(w.z & 0x7FFFFFFFu, w.w & 0x7FFFFFFFu)));
            } else {
                mx = __vmaxu2(mx, __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                                           __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu)));
            }
        };
        // four 16-byte loads in flight per thread, then the grid-stride tail
        int64_t i = gtid;
        for (; i + 3 * gstride < nv; i += 4 * gstride) {
            uint4 w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) w[u] = ld16(b + (i + u * gstride) * 16);
#pragma unroll
            for (int u = 0; u < 4; ++u) fold(w[u]);
        }
        for (; i < nv; i += gstride) fold(ld16(b + i * 16));
        if (XT != kF32) mx = max(mx & 0xFFFFu, mx >> 16);
        for (int64_t k = nv * per + gtid; k < n; k += gstride) {
            mx = max(mx, XT == kF32 ? (static_cast<const uint32_t *>(x)[k] & 0x7FFFFFFFu)
                                    : uint32_t(static_cast<const uint16_t *>(x)[k] & 0x7FFFu));
        }
    } else {
        for (int64_t k = gtid; k < n; k += gstride) {
            mx = max(mx, XT == kF32 ? (static_cast<const uint32_t *>(x)[k] & 0x7FFFFFFFu)
                                    : uint32_t(static_cast<const uint16_t *>(x)[k] & 0x7FFFu));
        }
    }
    // |x| bit patterns -> fp32 bit patterns of the same magnitude (monotone,
    // NaN above inf), so an unsigned max is the NaN-propagating fp32 max.
    uint32_t f;
    if (XT == kF32) f = mx;
    else if (XT == kBF16) f = mx << 16;
    else f = __float_as_uint(f16_bits_to_f32(mx));
    // one atomic per CTA: every CTA hits the same word, so per-warp atomics
    // would queue up at one L2 slice
    __shared__ uint32_t wmax[kThreads / 32];
    f = warp_max_u32(f);
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = f;
    __syncthreads();
    if (threadIdx.x < 32) {
        f = warp_max_u32(threadIdx.x < kThreads / 32 ? wmax[threadIdx.x] : 0u);
        if (threadIdx.x == 0 && f != 0) atomicMax(amax_bits, f);
    }
}

__global__ void quant_empty_kernel(float *amax, int amax_given, float *inv_scale, EpsFloor ef,
                                   float fmax, const int32_t *skip_if) {
    pdl_wait();
    pdl_trigger();
    if (skip_if && *skip_if) return;
    if (!amax_given) *amax = 0.0f;
    float s32, inv;
    tensor_scale(*amax, ef, fmax, s32, inv);
    *inv_scale = inv;
}

template <int XT, int FT>
cudaError_t launch_single(const void *x, int64_t rows, int64_t cols, uint8_t *out, uint8_t *out_t,
                          float *inv_scale, float *amax, int amax_given, double eps,
                          const int32_t *skip_if, int device, cudaStream_t s) {
    const int64_t n = rows * cols;
    if (!amax_given) {
        cudaError_t e = launch_pdl(amax_zero_kernel, dim3(1), dim3(1), 0, s, amax, skip_if);
        if (e != cudaSuccess) return e;
        const int64_t per = XT == kF32 ? 4 : 8;
        const int64_t want = (n / per + kThreads - 1) / kThreads;
        const int64_t cap = int64_t(sm_count(device)) * 8;
        const unsigned grid = (unsigned)std::max<int64_t>(1, std::min(want, cap));
        e = launch_pdl(amax_kernel<XT>, dim3(grid), dim3(kThreads), 0, s, x, n,
                       reinterpret_cast<unsigned int *>(amax), skip_if);
        if (e != cudaSuccess) return e;
    }
    const int64_t tiles = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
    return launch_pdl(quant_single_kernel<XT, FT>, dim3(unsigned(tiles)), dim3(kThreads), 0, s, x,
                      rows, cols, out, out_t, static_cast<const float *>(amax), inv_scale,
                      make_eps_floor(eps, fp8_max<FT>()), skip_if);
}

}  // namespace

cudaError_t launch_fp8_quant(const void *x, int xelem, int64_t rows, int64_t cols, int fp8,
                             double eps, uint8_t *out, uint8_t *out_t, float *inv_scale,
                             float *amax, int amax_given, const int32_t *skip_if, int device,
                             cudaStream_t s) {
    if (rows * cols == 0) {
        const float fmax = fp8 == kE4M3 ? fp8_max<kE4M3>() : fp8_max<kE5M2>();
        return launch_pdl(quant_empty_kernel, dim3(1), dim3(1), 0, s, amax, amax_given, inv_scale,
                          make_eps_floor(eps, fmax), fmax, skip_if);
    }
#define AMP_Q1(XT, FT) \
    launch_single<XT, FT>(x, rows, cols, out, out_t, inv_scale, amax, amax_given, eps, skip_if, \
                          device, s)
    if (fp8 == kE4M3) {
        if (xelem == kBF16) return AMP_Q1(kBF16, kE4M3);
        if (xelem == kF16) return AMP_Q1(kF16, kE4M3);
        return AMP_Q1(kF32, kE4M3);
    }
    if (xelem == kBF16) return AMP_Q1(kBF16, kE5M2);
    if (xelem == kF16) return AMP_Q1(kF16, kE5M2);
    return AMP_Q1(kF32, kE5M2);
#undef AMP_Q1
}

cudaError_t launch_fp8_quant_list(const ListView &x, int64_t n_tiles, bool any_empty, int xelem,
                                  const ListView &out, const ListView *out_t, int fp8,
                                  double eps, const float *amax, float *inv_scale,
                                  const int32_t *skip_if, cudaStream_t s, const int32_t *sr_step,
                                  uint64_t sr_seed, bool use_slots) {
    const int us = use_slots ? 1 : 0;
    if (any_empty) {
        if (fp8 == kE4M3) launch_pdl(quant_list_empty_kernel<kE4M3>, dim3(1), dim3(kThreads), 0, s,
                                     x, us, amax, inv_scale,
                                     make_eps_floor(eps, fp8_max<kE4M3>()), skip_if);
        else launch_pdl(quant_list_empty_kernel<kE5M2>, dim3(1), dim3(kThreads), 0, s, x, us, amax,
                        inv_scale, make_eps_floor(eps, fp8_max<kE5M2>()), skip_if);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (n_tiles == 0) return cudaSuccess;
    const ListView ot = out_t ? *out_t : ListView{};
    const int has_t = out_t != nullptr;
    const dim3 grid((unsigned)n_tiles), block(kThreads);
    const EpsFloor ef = make_eps_floor(eps, fp8 == kE4M3 ? fp8_max<kE4M3>() : fp8_max<kE5M2>());
#define AMP_QL(XT, FT)                                                                       \
    (sr_step ? launch_pdl(quant_list_sr_kernel<XT, FT>, grid, block, 0, s, x, out, ot, has_t, us, \
                          amax, inv_scale, ef, skip_if, sr_seed, sr_step)                        \
             : launch_pdl(quant_list_kernel<XT, FT>, grid, block, 0, s, x, out, ot, has_t, us,    \
                          amax, inv_scale, ef, skip_if))
    if (fp8 == kE4M3) {
        if (xelem == kBF16) AMP_QL(kBF16, kE4M3);
        else if (xelem == kF16) AMP_QL(kF16, kE4M3);
        else AMP_QL(kF32, kE4M3);
    } else {
        if (xelem == kBF16) AMP_QL(kBF16, kE5M2);
        else if (xelem == kF16) AMP_QL(kF16, kE5M2);
        else AMP_QL(kF32, kE5M2);
    }
#undef AMP_QL
    return cudaGetLastError();
}

}  // namespace amp
