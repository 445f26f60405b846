// fp8_rowwise.cu - rowwise FP8 scaling ("FP8训练：量化、自动微分、Torchao" §1:
// one scale per row instead of one per tensor, §2's formula per row; §4: the
// column-major copy for the backward GEMMs, whose reduction runs along the
// rows, carries one scale per column).
//
// Four launches, 6 bytes per element as for the tensorwise cast:
//   zero   amax_row[rows], amax_col[cols] <- +0 (skipped calls write nothing)
//   amax   one wave of CTAs reads x once (2 B/elt), S CTAs per column strip,
//          each taking every S-th 128x128 tile down its strip, so that the
//          wave sweeps x from top to bottom; every thread holds 8 rows x 8
//          columns of a tile; row maxima are combined across the 16 lanes
//          sharing a row (one atomicMax per row and tile), column maxima stay
//          in registers for the strip (one atomicMax per column at the end);
//          fp32 bit patterns of |x| (16-bit x: 16-bit patterns, widened for
//          the atomics): an unsigned max that propagates NaN
//   scale  per row and per column, fp32 multiplier and inverse written once,
//          by fp32 divisions equal to the fp64 formula rounded to fp32
//          (tensor_scale in fp8_tile.cuh)
//   cast   one CTA per tile reads it again (2 B/elt), casts each element twice
//          (row multiplier for the row-major bytes, column multiplier for the
//          transposed bytes) and writes both (1 + 1 B/elt), the transposed
//          tile through the swizzled shared-memory transpose.  The tiles go
//          in reverse row-major order, the reverse of the maxima pass's
//          sweep, so the first reads find x still in L2.
#include <algorithm>
#include <atomic>

#include "fp8_tile.cuh"
#include "internal.h"
#include "pdl.cuh"

namespace amp {
namespace {

// |x| of element k as the bit pattern of an fp32 magnitude (monotone in |x|,
// NaN above inf).
template <int XT>
__device__ __forceinline__ uint32_t abs_f32_bits(const void *x, int64_t k) {
    if (XT == kF32) return static_cast<const uint32_t *>(x)[k] & 0x7FFFFFFFu;
    const uint32_t h = static_cast<const uint16_t *>(x)[k] & 0x7FFFu;
    return XT == kBF16 ? (h << 16) : __float_as_uint(f16_bits_to_f32(h));
}

// A 16-bit magnitude pattern (sign clear) as the fp32 pattern of the same
// value, as abs_f32_bits gives it; 0 stays 0.
template <int XT>
__device__ __forceinline__ uint32_t widen16(uint32_t h) {
    return XT == kBF16 ? (h << 16) : __float_as_uint(f16_bits_to_f32(h));
}

// |x| bit patterns (as abs_f32_bits) of 8 consecutive elements held in one
// (16-bit types) or two (fp32) 16-byte words
template <int XT>
__device__ __forceinline__ void raw_abs(const uint4 *u, uint32_t (&a)[8]) {
    if (XT == kF32) {
        const uint32_t w[8] = {u[0].x, u[0].y, u[0].z, u[0].w, u[1].x, u[1].y, u[1].z, u[1].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = w[j] & 0x7FFFFFFFu;
    } else {
        const uint32_t w[4] = {u[0].x, u[0].y, u[0].z, u[0].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = w[j] & 0x7FFFu, hi = (w[j] >> 16) & 0x7FFFu;
            if (XT == kBF16) {
                a[2 * j] = lo << 16;
                a[2 * j + 1] = hi << 16;
            } else {
                a[2 * j] = __float_as_uint(f16_bits_to_f32(lo));
                a[2 * j + 1] = __float_as_uint(f16_bits_to_f32(hi));
            }
        }
    }
}

// 8 consecutive elements as fp32, from the one (16-bit types) or two (fp32)
// 16-byte words that hold them
template <int XT>
__device__ __forceinline__ void raw_to_f32(const uint4 *u, float (&y)[8]) {
    if (XT == kF32) {
        const uint32_t w[8] = {u[0].x, u[0].y, u[0].z, u[0].w, u[1].x, u[1].y, u[1].z, u[1].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = __uint_as_float(w[j]);
    } else {
        const uint32_t w[4] = {u[0].x, u[0].y, u[0].z, u[0].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            y[2 * j] = lowp_to_f32<XT>(w[j] & 0xFFFFu);
            y[2 * j + 1] = lowp_to_f32<XT>(w[j] >> 16);
        }
    }
}

__device__ __forceinline__ bool tile_fast(const void *x, int64_t rows, int64_t cols, int64_t r0,
                                          int64_t c0) {
    return r0 + kTile <= rows && c0 + kTile <= cols && (cols & 7) == 0 && aligned16(x);
}

__global__ void rowcol_zero_kernel(float *amax_row, int64_t rows, float *amax_col, int64_t cols,
                                   const int32_t *skip_if) {
    pdl_wait();
    pdl_trigger();
    if (skip_if && *skip_if) return;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < rows + cols;
         i += int64_t(gridDim.x) * blockDim.x) {
        if (i < rows) amax_row[i] = 0.0f;
        else if (amax_col) amax_col[i - rows] = 0.0f;
    }
}

// Row and column maxima of |x|.  The grid is S CTAs per 128-column strip:
// CTA b takes strip b mod C (C strips) and, in it, the tile rows b / C,
// b / C + S, b / C + 2S, ...  At step m the CTAs together read tile rows
// [m S, m S + S) of every strip, so the pass sweeps x from top to bottom (the
// cast then walks the tiles in reverse and meets the last reads in L2).  Per
// tile, each thread holds 8 rows x 8 columns.  Row maxima are combined across
// the 16 lanes sharing a row and sent with one atomicMax per row; for 16-bit
// x on packed magnitudes, by a transposing reduction of five shuffles that
// leaves each row in one lane pair.  Column maxima stay in registers for the
// whole strip and are combined through shared memory once, at the end.  The
// next tile's loads are issued before the current tile is reduced.  Tiles on
// a ragged edge, or with sizes/addresses that break 16-byte access, take an
// element path through shared memory.
template <int XT>
__global__ void __launch_bounds__(kThreads) rowcol_amax_kernel(const void *x, int64_t rows,
                                                               int64_t cols, unsigned *amax_row,
                                                               unsigned *amax_col, int per_strip,
                                                               const int32_t *skip_if) {
    pdl_wait();
    pdl_trigger();
    if (skip_if && *skip_if) return;
    __shared__ __align__(16) uint32_t colmax[kThreads / 32][kTile];
    __shared__ uint32_t s_row[kTile], s_col[kTile];
    constexpr int nw = XT == kF32 ? 2 : 1;
    constexpr int esz = XT == kF32 ? 4 : 2;
    const int64_t tiles_r = (rows + kTile - 1) / kTile, tiles_c = (cols + kTile - 1) / kTile;
    const int64_t strip = blockIdx.x % tiles_c, tr0 = blockIdx.x / tiles_c;
    const int c8 = threadIdx.x & 15, rb = threadIdx.x >> 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t cm[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint32_t cm2[4] = {0, 0, 0, 0};  // 16-bit x: packed column maxima of the fast tiles
    uint4 raw[8][nw];
    auto load = [&](int64_t r0, int64_t c0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const char *p = static_cast<const char *>(x) + ((r0 + rb + 16 * k) * cols + c0 + 8 * c8) * esz;
            raw[k][0] = ld16(p);
            if (nw == 2) raw[k][nw - 1] = ld16(p + 16);
        }
    };
    // column maxima gathered in registers for the strip -> one atomicMax per column
    auto flush = [&]() {
        if constexpr (XT != kF32) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                cm[2 * j] = max(cm[2 * j], widen16<XT>(cm2[j] & 0xFFFFu));
                cm[2 * j + 1] = max(cm[2 * j + 1], widen16<XT>(cm2[j] >> 16));
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) cm[j] = max(cm[j], __shfl_xor_sync(0xFFFFFFFFu, cm[j], 16));
        if (lane < 16) {
            uint4 *d = reinterpret_cast<uint4 *>(&colmax[warp][8 * c8]);
            d[0] = make_uint4(cm[0], cm[1], cm[2], cm[3]);
            d[1] = make_uint4(cm[4], cm[5], cm[6], cm[7]);
        }
        __syncthreads();
        if (threadIdx.x < kTile) {
            uint32_t m = 0;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) m = max(m, colmax[w][threadIdx.x]);
            const int64_t c = strip * kTile + threadIdx.x;
            if (amax_col && c < cols && m != 0) atomicMax(amax_col + c, m);
        }
    };
    const int64_t c0 = strip * kTile;
    if (tr0 < tiles_r && tile_fast(x, rows, cols, tr0 * kTile, c0)) load(tr0 * kTile, c0);
    for (int64_t tr = tr0; tr < tiles_r; tr += per_strip) {
        const int64_t r0 = tr * kTile, nr0 = r0 + int64_t(per_strip) * kTile;
        const bool has_next = tr + per_strip < tiles_r;
        if (XT != kF32 && tile_fast(x, rows, cols, r0, c0)) {
            // 16-bit x: packed magnitudes (unsigned order = order of |x|, NaN
            // above inf), widened to fp32 patterns only for the atomics
            uint32_t mg[8][4];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                mg[k][0] = raw[k][0].x & 0x7FFF7FFFu;
                mg[k][1] = raw[k][0].y & 0x7FFF7FFFu;
                mg[k][2] = raw[k][0].z & 0x7FFF7FFFu;
                mg[k][3] = raw[k][0].w & 0x7FFF7FFFu;
            }
            if (has_next && tile_fast(x, rows, cols, nr0, c0)) load(nr0, c0);
            // pk[i]: the maxima of rows rb + 32 i (low half) and rb + 32 i + 16
            uint32_t pk[4], r2[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
#pragma unroll
                for (int j = 0; j < 4; ++j) cm2[j] = __vmaxu2(cm2[j], mg[k][j]);
                r2[k] = __vmaxu2(__vmaxu2(mg[k][0], mg[k][1]), __vmaxu2(mg[k][2], mg[k][3]));
            }
            // rows 2i and 2i + 1: their low halves side by side against their
            // high halves, one packed max
#pragma unroll
            for (int i = 0; i < 4; ++i)
                pk[i] = __vmaxu2(__byte_perm(r2[2 * i], r2[2 * i + 1], 0x5410),
                                 __byte_perm(r2[2 * i], r2[2 * i + 1], 0x7632));
            // transposing reduction over the 16 lanes of the row (c8 bits 3..0):
            // each step hands half of the words to the partner and keeps the
            // other half, so lane c8 ends with pk[2 b3 + b2] over all 16 lanes
            const bool b3 = c8 & 8, b2 = c8 & 4;
            const uint32_t k0 = b3 ? pk[2] : pk[0], k1 = b3 ? pk[3] : pk[1];
            const uint32_t s0 = b3 ? pk[0] : pk[2], s1 = b3 ? pk[1] : pk[3];
            const uint32_t q0 = __vmaxu2(k0, __shfl_xor_sync(0xFFFFFFFFu, s0, 8));
            const uint32_t q1 = __vmaxu2(k1, __shfl_xor_sync(0xFFFFFFFFu, s1, 8));
            uint32_t rr = __vmaxu2(b2 ? q1 : q0, __shfl_xor_sync(0xFFFFFFFFu, b2 ? q0 : q1, 4));
            rr = __vmaxu2(rr, __shfl_xor_sync(0xFFFFFFFFu, rr, 2));
            rr = __vmaxu2(rr, __shfl_xor_sync(0xFFFFFFFFu, rr, 1));
            // lanes with c8 & 3 == 0 / 1 send the low / high row of pk[2 b3 + b2]
            if ((c8 & 2) == 0) {
                const int i = (b3 ? 2 : 0) + (b2 ? 1 : 0);
                const uint32_t h = (c8 & 1) ? (rr >> 16) : (rr & 0xFFFFu);
                const uint32_t v = widen16<XT>(h);
                if (v != 0) atomicMax(amax_row + r0 + rb + 32 * i + 16 * (c8 & 1), v);
            }
        } else if (tile_fast(x, rows, cols, r0, c0)) {
            uint32_t a[8][8];
#pragma unroll
            for (int k = 0; k < 8; ++k) raw_abs<XT>(raw[k], a[k]);
            if (has_next && tile_fast(x, rows, cols, nr0, c0)) load(nr0, c0);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint32_t rm = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    rm = max(rm, a[k][j]);
                    cm[j] = max(cm[j], a[k][j]);
                }
                // the 16 lanes holding this row: lanes 0-15 or 16-31 of the warp
#pragma unroll
                for (int off = 8; off > 0; off >>= 1)
                    rm = max(rm, __shfl_xor_sync(0xFFFFFFFFu, rm, off));
                if (c8 == 0 && rm != 0) atomicMax(amax_row + r0 + rb + 16 * k, rm);
            }
        } else {
            if (threadIdx.x < kTile) s_row[threadIdx.x] = s_col[threadIdx.x] = 0u;
            __syncthreads();
            for (int idx = threadIdx.x; idx < kTile * kTile; idx += kThreads) {
                const int64_t i = r0 + (idx >> 7), j = c0 + (idx & (kTile - 1));
                if (i < rows && j < cols) {
                    const uint32_t v = abs_f32_bits<XT>(x, i * cols + j);
                    atomicMax(&s_row[idx >> 7], v);
                    atomicMax(&s_col[idx & (kTile - 1)], v);
                }
            }
            __syncthreads();
            if (threadIdx.x < kTile) {
                const int u = threadIdx.x;
                if (r0 + u < rows && s_row[u] != 0) atomicMax(amax_row + r0 + u, s_row[u]);
                if (amax_col && c0 + u < cols && s_col[u] != 0) atomicMax(amax_col + c0 + u, s_col[u]);
            }
            __syncthreads();
            if (has_next && tile_fast(x, rows, cols, nr0, c0)) load(nr0, c0);
        }
    }
    flush();
}

__global__ void rowcol_scale_kernel(const float *amax_row, float *scale_row, float *inv_row,
                                    int64_t rows, const float *amax_col, float *scale_col,
                                    float *inv_col, int64_t cols, EpsFloor ef, float fmax,
                                    const int32_t *skip_if) {
    pdl_wait();
    pdl_trigger();
    if (skip_if && *skip_if) return;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < rows + cols;
         i += int64_t(gridDim.x) * blockDim.x) {
        if (i < rows) {
            tensor_scale(amax_row[i], ef, fmax, scale_row[i], inv_row[i]);
        } else if (amax_col) {
            const int64_t j = i - rows;
            tensor_scale(amax_col[j], ef, fmax, scale_col[j], inv_col[j]);
        }
    }
}

template <int XT, int FT>
__global__ void __launch_bounds__(kThreads) rowcol_cast_kernel(const void *x, int64_t rows,
                                                               int64_t cols, uint8_t *out,
                                                               uint8_t *out_t,
                                                               const float *scale_row,
                                                               const float *scale_col,
                                                               const int32_t *skip_if) {
    pdl_wait();
    pdl_trigger();
    if (skip_if && *skip_if) return;
    __shared__ __align__(16) uint32_t sm[kTile * 32];
    // tiles in reverse row-major order: the maxima pass's last reads first
    const int64_t tiles_c = (cols + kTile - 1) / kTile;
    const int64_t tile = int64_t(gridDim.x) - 1 - blockIdx.x;
    const int64_t r0 = (tile / tiles_c) * kTile;
    const int64_t c0 = (tile % tiles_c) * kTile;
    const bool fast = tile_fast(x, rows, cols, r0, c0) &&
                      (reinterpret_cast<uintptr_t>(out) & 7) == 0 &&
                      (out_t == nullptr || ((rows & 15) == 0 && aligned16(out_t)));
    if (fast) {
        const int c8 = threadIdx.x & 15, rb = threadIdx.x >> 4;
        float sc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) sc[j] = out_t ? scale_col[c0 + 8 * c8 + j] : 0.0f;
        // all eight rows' loads in flight before any store (x and out may
        // alias as far as the compiler knows, so it would not hoist them)
        constexpr int nw = XT == kF32 ? 2 : 1;
        uint4 raw[8][nw];
        float srow[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const char *p = static_cast<const char *>(x) +
                            ((r0 + rb + 16 * k) * cols + c0 + 8 * c8) * (XT == kF32 ? 4 : 2);
            raw[k][0] = ld16(p);
            if (nw == 2) raw[k][nw - 1] = ld16(p + 16);
            srow[k] = scale_row[r0 + rb + 16 * k];
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int r = rb + 16 * k;
            const int64_t e = (r0 + r) * cols + c0 + 8 * c8;
            float y[8];
            raw_to_f32<XT>(raw[k], y);
            const float sr = srow[k];
            uint32_t h[4], g[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float a0, a1, b0, b1;
                mul2_rn(y[2 * j], y[2 * j + 1], sr, sr, a0, a1);
                mul2_rn(y[2 * j], y[2 * j + 1], sc[2 * j], sc[2 * j + 1], b0, b1);
                h[j] = f32x2_to_fp8x2_raw<FT>(a0, a1);
                g[j] = f32x2_to_fp8x2_raw<FT>(b0, b1);
            }
            *reinterpret_cast<uint2 *>(out + e) =
                make_uint2(fp8x4_canonical_nan<FT>(h[0] | (h[1] << 16)),
                           fp8x4_canonical_nan<FT>(h[2] | (h[3] << 16)));
            if (out_t)
                *reinterpret_cast<uint2 *>(sm + swz(r, 2 * c8)) =
                    make_uint2(fp8x4_canonical_nan<FT>(g[0] | (g[1] << 16)),
                               fp8x4_canonical_nan<FT>(g[2] | (g[3] << 16)));
        }
        if (out_t) {
            __syncthreads();
            store_transposed_tile(sm, out_t, rows, r0, c0);
        }
    } else {
        for (int idx = threadIdx.x; idx < kTile * kTile; idx += kThreads) {
            const int64_t i = r0 + (idx >> 7), j = c0 + (idx & (kTile - 1));
            if (i < rows && j < cols) {
                const float v = XT == kF32 ? static_cast<const float *>(x)[i * cols + j]
                                           : lowp_to_f32<XT>(static_cast<const uint16_t *>(x)[i * cols + j]);
                out[i * cols + j] = quant1<FT>(v, scale_row[i]);
                if (out_t) out_t[j * rows + i] = quant1<FT>(v, scale_col[j]);
            }
        }
    }
}

template <int XT, int FT>
cudaError_t launch_rowwise_t(const void *x, int64_t rows, int64_t cols, uint8_t *out,
                             uint8_t *out_t, float *amax_row, float *scale_row, float *inv_row,
                             float *amax_col, float *scale_col, float *inv_col, double eps,
                             const int32_t *skip_if, int device, cudaStream_t s) {
    const int64_t n_rc = rows + (out_t ? cols : 0);
    const unsigned small_grid =
        (unsigned)std::max<int64_t>(1, std::min<int64_t>((n_rc + 255) / 256, sm_count(device) * 4));
    float *acol = out_t ? amax_col : nullptr;
    cudaError_t e = launch_pdl(rowcol_zero_kernel, dim3(small_grid), dim3(256), 0, s, amax_row,
                               rows, acol, int64_t(out_t ? cols : 0), skip_if);
    if (e != cudaSuccess) return e;
    const int64_t tiles = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
    if (tiles == 0) return cudaSuccess;
    // as many CTAs as fit on the GPU at once (each walks a run of tiles)
    static std::atomic<int> per_sm{0};
    if (per_sm.load(std::memory_order_relaxed) == 0) {
        int k = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, rowcol_amax_kernel<XT>, kThreads, 0) !=
                cudaSuccess || k < 1)
            k = 1;
        per_sm.store(k, std::memory_order_relaxed);
    }
    // S CTAs per column strip, so that the CTAs resident at once cover all
    // strips (at least one CTA per strip; no more than the strip's tiles)
    const int64_t tiles_r = (rows + kTile - 1) / kTile, tiles_c = (cols + kTile - 1) / kTile;
    const int64_t resident = int64_t(sm_count(device)) * per_sm.load(std::memory_order_relaxed);
    const int64_t per_strip = std::max<int64_t>(1, std::min<int64_t>(tiles_r, resident / tiles_c));
    e = launch_pdl(rowcol_amax_kernel<XT>, dim3((unsigned)(tiles_c * per_strip)), dim3(kThreads),
                   0, s, x, rows, cols, reinterpret_cast<unsigned *>(amax_row),
                   reinterpret_cast<unsigned *>(acol), int(per_strip), skip_if);
    if (e != cudaSuccess) return e;
    e = launch_pdl(rowcol_scale_kernel, dim3(small_grid), dim3(256), 0, s,
                   static_cast<const float *>(amax_row), scale_row, inv_row, rows,
                   static_cast<const float *>(acol), scale_col, inv_col,
                   int64_t(out_t ? cols : 0), make_eps_floor(eps, fp8_max<FT>()), fp8_max<FT>(),
                   skip_if);
    if (e != cudaSuccess) return e;
    return launch_pdl(rowcol_cast_kernel<XT, FT>, dim3((unsigned)tiles), dim3(kThreads), 0, s, x,
                      rows, cols, out, out_t, static_cast<const float *>(scale_row),
                      static_cast<const float *>(scale_col), skip_if);
}

}  // namespace

cudaError_t launch_fp8_quant_rowwise(const void *x, int xelem, int64_t rows, int64_t cols, int fp8,
                                     double eps, uint8_t *out, uint8_t *out_t, float *amax_row,
                                     float *scale_row, float *inv_row, float *amax_col,
                                     float *scale_col, float *inv_col, const int32_t *skip_if,
                                     int device, cudaStream_t s) {
#define AMP_RW(XT, FT)                                                                           \
    return launch_rowwise_t<XT, FT>(x, rows, cols, out, out_t, amax_row, scale_row, inv_row,     \
                                    amax_col, scale_col, inv_col, eps, skip_if, device, s)
    if (fp8 == kE4M3) {
        if (xelem == kBF16) AMP_RW(kBF16, kE4M3);
        if (xelem == kF16) AMP_RW(kF16, kE4M3);
        AMP_RW(kF32, kE4M3);
    }
    if (xelem == kBF16) AMP_RW(kBF16, kE5M2);
    if (xelem == kF16) AMP_RW(kF16, kE5M2);
    AMP_RW(kF32, kE5M2);
#undef AMP_RW
}

}  // namespace amp
