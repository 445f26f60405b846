// fp8_tile.cuh - pieces of the tensorwise FP8 cast shared by the standalone
// quantizer and the fused AdamW + FP8 step ("FP8训练：量化、自动微分、Torchao"
// §2 scale and cast, §4 column-major copy).
#pragma once

#include <cmath>

#include "common.cuh"

namespace amp {

// §2's scale: scale_d = fp8_max / max(double(amax), eps) in fp64, NaN
// propagating; the cast uses scale_d rounded to fp32 and inv_scale is
// 1 / scale_d rounded to fp32.  Both are formed with IEEE fp32 divisions,
// which give the same values:
//   - for amax >= eps, fp8_max / amax rounded to fp64 and then to fp32 equals
//     the correctly rounded fp32 quotient (double rounding is innocuous for
//     division when the wider format has at least 2p + 2 bits: 53 >= 50);
//   - 1 / scale_d rounded to fp32 equals amax / fp8_max correctly rounded:
//     fp8_max = 7 * 2^k, so amax / fp8_max lies at least 1/14 ulp from any
//     fp32 rounding boundary, far beyond the two fp64 rounding errors;
//   - amax = inf gives 0 and inf, NaN gives NaN (a NaN's payload is open).
// The EPS floor (amax < eps) takes two constants formed once on the host in
// fp64, so no fp64 arithmetic runs on the device.
struct EpsFloor {
    float eps32;   // the smallest fp32 value not below eps: amax < eps32 <=> double(amax) < eps
    float s_eps;   // float(fp8_max / eps)
    float inv_eps; // float(1 / (fp8_max / eps))
};

inline EpsFloor make_eps_floor(double eps, float fmax) {
    EpsFloor e;
    e.eps32 = float(eps);
    if (double(e.eps32) < eps) e.eps32 = std::nextafter(e.eps32, INFINITY);
    const double sd = double(fmax) / eps;
    e.s_eps = float(sd);
    e.inv_eps = float(1.0 / sd);
    return e;
}

__device__ __forceinline__ void tensor_scale(float amax, const EpsFloor &e, float fmax, float &s32,
                                             float &inv) {
    if (amax < e.eps32) {
        s32 = e.s_eps;
        inv = e.inv_eps;
    } else {
        s32 = __fdiv_rn(fmax, amax);
        inv = __fdiv_rn(amax, fmax);
    }
}

// Whether every product x * s32 of the elements that s32 was formed from is a
// number: true when 0 < s32 < inf.  Then no element of the group is NaN or
// infinite (a NaN amax gives a NaN scale, an infinite one the scale 0), and a
// finite x times a finite positive s32 saturates instead of turning NaN, so
// the raw conversion yields no NaN byte and needs no canonicalisation.
__device__ __forceinline__ bool scale_keeps_finite(float s32) {
    return s32 > 0.0f && s32 < __int_as_float(0x7F800000);
}

template <int FT>
__device__ __forceinline__ uint8_t quant1(float x, float s32) {
    return uint8_t(f32x2_to_fp8x2<FT>(__fmul_rn(x, s32), 0.0f) & 0xFFu);
}

// Eight bf16 values (a 16-byte word group) -> eight fp8 bytes of x * s32.
template <int FT>
__device__ __forceinline__ uint2 bf16x8_to_fp8x8(const uint4 &b, float s32) {
    const uint32_t w[4] = {b.x, b.y, b.z, b.w};
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float lo, hi;
        mul2_rn(bf16_bits_to_f32(w[j] & 0xFFFFu), bf16_bits_to_f32(w[j] >> 16), s32, s32, lo, hi);
        h[j] = f32x2_to_fp8x2_raw<FT>(lo, hi);
    }
    return make_uint2(fp8x4_canonical_nan<FT>(h[0] | (h[1] << 16)),
                      fp8x4_canonical_nan<FT>(h[2] | (h[3] << 16)));
}

// 4-byte word (row r, word w) of a 128x128 byte tile in shared memory,
// XOR-swizzled by 16-row band so the transposed read hits 32 distinct banks.
// RowWords is the row pitch in words: 32 for a dense tile, more when the tile
// sits in a wider buffer (any multiple of 32 keeps the banks distinct).
template <int RowWords = 32>
__device__ __forceinline__ int swz(int r, int w) {
    static_assert(RowWords % 32 == 0, "row pitch must be a multiple of the 32 banks");
    return r * RowWords + (w ^ (((r >> 4) & 7) << 2));
}

// Write the transposed copy of a full 128x128 byte tile held in `sm` (filled
// through swz) to out_t, which is [cols, rows] row-major: tile element
// (i, j) goes to out_t[(c0 + j) * rows + r0 + i].  256 threads; each reads 16
// words of one word-column (conflict-free), transposes 4x4 byte blocks with
// byte permutes and writes four 16-byte stores; 8 lanes cover one 128-byte
// segment of a transposed row.  Requires rows % 16 == 0 and a 16-byte aligned
// out_t.  RowWords: the row pitch the tile was written with (swz<RowWords>).
template <int RowWords = 32>
__device__ __forceinline__ void store_transposed_tile(const uint32_t *sm, uint8_t *out_t,
                                                      int64_t rows, int64_t r0, int64_t c0) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rg = lane & 7, wq = (lane >> 3) + 4 * warp;
    uint32_t wv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) wv[i] = sm[swz<RowWords>(16 * rg + i, wq)];
    uint32_t col[4][4];  // col[j][blk]: rows 4blk..4blk+3 of column 4wq+j
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
        const uint32_t a = wv[4 * blk], b = wv[4 * blk + 1], c = wv[4 * blk + 2],
                       d = wv[4 * blk + 3];
        const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(a, b, 0x7362);
        const uint32_t t2 = __byte_perm(c, d, 0x5140), t3 = __byte_perm(c, d, 0x7362);
        col[0][blk] = __byte_perm(t0, t2, 0x5410);
        col[1][blk] = __byte_perm(t0, t2, 0x7632);
        col[2][blk] = __byte_perm(t1, t3, 0x5410);
        col[3][blk] = __byte_perm(t1, t3, 0x7632);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t dst = (c0 + 4 * wq + j) * rows + r0 + 16 * rg;
        st16(out_t + dst, make_uint4(col[j][0], col[j][1], col[j][2], col[j][3]));
    }
}

}  // namespace amp
