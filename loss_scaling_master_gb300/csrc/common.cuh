// common.cuh - device-side building blocks shared by the libampfp8 kernels:
// list views, vector memory access, exact format conversions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace amp {

// Elements per chunk of a 1-D tensor list.  One CTA walks one chunk.
constexpr int kChunk = 16384;
// Threads per CTA of the streaming list kernels.
constexpr int kThreads = 256;
// Square tile edge of the FP8 quantization kernels (bytes of fp8 output).
constexpr int kTile = 128;

// Device view of a tensor list handle (all arrays live in the handle's
// device block).  chunks[c] = {tensor, chunk index within the tensor};
// tiles[k] = {tensor, tile index within the tensor, row-major over tiles}.
struct ListView {
    void *const *ptrs;
    const int64_t *numel;
    const int64_t *rows;
    const int64_t *cols;
    const int32_t *slots;
    const uint2 *chunks;
    const uint2 *tiles;
    double *partials;  // one fp64 slot per chunk (scratch of the norm pass)
    int n;
};

enum ElemType : int { kF32 = 0, kF16 = 1, kBF16 = 2 };
enum Fp8Type : int { kE4M3 = 0, kE5M2 = 1 };

// Canonical positive NaN codes written by the encoders.
constexpr uint16_t kBf16NaN = 0x7FC0u;
constexpr uint16_t kF16NaN = 0x7E00u;
constexpr uint8_t kE4M3NaN = 0x7Fu;
constexpr uint8_t kE5M2NaN = 0x7Eu;

__device__ __forceinline__ bool aligned16(const void *p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// 16-byte global loads/stores with the default cache policy.  (Evict-first
// hints on the streams measured 1.4 % slower for the AdamW pass on GB300: the
// read/write mix at the DRAM controller, not L2 capacity, is what limits it.)
__device__ __forceinline__ uint4 ld16(const void *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ void st16(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

// ---- exact widening conversions -----------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) {
    return __uint_as_float(b << 16);
}
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
    float f;
    asm("{ .reg .b16 t; mov.b16 t, %1; cvt.f32.f16 %0, t; }" : "=f"(f) : "h"((unsigned short)h));
    return f;
}
template <int ET>
__device__ __forceinline__ float lowp_to_f32(uint32_t bits) {
    return ET == kBF16 ? bf16_bits_to_f32(bits) : f16_bits_to_f32(bits);
}

// ---- round-to-nearest-even narrowing conversions ------------------------
// Two fp32 -> packed bf16x2 (lo in bits 0..15), NaN -> canonical 0x7FC0.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    if (lo != lo) r = (r & 0xFFFF0000u) | kBf16NaN;
    if (hi != hi) r = (r & 0x0000FFFFu) | (uint32_t(kBf16NaN) << 16);
    return r;
}
__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
    return (uint16_t)(f32x2_to_bf16x2(x, 0.0f) & 0xFFFFu);
}
__device__ __forceinline__ uint16_t f32_to_f16(float x) {
    unsigned short h;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return x != x ? kF16NaN : (uint16_t)h;
}

// Two fp32 -> packed fp8x2 (lo in bits 0..7), round-to-nearest-even with
// saturation to the largest finite value (the same bytes as clamping to
// +-fp8_max first), NaN -> canonical code.
// Two fp32 -> two fp8 bytes (lo in bits 0-7, hi in bits 8-15), round to
// nearest even with saturation to the largest finite value; NaN bytes are
// whatever the conversion gives (see fp8x4_canonical_nan).
template <int FT>
__device__ __forceinline__ uint32_t f32x2_to_fp8x2_raw(float lo, float hi) {
    unsigned short r;
    if (FT == kE4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Every NaN byte of four fp8 bytes -> the positive canonical NaN (e4m3fn 0x7F,
// e5m2 0x7E).  With saturation, finite and infinite inputs never convert to a
// NaN pattern (the largest outputs are e4m3fn 0x7E and e5m2 0x7B), so the
// NaN bytes are exactly those of NaN inputs.
template <int FT>
__device__ __forceinline__ uint32_t fp8x4_canonical_nan(uint32_t v) {
    if (FT == kE4M3) {
        const uint32_t m = __vcmpeq4(v | 0x80808080u, 0xFFFFFFFFu);  // bytes S.1111.111
        return v & ~(m & 0x80808080u);
    }
    const uint32_t m = __vcmpgtu4(v & 0x7F7F7F7Fu, 0x7C7C7C7Cu);  // bytes S.11111.xx, xx != 0
    return (v & ~m) | (kE5M2NaN * 0x01010101u & m);
}

template <int FT>
__device__ __forceinline__ uint32_t f32x2_to_fp8x2(float lo, float hi) {
    return fp8x4_canonical_nan<FT>(f32x2_to_fp8x2_raw<FT>(lo, hi));
}

// Lane-wise unsigned maximum of two pairs of 16-bit values.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// (a0 * b0, a1 * b1), each lane an IEEE fp32 multiply rounded to nearest even,
// as one packed instruction.
__device__ __forceinline__ void mul2_rn(float a0, float a1, float b0, float b1, float &o0,
                                        float &o1) {
    asm("{\n\t.reg .b64 pa, pb, pc;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pc, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pc;\n\t}"
        : "=f"(o0), "=f"(o1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

template <int FT>
__host__ __device__ constexpr float fp8_max() {
    return FT == kE4M3 ? 448.0f : 57344.0f;
}

// Warp-wide unsigned max.
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
    return __reduce_max_sync(0xFFFFFFFFu, v);
}

}  // namespace amp
