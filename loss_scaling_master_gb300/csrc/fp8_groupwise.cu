// fp8_groupwise.cu - group-wise FP8 scaling in one pass.
//
// "第20章 量化与混合精度训练" §20.5.18: a weight [out, in] is cut into groups
// of G consecutive elements along `in`, each with its own scale (g128: scales
// [out, in / 128]).  Each group follows §2 of "FP8训练：量化、自动微分、
// Torchao" (amax, scale_d = fp8_max / max(double(amax), EPS), clamp, RNE
// cast).  The column-major copy (§4) feeds the backward GEMM, whose reduction
// runs along the rows of x, so its groups are G consecutive rows of a column
// (scales [cols, rows / G]).
//
// With G dividing the 128x128 tile, every group lies inside one tile, so one
// CTA per tile reads x once and finishes everything: group maxima along rows
// (lane shuffles) and along columns (registers, then shared memory), the
// scales, the row-major bytes and the transposed bytes (through a swizzled
// byte tile).  2 bytes read + 1 + 1 written per element, one launch.  The
// tile of x sits in registers (16-bit x, G >= 64) or is staged in shared
// memory with cp.async (fp32 x, G = 32), where the byte tile then reuses the
// staging rows as they are consumed.  With the tile in registers, the lanes of
// a row group form its scales right after the row maxima and cast the
// row-major bytes in the same pass, so only the column scales and the
// transposed bytes wait for the CTA's barriers (and without the copy there
// are none).
//
// Instruction count is what bounds this pass after the loads, so: 16-bit x
// takes its maxima on packed pairs of 16-bit magnitudes, and the fp8 bytes
// skip the NaN canonicalisation in tiles whose scales all lie in (0, inf),
// where no NaN byte can arise.
//
// The scales come from tensor_scale (fp8_tile.cuh): fp32 divisions equal to
// §2's fp64 formula rounded to fp32.
#include <algorithm>
#include <type_traits>

#include "fp8_tile.cuh"
#include "internal.h"
#include "pdl.cuh"

namespace amp {
namespace {

template <int XT>
__device__ __forceinline__ float elem_f32(const void *x, int64_t k) {
    if (XT == kF32) return static_cast<const float *>(x)[k];
    return lowp_to_f32<XT>(static_cast<const uint16_t *>(x)[k]);
}

template <int XT>
__device__ __forceinline__ uint32_t elem_abs_bits(const void *x, int64_t k) {
    return __float_as_uint(elem_f32<XT>(x, k)) & 0x7FFFFFFFu;
}

// 8 consecutive elements held in one (16-bit) or two (fp32) 16-byte words
template <int XT>
__device__ __forceinline__ void words_to_f32(const uint4 *u, float (&y)[8]) {
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

struct GroupOut {
    uint8_t *out, *out_t;
    float *amax_rg, *scale_rg, *inv_rg;  // [rows, ngc]
    float *amax_cg, *scale_cg, *inv_cg;  // [cols, ngr]
};

// shared memory of one CTA besides the staging buffer (which also takes the
// fp8 tile for the transpose, row by row as its x rows are consumed)
template <int G>
struct GroupSmem {
    static constexpr int NG = kTile / G;
    uint32_t colmax[kThreads / 32][NG][kTile];  // per-warp column-group maxima
    uint32_t s_rmax[kTile][NG];                 // row-group maxima (bit patterns)
    float s_rsc[kTile][NG];                     // row-group multipliers
    float s_csc[NG][kTile];                     // column-group multipliers
    int canon;  // some scale of the tile is not in (0, inf): NaN bytes possible
};

// Where the vector path keeps its tile of x: in registers for 16-bit x and
// G >= 64 (measured a few per cent faster), in shared memory for fp32 x (64
// registers of data) and for G = 32, whose four column groups' maxima would
// push the register count to ~90.  The kernel's register cap keeps as many
// CTAs per SM as its shared memory allows: 4 for 16-bit x, 3 for fp32 x.
template <int XT, int G>
constexpr bool kGroupRegs = XT != kF32 && G >= 64;

// Whether a tile takes the vector path: full, 16-byte rows, aligned outputs.
__device__ __forceinline__ bool group_tile_fast(const void *x, int64_t rows, int64_t cols,
                                                int64_t r0, int64_t c0, const GroupOut &o) {
    return r0 + kTile <= rows && c0 + kTile <= cols && (cols & 7) == 0 && aligned16(x) &&
           (reinterpret_cast<uintptr_t>(o.out) & 7) == 0 &&
           (o.out_t == nullptr || ((rows & 15) == 0 && aligned16(o.out_t)));
}

// One 128x128 tile (one CTA): the vector path, or the element path for tiles
// on a ragged edge or with sizes/addresses that break 16-byte access.
template <int XT, int FT, int G>
__device__ __forceinline__ void group_tile(const void *x, int64_t rows, int64_t cols, int64_t r0,
                                           int64_t c0, const GroupOut &o, const EpsFloor &ef,
                                           bool fast, GroupSmem<G> &S, uint4 *stage) {
    constexpr int NG = kTile / G;  // groups per tile edge
    constexpr int nw = XT == kF32 ? 2 : 1;
    // With kGroupRegs, x stays in registers (8 x 16 B a thread) and `stage`
    // holds only the 16 KB fp8 tile for the transpose.  Otherwise x is staged
    // in shared memory: row r fills stage bytes [r * 256 nw, (r + 1) * 256 nw),
    // and its 128 fp8 bytes for the transpose go to the start of that span
    // once it is read.
    constexpr bool kRegs = kGroupRegs<XT, G>;
    constexpr int kRowWords = kRegs ? 32 : 64 * nw;
    uint32_t *sm = reinterpret_cast<uint32_t *>(stage);
    auto &colmax = S.colmax;
    auto &s_rmax = S.s_rmax;
    auto &s_rsc = S.s_rsc;
    auto &s_csc = S.s_csc;
    const float fmax = fp8_max<FT>();
    const int64_t ngc = (cols + G - 1) / G, ngr = (rows + G - 1) / G;
    const int64_t gc0 = c0 / G, gr0 = r0 / G;  // first group of this tile in each direction
    uint8_t *out = o.out, *out_t = o.out_t;
    if (fast) {
        constexpr int esz = XT == kF32 ? 4 : 2;
        const int c8 = threadIdx.x & 15, rb = threadIdx.x >> 4;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        uint4 xr[kRegs ? 8 : 1];
        if constexpr (kRegs) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                xr[k] = ld16(static_cast<const char *>(x) +
                             ((r0 + rb + 16 * k) * cols + c0 + 8 * c8) * esz);
        } else {
            // the tile goes to this thread's own staging slots with
            // asynchronous copies, so no registers are held while the loads
            // are in flight and the cast pass reads the data again
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const char *p =
                    static_cast<const char *>(x) + ((r0 + rb + 16 * k) * cols + c0 + 8 * c8) * esz;
#pragma unroll
                for (int u = 0; u < nw; ++u) {
                    const uint32_t d = static_cast<uint32_t>(
                        __cvta_generic_to_shared(stage + (k * kThreads + threadIdx.x) * nw + u));
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d),
                                 "l"(p + 16 * u)
                                 : "memory");
                }
            }
            asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        }
        auto raw = [&](int k) -> const uint4 * {
            if constexpr (kRegs) return &xr[k];
            else return stage + (k * kThreads + threadIdx.x) * nw;
        };
        if (threadIdx.x == 0) S.canon = 0;
        if constexpr (XT == kF32) {
            // |x| bit patterns (an unsigned max of them is the NaN-propagating
            // fp32 max); colg[q][j]: column 8 c8 + j over this thread's rows of
            // group q
            uint32_t colg[NG][8];
#pragma unroll
            for (int q = 0; q < NG; ++q)
#pragma unroll
                for (int j = 0; j < 8; ++j) colg[q][j] = 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float y[8];
                words_to_f32<XT>(raw(k), y);
                uint32_t rm = 0;
                const int q = (16 * k) / G;  // column group of row rb + 16k (rb < 16 <= G)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t a = __float_as_uint(y[j]) & 0x7FFFFFFFu;
                    rm = max(rm, a);
                    colg[q][j] = max(colg[q][j], a);
                }
                // the G / 8 lanes holding this row's group of G columns
#pragma unroll
                for (int off = G / 16; off > 0; off >>= 1)
                    rm = max(rm, __shfl_xor_sync(0xFFFFFFFFu, rm, off));
                if ((c8 & (G / 8 - 1)) == 0) s_rmax[rb + 16 * k][(8 * c8) / G] = rm;
            }
            if (out_t) {
                // lanes l and l ^ 16 hold the same columns (row groups 2w, 2w + 1)
#pragma unroll
                for (int q = 0; q < NG; ++q)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        colg[q][j] = max(colg[q][j], __shfl_xor_sync(0xFFFFFFFFu, colg[q][j], 16));
                if (lane < 16) {
#pragma unroll
                    for (int q = 0; q < NG; ++q) {
                        uint4 *d = reinterpret_cast<uint4 *>(&colmax[warp][q][8 * c8]);
                        d[0] = make_uint4(colg[q][0], colg[q][1], colg[q][2], colg[q][3]);
                        d[1] = make_uint4(colg[q][4], colg[q][5], colg[q][6], colg[q][7]);
                    }
                }
            }
        } else {
            // 16-bit x: |x| as 16-bit patterns, whose unsigned order is the
            // order of magnitudes (NaN above inf), so the maxima are taken on
            // packed pairs and widened to fp32 bit patterns at the end.
            // colg[q][j]: columns 8 c8 + 2j, 8 c8 + 2j + 1 over this thread's
            // rows of group q; rpair[i]: rows rb + 32i and rb + 32i + 16.
            auto widen = [](uint32_t h) {
                return __float_as_uint(lowp_to_f32<XT>(h & 0xFFFFu)) & 0x7FFFFFFFu;
            };
            uint32_t colg[NG][4], rpair[4], m2[8];
#pragma unroll
            for (int q = 0; q < NG; ++q)
#pragma unroll
                for (int j = 0; j < 4; ++j) colg[q][j] = 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint4 u = *raw(k);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                const int q = (16 * k) / G;
                m2[k] = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t a = w[j] & 0x7FFF7FFFu;
                    m2[k] = max_u16x2(m2[k], a);
                    colg[q][j] = max_u16x2(colg[q][j], a);
                }
            }
            // rows k = 2i, 2i + 1: low halves side by side against high halves
#pragma unroll
            for (int i = 0; i < 4; ++i)
                rpair[i] = max_u16x2(__byte_perm(m2[2 * i], m2[2 * i + 1], 0x5410),
                                     __byte_perm(m2[2 * i], m2[2 * i + 1], 0x7632));
            // rrow: G >= 64, after a transposing reduction over the G / 8 lanes
            // of the row group, lane gl = c8 mod (G / 8) holds (in the half gl
            // & 1) the maximum of row rb + 16 (gl mod 8): the words are halved
            // between partners on lane bits 2 and 1, then reduced whole over
            // the remaining bits.  G = 32 reduces every word over its 4 lanes.
            uint32_t rrow = 0;
            if constexpr (G >= 64) {
                const bool b2 = c8 & 4, b1 = c8 & 2;
                const uint32_t q0 = max_u16x2(b2 ? rpair[2] : rpair[0],
                                              __shfl_xor_sync(0xFFFFFFFFu, b2 ? rpair[0] : rpair[2], 4));
                const uint32_t q1 = max_u16x2(b2 ? rpair[3] : rpair[1],
                                              __shfl_xor_sync(0xFFFFFFFFu, b2 ? rpair[1] : rpair[3], 4));
                rrow = max_u16x2(b1 ? q1 : q0, __shfl_xor_sync(0xFFFFFFFFu, b1 ? q0 : q1, 2));
                rrow = max_u16x2(rrow, __shfl_xor_sync(0xFFFFFFFFu, rrow, 1));
                if (G == 128) rrow = max_u16x2(rrow, __shfl_xor_sync(0xFFFFFFFFu, rrow, 8));
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
#pragma unroll
                    for (int off = G / 16; off > 0; off >>= 1)
                        rpair[i] = max_u16x2(rpair[i], __shfl_xor_sync(0xFFFFFFFFu, rpair[i], off));
                    if ((c8 & (G / 8 - 1)) == 0) {
                        s_rmax[rb + 32 * i][(8 * c8) / G] = widen(rpair[i]);
                        s_rmax[rb + 32 * i + 16][(8 * c8) / G] = widen(rpair[i] >> 16);
                    }
                }
            }
            if constexpr (!kRegs && G >= 64) {
                const int gl = c8 & (G / 8 - 1);
                if (gl < 8) s_rmax[rb + 16 * gl][(8 * c8) / G] = widen((gl & 1) ? rrow >> 16 : rrow);
            }
            if constexpr (kRegs) {
                // Every lane of a row group now holds the maxima of its 8 rows.
                // Lane gl < 8 of the group forms the scale of row rb + 16 gl
                // and writes that row group's outputs; the row-major bytes are
                // cast here, each row's multiplier taken from its lane.
                const int gl = c8 & (G / 8 - 1);
                const int base = lane & ~(G / 8 - 1);
                float s32 = 0.0f;
                bool odd = false;
                if (gl < 8) {
                    const float a = __uint_as_float(widen((gl & 1) ? rrow >> 16 : rrow));
                    float inv;
                    tensor_scale(a, ef, fmax, s32, inv);
                    odd = !scale_keeps_finite(s32);
                    const int64_t k = (r0 + rb + 16 * gl) * ngc + gc0 + (8 * c8) / G;
                    o.amax_rg[k] = a;
                    o.scale_rg[k] = s32;
                    o.inv_rg[k] = inv;
                }
                // NaN bytes need a scale outside (0, inf): warps whose rows have
                // none skip the canonicalisation (a branch uniform over the warp)
                auto cast_rows = [&](auto canon_tag) {
                    constexpr bool kCanon = decltype(canon_tag)::value;
                    auto fix = [](uint32_t v) { return kCanon ? fp8x4_canonical_nan<FT>(v) : v; };
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float sr = __shfl_sync(0xFFFFFFFFu, s32, base + k);
                        float y[8];
                        words_to_f32<XT>(raw(k), y);
                        uint32_t h[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float a0, a1;
                            mul2_rn(y[2 * j], y[2 * j + 1], sr, sr, a0, a1);
                            h[j] = f32x2_to_fp8x2_raw<FT>(a0, a1);
                        }
                        *reinterpret_cast<uint2 *>(out + (r0 + rb + 16 * k) * cols + c0 + 8 * c8) =
                            make_uint2(fix(h[0] | (h[1] << 16)), fix(h[2] | (h[3] << 16)));
                    }
                };
                if (__any_sync(0xFFFFFFFFu, odd))
                    cast_rows(std::true_type{});
                else
                    cast_rows(std::false_type{});
            }
            if (out_t) {
#pragma unroll
                for (int q = 0; q < NG; ++q)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        colg[q][j] = max_u16x2(colg[q][j], __shfl_xor_sync(0xFFFFFFFFu, colg[q][j], 16));
                if (lane < 16) {
#pragma unroll
                    for (int q = 0; q < NG; ++q) {
                        uint4 *d = reinterpret_cast<uint4 *>(&colmax[warp][q][8 * c8]);
                        d[0] = make_uint4(widen(colg[q][0]), widen(colg[q][0] >> 16),
                                          widen(colg[q][1]), widen(colg[q][1] >> 16));
                        d[1] = make_uint4(widen(colg[q][2]), widen(colg[q][2] >> 16),
                                          widen(colg[q][3]), widen(colg[q][3] >> 16));
                    }
                }
            }
        }
        if (kRegs && out_t == nullptr) return;  // the row-major bytes are done
        __syncthreads();
        // scales: 128 x NG row groups (staged path; the register path formed
        // them in pass 1), and (with the copy) NG x 128 column groups
        if constexpr (!kRegs) {
            for (int idx = threadIdx.x; idx < kTile * NG; idx += kThreads) {
                const int r = idx / NG, q = idx % NG;
                const float a = __uint_as_float(s_rmax[r][q]);
                float s32, inv;
                tensor_scale(a, ef, fmax, s32, inv);
                if (!scale_keeps_finite(s32)) S.canon = 1;
                s_rsc[r][q] = s32;
                const int64_t k = (r0 + r) * ngc + gc0 + q;
                o.amax_rg[k] = a;
                o.scale_rg[k] = s32;
                o.inv_rg[k] = inv;
            }
        }
        if (out_t) {
            for (int idx = threadIdx.x; idx < kTile * NG; idx += kThreads) {
                const int q = idx / kTile, c = idx % kTile;
                uint32_t m = 0;
#pragma unroll
                for (int w = 0; w < kThreads / 32; ++w) m = max(m, colmax[w][q][c]);
                const float a = __uint_as_float(m);
                float s32, inv;
                tensor_scale(a, ef, fmax, s32, inv);
                if (!scale_keeps_finite(s32)) S.canon = 1;
                s_csc[q][c] = s32;
                const int64_t k = (c0 + c) * ngr + gr0 + q;
                o.amax_cg[k] = a;
                o.scale_cg[k] = s32;
                o.inv_cg[k] = inv;
            }
        }
        __syncthreads();
        [[maybe_unused]] const int qc = (8 * c8) / G;  // this thread's row group
        // the column multipliers of this thread's 8 columns, per column group
        float csc[NG][8];
        if (out_t) {
#pragma unroll
            for (int q = 0; q < NG; ++q) {
                const float4 a = *reinterpret_cast<const float4 *>(&s_csc[q][8 * c8]);
                const float4 b = *reinterpret_cast<const float4 *>(&s_csc[q][8 * c8 + 4]);
                csc[q][0] = a.x; csc[q][1] = a.y; csc[q][2] = a.z; csc[q][3] = a.w;
                csc[q][4] = b.x; csc[q][5] = b.y; csc[q][6] = b.z; csc[q][7] = b.w;
            }
        }
        // NaN bytes can only come from a scale outside (0, inf): tiles without
        // one skip the canonicalisation (a branch uniform over the CTA)
        auto cast_pass = [&](auto canon_tag) {
            constexpr bool kCanon = decltype(canon_tag)::value;
            auto fix = [](uint32_t v) { return kCanon ? fp8x4_canonical_nan<FT>(v) : v; };
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int r = rb + 16 * k;
                float y[8];
                words_to_f32<XT>(raw(k), y);
                // row r is read by this half-warp alone (lanes with this rb), in
                // this iteration: once all 16 have it, its span takes the fp8 bytes
                __syncwarp();
                if constexpr (!kRegs) {
                    const float sr = s_rsc[r][qc];
                    uint32_t h[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float a0, a1;
                        mul2_rn(y[2 * j], y[2 * j + 1], sr, sr, a0, a1);
                        h[j] = f32x2_to_fp8x2_raw<FT>(a0, a1);
                    }
                    *reinterpret_cast<uint2 *>(out + (r0 + r) * cols + c0 + 8 * c8) =
                        make_uint2(fix(h[0] | (h[1] << 16)), fix(h[2] | (h[3] << 16)));
                }
                if (out_t) {
                    const int q = (16 * k) / G;
                    uint32_t g[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float b0, b1;
                        mul2_rn(y[2 * j], y[2 * j + 1], csc[q][2 * j], csc[q][2 * j + 1], b0, b1);
                        g[j] = f32x2_to_fp8x2_raw<FT>(b0, b1);
                    }
                    *reinterpret_cast<uint2 *>(sm + swz<kRowWords>(r, 2 * c8)) =
                        make_uint2(fix(g[0] | (g[1] << 16)), fix(g[2] | (g[3] << 16)));
                }
            }
        };
        if (S.canon)
            cast_pass(std::true_type{});
        else
            cast_pass(std::false_type{});
        if (out_t) {
            __syncthreads();
            store_transposed_tile<kRowWords>(sm, out_t, rows, r0, c0);
        }
    } else {
        // element path (ragged edge, or sizes/addresses that break 16-byte
        // access): group maxima through shared-memory atomics, then the cast
        uint32_t(&rmax)[kTile][NG] = s_rmax;
        uint32_t *cmax = &colmax[0][0][0];  // [NG][kTile]
        for (int i = threadIdx.x; i < kTile * NG; i += kThreads) {
            (&rmax[0][0])[i] = 0u;
            cmax[i] = 0u;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < kTile * kTile; idx += kThreads) {
            const int ri = idx >> 7, cj = idx & (kTile - 1);
            const int64_t i = r0 + ri, j = c0 + cj;
            if (i < rows && j < cols) {
                const uint32_t v = elem_abs_bits<XT>(x, i * cols + j);
                atomicMax(&rmax[ri][cj / G], v);
                atomicMax(&cmax[(ri / G) * kTile + cj], v);
            }
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < kTile * NG; idx += kThreads) {
            const int r = idx / NG, q = idx % NG;
            if (r0 + r < rows && c0 + q * G < cols) {
                const float a = __uint_as_float(rmax[r][q]);
                float s32, inv;
                tensor_scale(a, ef, fmax, s32, inv);
                s_rsc[r][q] = s32;
                const int64_t k = (r0 + r) * ngc + gc0 + q;
                o.amax_rg[k] = a;
                o.scale_rg[k] = s32;
                o.inv_rg[k] = inv;
            }
            const int q2 = idx / kTile, c = idx % kTile;
            if (out_t && c0 + c < cols && r0 + q2 * G < rows) {
                const float a = __uint_as_float(cmax[q2 * kTile + c]);
                float s32, inv;
                tensor_scale(a, ef, fmax, s32, inv);
                s_csc[q2][c] = s32;
                const int64_t k = (c0 + c) * ngr + gr0 + q2;
                o.amax_cg[k] = a;
                o.scale_cg[k] = s32;
                o.inv_cg[k] = inv;
            }
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < kTile * kTile; idx += kThreads) {
            const int ri = idx >> 7, cj = idx & (kTile - 1);
            const int64_t i = r0 + ri, j = c0 + cj;
            if (i < rows && j < cols) {
                const float v = elem_f32<XT>(x, i * cols + j);
                out[i * cols + j] = quant1<FT>(v, s_rsc[ri][cj / G]);
                if (out_t) out_t[j * rows + i] = quant1<FT>(v, s_csc[ri / G][cj]);
            }
        }
    }
}

template <int XT, int FT, int G>
__device__ __forceinline__ void groupwise_body(const void *x, int64_t rows, int64_t cols,
                                               const GroupOut &o, const EpsFloor &ef,
                                               const int32_t *skip_if) {
    pdl_wait();
    pdl_trigger();
    if (skip_if && *skip_if) return;
    __shared__ __align__(16) GroupSmem<G> S;
    extern __shared__ __align__(16) uint4 stage[];  // the tile of x, or the fp8 tile
    const int64_t tiles_c = (cols + kTile - 1) / kTile;
    const int64_t r0 = int64_t(blockIdx.x / tiles_c) * kTile;
    const int64_t c0 = int64_t(blockIdx.x % tiles_c) * kTile;
    group_tile<XT, FT, G>(x, rows, cols, r0, c0, o, ef,
                          group_tile_fast(x, rows, cols, r0, c0, o), S, stage);
}

// Tiles held in registers: capped at 64 registers, so 4 CTAs share an SM.
template <int XT, int FT, int G>
__global__ void __launch_bounds__(kThreads, 4) groupwise_kernel(const void *x, int64_t rows,
                                                                int64_t cols, GroupOut o,
                                                                EpsFloor ef,
                                                                const int32_t *skip_if) {
    groupwise_body<XT, FT, G>(x, rows, cols, o, ef, skip_if);
}

// Tiles staged in shared memory (fp32 x, G = 32): the compiler's own choice.
template <int XT, int FT, int G>
__global__ void __launch_bounds__(kThreads) groupwise_staged_kernel(const void *x, int64_t rows,
                                                                    int64_t cols, GroupOut o,
                                                                    EpsFloor ef,
                                                                    const int32_t *skip_if) {
    groupwise_body<XT, FT, G>(x, rows, cols, o, ef, skip_if);
}

template <int XT, int FT, int G>
cudaError_t launch_group_t(const void *x, int64_t rows, int64_t cols, const GroupOut &o,
                           double eps, const int32_t *skip_if, cudaStream_t s) {
    const int64_t tiles = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
    if (tiles == 0) return cudaSuccess;
    const EpsFloor ef = make_eps_floor(eps, fp8_max<FT>());
    auto launch = [&](auto kern, int smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(kern, dim3((unsigned)tiles), dim3(kThreads), smem, s, x, rows, cols, o,
                          ef, skip_if);
    };
    if constexpr (kGroupRegs<XT, G>)
        return launch(groupwise_kernel<XT, FT, G>, kTile * kTile);  // the fp8 tile only
    else
        return launch(groupwise_staged_kernel<XT, FT, G>, kTile * kTile * (XT == kF32 ? 4 : 2));
}

template <int XT, int FT>
cudaError_t launch_group_g(int64_t group, const void *x, int64_t rows, int64_t cols,
                           const GroupOut &o, double eps, const int32_t *skip_if, cudaStream_t s) {
    if (group == 32) return launch_group_t<XT, FT, 32>(x, rows, cols, o, eps, skip_if, s);
    if (group == 64) return launch_group_t<XT, FT, 64>(x, rows, cols, o, eps, skip_if, s);
    return launch_group_t<XT, FT, 128>(x, rows, cols, o, eps, skip_if, s);
}

}  // namespace

cudaError_t launch_fp8_quant_groupwise(const void *x, int xelem, int64_t rows, int64_t cols,
                                       int64_t group, int fp8, double eps, uint8_t *out,
                                       uint8_t *out_t, float *amax_rg, float *scale_rg,
                                       float *inv_rg, float *amax_cg, float *scale_cg,
                                       float *inv_cg, const int32_t *skip_if, cudaStream_t s) {
    GroupOut o{out, out_t, amax_rg, scale_rg, inv_rg, amax_cg, scale_cg, inv_cg};
#define AMP_GW(XT, FT) launch_group_g<XT, FT>(group, x, rows, cols, o, eps, skip_if, s)
    if (fp8 == kE4M3) {
        if (xelem == kBF16) return AMP_GW(kBF16, kE4M3);
        if (xelem == kF16) return AMP_GW(kF16, kE4M3);
        return AMP_GW(kF32, kE4M3);
    }
    if (xelem == kBF16) return AMP_GW(kBF16, kE5M2);
    if (xelem == kF16) return AMP_GW(kF16, kE5M2);
    return AMP_GW(kF32, kE5M2);
#undef AMP_GW
}

}  // namespace amp
