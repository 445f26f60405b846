// adamw_master.cu - A2..A6: skip-on-inf, unscale, FP32-master AdamW, BF16
// working-copy emission and the per-tensor amax fold for FP8 weights.
//
//   "第20章 量化与混合精度训练" §20.5.13 Master Weights and "从 AMP 到 Mixed
//   Precision" sections "为什么需要 FP32 Master Weights" / "PyTorch AMP 与 FP32
//   Master Weights" (mode B): the optimizer updates an fp32 master and casts
//   it to the bf16 copy the forward pass uses; "06 · 混合精度" §三: master,
//   m and v are fp32, 12 bytes per parameter.
//
// Two launches per step:
//   prologue  one thread: reads found_inf and the step counter, forms the
//             bias-corrected scalars in fp64 once, advances the counter when
//             the step is not skipped, and leaves {skip, step_size, c2} in a
//             block of the master list's device block;
//   main      adamw_bulk_kernel, one CTA per chunk of 16384 elements; a
//             skipped step returns at once, otherwise the chunk streams
//             through shared memory with TMA bulk copies: 14 bytes read + 14
//             bytes written per parameter (fp16/bf16 grads, bf16 emission).
// The delayed-FP8 form adds adamw_fp8_tile_kernel, which updates the FP8
// weights by 128x128 tile and casts them in the same pass.
#include "bulk_copy.cuh"
#include "fp8_tile.cuh"
#include "internal.h"
#include "pdl.cuh"
#include "philox.cuh"

namespace amp {
namespace {

struct AdamwParams {
    ListView p, m, v, g, b;
    const float *scale;
    const AdamwStepScalars *scal;
    float *amax;
    float decay, b1, omb1, b2, omb2, eps;
    int use_slots;
    uint64_t sr_seed;  // stochastic bf16 rounding key
    int32_t *err;      // sticky error word (a bounded wait gave up)
};

struct Scal {
    float r, clip, decay, b1, omb1, b2, omb2, eps, step_size, c2;
};

// One element of the update; each operation rounded on its own (no fma).
// g = (float(grad) * (1/S)) * clip, where clip is exactly 1.0 unless the
// gradients are being norm-clipped (x * 1.0f == x, so that path is unchanged).
__device__ __forceinline__ void adamw_elem(float &p, float &m, float &v, float graw,
                                           const Scal &s) {
    const float g = __fmul_rn(__fmul_rn(graw, s.r), s.clip);
    p = __fmul_rn(p, s.decay);
    m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
    v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
    const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.c2), s.eps);
    p = __fsub_rn(p, __fmul_rn(s.step_size, __fdiv_rn(m, denom)));
}

template <int GT>
__device__ __forceinline__ float grad_at(const void *gp, int64_t k) {
    if (GT == kF32) return static_cast<const float *>(gp)[k];
    return lowp_to_f32<GT>(static_cast<const uint16_t *>(gp)[k]);
}

// Registers of one group of 8 consecutive elements.
template <int GT>
struct Group {
    uint4 p[2], m[2], v[2];
    uint4 g[GT == kF32 ? 2 : 1];
};

template <int GT>
__device__ __forceinline__ void load_group(Group<GT> &r, const float *pp, const float *mp,
                                           const float *vp, const void *gp, int64_t e) {
    r.p[0] = ld16(pp + e);
    r.p[1] = ld16(pp + e + 4);
    r.m[0] = ld16(mp + e);
    r.m[1] = ld16(mp + e + 4);
    r.v[0] = ld16(vp + e);
    r.v[1] = ld16(vp + e + 4);
    if constexpr (GT == kF32) {
        r.g[0] = ld16(static_cast<const float *>(gp) + e);
        r.g[1] = ld16(static_cast<const float *>(gp) + e + 4);
    } else {
        r.g[0] = ld16(static_cast<const uint16_t *>(gp) + e);
    }
}

__device__ __forceinline__ float u4_get(const uint4 &w, int j) {
    return __uint_as_float(j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w);
}
__device__ __forceinline__ void u4_set(uint4 &w, int j, float f) {
    const uint32_t b = __float_as_uint(f);
    if (j == 0) w.x = b; else if (j == 1) w.y = b; else if (j == 2) w.z = b; else w.w = b;
}

template <int GT, bool BF16, bool SR = false>
__device__ __forceinline__ uint4 compute_store_group(Group<GT> &r, float *pp, float *mp, float *vp,
                                                     uint16_t *bp, int64_t e, const Scal &s,
                                                     uint32_t &amax2, const uint4 *rnd = nullptr) {
    float p[8], m[8], v[8], g[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        p[j] = u4_get(r.p[j >> 2], j & 3);
        m[j] = u4_get(r.m[j >> 2], j & 3);
        v[j] = u4_get(r.v[j >> 2], j & 3);
    }
    if constexpr (GT == kF32) {
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = u4_get(r.g[j >> 2], j & 3);
    } else {
        const uint32_t w[4] = {r.g[0].x, r.g[0].y, r.g[0].z, r.g[0].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            g[2 * j] = lowp_to_f32<GT>(w[j] & 0xFFFFu);
            g[2 * j + 1] = lowp_to_f32<GT>(w[j] >> 16);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) adamw_elem(p[j], m[j], v[j], g[j], s);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        u4_set(r.p[j >> 2], j & 3, p[j]);
        u4_set(r.m[j >> 2], j & 3, m[j]);
        u4_set(r.v[j >> 2], j & 3, v[j]);
    }
    st16(pp + e, r.p[0]);
    st16(pp + e + 4, r.p[1]);
    st16(mp + e, r.m[0]);
    st16(mp + e + 4, r.m[1]);
    st16(vp + e, r.v[0]);
    st16(vp + e + 4, r.v[1]);
    if (BF16) {
        uint4 o;
        if constexpr (SR) {
            o = bf16x8_stochastic(p, *rnd);
        } else {
            o.x = f32x2_to_bf16x2(p[0], p[1]);
            o.y = f32x2_to_bf16x2(p[2], p[3]);
            o.z = f32x2_to_bf16x2(p[4], p[5]);
            o.w = f32x2_to_bf16x2(p[6], p[7]);
        }
        st16(bp + e, o);
        amax2 = __vmaxu2(amax2, __vmaxu2(__vmaxu2(o.x & 0x7FFF7FFFu, o.y & 0x7FFF7FFFu),
                                         __vmaxu2(o.z & 0x7FFF7FFFu, o.w & 0x7FFF7FFFu)));
        return o;
    }
    return make_uint4(0u, 0u, 0u, 0u);
}

template <int GT, bool BF16, bool SR = false>
__device__ __forceinline__ uint16_t scalar_elem(float *pp, float *mp, float *vp, const void *gp,
                                                uint16_t *bp, int64_t k, const Scal &s,
                                                uint32_t &amax1, uint32_t u16 = 0) {
    float p = pp[k], m = mp[k], v = vp[k];
    adamw_elem(p, m, v, grad_at<GT>(gp, k), s);
    pp[k] = p;
    mp[k] = m;
    vp[k] = v;
    if (BF16) {
        const uint16_t b = SR ? uint16_t(bf16_stochastic(p, u16)) : f32_to_bf16(p);
        bp[k] = b;
        amax1 = max(amax1, uint32_t(b & 0x7FFFu));
        return b;
    }
    return 0;
}

// 16 random bits of element k (an index within its tensor) for the SR path.
__device__ __forceinline__ uint32_t sr_u16(uint64_t seed, int32_t t, int tensor, int64_t k) {
    const uint4 r = sr_random8(seed, t, tensor, k >> 3);
    const int lane = int(k & 7);
    const uint32_t w = (lane >> 1) == 0 ? r.x : (lane >> 1) == 1 ? r.y : (lane >> 1) == 2 ? r.z : r.w;
    return (lane & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// ---------------------------------------------------------------------------
// The update pass over the plain (non-FP8-tiled) tensors, one CTA per chunk,
// streamed with TMA bulk copies: the chunk goes through kStages shared-memory
// stages of kSub elements.  One thread issues the cp.async.bulk loads of the
// p, m, v and g runs into a stage (completion counted by bytes on the stage's
// mbarrier) kStages sub-blocks ahead; every thread updates groups of 8
// elements in shared memory; the results go back with cp.async.bulk stores,
// whose reads of the stage are awaited before it is refilled.  On GB300 a
// plain copy streams ~5 % faster this way than with per-thread 16-byte
// loads/stores, and this kernel ~0.5 % faster than its per-thread form; 2
// stages of 2048 elements measured best (1024 x 2..4, 2048 x 3 and smaller
// stages were 0.6-50 % slower).  Every wait is bounded in time: one that
// gives up sets the sticky error word, lets its own loads land and returns.
// Chunks whose addresses do not allow 16-byte bulk copies, and the last
// (n mod 8) elements of a tensor, take the per-element path.
// ---------------------------------------------------------------------------
constexpr int kSub = 2048;    // elements per stage
constexpr int kStages = 2;    // stages in flight per CTA

template <int GT>
__host__ __device__ constexpr int bulk_stage_bytes() { return kSub * (12 + (GT == kF32 ? 4 : 2) + 2); }

template <int GT, bool BF16, bool SR>
__global__ void __launch_bounds__(kThreads) adamw_bulk_kernel(AdamwParams P) {
    pdl_wait();
    pdl_trigger();
    const AdamwStepScalars sc = *P.scal;
    if (sc.skip) return;  // A2: nothing is written on a skipped step
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar[kStages];
    const uint2 ch = P.p.chunks[blockIdx.x];
    const int t = int(ch.x);
    const int64_t start = int64_t(ch.y) * kChunk;
    const int64_t n = min(int64_t(kChunk), P.p.numel[t] - start);
    constexpr int gsz = GT == kF32 ? 4 : 2;
    float *pp = static_cast<float *>(P.p.ptrs[t]) + start;
    float *mp = static_cast<float *>(P.m.ptrs[t]) + start;
    float *vp = static_cast<float *>(P.v.ptrs[t]) + start;
    const char *gp = static_cast<const char *>(P.g.ptrs[t]) + start * gsz;
    uint16_t *bp = BF16 ? static_cast<uint16_t *>(P.b.ptrs[t]) + start : nullptr;

    Scal s;
    s.r = P.scale ? __fdiv_rn(1.0f, *P.scale) : 1.0f;
    s.clip = sc.clip;
    s.decay = P.decay;
    s.b1 = P.b1;
    s.omb1 = P.omb1;
    s.b2 = P.b2;
    s.omb2 = P.omb2;
    s.eps = P.eps;
    s.step_size = sc.step_size;
    s.c2 = sc.bc2_sqrt;

    uint32_t amax2 = 0, amax1 = 0;
    const bool vec = aligned16(pp) && aligned16(mp) && aligned16(vp) && aligned16(gp) &&
                     (!BF16 || aligned16(bp));
    int64_t done = 0;  // elements handled by the bulk pipeline
    if (vec) {
        constexpr int kStage = bulk_stage_bytes<GT>();
        const int64_t nb = n & ~int64_t(7);
        const int nsub = int((nb + kSub - 1) / kSub);
        if (threadIdx.x == 0) {
            for (int q = 0; q < kStages; ++q) mbar_init(&bar[q], 1);
            mbar_fence_init();
        }
        __syncthreads();
        // stage layout: p | m | v (fp32) | g | bf16
        auto stage_p = [&](int k) { return reinterpret_cast<float *>(smem + (k % kStages) * kStage); };
        auto issue = [&](int k) {
            const int64_t off = int64_t(k) * kSub;
            const uint32_t cnt = uint32_t(min(int64_t(kSub), nb - off));
            float *sp = stage_p(k);
            uint64_t *b = &bar[k % kStages];
            mbar_arrive_expect_tx(b, cnt * (12u + gsz));
            bulk_g2s(sp, pp + off, cnt * 4u, b);
            bulk_g2s(sp + kSub, mp + off, cnt * 4u, b);
            bulk_g2s(sp + 2 * kSub, vp + off, cnt * 4u, b);
            bulk_g2s(sp + 3 * kSub, gp + off * gsz, cnt * gsz, b);
        };
        if (threadIdx.x == 0)
            for (int q = 0; q < kStages && q < nsub; ++q) issue(q);
        uint32_t phases = 0;  // bit q: parity of stage q's next completion
        int failed_at = -1;   // sub-block whose wait gave up
        for (int k = 0; k < nsub; ++k) {
            const int64_t off = int64_t(k) * kSub;
            const int cnt = int(min(int64_t(kSub), nb - off));
            const int q = k % kStages;
            const bool w = mbar_wait(&bar[q], (phases >> q) & 1u);
            if (!__syncthreads_and(w)) {
                failed_at = k;
                break;
            }
            phases ^= 1u << q;
            float *sp = stage_p(k);
            for (int j = threadIdx.x; 8 * j < cnt; j += kThreads) {
                Group<GT> r;
                const uint4 *p4 = reinterpret_cast<const uint4 *>(sp) + 2 * j;
                const uint4 *m4 = reinterpret_cast<const uint4 *>(sp + kSub) + 2 * j;
                const uint4 *v4 = reinterpret_cast<const uint4 *>(sp + 2 * kSub) + 2 * j;
                r.p[0] = p4[0];
                r.p[1] = p4[1];
                r.m[0] = m4[0];
                r.m[1] = m4[1];
                r.v[0] = v4[0];
                r.v[1] = v4[1];
                const uint4 *g4 = reinterpret_cast<const uint4 *>(sp + 3 * kSub);
                if constexpr (GT == kF32) {
                    r.g[0] = g4[2 * j];
                    r.g[1] = g4[2 * j + 1];
                } else {
                    r.g[0] = g4[j];
                }
                uint4 rnd;
                if constexpr (SR) rnd = sr_random8(P.sr_seed, sc.t, t, ((start + off) >> 3) + j);
                // compute_store_group writes to p/m/v/b at the given element
                // offset: point it at this stage's shared buffers
                uint16_t *sb = reinterpret_cast<uint16_t *>(
                    reinterpret_cast<unsigned char *>(sp + 3 * kSub) + kSub * gsz);
                compute_store_group<GT, BF16, SR>(r, sp, sp + kSub, sp + 2 * kSub, sb,
                                                  int64_t(8) * j, s, amax2, &rnd);
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (threadIdx.x == 0) {
                bulk_s2g(pp + off, sp, uint32_t(cnt) * 4u);
                bulk_s2g(mp + off, sp + kSub, uint32_t(cnt) * 4u);
                bulk_s2g(vp + off, sp + 2 * kSub, uint32_t(cnt) * 4u);
                if (BF16)
                    bulk_s2g(bp + off,
                             reinterpret_cast<unsigned char *>(sp + 3 * kSub) + kSub * gsz,
                             uint32_t(cnt) * 2u);
                bulk_commit();
                if (k + kStages < nsub) {
                    bulk_wait_read_all();  // this stage's stores have read it
                    issue(k + kStages);
                }
            }
        }
        if (threadIdx.x == 0) {
            if (failed_at >= 0) {
                atomicExch(P.err, 1);
                // let the loads issued for sub-blocks failed_at .. failed_at+kStages-1
                // finish landing in this CTA's shared memory before it exits
                for (int k = failed_at; k < failed_at + kStages && k < nsub; ++k)
                    mbar_wait(&bar[k % kStages], (phases >> (k % kStages)) & 1u);
            }
            bulk_wait_all();
        }
        if (failed_at >= 0) return;
        done = nb;
    }
    for (int64_t k = done + threadIdx.x; k < n; k += kThreads)
        scalar_elem<GT, BF16, SR>(pp, mp, vp, gp, bp, k, s, amax1,
                                  SR ? sr_u16(P.sr_seed, sc.t, t, start + k) : 0u);
    if (BF16 && P.use_slots) {
        const int slot = P.b.slots[t];
        if (slot >= 0) {
            uint32_t a = max(max(amax2 & 0xFFFFu, amax2 >> 16), amax1);
            a = warp_max_u32(a);
            if ((threadIdx.x & 31) == 0 && a != 0)
                atomicMax(reinterpret_cast<unsigned int *>(P.amax) + slot, a << 16);
        }
    }
}

// Per-step scalars: skip flag, bias corrections (fp64, rounded once), clip
// factor; advances the step counter when the step is not skipped.
__device__ __forceinline__ AdamwStepScalars step_scalars(const int32_t *found_inf, int32_t *step,
                                                         double lr, double beta1, double beta2,
                                                         const double *clip_sumsq,
                                                         double max_norm) {
    AdamwStepScalars s;
    s.skip = found_inf ? (*found_inf != 0) : 0;
    s.step_size = 0.0f;
    s.bc2_sqrt = 1.0f;
    s.clip = 1.0f;
    s.t = *step;
    s.pad[0] = s.pad[1] = s.pad[2] = 0;
    if (clip_sumsq) {
        // min(1, max_norm / (||g|| + 1e-6)), NaN propagating
        const double c = max_norm / (sqrt(*clip_sumsq) + 1e-6);
        s.clip = float(c != c ? c : (c < 1.0 ? c : 1.0));
    }
    if (!s.skip) {
        const int32_t t = *step + 1;
        const double bc1 = 1.0 - pow(beta1, double(t));
        const double bc2 = 1.0 - pow(beta2, double(t));
        s.step_size = float(lr / bc1);
        s.bc2_sqrt = float(sqrt(bc2));
        s.t = t;
        *step = t;
    }
    return s;
}

__global__ void adamw_prologue_kernel(const int32_t *found_inf, int32_t *step, double lr,
                                      double beta1, double beta2, const double *clip_sumsq,
                                      double max_norm, AdamwStepScalars *out) {
    pdl_wait();
    pdl_trigger();
    *out = step_scalars(found_inf, step, lr, beta1, beta2, clip_sumsq, max_norm);
}

// ---------------------------------------------------------------------------
// AdamW + BF16 + FP8 with delayed scaling ("第20章 量化与混合精度训练" §20.5.9:
// each FP8 op keeps an amax history and casts with the scale of the previous
// steps' amax).  The scale is known before the pass, so the FP8 bytes and
// their transposed copy come out of the same pass as the update: 30 bytes per
// parameter for the FP8 weights instead of 28 + 4 in two passes.
// ---------------------------------------------------------------------------
struct Fp8StepParams {
    ListView p, m, v, g, b, q, qt;
    int has_t;
    const float *scale;
    const AdamwStepScalars *scal;
    const float *tscale;  // per tensor: the fp32 cast scale from the history
    float *amax;          // per tensor: max|bf16| of this step, for the history
    float decay, b1, omb1, b2, omb2, eps;
    uint64_t sr_seed;     // stochastic rounding of the bf16 and FP8 copies
};

// Tensor word of the bf16 copy's random counter for FP8 weight t of the
// delayed step (its plain tensors use their own list index, below 2^30).
constexpr uint32_t kSrFp8GroupBit = 0x40000000u;

// Eight bf16 values (a 16-byte word group of elements k0 .. k0+7 of FP8
// weight `tensor`) -> eight stochastically rounded fp8 bytes of x * s32.
template <int FT>
__device__ __forceinline__ uint2 bf16x8_to_fp8x8_sr(const uint4 &b, float s32, uint64_t seed,
                                                    int32_t step, int tensor, int64_t k0) {
    const uint32_t w[4] = {b.x, b.y, b.z, b.w};
    float y[8];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        mul2_rn(bf16_bits_to_f32(w[j] & 0xFFFFu), bf16_bits_to_f32(w[j] >> 16), s32, s32,
                y[2 * j], y[2 * j + 1]);
    return fp8x8_stochastic<FT>(y, seed, step, tensor, k0);
}

// One CTA: thread 0 the step scalars; every thread a strided share of the
// FP8 tensors' scales from their amax histories (NaN propagating max).
__global__ void adamw_fp8_prologue_kernel(const int32_t *found_inf, int32_t *step, double lr,
                                          double beta1, double beta2, AdamwStepScalars *out,
                                          const float *hist, int hist_len, int n8, EpsFloor ef,
                                          float fmax, float *tscale, float *inv_scale) {
    pdl_wait();
    pdl_trigger();
    const int skip = found_inf ? (*found_inf != 0) : 0;
    __syncthreads();  // every thread has read found_inf before thread 0 goes on
    if (threadIdx.x == 0) *out = step_scalars(found_inf, step, lr, beta1, beta2, nullptr, 0.0);
    if (skip) return;
    for (int j = threadIdx.x; j < n8; j += blockDim.x) {
        const float *h = hist + int64_t(j) * hist_len;
        float a = h[0];
        for (int k = 1; k < hist_len; ++k) a = (a != a || h[k] != h[k]) ? __int_as_float(0x7FC00000) : fmaxf(a, h[k]);
        float s32, inv;
        tensor_scale(a, ef, fmax, s32, inv);
        tscale[j] = s32;
        inv_scale[j] = inv;
    }
}

template <int GT, int FT, bool SR>
__device__ __forceinline__ void adamw_fp8_tile(const Fp8StepParams &P) {
    pdl_wait();
    pdl_trigger();
    const AdamwStepScalars sc = *P.scal;
    if (sc.skip) return;
    __shared__ __align__(16) uint32_t sm[kTile * 32];
    const uint2 tl = P.p.tiles[blockIdx.x];
    const int t = int(tl.x);
    const int64_t rows = P.p.rows[t], cols = P.p.cols[t];
    const int64_t tiles_c = (cols + kTile - 1) / kTile;
    const int64_t r0 = int64_t(tl.y / tiles_c) * kTile, c0 = int64_t(tl.y % tiles_c) * kTile;
    float *pp = static_cast<float *>(P.p.ptrs[t]);
    float *mp = static_cast<float *>(P.m.ptrs[t]);
    float *vp = static_cast<float *>(P.v.ptrs[t]);
    const void *gp = P.g.ptrs[t];
    uint16_t *bp = static_cast<uint16_t *>(P.b.ptrs[t]);
    uint8_t *qp = static_cast<uint8_t *>(P.q.ptrs[t]);
    uint8_t *qtp = P.has_t ? static_cast<uint8_t *>(P.qt.ptrs[t]) : nullptr;

    Scal s;
    s.r = P.scale ? __fdiv_rn(1.0f, *P.scale) : 1.0f;
    s.clip = sc.clip;
    s.decay = P.decay;
    s.b1 = P.b1;
    s.omb1 = P.omb1;
    s.b2 = P.b2;
    s.omb2 = P.omb2;
    s.eps = P.eps;
    s.step_size = sc.step_size;
    s.c2 = sc.bc2_sqrt;
    const float s32 = P.tscale[t];

    uint32_t amax2 = 0, amax1 = 0;
    const bool fast = r0 + kTile <= rows && c0 + kTile <= cols && (cols & 7) == 0 &&
                      aligned16(pp) && aligned16(mp) && aligned16(vp) && aligned16(gp) &&
                      aligned16(bp) && (reinterpret_cast<uintptr_t>(qp) & 7) == 0 &&
                      (qtp == nullptr || ((rows & 15) == 0 && aligned16(qtp)));
    if (fast && SR) {
        // The stochastic form loads the next two groups before it rounds the
        // FP8 bytes of the current two, so that the generator draws and the
        // roundings, which need no memory, run while those loads are in flight.
        const int c8 = threadIdx.x & 15, rb = threadIdx.x >> 4;
        const int32_t bid = int32_t(uint32_t(t) | kSrFp8GroupBit);
        int64_t ea = (r0 + rb) * cols + c0 + 8 * c8, eb = ea + 16 * cols;
        Group<GT> a, b;
        load_group<GT>(a, pp, mp, vp, gp, ea);
        load_group<GT>(b, pp, mp, vp, gp, eb);
#pragma unroll 1
        for (int k = 0; k < 8; k += 2) {
            const uint4 rna = sr_random8(P.sr_seed, sc.t, bid, ea >> 3);
            const uint4 rnb = sr_random8(P.sr_seed, sc.t, bid, eb >> 3);
            const uint4 oa = compute_store_group<GT, true, true>(a, pp, mp, vp, bp, ea, s, amax2,
                                                                 &rna);
            const uint4 ob = compute_store_group<GT, true, true>(b, pp, mp, vp, bp, eb, s, amax2,
                                                                 &rnb);
            const int64_t ea0 = ea, eb0 = eb;
            if (k + 2 < 8) {
                ea += 32 * cols;
                eb += 32 * cols;
                load_group<GT>(a, pp, mp, vp, gp, ea);
                load_group<GT>(b, pp, mp, vp, gp, eb);
            }
            const uint2 qa = bf16x8_to_fp8x8_sr<FT>(oa, s32, P.sr_seed, sc.t, t, ea0);
            const uint2 qb = bf16x8_to_fp8x8_sr<FT>(ob, s32, P.sr_seed, sc.t, t, eb0);
            *reinterpret_cast<uint2 *>(qp + ea0) = qa;
            *reinterpret_cast<uint2 *>(qp + eb0) = qb;
            if (qtp) {
                *reinterpret_cast<uint2 *>(sm + swz(rb + 16 * k, 2 * c8)) = qa;
                *reinterpret_cast<uint2 *>(sm + swz(rb + 16 * (k + 1), 2 * c8)) = qb;
            }
        }
    } else if (fast) {
        const int c8 = threadIdx.x & 15, rb = threadIdx.x >> 4;
#pragma unroll 1
        for (int k = 0; k < 8; k += 2) {
            const int ra = rb + 16 * k, rbb = rb + 16 * (k + 1);
            const int64_t ea = (r0 + ra) * cols + c0 + 8 * c8;
            const int64_t eb = (r0 + rbb) * cols + c0 + 8 * c8;
            Group<GT> a, b;
            load_group<GT>(a, pp, mp, vp, gp, ea);
            load_group<GT>(b, pp, mp, vp, gp, eb);
            const uint4 oa = compute_store_group<GT, true>(a, pp, mp, vp, bp, ea, s, amax2);
            const uint4 ob = compute_store_group<GT, true>(b, pp, mp, vp, bp, eb, s, amax2);
            const uint2 qa = bf16x8_to_fp8x8<FT>(oa, s32);
            const uint2 qb = bf16x8_to_fp8x8<FT>(ob, s32);
            *reinterpret_cast<uint2 *>(qp + ea) = qa;
            *reinterpret_cast<uint2 *>(qp + eb) = qb;
            if (qtp) {
                *reinterpret_cast<uint2 *>(sm + swz(ra, 2 * c8)) = qa;
                *reinterpret_cast<uint2 *>(sm + swz(rbb, 2 * c8)) = qb;
            }
        }
    }
    if (fast && qtp) {
        __syncthreads();
        store_transposed_tile(sm, qtp, rows, r0, c0);
    }
    if (!fast) {
        for (int idx = threadIdx.x; idx < kTile * kTile; idx += kThreads) {
            const int64_t i = r0 + (idx >> 7), j = c0 + (idx & (kTile - 1));
            if (i < rows && j < cols) {
                const int64_t e = i * cols + j;
                uint16_t bv;
                uint8_t q8;
                if constexpr (SR) {
                    bv = scalar_elem<GT, true, true>(
                        pp, mp, vp, gp, bp, e, s, amax1,
                        sr_u16(P.sr_seed, sc.t, int(uint32_t(t) | kSrFp8GroupBit), e));
                    q8 = uint8_t(fp8_stochastic<FT>(__fmul_rn(bf16_bits_to_f32(bv), s32),
                                                    sr8_word(P.sr_seed, sc.t, t, e)));
                } else {
                    bv = scalar_elem<GT, true>(pp, mp, vp, gp, bp, e, s, amax1);
                    q8 = quant1<FT>(bf16_bits_to_f32(bv), s32);
                }
                qp[e] = q8;
                if (qtp) qtp[j * rows + i] = q8;
            }
        }
    }
    uint32_t a = max(max(amax2 & 0xFFFFu, amax2 >> 16), amax1);
    a = warp_max_u32(a);
    if ((threadIdx.x & 31) == 0 && a != 0)
        atomicMax(reinterpret_cast<unsigned int *>(P.amax) + t, a << 16);
}

template <int GT, int FT>
__global__ void __launch_bounds__(kThreads) adamw_fp8_tile_kernel(Fp8StepParams P) {
    adamw_fp8_tile<GT, FT, false>(P);
}

// The stochastic form is held to 128 registers, so two CTAs share an SM as
// with the plain form (left to itself it took 143).
template <int GT, int FT>
__global__ void __launch_bounds__(kThreads, 2) adamw_fp8_tile_sr_kernel(Fp8StepParams P) {
    adamw_fp8_tile<GT, FT, true>(P);
}

// Self-test of the bounded wait: a barrier that nothing completes (one
// expected arrival, none made); the wait must give up after limit_ns and
// report through *err, leaving the context usable.
__global__ void bounded_wait_selftest_kernel(int32_t *err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        const bool done = mbar_wait(&bar, 0, limit_ns);
        *err = done ? 0 : 1;
    }
}

template <int GT, bool BF16, bool SR>
void bulk_launch(dim3 grid, dim3 block, cudaStream_t s, const AdamwParams &P) {
    constexpr int smem = kStages * bulk_stage_bytes<GT>();
    // above the 48 KB default: opt in (cheap, and valid for whichever device is current)
    cudaFuncSetAttribute(adamw_bulk_kernel<GT, BF16, SR>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    launch_pdl(adamw_bulk_kernel<GT, BF16, SR>, grid, block, smem, s, P);
}

}  // namespace

cudaError_t launch_adamw(const ListView &p, const ListView &m, const ListView &v,
                         const ListView &g, const ListView *b, int64_t n_chunks, int gelem,
                         const float *scale, const int32_t *found_inf, int32_t *step,
                         const AdamwConsts &c, AdamwStepScalars *scal, float *amax,
                         bool use_slots, cudaStream_t s, const double *clip_sumsq,
                         double max_norm, bool stochastic, uint64_t seed) {
    launch_pdl(adamw_prologue_kernel, dim3(1), dim3(1), 0, s, found_inf, step, c.lr, c.beta1,
               c.beta2, clip_sumsq, max_norm, scal);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_adamw_main(p, m, v, g, b, n_chunks, gelem, scale, c, scal, amax, use_slots, s,
                             stochastic, seed);
}

cudaError_t launch_adamw_main(const ListView &p, const ListView &m, const ListView &v,
                              const ListView &g, const ListView *b, int64_t n_chunks, int gelem,
                              const float *scale, const AdamwConsts &c,
                              const AdamwStepScalars *scal, float *amax, bool use_slots,
                              cudaStream_t s, bool stochastic, uint64_t seed) {
    // the sticky error word sits next to the step scalars in the same scratch block
    int32_t *err = reinterpret_cast<int32_t *>(const_cast<AdamwStepScalars *>(scal)) + kErrWordOffset;
    if (n_chunks == 0) return cudaSuccess;
    AdamwParams P;
    P.p = p;
    P.m = m;
    P.v = v;
    P.g = g;
    P.b = b ? *b : ListView{};
    P.scale = scale;
    P.scal = scal;
    P.amax = amax;
    P.decay = c.decay;
    P.b1 = c.b1;
    P.omb1 = c.omb1;
    P.b2 = c.b2;
    P.omb2 = c.omb2;
    P.eps = c.eps;
    P.use_slots = use_slots ? 1 : 0;
    P.sr_seed = seed;
    P.err = err;
    const dim3 grid((unsigned)n_chunks), block(kThreads);
    const bool bf = b != nullptr;
#define AMP_ADAMW_LAUNCH(GT)                                                         \
    do {                                                                             \
        if (bf && stochastic) bulk_launch<GT, true, true>(grid, block, s, P);         \
        else if (bf) bulk_launch<GT, true, false>(grid, block, s, P);                \
        else bulk_launch<GT, false, false>(grid, block, s, P);                       \
    } while (0)
    if (gelem == kF32) AMP_ADAMW_LAUNCH(kF32);
    else if (gelem == kF16) AMP_ADAMW_LAUNCH(kF16);
    else AMP_ADAMW_LAUNCH(kBF16);
#undef AMP_ADAMW_LAUNCH
    return cudaGetLastError();
}

cudaError_t launch_adamw_fp8_delayed(const Fp8DelayedLists &L, int gelem, int fp8,
                                     const float *scale, const int32_t *found_inf, int32_t *step,
                                     const AdamwConsts &c, AdamwStepScalars *scal,
                                     const float *hist, int hist_len, double eps, float *amax,
                                     float *inv_scale, cudaStream_t s, bool stochastic,
                                     uint64_t seed) {
    const float fmax = fp8 == kE4M3 ? fp8_max<kE4M3>() : fp8_max<kE5M2>();
    launch_pdl(adamw_fp8_prologue_kernel, dim3(1), dim3(256), 0, s, found_inf, step, c.lr, c.beta1,
               c.beta2, scal, hist, hist_len, L.n8, make_eps_floor(eps, fmax), fmax, L.tscale,
               inv_scale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (L.n_plain_chunks > 0) {
        e = launch_adamw_main(L.p, L.m, L.v, L.g, &L.b, L.n_plain_chunks, gelem, scale, c, scal,
                              nullptr, false, s, stochastic, seed);
        if (e != cudaSuccess) return e;
    }
    if (L.n_tiles == 0) return cudaSuccess;
    Fp8StepParams P;
    P.p = L.p8;
    P.m = L.m8;
    P.v = L.v8;
    P.g = L.g8;
    P.b = L.b8;
    P.q = L.q;
    P.qt = L.qt ? *L.qt : ListView{};
    P.has_t = L.qt != nullptr;
    P.scale = scale;
    P.scal = scal;
    P.tscale = L.tscale;
    P.amax = amax;
    P.decay = c.decay;
    P.b1 = c.b1;
    P.omb1 = c.omb1;
    P.b2 = c.b2;
    P.omb2 = c.omb2;
    P.eps = c.eps;
    P.sr_seed = seed;
    const dim3 grid((unsigned)L.n_tiles), block(kThreads);
    // A plain launch: with programmatic dependent launch this kernel ran 6 %
    // slower on GB300 (30.7 -> 32.5 ms on the 8B set), while the chunked pass
    // before it gained nothing from the overlap.
#define AMP_FP8_LAUNCH(GT)                                                                  \
    do {                                                                                    \
        if (stochastic) {                                                                   \
            if (fp8 == kE4M3) adamw_fp8_tile_sr_kernel<GT, kE4M3><<<grid, block, 0, s>>>(P);   \
            else adamw_fp8_tile_sr_kernel<GT, kE5M2><<<grid, block, 0, s>>>(P);              \
        } else {                                                                            \
            if (fp8 == kE4M3) adamw_fp8_tile_kernel<GT, kE4M3><<<grid, block, 0, s>>>(P);   \
            else adamw_fp8_tile_kernel<GT, kE5M2><<<grid, block, 0, s>>>(P);                \
        }                                                                                   \
    } while (0)
    if (gelem == kF32) AMP_FP8_LAUNCH(kF32);
    else if (gelem == kF16) AMP_FP8_LAUNCH(kF16);
    else AMP_FP8_LAUNCH(kBF16);
#undef AMP_FP8_LAUNCH
    return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(int32_t *err, double limit_s, cudaStream_t s) {
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(err, (unsigned long long)(limit_s * 1e9));
    return cudaGetLastError();
}

}  // namespace amp
