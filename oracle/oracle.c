/*
 * oracle.c - plain, slow, single-threaded CPU oracle for the mixed-precision
 * optimizer step (loss-scale unscale/check, scale state machine, FP32-master
 * AdamW with BF16 emission, tensorwise dynamic FP8 quantization).
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the smoke check and the CPU
 * baseline leg of bench.py load this file.  It shares no code, header, table
 * or constant with the CUDA library; it includes no CUDA header.  Build with
 *     gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared oracle.c -lm
 * (-ffp-contract=off: every float operation is rounded on its own, no fused
 * multiply-add is formed behind the reader's back).
 *
 * Sources (page title, then section):
 *   [CH20]  "第20章 量化与混合精度训练" (PyTorch book, ch. 20):
 *           §20.2.2 GradScaler, §20.5.13 Master Weights,
 *           §20.5.33 GradScaler 的 _growth_tracker 状态机细节.
 *   [MP]    "从 AMP 到 Mixed Precision：训练和推理为什么不使用同一种精度":
 *           "Gradient 和 Loss Scaling", "训练中到底哪些东西是低精度",
 *           "为什么需要 FP32 Master Weights", "PyTorch AMP 与 FP32 Master Weights".
 *   [FP8]   "FP8训练：量化、自动微分、Torchao": §2 量化数学, §3 格式选择,
 *           §4 _scaled_mm 布局要求.
 *   [NOTES] "AMP：Automatic Mixed Precision 技术笔记": §4 GradScaler.
 *   [MP06]  "06 · 混合精度": §一 五种数字格式, §三 主权重副本, §四 Loss Scaling.
 *
 * Readings of points the pages leave open:
 *   - AdamW is named but never written out on the pages; the oracle takes
 *     the published decoupled-weight-decay AdamW (Loshchilov & Hutter) with
 *     Adam's bias correction, in the parametrisation of torch.optim.AdamW
 *     (decay factor 1 - lr*wd, eps added after the square root), computed in
 *     fp32 because [MP] "训练中到底哪些东西是低精度" puts optimizer states and
 *     the master-weight update in FP32.  Per-step scalars in fp64.
 *   - Unscale multiplies by the correctly rounded fp32 value of 1/S.
 *   - NaN outputs of every encoder are the positive canonical quiet NaN of
 *     the target format (fp16 0x7E00, bf16 0x7FC0, e4m3fn 0x7F, e5m2 0x7E).
 *   - Growth that would make S non-finite keeps S.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

/* dtype codes understood by the oracle entry points */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_E4M3FN = 3, ORC_E5M2 = 4 };

/* ------------------------------------------------------------------------ */
/* Number formats, written from their definitions.                          */
/*   binary16 : 1 sign | 5 exponent (bias 15)  | 10 fraction, IEEE specials */
/*   bfloat16 : 1 sign | 8 exponent (bias 127) | 7 fraction, IEEE specials  */
/*   E5M2     : 1 sign | 5 exponent (bias 15)  | 2 fraction, IEEE specials  */
/*   E4M3FN   : 1 sign | 4 exponent (bias 7)   | 3 fraction, no infinity;   */
/*              exponent 1111 holds normal numbers, only S.1111.111 is NaN  */
/* ([MP06] §一 bit layouts; [FP8] §3 e4m3 max 448 / e5m2 max 57344).        */
/* ------------------------------------------------------------------------ */
typedef struct {
    int ebits, mbits, bias;
    int ieee;            /* 1: all-ones exponent is inf/NaN; 0: E4M3FN rule */
    uint32_t nan_code;   /* canonical positive NaN emitted by the encoder */
} orc_fmt;

static const orc_fmt FMT_F16  = {5, 10, 15, 1, 0x7E00u};
static const orc_fmt FMT_BF16 = {8, 7, 127, 1, 0x7FC0u};
static const orc_fmt FMT_E5M2 = {5, 2, 15, 1, 0x7Eu};
static const orc_fmt FMT_E4M3 = {4, 3, 7, 0, 0x7Fu};

/* largest finite magnitude of a format */
static double fmt_max(const orc_fmt *f)
{
    int top = (1 << f->ebits) - 1;
    if (f->ieee) /* exponent top-1, fraction all ones */
        return ldexp(2.0 - ldexp(1.0, -f->mbits), top - 1 - f->bias);
    /* E4M3FN: exponent top, fraction all ones except the last (that is NaN) */
    return ldexp(2.0 - 2.0 * ldexp(1.0, -f->mbits), top - f->bias);
}

static double fmt_decode(const orc_fmt *f, uint32_t bits)
{
    uint32_t top = (1u << f->ebits) - 1u, fmask = (1u << f->mbits) - 1u;
    int sign = (bits >> (f->ebits + f->mbits)) & 1u;
    uint32_t e = (bits >> f->mbits) & top, m = bits & fmask;
    double mag;
    if (f->ieee && e == top)
        mag = m ? NAN : INFINITY;
    else if (!f->ieee && e == top && m == fmask)
        mag = NAN;
    else if (e == 0) /* subnormal: m * 2^(1-bias-mbits) */
        mag = ldexp((double)m, 1 - f->bias - f->mbits);
    else
        mag = ldexp((double)((1u << f->mbits) + m), (int)e - f->bias - f->mbits);
    return sign ? -mag : mag;
}

/* Round-to-nearest, ties-to-even encoding of a real value x.  Overflow gives
 * infinity (IEEE-style formats) or NaN (E4M3FN has no infinity); callers that
 * want saturation clamp first, as the FP8 quantizer does. */
static uint32_t fmt_encode(const orc_fmt *f, double x)
{
    uint32_t sbit = 1u << (f->ebits + f->mbits);
    uint32_t top = (1u << f->ebits) - 1u;
    uint32_t sign = signbit(x) ? sbit : 0u;
    if (isnan(x))
        return f->nan_code;
    double a = fabs(x);
    if (isinf(a))
        return f->ieee ? (sign | (top << f->mbits)) : f->nan_code;
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2);           /* a = fr * 2^e2, fr in [0.5, 1) */
    int E = e2 - 1;                /* floor(log2 a) */
    int emin = 1 - f->bias;        /* exponent of the smallest normal */
    if (E < emin)
        E = emin;                  /* subnormal range shares the quantum */
    double q = ldexp(1.0, E - f->mbits); /* spacing of representable values */
    double r = a / q;              /* exact: division by a power of two */
    double n = floor(r), frac = r - n;
    if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) == 1.0))
        n += 1.0;
    double one = ldexp(1.0, f->mbits);
    if (n == 2.0 * one) {          /* rounded up into the next binade */
        n = one;
        E += 1;
    }
    if (n * ldexp(1.0, E - f->mbits) > fmt_max(f))
        return f->ieee ? (sign | (top << f->mbits)) : f->nan_code;
    uint32_t efield, mfield;
    if (n < one) {                 /* subnormal */
        efield = 0u;
        mfield = (uint32_t)n;
    } else {
        efield = (uint32_t)(E + f->bias);
        mfield = (uint32_t)(n - one);
    }
    return sign | (efield << f->mbits) | mfield;
}

static const orc_fmt *fmt_of(int dtype)
{
    switch (dtype) {
    case ORC_F16: return &FMT_F16;
    case ORC_BF16: return &FMT_BF16;
    case ORC_E4M3FN: return &FMT_E4M3;
    case ORC_E5M2: return &FMT_E5M2;
    default: return NULL;
    }
}

/* exported converters (used by the pin tests) */
double orc_fmt_max(int dtype) { return fmt_max(fmt_of(dtype)); }

void orc_decode(int dtype, const void *src, float *dst, int64_t n)
{
    const orc_fmt *f = fmt_of(dtype);
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = (dtype == ORC_E4M3FN || dtype == ORC_E5M2)
                         ? ((const uint8_t *)src)[i] : ((const uint16_t *)src)[i];
        dst[i] = (float)fmt_decode(f, b);
    }
}

void orc_encode(int dtype, const float *src, void *dst, int64_t n)
{
    const orc_fmt *f = fmt_of(dtype);
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = fmt_encode(f, (double)src[i]);
        if (dtype == ORC_E4M3FN || dtype == ORC_E5M2)
            ((uint8_t *)dst)[i] = (uint8_t)b;
        else
            ((uint16_t *)dst)[i] = (uint16_t)b;
    }
}

/* element k of a gradient buffer of the given dtype, as fp32 */
static float load_as_f32(int dtype, const void *p, int64_t k)
{
    if (dtype == ORC_F32)
        return ((const float *)p)[k];
    return (float)fmt_decode(fmt_of(dtype), ((const uint16_t *)p)[k]);
}

static void store_from_f32(int dtype, void *p, int64_t k, float v)
{
    if (dtype == ORC_F32)
        ((float *)p)[k] = v;
    else
        ((uint16_t *)p)[k] = (uint16_t)fmt_encode(fmt_of(dtype), (double)v);
}

/* ------------------------------------------------------------------------ */
/* Unscale + non-finite check.  [CH20] §20.2.2: the scaled gradients are     */
/* divided by the scale before the optimizer, then inspected for inf/NaN;    */
/* [NOTES] §4 steps 3-4; [MP] "Gradient 和 Loss Scaling".                    */
/* found_inf is OR-ed, never cleared here (several lists may feed one flag). */
/* ------------------------------------------------------------------------ */
void orc_unscale_check(int n_tensors, void *const *ptrs, const int64_t *numel,
                       int dtype, float scale, int32_t *found_inf, int inplace)
{
    float inv_s = 1.0f / scale;
    int found = 0;
    for (int t = 0; t < n_tensors; ++t) {
        for (int64_t k = 0; k < numel[t]; ++k) {
            float g = load_as_f32(dtype, ptrs[t], k) * inv_s;
            if (!isfinite(g))
                found = 1;
            if (inplace)
                store_from_f32(dtype, ptrs[t], k, g);
        }
    }
    if (found)
        *found_inf = 1;
}

/* ------------------------------------------------------------------------ */
/* Gradient-norm clipping after unscale.  "AMP：Automatic Mixed Precision 技术 */
/* 笔记" §6 and "06 · 混合精度" §四: with a loss scaler the gradients are       */
/* unscaled first and clipped afterwards (clip_grad_norm_(params, max_norm)),  */
/* otherwise the threshold would apply to the scaled values.  The pages call   */
/* the library routine without writing it out; the plain reading is the global */
/* L2 norm over every element of every gradient, and the factor               */
/* min(1, max_norm / (norm + 1e-6)) applied to each unscaled gradient.         */
/* ------------------------------------------------------------------------ */
double orc_grad_sumsq(int n_tensors, void *const *ptrs, const int64_t *numel, int dtype,
                      float scale)
{
    float inv_s = 1.0f / scale;
    double acc = 0.0;
    for (int t = 0; t < n_tensors; ++t)
        for (int64_t k = 0; k < numel[t]; ++k) {
            double g = (double)(load_as_f32(dtype, ptrs[t], k) * inv_s);
            acc += g * g;
        }
    return acc;
}

float orc_clip_coef(double sumsq, double max_norm)
{
    double c = max_norm / (sqrt(sumsq) + 1e-6);
    if (isnan(c))
        return (float)c; /* NaN propagates (the step is skipped anyway) */
    return (float)(c < 1.0 ? c : 1.0);
}

/* ------------------------------------------------------------------------ */
/* Dynamic loss-scale state machine, [CH20] §20.5.33: on inf/NaN multiply    */
/* the scale by backoff and reset the tracker; otherwise count the clean     */
/* step and multiply by growth once the count reaches the interval.          */
/* [MP06] 检查点: "没溢出就每隔 N 步把 S 翻倍; 出现 inf/nan 就 S 减半".       */
/* Afterwards the per-step flags are cleared for the next step.              */
/* ------------------------------------------------------------------------ */
void orc_update_scale(float *scale, int32_t *tracker, int32_t *found_inf,
                      float growth, float backoff, int32_t interval,
                      float *amax, int n_amax)
{
    if (*found_inf) {
        *scale = *scale * backoff;
        *tracker = 0;
    } else {
        *tracker = *tracker + 1;
        if (*tracker >= interval) {
            float grown = *scale * growth;
            if (isfinite(grown))
                *scale = grown;
            *tracker = 0;
        }
    }
    *found_inf = 0;
    for (int i = 0; i < n_amax; ++i)
        amax[i] = 0.0f;
}

/* ------------------------------------------------------------------------ */
/* FP32-master AdamW step with BF16 working-copy emission.                   */
/*   skip    : [CH20] §20.2.2 / [MP] "Gradient 和 Loss Scaling": a step whose */
/*             scaled gradients hold inf/NaN changes nothing.                */
/*   master  : [CH20] §20.5.13 and [MP] "为什么需要 FP32 Master Weights":     */
/*             the optimizer updates an fp32 copy, then casts it to bf16.    */
/*   state   : [MP06] §三: fp32 master 4 + m 4 + v 4 = 12 bytes/param.        */
/*   AdamW   : decoupled weight decay, bias-corrected moments (see header).  */
/* amax_slot[t] >= 0 also folds max|bf16| of tensor t into amax[slot]        */
/* (NaN-propagating), the input of the FP8 weight quantizer.                 */
/* ------------------------------------------------------------------------ */
void orc_adamw_master_step_clip(int n_tensors, float *const *master, float *const *exp_avg,
                                float *const *exp_avg_sq, void *const *grads, int gdtype,
                                uint16_t *const *bf16_out, const int64_t *numel,
                                const float *scale, int32_t found_inf, int32_t *step,
                                double lr, double beta1, double beta2, double eps, double wd,
                                const int32_t *amax_slot, float *amax, float clip_coef);
void orc_adamw_master_step_ex(int n_tensors, float *const *master, float *const *exp_avg,
                              float *const *exp_avg_sq, void *const *grads, int gdtype,
                              uint16_t *const *bf16_out, const int64_t *numel,
                              const float *scale, int32_t found_inf, int32_t *step,
                              double lr, double beta1, double beta2, double eps, double wd,
                              const int32_t *amax_slot, float *amax, float clip_coef,
                              int stochastic, uint64_t seed);
static uint32_t sr_bits(uint64_t seed, int32_t step, int32_t tensor, int64_t k);
uint16_t orc_bf16_stochastic(float p, uint32_t u);

void orc_adamw_master_step(int n_tensors, float *const *master, float *const *exp_avg,
                           float *const *exp_avg_sq, void *const *grads, int gdtype,
                           uint16_t *const *bf16_out, const int64_t *numel,
                           const float *scale, int32_t found_inf, int32_t *step,
                           double lr, double beta1, double beta2, double eps, double wd,
                           const int32_t *amax_slot, float *amax)
{
    orc_adamw_master_step_clip(n_tensors, master, exp_avg, exp_avg_sq, grads, gdtype, bf16_out,
                               numel, scale, found_inf, step, lr, beta1, beta2, eps, wd,
                               amax_slot, amax, 1.0f);
}

/* As above; every unscaled gradient is first multiplied by clip_coef (fp32),
 * the clipping factor of orc_clip_coef (1.0 leaves it unchanged). */
void orc_adamw_master_step_clip(int n_tensors, float *const *master, float *const *exp_avg,
                                float *const *exp_avg_sq, void *const *grads, int gdtype,
                                uint16_t *const *bf16_out, const int64_t *numel,
                                const float *scale, int32_t found_inf, int32_t *step,
                                double lr, double beta1, double beta2, double eps, double wd,
                                const int32_t *amax_slot, float *amax, float clip_coef)
{
    orc_adamw_master_step_ex(n_tensors, master, exp_avg, exp_avg_sq, grads, gdtype, bf16_out,
                             numel, scale, found_inf, step, lr, beta1, beta2, eps, wd, amax_slot,
                             amax, clip_coef, 0, 0);
}

/* As above; with stochastic != 0 the bf16 copy is rounded stochastically
 * (orc_bf16_stochastic, random bits of element k of tensor i at the new step
 * count t from sr_bits(seed, t, i, k)) instead of to nearest-even. */
/* As orc_adamw_master_step_ex; sr_ids[i] (when not NULL) replaces i as the
 * tensor word of the bf16 copy's random counter.  The delayed FP8 step walks
 * its plain tensors and its FP8 weights as two lists: plain tensor p uses p,
 * FP8 weight j uses j | 2^30. */
void orc_adamw_master_step_ids(int n_tensors, float *const *master, float *const *exp_avg,
                               float *const *exp_avg_sq, void *const *grads, int gdtype,
                               uint16_t *const *bf16_out, const int64_t *numel,
                               const float *scale, int32_t found_inf, int32_t *step,
                               double lr, double beta1, double beta2, double eps, double wd,
                               const int32_t *amax_slot, float *amax, float clip_coef,
                               int stochastic, uint64_t seed, const int32_t *sr_ids);

void orc_adamw_master_step_ex(int n_tensors, float *const *master, float *const *exp_avg,
                              float *const *exp_avg_sq, void *const *grads, int gdtype,
                              uint16_t *const *bf16_out, const int64_t *numel,
                              const float *scale, int32_t found_inf, int32_t *step,
                              double lr, double beta1, double beta2, double eps, double wd,
                              const int32_t *amax_slot, float *amax, float clip_coef,
                              int stochastic, uint64_t seed)
{
    orc_adamw_master_step_ids(n_tensors, master, exp_avg, exp_avg_sq, grads, gdtype, bf16_out,
                              numel, scale, found_inf, step, lr, beta1, beta2, eps, wd, amax_slot,
                              amax, clip_coef, stochastic, seed, NULL);
}

void orc_adamw_master_step_ids(int n_tensors, float *const *master, float *const *exp_avg,
                               float *const *exp_avg_sq, void *const *grads, int gdtype,
                               uint16_t *const *bf16_out, const int64_t *numel,
                               const float *scale, int32_t found_inf, int32_t *step,
                               double lr, double beta1, double beta2, double eps, double wd,
                               const int32_t *amax_slot, float *amax, float clip_coef,
                               int stochastic, uint64_t seed, const int32_t *sr_ids)
{
    if (found_inf)
        return; /* skipped step: no state, output or counter changes */

    /* per-step scalars: fp64, each rounded once to fp32 */
    int32_t t = *step + 1;
    double bc1 = 1.0 - pow(beta1, (double)t);
    double bc2 = 1.0 - pow(beta2, (double)t);
    float step_size = (float)(lr / bc1);
    float bc2_sqrt = (float)sqrt(bc2);
    float decay = (float)(1.0 - lr * wd);
    float b1 = (float)beta1, omb1 = (float)(1.0 - beta1);
    float b2 = (float)beta2, omb2 = (float)(1.0 - beta2);
    float epsf = (float)eps;
    float inv_s = scale ? 1.0f / *scale : 1.0f;

    for (int i = 0; i < n_tensors; ++i) {
        int slot = amax_slot ? amax_slot[i] : -1;
        for (int64_t k = 0; k < numel[i]; ++k) {
            float g = (load_as_f32(gdtype, grads[i], k) * inv_s) * clip_coef;
            float p = master[i][k], m = exp_avg[i][k], v = exp_avg_sq[i][k];
            p = p * decay;
            m = b1 * m + omb1 * g;
            v = b2 * v + omb2 * (g * g);
            float denom = sqrtf(v) / bc2_sqrt + epsf;
            p = p - step_size * (m / denom);
            master[i][k] = p;
            exp_avg[i][k] = m;
            exp_avg_sq[i][k] = v;
            if (bf16_out && bf16_out[i]) {
                int32_t id = sr_ids ? sr_ids[i] : i;
                uint16_t b = stochastic ? orc_bf16_stochastic(p, sr_bits(seed, t, id, k))
                                        : (uint16_t)fmt_encode(&FMT_BF16, (double)p);
                bf16_out[i][k] = b;
                if (slot >= 0) {
                    float a = fabsf((float)fmt_decode(&FMT_BF16, b));
                    if (isnan(a) || isnan(amax[slot]))
                        amax[slot] = NAN;
                    else if (a > amax[slot])
                        amax[slot] = a;
                }
            }
        }
    }
    *step = t;
}

/* ------------------------------------------------------------------------ */
/* Tensorwise dynamic FP8 quantization, [FP8] §2:                            */
/*   amax  = max |x| in fp32                                                 */
/*   scale = fp8_max / max(double(amax), EPS)          (fp64)                */
/*   q     = to_fp8(clamp(x_f32 * scale, -fp8_max, fp8_max))                 */
/*   inv_scale = 1 / scale                             (exported as fp32)    */
/* e4m3fn (max 448) for weights/activations, e5m2 (max 57344) for gradients  */
/* ([FP8] §3).  out_t is the same bytes laid out [cols, rows] row-major, the  */
/* column-major copy the backward GEMMs consume ([FP8] §4 _to_col_major).    */
/* x is [rows, cols] row-major of dtype xdtype (f32, f16 or bf16).           */
/* amax_given != 0 takes *amax as given instead of computing it.             */
/* ------------------------------------------------------------------------ */
void orc_fp8_quant_tensorwise(const void *x, int xdtype, int64_t rows, int64_t cols,
                              int fp8_dtype, double eps, uint8_t *out, uint8_t *out_t,
                              float *inv_scale, float *amax, int amax_given)
{
    const orc_fmt *f = fmt_of(fp8_dtype);
    int64_t n = rows * cols;
    float a = 0.0f;
    if (amax_given) {
        a = *amax;
    } else {
        for (int64_t k = 0; k < n; ++k) {
            float v = fabsf(load_as_f32(xdtype, x, k));
            if (isnan(v) || isnan(a))
                a = NAN;
            else if (v > a)
                a = v;
        }
        *amax = a;
    }
    double fmax = fmt_max(f);
    double ad = (double)a;
    double clamped = isnan(ad) ? ad : (ad < eps ? eps : ad); /* NaN propagates */
    double scale_d = fmax / clamped;
    float s32 = (float)scale_d;          /* the fp32 multiply uses scale as fp32 */
    *inv_scale = (float)(1.0 / scale_d);
    float lo = (float)-fmax, hi = (float)fmax;
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t j = 0; j < cols; ++j) {
            float y = load_as_f32(xdtype, x, i * cols + j) * s32;
            if (!isnan(y))
                y = y < lo ? lo : (y > hi ? hi : y);
            uint8_t q = (uint8_t)fmt_encode(f, (double)y);
            out[i * cols + j] = q;
            if (out_t)
                out_t[j * rows + i] = q;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Rowwise FP8 scaling.  "FP8训练：量化、自动微分、Torchao" §1: instead of one   */
/* scale per tensor, every row gets its own scale (§2's formula per row).     */
/* §4: the backward GEMMs consume the column-major copy, whose reduction runs */
/* along the rows of x - so that copy carries one scale per column of x (a    */
/* per-row scale would vary along its reduction dimension).  Reading: out has */
/* per-row scales, out_t (= [cols, rows] row-major) per-column scales.         */
/* Each scale is §2's scale_d = fp8_max / max(double(amax), EPS) of its own   */
/* row or column; the cast is §2's clamp and RNE.                              */
/* ------------------------------------------------------------------------ */
static double nan_max_abs_update(double acc, float v)
{
    float a = fabsf(v);
    if (isnan(a) || isnan(acc))
        return NAN;
    return a > acc ? a : acc;
}

static uint8_t cast_scaled(const orc_fmt *f, float x, float s32)
{
    double fmax = fmt_max(f);
    float lo = (float)-fmax, hi = (float)fmax;
    float y = x * s32;
    if (!isnan(y))
        y = y < lo ? lo : (y > hi ? hi : y);
    return (uint8_t)fmt_encode(f, (double)y);
}

static void scale_of(double fmax, double eps, float amax, float *s32, float *inv)
{
    double ad = (double)amax;
    double cl = isnan(ad) ? ad : (ad < eps ? eps : ad);
    double sd = fmax / cl;
    *s32 = (float)sd;
    *inv = (float)(1.0 / sd);
}

void orc_fp8_quant_rowwise(const void *x, int xdtype, int64_t rows, int64_t cols, int fp8_dtype,
                           double eps, uint8_t *out, uint8_t *out_t, float *amax_row,
                           float *scale_row, float *inv_row, float *amax_col, float *scale_col,
                           float *inv_col)
{
    const orc_fmt *f = fmt_of(fp8_dtype);
    double fmax = fmt_max(f);
    for (int64_t i = 0; i < rows; ++i) {
        double a = 0.0;
        for (int64_t j = 0; j < cols; ++j)
            a = nan_max_abs_update(a, load_as_f32(xdtype, x, i * cols + j));
        amax_row[i] = (float)a;
        scale_of(fmax, eps, amax_row[i], &scale_row[i], &inv_row[i]);
        for (int64_t j = 0; j < cols; ++j)
            out[i * cols + j] = cast_scaled(f, load_as_f32(xdtype, x, i * cols + j), scale_row[i]);
    }
    if (!out_t)
        return;
    for (int64_t j = 0; j < cols; ++j) {
        double a = 0.0;
        for (int64_t i = 0; i < rows; ++i)
            a = nan_max_abs_update(a, load_as_f32(xdtype, x, i * cols + j));
        amax_col[j] = (float)a;
        scale_of(fmax, eps, amax_col[j], &scale_col[j], &inv_col[j]);
        for (int64_t i = 0; i < rows; ++i)
            out_t[j * rows + i] = cast_scaled(f, load_as_f32(xdtype, x, i * cols + j), scale_col[j]);
    }
}

/* ------------------------------------------------------------------------ */
/* Group-wise FP8 scaling.  "第20章 量化与混合精度训练" §20.5.18: a weight     */
/* [out, in] is cut into groups of `group` consecutive elements along in, each */
/* with its own scale (g128: scales of shape [out, in / 128]).  Reading: §2's  */
/* recipe of "FP8训练：量化、自动微分、Torchao" per group - amax of the group,  */
/* scale_d = fp8_max / max(double(amax), EPS), clamp and RNE cast.  The        */
/* column-major copy out_t ([cols, rows], §4) feeds the backward GEMM, whose   */
/* reduction runs along the rows of x, so its groups are `group` consecutive   */
/* rows within one column (scales of shape [cols, rows / group]).  The last    */
/* group of a row (column) holds the remaining cols % group (rows % group).    */
/*   *_rg: [rows, ceil(cols / group)] row-major; *_cg: [cols, ceil(rows /     */
/*   group)] row-major.                                                       */
/* ------------------------------------------------------------------------ */
void orc_fp8_quant_groupwise(const void *x, int xdtype, int64_t rows, int64_t cols, int64_t group,
                             int fp8_dtype, double eps, uint8_t *out, uint8_t *out_t,
                             float *amax_rg, float *scale_rg, float *inv_rg, float *amax_cg,
                             float *scale_cg, float *inv_cg)
{
    const orc_fmt *f = fmt_of(fp8_dtype);
    double fmax = fmt_max(f);
    int64_t ngc = (cols + group - 1) / group, ngr = (rows + group - 1) / group;
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t g = 0; g < ngc; ++g) {
            int64_t j0 = g * group, j1 = j0 + group < cols ? j0 + group : cols;
            double a = 0.0;
            for (int64_t j = j0; j < j1; ++j)
                a = nan_max_abs_update(a, load_as_f32(xdtype, x, i * cols + j));
            int64_t k = i * ngc + g;
            amax_rg[k] = (float)a;
            scale_of(fmax, eps, amax_rg[k], &scale_rg[k], &inv_rg[k]);
            for (int64_t j = j0; j < j1; ++j)
                out[i * cols + j] = cast_scaled(f, load_as_f32(xdtype, x, i * cols + j), scale_rg[k]);
        }
    }
    if (!out_t)
        return;
    for (int64_t j = 0; j < cols; ++j) {
        for (int64_t g = 0; g < ngr; ++g) {
            int64_t i0 = g * group, i1 = i0 + group < rows ? i0 + group : rows;
            double a = 0.0;
            for (int64_t i = i0; i < i1; ++i)
                a = nan_max_abs_update(a, load_as_f32(xdtype, x, i * cols + j));
            int64_t k = j * ngr + g;
            amax_cg[k] = (float)a;
            scale_of(fmax, eps, amax_cg[k], &scale_cg[k], &inv_cg[k]);
            for (int64_t i = i0; i < i1; ++i)
                out_t[j * rows + i] = cast_scaled(f, load_as_f32(xdtype, x, i * cols + j), scale_cg[k]);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Stochastic rounding of the bf16 working copy.  "第20章 量化与混合精度训练"  */
/* §20.5.14: instead of round-to-nearest, round down or up with probability   */
/* proportional to the distance, so the expected value is the input.  For a  */
/* finite fp32 p between two neighbouring bf16 values lo (toward zero) and hi */
/* (away from zero, inf beyond the largest finite), the result is hi with     */
/* probability (|p| - |lo|) / (|hi| - |lo|): with 16 uniform random bits u,    */
/* hi exactly when u < the 16 low bits of p's magnitude pattern.  NaN gives   */
/* the canonical NaN, values already on the grid stay.                        */
/*                                                                            */
/* Random bits: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random   */
/* numbers: as easy as 1, 2, 3", SC 2011): a 4x32-bit counter, a 2x32-bit key, */
/* ten rounds of two 32x32->64 multiplies and xors, key bumped by the golden-  */
/* ratio and sqrt(3)-1 Weyl constants between rounds.                          */
/* Counter of element k of tensor t at optimizer step s: {k/8 low, k/8 high,   */
/* s, t}; key = the 64-bit seed {low, high}; element k takes the 16-bit half    */
/* (k%8)%2 (low half first) of output word (k%8)/2.                            */
/* ------------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* the 16 random bits of element k */
static uint32_t sr_bits(uint64_t seed, int32_t step, int32_t tensor, int64_t k)
{
    uint64_t grp = (uint64_t)k >> 3;
    uint32_t ctr[4] = {(uint32_t)grp, (uint32_t)(grp >> 32), (uint32_t)step, (uint32_t)tensor};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    orc_philox4x32_10(ctr, key, o);
    int lane = (int)(k & 7);
    uint32_t w = o[lane >> 1];
    return (lane & 1) ? (w >> 16) : (w & 0xFFFFu);
}

/* stochastic rounding of p to bf16 with the random 16 bits u */
uint16_t orc_bf16_stochastic(float p, uint32_t u)
{
    if (isnan(p))
        return (uint16_t)FMT_BF16.nan_code;
    uint32_t bits;
    memcpy(&bits, &p, 4);
    uint32_t sign = bits & 0x80000000u, mag = bits & 0x7FFFFFFFu;
    uint32_t lo = mag >> 16, frac = mag & 0xFFFFu;
    uint32_t r = lo + ((u & 0xFFFFu) < frac ? 1u : 0u);  /* P(up) = frac / 2^16 */
    return (uint16_t)((sign >> 16) | r);
}

void orc_bf16_stochastic_list(const float *p, uint16_t *out, int64_t n, uint64_t seed,
                              int32_t step, int32_t tensor)
{
    for (int64_t k = 0; k < n; ++k)
        out[k] = orc_bf16_stochastic(p[k], sr_bits(seed, step, tensor, k));
}

/* ------------------------------------------------------------------------ */
/* Stochastic rounding of the FP8 weight copies.  "第20章 量化与混合精度训练"  */
/* §20.5.14 rounds down or up with probability proportional to the distance  */
/* (so the expected value is the input) and says it matters most the lower   */
/* the precision, FP8 and FP4 included.  Reading: [FP8] §2's quantizer with   */
/* its round-to-nearest cast replaced by that rule, drawn with 16 random bits */
/* per element as for the bf16 copy:                                          */
/*   y = x_f32 * scale (fp32), clamped to +-fp8_max, NaN propagating;         */
/*   lo <= |y| < hi: the neighbouring FP8 magnitudes (|y| = fp8_max or on the */
/*   grid: the result is |y| itself);                                        */
/*   result = sign(y) * hi with probability                                   */
/*       floor(2^16 * (|y| - lo) / (hi - lo)) / 2^16,                         */
/*   else sign(y) * lo; NaN gives the canonical NaN.                          */
/* With 16 uniform random bits u the result is hi exactly when u is below    */
/* that numerator.  The probability is the distance ratio itself whenever the */
/* ratio is a multiple of 2^-16, else the ratio truncated to one: the mean is */
/* then low by less than 2^-16 of a quantum.  (The bf16 copy's rule is exact, */
/* since bf16 drops exactly 16 bits of an fp32 value; a scaled FP8 input      */
/* keeps up to 21 bits below the FP8 quantum.)                                */
/* Random bits: element k (row-major index within its tensor) takes the      */
/* 16-bit draw that the bf16 copy's layout assigns it (sr_bits above: half    */
/* (k%8)%2, low first, of Philox output word (k%8)/2 at counter {k/8 low,     */
/* k/8 high, step, w}, key = seed) with w = tensor | 2^31; bit 31 keeps these */
/* draws apart from the bf16 copy's, whose tensor words stay below 2^31.      */
/* The transposed copy holds the same bytes as the row-major one (one draw    */
/* per element).                                                              */
/* ------------------------------------------------------------------------ */

/* ascending finite non-negative magnitudes of an FP8 format (at most 128) */
static int fp8_grid(const orc_fmt *f, double *g)
{
    int n = 0;
    uint32_t codes = 1u << (f->ebits + f->mbits);   /* codes with sign bit clear */
    for (uint32_t c = 0; c < codes; ++c) {
        double v = fmt_decode(f, c);
        if (isfinite(v))
            g[n++] = v;                              /* decode is monotone in c */
    }
    return n;
}

uint8_t orc_fp8_stochastic(int fp8_dtype, float y, uint32_t u)
{
    const orc_fmt *f = fmt_of(fp8_dtype);
    if (isnan(y))
        return (uint8_t)f->nan_code;
    double grid[256];
    int n = fp8_grid(f, grid);
    double a = fabs((double)y), fmax = fmt_max(f);
    if (a > fmax)
        a = fmax;
    int i = 0;                                       /* largest grid[i] <= a */
    while (i + 1 < n && grid[i + 1] <= a)
        ++i;
    double r = grid[i];
    if (r < a) {
        double ratio = (a - grid[i]) / (grid[i + 1] - grid[i]);   /* exact: the gap is 2^k */
        double num = floor(ratio * 65536.0);
        if ((double)(u & 0xFFFFu) < num)
            r = grid[i + 1];
    }
    return (uint8_t)fmt_encode(f, signbit(y) ? -r : r);
}

static uint32_t sr8_bits(uint64_t seed, int32_t step, int32_t tensor, int64_t k)
{
    return sr_bits(seed, step, (int32_t)((uint32_t)tensor | 0x80000000u), k);
}

/* orc_fp8_quant_tensorwise with the stochastic cast: the same amax, scale and
 * inv_scale; element k of tensor `tensor` at optimizer step `step` rounds
 * with sr8_bits(seed, step, tensor, k). */
void orc_fp8_quant_tensorwise_sr(const void *x, int xdtype, int64_t rows, int64_t cols,
                                 int fp8_dtype, double eps, uint8_t *out, uint8_t *out_t,
                                 float *inv_scale, float *amax, int amax_given, uint64_t seed,
                                 int32_t step, int32_t tensor)
{
    const orc_fmt *f = fmt_of(fp8_dtype);
    int64_t n = rows * cols;
    float a = 0.0f;
    if (amax_given) {
        a = *amax;
    } else {
        for (int64_t k = 0; k < n; ++k) {
            float v = fabsf(load_as_f32(xdtype, x, k));
            if (isnan(v) || isnan(a))
                a = NAN;
            else if (v > a)
                a = v;
        }
        *amax = a;
    }
    double fmax = fmt_max(f);
    double ad = (double)a;
    double clamped = isnan(ad) ? ad : (ad < eps ? eps : ad);
    double scale_d = fmax / clamped;
    float s32 = (float)scale_d;
    *inv_scale = (float)(1.0 / scale_d);
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t j = 0; j < cols; ++j) {
            int64_t k = i * cols + j;
            float y = load_as_f32(xdtype, x, k) * s32;
            uint8_t q = orc_fp8_stochastic(fp8_dtype, y, sr8_bits(seed, step, tensor, k));
            out[k] = q;
            if (out_t)
                out_t[j * rows + i] = q;
        }
    }
}

/* the 16 random bits of element k (exported for the pin tests) */
uint32_t orc_sr8_bits(uint64_t seed, int32_t step, int32_t tensor, int64_t k)
{
    return sr8_bits(seed, step, tensor, k);
}

void orc_fp8_stochastic_list(int fp8_dtype, const float *y, const uint32_t *u, uint8_t *out,
                             int64_t n)
{
    for (int64_t k = 0; k < n; ++k)
        out[k] = orc_fp8_stochastic(fp8_dtype, y[k], u[k]);
}

void orc_sr8_bits_list(uint64_t seed, int32_t step, int32_t tensor, int64_t k0, int64_t n,
                       uint32_t *out)
{
    for (int64_t k = 0; k < n; ++k)
        out[k] = sr8_bits(seed, step, tensor, k0 + k);
}
