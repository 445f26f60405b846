/*
 * ampfp8.h - C ABI of libampfp8.so: the per-step mixed-precision optimizer
 * pipeline on one GPU (sm_103a).
 *
 *   amp_unscale_check        scaled low-precision gradients -> found_inf flag
 *   amp_adamw_master_step    skip-on-inf + unscale + FP32-master AdamW
 *                            + BF16 working copy (+ per-tensor amax fold)
 *   fp8_quant_tensorwise     tensorwise dynamic FP8 cast (+ transposed copy)
 *   fp8_quant_tensorwise_list  the same over a list of 2-D tensors
 *   amp_update_scale         dynamic loss-scale state machine
 *
 * Sources the operations follow (page title, section):
 *   [CH20]  "第20章 量化与混合精度训练": §20.2.2 GradScaler, §20.5.13 Master
 *           Weights, §20.5.33 GradScaler 的 _growth_tracker 状态机细节.
 *   [MP]    "从 AMP 到 Mixed Precision：训练和推理为什么不使用同一种精度":
 *           "Gradient 和 Loss Scaling", "为什么需要 FP32 Master Weights",
 *           "PyTorch AMP 与 FP32 Master Weights" (mode B: bf16 params + fp32 master).
 *   [FP8]   "FP8训练：量化、自动微分、Torchao": §2 量化数学, §3 格式选择,
 *           §4 _scaled_mm 布局要求.
 *   [NOTES] "AMP：Automatic Mixed Precision 技术笔记": §4 GradScaler.
 *   [MP06]  "06 · 混合精度": §三 (12 bytes/param of fp32 master + m + v),
 *           §四 Loss Scaling.
 *
 * Conventions shared by every entry point
 *   - Every pointer named *_dev, and every tensor a list refers to, is device
 *     memory owned by the caller.  Tensors are contiguous; 16-bit and 8-bit
 *     floating-point data are raw bit patterns.
 *   - Every call is asynchronous: it validates its arguments on the host,
 *     enqueues kernels on `stream` (NULL = the legacy default stream) and
 *     returns.  No per-step call synchronises the host with the device or
 *     allocates device memory; only the set-up calls on tensor lists do.
 *   - A negative status means nothing was enqueued (argument errors), or
 *     that a launch failed (AMP_ECUDA).  amp_last_error() then returns a
 *     message for the calling thread.  Faults inside kernels surface at the
 *     caller's next synchronisation, as for any CUDA work.
 *   - Calls that touch the same buffers must be ordered on one stream (or
 *     by events); the library takes no locks.
 *   - Within one call, buffers that are only read (x, grads) must not
 *     overlap buffers the call writes; only the buffers named as updated in
 *     place (master, m, v) are both read and written.
 *   - Pointers need no particular alignment: tensors whose addresses allow
 *     16-byte vector access take the vector path, others a scalar path that
 *     gives the same bits.
 *   - Kernels are launched as programmatic dependent launches: a kernel may
 *     be scheduled while the one before it in the stream drains, but waits
 *     (griddepcontrol.wait) for that kernel to complete before it touches
 *     memory, so results are those of plain stream order.  Other work on the
 *     stream, before or after, runs in plain stream order.
 *   - Every call opens an NVTX range named after itself, for profilers.
 */
#ifndef AMPFP8_H
#define AMPFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; declared here so the header needs
 * no CUDA include. */
typedef struct CUstream_st *amp_stream_t;

typedef enum {
    AMP_OK = 0,
    AMP_EINVAL = -1,  /* null pointer, negative or too large size (a side >= 2^48 or rows*cols past int64), mismatched list shapes */
    AMP_EDTYPE = -2,  /* element type not accepted by this entry point */
    AMP_ECUDA = -4,   /* a CUDA runtime call or kernel launch failed */
    AMP_ENOMEM = -5,  /* device allocation in amp_tensor_list_create failed */
    AMP_ETIMEOUT = -6 /* a kernel's bounded wait gave up (see amp_tensor_list_check) */
} amp_status;

typedef enum {
    AMP_DT_F32 = 1,
    AMP_DT_F16 = 2,     /* IEEE binary16 */
    AMP_DT_BF16 = 3,    /* bfloat16 */
    AMP_DT_E4M3FN = 4,  /* OCP FP8 E4M3, finite + NaN (max 448) */
    AMP_DT_E5M2 = 5     /* OCP FP8 E5M2, IEEE-like (max 57344) */
} amp_dtype;

/* ------------------------------------------------------------------------ */
/* Tensor lists.  Every step of the pages runs over all of a model's          */
/* parameters or gradients ([CH20] §20.2.2, [NOTES] §4, [MP06] §四); a handle */
/* is that list on the device.  Its layout has no counterpart on the pages.   */
/* ------------------------------------------------------------------------ */

/* Opaque handle describing a ragged list of n contiguous device tensors of
 * one dtype.  It owns only one device block with its copies of the pointer
 * and size arrays, the chunk table the list kernels walk (and, for 2-D
 * lists, the tile table of the FP8 kernels); it never owns tensor data. */
typedef struct amp_tensor_list_s *amp_tensor_list;

/* Create a list handle.
 *   n        number of tensors, >= 0
 *   dev_ptrs host array[n] of device pointers (a pointer may be NULL only
 *            when its tensor is empty)
 *   rows     host array[n]: element counts of 1-D tensors, or row counts
 *            when `cols` is given
 *   cols     host array[n] of column counts (2-D, row-major), or NULL
 *   dtype    element type of every tensor
 *   stream   the device block is filled with cudaMemcpyAsync on it
 * Allocates the device block with cudaMalloc (the only allocating call of
 * the library) and waits for the upload on `stream` (a one-time set-up
 * call, unlike the per-step entry points below).  Returns AMP_EINVAL for n < 0, a null array, a negative
 * size or a NULL pointer of a non-empty tensor; AMP_ENOMEM if allocation
 * fails.  *out is set only on success. */
amp_status amp_tensor_list_create(int n, void *const *dev_ptrs, const int64_t *rows,
                                  const int64_t *cols, amp_dtype dtype,
                                  amp_stream_t stream, amp_tensor_list *out);

/* Per-tensor amax slots of a list.  On the bf16 output of
 * amp_adamw_master_step (and amp_emit_bf16): slots[i] >= 0 folds max|bf16| of
 * tensor i into amax_dev[slots[i]]; -1 (the default) does not.  On the x list
 * of fp8_quant_tensorwise_list(_sr) (every slot >= 0): tensor i takes its
 * amax from, and writes its inv_scale to, entry slots[i] instead of i - so
 * the pieces of weights sharded over ranks can use the weights' global
 * numbering.  Host array[n], copied to the handle's device block on `stream`
 * (waits for the copy: set-up call). */
amp_status amp_tensor_list_set_amax_slots(amp_tensor_list list, const int32_t *slots,
                                          amp_stream_t stream);

/* Health check.  The AdamW kernels stream through shared memory with
 * asynchronous bulk copies whose completion they wait for with a time limit
 * (one second of GPU time) instead of forever; a wait that gives up leaves
 * its chunk not updated and sets a sticky error word in the device block of
 * the list that holds the step scalars: `master` for amp_adamw_master_step
 * and its _clip / _sr forms, `fp8_out` for amp_adamw_master_step_fp8_delayed.
 * This call waits for `stream`, reads and clears that word, and returns
 * AMP_ETIMEOUT if it was set, AMP_OK otherwise. */
amp_status amp_tensor_list_check(amp_tensor_list list, amp_stream_t stream);

/* Self-test of the bounded wait: one CTA waits on a barrier that nothing
 * completes, gives up after limit_seconds (0 < limit <= 10) of GPU time and
 * writes *err_dev = 1 (0 would mean the barrier completed).  No fault, no
 * hang; the context stays usable.  The pages have no counterpart. */
amp_status amp_selftest_bounded_wait(int32_t *err_dev, double limit_seconds, amp_stream_t stream);

/* Release the handle and its device block (cudaFree; synchronises the
 * device like any cudaFree).  NULL is accepted. */
amp_status amp_tensor_list_destroy(amp_tensor_list list);

/* Feed and read back a list from host memory.  The pages have no counterpart
 * (they run on framework tensors); these let a caller with host buffers drive
 * the step through this ABI alone.
 *   host_ptrs  n host pointers; host_ptrs[i] holds numel[i] elements of the
 *              list dtype (may be NULL for an empty tensor)
 * One cudaMemcpyAsync per non-empty tensor, in list order, on `stream`.  With
 * page-locked host memory (cudaHostAlloc / cudaHostRegister) the copies are
 * asynchronous; with pageable memory CUDA stages them and the call may return
 * only after they are done.  All pointers are checked before the first copy
 * (AMP_EINVAL, nothing enqueued); a copy that fails to enqueue returns
 * AMP_ECUDA with the earlier copies already enqueued. */
amp_status amp_tensor_list_copy_from_host(amp_tensor_list list, const void *const *host_ptrs,
                                          amp_stream_t stream);
amp_status amp_tensor_list_copy_to_host(amp_tensor_list list, void *const *host_ptrs,
                                        amp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* A1: unscale + non-finite check.  [CH20] §20.2.2, [MP] "Gradient 和 Loss    */
/* Scaling", [NOTES] §4 steps 3-4: before the optimizer the scaled gradients  */
/* are divided by S and inspected for inf/NaN.                                */
/* ------------------------------------------------------------------------ */

/* found_inf_dev |= OR over all elements of !isfinite(float(g) * (1/S)),
 * where 1/S is the correctly rounded fp32 reciprocal of *scale_dev (S = 1
 * when scale_dev is NULL).  The flag (int32, 0/1) is never cleared here, so
 * several lists can be checked into one flag; amp_update_scale clears it.
 *   grads    list of AMP_DT_F16, AMP_DT_BF16 or AMP_DT_F32 tensors
 *   inplace  0: read-only check (2 bytes/elt for 16-bit grads);
 *            1: also store g * (1/S) back, rounded to nearest-even in the
 *               gradient dtype (NaN as the canonical quiet NaN).
 * Errors: AMP_EINVAL (null list / flag), AMP_EDTYPE (fp8 list). */
amp_status amp_unscale_check(amp_tensor_list grads, const float *scale_dev,
                             int32_t *found_inf_dev, int inplace, amp_stream_t stream);

/* Gradient-norm clipping input ("AMP：Automatic Mixed Precision 技术笔记" §6,
 * "06 · 混合精度" §四: unscale first, then clip_grad_norm_).  Does everything
 * amp_unscale_check does (inplace = 0) and also writes
 *     *grad_sumsq_dev = sum over all elements of (float(g) * (1/S))^2   (fp64)
 * for amp_adamw_master_step_clip.  Each thread squares the stored values
 * (exact in fp32 for 16-bit gradients) in fused multiply-add chains of four,
 * adds the chain sums in compensated fp32, and chunks and the final total are
 * added in fp64 in a fixed order, so the value does not depend on scheduling;
 * (1/S)^2 is applied per chunk in fp64, which equals squaring the unscaled
 * fp32 gradient while 1/S is a power of two.  Relative error <= 6 ulp of
 * fp32 (3.6e-7).  A non-finite gradient makes the sum NaN (found_inf is set
 * and the step is skipped); squared fp32 gradients above 3.4e38 overflow the
 * per-thread sums.  The list handle's per-chunk scratch holds the partial
 * sums: calls on one list must not overlap on the GPU.
 * Errors: AMP_EINVAL (NULL argument), AMP_EDTYPE (fp8 list). */
amp_status amp_unscale_check_norm(amp_tensor_list grads, const float *scale_dev,
                                  int32_t *found_inf_dev, double *grad_sumsq_dev,
                                  amp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* A2-A6: skip decision + FP32-master AdamW + BF16 emission + amax fold.     */
/* [CH20] §20.5.13, [MP] "为什么需要 FP32 Master Weights" / "PyTorch AMP 与   */
/* FP32 Master Weights" mode B, [MP06] §三 12 bytes/param.                    */
/* ------------------------------------------------------------------------ */

/* AdamW hyper-parameters, as the user states them (fp64). */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
} amp_adamw_hyper;

/* If found_inf_dev is non-NULL and *found_inf_dev != 0 the step is skipped:
 * nothing below is written and *step_dev is unchanged.  Otherwise, with
 * t = *step_dev + 1 and per-step scalars computed once in fp64 and rounded
 * to fp32 (step_size = lr / (1 - beta1^t), c2 = sqrt(1 - beta2^t)), every
 * element does in fp32, each operation rounded to nearest-even and none
 * fused:
 *     g = float(grad) * (1/S)
 *     p = p * (1 - lr*wd)
 *     m = beta1*m + (1-beta1)*g
 *     v = beta2*v + (1-beta2)*(g*g)
 *     p = p - step_size * (m / (sqrt(v)/c2 + eps))
 * then bf16_out = RNE(p), and *step_dev = t.  The constants (1 - lr*wd),
 * (1-beta1), (1-beta2) are formed in fp64 and rounded once to fp32.
 *   master, exp_avg, exp_avg_sq  AMP_DT_F32 lists, updated in place
 *   grads      AMP_DT_F16 / AMP_DT_BF16 / AMP_DT_F32 list (scaled by S)
 *   bf16_out   AMP_DT_BF16 list or NULL; tensors with an amax slot also do
 *              amax_dev[slot] = max(amax_dev[slot], |bf16|) (fp32 bits,
 *              NaN-propagating), which the caller must have zeroed
 *              (amp_update_scale does at the end of each step)
 *   scale_dev  fp32 S, or NULL for S = 1
 *   step_dev   int32 count of completed (non-skipped) steps
 * All lists must have the same tensor count and element counts.
 * Errors: AMP_EINVAL (null / mismatched lists, null step or hyper, slots
 * without amax_dev), AMP_EDTYPE (wrong list dtypes). */
amp_status amp_adamw_master_step(amp_tensor_list master, amp_tensor_list exp_avg,
                                 amp_tensor_list exp_avg_sq, amp_tensor_list grads,
                                 amp_tensor_list bf16_out, const float *scale_dev,
                                 const int32_t *found_inf_dev, int32_t *step_dev,
                                 const amp_adamw_hyper *hyper, float *amax_dev,
                                 amp_stream_t stream);

/* A5 on its own ("从 AMP 到 Mixed Precision" sections "为什么需要 FP32 Master
 * Weights" and "PyTorch AMP 与 FP32 Master Weights", mode B: the model's bf16
 * parameters are the fp32 master rounded to bf16).  The AdamW entry points
 * emit this copy after every step; this call makes it before the first one,
 * for the first forward pass and, with amax slots, for the first amax of the
 * FP8 weights (the opening entry of a delayed-scaling history):
 *     bf16_out = RNE(master)   (NaN -> 0x7FC0)
 *     amax_dev[slot] = max(amax_dev[slot], |bf16|) for tensors with a slot
 *                   (amp_tensor_list_set_amax_slots on bf16_out; fp32 bits,
 *                   NaN propagating; the caller zeroes amax_dev first)
 *   master    AMP_DT_F32 list (read only)
 *   bf16_out  AMP_DT_BF16 list with master's tensor count and sizes
 * 6 bytes per element, one launch.
 * Errors: AMP_EINVAL (NULL / mismatched lists, slots without amax_dev),
 * AMP_EDTYPE (wrong list dtypes). */
amp_status amp_emit_bf16(amp_tensor_list master, amp_tensor_list bf16_out, float *amax_dev,
                         amp_stream_t stream);

/* amp_adamw_master_step with gradient-norm clipping: the per-step scalar
 *     clip = min(1, max_norm / (sqrt(*grad_sumsq_dev) + 1e-6))
 * is formed once in fp64 (NaN propagates) and rounded to fp32, and every
 * element uses g = (float(grad) * (1/S)) * clip in place of float(grad) * (1/S).
 * grad_sumsq_dev is the output of amp_unscale_check_norm for the same step.
 * Errors: as amp_adamw_master_step, plus AMP_EINVAL for a NULL
 * grad_sumsq_dev or a max_norm that is not finite and > 0. */
amp_status amp_adamw_master_step_clip(amp_tensor_list master, amp_tensor_list exp_avg,
                                      amp_tensor_list exp_avg_sq, amp_tensor_list grads,
                                      amp_tensor_list bf16_out, const float *scale_dev,
                                      const int32_t *found_inf_dev, int32_t *step_dev,
                                      const amp_adamw_hyper *hyper, float *amax_dev,
                                      const double *grad_sumsq_dev, double max_norm,
                                      amp_stream_t stream);

/* amp_adamw_master_step with the bf16 working copy rounded stochastically
 * ("第20章 量化与混合精度训练" §20.5.14: round down or up with probability
 * proportional to the distance, so the expected value is the input) instead
 * of to nearest-even; master, m, v and the amax fold are as in
 * amp_adamw_master_step.  For a finite fp32 p the result is the bf16 value
 * away from zero (inf beyond the largest finite) with probability
 * (16 dropped bits of |p|) / 2^16, else the one toward zero; values on the
 * bf16 grid and infinities are kept, NaN gives 0x7FC0.  Random bits:
 * Philox4x32-10 (Salmon et al., SC 2011) with key = seed and counter
 * {k/8 (low, high 32 bits), t, i} for element k of tensor i at step t (the
 * step counter after this step); element k uses 16-bit half (k%8)%2 (low
 * first) of output word (k%8)/2.  Deterministic for a given seed and step.
 * Errors: as amp_adamw_master_step, and AMP_EINVAL for a NULL bf16_out. */
amp_status amp_adamw_master_step_sr(amp_tensor_list master, amp_tensor_list exp_avg,
                                    amp_tensor_list exp_avg_sq, amp_tensor_list grads,
                                    amp_tensor_list bf16_out, const float *scale_dev,
                                    const int32_t *found_inf_dev, int32_t *step_dev,
                                    const amp_adamw_hyper *hyper, float *amax_dev, uint64_t seed,
                                    amp_stream_t stream);

/* amp_adamw_master_step_clip with the bf16 copy rounded stochastically as in
 * amp_adamw_master_step_sr (same random counters); the clip factor as in
 * amp_adamw_master_step_clip.
 * Errors: as amp_adamw_master_step_clip, and AMP_EINVAL for a NULL bf16_out. */
amp_status amp_adamw_master_step_clip_sr(amp_tensor_list master, amp_tensor_list exp_avg,
                                         amp_tensor_list exp_avg_sq, amp_tensor_list grads,
                                         amp_tensor_list bf16_out, const float *scale_dev,
                                         const int32_t *found_inf_dev, int32_t *step_dev,
                                         const amp_adamw_hyper *hyper, float *amax_dev,
                                         const double *grad_sumsq_dev, double max_norm,
                                         uint64_t seed, amp_stream_t stream);

/* Allocation-free form of amp_adamw_master_step.  The pages have no
 * counterpart: it exists for callers that cannot allocate device memory -
 * runtimes that serve all device memory from their own arena, loops that must
 * not take the device-wide synchronisation of cudaMalloc/cudaFree, processes
 * running with the GPU nearly full, and plain-C callers that cannot keep a
 * list handle alive.  The same arithmetic and kernels as
 * amp_adamw_master_step; the tensors come as host arrays of n device
 * pointers (bf16_out and amax_slots may be NULL) plus numel[n], and the
 * tables the kernels walk are copied on `stream` into one fixed device array
 * of about 4.1 MB built into the library (held on every GPU that loads it
 * until exit).  Limits: n <= 1024 tensors and at most 524,288 chunks of 16384
 * elements in total; larger calls return AMP_EINVAL with a message.
 *   - No cudaMalloc/cudaFree or other allocating routine is called.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.
 *   - The tables are uploaded with one cudaMemcpyAsync from pageable host
 *     memory.  CUDA stages such a copy itself and may first wait for the
 *     stream, so, unlike the handle-based entry points, a call can block the
 *     host until the work already enqueued on `stream` has drained.
 *   - It cannot be captured into a CUDA graph: on a capturing stream it
 *     returns AMP_EINVAL and enqueues nothing (a captured copy would replay
 *     from host memory freed when the call returns).
 *   - Every call shares the array: calls whose work can overlap on the GPU
 *     (unordered streams) race; order them on one stream.
 *   - Host allocation failure of the tables returns AMP_ENOMEM. */
amp_status amp_adamw_master_step_noalloc(int n, float *const *master, float *const *exp_avg,
                                         float *const *exp_avg_sq, const void *const *grads,
                                         amp_dtype grad_dtype, uint16_t *const *bf16_out,
                                         const int64_t *numel, const int32_t *amax_slots,
                                         const float *scale_dev, const int32_t *found_inf_dev,
                                         int32_t *step_dev, const amp_adamw_hyper *hyper,
                                         float *amax_dev, amp_stream_t stream);

/* amp_tensor_list_check for amp_adamw_master_step_noalloc: waits for
 * `stream`, reads and clears the sticky error word of the current device's
 * fixed array; AMP_ETIMEOUT if a bounded wait gave up since the last check.
 * Allocates nothing. */
amp_status amp_noalloc_check(amp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* A6-A9: tensorwise dynamic FP8 quantization.  [FP8] §2 (quant math), §3     */
/* (e4m3fn for weights/activations, e5m2 for gradients), §4 (column-major     */
/* copies for the backward GEMMs).                                            */
/* ------------------------------------------------------------------------ */

/* x is [rows, cols] row-major (AMP_DT_BF16, AMP_DT_F16 or AMP_DT_F32).
 *   amax      = max |x| in fp32 (NaN-propagating); written to *amax_dev
 *               unless amax_given != 0, in which case *amax_dev is read
 *   scale_d   = fp8_max / max(double(amax), eps)                  (fp64)
 *   out[i,j]  = fp8(clamp(float(x[i,j]) * float(scale_d), -fp8_max, fp8_max))
 *               round-to-nearest-even; NaN -> 0x7F (e4m3fn) / 0x7E (e5m2)
 *   out_t[j,i] = out[i,j]   ([cols, rows] row-major = column-major out), if
 *               out_t is non-NULL
 *   *inv_scale_dev = float(1 / scale_d)
 * fp8_dtype is AMP_DT_E4M3FN (max 448) or AMP_DT_E5M2 (max 57344); eps > 0
 * (1e-12 is the usual value).  If skip_if_dev is non-NULL and
 * *skip_if_dev != 0 nothing is written.  Empty tensors (rows*cols == 0)
 * write amax 0 and the matching inv_scale.
 * Errors: AMP_EINVAL (null out / inv_scale / amax, negative size,
 * eps <= 0), AMP_EDTYPE. */
amp_status fp8_quant_tensorwise(const void *x, amp_dtype x_dtype, int64_t rows, int64_t cols,
                                amp_dtype fp8_dtype, double eps, void *out, void *out_t,
                                float *inv_scale_dev, float *amax_dev, int amax_given,
                                const int32_t *skip_if_dev, amp_stream_t stream);

/* Group-wise scaling ("第20章 量化与混合精度训练" §20.5.18: a weight [out, in]
 * cut into groups of `group` consecutive elements along in, one scale per
 * group; g128 is the usual size).  x is [rows, cols] row-major (bf16, f16,
 * f32); group is 32, 64 or 128.  With ngc = ceil(cols / group), for every row
 * i and group g (columns g*group .. min((g+1)*group, cols) - 1), §2 of
 * "FP8训练：量化、自动微分、Torchao" on that group alone:
 *     amax_rg[i*ngc+g]  = max |x[i,j]| over the group  (fp32, NaN propagating)
 *     scale_d           = fp8_max / max(double(amax), eps)               (fp64)
 *     scale_rg[i*ngc+g] = float(scale_d), inv_rg[i*ngc+g] = float(1/scale_d)
 *     out[i,j]          = fp8(clamp(float(x[i,j]) * scale_rg, +-fp8_max)), RNE
 * If out_t is non-NULL it is the column-major copy ([cols, rows], §4) for the
 * GEMMs that reduce along the rows of x, so its groups are `group` consecutive
 * rows of one column: with ngr = ceil(rows / group), amax_cg / scale_cg /
 * inv_cg[j*ngr+g] and out_t[j,i] = fp8(clamp(float(x[i,j]) * scale_cg, ...)).
 * One launch, one CTA per 128x128 tile, 2 bytes read + 1 (+1) written per
 * element.  A set *skip_if_dev writes nothing.  Empty tensors return at once.
 * Errors: AMP_EINVAL (group not 32/64/128, NULL outputs, negative size,
 * eps <= 0), AMP_EDTYPE. */
amp_status fp8_quant_groupwise(const void *x, amp_dtype x_dtype, int64_t rows, int64_t cols,
                               int64_t group, amp_dtype fp8_dtype, double eps, void *out,
                               void *out_t, float *amax_rg, float *scale_rg, float *inv_rg,
                               float *amax_cg, float *scale_cg, float *inv_cg,
                               const int32_t *skip_if_dev, amp_stream_t stream);

/* Rowwise scaling ("FP8训练：量化、自动微分、Torchao" §1: one scale per row
 * instead of one per tensor).  x is [rows, cols] row-major (bf16, f16, f32).
 * For every row i, §2's recipe on that row alone:
 *     amax_row[i]  = max_j |x[i,j]|  (fp32, NaN propagating)
 *     scale_d      = fp8_max / max(double(amax_row[i]), eps)          (fp64)
 *     scale_row[i] = float(scale_d), inv_scale_row[i] = float(1/scale_d)
 *     out[i,j]     = fp8(clamp(float(x[i,j]) * scale_row[i], +-fp8_max)), RNE
 * If out_t is non-NULL it is the column-major copy for the GEMMs that reduce
 * along the rows of x (§4), so it takes one scale per column j, the same
 * recipe on column j: amax_col[j], scale_col[j], inv_scale_col[j], and
 * out_t[j,i] = fp8(clamp(float(x[i,j]) * scale_col[j], +-fp8_max)).
 * Four launches (zero, amax, scales, cast), 6 bytes per element.  A set
 * *skip_if_dev writes nothing.  Empty tensors return at once.
 * Errors: AMP_EINVAL (NULL outputs, negative size, eps <= 0), AMP_EDTYPE. */
amp_status fp8_quant_rowwise(const void *x, amp_dtype x_dtype, int64_t rows, int64_t cols,
                             amp_dtype fp8_dtype, double eps, void *out, void *out_t,
                             float *amax_row, float *scale_row, float *inv_scale_row,
                             float *amax_col, float *scale_col, float *inv_scale_col,
                             const int32_t *skip_if_dev, amp_stream_t stream);

/* The same over a list of 2-D tensors in one launch, with amax given per
 * tensor: tensor i uses amax_dev[i] (e.g. folded by amp_adamw_master_step
 * with slot i) and writes inv_scale_dev[i]; if x has amax slots, entry
 * slots[i] instead (amp_tensor_list_set_amax_slots).
 *   x      2-D list, AMP_DT_BF16 / AMP_DT_F16 / AMP_DT_F32
 *   out    2-D list of fp8_dtype with the shapes of x
 *   out_t  2-D list of fp8_dtype with the transposed shapes, or NULL
 * Errors: AMP_EINVAL (null / mismatched lists, 1-D list, eps <= 0),
 * AMP_EDTYPE. */
amp_status fp8_quant_tensorwise_list(amp_tensor_list x, amp_tensor_list out,
                                     amp_tensor_list out_t, amp_dtype fp8_dtype, double eps,
                                     const float *amax_dev, float *inv_scale_dev,
                                     const int32_t *skip_if_dev, amp_stream_t stream);

/* fp8_quant_tensorwise_list with the FP8 bytes rounded stochastically
 * ("第20章 量化与混合精度训练" §20.5.14: round down or up with probability
 * proportional to the distance; the lower the precision, FP8 included, the
 * more it matters).  The same amax, scale and inv_scale; each element's
 * y = float(x) * float(scale_d), clamped to +-fp8_max, becomes the FP8 value
 * away from zero with probability
 *     floor(2^16 * (|y| - lo) / (hi - lo)) / 2^16
 * (lo <= |y| < hi the neighbouring FP8 magnitudes: the distance ratio,
 * truncated to a multiple of 2^-16, so the mean is low by less than 2^-16 of
 * an FP8 quantum), else the one toward zero, with y's sign; values on the
 * grid stay, NaN gives 0x7F / 0x7E.  Random bits: 16 per element from
 * Philox4x32-10 (Salmon et al., SC 2011), key = seed, counter {k/8 (low,
 * high 32 bits), t, j | 2^31} for row-major element k of tensor j of the
 * list, t = *step_dev (the step count after this step's update); element k
 * takes the 16-bit half (k%8)%2 (low first) of output word (k%8)/2, the
 * layout of the bf16 copy's draws.  The transposed copy holds the same bytes.
 * Errors: as fp8_quant_tensorwise_list, and AMP_EINVAL for a NULL step_dev or
 * a list of 2^30 tensors or more. */
amp_status fp8_quant_tensorwise_list_sr(amp_tensor_list x, amp_tensor_list out,
                                        amp_tensor_list out_t, amp_dtype fp8_dtype, double eps,
                                        const float *amax_dev, float *inv_scale_dev,
                                        const int32_t *skip_if_dev, uint64_t seed,
                                        const int32_t *step_dev, amp_stream_t stream);

/* Delayed FP8 scaling fused into the update ("第20章 量化与混合精度训练"
 * §20.5.9: each FP8 op keeps an amax history and casts with the scale of the
 * previous steps' amax; §20.5.31 ScalingStrategy.DELAYED).  The pages have no
 * fused form: with the scale known before the pass, the FP8 weights' update,
 * bf16 copy, FP8 bytes and transposed FP8 bytes come out of one pass (30
 * bytes per parameter instead of 28 + 4 over two passes).
 * One optimizer step over two groups of tensors that share the step counter:
 *   plain group  - 1-D lists master, exp_avg, exp_avg_sq, grads, bf16_out:
 *                  exactly amp_adamw_master_step (no amax slots);
 *   FP8 group    - 2-D lists master8, exp_avg8, exp_avg_sq8, grads8, bf16_out8
 *                  and fp8_out (all with one shape set), fp8_t_out (the
 *                  transposed shapes, or NULL): the same update and bf16
 *                  copy, and per tensor j, in the same pass,
 *        amax_h  = max over amax_history[j*hist_len .. j*hist_len+hist_len)
 *                  (NaN propagating; newest first, see below)
 *        scale_d = fp8_max / max(double(amax_h), eps)              (fp64)
 *        fp8_out[j] = fp8(clamp(float(bf16) * float(scale_d), +-fp8_max)),
 *                  fp8_t_out[j] its [cols, rows] copy, RNE, NaN -> 0x7F/0x7E
 *        inv_scale_dev[j] = float(1 / scale_d)
 *        amax_dev[j] = max(amax_dev[j], max |bf16 of tensor j|)  (the caller
 *                  zeroes amax_dev; amp_update_scale_fp8_history does)
 * On a skipped step (*found_inf_dev != 0) nothing is written, inv_scale
 * included, and *step_dev is unchanged.  Either group may be empty (n = 0).
 * grads and grads8 share one dtype (f16, bf16 or f32); fp8_dtype is
 * AMP_DT_E4M3FN or AMP_DT_E5M2; eps > 0; hist_len >= 1.  The per-tensor scales
 * live in fp8_out's device block between the two launches of the call: calls
 * on one fp8_out list must not overlap on the GPU.
 * Errors: AMP_EINVAL (NULL / mismatched lists, hist_len < 1, eps <= 0),
 * AMP_EDTYPE. */
amp_status amp_adamw_master_step_fp8_delayed(
    amp_tensor_list master, amp_tensor_list exp_avg, amp_tensor_list exp_avg_sq,
    amp_tensor_list grads, amp_tensor_list bf16_out, amp_tensor_list master8,
    amp_tensor_list exp_avg8, amp_tensor_list exp_avg_sq8, amp_tensor_list grads8,
    amp_tensor_list bf16_out8, amp_tensor_list fp8_out, amp_tensor_list fp8_t_out,
    amp_dtype fp8_dtype, double eps, const float *amax_history, int hist_len, float *amax_dev,
    float *inv_scale_dev, const float *scale_dev, const int32_t *found_inf_dev,
    int32_t *step_dev, const amp_adamw_hyper *hyper, amp_stream_t stream);

/* amp_adamw_master_step_fp8_delayed with both copies rounded stochastically
 * ("第20章 量化与混合精度训练" §20.5.14): the bf16 copy as in
 * amp_adamw_master_step_sr, whose counter takes, as its tensor word, the list
 * index p for plain tensors and j | 2^30 for FP8 weight j; the FP8 bytes cast
 * from that copy with the delayed scale as in fp8_quant_tensorwise_list_sr
 * (tensor word j | 2^31); t is the step count after this step.
 * Errors: as amp_adamw_master_step_fp8_delayed, and AMP_EINVAL for a list of
 * 2^30 tensors or more. */
amp_status amp_adamw_master_step_fp8_delayed_sr(
    amp_tensor_list master, amp_tensor_list exp_avg, amp_tensor_list exp_avg_sq,
    amp_tensor_list grads, amp_tensor_list bf16_out, amp_tensor_list master8,
    amp_tensor_list exp_avg8, amp_tensor_list exp_avg_sq8, amp_tensor_list grads8,
    amp_tensor_list bf16_out8, amp_tensor_list fp8_out, amp_tensor_list fp8_t_out,
    amp_dtype fp8_dtype, double eps, const float *amax_history, int hist_len, float *amax_dev,
    float *inv_scale_dev, const float *scale_dev, const int32_t *found_inf_dev,
    int32_t *step_dev, const amp_adamw_hyper *hyper, uint64_t seed, amp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* A3: dynamic loss-scale state machine.  [CH20] §20.5.33, [MP06] §四.        */
/* ------------------------------------------------------------------------ */

/* One thread on the device:
 *   if *found_inf_dev: *scale_dev *= backoff_factor; *growth_tracker_dev = 0
 *   else: *growth_tracker_dev += 1; if it reaches growth_interval:
 *         *scale_dev *= growth_factor (kept unchanged if the product is not
 *         finite); *growth_tracker_dev = 0
 * then clears *found_inf_dev and amax_dev[0 .. n_amax) for the next step.
 * Errors: AMP_EINVAL (null state pointers, growth_interval < 1, n_amax < 0,
 * n_amax > 0 with amax_dev NULL). */
amp_status amp_update_scale(float *scale_dev, int32_t *growth_tracker_dev,
                            int32_t *found_inf_dev, float growth_factor, float backoff_factor,
                            int32_t growth_interval, float *amax_dev, int n_amax,
                            amp_stream_t stream);

/* amp_update_scale for the delayed-scaling step: the same state machine, and
 * when the step was not skipped (*found_inf_dev == 0 on entry) each FP8
 * tensor's amax of this step enters its history row of hist_len floats at
 * position 0, the older entries moving up by one and the oldest dropped.
 * amax_dev[0 .. n_fp8) and *found_inf_dev are cleared in every case.
 * Errors: as amp_update_scale, plus AMP_EINVAL for hist_len < 1 or NULL
 * amax / history with n_fp8 > 0. */
amp_status amp_update_scale_fp8_history(float *scale_dev, int32_t *growth_tracker_dev,
                                        int32_t *found_inf_dev, float growth_factor,
                                        float backoff_factor, int32_t growth_interval,
                                        float *amax_dev, float *amax_history, int n_fp8,
                                        int hist_len, amp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Monitoring.  The pages watch the loss scale (scaler.get_scale()) and fall  */
/* back to bf16 when it keeps halving ([CH20] §20.2.2 and "06 · 混合精度"      */
/* §四); these two calls serve that outside the step, and have no other       */
/* counterpart on the pages.                                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    float scale;
    int32_t growth_tracker;
    int32_t step;
    int32_t found_inf;
} amp_scaler_state;

/* Enqueue on `stream` a device-to-host copy of the scaler and step state into
 * *host_out (one 4-byte cudaMemcpyAsync per non-NULL pointer; the fields of
 * NULL pointers are left alone).  host_out should be page-locked for the
 * copies to be asynchronous; read it after synchronising `stream`.
 * Errors: AMP_EINVAL (host_out NULL), AMP_ECUDA. */
amp_status amp_read_state(const float *scale_dev, const int32_t *growth_tracker_dev,
                          const int32_t *step_dev, const int32_t *found_inf_dev,
                          amp_scaler_state *host_out, amp_stream_t stream);

/* Sticky health word of the loss scale, one thread on `stream`:
 *   *health_dev |= 1 if *scale_dev is not finite,
 *   *health_dev |= 2 if it is finite and below min_scale (it kept halving).
 * Bits are only ever set; the caller clears the word.  health_dev may point to
 * device memory or to page-locked host memory the device can address (memory
 * from cudaHostAlloc, or registered), so the host can poll it without
 * synchronising.  Errors: AMP_EINVAL (NULL pointer, min_scale < 0 or NaN). */
amp_status amp_scale_health(const float *scale_dev, float min_scale, int32_t *health_dev,
                            amp_stream_t stream);

/* Message describing the last non-OK status returned on this thread (no
 * counterpart on the pages; error reporting of this ABI). */
const char *amp_last_error(void);

/* ABI version of this header (incremented on incompatible changes; no
 * counterpart on the pages). */
int amp_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* AMPFP8_H */
