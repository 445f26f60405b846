// internal.h - host-side pieces shared by the C-ABI layer (api.cu) and the
// kernel translation units: the list handle and the launch functions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "ampfp8.h"
#include "common.cuh"

// An NVTX range around one ABI call, named after the entry point: visible to
// profilers that record NVTX ranges (ncu --nvtx, Nsight Systems); without an
// attached tool each push/pop is a call through an empty hook.
struct AmpTraceRange {
    explicit AmpTraceRange(const char *name) { nvtxRangePushA(name); }
    ~AmpTraceRange() { nvtxRangePop(); }
    AmpTraceRange(const AmpTraceRange &) = delete;
    AmpTraceRange &operator=(const AmpTraceRange &) = delete;
};
#define AMP_TRACE(name) AmpTraceRange amp_trace_range_(name)

struct amp_tensor_list_s {
    int n = 0;
    amp_dtype dtype = AMP_DT_F32;
    bool two_d = false;
    int device = 0;
    std::vector<void *> ptrs;
    std::vector<int64_t> numel, rows, cols;
    int64_t n_chunks = 0;
    int64_t n_tiles = 0;
    bool has_slots = false;  // some slot >= 0
    int32_t min_slot = -1;   // the smallest slot (a cast list needs every slot >= 0)
    void *block = nullptr;   // the single device allocation
    void *scratch = nullptr; // 256 bytes of it for per-call kernel scalars
    float *tscale = nullptr; // one float per tensor of it (per-call scratch)
    amp::ListView view{};    // pointers into `block`
};

namespace amp {

// Per-step AdamW constants prepared on the host (fp64 -> fp32 once).
struct AdamwConsts {
    double lr, beta1, beta2;          // per-step scalars are formed on device
    float decay, b1, omb1, b2, omb2, eps;
};

// Offset, in int32 words from the step-scalar block, of the sticky error word
// the bulk-copy kernels set when a bounded wait gives up (within the 256-byte
// per-list scratch; the step scalars take the first 32 bytes).
constexpr int kErrWordOffset = 32;

// Device scalars of one AdamW step, written by the prologue kernel.
struct AdamwStepScalars {
    int32_t skip;
    float step_size;
    float bc2_sqrt;
    float clip;  // gradient clipping factor, exactly 1.0 when not clipping
    int32_t t;   // the step being taken (step counter after it)
    int32_t pad[3];
};

int sm_count(int device);

// Set the calling thread's amp_last_error() message.
void set_last_error(const char *msg);

cudaError_t launch_unscale_check(const ListView &g, int64_t n_chunks, int elem, const float *scale,
                                 int32_t *found_inf, int inplace, cudaStream_t s);

cudaError_t launch_check_norm(const ListView &g, int64_t n_chunks, int elem, const float *scale,
                              int32_t *found_inf, double *sumsq, cudaStream_t s);

cudaError_t launch_adamw(const ListView &p, const ListView &m, const ListView &v,
                         const ListView &g, const ListView *b, int64_t n_chunks, int gelem,
                         const float *scale, const int32_t *found_inf, int32_t *step,
                         const AdamwConsts &c, AdamwStepScalars *scal, float *amax,
                         bool use_slots, cudaStream_t s, const double *clip_sumsq = nullptr,
                         double max_norm = 0.0, bool stochastic = false, uint64_t seed = 0);

cudaError_t launch_adamw_main(const ListView &p, const ListView &m, const ListView &v,
                              const ListView &g, const ListView *b, int64_t n_chunks, int gelem,
                              const float *scale, const AdamwConsts &c,
                              const AdamwStepScalars *scal, float *amax, bool use_slots,
                              cudaStream_t s, bool stochastic = false, uint64_t seed = 0);

// The lists of one delayed-scaling FP8 step: the tensors without FP8 copies
// (1-D, walked by chunks) and the FP8 weights (2-D, walked by 128x128 tiles).
struct Fp8DelayedLists {
    ListView p, m, v, g, b;          // plain tensors
    int64_t n_plain_chunks;
    ListView p8, m8, v8, g8, b8, q;  // FP8 weights (2-D) and their fp8 copies
    const ListView *qt;              // transposed copies or nullptr
    int64_t n_tiles;
    int n8;
    float *tscale;                   // per FP8 weight: fp32 cast scale (scratch)
};

cudaError_t launch_adamw_fp8_delayed(const Fp8DelayedLists &L, int gelem, int fp8,
                                     const float *scale, const int32_t *found_inf, int32_t *step,
                                     const AdamwConsts &c, AdamwStepScalars *scal,
                                     const float *hist, int hist_len, double eps, float *amax,
                                     float *inv_scale, cudaStream_t s, bool stochastic = false,
                                     uint64_t seed = 0);

cudaError_t launch_emit_bf16(const ListView &p, const ListView &b, int64_t n_chunks, float *amax,
                             bool use_slots, cudaStream_t s);

cudaError_t launch_bounded_wait_selftest(int32_t *err, double limit_s, cudaStream_t s);
cudaError_t launch_fp8_quant_groupwise(const void *x, int xelem, int64_t rows, int64_t cols,
                                       int64_t group, int fp8, double eps, uint8_t *out,
                                       uint8_t *out_t, float *amax_rg, float *scale_rg,
                                       float *inv_rg, float *amax_cg, float *scale_cg,
                                       float *inv_cg, const int32_t *skip_if, cudaStream_t s);
cudaError_t launch_scale_health(const float *scale, float min_scale, int32_t *health, cudaStream_t s);

cudaError_t launch_update_scale_hist(float *scale, int32_t *tracker, int32_t *found_inf,
                                     float growth, float backoff, int32_t interval, float *amax,
                                     float *hist, int n, int hist_len, cudaStream_t s);

cudaError_t launch_update_scale(float *scale, int32_t *tracker, int32_t *found_inf, float growth,
                                float backoff, int32_t interval, float *amax, int n_amax,
                                cudaStream_t s);

cudaError_t launch_fp8_quant(const void *x, int xelem, int64_t rows, int64_t cols, int fp8,
                             double eps, uint8_t *out, uint8_t *out_t, float *inv_scale,
                             float *amax, int amax_given, const int32_t *skip_if, int device,
                             cudaStream_t s);

cudaError_t launch_fp8_quant_rowwise(const void *x, int xelem, int64_t rows, int64_t cols, int fp8,
                                     double eps, uint8_t *out, uint8_t *out_t, float *amax_row,
                                     float *scale_row, float *inv_row, float *amax_col,
                                     float *scale_col, float *inv_col, const int32_t *skip_if,
                                     int device, cudaStream_t s);

// sr_step non-NULL: the stochastic cast, random counters from the step count
// *sr_step and sr_seed.  use_slots: tensor t takes amax / inv_scale (and the
// random counter's tensor word) at x.slots[t] instead of t.
cudaError_t launch_fp8_quant_list(const ListView &x, int64_t n_tiles, bool any_empty, int xelem,
                                  const ListView &out, const ListView *out_t, int fp8,
                                  double eps, const float *amax, float *inv_scale,
                                  const int32_t *skip_if, cudaStream_t s,
                                  const int32_t *sr_step = nullptr, uint64_t sr_seed = 0,
                                  bool use_slots = false);

}  // namespace amp
