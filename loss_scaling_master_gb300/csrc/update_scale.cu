// update_scale.cu - A3: the dynamic loss-scale state machine
// ("第20章 量化与混合精度训练" §20.5.33 GradScaler 的 _growth_tracker 状态机细节;
// "06 · 混合精度" §四: skip and halve on inf/NaN, double after N clean steps).
// One thread updates {scale, tracker} in place from found_inf; the block then
// clears found_inf and the per-tensor amax slots for the next step, so the
// host never reads the state back.
#include "internal.h"
#include "pdl.cuh"

namespace amp {
namespace {

__global__ void update_scale_kernel(float *scale, int32_t *tracker, int32_t *found_inf,
                                    float growth, float backoff, int32_t interval, float *amax,
                                    int n_amax) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) {
        const int32_t fi = *found_inf;
        float s = *scale;
        int32_t t = *tracker;
        if (fi) {
            s = __fmul_rn(s, backoff);
            t = 0;
        } else {
            t = t + 1;
            if (t >= interval) {
                const float grown = __fmul_rn(s, growth);
                if (isfinite(grown)) s = grown;
                t = 0;
            }
        }
        *scale = s;
        *tracker = t;
        *found_inf = 0;
    }
    for (int i = threadIdx.x; i < n_amax; i += blockDim.x) amax[i] = 0.0f;
}

// As update_scale_kernel, and on a step that was not skipped each FP8
// tensor's amax of this step is pushed into its history (newest first, the
// oldest dropped); amax is cleared either way.
__global__ void update_scale_hist_kernel(float *scale, int32_t *tracker, int32_t *found_inf,
                                         float growth, float backoff, int32_t interval,
                                         float *amax, float *hist, int n, int hist_len) {
    pdl_wait();
    pdl_trigger();
    const int32_t fi = *found_inf;
    __syncthreads();  // every thread has read the flag before thread 0 clears it
    if (threadIdx.x == 0) {
        float s = *scale;
        int32_t t = *tracker;
        if (fi) {
            s = __fmul_rn(s, backoff);
            t = 0;
        } else {
            t = t + 1;
            if (t >= interval) {
                const float grown = __fmul_rn(s, growth);
                if (isfinite(grown)) s = grown;
                t = 0;
            }
        }
        *scale = s;
        *tracker = t;
        *found_inf = 0;
    }
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        if (!fi) {
            float *h = hist + int64_t(j) * hist_len;
            for (int k = hist_len - 1; k > 0; --k) h[k] = h[k - 1];
            h[0] = amax[j];
        }
        amax[j] = 0.0f;
    }
}

}  // namespace

cudaError_t launch_update_scale_hist(float *scale, int32_t *tracker, int32_t *found_inf,
                                     float growth, float backoff, int32_t interval, float *amax,
                                     float *hist, int n, int hist_len, cudaStream_t s) {
    launch_pdl(update_scale_hist_kernel, dim3(1), dim3(256), 0, s, scale, tracker, found_inf,
               growth, backoff, interval, amax, hist, n, hist_len);
    return cudaGetLastError();
}

cudaError_t launch_update_scale(float *scale, int32_t *tracker, int32_t *found_inf, float growth,
                                float backoff, int32_t interval, float *amax, int n_amax,
                                cudaStream_t s) {
    launch_pdl(update_scale_kernel, dim3(1), dim3(256), 0, s, scale, tracker, found_inf, growth,
               backoff, interval, amax, n_amax);
    return cudaGetLastError();
}

namespace {

// Health of the loss scale: "第20章 量化与混合精度训练" and "06 · 混合精度" watch
// the scale (scaler.get_scale()) and switch to bf16 when it keeps halving.
// bit 0: the scale is not finite; bit 1: it fell below min_scale.  Bits are
// only ever set.
__global__ void scale_health_kernel(const float *scale, float min_scale, int32_t *health) {
    pdl_wait();
    pdl_trigger();
    const float s = *scale;
    const int32_t h = !isfinite(s) ? 1 : (s < min_scale ? 2 : 0);
    if (h) {
        volatile int32_t *p = health;
        *p = *p | h;
        __threadfence_system();
    }
}

}  // namespace

cudaError_t launch_scale_health(const float *scale, float min_scale, int32_t *health, cudaStream_t s) {
    return launch_pdl(scale_health_kernel, dim3(1), dim3(1), 0, s, scale, min_scale, health);
}

}  // namespace amp
