// api.cu - the extern "C" boundary of libampfp8.so: argument validation,
// tensor-list handles and kernel launches.  Every entry point is declared and
// documented in include/ampfp8.h.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"

namespace {

thread_local char g_err[512] = "";

amp_status fail(amp_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

amp_status cuda_fail(cudaError_t e, const char *what) {
    return fail(AMP_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

int elem_code(amp_dtype d) {
    switch (d) {
    case AMP_DT_F32: return amp::kF32;
    case AMP_DT_F16: return amp::kF16;
    case AMP_DT_BF16: return amp::kBF16;
    default: return -1;
    }
}

int fp8_code(amp_dtype d) {
    return d == AMP_DT_E4M3FN ? amp::kE4M3 : d == AMP_DT_E5M2 ? amp::kE5M2 : -1;
}

size_t elem_size(amp_dtype d) {
    switch (d) {
    case AMP_DT_F32: return 4;
    case AMP_DT_F16:
    case AMP_DT_BF16: return 2;
    case AMP_DT_E4M3FN:
    case AMP_DT_E5M2: return 1;
    }
    return 0;
}

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

bool same_shapes(const amp_tensor_list_s *a, const amp_tensor_list_s *b) {
    return a->n == b->n && a->numel == b->numel;
}

}  // namespace

namespace amp {
void set_last_error(const char *msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

int sm_count(int device) {
    static std::mutex mu;
    static std::vector<int> cache;
    std::lock_guard<std::mutex> lock(mu);
    if (device >= int(cache.size())) cache.resize(device + 1, 0);
    if (cache[device] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0)
            v = 148;
        cache[device] = v;
    }
    return cache[device];
}
}  // namespace amp

extern "C" {

const char *amp_last_error(void) { return g_err; }

int amp_abi_version(void) { return 11; }

// A [rows, cols] shape the launch arithmetic can hold: non-negative, each side
// below 2^48 and rows * cols without int64 overflow.
static bool bad_shape(int64_t rows, int64_t cols) {
    const int64_t lim = int64_t(1) << 48;
    return rows < 0 || cols < 0 || rows >= lim || cols >= lim || (cols > 0 && rows > INT64_MAX / cols);
}

// The body of amp_tensor_list_create; host allocations may throw
// std::bad_alloc, which the entry point turns into AMP_ENOMEM.
static amp_status list_create(int n, void *const *dev_ptrs, const int64_t *rows,
                              const int64_t *cols, amp_dtype dtype, amp_stream_t stream,
                              amp_tensor_list *out) {
    if (!out) return fail(AMP_EINVAL, "amp_tensor_list_create: out is NULL");
    if (n < 0) return fail(AMP_EINVAL, "amp_tensor_list_create: n < 0");
    if (n > 0 && (!dev_ptrs || !rows))
        return fail(AMP_EINVAL, "amp_tensor_list_create: dev_ptrs / rows is NULL");
    if (elem_size(dtype) == 0) return fail(AMP_EDTYPE, "amp_tensor_list_create: unknown dtype");
    auto owner = std::make_unique<amp_tensor_list_s>();
    amp_tensor_list_s *L = owner.get();
    L->n = n;
    L->dtype = dtype;
    L->two_d = cols != nullptr;
    L->ptrs.resize(n);
    L->numel.resize(n);
    L->rows.resize(n);
    L->cols.resize(n);
    std::vector<uint2> chunks, tiles;
    for (int i = 0; i < n; ++i) {
        const int64_t r = rows[i], c = cols ? cols[i] : 1;
        if (bad_shape(r, c)) {
            return fail(AMP_EINVAL, "amp_tensor_list_create: negative or too large size at tensor %d", i);
        }
        const int64_t ne = r * c;
        if (ne > 0 && dev_ptrs[i] == nullptr) {
            return fail(AMP_EINVAL, "amp_tensor_list_create: NULL pointer of non-empty tensor %d", i);
        }
        // the tables are bounded before they grow, so an absurd shape fails
        // here instead of exhausting host memory
        const int64_t nc = (ne + amp::kChunk - 1) / amp::kChunk;
        const int64_t nt =
            cols ? ((r + amp::kTile - 1) / amp::kTile) * ((c + amp::kTile - 1) / amp::kTile) : 0;
        if (nc > int64_t(INT32_MAX) - int64_t(chunks.size()) ||
            nt > int64_t(INT32_MAX) - int64_t(tiles.size())) {
            return fail(AMP_EINVAL, "amp_tensor_list_create: tensor %d too large", i);
        }
        L->ptrs[i] = dev_ptrs[i];
        L->numel[i] = ne;
        L->rows[i] = r;
        L->cols[i] = c;
        for (int64_t k = 0; k < nc; ++k) chunks.push_back(make_uint2(i, uint32_t(k)));
        for (int64_t k = 0; k < nt; ++k) tiles.push_back(make_uint2(i, uint32_t(k)));
    }
    L->n_chunks = int64_t(chunks.size());
    L->n_tiles = int64_t(tiles.size());

    // one device block: ptrs | numel | rows | cols | slots | chunks | tiles | scratch
    const size_t nn = size_t(n > 0 ? n : 1);
    const size_t o_ptrs = 0;
    const size_t o_numel = align_up(o_ptrs + nn * sizeof(void *));
    const size_t o_rows = align_up(o_numel + nn * sizeof(int64_t));
    const size_t o_cols = align_up(o_rows + nn * sizeof(int64_t));
    const size_t o_slots = align_up(o_cols + nn * sizeof(int64_t));
    const size_t o_chunks = align_up(o_slots + nn * sizeof(int32_t));
    const size_t o_tiles = align_up(o_chunks + std::max<size_t>(1, chunks.size()) * sizeof(uint2));
    const size_t o_partials = align_up(o_tiles + std::max<size_t>(1, tiles.size()) * sizeof(uint2));
    const size_t o_tscale = align_up(o_partials + std::max<size_t>(1, chunks.size()) * sizeof(double));
    const size_t o_scratch = align_up(o_tscale + nn * sizeof(float));
    const size_t total = align_up(o_scratch + 256);
    std::vector<char> host(total, 0);
    std::memcpy(host.data() + o_ptrs, L->ptrs.data(), n * sizeof(void *));
    std::memcpy(host.data() + o_numel, L->numel.data(), n * sizeof(int64_t));
    std::memcpy(host.data() + o_rows, L->rows.data(), n * sizeof(int64_t));
    std::memcpy(host.data() + o_cols, L->cols.data(), n * sizeof(int64_t));
    std::vector<int32_t> slots(nn, -1);
    std::memcpy(host.data() + o_slots, slots.data(), nn * sizeof(int32_t));
    std::memcpy(host.data() + o_chunks, chunks.data(), chunks.size() * sizeof(uint2));
    std::memcpy(host.data() + o_tiles, tiles.data(), tiles.size() * sizeof(uint2));

    cudaError_t e = cudaGetDevice(&L->device);
    if (e != cudaSuccess) {
        return cuda_fail(e, "amp_tensor_list_create: cudaGetDevice");
    }
    e = cudaMalloc(&L->block, total);
    if (e != cudaSuccess) {
        return fail(AMP_ENOMEM, "amp_tensor_list_create: cudaMalloc(%zu): %s", total,
                    cudaGetErrorString(e));
    }
    // The host staging buffer must outlive the asynchronous copy.
    e = cudaMemcpyAsync(L->block, host.data(), total, cudaMemcpyHostToDevice,
                        reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaFree(L->block);
        return cuda_fail(e, "amp_tensor_list_create: upload");
    }
    char *b = static_cast<char *>(L->block);
    L->view.ptrs = reinterpret_cast<void *const *>(b + o_ptrs);
    L->view.numel = reinterpret_cast<const int64_t *>(b + o_numel);
    L->view.rows = reinterpret_cast<const int64_t *>(b + o_rows);
    L->view.cols = reinterpret_cast<const int64_t *>(b + o_cols);
    L->view.slots = reinterpret_cast<const int32_t *>(b + o_slots);
    L->view.chunks = reinterpret_cast<const uint2 *>(b + o_chunks);
    L->view.tiles = reinterpret_cast<const uint2 *>(b + o_tiles);
    L->view.partials = reinterpret_cast<double *>(b + o_partials);
    L->view.n = n;
    L->scratch = b + o_scratch;
    L->tscale = reinterpret_cast<float *>(b + o_tscale);
    *out = owner.release();
    return AMP_OK;
}

amp_status amp_tensor_list_create(int n, void *const *dev_ptrs, const int64_t *rows,
                                  const int64_t *cols, amp_dtype dtype, amp_stream_t stream,
                                  amp_tensor_list *out) {
    AMP_TRACE("amp_tensor_list_create");
    try {
        return list_create(n, dev_ptrs, rows, cols, dtype, stream, out);
    } catch (const std::bad_alloc &) {
        return fail(AMP_ENOMEM, "amp_tensor_list_create: host allocation failed");
    }
}

amp_status amp_tensor_list_set_amax_slots(amp_tensor_list list, const int32_t *slots,
                                          amp_stream_t stream) {
    AMP_TRACE("amp_tensor_list_set_amax_slots");
    if (!list || (list->n > 0 && !slots))
        return fail(AMP_EINVAL, "amp_tensor_list_set_amax_slots: NULL argument");
    if (list->n == 0) return AMP_OK;
    std::vector<int32_t> h(slots, slots + list->n);
    bool any = false;
    int32_t lo = INT32_MAX;
    for (int32_t s : h) {
        any |= s >= 0;
        lo = std::min(lo, s);
    }
    cudaError_t e = cudaMemcpyAsync(const_cast<int32_t *>(list->view.slots), h.data(),
                                    h.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "amp_tensor_list_set_amax_slots");
    list->has_slots = any;
    list->min_slot = lo;
    return AMP_OK;
}

amp_status amp_tensor_list_destroy(amp_tensor_list list) {
    AMP_TRACE("amp_tensor_list_destroy");
    if (!list) return AMP_OK;
    cudaError_t e = list->block ? cudaFree(list->block) : cudaSuccess;
    delete list;
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, "amp_tensor_list_destroy");
}

static amp_status list_copy_host(amp_tensor_list list, void *const *host_ptrs, bool to_host,
                                 amp_stream_t stream) {
    const char *fn = to_host ? "amp_tensor_list_copy_to_host" : "amp_tensor_list_copy_from_host";
    if (!list) return fail(AMP_EINVAL, "%s: NULL list", fn);
    if (list->n > 0 && !host_ptrs) return fail(AMP_EINVAL, "%s: host_ptrs is NULL", fn);
    for (int i = 0; i < list->n; ++i)
        if (list->numel[i] > 0 && !host_ptrs[i])
            return fail(AMP_EINVAL, "%s: NULL host pointer of non-empty tensor %d", fn, i);
    const size_t es = elem_size(list->dtype);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int i = 0; i < list->n; ++i) {
        if (list->numel[i] == 0) continue;
        const size_t bytes = size_t(list->numel[i]) * es;
        cudaError_t e = to_host
            ? cudaMemcpyAsync(host_ptrs[i], list->ptrs[i], bytes, cudaMemcpyDeviceToHost, s)
            : cudaMemcpyAsync(list->ptrs[i], host_ptrs[i], bytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    return AMP_OK;
}

amp_status amp_tensor_list_copy_from_host(amp_tensor_list list, const void *const *host_ptrs,
                                          amp_stream_t stream) {
    AMP_TRACE("amp_tensor_list_copy_from_host");
    return list_copy_host(list, const_cast<void *const *>(host_ptrs), false, stream);
}

amp_status amp_tensor_list_copy_to_host(amp_tensor_list list, void *const *host_ptrs,
                                        amp_stream_t stream) {
    AMP_TRACE("amp_tensor_list_copy_to_host");
    return list_copy_host(list, host_ptrs, true, stream);
}

amp_status amp_tensor_list_check(amp_tensor_list list, amp_stream_t stream) {
    AMP_TRACE("amp_tensor_list_check");
    if (!list) return fail(AMP_EINVAL, "amp_tensor_list_check: NULL list");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t *word = reinterpret_cast<int32_t *>(list->scratch) + amp::kErrWordOffset;
    int32_t v = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "amp_tensor_list_check");
    if (v != 0) {
        const int32_t zero = 0;
        e = cudaMemcpy(word, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "amp_tensor_list_check");
        return fail(AMP_ETIMEOUT,
                    "amp_tensor_list_check: a kernel's bounded wait for its asynchronous copies "
                    "gave up; the chunks it held were not updated");
    }
    return AMP_OK;
}

amp_status amp_selftest_bounded_wait(int32_t *err_dev, double limit_seconds, amp_stream_t stream) {
    AMP_TRACE("amp_selftest_bounded_wait");
    if (!err_dev || !(limit_seconds > 0.0) || limit_seconds > 10.0)
        return fail(AMP_EINVAL, "amp_selftest_bounded_wait: err_dev NULL or limit not in (0, 10] s");
    cudaError_t e = amp::launch_bounded_wait_selftest(err_dev, limit_seconds,
                                                      reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, "amp_selftest_bounded_wait");
}

amp_status amp_unscale_check(amp_tensor_list grads, const float *scale_dev, int32_t *found_inf_dev,
                             int inplace, amp_stream_t stream) {
    AMP_TRACE("amp_unscale_check");
    if (!grads || !found_inf_dev) return fail(AMP_EINVAL, "amp_unscale_check: NULL argument");
    const int ec = elem_code(grads->dtype);
    if (ec < 0) return fail(AMP_EDTYPE, "amp_unscale_check: gradients must be f32/f16/bf16");
    cudaError_t e = amp::launch_unscale_check(grads->view, grads->n_chunks, ec, scale_dev,
                                              found_inf_dev, inplace ? 1 : 0,
                                              reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, "amp_unscale_check");
}

static amp_status adamw_entry(amp_tensor_list master, amp_tensor_list exp_avg,
                              amp_tensor_list exp_avg_sq, amp_tensor_list grads,
                              amp_tensor_list bf16_out, const float *scale_dev,
                              const int32_t *found_inf_dev, int32_t *step_dev,
                              const amp_adamw_hyper *hyper, float *amax_dev,
                              const double *clip_sumsq, double max_norm, amp_stream_t stream,
                              bool stochastic = false, uint64_t seed = 0) {
    if (!master || !exp_avg || !exp_avg_sq || !grads || !step_dev || !hyper)
        return fail(AMP_EINVAL, "amp_adamw_master_step: NULL argument");
    if (master->dtype != AMP_DT_F32 || exp_avg->dtype != AMP_DT_F32 ||
        exp_avg_sq->dtype != AMP_DT_F32)
        return fail(AMP_EDTYPE, "amp_adamw_master_step: master/exp_avg/exp_avg_sq must be f32");
    const int gc = elem_code(grads->dtype);
    if (gc < 0) return fail(AMP_EDTYPE, "amp_adamw_master_step: gradients must be f32/f16/bf16");
    if (bf16_out && bf16_out->dtype != AMP_DT_BF16)
        return fail(AMP_EDTYPE, "amp_adamw_master_step: bf16_out must be bf16");
    if (!same_shapes(master, exp_avg) || !same_shapes(master, exp_avg_sq) ||
        !same_shapes(master, grads) || (bf16_out && !same_shapes(master, bf16_out)))
        return fail(AMP_EINVAL, "amp_adamw_master_step: lists differ in tensor count or sizes");
    const bool slots = bf16_out && bf16_out->has_slots;
    if (slots && !amax_dev)
        return fail(AMP_EINVAL, "amp_adamw_master_step: bf16_out has amax slots but amax_dev is NULL");
    const amp_adamw_hyper &h = *hyper;
    amp::AdamwConsts c;
    c.lr = h.lr;
    c.beta1 = h.beta1;
    c.beta2 = h.beta2;
    c.decay = float(1.0 - h.lr * h.weight_decay);
    c.b1 = float(h.beta1);
    c.omb1 = float(1.0 - h.beta1);
    c.b2 = float(h.beta2);
    c.omb2 = float(1.0 - h.beta2);
    c.eps = float(h.eps);
    cudaError_t e = amp::launch_adamw(
        master->view, exp_avg->view, exp_avg_sq->view, grads->view,
        bf16_out ? &bf16_out->view : nullptr, master->n_chunks, gc, scale_dev, found_inf_dev,
        step_dev, c, reinterpret_cast<amp::AdamwStepScalars *>(master->scratch), amax_dev, slots,
        reinterpret_cast<cudaStream_t>(stream), clip_sumsq, max_norm, stochastic, seed);
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, "amp_adamw_master_step");
}

amp_status amp_emit_bf16(amp_tensor_list master, amp_tensor_list bf16_out, float *amax_dev,
                         amp_stream_t stream) {
    AMP_TRACE("amp_emit_bf16");
    const char *fn = "amp_emit_bf16";
    if (!master || !bf16_out) return fail(AMP_EINVAL, "%s: NULL list", fn);
    if (master->dtype != AMP_DT_F32 || bf16_out->dtype != AMP_DT_BF16)
        return fail(AMP_EDTYPE, "%s: master must be f32 and bf16_out bf16", fn);
    if (!same_shapes(master, bf16_out))
        return fail(AMP_EINVAL, "%s: lists differ in tensor count or sizes", fn);
    const bool slots = bf16_out->has_slots;
    if (slots && !amax_dev)
        return fail(AMP_EINVAL, "%s: bf16_out has amax slots but amax_dev is NULL", fn);
    cudaError_t e = amp::launch_emit_bf16(master->view, bf16_out->view, master->n_chunks,
                                          amax_dev, slots, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, fn);
}

amp_status amp_adamw_master_step_sr(amp_tensor_list master, amp_tensor_list exp_avg,
                                    amp_tensor_list exp_avg_sq, amp_tensor_list grads,
                                    amp_tensor_list bf16_out, const float *scale_dev,
                                    const int32_t *found_inf_dev, int32_t *step_dev,
                                    const amp_adamw_hyper *hyper, float *amax_dev, uint64_t seed,
                                    amp_stream_t stream) {
    AMP_TRACE("amp_adamw_master_step_sr");
    if (!bf16_out) return fail(AMP_EINVAL, "amp_adamw_master_step_sr: bf16_out is NULL");
    return adamw_entry(master, exp_avg, exp_avg_sq, grads, bf16_out, scale_dev, found_inf_dev,
                       step_dev, hyper, amax_dev, nullptr, 0.0, stream, true, seed);
}

amp_status amp_adamw_master_step(amp_tensor_list master, amp_tensor_list exp_avg,
                                 amp_tensor_list exp_avg_sq, amp_tensor_list grads,
                                 amp_tensor_list bf16_out, const float *scale_dev,
                                 const int32_t *found_inf_dev, int32_t *step_dev,
                                 const amp_adamw_hyper *hyper, float *amax_dev,
                                 amp_stream_t stream) {
    AMP_TRACE("amp_adamw_master_step");
    return adamw_entry(master, exp_avg, exp_avg_sq, grads, bf16_out, scale_dev, found_inf_dev,
                       step_dev, hyper, amax_dev, nullptr, 0.0, stream);
}

amp_status amp_adamw_master_step_clip(amp_tensor_list master, amp_tensor_list exp_avg,
                                      amp_tensor_list exp_avg_sq, amp_tensor_list grads,
                                      amp_tensor_list bf16_out, const float *scale_dev,
                                      const int32_t *found_inf_dev, int32_t *step_dev,
                                      const amp_adamw_hyper *hyper, float *amax_dev,
                                      const double *grad_sumsq_dev, double max_norm,
                                      amp_stream_t stream) {
    AMP_TRACE("amp_adamw_master_step_clip");
    if (!grad_sumsq_dev) return fail(AMP_EINVAL, "amp_adamw_master_step_clip: grad_sumsq_dev is NULL");
    if (!(max_norm > 0.0) || max_norm > 1e300)
        return fail(AMP_EINVAL, "amp_adamw_master_step_clip: max_norm must be finite and > 0");
    return adamw_entry(master, exp_avg, exp_avg_sq, grads, bf16_out, scale_dev, found_inf_dev,
                       step_dev, hyper, amax_dev, grad_sumsq_dev, max_norm, stream);
}

static amp_status delayed_entry(
    const char *fn, amp_tensor_list master, amp_tensor_list exp_avg, amp_tensor_list exp_avg_sq,
    amp_tensor_list grads, amp_tensor_list bf16_out, amp_tensor_list master8,
    amp_tensor_list exp_avg8, amp_tensor_list exp_avg_sq8, amp_tensor_list grads8,
    amp_tensor_list bf16_out8, amp_tensor_list fp8_out, amp_tensor_list fp8_t_out,
    amp_dtype fp8_dtype, double eps, const float *amax_history, int hist_len, float *amax_dev,
    float *inv_scale_dev, const float *scale_dev, const int32_t *found_inf_dev, int32_t *step_dev,
    const amp_adamw_hyper *hyper, amp_stream_t stream, bool stochastic, uint64_t seed) {
    if (!master || !exp_avg || !exp_avg_sq || !grads || !bf16_out || !master8 || !exp_avg8 ||
        !exp_avg_sq8 || !grads8 || !bf16_out8 || !fp8_out || !amax_history || !amax_dev ||
        !inv_scale_dev || !step_dev || !hyper)
        return fail(AMP_EINVAL, "%s: NULL argument", fn);
    if (hist_len < 1) return fail(AMP_EINVAL, "%s: hist_len < 1", fn);
    if (!(eps > 0.0)) return fail(AMP_EINVAL, "%s: eps must be > 0", fn);
    const int fc = fp8_code(fp8_dtype);
    const int gc = elem_code(grads->dtype);
    if (fc < 0 || gc < 0 || grads8->dtype != grads->dtype)
        return fail(AMP_EDTYPE, "%s: unsupported or mixed gradient / fp8 dtype", fn);
    for (amp_tensor_list l : {master, exp_avg, exp_avg_sq, master8, exp_avg8, exp_avg_sq8})
        if (l->dtype != AMP_DT_F32) return fail(AMP_EDTYPE, "%s: master/m/v must be f32", fn);
    if (bf16_out->dtype != AMP_DT_BF16 || bf16_out8->dtype != AMP_DT_BF16 ||
        fp8_out->dtype != fp8_dtype || (fp8_t_out && fp8_t_out->dtype != fp8_dtype))
        return fail(AMP_EDTYPE, "%s: bf16 / fp8 output dtypes", fn);
    if (!same_shapes(master, exp_avg) || !same_shapes(master, exp_avg_sq) ||
        !same_shapes(master, grads) || !same_shapes(master, bf16_out))
        return fail(AMP_EINVAL, "%s: plain lists differ in tensor count or sizes", fn);
    for (amp_tensor_list l : {master8, exp_avg8, exp_avg_sq8, grads8, bf16_out8, fp8_out})
        if (!l->two_d || l->n != fp8_out->n || l->rows != fp8_out->rows || l->cols != fp8_out->cols)
            return fail(AMP_EINVAL, "%s: FP8-weight lists must be 2-D with one shape set", fn);
    if (fp8_t_out && (!fp8_t_out->two_d || fp8_t_out->n != fp8_out->n ||
                      fp8_t_out->rows != fp8_out->cols || fp8_t_out->cols != fp8_out->rows))
        return fail(AMP_EINVAL, "%s: fp8_t_out shapes are not the FP8 weights transposed", fn);
    const amp_adamw_hyper &h = *hyper;
    amp::AdamwConsts c;
    c.lr = h.lr;
    c.beta1 = h.beta1;
    c.beta2 = h.beta2;
    c.decay = float(1.0 - h.lr * h.weight_decay);
    c.b1 = float(h.beta1);
    c.omb1 = float(1.0 - h.beta1);
    c.b2 = float(h.beta2);
    c.omb2 = float(1.0 - h.beta2);
    c.eps = float(h.eps);
    amp::Fp8DelayedLists L;
    L.p = master->view;
    L.m = exp_avg->view;
    L.v = exp_avg_sq->view;
    L.g = grads->view;
    L.b = bf16_out->view;
    L.n_plain_chunks = master->n_chunks;
    L.p8 = master8->view;
    L.m8 = exp_avg8->view;
    L.v8 = exp_avg_sq8->view;
    L.g8 = grads8->view;
    L.b8 = bf16_out8->view;
    L.q = fp8_out->view;
    L.qt = fp8_t_out ? &fp8_t_out->view : nullptr;
    L.n_tiles = master8->n_tiles;
    L.n8 = fp8_out->n;
    L.tscale = fp8_out->tscale;
    if (stochastic && (master->n >= (1 << 30) || fp8_out->n >= (1 << 30)))
        return fail(AMP_EINVAL, "%s: 2^30 tensors or more per list", fn);
    cudaError_t e = amp::launch_adamw_fp8_delayed(
        L, gc, fc, scale_dev, found_inf_dev, step_dev, c,
        reinterpret_cast<amp::AdamwStepScalars *>(fp8_out->scratch), amax_history, hist_len, eps,
        amax_dev, inv_scale_dev, reinterpret_cast<cudaStream_t>(stream), stochastic, seed);
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, fn);
}

amp_status amp_adamw_master_step_clip_sr(amp_tensor_list master, amp_tensor_list exp_avg,
                                         amp_tensor_list exp_avg_sq, amp_tensor_list grads,
                                         amp_tensor_list bf16_out, const float *scale_dev,
                                         const int32_t *found_inf_dev, int32_t *step_dev,
                                         const amp_adamw_hyper *hyper, float *amax_dev,
                                         const double *grad_sumsq_dev, double max_norm,
                                         uint64_t seed, amp_stream_t stream) {
    AMP_TRACE("amp_adamw_master_step_clip_sr");
    const char *fn = "amp_adamw_master_step_clip_sr";
    if (!grad_sumsq_dev) return fail(AMP_EINVAL, "%s: grad_sumsq_dev is NULL", fn);
    if (!(max_norm > 0.0) || max_norm > 1e300)
        return fail(AMP_EINVAL, "%s: max_norm must be finite and > 0", fn);
    if (!bf16_out) return fail(AMP_EINVAL, "%s: bf16_out is NULL", fn);
    return adamw_entry(master, exp_avg, exp_avg_sq, grads, bf16_out, scale_dev, found_inf_dev,
                       step_dev, hyper, amax_dev, grad_sumsq_dev, max_norm, stream, true, seed);
}

amp_status amp_adamw_master_step_fp8_delayed(
    amp_tensor_list master, amp_tensor_list exp_avg, amp_tensor_list exp_avg_sq,
    amp_tensor_list grads, amp_tensor_list bf16_out, amp_tensor_list master8,
    amp_tensor_list exp_avg8, amp_tensor_list exp_avg_sq8, amp_tensor_list grads8,
    amp_tensor_list bf16_out8, amp_tensor_list fp8_out, amp_tensor_list fp8_t_out,
    amp_dtype fp8_dtype, double eps, const float *amax_history, int hist_len, float *amax_dev,
    float *inv_scale_dev, const float *scale_dev, const int32_t *found_inf_dev, int32_t *step_dev,
    const amp_adamw_hyper *hyper, amp_stream_t stream) {
    AMP_TRACE("amp_adamw_master_step_fp8_delayed");
    return delayed_entry("amp_adamw_master_step_fp8_delayed", master, exp_avg, exp_avg_sq, grads,
                         bf16_out, master8, exp_avg8, exp_avg_sq8, grads8, bf16_out8, fp8_out,
                         fp8_t_out, fp8_dtype, eps, amax_history, hist_len, amax_dev,
                         inv_scale_dev, scale_dev, found_inf_dev, step_dev, hyper, stream, false,
                         0);
}

amp_status amp_adamw_master_step_fp8_delayed_sr(
    amp_tensor_list master, amp_tensor_list exp_avg, amp_tensor_list exp_avg_sq,
    amp_tensor_list grads, amp_tensor_list bf16_out, amp_tensor_list master8,
    amp_tensor_list exp_avg8, amp_tensor_list exp_avg_sq8, amp_tensor_list grads8,
    amp_tensor_list bf16_out8, amp_tensor_list fp8_out, amp_tensor_list fp8_t_out,
    amp_dtype fp8_dtype, double eps, const float *amax_history, int hist_len, float *amax_dev,
    float *inv_scale_dev, const float *scale_dev, const int32_t *found_inf_dev, int32_t *step_dev,
    const amp_adamw_hyper *hyper, uint64_t seed, amp_stream_t stream) {
    AMP_TRACE("amp_adamw_master_step_fp8_delayed_sr");
    return delayed_entry("amp_adamw_master_step_fp8_delayed_sr", master, exp_avg, exp_avg_sq,
                         grads, bf16_out, master8, exp_avg8, exp_avg_sq8, grads8, bf16_out8,
                         fp8_out, fp8_t_out, fp8_dtype, eps, amax_history, hist_len, amax_dev,
                         inv_scale_dev, scale_dev, found_inf_dev, step_dev, hyper, stream, true,
                         seed);
}

amp_status amp_update_scale_fp8_history(float *scale_dev, int32_t *growth_tracker_dev,
                                        int32_t *found_inf_dev, float growth_factor,
                                        float backoff_factor, int32_t growth_interval,
                                        float *amax_dev, float *amax_history, int n_fp8,
                                        int hist_len, amp_stream_t stream) {
    AMP_TRACE("amp_update_scale_fp8_history");
    const char *fn = "amp_update_scale_fp8_history";
    if (!scale_dev || !growth_tracker_dev || !found_inf_dev)
        return fail(AMP_EINVAL, "%s: NULL state pointer", fn);
    if (growth_interval < 1) return fail(AMP_EINVAL, "%s: growth_interval < 1", fn);
    if (n_fp8 < 0 || hist_len < 1 || (n_fp8 > 0 && (!amax_dev || !amax_history)))
        return fail(AMP_EINVAL, "%s: bad amax / history arguments", fn);
    cudaError_t e = amp::launch_update_scale_hist(scale_dev, growth_tracker_dev, found_inf_dev,
                                                  growth_factor, backoff_factor, growth_interval,
                                                  amax_dev, amax_history, n_fp8, hist_len,
                                                  reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, fn);
}

amp_status amp_unscale_check_norm(amp_tensor_list grads, const float *scale_dev,
                                  int32_t *found_inf_dev, double *grad_sumsq_dev,
                                  amp_stream_t stream) {
    AMP_TRACE("amp_unscale_check_norm");
    if (!grads || !found_inf_dev || !grad_sumsq_dev)
        return fail(AMP_EINVAL, "amp_unscale_check_norm: NULL argument");
    const int ec = elem_code(grads->dtype);
    if (ec < 0) return fail(AMP_EDTYPE, "amp_unscale_check_norm: gradients must be f32/f16/bf16");
    cudaError_t e = amp::launch_check_norm(grads->view, grads->n_chunks, ec, scale_dev,
                                           found_inf_dev, grad_sumsq_dev,
                                           reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, "amp_unscale_check_norm");
}

amp_status fp8_quant_tensorwise(const void *x, amp_dtype x_dtype, int64_t rows, int64_t cols,
                                amp_dtype fp8_dtype, double eps, void *out, void *out_t,
                                float *inv_scale_dev, float *amax_dev, int amax_given,
                                const int32_t *skip_if_dev, amp_stream_t stream) {
    AMP_TRACE("fp8_quant_tensorwise");
    if (bad_shape(rows, cols)) return fail(AMP_EINVAL, "fp8_quant_tensorwise: negative or too large size");
    if (!inv_scale_dev || !amax_dev) return fail(AMP_EINVAL, "fp8_quant_tensorwise: NULL inv_scale/amax");
    if (rows * cols > 0 && (!x || !out)) return fail(AMP_EINVAL, "fp8_quant_tensorwise: NULL x/out");
    if (!(eps > 0.0)) return fail(AMP_EINVAL, "fp8_quant_tensorwise: eps must be > 0");
    const int xc = elem_code(x_dtype), fc = fp8_code(fp8_dtype);
    if (xc < 0 || fc < 0) return fail(AMP_EDTYPE, "fp8_quant_tensorwise: unsupported dtype");
    const int64_t tiles = ((rows + amp::kTile - 1) / amp::kTile) * ((cols + amp::kTile - 1) / amp::kTile);
    if (tiles > int64_t(INT32_MAX)) return fail(AMP_EINVAL, "fp8_quant_tensorwise: tensor too large");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "fp8_quant_tensorwise: cudaGetDevice");
    e = amp::launch_fp8_quant(x, xc, rows, cols, fc, eps, static_cast<uint8_t *>(out),
                              static_cast<uint8_t *>(out_t), inv_scale_dev, amax_dev,
                              amax_given ? 1 : 0, skip_if_dev, dev,
                              reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, "fp8_quant_tensorwise");
}

amp_status fp8_quant_rowwise(const void *x, amp_dtype x_dtype, int64_t rows, int64_t cols,
                             amp_dtype fp8_dtype, double eps, void *out, void *out_t,
                             float *amax_row, float *scale_row, float *inv_scale_row,
                             float *amax_col, float *scale_col, float *inv_scale_col,
                             const int32_t *skip_if_dev, amp_stream_t stream) {
    AMP_TRACE("fp8_quant_rowwise");
    const char *fn = "fp8_quant_rowwise";
    if (bad_shape(rows, cols)) return fail(AMP_EINVAL, "%s: negative or too large size", fn);
    if (rows * cols > 0 && (!x || !out || !amax_row || !scale_row || !inv_scale_row))
        return fail(AMP_EINVAL, "%s: NULL x / out / row outputs", fn);
    if (out_t && rows * cols > 0 && (!amax_col || !scale_col || !inv_scale_col))
        return fail(AMP_EINVAL, "%s: out_t needs the column outputs", fn);
    if (!(eps > 0.0)) return fail(AMP_EINVAL, "%s: eps must be > 0", fn);
    const int xc = elem_code(x_dtype), fc = fp8_code(fp8_dtype);
    if (xc < 0 || fc < 0) return fail(AMP_EDTYPE, "%s: unsupported dtype", fn);
    const int64_t tiles = ((rows + amp::kTile - 1) / amp::kTile) * ((cols + amp::kTile - 1) / amp::kTile);
    if (tiles > int64_t(INT32_MAX)) return fail(AMP_EINVAL, "%s: tensor too large", fn);
    if (rows * cols == 0) return AMP_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    e = amp::launch_fp8_quant_rowwise(x, xc, rows, cols, fc, eps, static_cast<uint8_t *>(out),
                                      static_cast<uint8_t *>(out_t), amax_row, scale_row,
                                      inv_scale_row, amax_col, scale_col, inv_scale_col,
                                      skip_if_dev, dev, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, fn);
}

amp_status fp8_quant_groupwise(const void *x, amp_dtype x_dtype, int64_t rows, int64_t cols,
                               int64_t group, amp_dtype fp8_dtype, double eps, void *out,
                               void *out_t, float *amax_rg, float *scale_rg, float *inv_rg,
                               float *amax_cg, float *scale_cg, float *inv_cg,
                               const int32_t *skip_if_dev, amp_stream_t stream) {
    AMP_TRACE("fp8_quant_groupwise");
    const char *fn = "fp8_quant_groupwise";
    if (bad_shape(rows, cols)) return fail(AMP_EINVAL, "%s: negative or too large size", fn);
    if (group != 32 && group != 64 && group != 128)
        return fail(AMP_EINVAL, "%s: group must be 32, 64 or 128", fn);
    if (rows * cols > 0 && (!x || !out || !amax_rg || !scale_rg || !inv_rg))
        return fail(AMP_EINVAL, "%s: NULL x / out / row-group outputs", fn);
    if (out_t && rows * cols > 0 && (!amax_cg || !scale_cg || !inv_cg))
        return fail(AMP_EINVAL, "%s: out_t needs the column-group outputs", fn);
    if (!(eps > 0.0)) return fail(AMP_EINVAL, "%s: eps must be > 0", fn);
    const int xc = elem_code(x_dtype), fc = fp8_code(fp8_dtype);
    if (xc < 0 || fc < 0) return fail(AMP_EDTYPE, "%s: unsupported dtype", fn);
    const int64_t tiles = ((rows + amp::kTile - 1) / amp::kTile) * ((cols + amp::kTile - 1) / amp::kTile);
    if (tiles > int64_t(INT32_MAX)) return fail(AMP_EINVAL, "%s: tensor too large", fn);
    if (rows * cols == 0) return AMP_OK;
    cudaError_t e = amp::launch_fp8_quant_groupwise(
        x, xc, rows, cols, group, fc, eps, static_cast<uint8_t *>(out),
        static_cast<uint8_t *>(out_t), amax_rg, scale_rg, inv_rg, amax_cg, scale_cg, inv_cg,
        skip_if_dev, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, fn);
}

static amp_status quant_list_entry(amp_tensor_list x, amp_tensor_list out, amp_tensor_list out_t,
                                   amp_dtype fp8_dtype, double eps, const float *amax_dev,
                                   float *inv_scale_dev, const int32_t *skip_if_dev,
                                   amp_stream_t stream, const int32_t *sr_step, uint64_t seed);

amp_status fp8_quant_tensorwise_list(amp_tensor_list x, amp_tensor_list out, amp_tensor_list out_t,
                                     amp_dtype fp8_dtype, double eps, const float *amax_dev,
                                     float *inv_scale_dev, const int32_t *skip_if_dev,
                                     amp_stream_t stream) {
    AMP_TRACE("fp8_quant_tensorwise_list");
    return quant_list_entry(x, out, out_t, fp8_dtype, eps, amax_dev, inv_scale_dev, skip_if_dev,
                            stream, nullptr, 0);
}

amp_status fp8_quant_tensorwise_list_sr(amp_tensor_list x, amp_tensor_list out,
                                        amp_tensor_list out_t, amp_dtype fp8_dtype, double eps,
                                        const float *amax_dev, float *inv_scale_dev,
                                        const int32_t *skip_if_dev, uint64_t seed,
                                        const int32_t *step_dev, amp_stream_t stream) {
    AMP_TRACE("fp8_quant_tensorwise_list_sr");
    if (!step_dev) return fail(AMP_EINVAL, "fp8_quant_tensorwise_list_sr: step_dev is NULL");
    if (x && x->n >= (1 << 30))
        return fail(AMP_EINVAL, "fp8_quant_tensorwise_list_sr: 2^30 tensors or more");
    return quant_list_entry(x, out, out_t, fp8_dtype, eps, amax_dev, inv_scale_dev, skip_if_dev,
                            stream, step_dev, seed);
}

static amp_status quant_list_entry(amp_tensor_list x, amp_tensor_list out, amp_tensor_list out_t,
                                   amp_dtype fp8_dtype, double eps, const float *amax_dev,
                                   float *inv_scale_dev, const int32_t *skip_if_dev,
                                   amp_stream_t stream, const int32_t *sr_step, uint64_t seed) {
    if (!x || !out || !amax_dev || !inv_scale_dev)
        return fail(AMP_EINVAL, "fp8_quant_tensorwise_list: NULL argument");
    if (x->has_slots && x->min_slot < 0)
        return fail(AMP_EINVAL,
                    "fp8_quant_tensorwise_list: x has amax slots, so every tensor needs one >= 0");
    if (!x->two_d || !out->two_d || (out_t && !out_t->two_d))
        return fail(AMP_EINVAL, "fp8_quant_tensorwise_list: lists must be 2-D");
    if (!(eps > 0.0)) return fail(AMP_EINVAL, "fp8_quant_tensorwise_list: eps must be > 0");
    const int xc = elem_code(x->dtype), fc = fp8_code(fp8_dtype);
    if (xc < 0 || fc < 0 || out->dtype != fp8_dtype || (out_t && out_t->dtype != fp8_dtype))
        return fail(AMP_EDTYPE, "fp8_quant_tensorwise_list: unsupported or mismatched dtype");
    if (out->n != x->n || out->rows != x->rows || out->cols != x->cols)
        return fail(AMP_EINVAL, "fp8_quant_tensorwise_list: out shapes differ from x");
    if (out_t && (out_t->n != x->n || out_t->rows != x->cols || out_t->cols != x->rows))
        return fail(AMP_EINVAL, "fp8_quant_tensorwise_list: out_t shapes are not x transposed");
    const bool any_empty =
        std::any_of(x->numel.begin(), x->numel.end(), [](int64_t k) { return k == 0; });
    cudaError_t e = amp::launch_fp8_quant_list(x->view, x->n_tiles, any_empty, xc, out->view,
                                               out_t ? &out_t->view : nullptr, fc, eps, amax_dev,
                                               inv_scale_dev, skip_if_dev,
                                               reinterpret_cast<cudaStream_t>(stream), sr_step,
                                               seed, x->has_slots);
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, "fp8_quant_tensorwise_list");
}

amp_status amp_update_scale(float *scale_dev, int32_t *growth_tracker_dev, int32_t *found_inf_dev,
                            float growth_factor, float backoff_factor, int32_t growth_interval,
                            float *amax_dev, int n_amax, amp_stream_t stream) {
    AMP_TRACE("amp_update_scale");
    if (!scale_dev || !growth_tracker_dev || !found_inf_dev)
        return fail(AMP_EINVAL, "amp_update_scale: NULL state pointer");
    if (growth_interval < 1) return fail(AMP_EINVAL, "amp_update_scale: growth_interval < 1");
    if (n_amax < 0 || (n_amax > 0 && !amax_dev))
        return fail(AMP_EINVAL, "amp_update_scale: bad amax arguments");
    cudaError_t e = amp::launch_update_scale(scale_dev, growth_tracker_dev, found_inf_dev,
                                             growth_factor, backoff_factor, growth_interval,
                                             amax_dev, n_amax,
                                             reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, "amp_update_scale");
}

amp_status amp_read_state(const float *scale_dev, const int32_t *growth_tracker_dev,
                          const int32_t *step_dev, const int32_t *found_inf_dev,
                          amp_scaler_state *host_out, amp_stream_t stream) {
    AMP_TRACE("amp_read_state");
    if (!host_out) return fail(AMP_EINVAL, "amp_read_state: host_out is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const void *src[4] = {scale_dev, growth_tracker_dev, step_dev, found_inf_dev};
    void *dst[4] = {&host_out->scale, &host_out->growth_tracker, &host_out->step,
                    &host_out->found_inf};
    for (int i = 0; i < 4; ++i) {
        if (!src[i]) continue;
        cudaError_t e = cudaMemcpyAsync(dst[i], src[i], 4, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e, "amp_read_state");
    }
    return AMP_OK;
}

amp_status amp_scale_health(const float *scale_dev, float min_scale, int32_t *health_dev,
                            amp_stream_t stream) {
    AMP_TRACE("amp_scale_health");
    if (!scale_dev || !health_dev) return fail(AMP_EINVAL, "amp_scale_health: NULL pointer");
    if (!(min_scale >= 0.0f)) return fail(AMP_EINVAL, "amp_scale_health: min_scale must be >= 0");
    cudaError_t e = amp::launch_scale_health(scale_dev, min_scale, health_dev,
                                             reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? AMP_OK : cuda_fail(e, "amp_scale_health");
}

}  // extern "C"
