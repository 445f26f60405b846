// adamw_noalloc.cu - amp_adamw_master_step_noalloc: the FP32-master AdamW
// step for callers that cannot allocate device memory.
//
// Who needs it: amp_adamw_master_step works on tensor-list handles, and
// creating a handle calls cudaMalloc for the handle's tables.  Some callers
// cannot do that - runtimes that hand out every byte of device memory from
// their own arena and reject allocations made behind their back, training
// loops that must not hit the implicit device synchronisation of
// cudaMalloc/cudaFree, processes running with the GPU nearly full where a late
// allocation could fail mid-run, and plain-C callers that cannot manage a
// handle's lifetime.  This entry point takes the tensors as plain arrays and
// keeps everything else it needs in one fixed device array compiled into the
// library.
//
// The array: kNoallocScratchBytes (about 4.1 MB) in a file-scope static
// __device__ buffer that every GPU loading the library holds until the process
// exits.  It holds the per-call tables (tensor pointers, sizes, amax slots,
// the chunk table) and the 16-byte per-step scalar block the AdamW prologue
// writes.  Limits: at most kNoallocMaxTensors tensors and kNoallocMaxChunks
// chunks of 16384 elements (8,589,934,592 elements in all); larger calls are
// rejected with AMP_EINVAL.
//
// Every call shares the array and it keeps the last call's contents.  Each
// call rewrites the tables it reads, and the prologue writes the step scalars
// before the main kernel reads them, so none of those need to start at zero.
// The one word that does is the sticky error word next to the step scalars:
// it relies on the array's static zero-initialisation, is set only by a
// bounded wait that gives up, and is cleared only by amp_noalloc_check.
// Calls whose work overlaps on the GPU (different streams without ordering)
// race on the array; order them on one stream.
//
// The tables travel with one cudaMemcpyAsync from a pageable host vector
// (pinning it would be an allocation).  CUDA stages a pageable copy through
// its own buffers and may wait for the stream to drain before it returns, so
// a call can block the host until earlier work on `stream` is done.  A copy
// from pageable memory cannot be recorded into a CUDA graph, and a recorded
// one would replay from a vector freed on return, so a call on a capturing
// stream is refused with AMP_EINVAL before anything is enqueued.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"

namespace {

constexpr int kNoallocMaxTensors = 1024;
constexpr int64_t kNoallocMaxChunks = 524288;
constexpr size_t kAlign = 256;
constexpr size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
// scalars | 5 pointer arrays | numel | slots | chunks, each 256-byte aligned
constexpr size_t kNoallocScratchBytes =
    kAlign + 5 * align_up(kNoallocMaxTensors * sizeof(void *)) +
    align_up(kNoallocMaxTensors * sizeof(int64_t)) + align_up(kNoallocMaxTensors * sizeof(int32_t)) +
    align_up(size_t(kNoallocMaxChunks) * sizeof(uint2));

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device.  In host
// code the symbol name is only a host-side stand-in for the array; handing it
// to a kernel would read the wrong memory.
std::mutex g_mu;
std::vector<unsigned char *> g_scratch_ptr;

cudaError_t scratch_on_current_device(unsigned char **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    if (dev >= int(g_scratch_ptr.size())) g_scratch_ptr.resize(dev + 1, nullptr);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

// Report through the library-wide per-thread message (amp_last_error).
amp_status noalloc_fail(amp_status st, const char *fmt, ...) {
    char msg[256];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof(msg), fmt, ap);
    va_end(ap);
    amp::set_last_error(msg);
    return st;
}

// The body of amp_adamw_master_step_noalloc; its host vectors may throw
// std::bad_alloc, which the entry point reports as AMP_ENOMEM.
amp_status noalloc_step(int n, float *const *master, float *const *exp_avg,
                        float *const *exp_avg_sq, const void *const *grads, amp_dtype grad_dtype,
                        uint16_t *const *bf16_out, const int64_t *numel,
                        const int32_t *amax_slots, const float *scale_dev,
                        const int32_t *found_inf_dev, int32_t *step_dev,
                        const amp_adamw_hyper *hyper, float *amax_dev, amp_stream_t stream) {
    const char *fn = "amp_adamw_master_step_noalloc";
    if (n < 0 || (n > 0 && (!master || !exp_avg || !exp_avg_sq || !grads || !numel)) ||
        !step_dev || !hyper)
        return noalloc_fail(AMP_EINVAL, "%s: NULL argument or n < 0", fn);
    if (n > kNoallocMaxTensors)
        return noalloc_fail(AMP_EINVAL, "%s: %d tensors exceed the limit of %d", fn, n,
                            kNoallocMaxTensors);
    int gelem = -1;
    if (grad_dtype == AMP_DT_F32) gelem = amp::kF32;
    if (grad_dtype == AMP_DT_F16) gelem = amp::kF16;
    if (grad_dtype == AMP_DT_BF16) gelem = amp::kBF16;
    if (gelem < 0) return noalloc_fail(AMP_EDTYPE, "%s: gradients must be f32/f16/bf16", fn);
    bool any_slot = false;
    int64_t n_chunks = 0;
    for (int i = 0; i < n; ++i) {
        if (numel[i] < 0) return noalloc_fail(AMP_EINVAL, "%s: negative size at tensor %d", fn, i);
        if (numel[i] > 0 && (!master[i] || !exp_avg[i] || !exp_avg_sq[i] || !grads[i] ||
                             (bf16_out && !bf16_out[i])))
            return noalloc_fail(AMP_EINVAL, "%s: NULL pointer of non-empty tensor %d", fn, i);
        // ceil without forming numel + kChunk - 1, which could pass INT64_MAX;
        // each term is below 2^50 and there are at most 1024 of them
        n_chunks += numel[i] / amp::kChunk + (numel[i] % amp::kChunk != 0);
        if (amax_slots && bf16_out && amax_slots[i] >= 0) any_slot = true;
    }
    if (n_chunks > kNoallocMaxChunks)
        return noalloc_fail(AMP_EINVAL,
                            "%s: %lld chunks of %d elements exceed the limit of %lld", fn,
                            (long long)n_chunks, amp::kChunk, (long long)kNoallocMaxChunks);
    if (any_slot && !amax_dev)
        return noalloc_fail(AMP_EINVAL, "%s: amax slots given but amax_dev is NULL", fn);

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess)
        return noalloc_fail(AMP_ECUDA, "%s: cudaStreamIsCapturing: %s", fn, cudaGetErrorString(e));
    if (cap != cudaStreamCaptureStatusNone)
        return noalloc_fail(AMP_EINVAL,
                            "%s: the stream is capturing a CUDA graph; this entry point uploads "
                            "its tables from pageable host memory and cannot be captured", fn);

    unsigned char *base = nullptr;
    e = scratch_on_current_device(&base);
    if (e != cudaSuccess)
        return noalloc_fail(AMP_ECUDA, "%s: cudaGetSymbolAddress: %s", fn, cudaGetErrorString(e));

    // Compact per-call layout after the scalar block.
    const size_t nn = size_t(n > 0 ? n : 1);
    const size_t o_ptr[5] = {kAlign, kAlign + align_up(nn * 8), kAlign + 2 * align_up(nn * 8),
                             kAlign + 3 * align_up(nn * 8), kAlign + 4 * align_up(nn * 8)};
    const size_t o_numel = kAlign + 5 * align_up(nn * 8);
    const size_t o_slots = o_numel + align_up(nn * sizeof(int64_t));
    const size_t o_chunks = o_slots + align_up(nn * sizeof(int32_t));
    const size_t end = o_chunks + size_t(n_chunks) * sizeof(uint2);
    std::vector<unsigned char> host(end - kAlign, 0);
    auto put = [&](size_t off, const void *src, size_t bytes) {
        if (bytes) std::memcpy(host.data() + (off - kAlign), src, bytes);
    };
    put(o_ptr[0], master, n * sizeof(void *));
    put(o_ptr[1], exp_avg, n * sizeof(void *));
    put(o_ptr[2], exp_avg_sq, n * sizeof(void *));
    put(o_ptr[3], grads, n * sizeof(void *));
    if (bf16_out) put(o_ptr[4], bf16_out, n * sizeof(void *));
    put(o_numel, numel, n * sizeof(int64_t));
    std::vector<int32_t> slots(nn, -1);
    if (amax_slots && bf16_out)
        for (int i = 0; i < n; ++i) slots[i] = amax_slots[i];
    put(o_slots, slots.data(), nn * sizeof(int32_t));
    std::vector<uint2> chunks;
    chunks.reserve(size_t(n_chunks));
    for (int i = 0; i < n; ++i)
        for (int64_t k = 0; k * amp::kChunk < numel[i]; ++k) chunks.push_back(make_uint2(i, uint32_t(k)));
    put(o_chunks, chunks.data(), chunks.size() * sizeof(uint2));

    // Pageable source: the runtime stages it before returning (waiting for the
    // stream if it must), so `host` may go out of scope; the copy is ordered
    // before the kernels on `s`.
    e = cudaMemcpyAsync(base + kAlign, host.data(), host.size(), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess)
        return noalloc_fail(AMP_ECUDA, "%s: table upload: %s", fn, cudaGetErrorString(e));

    amp::ListView v[5];
    for (int k = 0; k < 5; ++k) {
        v[k] = amp::ListView{};
        v[k].ptrs = reinterpret_cast<void *const *>(base + o_ptr[k]);
        v[k].numel = reinterpret_cast<const int64_t *>(base + o_numel);
        v[k].slots = reinterpret_cast<const int32_t *>(base + o_slots);
        v[k].chunks = reinterpret_cast<const uint2 *>(base + o_chunks);
        v[k].n = n;
    }
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
    e = amp::launch_adamw(v[0], v[1], v[2], v[3], bf16_out ? &v[4] : nullptr, n_chunks, gelem,
                          scale_dev, found_inf_dev, step_dev, c,
                          reinterpret_cast<amp::AdamwStepScalars *>(base), amax_dev, any_slot, s);
    if (e != cudaSuccess) return noalloc_fail(AMP_ECUDA, "%s: %s", fn, cudaGetErrorString(e));
    return AMP_OK;
}

}  // namespace

extern "C" amp_status amp_adamw_master_step_noalloc(
    int n, float *const *master, float *const *exp_avg, float *const *exp_avg_sq,
    const void *const *grads, amp_dtype grad_dtype, uint16_t *const *bf16_out,
    const int64_t *numel, const int32_t *amax_slots, const float *scale_dev,
    const int32_t *found_inf_dev, int32_t *step_dev, const amp_adamw_hyper *hyper,
    float *amax_dev, amp_stream_t stream) {
    AMP_TRACE("amp_adamw_master_step_noalloc");
    try {
        return noalloc_step(n, master, exp_avg, exp_avg_sq, grads, grad_dtype, bf16_out, numel,
                            amax_slots, scale_dev, found_inf_dev, step_dev, hyper, amax_dev,
                            stream);
    } catch (const std::bad_alloc &) {
        return noalloc_fail(AMP_ENOMEM,
                            "amp_adamw_master_step_noalloc: host allocation of the tables failed");
    }
}

extern "C" amp_status amp_noalloc_check(amp_stream_t stream) {
    AMP_TRACE("amp_noalloc_check");
    const char *fn = "amp_noalloc_check";
    unsigned char *base = nullptr;
    cudaError_t e = scratch_on_current_device(&base);
    if (e != cudaSuccess)
        return noalloc_fail(AMP_ECUDA, "%s: cudaGetSymbolAddress: %s", fn, cudaGetErrorString(e));
    int32_t *word = reinterpret_cast<int32_t *>(base) + amp::kErrWordOffset;
    int32_t v = 0;
    e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && v != 0) {
        const int32_t zero = 0;
        e = cudaMemcpy(word, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e == cudaSuccess)
            return noalloc_fail(AMP_ETIMEOUT,
                                "%s: a kernel's bounded wait for its asynchronous copies gave up; "
                                "the chunks it held were not updated", fn);
    }
    if (e != cudaSuccess) return noalloc_fail(AMP_ECUDA, "%s: %s", fn, cudaGetErrorString(e));
    return AMP_OK;
}
