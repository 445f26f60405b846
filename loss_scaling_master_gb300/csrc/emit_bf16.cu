// emit_bf16.cu - A5 on its own: the bf16 working copy of an fp32 master list,
// with the per-tensor amax fold of the FP8 weights.
//
//   "从 AMP 到 Mixed Precision" section "PyTorch AMP 与 FP32 Master Weights"
//   (mode B: the model holds bf16 parameters, the optimizer an fp32 master of
//   each) and "为什么需要 FP32 Master Weights": the working copy is the master
//   rounded to bf16.  The AdamW pass emits it after every step; a run needs it
//   once more before its first step, for the first forward pass, and the
//   delayed FP8 scaling of "第20章 量化与混合精度训练" §20.5.9 needs the amax
//   of that first copy to open its history.
//
// One CTA per chunk of 16384 elements: 16-byte loads of 8 fp32 values, one
// 16-byte store of 8 bf16 values (cvt.rn.bf16x2.f32, NaN -> 0x7FC0), and the
// amax of |bf16| by lane-wise 16-bit maxima and one atomicMax per warp on the
// fp32 bit pattern, as in the AdamW pass.  6 bytes per element.
#include "internal.h"
#include "pdl.cuh"

namespace amp {
namespace {

struct EmitParams {
    ListView p, b;
    float *amax;
    int use_slots;
};

__global__ void __launch_bounds__(kThreads) emit_bf16_kernel(EmitParams P) {
    pdl_wait();
    pdl_trigger();
    const uint2 ch = P.p.chunks[blockIdx.x];
    const int t = int(ch.x);
    const int64_t start = int64_t(ch.y) * kChunk;
    const int64_t n = min(int64_t(kChunk), P.p.numel[t] - start);
    const float *pp = static_cast<const float *>(P.p.ptrs[t]) + start;
    uint16_t *bp = static_cast<uint16_t *>(P.b.ptrs[t]) + start;
    uint32_t amax2 = 0, amax1 = 0;
    int64_t done = 0;
    if (aligned16(pp) && aligned16(bp)) {
        const int64_t nb = n & ~int64_t(7);
#pragma unroll 2
        for (int64_t e = 8 * int64_t(threadIdx.x); e < nb; e += 8 * kThreads) {
            const uint4 a = ld16(pp + e), c = ld16(pp + e + 4);
            uint4 o;
            o.x = f32x2_to_bf16x2(__uint_as_float(a.x), __uint_as_float(a.y));
            o.y = f32x2_to_bf16x2(__uint_as_float(a.z), __uint_as_float(a.w));
            o.z = f32x2_to_bf16x2(__uint_as_float(c.x), __uint_as_float(c.y));
            o.w = f32x2_to_bf16x2(__uint_as_float(c.z), __uint_as_float(c.w));
            st16(bp + e, o);
            amax2 = __vmaxu2(amax2, __vmaxu2(__vmaxu2(o.x & 0x7FFF7FFFu, o.y & 0x7FFF7FFFu),
                                             __vmaxu2(o.z & 0x7FFF7FFFu, o.w & 0x7FFF7FFFu)));
        }
        done = nb;
    }
    for (int64_t k = done + threadIdx.x; k < n; k += kThreads) {
        const uint16_t b = f32_to_bf16(pp[k]);
        bp[k] = b;
        amax1 = max(amax1, uint32_t(b & 0x7FFFu));
    }
    if (P.use_slots) {
        const int slot = P.b.slots[t];
        if (slot >= 0) {
            // |bf16| bit patterns order like their values, NaN (0x7FC0) above inf
            uint32_t a = max(max(amax2 & 0xFFFFu, amax2 >> 16), amax1);
            a = warp_max_u32(a);
            if ((threadIdx.x & 31) == 0 && a != 0)
                atomicMax(reinterpret_cast<unsigned int *>(P.amax) + slot, a << 16);
        }
    }
}

}  // namespace

cudaError_t launch_emit_bf16(const ListView &p, const ListView &b, int64_t n_chunks, float *amax,
                             bool use_slots, cudaStream_t s) {
    if (n_chunks == 0) return cudaSuccess;
    EmitParams P;
    P.p = p;
    P.b = b;
    P.amax = amax;
    P.use_slots = use_slots ? 1 : 0;
    cudaError_t e = launch_pdl(emit_bf16_kernel, dim3((unsigned)n_chunks), dim3(kThreads), 0, s, P);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace amp
