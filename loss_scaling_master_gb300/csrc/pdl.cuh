// pdl.cuh - programmatic dependent launch: a kernel of the chain may be
// scheduled while the kernel before it in the stream drains, so its launch
// and CTA ramp-up overlap that tail instead of following it.
//
// Contract of every kernel launched with launch_pdl: it calls pdl_wait()
// before its first global-memory access.  griddepcontrol.wait returns once
// every prerequisite grid has completed and its memory operations are
// visible, so data dependencies (read-after-write and write-after-read) are
// exactly those of plain stream order.  pdl_trigger() after the wait lets the
// next kernel of the stream be scheduled as soon as every CTA of this one has
// started; it never lets that kernel read before this one completes, because
// it waits in turn.  The wait is the hardware's own dependency mechanism, not
// a spin loop.  Where the stream holds no kernel before it, or the previous
// kernel never triggers, the wait returns when plain stream order would have
// started the kernel.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace amp {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace amp
