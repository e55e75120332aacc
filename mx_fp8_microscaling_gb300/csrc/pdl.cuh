// Programmatic dependent launch for the libmx kernels.
//
// Every kernel is launched with programmatic stream serialization allowed,
// so the next kernel on a stream may be scheduled before the current one has
// finished.  Each kernel calls pdl_allow_next() as it starts: the next grid
// is launched once every block of the current grid has made that call (so
// all of them are already running, and none can be starved of an SM by the
// next grid).  Each kernel calls pdl_wait_prior() before it reads or writes
// any memory another kernel may touch; the wait returns when every earlier
// grid on the stream has completed and its memory operations are visible.
// What overlaps the previous kernel's tail is therefore only launch latency
// and set-up (index math, barrier initialisation, tensor-memory allocation).
// Without a programmatic predecessor (a copy, an event wait, a kernel
// launched without the attribute) the wait returns at once.
#pragma once

#include <cuda_runtime.h>

namespace mx {
namespace dev {

__device__ __forceinline__ void pdl_allow_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void pdl_wait_prior() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace dev

inline cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute a{};
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

// kernel<<<grid, block, smem, stream>>>(args...) with the attribute above.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace mx
