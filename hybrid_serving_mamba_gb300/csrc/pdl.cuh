// Programmatic dependent launch: a kernel launched this way may be scheduled while the stream's
// previous kernel drains (once that kernel's CTAs have executed griddepcontrol.launch_dependents or
// exited); it must execute griddepcontrol.wait, which returns once that grid has completed and its
// writes are visible, before it reads anything the grid writes.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace ssm {

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}

}  // namespace ssm
