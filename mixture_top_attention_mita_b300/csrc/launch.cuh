// Chained launches: programmatic dependent launch between the kernels of one
// stream.  A chained launch may begin while the previous kernel on the stream
// is still running its last blocks; every kernel of a chain therefore starts
// with chain_wait_and_trigger():
//   griddepcontrol.wait               no read (and no tensor-memory
//                                     allocation) before the previous grid
//                                     has completed and its writes are
//                                     visible; a no-op for a plain launch
//   griddepcontrol.launch_dependents  the next chained kernel may launch
//                                     once every block of this one has begun
// Because every block of every chained kernel waits before it can finish, a
// kernel completes only after all kernels before it on the stream: results
// of any earlier kernel in the chain are visible, not only the previous one's.
#pragma once

#include <cuda_runtime.h>

#include <utility>

#include "common.cuh"

namespace mita {

MITA_DEV void chain_wait_and_trigger() {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// `overlap` false gives a plain launch (the kernel's wait is then a no-op).
template <typename... P, typename... A>
cudaError_t launch_chained(bool overlap, void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                           A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

}  // namespace mita
