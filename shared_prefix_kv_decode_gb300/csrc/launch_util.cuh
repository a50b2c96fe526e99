// launch_util.cuh -- kernel launch helpers: programmatic dependent launch and the shared-memory
// carveout.
//
// Programmatic dependent launch (PDL): a kernel launched with the programmatic stream
// serialisation attribute may be scheduled while the kernel before it in the stream is still
// running, once every CTA of that kernel has executed griddepcontrol.launch_dependents (or
// exited).  It then runs its set-up (barrier init, TMEM allocation, plan loads) early and
// blocks in griddepcontrol.wait until the earlier kernel has completed and its writes are
// visible.  Every kernel of the decode path executes griddepcontrol.wait before it reads data
// that earlier work in the stream may write (q, the pools, the token tables, partial records)
// and before it writes anything, so a chain of such kernels keeps stream order for memory.
// Without the attribute both instructions are no-ops.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace granikv {

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Ask for the largest shared-memory carveout, so that an SM switching between this kernel and
// the tensor-core kernels (which need nearly all of it) does not reconfigure its L1/shared split.
template <typename K>
inline cudaError_t prefer_max_shared(K kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

}  // namespace granikv
