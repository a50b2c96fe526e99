// kernels_suffix_mma.cu -- the COLD suffix kernel on its own (serial path, and the concurrent
// path when the prefix does not run on the dense tensor-core kernel); its body, with the design
// notes, is in suffix_mma_body.cuh.
#include "suffix_mma_body.cuh"

namespace granikv {
namespace {

__global__ void __launch_bounds__(sfx::kThreads, 1) suffix_mma_kernel(AttnParams p, const int32_t* __restrict__ cta_begin) {
  extern __shared__ __align__(128) unsigned char smem[];
  sfx::suffix_mma_body(p, cta_begin, blockIdx.x, blockIdx.y, smem);
}

}  // namespace

cudaError_t launch_suffix_mma(const AttnParams& p, const int32_t* cta_begin, int32_t n_cta, cudaStream_t s,
                              bool pdl) {
  if (n_cta <= 0) return cudaSuccess;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(suffix_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sfx::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  dim3 grid(n_cta, (p.n_kv + sfx::kWarps - 1) / sfx::kWarps);
  return launch_kernel(suffix_mma_kernel, grid, dim3(sfx::kThreads), sfx::kSmemBytes, s, pdl, p, cta_begin);
}

}  // namespace granikv
