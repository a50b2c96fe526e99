// kernels_dense_tc.cu -- the tensor-core decode kernels: the dense prefix kernel on its own,
// and the prefix-and-suffix kernel whose first CTAs run dense prefix work items and the rest
// suffix token-CTAs (one launch for both, so the merge kernel can follow it directly).  The
// bodies, with the design notes, are in dense_tc_body.cuh and suffix_mma_body.cuh.
#include "dense_tc_body.cuh"
#include "suffix_mma_body.cuh"

namespace granikv {
namespace {

__global__ void __launch_bounds__(dns::kThreads, 1)
    dense_tc_kernel(AttnParams p, int32_t first_item, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmq) {
  extern __shared__ unsigned char smem_raw[];
  dns::dense_tc_body(p, first_item + (int32_t)blockIdx.x, &tmk, &tmv, &tmq, smem_raw);
}

constexpr int kPsSmemBytes = dns::kSmemBytes > sfx::kSmemBytes ? dns::kSmemBytes : sfx::kSmemBytes;
static_assert(sfx::kThreads <= dns::kThreads, "the suffix body runs on the dense block size");

// CTAs [0, n_dense) run prefix items first_item.., the rest suffix token-CTAs: CTA n_dense + k
// is token-CTA k % n_scta of KV-head group k / n_scta.
__global__ void __launch_bounds__(dns::kThreads, 1)
    prefix_suffix_tc_kernel(AttnParams p, int32_t first_item, int32_t n_dense, const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmq,
                            const int32_t* __restrict__ cta_begin, int32_t n_scta) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  if ((int32_t)blockIdx.x < n_dense) {
    dns::dense_tc_body(p, first_item + (int32_t)blockIdx.x, &tmk, &tmv, &tmq, smem_raw);
  } else {
    const int32_t k = (int32_t)blockIdx.x - n_dense;
    sfx::suffix_mma_body(p, cta_begin, k % n_scta, k / n_scta, smem_raw);
  }
}

}  // namespace

cudaError_t launch_dense_tc(const AttnParams& p, int32_t first_item, int32_t n_items, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, const CUtensorMap& tmq, cudaStream_t s, bool pdl) {
  if (n_items <= 0) return cudaSuccess;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(dense_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dns::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  return launch_kernel(dense_tc_kernel, dim3(n_items), dim3(dns::kThreads), dns::kSmemBytes, s, pdl, p, first_item, tmk, tmv, tmq);
}

cudaError_t launch_prefix_suffix_tc(const AttnParams& p, int32_t first_item, int32_t n_dense, const CUtensorMap& tmk,
                                    const CUtensorMap& tmv, const CUtensorMap& tmq, const int32_t* cta_begin,
                                    int32_t n_scta, cudaStream_t s, bool pdl) {
  const int32_t groups = (p.n_kv + sfx::kWarps - 1) / sfx::kWarps;
  const int64_t n = (int64_t)n_dense + (int64_t)n_scta * groups;
  if (n <= 0) return cudaSuccess;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(prefix_suffix_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPsSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  return launch_kernel(prefix_suffix_tc_kernel, dim3((unsigned)n), dim3(dns::kThreads), kPsSmemBytes, s, pdl, p,
                       first_item, n_dense, tmk, tmv, tmq, cta_begin, n_scta);
}

}  // namespace granikv
