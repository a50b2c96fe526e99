// kernels_dense_tc.cu -- the tensor-core decode kernels: the dense prefix kernel and the
// streaming cascade kernel on their own, and the prefix-and-suffix kernel whose first CTAs run
// prefix work items (dense, then streaming cascade) and the rest suffix token-CTAs (one launch
// for all, so the merge kernel can follow it directly).  The bodies, with the design notes, are
// in dense_tc_body.cuh, cascade_stream_body.cuh and suffix_mma_body.cuh.
#include "cascade_stream_body.cuh"
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

constexpr int kPsSmemBytes0 = dns::kSmemBytes > sfx::kSmemBytes ? dns::kSmemBytes : sfx::kSmemBytes;
constexpr int kPsSmemBytes = kPsSmemBytes0 > csc::kSmemBytes ? kPsSmemBytes0 : csc::kSmemBytes;
static_assert(sfx::kThreads <= dns::kThreads, "the suffix body runs on the dense block size");
static_assert(csc::kThreads <= dns::kThreads, "the cascade body runs on the dense block size");

// CTAs [0, n_dense) run dense prefix items first_dense.., the next n_casc streaming cascade
// items first_casc.., the rest suffix token-CTAs: CTA n_dense + n_casc + k is token-CTA
// k % n_scta of KV-head group k / n_scta.  Dense CTA c < n_tail then runs suffix token-CTA
// n_scta + c (one KV-head group only): suffix work the plan gives the dense CTAs for after
// their prefix piece, so that both sides of the grid end together.
__global__ void __launch_bounds__(dns::kThreads, 1)
    prefix_suffix_tc_kernel(AttnParams p, int32_t first_dense, int32_t n_dense, int32_t first_casc, int32_t n_casc,
                            const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                            const __grid_constant__ CUtensorMap tmq, const int32_t* __restrict__ cta_begin,
                            int32_t n_scta, int32_t n_tail) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int32_t c = (int32_t)blockIdx.x;
  if (c < n_dense) {
    dns::dense_tc_body(p, first_dense + c, &tmk, &tmv, &tmq, smem_raw);
    if (c < n_tail) {
      // the dense body has returned on every thread: its copies have landed, its MMAs have
      // completed and its tensor memory is freed, so its shared memory is free for the suffix
      // body (which initialises its own barriers)
      __syncthreads();
      fence_proxy_async_smem();
      sfx::suffix_mma_body(p, cta_begin, n_scta + c, 0, smem_raw);
    }
  } else if (c < n_dense + n_casc) {
    csc::cascade_stream_body(p, first_casc + (c - n_dense), smem_raw);
  } else {
    const int32_t k = c - n_dense - n_casc;
    sfx::suffix_mma_body(p, cta_begin, k % n_scta, k / n_scta, smem_raw);
  }
}

__global__ void __launch_bounds__(csc::kThreads, 1) cascade_stream_kernel(AttnParams p, int32_t first_item) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  csc::cascade_stream_body(p, first_item + (int32_t)blockIdx.x, smem_raw);
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

cudaError_t launch_cascade_stream(const AttnParams& p, int32_t first_item, int32_t n_items, cudaStream_t s, bool pdl) {
  if (n_items <= 0) return cudaSuccess;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(cascade_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, csc::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  return launch_kernel(cascade_stream_kernel, dim3(n_items), dim3(csc::kThreads), csc::kSmemBytes, s, pdl, p,
                       first_item);
}

cudaError_t launch_prefix_suffix_tc(const AttnParams& p, int32_t first_dense, int32_t n_dense, int32_t first_casc,
                                    int32_t n_casc, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                    const CUtensorMap& tmq, const int32_t* cta_begin, int32_t n_scta, int32_t n_tail,
                                    cudaStream_t s, bool pdl) {
  const int32_t groups = (p.n_kv + sfx::kWarps - 1) / sfx::kWarps;
  const int64_t n = (int64_t)n_dense + n_casc + (int64_t)n_scta * groups;
  if (n <= 0) return cudaSuccess;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(prefix_suffix_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPsSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  return launch_kernel(prefix_suffix_tc_kernel, dim3((unsigned)n), dim3(dns::kThreads), kPsSmemBytes, s, pdl, p,
                       first_dense, n_dense, first_casc, n_casc, tmk, tmv, tmq, cta_begin, n_scta, n_tail);
}

}  // namespace granikv
