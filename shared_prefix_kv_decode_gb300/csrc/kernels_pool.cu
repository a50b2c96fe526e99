// kernels_pool.cu -- COLD pool kernels: slot allocation from the free ring, slot release, and
// the scatter of new tokens' K/V into their slots.
//
// GraniKV (arXiv:2608.15584), "1 Introduction" and "3 GraniKV": suffix and decoded tokens
// live in a token-level COLD pool with page size 1; the card page calls its allocator a
// token-level free list.  The ring's head and tail are tracked on the host (every allocation
// and release passes through the host API with host-known counts) and mirrored in a device
// word pair that these kernels keep current, so that the graph-safe allocation (which must not
// depend on host state captured once) can read the ring position on the device.
#include "internal.h"

namespace granikv {
namespace {

__device__ __forceinline__ void latch(int32_t* err, int32_t code) { atomicCAS(err, 0, code); }

// One block per request: pop excl[b+1]-excl[b] ring entries starting at head + excl[b],
// append them to the request's token table and (optionally) to slots_out.
__global__ void cold_alloc_kernel(const int32_t* __restrict__ excl, int32_t B,
                                  const int32_t* __restrict__ ring, int64_t n_cold, int64_t head,
                                  int32_t* __restrict__ req_to_slot, int32_t* __restrict__ suffix_len,
                                  int32_t cap, int32_t* __restrict__ slots_out, int64_t* ring_pos,
                                  int32_t* err) {
  if (blockIdx.x == 0 && threadIdx.x == 0) ring_pos[0] = head + excl[B];  // nothing here reads it
  for (int32_t b = blockIdx.x; b < B; b += gridDim.x) {
    const int32_t start = excl[b];
    const int32_t n = excl[b + 1] - start;
    if (n == 0) continue;
    const int32_t len = suffix_len[b];
    __syncthreads();  // every thread has read suffix_len[b] before thread 0 updates it
    if (len < 0 || (int64_t)len + n > cap) {
      if (threadIdx.x == 0) latch(err, kDevTableOverflow);
      continue;
    }
    int32_t* row = req_to_slot + (int64_t)b * cap + len;
    for (int32_t i = threadIdx.x; i < n; i += blockDim.x) {
      const int32_t slot = ring[(head + start + i) % n_cold];
      row[i] = slot;
      if (slots_out) slots_out[start + i] = slot;
    }
    __syncthreads();
    if (threadIdx.x == 0) suffix_len[b] = len + n;
  }
}

// Allocation of n slots for each of requests 0..B-1 that takes the ring position from the
// device (ring_pos = {head, tail}, absolute counts) and checks there that enough slots are free
// (else nothing is popped and kDevColdEmpty is latched).  One block: every thread reads the
// position before it moves; one thread per request (n is small: decode steps use 1).
__global__ void cold_alloc_uniform_kernel(int32_t n, int32_t B, const int32_t* __restrict__ ring, int64_t n_cold,
                                          int32_t* __restrict__ req_to_slot, int32_t* __restrict__ suffix_len,
                                          int32_t cap, int32_t* __restrict__ slots_out, int64_t* ring_pos,
                                          int32_t* err) {
  __shared__ int64_t s_head;
  __shared__ int s_ok;
  const int64_t total = (int64_t)n * B;
  if (threadIdx.x == 0) {
    const int64_t head = ring_pos[0], tail = ring_pos[1];
    s_head = head;
    s_ok = tail - head >= total ? 1 : 0;
    if (!s_ok) latch(err, kDevColdEmpty);
  }
  __syncthreads();
  if (!s_ok) return;
  const int64_t head = s_head;
  for (int32_t b = threadIdx.x; b < B; b += blockDim.x) {
    const int32_t len = suffix_len[b];
    if (len < 0 || (int64_t)len + n > cap) {
      latch(err, kDevTableOverflow);
      continue;
    }
    int32_t* row = req_to_slot + (int64_t)b * cap + len;
    for (int32_t i = 0; i < n; ++i) {
      const int32_t slot = ring[(head + (int64_t)b * n + i) % n_cold];
      row[i] = slot;
      if (slots_out) slots_out[(int64_t)b * n + i] = slot;
    }
    suffix_len[b] = len + n;
  }
  __syncthreads();
  if (threadIdx.x == 0) ring_pos[0] = head + total;
}

__global__ void cold_free_kernel(const int32_t* __restrict__ slots, int32_t n, int32_t* __restrict__ ring,
                                 int64_t n_cold, int64_t tail, int64_t n_hot, int64_t n_slots,
                                 int32_t checks, int64_t* ring_pos, int32_t* err) {
  if (blockIdx.x == 0 && threadIdx.x == 0) ring_pos[1] = tail + n;  // nothing here reads it
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t s = slots[i];
    if (checks && (s < n_hot || s >= n_slots)) {
      latch(err, kDevBadSlot);
      continue;
    }
    ring[(tail + i) % n_cold] = s;
  }
}

// One block per token: copy its K and V rows (row_bytes each, a multiple of 16) with 16-byte
// vector accesses.
__global__ void cold_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                   const int32_t* __restrict__ slots, int32_t N,
                                   uint4* __restrict__ kpool, uint4* __restrict__ vpool,
                                   int64_t row_vec, int64_t n_hot, int64_t n_slots, int32_t* err) {
  for (int32_t t = blockIdx.x; t < N; t += gridDim.x) {
    const int32_t s = slots[t];
    if (s < n_hot || s >= n_slots) {
      if (threadIdx.x == 0) latch(err, kDevBadSlot);
      continue;
    }
    const uint4* ks = k_new + (int64_t)t * row_vec;
    const uint4* vs = v_new + (int64_t)t * row_vec;
    uint4* kd = kpool + (int64_t)s * row_vec;
    uint4* vd = vpool + (int64_t)s * row_vec;
    for (int64_t i = threadIdx.x; i < row_vec; i += blockDim.x) {
      kd[i] = ks[i];
      vd[i] = vs[i];
    }
  }
}

}  // namespace

cudaError_t launch_cold_alloc(const int32_t* excl, int32_t B, const int32_t* ring, int64_t n_cold,
                              int64_t head, int32_t* req_to_slot, int32_t* suffix_len, int32_t cap,
                              int32_t* slots_out, int64_t* ring_pos, int32_t* err, cudaStream_t s) {
  const int grid = B < 4096 ? B : 4096;
  cold_alloc_kernel<<<grid, 128, 0, s>>>(excl, B, ring, n_cold, head, req_to_slot, suffix_len, cap, slots_out,
                                         ring_pos, err);
  return cudaGetLastError();
}

cudaError_t launch_cold_alloc_uniform(int32_t n, int32_t B, const int32_t* ring, int64_t n_cold, int32_t* req_to_slot,
                                      int32_t* suffix_len, int32_t cap, int32_t* slots_out, int64_t* ring_pos,
                                      int32_t* err, cudaStream_t s) {
  cold_alloc_uniform_kernel<<<1, 256, 0, s>>>(n, B, ring, n_cold, req_to_slot, suffix_len, cap, slots_out, ring_pos,
                                              err);
  return cudaGetLastError();
}

cudaError_t launch_cold_free(const int32_t* slots, int32_t n, int32_t* ring, int64_t n_cold,
                             int64_t tail, int64_t n_hot, int64_t n_slots, int32_t checks,
                             int64_t* ring_pos, int32_t* err, cudaStream_t s) {
  int grid = (n + 255) / 256;
  if (grid > 4096) grid = 4096;
  cold_free_kernel<<<grid, 256, 0, s>>>(slots, n, ring, n_cold, tail, n_hot, n_slots, checks, ring_pos, err);
  return cudaGetLastError();
}

cudaError_t launch_cold_append(int32_t dtype, const void* k_new, const void* v_new,
                               const int32_t* slots, int32_t N, void* kpool, void* vpool,
                               int64_t row_elems, int64_t n_hot, int64_t n_slots, int32_t checks,
                               int32_t* err, cudaStream_t s) {
  (void)checks;  // slot ids are always range-checked here: a bad id would write outside the pool
  const int64_t row_bytes = row_elems * (dtype == 1 ? 2 : 4);
  if (row_bytes % 16) return cudaErrorInvalidValue;
  if (((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)kpool | (uintptr_t)vpool) % 16)
    return cudaErrorInvalidValue;
  const int64_t row_vec = row_bytes / 16;
  const int grid = N < 8192 ? N : 8192;
  const int block = row_vec >= 128 ? 128 : (row_vec >= 64 ? 64 : 32);
  cold_append_kernel<<<grid, block, 0, s>>>((const uint4*)k_new, (const uint4*)v_new, slots, N,
                                            (uint4*)kpool, (uint4*)vpool, row_vec, n_hot, n_slots,
                                            err);
  return cudaGetLastError();
}

}  // namespace granikv
