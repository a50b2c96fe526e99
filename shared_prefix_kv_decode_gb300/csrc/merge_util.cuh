// merge_util.cuh -- the log-sum-exp merge of a request's partial attention states, done by the
// producer that finishes last.
//
// GraniKV (arXiv:2608.15584), "2 Related Work", prefix-suffix attention: prefix and suffix
// partial attentions are merged with log-sum-exp.  Every (request b, query head h) row has
// n_parts partial states (one per prefix piece and per suffix segment).  Each producer writes
// its record, fences, and increments the row's ticket; the producer whose increment completes
// the count merges the row:
//     lse = M + ln sum_i e^(lse_i - M),   o = sum_i e^(lse_i - lse) o_i,
// and resets the ticket to zero for the next call.  No thread waits for another, so nothing
// here can hang.  Records written by other CTAs are read through L2 (ld.global.cg).
#pragma once

#include <cuda_bf16.h>

#include "internal.h"

namespace granikv {

// Merge up to four rows at once: lanes 8k..8k+7 take row k (valid when `have`), each lane
// owns 16 consecutive elements of head_dim 128.  One pass over the records with a running
// log-sum-exp (m, den) per row; the loads of four records are in flight together.
__device__ __forceinline__ void warp_merge_rows4_bf16_d128(const AttnParams& p, bool have, int32_t b, int32_t h,
                                                          int lane) {
  constexpr float kLog2e = 1.4426950408889634f;
  const int sub = lane & 7;  // which 16-element slice of the row
  int32_t n = 0;
  const float* lse_rec = nullptr;
  const float4* orec = nullptr;
  if (have) {
    const DevReq r = p.reqs[b];
    n = r.n_parts;
    lse_rec = p.rec_lse + (int64_t)r.rec_base * p.n_q + h;
    orec = reinterpret_cast<const float4*>(p.rec_o + ((int64_t)r.rec_base * p.n_q + h) * 128) + sub * 4;
  }
  const int64_t lstride = p.n_q;                      // floats between a row's records (lse)
  const int64_t ostride = (int64_t)p.n_q * 128 / 4;   // float4s between a row's records (o)
  float m = -INFINITY, den = 0.f;
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int32_t i = 0; i < n; i += 4) {
    float l[4];
    float4 x[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = i + u < n;
      l[u] = ok ? __ldcg(lse_rec + (i + u) * lstride) : -INFINITY;
#pragma unroll
      for (int k = 0; k < 4; ++k) x[u][k] = ok ? __ldcg(orec + (i + u) * ostride + k) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (l[u] == -INFINITY) continue;
      const float mn = fmaxf(m, l[u]);
      const float a = exp2f((m - mn) * kLog2e);   // 0 when m is still -inf
      const float w = exp2f((l[u] - mn) * kLog2e);
      den = den * a + w;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k].x = acc[k].x * a + w * x[u][k].x;
        acc[k].y = acc[k].y * a + w * x[u][k].y;
        acc[k].z = acc[k].z * a + w * x[u][k].z;
        acc[k].w = acc[k].w * a + w * x[u][k].w;
      }
      m = mn;
    }
  }
  if (!have) return;
  const int64_t row = (int64_t)b * p.n_q + h;
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.o) + row * 128 + sub * 16;
  uint32_t packed[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
    packed[2 * k] = *reinterpret_cast<uint32_t*>(&lo);
    packed[2 * k + 1] = *reinterpret_cast<uint32_t*>(&hi);
  }
  *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  *reinterpret_cast<uint4*>(dst + 8) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  if (sub == 0) p.lse[row] = den > 0.f ? m + logf(den) : -INFINITY;
}

// Ticket increment for row (b, h); returns whether this arrival completed the row.  Every
// thread that stored part of the record must have executed __threadfence() before this call
// (and the warp synchronised), so the record is visible before the ticket moves.
__device__ __forceinline__ bool arrive_row(const AttnParams& p, int32_t b, int32_t h) {
  const int32_t n = p.reqs[b].n_parts;
  const int32_t prev = atomicAdd(p.tickets + (int64_t)b * p.n_q + h, 1);
  return prev == n - 1;
}

// Every lane with `mine` set arrived last for (b_l, h_l); the warp merges those rows four at
// a time and resets their tickets.
__device__ __forceinline__ void warp_merge_completed(const AttnParams& p, bool mine, int32_t b_l, int32_t h_l,
                                                     int lane) {
  unsigned todo = __ballot_sync(0xffffffffu, mine);
  if (!todo) return;
  __threadfence();  // the other producers' records are visible before they are read
  while (todo) {
    // take up to four pending rows; lanes 8k..8k+7 work on the k-th
    const int k = lane >> 3;
    int my_src = -1;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int src = todo ? __ffs(todo) - 1 : -1;
      if (todo) todo &= todo - 1;
      if (q == k) my_src = src;
    }
    const int32_t b = __shfl_sync(0xffffffffu, b_l, my_src < 0 ? 0 : my_src);
    const int32_t h = __shfl_sync(0xffffffffu, h_l, my_src < 0 ? 0 : my_src);
    warp_merge_rows4_bf16_d128(p, my_src >= 0, b, h, lane);
    if (my_src >= 0 && (lane & 7) == 0) atomicExch(p.tickets + (int64_t)b * p.n_q + h, 0);
  }
}

}  // namespace granikv
