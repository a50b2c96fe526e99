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

// One warp merges row (b, h) of a head_dim-128 bf16 output; lane owns elements 4*lane..4*lane+3.
__device__ __forceinline__ void warp_merge_row_bf16_d128(const AttnParams& p, int32_t b, int32_t h, int lane) {
  constexpr float kLog2e = 1.4426950408889634f;
  const DevReq r = p.reqs[b];
  const float* lse_rec = p.rec_lse + (int64_t)r.rec_base * p.n_q + h;
  float M = -INFINITY;
  for (int32_t i = lane; i < r.n_parts; i += 32) M = fmaxf(M, __ldcg(lse_rec + (int64_t)i * p.n_q));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const int64_t row = (int64_t)b * p.n_q + h;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.o) + row * 128 + lane * 4;
  if (M == -INFINITY) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
    if (lane == 0) p.lse[row] = -INFINITY;
    return;
  }
  float tot = 0.f;
  for (int32_t i = lane; i < r.n_parts; i += 32) tot += exp2f((__ldcg(lse_rec + (int64_t)i * p.n_q) - M) * kLog2e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float lse = M + logf(tot);
  const float4* orec = reinterpret_cast<const float4*>(p.rec_o + ((int64_t)r.rec_base * p.n_q + h) * 128) + lane;
  const int64_t stride = (int64_t)p.n_q * 128 / 4;  // float4s between consecutive records of this row
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int32_t i = 0;
  for (; i + 4 <= r.n_parts; i += 4) {
    float w[4];
    float4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      w[u] = exp2f((__ldcg(lse_rec + (int64_t)(i + u) * p.n_q) - lse) * kLog2e);
      x[u] = __ldcg(orec + (i + u) * stride);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc.x += w[u] * x[u].x;
      acc.y += w[u] * x[u].y;
      acc.z += w[u] * x[u].z;
      acc.w += w[u] * x[u].w;
    }
  }
  for (; i < r.n_parts; ++i) {
    const float w = exp2f((__ldcg(lse_rec + (int64_t)i * p.n_q) - lse) * kLog2e);
    const float4 x = __ldcg(orec + i * stride);
    acc.x += w * x.x;
    acc.y += w * x.y;
    acc.z += w * x.z;
    acc.w += w * x.w;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  if (lane == 0) p.lse[row] = lse;
}

// Ticket increment for row (b, h); returns whether this arrival completed the row.  Every
// thread that stored part of the record must have executed __threadfence() before this call
// (and the warp synchronised), so the record is visible before the ticket moves.
__device__ __forceinline__ bool arrive_row(const AttnParams& p, int32_t b, int32_t h) {
  const int32_t n = p.reqs[b].n_parts;
  const int32_t prev = atomicAdd(p.tickets + (int64_t)b * p.n_q + h, 1);
  return prev == n - 1;
}

// Every lane with `mine` set arrived last for (b_l, h_l); the warp merges those rows one by one
// and resets their tickets.
__device__ __forceinline__ void warp_merge_completed(const AttnParams& p, bool mine, int32_t b_l, int32_t h_l,
                                                     int lane) {
  unsigned todo = __ballot_sync(0xffffffffu, mine);
  if (!todo) return;
  __threadfence();  // the other producers' records are visible before they are read
  while (todo) {
    const int src = __ffs(todo) - 1;
    todo &= todo - 1;
    const int32_t b = __shfl_sync(0xffffffffu, b_l, src);
    const int32_t h = __shfl_sync(0xffffffffu, h_l, src);
    warp_merge_row_bf16_d128(p, b, h, lane);
    if (lane == 0) atomicExch(p.tickets + (int64_t)b * p.n_q + h, 0);
  }
}

}  // namespace granikv
