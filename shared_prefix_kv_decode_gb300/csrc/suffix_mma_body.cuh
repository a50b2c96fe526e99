// suffix_mma_body.cuh -- COLD suffix partial attention: bulk-copy gather, warp-level bf16
// tensor cores.
//
// GraniKV (arXiv:2608.15584), "1 Introduction" / "3 GraniKV": suffix and decoded tokens sit in
// a token-level COLD pool (page size 1), so every token is gathered through the request's
// token table; "2 Related Work", prefix-suffix attention: the suffix is attended separately
// and merged with the prefix by log-sum-exp.
//
// Shape: head_dim 128, bf16, g = n_q/n_kv <= 8.  One consumer warp owns one KV head of one
// request segment.  Because only g query heads share a KV head, tokens are the MMA's M
// dimension and the g heads its N dimension (8 columns):
//     S^T[16 tok x 8 heads] = K[16 tok x 128] . Q^T[128 x 8]          (8 mma.m16n8k16)
//     O^T[128 x 8 heads]   += V^T[128 x 16 tok] . P^T[16 tok x 8 heads] (8 mma.m16n8k16)
// P^T goes from the accumulator layout to the B-operand layout with movmatrix.  The online
// softmax (running max and sum per head column) reduces across lanes with warp shuffles.
//
// Work split: the plan cuts the concatenation of all requests' COLD tokens into one contiguous
// run per token-CTA (stream-K style, cut on 16-token tile boundaries of each request), so that
// every CTA's tiles plus one tile per request segment come to the same count; each request
// segment inside a run writes one partial-state record.  In one grid whose dense CTAs finish
// early, the dense CTAs run the last runs after their prefix pieces.  A second index picks a group of
// up to eight KV heads, whose K (and V) rows of one slot are contiguous in the pool (2 KB for
// eight heads).
//
// Gather: a producer warp streams 16-token tiles through a 3-stage shared-memory ring with
// asynchronous bulk copies (cp.async.bulk, one per token row of K and of V, completing on the
// stage's mbarrier), so the copies bypass L1 and the ring holds two tiles (128 KB) in flight
// per SM.  Token rows are stored 2064 bytes apart (2048 + 16), which puts the eight rows an
// ldmatrix reads into eight different bank groups.  Rows past a segment's end are copied from
// a zero row in global memory, so masked tokens hold finite values.  Every mbarrier wait is
// bounded in time; on expiry the CTA raises an abort flag and latches an error, and the
// producer waits (again bounded) for its copies in flight before the CTA exits.
#pragma once

#include "internal.h"
#include "launch_util.cuh"
#include "merge_util.cuh"
#include "mma_util.cuh"
#include "tc_util.cuh"

namespace granikv {
namespace sfx {
namespace {


constexpr int kD = 128;
constexpr int kTile = 16;                          // tokens per tile (MMA M)
constexpr int kStages = 3;
constexpr int kWarps = 8;                          // consumer warps: KV heads per CTA
constexpr int kThreads = (kWarps + 1) * 32;        // + the producer warp
constexpr int kRowBytes = kD * 2;                  // one head's K (or V) row: 256 B
constexpr int kGroupBytes = kWarps * kRowBytes;    // one slot's row of a head group: 2 KB
constexpr int kRowStride = kGroupBytes + 16;       // shared-memory stride of token rows
constexpr int kTileBytes = kTile * kRowStride;     // 33,024 B
constexpr int kStageBytes = 2 * kTileBytes;        // K + V
constexpr int kOffSlots = kStages * kStageBytes;
constexpr int kSlotBytes = kSuffixMaxCtaTokens * 4;  // the CTA's slot ids, loaded once
constexpr int kSegSmem = 256;                      // segment descriptors staged in shared memory
constexpr int kOffSegs = kOffSlots + kSlotBytes;
constexpr int kOffNew = kOffSegs + kSegSmem * (int)sizeof(DevSuffixItem);  // newest token per segment
constexpr int kOffBar = kOffNew + kSegSmem * 4;
constexpr int kSmemBytes = kOffBar + 8 * 2 * kStages + 16;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kRowStride % 16 == 0 && kStageBytes % 16 == 0, "bulk copies need 16-byte alignment");
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Source of the rows of masked tokens (one copy per translation unit; zero-initialised at
// module load, never written).
__device__ __align__(128) uint4 g_zero_row[kGroupBytes / 16];

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(mbar)
      : "memory");
}

// One token-CTA `cta` of the suffix work list, for KV-head group `group`, on `smem` (at least
// kSmemBytes, 128-byte aligned), run by kThreads or more threads (the extra warps only take
// part in the set-up barrier).
__device__ __forceinline__ void suffix_mma_body(const AttnParams& p, const int32_t* __restrict__ cta_begin, int cta,
                                                int group, unsigned char* smem) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int seg_begin = cta_begin[cta];
  const int seg_end = cta_begin[cta + 1];
  if (seg_begin >= seg_end) return;
  const int j0 = group * kWarps;                      // first KV head of this CTA's group
  const int nh = min(kWarps, p.n_kv - j0);            // heads in the group
  const uint32_t gbytes = (uint32_t)nh * kRowBytes;   // bytes per slot row of the group
  const uint32_t sbase = smem_u32(smem);
  auto full_bar = [&](int st) { return sbase + kOffBar + 8 * st; };
  auto empty_bar = [&](int st) { return sbase + kOffBar + 8 * (kStages + st); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 16 * kStages);

  // The slot ids of all of this CTA's tokens (its segments back to back) and its segment
  // descriptors go to shared memory once, so neither the copy issue nor a segment change waits
  // on a global load.  The plan keeps a CTA's tokens within kSuffixMaxCtaTokens; a CTA with more
  // than kSegSmem segments reads the descriptors beyond that from global memory.
  int32_t* sslot = reinterpret_cast<int32_t*>(smem + kOffSlots);
  DevSuffixItem* sseg = reinterpret_cast<DevSuffixItem*>(smem + kOffSegs);
  const int n_seg = seg_end - seg_begin;
  for (int k = threadIdx.x; k < min(n_seg, kSegSmem); k += blockDim.x) sseg[k] = p.sitems[seg_begin + k];
  // the token tables, lengths, pools and q are read only after the previous kernel in the
  // stream completed
  grid_dep_wait();
  grid_dep_launch_dependents();
  // a plan made for more tokens than exist yet: each segment ends at its request's live length
  auto clamp = [&](DevSuffixItem sgi) {
    if (p.live_len) sgi.t1 = max(sgi.t0, min(sgi.t1, p.live_len[sgi.b]));
    return sgi;
  };
  if (p.live_len) {
    __syncthreads();  // the staged descriptors are complete
    for (int k = threadIdx.x; k < min(n_seg, kSegSmem); k += blockDim.x) sseg[k] = clamp(sseg[k]);
    __syncthreads();
  }
  auto seg_at = [&](int k) { return k < kSegSmem ? sseg[k] : clamp(p.sitems[seg_begin + k]); };
  // fused COLD append: each request's newest token (the last of its list) is read from
  // k_new/v_new row b instead of the pool, and the consumer warps write it to its slot; the
  // index of that token per segment is staged next to the descriptors
  const bool fuse_new = p.k_new != nullptr;
  int32_t* snew = reinterpret_cast<int32_t*>(smem + kOffNew);
  auto newest_of = [&](int32_t b) { return (p.live_len ? p.live_len[b] : p.reqs[b].seq_len) - 1; };
  if (fuse_new)
    for (int k = threadIdx.x; k < min(n_seg, kSegSmem); k += blockDim.x) snew[k] = newest_of(p.sitems[seg_begin + k].b);
  auto new_at = [&](int k) { return !fuse_new ? -1 : k < kSegSmem ? snew[k] : newest_of(p.sitems[seg_begin + k].b); };
  const int64_t tok_bytes = (int64_t)p.n_kv * kRowBytes;
  int n_tok = 0;
  for (int sg = seg_begin; sg < seg_end; ++sg) {
    // from global memory: the staged copies are not complete before the barrier below
    const DevSuffixItem seg = clamp(p.sitems[sg]);
    const int len = seg.t1 - seg.t0;
    const int32_t* row = p.req_to_slot + (int64_t)seg.b * p.cap + seg.t0;
    for (int k = threadIdx.x; k < len && n_tok + k < kSuffixMaxCtaTokens; k += blockDim.x) sslot[n_tok + k] = row[k];
    n_tok += len;
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), (uint32_t)nh);
    }
    *abort_flag = 0;
    mbar_fence_init();
    if (n_tok > kSuffixMaxCtaTokens) latch_err(p.err, kDevBadRecord);
  }
  __syncthreads();
  if (n_tok > kSuffixMaxCtaTokens) return;

  if (warp == kWarps) {
    // ---------------- producer: one bulk copy per token row (lanes 0-15 K, 16-31 V) -------
    const bool is_v = lane >= kTile;
    const char* src_base = static_cast<const char*>(is_v ? p.vpool : p.kpool) + (int64_t)j0 * kRowBytes;
    const int r = lane & (kTile - 1);
    int n = 0;      // tiles issued
    int pos = 0;    // position of the current segment's first token in sslot
    bool stop = false;
    // test hook: token-CTA 0 of group 0 withholds its first tile
    const bool skip0 = p.inject_stall != 0 && cta == 0 && group == 0;
    const char* new_base =
        fuse_new ? static_cast<const char*>(is_v ? p.v_new : p.k_new) + (int64_t)j0 * kRowBytes : nullptr;
    for (int sg = 0; sg < n_seg && !stop; ++sg) {
      const DevSuffixItem seg = seg_at(sg);
      const int newest = new_at(sg);
      for (int t = seg.t0; t < seg.t1; t += kTile, ++n) {
        const int st = n % kStages;
        // every lane polls; the warp goes on only if all of them saw the phase complete
        const bool free_ok = n < kStages || mbar_wait_bounded(empty_bar(st), ((n / kStages) - 1) & 1, abort_flag,
                                                              p.err, kDevTimeout, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, free_ok)) {
          stop = true;
          break;
        }
        const void* src = g_zero_row;
        if (t + r < seg.t1) {
          const int32_t slot = sslot[pos + (t - seg.t0) + r];
          if (t + r == newest)
            src = new_base + (int64_t)seg.b * tok_bytes;
          else if (slot >= p.n_hot && slot < p.n_slots)
            src = src_base + (int64_t)slot * tok_bytes;
          else
            latch_err(p.err, kDevBadSlot);
        }
        if (skip0 && n == 0) continue;
        if (lane == 0) mbar_arrive_expect_tx(full_bar(st), 2u * kTile * gbytes);
        __syncwarp();
        const uint32_t dst = sbase + st * kStageBytes + (is_v ? kTileBytes : 0) + r * kRowStride;
        bulk_load(dst, src, gbytes, full_bar(st));
      }
      pos += seg.t1 - seg.t0;
    }
    // never leave with a copy in flight: wait for the last issued tiles to land
    if (lane == 0) {
      for (int i = max(skip0 ? 1 : 0, n - kStages); i < n; ++i) {
        const uint64_t t_start = globaltimer_ns();
        while (!mbar_try_wait(full_bar(i % kStages), (i / kStages) & 1)) {
          if (globaltimer_ns() - t_start > kWaitLimitNs) {
            atomicCAS(p.err, 0, kDevTimeout);
            break;
          }
        }
      }
    }
    return;
  }
  if (warp >= nh) return;  // no CTA-wide barrier is used below

  // ---------------- consumers: warp `warp` owns KV head j ----------------
  const int j = j0 + warp;
  const float scale = p.scale_log2;
  const int g = p.g;
  const int h0 = 2 * (lane & 3);  // this thread's two head columns: h0, h0 + 1
  // Q^T as B fragments (column n = lane/4 is head j*g + n); the next segment's are loaded one
  // segment ahead so their latency hides behind the current segment's tiles
  uint32_t qn[8][2];
  auto load_q = [&](int sg) {
    const int nn = lane >> 2;
    if (sg < n_seg && nn < g) {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          static_cast<const __nv_bfloat16*>(p.q) + ((int64_t)seg_at(sg).b * p.n_q + j * g + nn) * kD);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qn[kk][0] = qrow[kk * 8 + (lane & 3)];
        qn[kk][1] = qrow[kk * 8 + 4 + (lane & 3)];
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) qn[kk][0] = qn[kk][1] = 0u;
    }
  };
  load_q(0);
  const uint32_t head_off = (uint32_t)warp * kRowBytes;
  int tile = 0;  // tiles consumed so far
  int cpos = 0;  // position of the next segment's first token in sslot
  for (int sg = 0; sg < n_seg; ++sg) {
    const DevSuffixItem seg = seg_at(sg);
    const int seg_pos = cpos;
    cpos += seg.t1 - seg.t0;
    const int newest = new_at(sg);
    uint32_t qf[8][2];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qf[kk][0] = qn[kk][0];
      qf[kk][1] = qn[kk][1];
    }
    load_q(sg + 1);
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    bool ok = true;
    for (int t = seg.t0; t < seg.t1; t += kTile, ++tile) {
      const int st = tile % kStages;
      const bool landed = mbar_wait_bounded(full_bar(st), (tile / kStages) & 1, abort_flag, p.err, kDevTimeout,
                                            kWaitLimitNs);
      if (!__all_sync(0xffffffffu, landed)) {
        ok = false;
        break;
      }
      const uint32_t kst = sbase + st * kStageBytes + head_off;
      const uint32_t vst = kst + kTileBytes;

      // S^T = K . Q^T
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int mi = lane >> 3;
        const int r = (lane & 7) + (mi & 1) * 8;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kst + r * kRowStride + (kk * 2 + (mi >> 1)) * 16, a0, a1, a2, a3);
          mma_bf16_16816(s, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        }
      }
      const int rem = seg.t1 - t;  // valid tokens in this tile (may exceed 16)
      const int r0 = lane >> 2, r1 = r0 + 8;
      s[0] = r0 < rem ? s[0] * scale : -INFINITY;
      s[1] = r0 < rem ? s[1] * scale : -INFINITY;
      s[2] = r1 < rem ? s[2] * scale : -INFINITY;
      s[3] = r1 < rem ? s[3] * scale : -INFINITY;
      float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
      const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
      const float p0 = exp2f(s[0] - mu0), p1 = exp2f(s[1] - mu1);
      const float p2 = exp2f(s[2] - mu0), p3 = exp2f(s[3] - mu1);
      l0 = l0 * al0 + p0 + p2;
      l1 = l1 * al1 + p1 + p3;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= al0;
        o[mt][2] *= al0;
        o[mt][1] *= al1;
        o[mt][3] *= al1;
      }
      // P^T in B-operand layout
      const uint32_t b0 = movmatrix_t(pack_bf16(p0, p1));
      const uint32_t b1 = movmatrix_t(pack_bf16(p2, p3));
      // O^T += V^T . P^T
      {
        const int mi = lane >> 3;
        const int r = (lane & 7) + (mi >> 1) * 8;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(vst + r * kRowStride + (mt * 2 + (mi & 1)) * 16, a0, a1, a2, a3);
          mma_bf16_16816(o[mt], a0, a1, a2, a3, b0, b1);
        }
      }
      // fused append: the step's new token of this request is in this tile (it came from
      // k_new/v_new); head j's K row (lanes 0-15) and V row (16-31) go from the tile to its slot.
      // No CTA of this launch reads that slot.
      if (newest >= t && newest < t + kTile && newest < seg.t1) {
        const int32_t slot = sslot[seg_pos + (newest - seg.t0)];
        if (slot >= p.n_hot && slot < p.n_slots) {
          const uint32_t row = (lane < 16 ? kst : vst) + (uint32_t)(newest - t) * kRowStride + (lane & 15) * 16;
          const uint4 v = *reinterpret_cast<const uint4*>(smem + (row - sbase));
          char* pool = static_cast<char*>(lane < 16 ? p.kpool : p.vpool);
          *reinterpret_cast<uint4*>(pool + (int64_t)slot * tok_bytes + (int64_t)j * kRowBytes + (lane & 15) * 16) = v;
        }
      }
      // this warp is done reading the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(st));
    }
    if (!ok) break;

    // finish the segment: full column sums, normalise, write the record
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const int32_t rec = seg.rec;
    if (rec < 0 || rec >= p.n_records) {
      if (lane == 0) latch_err(p.err, kDevBadRecord);
      continue;
    }
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
    const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const int hq0 = j * g + h0;
    float* dst0 = p.rec_o + ((int64_t)rec * p.n_q + hq0) * kD + (lane >> 2);
    float* dst1 = dst0 + kD;
    const bool w0 = h0 < g, w1 = h0 + 1 < g;
    const uint64_t keep = l2_policy_keep();
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      if (w0) {
        st_record(dst0 + mt * 16, o[mt][0] * inv0, keep);
        st_record(dst0 + mt * 16 + 8, o[mt][2] * inv0, keep);
      }
      if (w1) {
        st_record(dst1 + mt * 16, o[mt][1] * inv1, keep);
        st_record(dst1 + mt * 16 + 8, o[mt][3] * inv1, keep);
      }
    }
    if (lane < 4) {
      float* ldst = p.rec_lse + (int64_t)rec * p.n_q + hq0;
      if (w0) st_record(ldst, l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY, keep);
      if (w1) st_record(ldst + 1, l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY, keep);
    }
    if (p.fused_merge) {
      __threadfence();
      __syncwarp();
      bool last0 = false, last1 = false;
      if (lane < 4) {
        if (w0) last0 = arrive_row(p, seg.b, hq0);
        if (w1) last1 = arrive_row(p, seg.b, hq0 + 1);
      }
      warp_merge_completed(p, last0, seg.b, hq0, lane);
      warp_merge_completed(p, last1, seg.b, hq0 + 1, lane);
    }
  }
}


}  // namespace
}  // namespace sfx
}  // namespace granikv
