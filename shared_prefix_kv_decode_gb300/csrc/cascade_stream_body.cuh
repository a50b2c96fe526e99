// cascade_stream_body.cuh -- cascade prefix backend as a bandwidth kernel: the contiguous HOT
// slab streamed once per step, all KV heads of a token together, warp-level bf16 tensor cores.
//
// GraniKV (arXiv:2608.15584), "2 Related Work": cascade inference reads the shared prefix once
// per step, cutting its HBM reads from O(B) to O(1); "3 GraniKV", dual attention backends:
// cascade serves the memory-bound steps (few rows per KV head), dense the compute-bound ones;
// the HOT slab makes the prefix one contiguous run of slots.
//
// Work item: (prefix group, KV-head group of up to 8 heads, column chunk, L_p piece).  A slot's
// K (or V) row for the eight heads of a group is 2 KB of contiguous memory, so each CTA streams
// whole 2 KB rows of consecutive slots -- every DRAM page it opens is read in full, unlike a
// per-head kernel that takes 256 B of every 2 KB row.  One consumer warp per KV head j; the
// chunk's query columns (request r, head-in-group i) -> query head j*g + i, at most 16 of them,
// are the MMA's N dimension and the tile's 16 tokens its M dimension:
//     S^T[16 tok x N] = K_j[16 tok x 128] . Q_j^T[128 x N]            (8 k-steps x N/8 mma.m16n8k16)
//     O^T[128 x N]   += V_j^T[128 x 16 tok] . P^T[16 tok x N]         (8 m-tiles x N/8 mma.m16n8k16)
// with an online softmax per column (running max and sum, lane shuffles over the 16 tokens).
// P^T goes from the accumulator layout to the B-operand layout with movmatrix.
//
// Loads: a producer warp streams 16-token tiles (K and V, 32 KB each for eight heads) through a
// 3-stage shared-memory ring with cp.async.bulk, one copy per 2 KB token row (lanes 0-15 K,
// 16-31 V), completing on the stage's mbarrier; rows are stored 2064 bytes apart so the eight
// rows an ldmatrix reads fall in eight bank groups.  Rows past the piece's end are copied from
// a zero row, so masked tokens hold finite values.  Every wait is bounded in time; on expiry
// the CTA raises its abort flag, latches an error, and the producer waits (bounded) for its
// copies in flight before the CTA exits.
//
// Output: per (request, query head) row, the piece's normalised partial state (o, lse) goes to
// the request's record for that piece; the merge combines a row's records by log-sum-exp.
#pragma once

#include "internal.h"
#include "launch_util.cuh"
#include "merge_util.cuh"
#include "mma_util.cuh"
#include "tc_util.cuh"

namespace granikv {
namespace csc {
namespace {

constexpr int kD = 128;
constexpr int kSub = kCascadeStreamTile;           // tokens per MMA sub-tile (MMA M)
constexpr int kStages = 3;
constexpr int kWarps = 8;                          // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;        // + the producer warp
constexpr int kWarpCols = kCascadeStreamCols;      // query columns per consumer warp
constexpr int kRowBytes = kD * 2;                  // one head's K (or V) row: 256 B
// Stage layout for WPH consumer warps per KV head (8 / WPH heads per CTA): K then V, each
// 16 * WPH token rows of the heads' bytes plus 16 bytes of padding.
template <int WPH>
struct Geo {
  static constexpr int kHeads = kWarps / WPH;
  static constexpr int kTok = kSub * WPH;                       // tokens per stage
  static constexpr int kRowStride = kHeads * kRowBytes + 16;    // 2064 / 1040 / 528 / 272 B
  static constexpr int kTileBytes = kTok * kRowStride;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOffBar = kStages * kStageBytes;
};
constexpr int max2(int a, int b) { return a > b ? a : b; }
constexpr int kOffBarMax = max2(max2(Geo<1>::kOffBar, Geo<2>::kOffBar), max2(Geo<4>::kOffBar, Geo<8>::kOffBar));
constexpr int kSmemBytes = kOffBarMax + 8 * 2 * kStages + 16;  // full and empty barriers, abort flag, done barrier
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(Geo<1>::kRowStride % 16 == 0 && Geo<8>::kRowStride % 16 == 0 && Geo<1>::kStageBytes % 16 == 0 &&
                  Geo<2>::kStageBytes % 16 == 0 && Geo<4>::kStageBytes % 16 == 0 && Geo<8>::kStageBytes % 16 == 0,
              "bulk copies need 16-byte alignment");
static_assert(kSub == 16 && kWarpCols == 16, "the MMA tiling below assumes 16 tokens and two 8-column n-tiles");
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Source of the rows of masked tokens (zero-initialised at module load, never written).
__device__ __align__(128) uint4 g_zero_row[kWarps * kRowBytes / 16];

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(mbar)
      : "memory");
}

// The consumer loop of one warp: KV head j (its rows at byte `head_off` of every token row),
// query columns [c0, c0 + ncols) of the chunk (ncols <= 8 * NT), over the piece's n_stages
// stages of Geo<WPH>::kTok tokens.  Sub-tiles are taken in pairs (WPH >= 2), each pair with one
// running-max update, and every S^T product runs as two independent accumulation chains over
// the two halves of head_dim, so a warp keeps several MMAs in flight.  At the end the warp
// waits (bounded) until every consumer warp is done with the ring, stages its normalised
// O^T in the ring's shared memory, and writes each column's record as one 512-byte row.
// Returns false if a wait gave up.
template <int WPH, int NT>
__device__ __forceinline__ bool consume(const AttnParams& p, const DevGroup& gr, const DevPrefixItem& it, int j,
                                        uint32_t head_off, int warp, int lane, int r0, int c0, int ncols,
                                        int n_valid, int n_stages, unsigned char* smem, volatile int* abort_flag) {
  using G = Geo<WPH>;
  constexpr int kPair = WPH >= 2 ? 2 : 1;           // sub-tiles per softmax update
  const int g = p.g;
  const uint32_t sbase = smem_u32(smem);
  auto full_bar = [&](int st) { return sbase + G::kOffBar + 8 * st; };
  auto empty_bar = [&](int st) { return sbase + G::kOffBar + 8 * (kStages + st); };
  const uint32_t done_bar = sbase + G::kOffBar + 16 * kStages + 8;
  // Q^T as B fragments: column n = c0 + t*8 + lane/4 of the chunk is (request r0 + n/g, query
  // head j*g + n%g)
  uint32_t qf[NT][8][2];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int n = t * 8 + (lane >> 2);
    if (n < ncols) {
      const int cn = c0 + n;
      const int32_t b = p.group_req[gr.req_begin + r0 + cn / g];
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          static_cast<const __nv_bfloat16*>(p.q) + ((int64_t)b * p.n_q + j * g + cn % g) * kD);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qf[t][kk][0] = qrow[kk * 8 + (lane & 3)];
        qf[t][kk][1] = qrow[kk * 8 + 4 + (lane & 3)];
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) qf[t][kk][0] = qf[t][kk][1] = 0u;
    }
  }
  const float scale = p.scale_log2;
  // this thread's columns: t*8 + 2*(lane%4) and the next; rows (tokens) lane/4 and lane/4 + 8
  float m[NT][2], l[NT][2];
  float o[NT][8][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    m[t][0] = m[t][1] = -INFINITY;
    l[t][0] = l[t][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[t][mt][0] = o[t][mt][1] = o[t][mt][2] = o[t][mt][3] = 0.f;
  }
  const int mi = lane >> 3;
  const int t0r = lane >> 2, t1r = t0r + 8;
  bool ok = true;
  for (int stage = 0; stage < n_stages && ok; ++stage) {
    const int st = stage % kStages;
    const bool landed =
        mbar_wait_bounded(full_bar(st), (stage / kStages) & 1, abort_flag, p.err, kDevTimeout, kWaitLimitNs);
    if (!__all_sync(0xffffffffu, landed)) {
      ok = false;
      break;
    }
#pragma unroll 1
    for (int u = 0; u < WPH; u += kPair) {
      const int rem0 = n_valid - stage * G::kTok - u * kSub;  // valid tokens from this pair's first row
      if (rem0 <= 0) break;
      const uint32_t kst = sbase + st * G::kStageBytes + u * kSub * G::kRowStride + head_off;
      const uint32_t vst = kst + G::kTileBytes;

      // S^T = K . Q^T for the pair's sub-tiles, head_dim in two halves (independent chains)
      float s[kPair][NT][4];
      {
        float sb[kPair][NT][4];
#pragma unroll
        for (int v = 0; v < kPair; ++v)
#pragma unroll
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[v][t][e] = sb[v][t][e] = 0.f;
        const int r = (lane & 7) + (mi & 1) * 8;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
          for (int v = 0; v < kPair; ++v) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            const uint32_t row = kst + (v * kSub + r) * G::kRowStride + (mi >> 1) * 16;
            ldsm_x4(row + kk * 32, a0, a1, a2, a3);
            ldsm_x4(row + (kk + 4) * 32, b0, b1, b2, b3);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              mma_bf16_16816(s[v][t], a0, a1, a2, a3, qf[t][kk][0], qf[t][kk][1]);
              mma_bf16_16816(sb[v][t], b0, b1, b2, b3, qf[t][kk + 4][0], qf[t][kk + 4][1]);
            }
          }
        }
#pragma unroll
        for (int v = 0; v < kPair; ++v)
#pragma unroll
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[v][t][e] += sb[v][t][e];
      }
      uint32_t pb[kPair][NT][2];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int v = 0; v < kPair; ++v) {
          const int rem = rem0 - v * kSub;
          s[v][t][0] = t0r < rem ? s[v][t][0] * scale : -INFINITY;
          s[v][t][1] = t0r < rem ? s[v][t][1] * scale : -INFINITY;
          s[v][t][2] = t1r < rem ? s[v][t][2] * scale : -INFINITY;
          s[v][t][3] = t1r < rem ? s[v][t][3] * scale : -INFINITY;
          mx0 = fmaxf(mx0, fmaxf(s[v][t][0], s[v][t][2]));
          mx1 = fmaxf(mx1, fmaxf(s[v][t][1], s[v][t][3]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[t][0], mx0), mn1 = fmaxf(m[t][1], mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
        const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = ex2_approx(m[t][0] - mu0), al1 = ex2_approx(m[t][1] - mu1);
        m[t][0] = mn0;
        m[t][1] = mn1;
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int v = 0; v < kPair; ++v) {
          const float p0 = ex2_approx(s[v][t][0] - mu0), p1 = ex2_approx(s[v][t][1] - mu1);
          const float p2 = ex2_approx(s[v][t][2] - mu0), p3 = ex2_approx(s[v][t][3] - mu1);
          ls0 += p0 + p2;
          ls1 += p1 + p3;
          pb[v][t][0] = movmatrix_t(pack_bf16(p0, p1));
          pb[v][t][1] = movmatrix_t(pack_bf16(p2, p3));
        }
        l[t][0] = l[t][0] * al0 + ls0;
        l[t][1] = l[t][1] * al1 + ls1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[t][mt][0] *= al0;
          o[t][mt][2] *= al0;
          o[t][mt][1] *= al1;
          o[t][mt][3] *= al1;
        }
      }
      // O^T += V^T . P^T over the pair's sub-tiles
      {
        const int r = (lane & 7) + (mi >> 1) * 8;
#pragma unroll
        for (int v = 0; v < kPair; ++v) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vst + (v * kSub + r) * G::kRowStride + (mt * 2 + (mi & 1)) * 16, a0, a1, a2, a3);
#pragma unroll
            for (int t = 0; t < NT; ++t) mma_bf16_16816(o[t][mt], a0, a1, a2, a3, pb[v][t][0], pb[v][t][1]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(st));
  }
  // every consumer warp is done with the ring before it holds the epilogue's staging rows
  if (lane == 0) mbar_arrive(done_bar);
  if (!ok) return false;
  const bool all_done = mbar_wait_bounded(done_bar, 0, abort_flag, p.err, kDevTimeout, kWaitLimitNs);
  if (!__all_sync(0xffffffffu, all_done)) return false;

  // full column sums over the 16 tokens' lanes, normalise, stage O^T as [column][d] fp32 rows
  // (stride 132 floats: the four columns a store instruction covers fall in different banks)
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l[t][0] += __shfl_xor_sync(0xffffffffu, l[t][0], off);
      l[t][1] += __shfl_xor_sync(0xffffffffu, l[t][1], off);
    }
  }
  constexpr int kStageStride = kD + 4;
  float* so = reinterpret_cast<float*>(smem) + warp * (kWarpCols * kStageStride);
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float lsum = l[t][c];
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      float* dst = so + (t * 8 + 2 * (lane & 3) + c) * kStageStride + (lane >> 2);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        dst[mt * 16] = o[t][mt][c] * inv;
        dst[mt * 16 + 8] = o[t][mt][2 + c] * inv;
      }
    }
  }
  // lane n < ncols finds column n's record row (all in parallel), then each column's record is
  // written as one 512-byte row
  int64_t row_l = -1;
  int32_t b_l = -1;
  if (lane < ncols) {
    const int cn = c0 + lane;
    b_l = p.group_req[gr.req_begin + r0 + cn / g];
    const int32_t rec = p.reqs[b_l].rec_base + it.split;
    if (rec >= 0 && rec < p.n_records) row_l = (int64_t)rec * p.n_q + j * g + cn % g;
    else latch_err(p.err, kDevBadRecord);
  }
  __syncwarp();
  const uint64_t keep = l2_policy_keep();
  for (int n = 0; n < ncols; ++n) {
    const int64_t row = __shfl_sync(0xffffffffu, row_l, n);
    if (row < 0) continue;
    const float4 v4 = *reinterpret_cast<const float4*>(so + n * kStageStride + lane * 4);
    st_record4(p.rec_o + row * kD + lane * 4, v4, keep);
  }
  // lse of each column, from the lanes that hold its sum (lanes 0-3: columns t*8 + 2*lane + c)
  int32_t bcol[NT][2], hcol[NT][2];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int n = t * 8 + 2 * (lane & 3) + c;  // < 16 always
      const int64_t row = __shfl_sync(0xffffffffu, row_l, n);
      const int32_t b = __shfl_sync(0xffffffffu, b_l, n);
      const bool have = n < ncols && row >= 0;
      bcol[t][c] = have ? b : -1;
      hcol[t][c] = j * g + (c0 + n) % g;
      const float lsum = l[t][c];
      if (have && lane < 4) st_record(p.rec_lse + row, lsum > 0.f ? (m[t][c] + log2f(lsum)) * kLn2 : -INFINITY, keep);
    }
  }
  if (p.fused_merge) {
    __threadfence();
    __syncwarp();
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const bool mine = lane < 4 && bcol[t][c] >= 0 && arrive_row(p, bcol[t][c], hcol[t][c]);
        warp_merge_completed(p, mine, bcol[t][c], hcol[t][c], lane);
      }
  }
  return true;
}

// One work item with WPH consumer warps per KV head (see cascade_stream_body).
template <int WPH>
__device__ __forceinline__ void cascade_stream_run(const AttnParams& p, const DevPrefixItem& it, const DevGroup& gr,
                                                   unsigned char* smem) {
  using G = Geo<WPH>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int j0 = it.kv_head * G::kHeads;              // first KV head of this CTA's head group
  const int nh = min(G::kHeads, p.n_kv - j0);         // heads present in the group
  const uint32_t gbytes = (uint32_t)nh * kRowBytes;   // bytes copied per token row
  int32_t t0, t1;
  piece_range(gr, it.split, t0, t1);
  const int n_valid = t1 - t0;
  const int n_stages = (n_valid + G::kTok - 1) / G::kTok;
  const int g = p.g;
  const int R = gr.rows_per_cta / g;                  // requests per column chunk
  const int r0 = it.row_block * R;
  const int ncols = min(R, gr.n_req - r0) * g;        // columns of this chunk
  const int parts = min(WPH, (ncols + kWarpCols - 1) / kWarpCols);  // warps per head with columns
  const uint32_t sbase = smem_u32(smem);
  auto full_bar = [&](int st) { return sbase + G::kOffBar + 8 * st; };
  auto empty_bar = [&](int st) { return sbase + G::kOffBar + 8 * (kStages + st); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::kOffBar + 16 * kStages);
  const uint32_t done_bar = sbase + G::kOffBar + 16 * kStages + 8;
  const bool bad_slab = gr.slab_off < 0 || gr.slab_off + gr.L_p > p.n_hot;
  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), (uint32_t)(max(nh, 1) * max(parts, 1)));
    }
    mbar_init(done_bar, (uint32_t)(max(nh, 1) * max(parts, 1)));
    *abort_flag = 0;
    mbar_fence_init();
    if (bad_slab) latch_err(p.err, kDevBadSlab);
  }
  __syncthreads();
  // q and the pools are read only after the previous kernel in the stream completed
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (bad_slab || n_stages <= 0 || ncols <= 0 || nh <= 0 || warp > kWarps) return;

  if (warp == kWarps) {
    // ---------------- producer: one bulk copy per token row of K and of V -----------------
    const int64_t tok_bytes = (int64_t)p.n_kv * kRowBytes;
    const char* kbase = static_cast<const char*>(p.kpool) + (gr.slab_off + t0) * tok_bytes + (int64_t)j0 * kRowBytes;
    const char* vbase = static_cast<const char*>(p.vpool) + (gr.slab_off + t0) * tok_bytes + (int64_t)j0 * kRowBytes;
    int n = 0;
    for (; n < n_stages; ++n) {
      const int st = n % kStages;
      const bool free_ok = n < kStages || mbar_wait_bounded(empty_bar(st), ((n / kStages) - 1) & 1, abort_flag,
                                                            p.err, kDevTimeout, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, free_ok)) break;
      if (lane == 0) mbar_arrive_expect_tx(full_bar(st), 2u * G::kTok * gbytes);
      __syncwarp();
#pragma unroll
      for (int k = 0; k < (2 * G::kTok) / 32; ++k) {
        const int c = lane + 32 * k;          // copies [0, kTok) are K rows, the rest V rows
        const bool is_v = c >= G::kTok;
        const int r = is_v ? c - G::kTok : c;
        const int tok = n * G::kTok + r;
        const char* base = is_v ? vbase : kbase;
        const void* src = tok < n_valid ? static_cast<const void*>(base + (int64_t)tok * tok_bytes)
                                        : static_cast<const void*>(g_zero_row);
        const uint32_t dst = sbase + st * G::kStageBytes + (is_v ? G::kTileBytes : 0) + r * G::kRowStride;
        bulk_load(dst, src, gbytes, full_bar(st));
      }
    }
    // never leave with a copy in flight: wait for the last issued stages to land
    if (lane == 0) {
      for (int i = max(0, n - kStages); i < n; ++i) {
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
  const int hw = warp / WPH, part = warp % WPH;       // this warp's head in the group and column part
  if (hw >= nh || part >= parts) return;              // no CTA-wide barrier is used below
  const int c0 = part * kWarpCols;
  const int my_cols = min(kWarpCols, ncols - c0);
  const uint32_t head_off = (uint32_t)hw * kRowBytes;
  if (my_cols > 8)
    consume<WPH, 2>(p, gr, it, j0 + hw, head_off, warp, lane, r0, c0, my_cols, n_valid, n_stages, smem, abort_flag);
  else
    consume<WPH, 1>(p, gr, it, j0 + hw, head_off, warp, lane, r0, c0, my_cols, n_valid, n_stages, smem, abort_flag);
}

// Prefix work item `item` (an index into p.pitems) on `smem` (at least kSmemBytes, 128-byte
// aligned), run by kThreads or more threads (the extra warps only take part in the set-up
// barrier).  The group's `sub` field is the number of consumer warps per KV head (1, 2, 4 or 8):
// a CTA covers 8 / sub KV heads and 16 * sub query columns of each, streaming 16 * sub tokens
// of those heads per stage.
__device__ __forceinline__ void cascade_stream_body(const AttnParams& p, int32_t item, unsigned char* smem) {
  const DevPrefixItem it = p.pitems[item];
  const DevGroup gr = p.groups[it.group];
  switch (gr.sub) {
    case 2: cascade_stream_run<2>(p, it, gr, smem); break;
    case 4: cascade_stream_run<4>(p, it, gr, smem); break;
    case 8: cascade_stream_run<8>(p, it, gr, smem); break;
    default: cascade_stream_run<1>(p, it, gr, smem); break;
  }
}

}  // namespace
}  // namespace csc
}  // namespace granikv
