// dense_tc_body.cuh -- dense prefix backend on the 5th-generation tensor cores (tcgen05/TMEM).
//
// GraniKV (arXiv:2608.15584), "2 Related Work": HydraGen-style attention batches all queries
// that share a prefix into one matrix-matrix product against the prefix K/V; "3 GraniKV":
// the dense backend targets compute-bound steps, and is possible only because the HOT slab
// stores the prefix contiguously (the card page: paged prefixes force a gather instead).
//
// One CTA takes one (prefix group, KV head j, 128-row block, L_p piece).  Rows are the group's
// (request, head-in-group) pairs of KV head j, so M = 128 query rows share every K/V tile.
// Per 128-token tile i:
//     S(i) = Q K(i)^T   (M=128, N=128, K=128: 8 tcgen05.mma from shared memory, fp32 in TMEM)
//     P(i) = 2^(S(i)*scale*log2e - m)   (softmax warps; bf16, written back over S(i) in TMEM;
//            scale and shift two columns per packed f32x2 operation, exponentials on MUFU)
//     O   += P(i) V(i)  (M=128, N=128, K=128: 8 tcgen05.mma with A = P(i) read from TMEM)
// Every MMA is 128x128x16, so one issuing thread keeps the tensor core fed.
// The same CTA runs the causal prefill of a slab (a group flagged causal): its "requests" are the
// slab's own tokens, row r is token r/g, the CTA reads keys only up to its block's last token,
// and each row masks the keys after its own token in the tiles at the diagonal.
// Roles:
//  * warps 0-7, softmax and epilogue: warp w serves TMEM lanes 32*(w%4).. (row r = lane r), all
//    128 columns of the tiles i with i % 2 == w / 4.  The two warps of a row quarter sit on the
//    same SM sub-partition and take turns, half a tile apart, so one issues exponentials while
//    the other waits on its TMEM loads.  The running max is a chain over the tiles: the warp of
//    tile i reads the max used for tile i-1 from shared memory (published by the other warp at
//    a time-bounded mbarrier as soon as it was decided), keeps it unless the tile's row max
//    exceeds it by more than 2^8, publishes its own, and writes P(i) over S(i)'s columns.
//  * warps 8 and 9, TMA loads (two 64-dim halves per tile, 128-byte swizzle), each in a warp of
//    its own: warp 8 fills a 3-slot K ring whose slots free up as soon as S(i) completes, warp 9
//    a 2-slot V ring freed by PV(i); warp 9 also zeroes the rows of a ragged last V tile past
//    the piece's end before PV may use it.
//  * warp 10, the MMAs, issued as their inputs become ready: S(j) up to three tiles ahead of
//    the PV products (three S/P buffers in TMEM), PV(i) once the softmax has written P(i).
// The K producer initialises the barriers and issues the first K and V tiles before the Q
// gather, so their HBM latency overlaps it.
// The running max is only moved (and O rescaled in TMEM) when it grows by more than 2^8; the
// final normalisation uses the same max, so the result is the exact softmax.  Every mbarrier
// wait is bounded in time; on expiry the CTA raises an abort flag, latches an error, drains what
// it issued and frees its TMEM.
#pragma once

#include <cuda.h>

#include "internal.h"
#include "launch_util.cuh"
#include "merge_util.cuh"
#include "mma_util.cuh"
#include "tc_util.cuh"

namespace granikv {
namespace dns {
namespace {


constexpr int kD = 128;
constexpr int kM = kDenseRows;                // 128 query rows per CTA
constexpr int kN = kDenseTile;                // 128 tokens per tile
static_assert(kN == 128, "the TMEM layout and the MMA shapes below assume 128-token tiles");
constexpr int kHalfCols = kN / 2;             // S columns per softmax thread
constexpr int kKSlots = 3;                    // slots of the K ring
constexpr int kVSlots = 2;                    // slots of the V ring
constexpr int kSBufs = 3;                     // S/P buffers in TMEM
// Only in-order waiters use the V barriers (the MMA for PV(i), the V producer for the tiles it
// issued), so two V slots suffice; the ragged last V tile is cleared by the V producer itself.
constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kWarpTmaK = 8, kWarpTmaV = 9, kWarpMma = 10;
constexpr int kThreads = 352;
constexpr int kHalf = kN * 128;               // one 64-dim half of a K or V tile: 16 KB
constexpr int kTile = 2 * kHalf;              // 32 KB
constexpr int kQBytes = kM * kD * 2;          // 32 KB (two 64-dim K-blocks)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;           // K slot s at kOffK + s*kTile
constexpr int kOffV = kOffK + kKSlots * kTile;   // V slot s at kOffV + s*kTile
constexpr int kOffRed = kOffV + kVSlots * kTile; // [2][2 tile parities][128 rows]: row sums, maxima
constexpr int kOffMPub = kOffRed + 2 * 2 * kM * 4;  // [4 quarters][2 tile parities][32 rows] maxima
constexpr int kOffBar = kOffMPub + 4 * 2 * 32 * 4;
constexpr int kBarArea = 512;
constexpr int kSmemBytes = kOffBar + kBarArea + 1024;  // barriers + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kKSlots * kTile >= kM * kD * 4, "the epilogue stages the fp32 record rows in the K ring");
static_assert(kVSlots * kTile >= kM * 8, "the epilogue keeps the rows' record offsets in the V ring");
constexpr uint32_t kTmemCols = 512;           // S/P buffers at 0, 128, 256; O at 384
constexpr uint32_t kColO = 384;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;     // log2 of the largest growth tolerated in P
constexpr uint64_t kWaitLimitNs = 2000000000ull;

enum : int {
  kBarKFull = 0,                            // [kKSlots] TMA -> MMA (K)
  kBarKEmpty = kBarKFull + kKSlots,         // [kKSlots] MMA (S done) -> TMA
  kBarVFull = kBarKEmpty + kKSlots,         // [kVSlots] TMA -> MMA and last-tile softmax (V)
  kBarVEmpty = kBarVFull + kVSlots,         // [kVSlots] MMA (PV done) -> TMA
  kBarSFull = kBarVEmpty + kVSlots,         // [kSBufs] S(i) in TMEM -> softmax
  kBarPFull = kBarSFull + kSBufs,           // [kSBufs] P(i) in TMEM -> MMA (128 arrivals)
  kBarPvDone = kBarPFull + kSBufs,          // [kSBufs] PV(i) done -> softmax
  kBarDrain = kBarPvDone + kSBufs,          // all MMAs done -> teardown
  kBarPair = kBarDrain + 1,                 // [4] the two softmax warps of a row quarter, epilogue (64)
  kBarQFull = kBarPair + 4,                 // Q tile loaded by TMA -> MMA
  kBarVZero = kBarQFull + 1,                // ragged last V tile cleared past its end -> MMA
  kBarMPub = kBarVZero + 1,                 // [4 quarters][2 parities] max of a tile published (32)
  kNumBars = kBarMPub + 8
};
static_assert(8 * kNumBars + 16 <= kBarArea, "barrier area");


// Prefix work item `item` (one CTA) on `smem_raw` (at least kSmemBytes), run by kThreads
// threads.  tmk/tmv: the layer's K and V tensor maps, kernel parameters (__grid_constant__).
__device__ __forceinline__ void dense_tc_body(const AttnParams& p, int32_t item, const CUtensorMap* tmk,
                                              const CUtensorMap* tmv, const CUtensorMap* tmq, unsigned char* smem_raw) {
  // 1024-byte alignment for the 128-byte-swizzle atoms
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base = (raw_u + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw_u);
  const uint32_t sQ = base + kOffQ, sK = base + kOffK, sV = base + kOffV;
  float* red = reinterpret_cast<float*>(smem + kOffRed);  // red[(kind*2 + parity)*kM + row]
  const uint32_t sBar = base + kOffBar;
  auto bar = [&](int i) { return sBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars + 8);

  const DevPrefixItem it = p.pitems[item];
  const DevGroup gr = p.groups[it.group];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = p.g;
  const int j = it.kv_head;
  const int32_t rows = gr.n_req * g;
  int32_t t0, t1;
  piece_range(gr, it.split, t0, t1);
  // causal prefill: row r is token r/g of the slab and sees keys [0, r/g], so the block's last
  // token ends the keys this CTA reads.  Every row sees key 0 in the first tile; a later tile
  // in which all of a row's keys lie past its token only adds zero weights.
  const bool causal = gr.causal != 0;
  if (causal) t1 = min(t1, (it.row_block * kM + kM - 1) / g + 1);
  const int n_tiles = t1 > t0 ? (t1 - t0 + kN - 1) / kN : 0;
  const int valid_last = n_tiles > 0 ? (t1 - t0) - (n_tiles - 1) * kN : kN;  // tokens of the last tile
  const bool ragged = valid_last < kN;
  const bool slab_ok = gr.slab_off >= 0 && gr.slab_off + gr.L_p <= p.n_hot && n_tiles > 0;
  // Q by TMA when the group's requests are consecutive in the batch: the row block is then a
  // (64 dims, g heads, 128/g requests) box of q [B, n_q, 128]; otherwise the threads gather it
  const bool q_tma = p.q_tma != 0 && gr.q_b0 >= 0;
  const int32_t rbase = it.row_block * kM;

  // The K producer thread initialises the barriers and issues the first K and V tiles at once,
  // so their HBM latency overlaps the Q gather below; its loop later starts after them.
  const int k_pre = min(n_tiles, kKSlots), v_pre = min(n_tiles, kVSlots);
  auto issue_tile = [&](bool is_k, int i) {
    const CUtensorMap* tm = is_k ? tmk : tmv;
    const int slots = is_k ? kKSlots : kVSlots;
    const int full = (is_k ? kBarKFull : kBarVFull) + i % slots;
    const uint32_t dst = (is_k ? sK : sV) + (i % slots) * kTile;
    const int32_t z = (int32_t)(gr.slab_off + t0 + i * kN);
    mbar_arrive_expect_tx(bar(full), kTile);
    tma_load_3d(dst, tm, 0, j, z, bar(full));
    tma_load_3d(dst + kHalf, tm, 64, j, z, bar(full));
  };
  // Read-ahead into L2 (p.l2_ahead > 0): when a ring slot is refilled with tile i, tile
  // i + l2_ahead of the same tensor is requested into L2, so this CTA keeps more of its bytes
  // in flight than its shared-memory ring holds.  Next to suffix CTAs that keep HBM busy, this
  // raises the prefix side's share of the bandwidth; the first tiles are not read ahead, which
  // would hold back the tiles the pipeline waits for first.
  const int l2_ahead = p.l2_ahead;
  auto read_ahead = [&](bool is_k, int i) {
    if (l2_ahead <= 0 || i >= n_tiles) return;
    const CUtensorMap* tm = is_k ? tmk : tmv;
    const int32_t z = (int32_t)(gr.slab_off + t0 + i * kN);
    tma_prefetch_l2_3d(tm, 0, j, z);
    tma_prefetch_l2_3d(tm, 64, j, z);
  };
  if (warp == kWarpTmaK && lane == 0) {
    tma_prefetch_desc(tmk);
    tma_prefetch_desc(tmv);
    if (q_tma) tma_prefetch_desc(tmq);
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1u;
      if (i >= kBarPFull && i < kBarPFull + kSBufs) count = kSoftmaxThreads / 2;
      if (i >= kBarPair && i < kBarPair + 4) count = 64u;
      if (i >= kBarMPub && i < kBarMPub + 8) count = 32u;
      mbar_init(bar(i), count);
    }
    *abort_flag = slab_ok ? 0 : 1;
    if (!slab_ok) atomicCAS(p.err, 0, (int32_t)kDevBadSlab);
    mbar_fence_init();
    fence_proxy_async_smem();
    grid_dep_wait();  // the slab may have been written by the work before this kernel
    if (slab_ok) {
      if (q_tma) {
        const int32_t z = gr.q_b0 + rbase / g;
        mbar_arrive_expect_tx(bar(kBarQFull), kQBytes);
        tma_load_3d(sQ, tmq, 0, j * g, z, bar(kBarQFull));
        tma_load_3d(sQ + kM * 128, tmq, 64, j * g, z, bar(kBarQFull));
      }
      for (int i = 0; i < k_pre; ++i) issue_tile(true, i);
      for (int i = 0; i < v_pre; ++i) issue_tile(false, i);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // q and the records are touched only after the previous kernel in the stream has completed
  grid_dep_wait();
  grid_dep_launch_dependents();
  // Q rows of this block -> shared memory, K-major with 128-byte swizzle: row r, 16-byte
  // chunk c lives in 64-dim block c/8 at r*128 + ((c%8) ^ (r%8))*16 (the layout the TMA box
  // load produces); rows past the group are 0.  A thread's chunks are gathered in three passes
  // (all request lookups, then all q loads, then the stores), so its loads are in flight together
  if (!q_tma) {
    constexpr int kQIters = (kM * 16 + kThreads - 1) / kThreads;
    int32_t qoff[kQIters];
#pragma unroll
    for (int k = 0; k < kQIters; ++k) {
      const int idx = tid + k * kThreads;
      const int32_t row = rbase + (idx >> 4);
      qoff[k] = -1;
      if (idx < kM * 16 && row < rows) qoff[k] = p.group_req[gr.req_begin + row / g];
    }
    uint4 qv[kQIters];
#pragma unroll
    for (int k = 0; k < kQIters; ++k) {
      const int idx = tid + k * kThreads;
      const int32_t row = rbase + (idx >> 4);
      qv[k] = make_uint4(0u, 0u, 0u, 0u);
      if (qoff[k] >= 0)
        qv[k] = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                               ((int64_t)qoff[k] * p.n_q + j * g + row % g) * kD)[idx & 15];
    }
#pragma unroll
    for (int k = 0; k < kQIters; ++k) {
      const int idx = tid + k * kThreads;
      if (idx < kM * 16) {
        const int r = idx >> 4;
        const int c = idx & 15;
        const uint32_t dst = sQ + (c >> 3) * (kM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(qv[k].x), "r"(qv[k].y), "r"(qv[k].z),
                     "r"(qv[k].w)
                     : "memory");
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTmaK || warp == kWarpTmaV) {
    // ---------------- TMA producers: warp 8 the K ring, warp 9 the V ring ----------------
    const bool is_k = warp == kWarpTmaK;
    const int full = is_k ? kBarKFull : kBarVFull;
    const int empty = is_k ? kBarKEmpty : kBarVEmpty;
    const int slots = is_k ? kKSlots : kVSlots;
    // the first `slots` tiles were issued before the block-wide barrier (when the slab is valid)
    int issued = slab_ok ? (is_k ? k_pre : v_pre) : 0;
    if (lane == 0) {
      for (int i = issued; i < n_tiles && !*abort_flag; ++i) {
        const int st = i % slots;
        if (!mbar_wait_bounded(bar(empty + st), ((i / slots) - 1) & 1, abort_flag, p.err, kDevTimeout,
                               kWaitLimitNs))
          break;
        issue_tile(is_k, i);
        read_ahead(is_k, i + l2_ahead);
        issued = i + 1;
      }
    }
    issued = __shfl_sync(0xffffffffu, issued, 0);
    if (!is_k && ragged && issued == n_tiles) {
      // the last V tile runs past the piece: once it has landed (this warp issued it after its
      // slot's previous tile was consumed, so the parity wait is unambiguous), zero its rows
      // from `valid_last` on, so that 0 * garbage cannot reach O, then let the MMA use it
      const int last = n_tiles - 1;
      bool landed = mbar_wait_bounded(bar(kBarVFull + last % kVSlots), (last / kVSlots) & 1, abort_flag, p.err,
                                      kDevTimeout, kWaitLimitNs);
      landed = __all_sync(0xffffffffu, landed);
      if (landed) {
        const uint32_t vt = sV + (last % kVSlots) * kTile;
        for (int idx = lane; idx < (kN - valid_last) * 16; idx += 32) {
          const int r = valid_last + idx / 16;
          const uint32_t a = vt + ((idx >> 3) & 1) * kHalf + r * 128 + (idx & 7) * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(a), "r"(0u) : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarVZero));
      }
    }
    if (lane == 0) {
      // never leave with a copy in flight: wait for every issued tile (and Q) to land
      if (is_k && q_tma && slab_ok) {
        const uint64_t t_start = globaltimer_ns();
        while (!mbar_try_wait(bar(kBarQFull), 0)) {
          if (globaltimer_ns() - t_start > kWaitLimitNs) {
            atomicCAS(p.err, 0, kDevTimeout);
            break;
          }
        }
      }
      for (int i = max(0, issued - slots); i < issued; ++i) {
        const int st = i % slots;
        const uint64_t t_start = globaltimer_ns();
        while (!mbar_try_wait(bar(full + st), (i / slots) & 1)) {
          if (globaltimer_ns() - t_start > kWaitLimitNs) {
            atomicCAS(p.err, 0, kDevTimeout);
            break;
          }
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && !*abort_flag) {
      constexpr uint32_t idS = idesc_bf16_f32(kM, kN, false);
      constexpr uint32_t idO = idesc_bf16_f32(kM, kD, true);
      // descriptors are built once; a byte offset into shared memory moves the start-address
      // field (bits 0..13, in 16-byte units), which never carries out for addresses < 256 KB
      const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sK, 16, 1024);
      // V tile as an MN-major B operand: 16 tokens per step (2048 bytes), the two 64-dim halves
      // kHalf apart (leading offset), 8-token groups 1024 bytes apart (stride)
      const uint64_t dv0 = smem_desc_sw128(sV, kHalf, 1024);
      int committed = 0;
      // Event-driven issue (non-blocking barrier tests): PV(i) as soon as P(i) and V(i) are
      // ready, S(j) as soon as K(j) has landed and its TMEM buffer is free.  S(j) overwrites S(j-3)/P(j-3), so it may go in once
      // PV(j-3), the last reader of P(j-3), has been issued (tcgen05 MMAs of one thread execute
      // in order; the softmax finished with S(j-3) before it produced P(j-3)).  Polling both
      // conditions keeps the issuing thread from sitting on one while the other is ready.
      int next_s = 0, next_pv = 0;
      if (q_tma && !mbar_wait_bounded(bar(kBarQFull), 0, abort_flag, p.err, kDevTimeout, kWaitLimitNs))
        next_pv = n_tiles;  // gave up (abort raised): issue nothing
      tc_fence_after();
      uint64_t t_last = globaltimer_ns();
      while (next_pv < n_tiles) {
        bool progressed = false;
        if (next_pv < next_s) {
          const int i = next_pv;
          const int st = i % kVSlots;
          const int sb = i % kSBufs;
          if (mbar_test_wait(bar(kBarPFull + sb), (i / kSBufs) & 1) &&
              mbar_test_wait(bar(kBarVFull + st), (i / kVSlots) & 1) &&
              (!ragged || i != n_tiles - 1 || mbar_test_wait(bar(kBarVZero), 0))) {
            tc_fence_after();
            const uint32_t pa = tmem + (uint32_t)(sb * kN);  // P(i): 64 columns, two tokens per column
            const uint64_t dv = dv0 + (uint64_t)((st * kTile) >> 4);
#pragma unroll
            for (int ks = 0; ks < kN / 16; ++ks)
              umma_f16_ts(tmem + kColO, pa + (uint32_t)(ks * 8), dv + (uint64_t)((ks * 2048) >> 4), idO,
                          (i > 0 || ks > 0) ? 1u : 0u);
            umma_commit(bar(kBarVEmpty + st));
            umma_commit(bar(kBarPvDone + sb));
            committed += 2;
            ++next_pv;
            progressed = true;
          }
        }
        if (next_s < n_tiles && next_s < next_pv + kSBufs) {
          const int i = next_s;
          const int st = i % kKSlots;
          if (mbar_test_wait(bar(kBarKFull + st), (i / kKSlots) & 1)) {
            tc_fence_after();
            const uint32_t dS = tmem + (uint32_t)((i % kSBufs) * kN);
            const uint64_t dk = dk0 + (uint64_t)((st * kTile) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t a = dq0 + (uint64_t)(((kk >> 2) * (kM * 128) + (kk & 3) * 32) >> 4);
              const uint64_t b = dk + (uint64_t)(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4);
              umma_f16(dS, a, b, idS, kk > 0 ? 1u : 0u);
            }
            umma_commit(bar(kBarSFull + i % kSBufs));
            umma_commit(bar(kBarKEmpty + st));
            committed += 2;
            ++next_s;
            progressed = true;
          }
        }
        if (progressed) {
          t_last = globaltimer_ns();
        } else if (*abort_flag) {
          break;
        } else if (globaltimer_ns() - t_last > kWaitLimitNs) {
          *abort_flag = 1;
          atomicCAS(p.err, 0, (int32_t)kDevTimeout);
          break;
        }
      }
      // drain: every tcgen05 op this thread issued completes before the CTA frees TMEM
      if (committed > 0) {
        umma_commit(bar(kBarDrain));
        const uint64_t t_start = globaltimer_ns();
        while (!mbar_try_wait(bar(kBarDrain), 0)) {
          if (globaltimer_ns() - t_start > kWaitLimitNs) {
            atomicCAS(p.err, 0, kDevTimeout);
            break;
          }
        }
      }
    }
  } else {
    // ---------------- softmax warps 0-7: rows of quarter `quad`, tiles of parity `par` ----------------
    const int quad = warp & 3;
    const int par = warp >> 2;
    const int half = par;                           // the epilogue's column half of O
    const int r = quad * 32 + lane;                 // row = TMEM lane
    const uint32_t lane_off = (uint32_t)((quad * 32) << 16);
    const int pair_bar = kBarPair + quad;           // mbarrier of the two warps sharing rows
    float* mpub = reinterpret_cast<float*>(smem + kOffMPub) + quad * 64;  // [tile parity][lane]
    const float scale = p.scale_log2;
    // this row's request, head and record, looked up now so the loads finish during the tiles
    const int32_t row = rbase + r;
    int32_t b = -1, h = 0, rec = -1;
    if (row < rows) {
      b = p.group_req[gr.req_begin + row / g];
      h = j * g + row % g;
      rec = p.reqs[b].rec_base + it.split;
    }
    // keys this row may see end at row_end (slab coordinates): its own token + 1 when causal
    const int32_t row_end = (causal && row < rows) ? min(t1, row / g + 1) : t1;
    float m_own = -INFINITY;   // max (scaled, base-2 units) used for this warp's latest tile
    float l = 0.f;             // this warp's share of the row sum, relative to m_own
    int pair_phase = 0;
    bool ok = !*abort_flag;
    for (int i = par; ok && i < n_tiles; i += 2) {
      const int sb = i % kSBufs;
      ok = mbar_wait_bounded(bar(kBarSFull + sb), (i / kSBufs) & 1, abort_flag, p.err, kDevTimeout, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);  // the TMEM loads below are warp-collective
      if (!ok) break;
      tc_fence_after();
      const int valid = min(kN, t1 - t0 - i * kN);               // tokens of the tile in range
      const int valid_row = min(valid, row_end - t0 - i * kN);    // of those, keys this row sees
      const uint32_t ts = tmem + lane_off + (uint32_t)(sb * kN);
      // row max over the 128 columns (scale > 0 commutes with max); S(i) is read again below
      // for the exponentials, which keeps the thread's registers within the launch's budget
      float mx;
      {
        static_assert(kN == 128, "the max tree below covers 128 columns");
        uint32_t u[4][32];
        GRANIKV_TMEM_LD32(ts, u[0]);
        GRANIKV_TMEM_LD32(ts + 32, u[1]);
        GRANIKV_TMEM_LD32(ts + 64, u[2]);
        GRANIKV_TMEM_LD32(ts + 96, u[3]);
        tmem_wait_ld();
        if (valid_row < kN) {
#pragma unroll
          for (int k = 0; k < kN; ++k) u[k >> 5][k & 31] = k < valid_row ? u[k >> 5][k & 31] : 0xff800000u;
        }
        float sv[kN];
#pragma unroll
        for (int k = 0; k < kN; ++k) sv[k] = __uint_as_float(u[k >> 5][k & 31]);
        float t[43], w[15];
#pragma unroll
        for (int k = 0; k < 42; ++k) t[k] = max3f(sv[3 * k], sv[3 * k + 1], sv[3 * k + 2]);
        t[42] = fmaxf(sv[126], sv[127]);
#pragma unroll
        for (int k = 0; k < 14; ++k) w[k] = max3f(t[3 * k], t[3 * k + 1], t[3 * k + 2]);
        w[14] = t[42];
        const float v0 = max3f(w[0], w[1], w[2]), v1 = max3f(w[3], w[4], w[5]), v2 = max3f(w[6], w[7], w[8]);
        const float v3 = max3f(w[9], w[10], w[11]), v4 = max3f(w[12], w[13], w[14]);
        mx = fmaxf(max3f(v0, v1, v2), fmaxf(v3, v4)) * scale;
      }
      // the max used for tile i: that of tile i-1 (decided by the other warp of the quarter),
      // moved only when this tile's row max exceeds it by more than 2^kRescaleThreshold
      float m_i = mx;
      bool warp_need = false;
      float m_prev = -INFINITY;
      if (i > 0) {
        const int pp = (i - 1) & 1;
        ok = mbar_wait_bounded(bar(kBarMPub + quad * 2 + pp), ((i - 1) >> 1) & 1, abort_flag, p.err, kDevTimeout,
                               kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        m_prev = mpub[pp * 32 + lane];
        warp_need = __any_sync(0xffffffffu, mx > m_prev + kRescaleThreshold);
        m_i = warp_need ? fmaxf(m_prev, mx) : m_prev;
      }
      // publish at once, so the warp of tile i+1 is not held up by the rescale below (the slot's
      // previous value, tile i-2's, was read by that warp before it published tile i-1's)
      mpub[par * 32 + lane] = m_i;
      mbar_arrive(bar(kBarMPub + quad * 2 + par));
      if (warp_need) {
        // O must hold PV(i-1) before it is rescaled, and PV(i) waits for P(i), written below
        ok = mbar_wait_bounded(bar(kBarPvDone + (i - 1) % kSBufs), ((i - 1) / kSBufs) & 1, abort_flag, p.err,
                               kDevTimeout, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float alpha = ex2_approx(m_prev - m_i);
        uint32_t u[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t ta = tmem + lane_off + kColO + c * 32;
          GRANIKV_TMEM_LD32(ta, u);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) u[k] = __float_as_uint(__uint_as_float(u[k]) * alpha);
          GRANIKV_TMEM_ST32(ta, u);
        }
        tmem_wait_st();
      }
      if (m_own != m_i && m_own != -INFINITY) l *= ex2_approx(m_own - m_i);
      m_own = m_i;
      // P = 2^(s*scale - m) for the 128 columns, packed two per 32-bit column and written over
      // columns [0, 64) of the S(i) buffer: S columns [64*hb, 64*hb + 64) are in registers
      // before their P goes to columns [32*hb, 32*hb + 32).  Every exponential goes to MUFU:
      // moving a share of them to a polynomial on the FMA pipe made the tile slower on this GPU
      // (the extra instructions cost more than MUFU time saved)
      const uint64_t scale2 = f2_pack(scale, scale), nm2 = f2_pack(-m_i, -m_i);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};  // packed partial row sums (0.0f bit patterns)
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t u[2][32];
        GRANIKV_TMEM_LD32(ts + hb * 64, u[0]);
        GRANIKV_TMEM_LD32(ts + hb * 64 + 32, u[1]);
        tmem_wait_ld();
        if (valid_row < kN) {  // masked keys: -inf, so their weight is 0
#pragma unroll
          for (int k = 0; k < 64; ++k) u[k >> 5][k & 31] = 64 * hb + k < valid_row ? u[k >> 5][k & 31] : 0xff800000u;
        }
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float sa = __uint_as_float(u[k >> 4][(2 * k) & 31]);
          const float sb2 = __uint_as_float(u[k >> 4][(2 * k + 1) & 31]);
          const uint64_t x = f2_fma(f2_pack(sa, sb2), scale2, nm2);
          float xa, xb;
          f2_unpack(x, xa, xb);
          const uint64_t e = f2_pack(ex2_approx(xa), ex2_approx(xb));
          acc[k & 3] = f2_add(acc[k & 3], e);
          float a, b2;
          f2_unpack(e, a, b2);
          pk[k] = pack_bf16(a, b2);
        }
        GRANIKV_TMEM_ST32(tmem + lane_off + (uint32_t)(sb * kN + hb * 32), pk);
      }
      {
        const uint64_t t2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
        float la, lb;
        f2_unpack(t2, la, lb);
        l += la + lb;
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + sb));
    }
    // epilogue: wait for the last PV, combine the two warps' row sums (each relative to the max
    // of its own latest tile; the last tile's max is the final one), normalise, write the record
    if (ok) {
      const int last = n_tiles - 1;
      ok = mbar_wait_bounded(bar(kBarPvDone + last % kSBufs), (last / kSBufs) & 1, abort_flag, p.err, kDevTimeout,
                             kWaitLimitNs);
    }
    ok = __all_sync(0xffffffffu, ok);
    // swap the row sums and maxima with the other warp at the pair barrier; a warp that left the
    // tile loop early may stop waiting for published maxima, so its partner's bounded waits give
    // up and both skip the record
    red[par * kM + r] = ok ? l : -1.f;
    red[2 * kM + par * kM + r] = m_own;
    mbar_arrive(bar(pair_bar));
    bool pair_ok = mbar_wait_bounded(bar(pair_bar), pair_phase & 1, abort_flag, p.err, kDevTimeout, kWaitLimitNs);
    ++pair_phase;
    pair_ok = __all_sync(0xffffffffu, pair_ok);
    const float l0 = pair_ok ? red[r] : -1.f, l1 = pair_ok ? red[kM + r] : -1.f;
    ok = __all_sync(0xffffffffu, l0 >= 0.f && l1 >= 0.f);
    if (ok) {
      tc_fence_after();
      const float m_used = n_tiles > 0 ? red[2 * kM + ((n_tiles - 1) & 1) * kM + r] : -INFINITY;
      const float m0 = red[2 * kM + r], m1 = red[2 * kM + kM + r];
      const float lt = (l0 > 0.f ? l0 * ex2_approx(m0 - m_used) : 0.f) + (l1 > 0.f ? l1 * ex2_approx(m1 - m_used) : 0.f);
      if (!causal && row < rows && (rec < 0 || rec >= p.n_records)) {
        if (half == 0) atomicCAS(p.err, 0, (int32_t)kDevBadRecord);
        rec = -1;
      }
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      uint32_t u[2][32];
      GRANIKV_TMEM_LD32(tmem + lane_off + kColO + half * 64, u[0]);
      GRANIKV_TMEM_LD32(tmem + lane_off + kColO + half * 64 + 32, u[1]);
      tmem_wait_ld();
      // Stage the normalised half row in shared memory (the K and V rings are idle: every MMA
      // has completed), 16-byte chunk c of row r at chunk c ^ (r % 32), so that a warp's 32
      // rows hit all banks; the pair then stores whole 512-byte rows, one per warp instruction.
      fence_proxy_async_smem();
      unsigned char* stage = smem + kOffK;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          const int chunk = half * 16 + c * 8 + k / 4;
          *reinterpret_cast<float4*>(stage + r * 512 + ((chunk ^ (r & 31)) << 4)) =
              make_float4(__uint_as_float(u[c][k]) * inv, __uint_as_float(u[c][k + 1]) * inv,
                          __uint_as_float(u[c][k + 2]) * inv, __uint_as_float(u[c][k + 3]) * inv);
        }
      if (half == 0) {
        const float lse_row = lt > 0.f ? (m_used + __log2f(lt)) * kLn2 : -INFINITY;
        if (causal) {
          // a prefill row has exactly one record: the final o (bf16) and lse go out directly
          const int64_t orow = (int64_t)b * p.n_q + h;
          reinterpret_cast<int64_t*>(smem + kOffV)[r] = row < rows ? orow * kD : -1;
          if (row < rows) p.lse[orow] = lse_row;
        } else {
          reinterpret_cast<int64_t*>(smem + kOffV)[r] = rec >= 0 ? ((int64_t)rec * p.n_q + h) * kD : -1;
          if (rec >= 0) st_record(p.rec_lse + (int64_t)rec * p.n_q + h, lse_row, l2_policy_keep());
        }
      }
    }
    // both halves of the quarter's 32 rows are staged (both warps of a pair agree on `ok`)
    mbar_arrive(bar(pair_bar));
    bool staged = mbar_wait_bounded(bar(pair_bar), pair_phase & 1, abort_flag, p.err, kDevTimeout, kWaitLimitNs);
    ++pair_phase;
    staged = __all_sync(0xffffffffu, staged) && ok;
    if (staged) {
      const unsigned char* stage = smem + kOffK;
      const int64_t* sdst = reinterpret_cast<const int64_t*>(smem + kOffV);
      const uint64_t keep = l2_policy_keep();
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int rr = quad * 32 + half * 16 + i;
        const int64_t d = sdst[rr];
        if (d < 0) continue;
        const float4 x = *reinterpret_cast<const float4*>(stage + rr * 512 + ((lane ^ (rr & 31)) << 4));
        if (causal) {
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + d + lane * 4) =
              make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
        } else {
          st_record4(p.rec_o + d + lane * 4, x, keep);
        }
      }
      if (p.fused_merge && !causal) {
        // the row's record is complete (both warps stored their rows) before its ticket moves
        __threadfence();
        mbar_arrive(bar(pair_bar));
        bool stored = mbar_wait_bounded(bar(pair_bar), pair_phase & 1, abort_flag, p.err, kDevTimeout, kWaitLimitNs);
        ++pair_phase;
        stored = __all_sync(0xffffffffu, stored);
        if (half == 0 && stored) {
          const bool last_arrival = rec >= 0 && arrive_row(p, b, h);
          warp_merge_completed(p, last_arrival, b, h, lane);
        }
      }
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


}  // namespace
}  // namespace dns
}  // namespace granikv
