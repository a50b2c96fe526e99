// kernels_dense_tc.cu -- dense prefix backend on the 5th-generation tensor cores (tcgen05/TMEM).
//
// GraniKV (arXiv:2608.15584), "2 Related Work": HydraGen-style attention batches all queries
// that share a prefix into one matrix-matrix product against the prefix K/V; "3 GraniKV":
// the dense backend targets compute-bound steps, and is possible only because the HOT slab
// stores the prefix contiguously (the card page: paged prefixes force a gather instead).
//
// One CTA takes one (prefix group, KV head j, 128-row block, L_p piece).  Rows are the group's
// (request, head-in-group) pairs of KV head j, so M = 128 query rows share every K/V tile.
// Per 64-token tile:
//     S = Q K^T   (M=128, N=64, K=128: 8 tcgen05.mma, fp32 accumulator in TMEM)
//     P = 2^(S*scale*log2e - m)   (softmax warps, one row per thread, P -> shared memory)
//     O += P V    (M=128, N=128, K=64: 4 tcgen05.mma, O stays in TMEM for the whole piece)
// Roles: warps 0-3 do the softmax and the epilogue (thread r owns row r, TMEM lane r), warp 4
// issues the TMA loads of K/V tiles (two 64-dim halves each, 128-byte swizzle) into a 5-stage
// ring, so up to four tiles (128 KB) are in flight per SM, warp 5 issues the MMAs.  S is
// double-buffered in TMEM so S(i+1) overlaps the softmax of tile i.  The
// running max is only moved (and O rescaled in TMEM) when it grows by more than 2^8, so most
// tiles skip the rescale; the final normalisation uses the same max, so the result is exact.
// Every mbarrier wait is bounded in time; on expiry the CTA raises an abort flag, latches an
// error, drains what it issued and frees its TMEM.
#include <cuda.h>

#include "internal.h"
#include "merge_util.cuh"
#include "mma_util.cuh"
#include "tc_util.cuh"

namespace granikv {
namespace {

constexpr int kD = 128;
constexpr int kM = kDenseRows;                // 128 query rows per CTA
constexpr int kN = kDenseTile;                // 64 tokens per tile
static_assert(kN == 64, "the P layout and the MMA shapes below assume 64-token tiles");
constexpr int kStages = 5;                    // K/V tile ring
constexpr int kThreads = 192;
constexpr int kHalf = kN * 128;               // one 64-dim half of a K or V tile: 8 KB
constexpr int kTile = 2 * kHalf;              // 16 KB
constexpr int kQBytes = kM * kD * 2;          // 32 KB (two 64-dim K-blocks)
constexpr int kPBytes = kM * kN * 2;          // 16 KB (one 64-token K-block)
constexpr int kOffQ = 0;
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffKV = kOffP + kPBytes;       // stage s: K at kOffKV + s*2*kTile, V after it
constexpr int kOffBar = kOffKV + kStages * 2 * kTile;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // barriers + alignment slack
constexpr uint32_t kTmemCols = 256;           // S0 [0,64), S1 [64,128), O [128,256)
constexpr uint32_t kColO = 128;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;     // log2 of the largest growth tolerated in P
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int32_t kDevTimeout = 6;

// barrier slots (8 bytes each) inside the barrier area
enum : int {
  kBarKvFull = 0,                  // [kStages] TMA -> MMA
  kBarKvEmpty = kStages,           // [kStages] MMA (PV done) -> TMA
  kBarSFull = 2 * kStages,         // [2] S(i) in TMEM -> softmax
  kBarPFull = 2 * kStages + 2,     // P(i) in shared memory -> MMA (128 arrivals)
  kBarPvDone = 2 * kStages + 3,    // [2] PV(i) done -> softmax
  kBarDrain = 2 * kStages + 5,     // all MMAs done -> teardown
  kNumBars = 2 * kStages + 6
};
static_assert(8 * kNumBars + 16 <= 256, "barrier area");

__global__ void __launch_bounds__(kThreads, 1)
    dense_tc_kernel(AttnParams p, int32_t first_item, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzle atoms
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base = (raw_u + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw_u);
  const uint32_t sQ = base + kOffQ, sP = base + kOffP, sKV = base + kOffKV;
  const uint32_t sBar = base + kOffBar;
  auto bar = [&](int i) { return sBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars + 8);

  const DevPrefixItem it = p.pitems[first_item + blockIdx.x];
  const DevGroup gr = p.groups[it.group];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = p.g;
  const int j = it.kv_head;
  const int32_t rows = gr.n_req * g;
  int32_t t0, t1;
  piece_range(gr, it.split, t0, t1);
  const int n_tiles = (t1 - t0 + kN - 1) / kN;
  const bool slab_ok = gr.slab_off >= 0 && gr.slab_off + gr.L_p <= p.n_hot && n_tiles > 0;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), i == kBarPFull ? 128u : 1u);
    *abort_flag = slab_ok ? 0 : 1;
    if (!slab_ok) atomicCAS(p.err, 0, (int32_t)kDevBadSlab);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  // Q rows of this block -> shared memory, K-major with 128-byte swizzle: row r, 16-byte
  // chunk c lives in 64-dim block c/8 at r*128 + ((c%8) ^ (r%8))*16; rows past the group are 0
  const int32_t rbase = it.row_block * kM;
  for (int idx = tid; idx < kM * 16; idx += kThreads) {
    const int r = idx >> 4;
    const int c = idx & 15;
    const int32_t row = rbase + r;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < rows) {
      const int32_t b = p.group_req[gr.req_begin + row / g];
      const int32_t h = j * g + row % g;
      v = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + ((int64_t)b * p.n_q + h) * kD)[c];
    }
    const uint32_t dst = sQ + (c >> 3) * (kM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && !*abort_flag) {
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kStages;
        if (i >= kStages &&
            !mbar_wait_bounded(bar(kBarKvEmpty + st), ((i / kStages) - 1) & 1, abort_flag, p.err, kDevTimeout,
                               kWaitLimitNs))
          break;
        const uint32_t kdst = sKV + st * 2 * kTile;
        const uint32_t vdst = kdst + kTile;
        const int32_t z = (int32_t)(gr.slab_off + t0 + i * kN);
        mbar_arrive_expect_tx(bar(kBarKvFull + st), 2 * kTile);
        tma_load_3d(kdst, &tmk, 0, j, z, bar(kBarKvFull + st));
        tma_load_3d(kdst + kHalf, &tmk, 64, j, z, bar(kBarKvFull + st));
        tma_load_3d(vdst, &tmv, 0, j, z, bar(kBarKvFull + st));
        tma_load_3d(vdst + kHalf, &tmv, 64, j, z, bar(kBarKvFull + st));
        issued = i + 1;
      }
      // never leave with a copy in flight: wait for every issued tile to land
      for (int i = max(0, issued - kStages); i < issued; ++i) {
        const int st = i % kStages;
        const uint64_t t_start = globaltimer_ns();
        while (!mbar_try_wait(bar(kBarKvFull + st), (i / kStages) & 1)) {
          if (globaltimer_ns() - t_start > kWaitLimitNs) {
            atomicCAS(p.err, 0, kDevTimeout);
            break;
          }
        }
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && !*abort_flag) {
      constexpr uint32_t idS = idesc_bf16_f32(kM, kN, false);
      constexpr uint32_t idO = idesc_bf16_f32(kM, kD, true);
      bool ok = true;
      int committed = 0;  // tcgen05 commits issued, for the drain below
      auto issue_s = [&](int i) -> bool {
        const int st = i % kStages;
        if (!mbar_wait_bounded(bar(kBarKvFull + st), (i / kStages) & 1, abort_flag, p.err, kDevTimeout, kWaitLimitNs))
          return false;
        tc_fence_after();
        const uint32_t kst = sKV + st * 2 * kTile;
        const uint32_t dS = tmem + (uint32_t)((i & 1) * kN);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * (kM * 128) + (kk & 3) * 32;
          const uint64_t a = smem_desc_sw128(sQ + off, 16, 1024);
          const uint64_t b = smem_desc_sw128(kst + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
          umma_f16(dS, a, b, idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(kBarSFull + (i & 1)));
        ++committed;
        return true;
      };
      ok = issue_s(0);
      for (int i = 0; ok && i < n_tiles; ++i) {
        if (i + 1 < n_tiles && !issue_s(i + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait_bounded(bar(kBarPFull), i & 1, abort_flag, p.err, kDevTimeout, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int st = i % kStages;
        const uint32_t vst = sKV + st * 2 * kTile + kTile;
#pragma unroll
        for (int ks = 0; ks < kN / 16; ++ks) {
          const uint64_t a = smem_desc_sw128(sP + ks * 32, 16, 1024);
          // V tile as an MN-major B operand: 16 tokens per step (2048 bytes), the two 64-dim
          // halves kHalf apart (leading offset), 8-token groups 1024 bytes apart (stride)
          const uint64_t b = smem_desc_sw128(vst + ks * 2048, kHalf, 1024);
          umma_f16(tmem + kColO, a, b, idO, (i > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(bar(kBarKvEmpty + st));
        umma_commit(bar(kBarPvDone + (i & 1)));
        committed += 2;
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
    // ---------------- softmax warps 0-3: thread r owns row r ----------------
    const int r = tid;  // 0..127, TMEM lane r
    const uint32_t lane_off = (uint32_t)((warp * 32) << 16);
    const float scale = p.scale_log2;
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = !*abort_flag;
    for (int i = 0; ok && i < n_tiles; ++i) {
      ok = mbar_wait_bounded(bar(kBarSFull + (i & 1)), (i >> 1) & 1, abort_flag, p.err, kDevTimeout, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);  // the TMEM loads below are warp-collective
      if (!ok) break;
      tc_fence_after();
      const int valid = min(kN, t1 - t0 - i * kN);
      float s[kN];
      {
        uint32_t u[2][32];
        const uint32_t ts = tmem + lane_off + (uint32_t)((i & 1) * kN);
        GRANIKV_TMEM_LD32(ts, u[0]);
        GRANIKV_TMEM_LD32(ts + 32, u[1]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int k = 0; k < 32; ++k) s[c * 32 + k] = __uint_as_float(u[c][k]);
      }
      float mx = -INFINITY;
      if (valid == kN) {
#pragma unroll
        for (int k = 0; k < kN; ++k) {
          s[k] *= scale;
          mx = fmaxf(mx, s[k]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < kN; ++k) {
          s[k] = k < valid ? s[k] * scale : -INFINITY;
          mx = fmaxf(mx, s[k]);
        }
      }
      // move the running max only when it grows by more than 2^kRescaleThreshold
      const bool first = (i == 0);
      const bool need = first ? true : (mx > m_used + kRescaleThreshold);
      const bool warp_need = __any_sync(0xffffffffu, need && !first);
      if (first) {
        m_used = mx;
      } else if (warp_need) {
        // O must hold PV(i-1) before it is rescaled
        if (!mbar_wait_bounded(bar(kBarPvDone + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag, p.err, kDevTimeout,
                               kWaitLimitNs)) {
          ok = false;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float m_new = fmaxf(m_used, mx);
        const float alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
        l *= alpha;
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
      float psum = 0.f;
      uint32_t pk[kN / 2];
#pragma unroll
      for (int k = 0; k < kN / 2; ++k) {
        const float a = ex2_approx(s[2 * k] - m_used);
        const float b = ex2_approx(s[2 * k + 1] - m_used);
        psum += a + b;
        pk[k] = pack_bf16(a, b);
      }
      l += psum;
      // P(i) overwrites P(i-1): PV(i-1) must be done
      if (i > 0 && !mbar_wait_bounded(bar(kBarPvDone + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag, p.err,
                                      kDevTimeout, kWaitLimitNs)) {
        ok = false;
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // row r of P: 8 chunks of 8 tokens in one 64-token K-block, swizzled
#pragma unroll
      for (int c = 0; c < kN / 8; ++c) {
        const uint32_t dst = sP + r * 128 + (((c & 7) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(pk[4 * c]), "r"(pk[4 * c + 1]),
                     "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                     : "memory");
      }
      // zero V rows past the piece in the last tile so 0 * garbage cannot reach O
      if (valid < kN && r >= valid && r < kN) {
        const uint32_t vst = sKV + (i % kStages) * 2 * kTile + kTile;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vst + r * 128 + c * 16), "r"(0u) : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vst + kHalf + r * 128 + c * 16), "r"(0u)
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull));
    }
    // epilogue: wait for the last PV, normalise, write this row's record
    if (ok) {
      const int last = n_tiles - 1;
      ok = mbar_wait_bounded(bar(kBarPvDone + (last & 1)), (last >> 1) & 1, abort_flag, p.err, kDevTimeout,
                             kWaitLimitNs);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const int32_t row = rbase + r;
      int32_t b = -1, h = 0, rec = -1;
      if (row < rows) {
        b = p.group_req[gr.req_begin + row / g];
        h = j * g + row % g;
        rec = p.reqs[b].rec_base + it.split;
        if (rec < 0 || rec >= p.n_records) {
          atomicCAS(p.err, 0, (int32_t)kDevBadRecord);
          rec = -1;
        }
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* dst = rec >= 0 ? p.rec_o + ((int64_t)rec * p.n_q + h) * kD : nullptr;
      uint32_t u[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        GRANIKV_TMEM_LD32(tmem + lane_off + kColO + c * 32, u);
        tmem_wait_ld();
        if (dst) {
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(dst + c * 32 + k) =
                make_float4(__uint_as_float(u[k]) * inv, __uint_as_float(u[k + 1]) * inv,
                            __uint_as_float(u[k + 2]) * inv, __uint_as_float(u[k + 3]) * inv);
        }
      }
      if (rec >= 0) p.rec_lse[(int64_t)rec * p.n_q + h] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
      if (p.fused_merge) {
        __threadfence();
        __syncwarp();
        const bool last = rec >= 0 && arrive_row(p, b, h);
        warp_merge_completed(p, last, b, h, lane);
      }
    }
  }

  // ---------------- teardown ----------------
  // If the CTA aborted, wait (bounded) until every MMA this CTA issued has completed: the last
  // commit of each kind is observed through the PV barriers.  Then free TMEM.
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_dense_tc(const AttnParams& p, int32_t first_item, int32_t n_items, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, cudaStream_t s) {
  if (n_items <= 0) return cudaSuccess;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(dense_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  dense_tc_kernel<<<n_items, kThreads, kSmemBytes, s>>>(p, first_item, tmk, tmv);
  return cudaGetLastError();
}

}  // namespace granikv
