// kernels_suffix_mma.cu -- COLD suffix partial attention on warp-level bf16 tensor cores.
//
// GraniKV (arXiv:2608.15584), "1 Introduction" / "3 GraniKV": suffix and decoded tokens sit in
// a token-level COLD pool (page size 1), so every token is gathered through the request's
// token table; "2 Related Work", prefix-suffix attention: the suffix is attended separately
// and merged with the prefix by log-sum-exp.
//
// Shape: head_dim 128, bf16, g = n_q/n_kv <= 8.  One warp owns one KV head of one request
// segment.  Because only g query heads share a KV head, tokens are the MMA's M dimension and
// the g heads its N dimension (8 columns):
//     S^T[16 tok x 8 heads] = K[16 tok x 128] . Q^T[128 x 8]          (8 mma.m16n8k16)
//     O^T[128 x 8 heads]   += V^T[128 x 16 tok] . P^T[16 tok x 8 heads] (8 mma.m16n8k16)
// P^T goes from the accumulator layout to the B-operand layout with movmatrix.  The online
// softmax (running max and sum per head column) reduces across lanes with warp shuffles.
//
// Work split: the plan cuts the concatenation of all requests' COLD tokens into one contiguous
// run per token-CTA (stream-K style), so every CTA streams the same number of tokens; each
// request segment inside a run writes one partial-state record.  blockIdx.y picks a group of
// eight KV heads (one group for the Llama and Qwen shapes), so the warps of a CTA fetch all
// heads of a slot's K and V rows (2 KB each) at the same time.  Each warp runs its own 3-stage cp.async pipeline: slot ids are read from the
// table, each token's 256-byte K and V rows are copied into a 16-byte-chunk-swizzled tile, and
// the pipeline runs on across segment boundaries.
#include "internal.h"
#include "merge_util.cuh"
#include "mma_util.cuh"

namespace granikv {
namespace {

constexpr int kD = 128;
constexpr int kTile = 16;                     // tokens per tile (MMA M)
constexpr int kStages = 3;
constexpr int kWarps = 8;                     // KV heads per CTA (all of them for n_kv <= 8)
constexpr int kRowBytes = kD * 2;             // one head's K (or V) row: 256 B
constexpr int kTileBytes = kTile * kRowBytes; // 4 KB
constexpr int kStageBytes = 2 * kTileBytes;   // K + V
constexpr int kWarpSmem = kStages * kStageBytes;
constexpr int kSlotBytes = kSuffixMaxCtaTokens * 4;  // the CTA's slot ids, loaded once
constexpr int kSmemBytes = kWarps * kWarpSmem + kSlotBytes;  // 192 KB + 16 KB
constexpr float kLn2 = 0.6931471805599453f;

// byte offset of 16-byte chunk c of row r in a tile of 256-byte rows (XOR swizzle so the 8
// rows of an ldmatrix hit 8 different bank groups)
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * kRowBytes + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kWarps * 32) suffix_mma_kernel(AttnParams p, const int32_t* __restrict__ cta_begin) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.y * kWarps + warp;  // KV head of this warp
  const int seg_begin = cta_begin[blockIdx.x];
  const int seg_end = cta_begin[blockIdx.x + 1];
  if (seg_begin >= seg_end) return;
  // The slot ids of all of this CTA's tokens (its segments back to back) go to shared memory
  // once, so the copy issue never waits on a table load.  The plan keeps a CTA's tokens within
  // kSuffixMaxCtaTokens.
  int32_t* sslot = reinterpret_cast<int32_t*>(smem + kWarps * kWarpSmem);
  {
    int base = 0;
    for (int sg = seg_begin; sg < seg_end; ++sg) {
      const DevSuffixItem seg = p.sitems[sg];
      const int len = seg.t1 - seg.t0;
      const int32_t* row = p.req_to_slot + (int64_t)seg.b * p.cap + seg.t0;
      for (int k = threadIdx.x; k < len && base + k < kSuffixMaxCtaTokens; k += blockDim.x) sslot[base + k] = row[k];
      base += len;
    }
    if (base > kSuffixMaxCtaTokens && threadIdx.x == 0) latch_err(p.err, kDevBadRecord);
    __syncthreads();
    if (base > kSuffixMaxCtaTokens) return;
  }
  if (j >= p.n_kv) return;  // no CTA-wide barrier is used below

  const uint32_t wsm = smem_u32(smem) + warp * kWarpSmem;
  const int64_t tok_bytes = (int64_t)p.n_kv * kRowBytes;
  const char* kbase = static_cast<const char*>(p.kpool) + (int64_t)j * kRowBytes;
  const char* vbase = static_cast<const char*>(p.vpool) + (int64_t)j * kRowBytes;
  const float scale = p.scale_log2;
  const int g = p.g;

  // ---- producer cursor: next tile to stage ---------------------------------------------
  int is = seg_begin;
  int it0 = p.sitems[is].t0;
  int is_base = 0;  // position of segment `is` in sslot
  constexpr int32_t kNoToken = INT32_MIN;  // rows past the segment: zero-filled, masked
  auto issue = [&](int stage) {
    if (is < seg_end) {
      const DevSuffixItem seg = p.sitems[is];
      int32_t slot = lane < min(kTile, seg.t1 - it0) ? sslot[is_base + (it0 - seg.t0) + lane] : kNoToken;
      if (slot != kNoToken && (slot < p.n_hot || slot >= p.n_slots)) {
        latch_err(p.err, kDevBadSlot);
        slot = kNoToken;
      }
      const uint32_t kdst = wsm + stage * kStageBytes;
      const uint32_t vdst = kdst + kTileBytes;
#pragma unroll
      for (int i = 0; i < (kTile * 16) / 32; ++i) {
        const int c = lane + 32 * i;
        const int row = c >> 4;
        const int piece = c & 15;
        const int32_t sl = __shfl_sync(0xffffffffu, slot, row);
        const bool ok = sl >= 0;
        const int64_t off = ok ? (int64_t)sl * tok_bytes + piece * 16 : 0;
        cp_async16(kdst + swz(row, piece), kbase + off, ok ? 16 : 0);
        cp_async16(vdst + swz(row, piece), vbase + off, ok ? 16 : 0);
      }
      it0 += kTile;
      if (it0 >= seg.t1) {
        is_base += seg.t1 - seg.t0;
        ++is;
        if (is < seg_end) it0 = p.sitems[is].t0;
      }
    }
    cp_async_commit();  // an empty group at the tail keeps the group count uniform
  };

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) issue(s);

  int tile = 0;  // tiles consumed so far
  const int h0 = 2 * (lane & 3);  // this thread's two head columns: h0, h0 + 1
  // Q^T as B fragments (column n = lane/4 is head j*g + n); the next segment's are loaded one
  // segment ahead so their latency hides behind the current segment's tiles
  uint32_t qn[8][2];
  auto load_q = [&](int sg) {
    const int n = lane >> 2;
    if (sg < seg_end && n < g) {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          static_cast<const __nv_bfloat16*>(p.q) + ((int64_t)p.sitems[sg].b * p.n_q + j * g + n) * kD);
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
  load_q(seg_begin);
  for (int sg = seg_begin; sg < seg_end; ++sg) {
    const DevSuffixItem seg = p.sitems[sg];
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

    for (int t = seg.t0; t < seg.t1; t += kTile, ++tile) {
      const int stage = tile % kStages;
      cp_async_wait<kStages - 2>();
      __syncwarp();
      issue((tile + kStages - 1) % kStages);
      const uint32_t kst = wsm + stage * kStageBytes;
      const uint32_t vst = kst + kTileBytes;

      // S^T = K . Q^T
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int mi = lane >> 3;
        const int r = (lane & 7) + (mi & 1) * 8;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kst + swz(r, kk * 2 + (mi >> 1)), a0, a1, a2, a3);
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
          ldsm_x4_t(vst + swz(r, mt * 2 + (mi & 1)), a0, a1, a2, a3);
          mma_bf16_16816(o[mt], a0, a1, a2, a3, b0, b1);
        }
      }
    }

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
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      if (w0) {
        dst0[mt * 16] = o[mt][0] * inv0;
        dst0[mt * 16 + 8] = o[mt][2] * inv0;
      }
      if (w1) {
        dst1[mt * 16] = o[mt][1] * inv1;
        dst1[mt * 16 + 8] = o[mt][3] * inv1;
      }
    }
    if (lane < 4) {
      float* ldst = p.rec_lse + (int64_t)rec * p.n_q + hq0;
      if (w0) ldst[0] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
      if (w1) ldst[1] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
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
  cp_async_wait<0>();
}

}  // namespace

cudaError_t launch_suffix_mma(const AttnParams& p, const int32_t* cta_begin, int32_t n_cta, cudaStream_t s) {
  if (n_cta <= 0) return cudaSuccess;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(suffix_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  dim3 grid(n_cta, (p.n_kv + kWarps - 1) / kWarps);
  suffix_mma_kernel<<<grid, kWarps * 32, kSmemBytes, s>>>(p, cta_begin);
  return cudaGetLastError();
}

}  // namespace granikv
