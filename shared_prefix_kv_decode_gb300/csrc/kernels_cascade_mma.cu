// kernels_cascade_mma.cu -- cascade prefix backend on warp-level bf16 tensor cores.
//
// GraniKV (arXiv:2608.15584), "2 Related Work": cascade inference reads the shared prefix
// once per step, cutting its HBM reads from O(B) to O(1); "3 GraniKV", dual attention
// backends: cascade is the backend for memory-bound steps, and the HOT slab makes the prefix
// a contiguous run of slots ("3 GraniKV": dense, indirection-free prefix reads).
//
// One CTA takes one (prefix group, KV head j, L_p piece, block of 128 query rows).  Rows are
// the group's (request, head-in-group) pairs of KV head j (grouped-query packing), so every
// K/V tile staged in shared memory serves up to 128 queries.  Eight warps own 16 rows each:
//     S = Q . K^T   (16 x 64 per warp per tile)       P = softmax part,   O += P . V
// with m16n8k16 bf16 MMAs, fp32 accumulators and a running (max, sum) per row.  A block of at
// most 16 rows (B * g <= 16: a few requests) would leave seven warps without rows and every
// tile waiting on one warp's chain; there all eight warps take the same rows, each its own 8
// tokens of every tile (S by m16n8k16, P V by m16n8k8), and their eight states are merged by
// log-sum-exp in shared memory at the end, into warp 0, which writes the record.  K/V tiles of
// 64 tokens x 128 dims (16 KB each) move through a 3-stage cp.async ring with 16-byte chunks,
// XOR-swizzled so ldmatrix reads are conflict-free.  The piece's partial state (normalised o
// and lse per row) goes to the request's record for that piece.
#include "internal.h"
#include "merge_util.cuh"
#include "mma_util.cuh"

namespace granikv {
namespace {

constexpr int kD = 128;
constexpr int kTok = kCascadeTile;              // 64 tokens per tile
constexpr int kStages = 3;
constexpr int kWarps = 8;
constexpr int kRows = kWarps * 16;              // 128 query rows per CTA
static_assert(kRows == kCascadeRows, "planner and kernel disagree on rows per CTA");
constexpr int kRowBytes = kD * 2;               // 256 B
constexpr int kTileBytes = kTok * kRowBytes;    // 16 KB
constexpr int kStageBytes = 2 * kTileBytes;     // K + V
constexpr int kSmemBytes = kStages * kStageBytes;  // 96 KB
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * kRowBytes + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kWarps * 32, 1) cascade_mma_kernel(AttnParams p, int32_t first_item) {
  extern __shared__ __align__(128) unsigned char smem[];
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
  if (gr.slab_off < 0 || gr.slab_off + gr.L_p > p.n_hot) {
    if (tid == 0) latch_err(p.err, kDevBadSlab);
    return;
  }
  const int64_t tok_bytes = (int64_t)p.n_kv * kRowBytes;
  const char* kbase = static_cast<const char*>(p.kpool) + (gr.slab_off + t0) * tok_bytes + (int64_t)j * kRowBytes;
  const char* vbase = static_cast<const char*>(p.vpool) + (gr.slab_off + t0) * tok_bytes + (int64_t)j * kRowBytes;
  const uint32_t sbase = smem_u32(smem);
  const int n_tiles = (t1 - t0 + kTok - 1) / kTok;

  auto issue = [&](int tile, int stage) {
    if (tile < n_tiles) {
      const uint32_t kdst = sbase + stage * kStageBytes;
      const uint32_t vdst = kdst + kTileBytes;
      const int valid = min(kTok, t1 - t0 - tile * kTok);
#pragma unroll
      for (int i = 0; i < (kTok * 16) / (kWarps * 32); ++i) {
        const int c = tid + kWarps * 32 * i;
        const int row = c >> 4;
        const int piece = c & 15;
        const bool ok = row < valid;
        const int64_t off = ok ? (int64_t)(tile * kTok + row) * tok_bytes + piece * 16 : 0;
        cp_async16(kdst + swz(row, piece), kbase + off, ok ? 16 : 0);
        cp_async16(vdst + swz(row, piece), vbase + off, ok ? 16 : 0);
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) issue(s, s);

  // Q as A fragments: rows r_lo = base + lane/4 and r_hi = r_lo + 8 of this warp (of the block
  // for every warp when the block's rows fit one warp)
  const bool split = rows - it.row_block * kRows <= 16;
  const int32_t rbase = it.row_block * kRows + (split ? 0 : warp * 16);
  const bool warp_active = rbase < rows;
  uint32_t qf[8][4];
  int32_t b_lo = -1, h_lo = 0, b_hi = -1, h_hi = 0;
  {
    const int32_t r_lo = rbase + (lane >> 2), r_hi = r_lo + 8;
    if (r_lo < rows) {
      b_lo = p.group_req[gr.req_begin + r_lo / g];
      h_lo = j * g + r_lo % g;
    }
    if (r_hi < rows) {
      b_hi = p.group_req[gr.req_begin + r_hi / g];
      h_hi = j * g + r_hi % g;
    }
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q);
    const uint32_t* qlo = b_lo >= 0 ? reinterpret_cast<const uint32_t*>(qb + ((int64_t)b_lo * p.n_q + h_lo) * kD) : nullptr;
    const uint32_t* qhi = b_hi >= 0 ? reinterpret_cast<const uint32_t*>(qb + ((int64_t)b_hi * p.n_q + h_hi) * kD) : nullptr;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int w = kk * 8 + (lane & 3);
      qf[kk][0] = qlo ? qlo[w] : 0u;
      qf[kk][1] = qhi ? qhi[w] : 0u;
      qf[kk][2] = qlo ? qlo[w + 4] : 0u;
      qf[kk][3] = qhi ? qhi[w + 4] : 0u;
    }
  }

  const float scale = p.scale_log2;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float o[16][4];
#pragma unroll
  for (int dt = 0; dt < 16; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;

  for (int tile = 0; tile < n_tiles; ++tile) {
    const int stage = tile % kStages;
    cp_async_wait<kStages - 2>();
    __syncthreads();
    issue(tile + kStages - 1, (tile + kStages - 1) % kStages);
    if (!warp_active) continue;
    const uint32_t kst = sbase + stage * kStageBytes;
    const uint32_t vst = kst + kTileBytes;
    const int valid = min(kTok, t1 - t0 - tile * kTok);

    if (split) {
      // this warp's 8 tokens of the tile: S (16 x 8) = Q K_w^T, one n-tile, 8 k-steps
      const int mi = lane >> 3;
      const int trow = warp * 8 + (lane & 7);
      float sw[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kst + swz(trow, kq * 4 + mi), b0, b1, b2, b3);
        mma_bf16_16816(sw, qf[kq * 2][0], qf[kq * 2][1], qf[kq * 2][2], qf[kq * 2][3], b0, b1);
        mma_bf16_16816(sw, qf[kq * 2 + 1][0], qf[kq * 2 + 1][1], qf[kq * 2 + 1][2], qf[kq * 2 + 1][3], b2, b3);
      }
      const int c0 = warp * 8 + 2 * (lane & 3);
      sw[0] = c0 < valid ? sw[0] * scale : -INFINITY;
      sw[1] = c0 + 1 < valid ? sw[1] * scale : -INFINITY;
      sw[2] = c0 < valid ? sw[2] * scale : -INFINITY;
      sw[3] = c0 + 1 < valid ? sw[3] * scale : -INFINITY;
      float mx_lo = fmaxf(sw[0], sw[1]), mx_hi = fmaxf(sw[2], sw[3]);
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, off));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, off));
      }
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float mu_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
      const float mu_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
      const float al_lo = exp2f(m_lo - mu_lo), al_hi = exp2f(m_hi - mu_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      const float p0 = exp2f(sw[0] - mu_lo), p1 = exp2f(sw[1] - mu_lo);
      const float p2 = exp2f(sw[2] - mu_hi), p3 = exp2f(sw[3] - mu_hi);
      l_lo = l_lo * al_lo + (p0 + p1);
      l_hi = l_hi * al_hi + (p2 + p3);
      const uint32_t a0 = pack_bf16(p0, p1), a1 = pack_bf16(p2, p3);
      // O += P V_w: one k-step of 8 tokens, 16 n-tiles of 8 dims
#pragma unroll
      for (int dq = 0; dq < 4; ++dq) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vst + swz(trow, dq * 4 + mi), b0, b1, b2, b3);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float(&od)[4] = o[dq * 4 + i];
          od[0] *= al_lo;
          od[1] *= al_lo;
          od[2] *= al_hi;
          od[3] *= al_hi;
        }
        mma_bf16_1688(o[dq * 4 + 0], a0, a1, b0);
        mma_bf16_1688(o[dq * 4 + 1], a0, a1, b1);
        mma_bf16_1688(o[dq * 4 + 2], a0, a1, b2);
        mma_bf16_1688(o[dq * 4 + 3], a0, a1, b3);
      }
      continue;
    }

    // S = Q K^T over 64 tokens: 8 n-tiles of 8 tokens
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    {
      const int mi = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int row = (np * 2 + (mi >> 1)) * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kst + swz(row, kk * 2 + (mi & 1)), b0, b1, b2, b3);
          mma_bf16_16816(s[np * 2], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
          mma_bf16_16816(s[np * 2 + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
        }
      }
    }
    // scale, mask the ragged tail, row max
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int c0 = nt * 8 + 2 * (lane & 3);
      s[nt][0] = c0 < valid ? s[nt][0] * scale : -INFINITY;
      s[nt][1] = c0 + 1 < valid ? s[nt][1] * scale : -INFINITY;
      s[nt][2] = c0 < valid ? s[nt][2] * scale : -INFINITY;
      s[nt][3] = c0 + 1 < valid ? s[nt][3] * scale : -INFINITY;
      mx_lo = fmaxf(mx_lo, fmaxf(s[nt][0], s[nt][1]));
      mx_hi = fmaxf(mx_hi, fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, off));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, off));
    }
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float mu_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
    const float mu_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
    const float al_lo = exp2f(m_lo - mu_lo), al_hi = exp2f(m_hi - mu_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    float ps_lo = 0.f, ps_hi = 0.f;
    uint32_t pa[4][4];  // P as A fragments, one per 16-token k-step
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = exp2f(s[nt][0] - mu_lo), p1 = exp2f(s[nt][1] - mu_lo);
      const float p2 = exp2f(s[nt][2] - mu_hi), p3 = exp2f(s[nt][3] - mu_hi);
      ps_lo += p0 + p1;
      ps_hi += p2 + p3;
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
    l_lo = l_lo * al_lo + ps_lo;
    l_hi = l_hi * al_hi + ps_hi;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      o[dt][0] *= al_lo;
      o[dt][1] *= al_lo;
      o[dt][2] *= al_hi;
      o[dt][3] *= al_hi;
    }
    // O += P V: 4 k-steps of 16 tokens, 16 n-tiles of 8 dims
    {
      const int mi = lane >> 3;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int row = ks * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vst + swz(row, dp * 2 + (mi >> 1)), b0, b1, b2, b3);
          mma_bf16_16816(o[dp * 2], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b0, b1);
          mma_bf16_16816(o[dp * 2 + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b2, b3);
        }
      }
    }
  }
  cp_async_wait<0>();
  if (split) {
    // Merge the eight warps' states of the block's 16 rows (each over its own tokens) by
    // log-sum-exp, in the ring's shared memory, into warp 0's registers in the layout below.
    constexpr int kR = 16;
    float* so = reinterpret_cast<float*>(smem);  // [warp][row][dim]
    float* sm = so + kWarps * kR * kD;           // [warp][row] running max (log2 units)
    float* sl = sm + kWarps * kR;                // [warp][row] sum
    float* sc = sl + kWarps * kR;                // [row][dim] merged, unnormalised
    float* sM = sc + kR * kD;                    // [row]
    float* sL = sM + kR;                         // [row]
    static_assert((kWarps * kR * kD + 2 * kWarps * kR + kR * kD + 2 * kR) * 4 <= kSmemBytes, "merge space");
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      l_lo += __shfl_xor_sync(0xffffffffu, l_lo, off);
      l_hi += __shfl_xor_sync(0xffffffffu, l_hi, off);
    }
    const int gq = lane >> 2, tq = lane & 3;
    __syncthreads();  // every warp is done reading the ring
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      *reinterpret_cast<float2*>(so + (warp * kR + gq) * kD + dt * 8 + 2 * tq) = make_float2(o[dt][0], o[dt][1]);
      *reinterpret_cast<float2*>(so + (warp * kR + gq + 8) * kD + dt * 8 + 2 * tq) = make_float2(o[dt][2], o[dt][3]);
    }
    if (tq == 0) {
      sm[warp * kR + gq] = m_lo;
      sm[warp * kR + gq + 8] = m_hi;
      sl[warp * kR + gq] = l_lo;
      sl[warp * kR + gq + 8] = l_hi;
    }
    __syncthreads();
    {
      const int r = tid >> 4;          // 16 threads a row
      const int d0 = (tid & 15) * 8;   // 8 dims a thread
      float mx = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, sm[w * kR + r]);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float den = 0.f;
      if (mx != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float mw = sm[w * kR + r];
          const float a = mw == -INFINITY ? 0.f : exp2f(mw - mx);
          den += a * sl[w * kR + r];
          const float4* src = reinterpret_cast<const float4*>(so + (w * kR + r) * kD + d0);
          const float4 x = src[0], y = src[1];
          acc[0] += a * x.x; acc[1] += a * x.y; acc[2] += a * x.z; acc[3] += a * x.w;
          acc[4] += a * y.x; acc[5] += a * y.y; acc[6] += a * y.z; acc[7] += a * y.w;
        }
      }
      float4* dst = reinterpret_cast<float4*>(sc + r * kD + d0);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      if ((tid & 15) == 0) {
        sM[r] = mx;
        sL[r] = den;
      }
    }
    __syncthreads();
    if (warp != 0) return;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      const float2 x = *reinterpret_cast<const float2*>(sc + gq * kD + dt * 8 + 2 * tq);
      const float2 y = *reinterpret_cast<const float2*>(sc + (gq + 8) * kD + dt * 8 + 2 * tq);
      o[dt][0] = x.x;
      o[dt][1] = x.y;
      o[dt][2] = y.x;
      o[dt][3] = y.y;
    }
    m_lo = sM[gq];
    m_hi = sM[gq + 8];
    l_lo = tq == 0 ? sL[gq] : 0.f;  // the quad sum below restores the row's sum
    l_hi = tq == 0 ? sL[gq + 8] : 0.f;
  }
  if (!warp_active) return;

  // full row sums over the quad, normalise, write each row's record for this piece
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, off);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, off);
  }
  const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
  const float inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
  const int dcol = 2 * (lane & 3);
  int32_t rec_lo = -1, rec_hi = -1;
  if (b_lo >= 0) {
    const int32_t rec = p.reqs[b_lo].rec_base + it.split;
    if (rec >= 0 && rec < p.n_records) {
      rec_lo = rec;
      float* dst = p.rec_o + ((int64_t)rec * p.n_q + h_lo) * kD + dcol;
#pragma unroll
      for (int dt = 0; dt < 16; ++dt)
        *reinterpret_cast<float2*>(dst + dt * 8) = make_float2(o[dt][0] * inv_lo, o[dt][1] * inv_lo);
      if ((lane & 3) == 0)
        p.rec_lse[(int64_t)rec * p.n_q + h_lo] = l_lo > 0.f ? (m_lo + log2f(l_lo)) * kLn2 : -INFINITY;
    } else if ((lane & 3) == 0) {
      latch_err(p.err, kDevBadRecord);
    }
  }
  if (b_hi >= 0) {
    const int32_t rec = p.reqs[b_hi].rec_base + it.split;
    if (rec >= 0 && rec < p.n_records) {
      rec_hi = rec;
      float* dst = p.rec_o + ((int64_t)rec * p.n_q + h_hi) * kD + dcol;
#pragma unroll
      for (int dt = 0; dt < 16; ++dt)
        *reinterpret_cast<float2*>(dst + dt * 8) = make_float2(o[dt][2] * inv_hi, o[dt][3] * inv_hi);
      if ((lane & 3) == 0)
        p.rec_lse[(int64_t)rec * p.n_q + h_hi] = l_hi > 0.f ? (m_hi + log2f(l_hi)) * kLn2 : -INFINITY;
    } else if ((lane & 3) == 0) {
      latch_err(p.err, kDevBadRecord);
    }
  }
  if (p.fused_merge) {
    __threadfence();
    __syncwarp();
    const bool lead = (lane & 3) == 0;
    const bool last_lo = lead && rec_lo >= 0 && arrive_row(p, b_lo, h_lo);
    const bool last_hi = lead && rec_hi >= 0 && arrive_row(p, b_hi, h_hi);
    warp_merge_completed(p, last_lo, b_lo, h_lo, lane);
    warp_merge_completed(p, last_hi, b_hi, h_hi, lane);
  }
}

}  // namespace

cudaError_t launch_cascade_mma(const AttnParams& p, int32_t first_item, int32_t n_items, cudaStream_t s) {
  if (n_items <= 0) return cudaSuccess;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(cascade_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  cascade_mma_kernel<<<n_items, kWarps * 32, kSmemBytes, s>>>(p, first_item);
  return cudaGetLastError();
}

}  // namespace granikv
