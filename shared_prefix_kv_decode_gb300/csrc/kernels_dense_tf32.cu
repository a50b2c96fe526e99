// kernels_dense_tf32.cu -- dense prefix backend for fp32 K/V on the 5th-generation tensor cores
// (tcgen05.mma kind::tf32, accumulators in TMEM).
//
// GraniKV (arXiv:2608.15584), "2 Related Work": HydraGen-style attention batches all queries
// that share a prefix into one matrix-matrix product against the prefix K/V; "3 GraniKV": the
// dense backend serves the compute-bound steps and reads the prefix from its contiguous HOT
// slab.  This is that backend for fp32 pools (any head_dim that is a multiple of 32, up to 128),
// so that forced dense and forced cascade run different kernels for fp32 too: the cascade
// backend of fp32 groups stays the CUDA-core kernel.
//
// One CTA of 128 threads per (prefix group, KV head j, 128-row block, L_p piece); thread t owns
// query row t of the block (TMEM lane t).  Per 32-token tile:
//     S = Q K^T          (M=128, N=32, K=d, fp32 accumulator in TMEM)
//     P = 2^(S*scale*log2e - m)   (each thread its row: running max m and sum l; P stored to
//                                  shared memory as the next product's A operand)
//     O = O*alpha + P V  (M=128, N=d, K=32, into O in TMEM; O is rescaled in TMEM when a row's
//                         max moves)
// Split precision: an MMA reads only the tf32 part of each fp32 operand (10 explicit mantissa
// bits), so every operand x is stored as x_hi (x with its 13 low mantissa bits cleared, exact
// in tf32) and x_lo = x - x_hi (exact in fp32), and each product runs as
// A_hi B_hi + A_hi B_lo + A_lo B_hi (the dropped A_lo B_lo and the tf32 reading of the lo parts
// are below 2^-20 of |a b|): fp32-level results from the tensor cores at three times the MMAs.
// All operands are K-major with the 128-byte swizzle (32 fp32 of K per 128-byte atom row, 8 rows
// per 1024-byte atom).  V is transposed while it is staged, so V^T (rows = head dims, K = tokens)
// is K-major too.  Tiles are staged with plain loads and each tile's MMAs complete before the
// next tile is staged: this path serves small fp32 problems; the pipelined, TMA-fed kernel is
// the bf16 one.
//
// Every mbarrier wait is bounded in time; on expiry the CTA latches an error, waits (bounded)
// for the MMAs it issued and frees its TMEM.
#include <cuda_runtime.h>

#include "internal.h"
#include "launch_util.cuh"
#include "mma_util.cuh"
#include "tc_util.cuh"

namespace granikv {
namespace {

constexpr int kRows = kDenseTf32Rows;  // query rows per CTA (MMA M)
constexpr int kTok = kDenseTf32Tile;   // tokens per tile (N of S, K of P V)
static_assert(kTok == 32, "one 32-wide column block of P and V^T per tile");
constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 256;    // S at column 0 (32 columns), O at 128 (d <= 128 columns)
constexpr uint32_t kColO = 128;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Each operand twice, hi part then lo part (`kLo` bytes further on).
template <int D>
struct Tf32Layout {
  static constexpr int kQ = 0;                         // [128 rows x D], K-major
  static constexpr int kQLo = kRows * D * 4;
  static constexpr int kK = kQ + 2 * kQLo;             // [32 tokens x D], K-major
  static constexpr int kKLo = kTok * D * 4;
  static constexpr int kV = kK + 2 * kKLo;             // V^T: [D dims x 32 tokens], K-major
  static constexpr int kVLo = D * kTok * 4;
  static constexpr int kP = kV + 2 * kVLo;             // [128 rows x 32 tokens], K-major
  static constexpr int kPLo = kRows * kTok * 4;
  static constexpr int kBar = kP + 2 * kPLo;           // S done, O done, drain; abort flag; TMEM slot
  static constexpr int kBytes = kBar + 64 + 1024;      // + alignment slack for the 1024-byte atoms
  static_assert(kQLo % 1024 == 0 && kKLo % 1024 == 0 && kVLo % 1024 == 0 && kPLo % 1024 == 0, "atom alignment");
  static_assert(kBytes <= 232448, "shared memory per CTA");
};

// Instruction descriptor of tcgen05.mma kind::tf32: fp32 accumulator, tf32 A and B, both
// K-major, M x N tile (same field positions as kind::f16; operand format 2 = tf32).
constexpr uint32_t idesc_tf32_f32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Byte offset of element (row r, k) of a K-major fp32 operand with `rows` rows: 32-element
// column block k/32 (rows * 128 bytes each), row r, 16-byte chunk (k % 32) / 4 at position
// chunk ^ (r % 8) of the row (the 128-byte swizzle), word k % 4.
__device__ __forceinline__ uint32_t sw_off(int rows, int r, int k) {
  return (uint32_t)((k >> 5) * rows * 128 + r * 128 + ((((k >> 2) & 7) ^ (r & 7)) << 4) + (k & 3) * 4);
}

// x = hi + lo with hi exact in tf32 (the low 13 of the 23 mantissa bits cleared); lo = x - hi
// is exact in fp32 (0 for 0, inf and nan inputs never reach here: masked tokens hold zeros)
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }

__device__ __forceinline__ void st_shared_v4(uint32_t a, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_shared_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
// store x's hi part at a and its lo part at a + lo_off
__device__ __forceinline__ void st_split_v4(uint32_t a, uint32_t lo_off, float4 x) {
  const float4 h = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
  st_shared_v4(a, h);
  st_shared_v4(a + lo_off, make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w));
}
__device__ __forceinline__ void st_split_f32(uint32_t a, uint32_t lo_off, float x) {
  const float h = tf32_hi(x);
  st_shared_f32(a, h);
  st_shared_f32(a + lo_off, x - h);
}

// D (+)= A B over k_steps K-steps of 8, as A_hi B_hi + A_hi B_lo + A_lo B_hi; A and B are
// K-major swizzled operands with a_rows / b_rows rows whose lo parts lie a_lo / b_lo bytes after
// their hi parts.  Issued by one thread.
__device__ __forceinline__ void mma_split(uint32_t d_tmem, uint32_t sa, int a_rows, uint32_t a_lo, uint32_t sb,
                                          int b_rows, uint32_t b_lo, int k_steps, uint32_t idesc, bool accumulate) {
  const uint32_t offs[3][2] = {{0u, 0u}, {0u, b_lo}, {a_lo, 0u}};
#pragma unroll
  for (int t = 0; t < 3; ++t)
    for (int kk = 0; kk < k_steps; ++kk) {
      const uint64_t a = smem_desc_sw128(sa + offs[t][0] + (kk >> 2) * (a_rows * 128) + (kk & 3) * 32, 16, 1024);
      const uint64_t b = smem_desc_sw128(sb + offs[t][1] + (kk >> 2) * (b_rows * 128) + (kk & 3) * 32, 16, 1024);
      umma_tf32(d_tmem, a, b, idesc, (accumulate || t > 0 || kk > 0) ? 1u : 0u);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) dense_tf32_kernel(AttnParams p, int32_t first_item) {
  using L = Tf32Layout<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base = (raw_u + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw_u);
  const uint32_t sQ = base + L::kQ, sK = base + L::kK, sV = base + L::kV, sP = base + L::kP;
  const uint32_t bar_s = base + L::kBar, bar_o = bar_s + 8, bar_drain = bar_s + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 24);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 32);

  const DevPrefixItem it = p.pitems[first_item + blockIdx.x];
  const DevGroup gr = p.groups[it.group];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int g = p.g, j = it.kv_head;
  const int32_t rows = gr.n_req * g;
  const int32_t row = it.row_block * kRows + tid;
  int32_t t0, t1;
  piece_range(gr, it.split, t0, t1);
  const int n_tiles = t1 > t0 ? (t1 - t0 + kTok - 1) / kTok : 0;
  if (gr.slab_off < 0 || gr.slab_off + gr.L_p > p.n_hot) {
    if (tid == 0) atomicCAS(p.err, 0, (int32_t)kDevBadSlab);
    return;
  }
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

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // this row of Q -> shared memory (rows past the group are 0)
  {
    const float4* qrow = row < rows ? reinterpret_cast<const float4*>(static_cast<const float*>(p.q) +
                                                                     ((int64_t)b * p.n_q + h) * D)
                                    : nullptr;
#pragma unroll 4
    for (int c = 0; c < D / 4; ++c)
      st_split_v4(sQ + sw_off(kRows, tid, 4 * c), L::kQLo, qrow ? qrow[c] : make_float4(0.f, 0.f, 0.f, 0.f));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_off = (uint32_t)((warp * 32) << 16);
  const float scale = p.scale_log2;
  const int64_t tok_stride = (int64_t)p.n_kv * D;
  const float* kslab = static_cast<const float*>(p.kpool) + (gr.slab_off + t0) * tok_stride + (int64_t)j * D;
  const float* vslab = static_cast<const float*>(p.vpool) + (gr.slab_off + t0) * tok_stride + (int64_t)j * D;

  float m = -INFINITY, l = 0.f;
  bool ok = true, issued = false;
  for (int i = 0; i < n_tiles; ++i) {
    const int valid = min(kTok, t1 - t0 - i * kTok);
    // stage K (threads 0-63) and V^T (threads 64-127): token row n = tid % 32, column half
    // (tid / 32) % 2 of it; rows past the piece are 0, so masked tokens hold finite values
    {
      const int n = tid & (kTok - 1);
      const int c0 = ((tid >> 5) & 1) * (D / 8);
      const bool in = n < valid;
      if (tid < 2 * kTok) {
        const float4* src = reinterpret_cast<const float4*>(kslab + (int64_t)(i * kTok + n) * tok_stride);
#pragma unroll 4
        for (int c = c0; c < c0 + D / 8; ++c)
          st_split_v4(sK + sw_off(kTok, n, 4 * c), L::kKLo, in ? src[c] : make_float4(0.f, 0.f, 0.f, 0.f));
      } else {
        const float4* src = reinterpret_cast<const float4*>(vslab + (int64_t)(i * kTok + n) * tok_stride);
#pragma unroll 4
        for (int c = c0; c < c0 + D / 8; ++c) {
          const float4 v = in ? src[c] : make_float4(0.f, 0.f, 0.f, 0.f);
          st_split_f32(sV + sw_off(D, 4 * c + 0, n), L::kVLo, v.x);
          st_split_f32(sV + sw_off(D, 4 * c + 1, n), L::kVLo, v.y);
          st_split_f32(sV + sw_off(D, 4 * c + 2, n), L::kVLo, v.z);
          st_split_f32(sV + sw_off(D, 4 * c + 3, n), L::kVLo, v.w);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();
    if (tid == 0) {
      mma_split(tmem, sQ, kRows, L::kQLo, sK, kTok, L::kKLo, D / 8, idesc_tf32_f32(kRows, kTok), false);
      umma_commit(bar_s);
      issued = true;
    }
    ok = mbar_wait_bounded(bar_s, i & 1, abort_flag, p.err, kDevTimeout, kWaitLimitNs);
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();

    // softmax of this thread's row over the tile
    uint32_t u[32];
    GRANIKV_TMEM_LD32(tmem + lane_off, u);
    tmem_wait_ld();
    float s[kTok];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < kTok; ++k) {
      s[k] = k < valid ? __uint_as_float(u[k]) : -INFINITY;
      mx = fmaxf(mx, s[k]);
    }
    const float m_new = fmaxf(m, mx * scale);
    const float alpha = m == -INFINITY ? 0.f : ex2_approx(m - m_new);
    float psum = 0.f;
#pragma unroll
    for (int c = 0; c < kTok / 4; ++c) {
      float4 pv;
      pv.x = ex2_approx(s[4 * c + 0] * scale - m_new);
      pv.y = ex2_approx(s[4 * c + 1] * scale - m_new);
      pv.z = ex2_approx(s[4 * c + 2] * scale - m_new);
      pv.w = ex2_approx(s[4 * c + 3] * scale - m_new);
      psum += (pv.x + pv.y) + (pv.z + pv.w);
      st_split_v4(sP + sw_off(kRows, tid, 4 * c), L::kPLo, pv);
    }
    l = l * alpha + psum;
    m = m_new;
    // O (complete up to the previous tile) follows the row's new max
    if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        GRANIKV_TMEM_LD32(tmem + lane_off + kColO + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
        GRANIKV_TMEM_ST32(tmem + lane_off + kColO + c * 32, o);
      }
      tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      mma_split(tmem + kColO, sP, kRows, L::kPLo, sV, D, L::kVLo, kTok / 8, idesc_tf32_f32(kRows, D), i > 0);
      umma_commit(bar_o);
    }
    ok = mbar_wait_bounded(bar_o, i & 1, abort_flag, p.err, kDevTimeout, kWaitLimitNs);
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();
  }

  if (ok) {
    // the record: o = O / l, lse = (m + log2 l) ln 2; a piece with no tokens leaves o = 0
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* dst = rec >= 0 ? p.rec_o + ((int64_t)rec * p.n_q + h) * D : nullptr;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      if (n_tiles > 0) {
        GRANIKV_TMEM_LD32(tmem + lane_off + kColO + c * 32, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = 0u;
      }
      if (dst) {
#pragma unroll
        for (int k = 0; k < 32; k += 4)
          *reinterpret_cast<float4*>(dst + c * 32 + k) =
              make_float4(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv,
                          __uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
      }
    }
    if (rec >= 0) p.rec_lse[(int64_t)rec * p.n_q + h] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
  }
  // teardown: every MMA this CTA issued completes before its TMEM is freed
  if (tid == 0 && issued && !ok) {
    umma_commit(bar_drain);
    const uint64_t t_start = globaltimer_ns();
    while (!mbar_try_wait(bar_drain, 0)) {
      if (globaltimer_ns() - t_start > kWaitLimitNs) {
        atomicCAS(p.err, 0, (int32_t)kDevTimeout);
        break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_tf32_d(const AttnParams& p, int32_t first_item, int32_t n_items, cudaStream_t s) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(dense_tf32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Tf32Layout<D>::kBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  return launch_kernel(dense_tf32_kernel<D>, dim3(n_items), dim3(kThreads), Tf32Layout<D>::kBytes, s, false, p,
                       first_item);
}

}  // namespace

cudaError_t launch_dense_tf32(const AttnParams& p, int32_t first_item, int32_t n_items, cudaStream_t s) {
  if (n_items <= 0) return cudaSuccess;
  switch (p.d) {
    case 32: return launch_tf32_d<32>(p, first_item, n_items, s);
    case 64: return launch_tf32_d<64>(p, first_item, n_items, s);
    case 96: return launch_tf32_d<96>(p, first_item, n_items, s);
    case 128: return launch_tf32_d<128>(p, first_item, n_items, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace granikv
