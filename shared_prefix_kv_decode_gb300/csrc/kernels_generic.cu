// kernels_generic.cu -- CUDA-core decode attention for any head_dim that is a multiple of 32
// (up to 256), fp32 or bf16: the prefix pass, the COLD suffix pass and the log-sum-exp merge.
//
// GraniKV (arXiv:2608.15584), "2 Related Work", prefix-suffix attention: the shared prefix
// and each request's suffix are attended separately and their partial states merged with
// log-sum-exp.  One warp owns one query row; each lane holds head_dim/32 consecutive elements
// of q and of the running output, the q.k dot product is reduced with warp shuffles, and the
// softmax is the usual online (running max, running sum) form in base 2.
//
// These kernels serve the fp32 path and every shape the tensor-core kernels do not cover.
#include "internal.h"
#include "launch_util.cuh"
#include "tc_util.cuh"

#include <cuda_bf16.h>

namespace granikv {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void latch(int32_t* err, int32_t code) { atomicCAS(err, 0, code); }

template <typename T, int VPL>
__device__ __forceinline__ void load_row(const T* p, float (&x)[VPL]);

template <int VPL>
__device__ __forceinline__ void load_row(const float* p, float (&x)[VPL]) {
#pragma unroll
  for (int i = 0; i < VPL; ++i) x[i] = p[i];
}

template <int VPL>
__device__ __forceinline__ void load_row(const __nv_bfloat16* p, float (&x)[VPL]) {
#pragma unroll
  for (int i = 0; i < VPL; ++i) x[i] = __bfloat162float(p[i]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Online softmax state of one query row, spread over a warp.
template <int VPL>
struct RowState {
  float m = -INFINITY;  // running max of the base-2 logits
  float l = 0.f;        // running sum of 2^(logit - m)
  float acc[VPL];
  __device__ RowState() {
#pragma unroll
    for (int i = 0; i < VPL; ++i) acc[i] = 0.f;
  }
  __device__ __forceinline__ void add(float s2, const float (&v)[VPL]) {
    const float m_new = fmaxf(m, s2);
    const float alpha = exp2f(m - m_new);
    const float p = exp2f(s2 - m_new);
    l = l * alpha + p;
#pragma unroll
    for (int i = 0; i < VPL; ++i) acc[i] = acc[i] * alpha + p * v[i];
    m = m_new;
  }
};

template <int VPL>
__device__ __forceinline__ void store_record(const AttnParams& p, const RowState<VPL>& st, int32_t rec,
                                             int32_t h, int lane) {
  if (p.checks && (rec < 0 || rec >= p.n_records)) {
    if (lane == 0) latch(p.err, kDevBadRecord);
    return;
  }
  float* dst = p.rec_o + ((int64_t)rec * p.n_q + h) * p.d + lane * VPL;
  const float inv = st.l > 0.f ? 1.f / st.l : 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) dst[i] = st.acc[i] * inv;
  if (lane == 0) p.rec_lse[(int64_t)rec * p.n_q + h] = st.l > 0.f ? (st.m + log2f(st.l)) * kLn2 : -INFINITY;
}

// Prefix pass: one CTA per prefix work item (group, KV head, row block, L_p piece).  The
// slab is contiguous, so token t of the piece is slot slab_off + t.
template <typename T, int VPL>
__global__ void __launch_bounds__(256) prefix_generic_kernel(AttnParams p, int32_t first_item) {
  const DevPrefixItem it = p.pitems[first_item + blockIdx.x];
  const DevGroup gr = p.groups[it.group];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t rows = gr.n_req * p.g;
  const int32_t r0 = it.row_block * gr.rows_per_cta;
  const int32_t r1 = min(rows, r0 + gr.rows_per_cta);
  int32_t t0, t1;
  piece_range(gr, it.split, t0, t1);
  if (p.checks && (gr.slab_off < 0 || gr.slab_off + gr.L_p > p.n_hot)) {
    if (threadIdx.x == 0) latch(p.err, kDevBadSlab);
    return;
  }
  const int64_t tok_stride = (int64_t)p.n_kv * p.d;
  const T* kbase = (const T*)p.kpool + gr.slab_off * tok_stride + (int64_t)it.kv_head * p.d + lane * VPL;
  const T* vbase = (const T*)p.vpool + gr.slab_off * tok_stride + (int64_t)it.kv_head * p.d + lane * VPL;
  for (int32_t r = r0 + warp; r < r1; r += blockDim.x >> 5) {
    const int32_t b = p.group_req[gr.req_begin + r / p.g];
    const int32_t h = it.kv_head * p.g + r % p.g;
    float q[VPL];
    load_row<VPL>((const T*)p.q + ((int64_t)b * p.n_q + h) * p.d + lane * VPL, q);
#pragma unroll
    for (int i = 0; i < VPL; ++i) q[i] *= p.scale_log2;
    RowState<VPL> st;
    for (int32_t t = t0; t < t1; ++t) {
      float k[VPL], v[VPL];
      load_row<VPL>(kbase + t * tok_stride, k);
      load_row<VPL>(vbase + t * tok_stride, v);
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < VPL; ++i) dot += q[i] * k[i];
      st.add(warp_sum(dot), v);
    }
    store_record<VPL>(p, st, p.reqs[b].rec_base + it.split, h, lane);
  }
}

// Suffix pass: one CTA per (request, token chunk) of its COLD token table; token t lives at
// slot req_to_slot[b, t].  Warps take the query heads in turn.
template <typename T, int VPL>
__global__ void __launch_bounds__(256) suffix_generic_kernel(AttnParams p) {
  DevSuffixItem it = p.sitems[blockIdx.x];
  if (p.live_len) it.t1 = max(it.t0, min(it.t1, p.live_len[it.b]));  // tokens that exist now
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tok_stride = (int64_t)p.n_kv * p.d;
  const int32_t* table = p.req_to_slot + (int64_t)it.b * p.cap;
  // fused COLD append: the request's newest token is read from k_new/v_new (row b), and the warp
  // of each KV head's first query head writes it to the token's slot; no CTA of this launch reads
  // that slot from the pool
  const int32_t newest = p.k_new ? (p.live_len ? p.live_len[it.b] : p.reqs[it.b].seq_len) - 1 : -1;
  for (int32_t h = warp; h < p.n_q; h += blockDim.x >> 5) {
    const int32_t j = h / p.g;
    float q[VPL];
    load_row<VPL>((const T*)p.q + ((int64_t)it.b * p.n_q + h) * p.d + lane * VPL, q);
#pragma unroll
    for (int i = 0; i < VPL; ++i) q[i] *= p.scale_log2;
    RowState<VPL> st;
    for (int32_t t = it.t0; t < it.t1; ++t) {
      const int32_t slot = table[t];
      if (slot < p.n_hot || slot >= p.n_slots) {
        if (lane == 0) latch(p.err, kDevBadSlot);
        continue;
      }
      T* kslot = static_cast<T*>(p.kpool) + slot * tok_stride + (int64_t)j * p.d;
      T* vslot = static_cast<T*>(p.vpool) + slot * tok_stride + (int64_t)j * p.d;
      const T* krow = kslot;
      const T* vrow = vslot;
      if (t == newest) {
        const T* kn = static_cast<const T*>(p.k_new) + (int64_t)it.b * tok_stride + (int64_t)j * p.d;
        const T* vn = static_cast<const T*>(p.v_new) + (int64_t)it.b * tok_stride + (int64_t)j * p.d;
        if (h % p.g == 0)
          for (int32_t i = lane; i < p.d; i += 32) {
            kslot[i] = kn[i];
            vslot[i] = vn[i];
          }
        krow = kn;
        vrow = vn;
      }
      float k[VPL], v[VPL];
      load_row<VPL>(krow + lane * VPL, k);
      load_row<VPL>(vrow + lane * VPL, v);
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < VPL; ++i) dot += q[i] * k[i];
      st.add(warp_sum(dot), v);
    }
    store_record<VPL>(p, st, it.rec, h, lane);
  }
}

template <typename T>
__device__ __forceinline__ void store_out(T* dst, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* dst, float v) { *dst = v; }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* dst, float v) {
  *dst = __float2bfloat16_rn(v);
}

// Merge: one warp per (request, head).  lse = M + ln sum_i e^(lse_i - M) and
// o = sum_i e^(lse_i - lse) o_i over the request's partial-state records; each lane owns
// head_dim/32 consecutive elements, so every record row is read with coalesced accesses, and
// the records loop is unrolled so several rows are in flight at once.
template <typename T, int VPL>
__global__ void __launch_bounds__(256) merge_kernel(AttnParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;  // b * n_q + h
  if (row >= (int64_t)p.B * p.n_q) return;
  const int32_t b = (int32_t)(row / p.n_q);
  const int32_t h = (int32_t)(row % p.n_q);
  const DevReq r = p.reqs[b];
  const float* lse_rec = p.rec_lse + (int64_t)r.rec_base * p.n_q + h;
  float M = -INFINITY;
  for (int32_t i = lane; i < r.n_parts; i += 32) M = fmaxf(M, lse_rec[(int64_t)i * p.n_q]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  T* dst = (T*)p.o + row * p.d + lane * VPL;
  if (M == -INFINITY) {  // no tokens at all (only reachable after a latched device check)
#pragma unroll
    for (int k = 0; k < VPL; ++k) store_out<T>(dst + k, 0.f);
    if (lane == 0) p.lse[row] = -INFINITY;
    return;
  }
  float tot = 0.f;
  for (int32_t i = lane; i < r.n_parts; i += 32) tot += exp2f((lse_rec[(int64_t)i * p.n_q] - M) * kLog2e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float lse = M + logf(tot);
  float acc[VPL];
#pragma unroll
  for (int k = 0; k < VPL; ++k) acc[k] = 0.f;
  const float* orec = p.rec_o + ((int64_t)r.rec_base * p.n_q + h) * p.d + lane * VPL;
  const int64_t rec_stride = (int64_t)p.n_q * p.d;
  int32_t i = 0;
  for (; i + 4 <= r.n_parts; i += 4) {
    float w[4], x[4][VPL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      w[u] = exp2f((lse_rec[(int64_t)(i + u) * p.n_q] - lse) * kLog2e);
#pragma unroll
      for (int k = 0; k < VPL; ++k) x[u][k] = orec[(i + u) * rec_stride + k];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int k = 0; k < VPL; ++k) acc[k] += w[u] * x[u][k];
  }
  for (; i < r.n_parts; ++i) {
    const float w = exp2f((lse_rec[(int64_t)i * p.n_q] - lse) * kLog2e);
#pragma unroll
    for (int k = 0; k < VPL; ++k) acc[k] += w * orec[i * rec_stride + k];
  }
#pragma unroll
  for (int k = 0; k < VPL; ++k) store_out<T>(dst + k, acc[k]);
  if (lane == 0) p.lse[row] = lse;
}

template <typename T, int VPL>
cudaError_t launch_prefix_vpl(const AttnParams& p, int32_t first, int32_t n, cudaStream_t s) {
  prefix_generic_kernel<T, VPL><<<n, 256, 0, s>>>(p, first);
  return cudaGetLastError();
}

template <typename T, int VPL>
cudaError_t launch_suffix_vpl(const AttnParams& p, cudaStream_t s) {
  suffix_generic_kernel<T, VPL><<<p.n_sitems, 256, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefix_t(const AttnParams& p, int32_t first, int32_t n, cudaStream_t s) {
  switch (p.d / 32) {
    case 1: return launch_prefix_vpl<T, 1>(p, first, n, s);
    case 2: return launch_prefix_vpl<T, 2>(p, first, n, s);
    case 3: return launch_prefix_vpl<T, 3>(p, first, n, s);
    case 4: return launch_prefix_vpl<T, 4>(p, first, n, s);
    case 5: return launch_prefix_vpl<T, 5>(p, first, n, s);
    case 6: return launch_prefix_vpl<T, 6>(p, first, n, s);
    case 7: return launch_prefix_vpl<T, 7>(p, first, n, s);
    case 8: return launch_prefix_vpl<T, 8>(p, first, n, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_suffix_t(const AttnParams& p, cudaStream_t s) {
  switch (p.d / 32) {
    case 1: return launch_suffix_vpl<T, 1>(p, s);
    case 2: return launch_suffix_vpl<T, 2>(p, s);
    case 3: return launch_suffix_vpl<T, 3>(p, s);
    case 4: return launch_suffix_vpl<T, 4>(p, s);
    case 5: return launch_suffix_vpl<T, 5>(p, s);
    case 6: return launch_suffix_vpl<T, 6>(p, s);
    case 7: return launch_suffix_vpl<T, 7>(p, s);
    case 8: return launch_suffix_vpl<T, 8>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefix_generic(int32_t dtype, const AttnParams& p, int32_t first_item,
                                  int32_t n_items, cudaStream_t s) {
  if (n_items <= 0) return cudaSuccess;
  return dtype == 1 ? launch_prefix_t<__nv_bfloat16>(p, first_item, n_items, s)
                    : launch_prefix_t<float>(p, first_item, n_items, s);
}

cudaError_t launch_suffix_generic(int32_t dtype, const AttnParams& p, cudaStream_t s) {
  if (p.n_sitems <= 0) return cudaSuccess;
  return dtype == 1 ? launch_suffix_t<__nv_bfloat16>(p, s) : launch_suffix_t<float>(p, s);
}

// bf16, head_dim 128: W warps per (request, head) row (W = 1, 2, 4 or 8), lane owns 4
// elements.  Warp w of a row takes the row's records w, w + W, w + 2W, ... in one pass with a
// running log-sum-exp, 8, 8, 16 or 24 records' loads in flight at a time (W = 1, 2, 4, 8); the W
// partial states are then combined in shared memory, in warp order, by the row's first warp.  A
// row of the one-grid split has five to nine records (one memory round trip); a cascade step
// over all SMs has one record per L_p piece, up to ~150, which W = 8 also covers in one.
// Records are read with streaming loads (they are not read again).  Two CTAs per SM (at most 128
// registers per thread): with programmatic dependent launch the CTAs become resident as the
// decode CTAs leave, spread over about 128 SMs rather than packed four to an SM on the first
// ones freed, which measured 1.5-2 us shorter from the release to the end.  A one-warp merge
// with more rows than two CTAs an SM hold at once (more than one wave) takes a build limited to
// 64 registers, four CTAs an SM, six records a batch: Qwen-2.5 shape (5,120 rows) 83.0 -> 82.4
// us a call with three CTAs an SM (80 registers), 80.8 -> 80.4 us more with four; eight prefixes
// 107.5 -> 106.8 -> 106.9 us; with one wave the two-CTA build stays (the headline's 2,048 rows:
// 38.7 against 39.2 us with three CTAs an SM).
// Records per warp loaded together: one memory round trip for rows of up to W * kBatch records.
template <int W>
struct MergeCfg {
  static constexpr int kBatch = W >= 8 ? 24 : W >= 4 ? 16 : 8;
  static constexpr int kMinBlocks = W >= 4 ? 1 : 2;  // registers for the larger batches
};

template <int W, int kBlocks = MergeCfg<W>::kMinBlocks>
__global__ void __launch_bounds__(256, kBlocks) merge_bf16_d128_kernel(AttnParams p) {
  constexpr int kMergeBatch = kBlocks >= 4 ? 6 : MergeCfg<W>::kBatch;  // 64 registers at four CTAs an SM
  constexpr int kRowsPerCta = 8 / W;
  __shared__ float4 s_acc[W > 1 ? 8 : 1][32];
  __shared__ float s_m[W > 1 ? 8 : 1], s_den[W > 1 ? 8 : 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = warp % W;
  const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + warp / W;  // b * n_q + h
  const bool have = row < (int64_t)p.B * p.n_q;
  DevReq r{0, 0, 0, 0};
  int32_t h = 0;
  if (have) {
    const int32_t b = (int32_t)(row / p.n_q);
    h = (int32_t)(row % p.n_q);
    r = p.reqs[b];  // the plan: written before the kernels of the call
  }
  grid_dep_wait();  // the records are complete once the kernels before this one are
  grid_dep_launch_dependents();
  const float* lse_rec = p.rec_lse + (int64_t)r.rec_base * p.n_q + h;
  const float4* orec = reinterpret_cast<const float4*>(p.rec_o + ((int64_t)r.rec_base * p.n_q + h) * 128) + lane;
  const int64_t lstride = (int64_t)p.n_q * W;
  const int64_t ostride = (int64_t)p.n_q * 32 * W;  // float4s between this warp's consecutive records
  lse_rec += (int64_t)part * p.n_q;
  orec += (int64_t)part * p.n_q * 32;
  const int32_t n_mine = have && r.n_parts > part ? (r.n_parts - part + W - 1) / W : 0;
  float m = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int32_t i = 0; i < n_mine; i += kMergeBatch) {
    float l[kMergeBatch];
    float4 x[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const bool ok = i + u < n_mine;
      l[u] = ok ? __ldcs(lse_rec + (i + u) * lstride) : -INFINITY;
      x[u] = ok ? __ldcs(orec + (i + u) * ostride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mb = m;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) mb = fmaxf(mb, l[u]);
    if (mb == -INFINITY) continue;
    const float a = ex2_approx((m - mb) * kLog2e);  // 0 while m is still -inf
    den *= a;
    acc.x *= a;
    acc.y *= a;
    acc.z *= a;
    acc.w *= a;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const float w = ex2_approx((l[u] - mb) * kLog2e);  // 0 for absent records
      den += w;
      acc.x += w * x[u].x;
      acc.y += w * x[u].y;
      acc.z += w * x[u].z;
      acc.w += w * x[u].w;
    }
    m = mb;
  }
  if constexpr (W > 1) {
    s_acc[warp][lane] = acc;
    if (lane == 0) {
      s_m[warp] = m;
      s_den[warp] = den;
    }
    __syncthreads();
    if (part != 0) return;
    float M = m;
#pragma unroll
    for (int q = 1; q < W; ++q) M = fmaxf(M, s_m[warp + q]);
    if (M != -INFINITY) {
      const float a0 = ex2_approx((m - M) * kLog2e);
      den *= a0;
      acc.x *= a0;
      acc.y *= a0;
      acc.z *= a0;
      acc.w *= a0;
#pragma unroll
      for (int q = 1; q < W; ++q) {
        const float a = ex2_approx((s_m[warp + q] - M) * kLog2e);  // 0 for a warp without records
        const float4 y = s_acc[warp + q][lane];
        den += a * s_den[warp + q];
        acc.x += a * y.x;
        acc.y += a * y.y;
        acc.z += a * y.z;
        acc.w += a * y.w;
      }
    }
    m = M;
  }
  if (!have) return;
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + row * 128)[lane] =
      make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  if (lane == 0) p.lse[row] = den > 0.f ? m + logf(den) : -INFINITY;
}

template <int W>
cudaError_t launch_merge_w(const AttnParams& p, cudaStream_t s, bool pdl) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = prefer_max_shared(merge_bf16_d128_kernel<W>);
    if (e == cudaSuccess && W == 1) e = prefer_max_shared(merge_bf16_d128_kernel<1, 4>);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int64_t rows = (int64_t)p.B * p.n_q;
  const int64_t per_cta = 8 / W;
  const dim3 grid((unsigned)((rows + per_cta - 1) / per_cta));
  if constexpr (W == 1) {
    int dev = 0, num_sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        (int64_t)grid.x > 2LL * num_sms)
      return launch_kernel(merge_bf16_d128_kernel<1, 4>, grid, dim3(256), 0, s, pdl, p);
  }
  return launch_kernel(merge_bf16_d128_kernel<W>, grid, dim3(256), 0, s, pdl, p);
}

template <typename T, int VPL>
cudaError_t launch_merge_vpl(const AttnParams& p, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.n_q;
  const int grid = (int)((rows + 7) / 8);
  merge_kernel<T, VPL><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_merge_t(const AttnParams& p, cudaStream_t s) {
  switch (p.d / 32) {
    case 1: return launch_merge_vpl<T, 1>(p, s);
    case 2: return launch_merge_vpl<T, 2>(p, s);
    case 3: return launch_merge_vpl<T, 3>(p, s);
    case 4: return launch_merge_vpl<T, 4>(p, s);
    case 5: return launch_merge_vpl<T, 5>(p, s);
    case 6: return launch_merge_vpl<T, 6>(p, s);
    case 7: return launch_merge_vpl<T, 7>(p, s);
    case 8: return launch_merge_vpl<T, 8>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_merge(int32_t dtype, const AttnParams& p, cudaStream_t s, bool pdl) {
  if (dtype == 1 && p.d == 128) return launch_merge_w<1>(p, s, pdl);
  return dtype == 1 ? launch_merge_t<__nv_bfloat16>(p, s) : launch_merge_t<float>(p, s);
}

cudaError_t launch_merge_rows(const AttnParams& p, int32_t warps_per_row, cudaStream_t s, bool pdl) {
  switch (warps_per_row) {
    case 1: return launch_merge_w<1>(p, s, pdl);
    case 2: return launch_merge_w<2>(p, s, pdl);
    case 4: return launch_merge_w<4>(p, s, pdl);
    case 8: return launch_merge_w<8>(p, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace granikv
