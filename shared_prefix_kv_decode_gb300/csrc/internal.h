// internal.h -- shared between the host library and the CUDA kernels of libgranikv.
//
// The per-step plan built by the dispatcher is a flat image of the structs below.  The host
// builds it, granikv_decode_attention copies it into the front of the caller's workspace, and
// the kernels read their work items from there.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace granikv {

// Error codes latched in the device error word (first failure wins).
enum DevErr : int32_t {
  kDevOk = 0,
  kDevBadSlot = 1,        // a COLD slot id outside [n_hot, n_slots)
  kDevTableOverflow = 2,  // a token table row would pass cap
  kDevBadSlab = 3,        // a slab range outside [0, n_hot)
  kDevBadRecord = 4,      // a partial-state record index outside the workspace
  kDevSmemAlign = 5,      // a kernel's dynamic shared memory was not aligned as its layout needs
  kDevTimeout = 6,        // a bounded mbarrier wait expired (the CTA drained and gave up)
  kDevColdEmpty = 7,      // a device-side COLD allocation found fewer free slots than asked
};

// Kernel implementations a prefix group or the suffix pass can run on.
enum Impl : int32_t {
  kImplGeneric = 0,   // CUDA-core kernel, any head_dim % 32 == 0 up to 256, f32 or bf16
  kImplCascadeMma = 1,// bf16, head_dim 128: warp-level tensor-core cascade kernel
  kImplDenseTc = 2,   // bf16, head_dim 128: tcgen05/TMEM dense kernel
  kImplSuffixMma = 3, // bf16, head_dim 128, g <= 8: warp-level tensor-core suffix kernel
  kImplCascadeStream = 4,  // bf16, head_dim 128, g <= 128: cascade over whole 2 KB slot rows
  kImplDenseTf32 = 5,      // f32, head_dim % 32 == 0 up to 128: tcgen05 kind::tf32 dense kernel
};

// Geometry of each prefix kernel: query rows per CTA and tokens per tile.  The planner and the
// kernels both use these.
constexpr int kGenericRows = 16, kGenericTile = 32;
constexpr int kCascadeRows = 128, kCascadeTile = 64;
constexpr int kDenseRows = 128, kDenseTile = 128;
constexpr int kDenseTf32Rows = 128, kDenseTf32Tile = 32;
// The streaming cascade kernel: eight consumer warps, each over 16-token sub-tiles and at most 16
// query columns (request, head-in-group pairs) of one KV head; with `sub` warps per KV head a
// CTA covers 8 / sub KV heads and 16 * sub columns of each.
constexpr int kCascadeStreamTile = 16, kCascadeStreamCols = 16, kCascadeStreamWarps = 8;
// Largest number of COLD tokens one suffix CTA streams (its slot ids are staged in shared memory).
constexpr int kSuffixMaxCtaTokens = 4096;

struct DevGroup {        // one prefix group: the requests sharing one HOT slab
  int64_t slab_off;      // first slot of the slab
  int32_t L_p;
  int32_t n_req;
  int32_t req_begin;     // index into the group_req array
  int32_t n_splits;      // pieces along L_p
  int32_t split_len;     // tokens of a short piece (a multiple of `tile`)
  int32_t backend;       // GRANIKV_BACKEND_DENSE / _CASCADE
  int32_t impl;          // Impl
  int32_t rows_per_cta;  // query rows (request, head-in-group) pairs per CTA
  int32_t row_blocks;    // ceil(n_req * g / rows_per_cta)
  int32_t n_long;        // the first n_long pieces are one tile longer than split_len
  int32_t tile;          // token granularity of the pieces
  int32_t q_b0;          // dense: the group's requests are q_b0, q_b0+1, ... (q rows by TMA), else -1
  int32_t causal;        // dense prefill of the slab's own tokens: request b of the group is token b
                         // of the slab and attends keys [0, b] (0 for decode groups)
  int32_t sub;           // streaming cascade: consumer warps per KV head (1, 2, 4, 8), else 0
};
static_assert(sizeof(DevGroup) == 64, "DevGroup layout");

// Token range [t0, t1) of piece `split` of a group's prefix: pieces of split_len or
// split_len + tile tokens (the longer ones first), clipped to L_p.
__host__ __device__ inline void piece_range(const DevGroup& g, int32_t split, int32_t& t0, int32_t& t1) {
  const int32_t lo = split < g.n_long ? split : g.n_long;
  t0 = split * g.split_len + lo * g.tile;
  const int32_t len = g.split_len + (split < g.n_long ? g.tile : 0);
  t1 = t0 + len < g.L_p ? t0 + len : g.L_p;
}

struct DevReq {          // per request of the batch
  int32_t rec_base;      // first partial-state record of this request
  int32_t n_prefix;      // records written by the prefix pass (0 without a HOT prefix)
  int32_t n_parts;       // records in total (prefix pieces + suffix chunks)
  int32_t seq_len;       // tokens in the COLD token table
};

struct DevPrefixItem {   // one CTA of a prefix kernel
  int32_t group, kv_head, row_block, split;  // the streaming cascade kernel: kv_head is the index of
                                             // a group of eight KV heads, row_block a column chunk
};

struct DevSuffixItem {   // one CTA of a suffix kernel
  int32_t b, t0, t1, rec;  // request, token range [t0, t1) of its COLD table, record index
};

// Everything an attention kernel needs, passed by value.
struct AttnParams {
  const void* q;          // [B, n_q, d]
  void* o;                // [B, n_q, d]
  float* lse;             // [B, n_q]
  void* kpool;            // [n_slots, n_kv, d]; written only by the fused COLD append
  void* vpool;
  const int32_t* req_to_slot;  // [B, cap]
  int64_t n_slots, n_hot;
  int32_t cap, B, n_q, n_kv, d, g;
  float scale_log2;       // softmax scale * log2(e)
  const DevGroup* groups;
  const int32_t* group_req;
  const DevReq* reqs;
  const DevPrefixItem* pitems;
  int32_t n_pitems;
  const DevSuffixItem* sitems;
  int32_t n_sitems;
  const int32_t* scta_begin;  // [n_scta + 1]: first suffix item of each suffix token-CTA
  int32_t n_scta;
  float* rec_o;           // [n_records, n_q, d]
  float* rec_lse;         // [n_records, n_q]
  int32_t n_records;
  int32_t* err;           // device error word
  int32_t checks;
  int32_t* tickets;       // [B, n_q] arrivals per row (fused merge), zero between calls
  int32_t fused_merge;    // 1: the last producer of a row merges it (no merge kernel)
  int32_t q_tma;          // 1: the q tensor map passed to the dense kernel is valid
  int32_t l2_ahead;       // dense kernel: K/V tiles requested into L2 ahead of its ring (0: none)
  int32_t inject_stall;   // test hook: suffix token-CTA 0 withholds its first tile (see header)
  const void* k_new;        // [B, n_kv, d] or NULL: K of each request's last COLD token, read from
  const void* v_new;        // here (not the pool) and written to its slot by the suffix CTA
  const int32_t* live_len;  // [B] device token counts that end each request's suffix segments early
                            // (the plan may cover more tokens than exist yet); NULL: the plan's
};

// ---- launchers (kernels_*.cu) ------------------------------------------------------------
// `pdl`: launch as a programmatic dependent of the previous kernel in the stream (see
// launch_util.cuh); only for a kernel whose stream predecessor is a kernel of this library.
cudaError_t launch_cold_alloc(const int32_t* excl /*[B+1]*/, int32_t B, const int32_t* ring, int64_t n_cold,
                              int64_t head, int32_t* req_to_slot, int32_t* suffix_len, int32_t cap,
                              int32_t* slots_out, int64_t* ring_pos, int32_t* err, cudaStream_t s);
// n slots for each of requests 0..B-1, the ring position read from and written back to
// ring_pos[0..1] (head, tail) on the device, the free count checked there (one block).
cudaError_t launch_cold_alloc_uniform(int32_t n, int32_t B, const int32_t* ring, int64_t n_cold, int32_t* req_to_slot,
                                      int32_t* suffix_len, int32_t cap, int32_t* slots_out, int64_t* ring_pos,
                                      int32_t* err, cudaStream_t s);
cudaError_t launch_cold_free(const int32_t* slots, int32_t n, int32_t* ring, int64_t n_cold,
                             int64_t tail, int64_t n_hot, int64_t n_slots, int32_t checks,
                             int64_t* ring_pos, int32_t* err, cudaStream_t s);
cudaError_t launch_cold_append(int32_t dtype, const void* k_new, const void* v_new,
                               const int32_t* slots, int32_t N, void* kpool, void* vpool,
                               int64_t row_elems, int64_t n_hot, int64_t n_slots,
                               int32_t checks, int32_t* err, cudaStream_t s);

cudaError_t launch_prefix_generic(int32_t dtype, const AttnParams& p, int32_t first_item,
                                  int32_t n_items, cudaStream_t s);
cudaError_t launch_suffix_generic(int32_t dtype, const AttnParams& p, cudaStream_t s);
cudaError_t launch_merge(int32_t dtype, const AttnParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_suffix_mma(const AttnParams& p, const int32_t* cta_begin, int32_t n_cta, cudaStream_t s,
                              bool pdl);
cudaError_t launch_cascade_mma(const AttnParams& p, int32_t first_item, int32_t n_items, cudaStream_t s);
cudaError_t launch_dense_tc(const AttnParams& p, int32_t first_item, int32_t n_items, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, const CUtensorMap& tmq, cudaStream_t s, bool pdl);
cudaError_t launch_cascade_stream(const AttnParams& p, int32_t first_item, int32_t n_items, cudaStream_t s, bool pdl);
// fp32 dense prefix items on the tcgen05 tensor cores (kind::tf32); head_dim 32, 64, 96 or 128.
cudaError_t launch_dense_tf32(const AttnParams& p, int32_t first_item, int32_t n_items, cudaStream_t s);
// One launch for the prefix and suffix work: CTAs [0, n_dense) run dense prefix items
// first_dense.., the next n_casc the streaming cascade items first_casc.., the rest the suffix
// token-CTAs (n_scta per KV-head group of eight); dense CTA c < n_tail then runs suffix
// token-CTA n_scta + c of a plan with one KV-head group.
cudaError_t launch_prefix_suffix_tc(const AttnParams& p, int32_t first_dense, int32_t n_dense, int32_t first_casc,
                                    int32_t n_casc, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                    const CUtensorMap& tmq, const int32_t* cta_begin, int32_t n_scta, int32_t n_tail,
                                    cudaStream_t s, bool pdl);
// The merge kernel, bf16 and head_dim 128, with `warps_per_row` warps (1, 2, 4 or 8) sharing
// each row's records.
cudaError_t launch_merge_rows(const AttnParams& p, int32_t warps_per_row, cudaStream_t s, bool pdl);

constexpr int kNumImpl = 6;

}  // namespace granikv

struct granikv_ctx;
struct granikv_plan;

namespace granikv {
// Host-side helpers shared between the library's translation units (not part of the C ABI).
int32_t granikv_internal_device(const granikv_ctx* ctx, int* device);        // a granikv_status
// Drop the record of which plan image a workspace holds, so the next decode call on it copies
// its work list in again (and zeroes its merge tickets).
void granikv_internal_forget_workspace(const void* ws);
// HOT pool as it would be if the live slabs slabs[0..n) were released as well (nothing is
// changed): the largest free extent, and the number of unused slab ids.
void granikv_internal_hot_if_released(const granikv_ctx* ctx, const int32_t* slabs, int32_t n,
                                      int64_t* largest_free, int32_t* free_ids);

}  // namespace granikv
