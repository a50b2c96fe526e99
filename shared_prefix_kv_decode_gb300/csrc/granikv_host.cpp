// granikv_host.cpp -- host side of libgranikv: context, HOT first-fit pool, COLD ring
// bookkeeping, the per-step dispatcher and planner, and the C ABI entry points.
//
// GraniKV (arXiv:2608.15584): "3 GraniKV" (asymmetric HOT/COLD paging, dual backends,
// per-step dispatch), "B.8 Multi-prefix sensitivity" (first-fit packing, class-local dense
// batching), "B.10 Cross-pool admission and promotion policy" (HOT first, COLD fallback, no
// demotion).
#include "../../include/granikv.h"
#include "internal.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

using namespace granikv;

namespace {

constexpr int32_t kDefaultMaxSlabs = 1024;
constexpr int32_t kDefaultMaxBatch = 4096;
// Dense/cascade crossover on GB300 for the Llama-3.1-8B shape, re-fitted from the L_p x B
// sweep of msat_fit.py, recorded in msat_gb300.json next to this package (the pages' A100 value
// is 1024 and they state other GPUs need a re-fit).  The least-regret fit lands on the sweep's
// smallest M_eff (4): the tcgen05 dense kernel is the faster backend in all but one cell, and
// there the streaming cascade kernel wins by 1 % (0.13 us; the strict rule, dense no slower in
// every cell from M_sat up, therefore reads 32).  The cascade comes within 1-8 %
// at M_eff <= 32 (both are bandwidth-bound there) and falls far behind above, where its
// warp-level MMAs run out of throughput.
constexpr int32_t kDefaultMsat = 4;

struct Extent {
  int64_t off, len;
};
struct Slab {
  int64_t off = 0;
  int32_t len = 0;
  bool live = false;
};

}  // namespace

struct granikv_ctx {
  granikv_config cfg{};
  std::vector<void*> kpool, vpool;
  int64_t n_hot = 0, n_cold = 0;
  int32_t g = 1;
  // HOT pool: free extents sorted by offset, slab table
  std::vector<Extent> free_ext;
  std::vector<Slab> slabs;
  // COLD ring: entries [head, tail) are free; positions are taken modulo n_cold
  int64_t head = 0, tail = 0;
  // device resources
  int32_t* d_ring = nullptr;
  int32_t* d_err = nullptr;
  int32_t* d_stage = nullptr;  // [max_batch + 1] exclusive offsets for cold_alloc
  int64_t* d_ring_pos = nullptr;  // {head, tail} of the COLD ring on the device (absolute counts)
  int32_t num_sms = 152;
  int32_t cc_major = 0, cc_minor = 0;
  // dispatch state
  int32_t m_sat = kDefaultMsat;
  int32_t forced = GRANIKV_BACKEND_AUTO;
  int32_t checks = 1;
  granikv_plan* own_plan = nullptr;
  // enqueued work, for attribution
  int64_t n_kernels = 0, n_copies = 0;
  // prefix/suffix concurrency: an auxiliary stream forked from / joined into the caller's
  cudaStream_t aux = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  int32_t concurrent = 1;
  float prefix_share = 0.0f;  // 0: automatic
  int32_t inject_stall = 0;   // test hook for the next decode call
  int32_t fused_merge = 0;  // merge by the last producer instead of a merge kernel
  int32_t l2_ahead = -1;    // dense kernel's L2 read-ahead in tiles; -1: chosen per step
  // tickets of the last call (zeroed again after a device check failure)
  void* last_tickets = nullptr;
  size_t last_tickets_bytes = 0;
  std::vector<unsigned char> prefill_blob;  // host image of the last prefill call's plan
  // TMA descriptors of each layer's K and V pools (dense backend), valid when has_tmaps
  std::vector<CUtensorMap> tmap_k, tmap_v;
  bool has_tmaps = false;
};

struct granikv_plan {
  granikv_ctx* ctx = nullptr;
  std::vector<unsigned char> blob;  // device image of the plan
  size_t off_groups = 0, off_group_req = 0, off_req = 0, off_pitems = 0, off_sitems = 0, off_scta = 0;
  int32_t n_groups = 0, n_pitems = 0, n_sitems = 0, n_scta = 0, B = 0, n_records = 0;
  int64_t n_prefix_records = 0;
  bool fused = false;       // the last producer of a row merges it (no merge kernel)
  bool concurrent = false;  // suffix kernel on the auxiliary stream next to the prefix kernel
  int32_t suffix_impl = kImplGeneric;
  int32_t merge_warps = 1;  // warps of the merge kernel per (request, head) row
  int32_t l2_ahead = 0;     // dense kernel's L2 read-ahead in tiles
  int32_t n_tail = 0;       // suffix runs (the last of n_scta) taken by the one grid's dense CTAs
  int32_t pitem_first[kNumImpl] = {};  // prefix items are ordered by implementation
  int32_t pitem_count[kNumImpl] = {};
  std::vector<granikv_group_info> info;
  std::vector<int32_t> group_impl;
  uint64_t uid = 0;      // unique over the process (never reused), so a workspace record can name it
  uint64_t version = 0;  // bumped by every dispatch into this plan
  bool valid = false;
  // granikv_dispatch's working arrays, kept with the plan so that the dispatches of a serving
  // loop reuse their capacity instead of allocating each step
  struct Scratch {
    std::vector<int32_t> slot_of_slab;  // slab id -> group, -1 between dispatches
    std::vector<int32_t> grp_slab, grp_count, req_group, begin, group_req, fill, scta_begin;
    std::vector<DevGroup> groups;
    std::vector<DevPrefixItem> pitems;
    std::vector<int32_t> grp_np;          // prefix records of a request by its group + 1
    // What the last successful dispatch derived from the batch's slab ids alone (the groups,
    // their members, whether each group's requests are consecutive) and from the groups' shapes
    // alone (the prefix work items): a serving loop re-dispatches the same requests step after
    // step with only their lengths grown, and then rebuilds neither.
    bool groups_cached = false;
    std::vector<int32_t> cache_slab_id;   // the batch's slab ids
    std::vector<Slab> cache_slab;         // each group's slab (offset, length) when cached
    std::vector<char> grp_contig;         // group's requests consecutive in the batch
    bool pitems_cached = false;
    std::vector<int32_t> pitems_key;      // the group fields the prefix items depend on
    // The serial dense schedule's choice of piece length (see the planner), memoised on the
    // groups' tile counts: tail_key -> tail_len (0: the balanced one-wave pieces).
    std::vector<int64_t> tail_key, tail_key_now, sim_heap;
    int64_t tail_len = 0;
    std::vector<char> grp_tail;           // group's last piece is a shorter remainder
  } scratch;
};

namespace {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int elem_size(int32_t dtype) { return dtype == GRANIKV_DTYPE_BF16 ? 2 : 4; }

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

granikv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GRANIKV_OK : GRANIKV_ERR_CUDA; }

bool has_device(const granikv_ctx* c) { return c && !c->cfg.host_only && c->d_ring; }

// Which prefix implementation serves a group of this shape and backend.
int32_t prefix_impl_for(const granikv_ctx* c, int32_t backend) {
  if (c->cfg.dtype == GRANIKV_DTYPE_BF16 && c->cfg.head_dim == 128) {
    if (backend == GRANIKV_BACKEND_DENSE && (c->has_tmaps || c->cfg.host_only)) return kImplDenseTc;
    if (c->g <= kCascadeStreamCols * kCascadeStreamWarps) return kImplCascadeStream;
    return kImplCascadeMma;
  }
  if (c->cfg.dtype == GRANIKV_DTYPE_F32 && backend == GRANIKV_BACKEND_DENSE && c->cfg.head_dim % 32 == 0 &&
      c->cfg.head_dim <= 128)
    return kImplDenseTf32;
  return kImplGeneric;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// A pool [n_slots, n_kv, 128] bf16 as a 3-D tensor (dim, head, slot) with 64 x 1 x 64 boxes and
// the 128-byte swizzle the tcgen05 operand descriptors expect.
bool encode_pool_map(CUtensorMap* m, void* base, int64_t n_slots, int32_t n_kv) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)n_kv, (cuuint64_t)n_slots};
  cuuint64_t strides[2] = {256, (cuuint64_t)n_kv * 256};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kDenseTile};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// q [B, n_q, 128] bf16 as a 3-D tensor (dim, head, request) with (64, g, 128/g) boxes: one box
// is a dense row block's q rows of one 64-dim half, in the layout the operand descriptors expect.
bool encode_q_map(CUtensorMap* m, const void* q, int32_t B, int32_t n_q, int32_t g) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || ((uintptr_t)q % 16) != 0 || g < 1 || kDenseRows % g != 0) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)n_q, (cuuint64_t)B};
  cuuint64_t strides[2] = {256, (cuuint64_t)n_q * 256};
  cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)(kDenseRows / g)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Streaming cascade: consumer warps per KV head for a group of n_req requests, the fewest (so
// the most KV heads per CTA, whole 2 KB slot rows at one warp) whose 16 * sub query columns hold
// the group's columns, or at least one request's g columns.
int32_t stream_sub_for(int32_t n_req, int32_t g) {
  const int64_t cols = (int64_t)n_req * g;
  int32_t sub = 1;
  while (sub < kCascadeStreamWarps && ((int64_t)kCascadeStreamCols * sub < cols || kCascadeStreamCols * sub < g)) sub *= 2;
  return sub;
}

// Query rows (request, head-in-group pairs of one KV head) one CTA of a prefix kernel takes;
// the streaming cascade kernel takes whole requests, as many as fit its query columns.
int32_t rows_per_cta_for(int32_t impl, int32_t g, int32_t sub) {
  switch (impl) {
    case kImplDenseTc: return kDenseRows;
    case kImplDenseTf32: return kDenseTf32Rows;
    case kImplCascadeMma: return kCascadeRows;
    case kImplCascadeStream: return (kCascadeStreamCols * sub / g) * g;
    default: return kGenericRows;
  }
}

int32_t tile_tokens_for(int32_t impl, int32_t sub) {
  switch (impl) {
    case kImplDenseTc: return kDenseTile;
    case kImplDenseTf32: return kDenseTf32Tile;
    case kImplCascadeMma: return kCascadeTile;
    case kImplCascadeStream: return kCascadeStreamTile * sub;
    default: return kGenericTile;
  }
}

// KV heads one CTA of the streaming cascade kernel covers.
int32_t stream_heads(int32_t sub) { return kCascadeStreamWarps / sub; }

// CTAs of one L_p piece of a group: one per (KV head, row block), or for the streaming cascade
// kernel one per (group of 8 / sub KV heads, column chunk).
int64_t ctas_per_piece(const DevGroup& dg, int32_t n_kv) {
  if (dg.impl == kImplCascadeStream) {
    const int32_t hpc = stream_heads(dg.sub);
    return (int64_t)((n_kv + hpc - 1) / hpc) * dg.row_blocks;
  }
  return (int64_t)n_kv * dg.row_blocks;
}

// Which plan image each workspace holds at its front.  A decode call copies its plan's work list
// into the workspace only when the record for that address names another plan, another
// dispatch of the same plan, or nothing; whatever else writes a workspace's front (a prefill,
// an upload by another plan or context, the built-in static workspace's next user) replaces or
// drops the record.  Process-wide, since several contexts may share one buffer.  Bounded: the
// oldest records are dropped first, which only costs a re-upload.
struct WsRecord {
  const void* ws;
  uint64_t plan_uid;  // 0: the front holds no plan image (e.g. a prefill's)
  uint64_t version;
};
std::mutex g_ws_mutex;
std::vector<WsRecord> g_ws_records;
std::atomic<uint64_t> g_next_plan_uid{1};
constexpr size_t kMaxWsRecords = 64;

bool ws_holds(const void* ws, uint64_t uid, uint64_t version) {
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  for (const WsRecord& r : g_ws_records)
    if (r.ws == ws) return r.plan_uid == uid && r.version == version;
  return false;
}

void ws_record(const void* ws, uint64_t uid, uint64_t version) {
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  for (size_t i = 0; i < g_ws_records.size(); ++i)
    if (g_ws_records[i].ws == ws) {
      g_ws_records.erase(g_ws_records.begin() + i);
      break;
    }
  if (g_ws_records.size() >= kMaxWsRecords) g_ws_records.erase(g_ws_records.begin());
  g_ws_records.push_back({ws, uid, version});
}

void ws_forget(const void* ws) {
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  for (size_t i = 0; i < g_ws_records.size(); ++i)
    if (g_ws_records[i].ws == ws) {
      g_ws_records.erase(g_ws_records.begin() + i);
      return;
    }
}

// The suffix's COLD tokens are counted in 16-token tiles per request; a segment (one request's
// part of one token-CTA run) costs its CTA about one tile on top of its tiles.
constexpr int64_t kSTile = 16;
constexpr int64_t kSegTiles = 1;

struct SuffixCut {
  int32_t n_items = 0;         // suffix work items written
  int32_t max_parts = 0;       // most records of one request
  int64_t records = 0;         // records of the batch
  int64_t prefix_records = 0;  // of them, prefix records
};

// Cuts the concatenation of the B requests' COLD tiles into n_scta token-CTA runs, cuts falling
// on a request's tile boundaries.  U is the batch's tiles plus segment costs when every cut is
// counted as splitting a request (one more segment); the first n_scta - n_tail runs share
// U - U_tail, the last n_tail runs U_tail.  Each run's target is set when it starts, as an equal
// share of what is left: U less the units given out so far and less one for every cut so far
// that fell between two requests (it added no segment), so that short requests, which most cuts
// do not split, leave no run short at the end.  Writes every request's record layout
// (np_of[rg[b]] prefix records, then one per segment), one suffix item per segment and each
// run's first item (scta_begin[0..n_scta]).  Out of line so that its loop's counters stay in
// registers.
__attribute__((noinline)) SuffixCut cut_suffix_runs(int32_t B, const int32_t* __restrict__ np_of,
                                                    const int32_t* __restrict__ rg,
                                                    const int32_t* __restrict__ seq_len, int32_t n_scta,
                                                    int32_t n_tail, int64_t U, int64_t U_tail,
                                                    DevReq* __restrict__ reqs, DevSuffixItem* __restrict__ si,
                                                    int32_t* __restrict__ scta_begin) {
  const int32_t n_main = n_scta - n_tail;
  int32_t n_si = 0;
  int64_t rec = 0;
  int32_t cta = 0;
  int64_t done = 0;         // tiles plus segment costs given to the CTAs so far
  int64_t whole_cuts = 0;   // cuts so far that fell between two requests
  bool cta_open = false;    // the current CTA has a segment
  // where run k (starting now, at `done`) ends: one division per run, not per segment
  auto run_end = [&](int64_t k) {
    const int64_t left = U - done - whole_cuts;
    if (k < n_main) return done + (left - U_tail) / (n_main - k);
    return done + left / (n_scta - k);
  };
  int64_t end_cur = n_scta > 0 ? run_end(0) : 0;
  int32_t max_parts = 0;
  int64_t n_prefix_records = 0;
  for (int32_t b = 0; b < B; ++b) {
    DevReq& r = reqs[b];
    const int32_t n_prefix = np_of[rg[b]];
    const int32_t L = seq_len[b];
    r.rec_base = (int32_t)rec;
    r.n_prefix = n_prefix;
    r.seq_len = L;
    n_prefix_records += n_prefix;
    int32_t k = 0;
    const int64_t n_t = (L + kSTile - 1) / kSTile;
    // the common case: the whole request fits the current run with room to spare (the loop
    // below would take it in one segment and leave the run open)
    if (n_t > 0 && (cta >= n_scta - 1 || end_cur - done - kSegTiles > n_t)) {
      DevSuffixItem& it = si[n_si++];
      it.b = b;
      it.t0 = 0;
      it.t1 = L;
      it.rec = (int32_t)(rec + n_prefix);
      done += kSegTiles + n_t;
      cta_open = true;
      r.n_parts = n_prefix + 1;
      max_parts = std::max(max_parts, r.n_parts);
      rec += r.n_parts;
      continue;
    }
    for (int64_t t = 0; t < n_t;) {
      const bool last_cta = cta >= n_scta - 1;
      int64_t room = last_cta ? n_t - t : end_cur - done - kSegTiles;
      if (room <= 0 && cta_open) {
        // no tile more fits in this CTA: the request goes on in the next one
        ++cta;
        scta_begin[cta] = n_si;
        cta_open = false;
        whole_cuts += t == 0 ? 1 : 0;
        end_cur = run_end(cta);
        continue;
      }
      const int64_t take = std::min<int64_t>(n_t - t, std::max<int64_t>(room, 1));
      DevSuffixItem& it = si[n_si++];
      it.b = b;
      it.t0 = (int32_t)(t * kSTile);
      it.t1 = (int32_t)std::min<int64_t>((t + take) * kSTile, L);
      it.rec = (int32_t)(rec + n_prefix + k);
      ++k;
      t += take;
      done += kSegTiles + take;
      cta_open = true;
      if (!last_cta && done >= end_cur) {
        ++cta;
        scta_begin[cta] = n_si;
        cta_open = false;
        whole_cuts += t == n_t ? 1 : 0;
        end_cur = run_end(cta);
      }
    }
    r.n_parts = n_prefix + k;
    max_parts = std::max(max_parts, r.n_parts);
    rec += r.n_parts;
  }
  for (int32_t i = std::min(cta + 1, n_scta); i <= n_scta; ++i) scta_begin[i] = n_si;
  SuffixCut out;
  out.n_items = n_si;
  out.max_parts = max_parts;
  out.records = rec;
  out.prefix_records = n_prefix_records;
  return out;
}

}  // namespace

extern "C" {

const char* granikv_status_string(granikv_status s) {
  switch (s) {
    case GRANIKV_OK: return "ok";
    case GRANIKV_ERR_INVALID: return "invalid argument or descriptor";
    case GRANIKV_ERR_NO_HOT_SPACE: return "no HOT extent large enough (or slab table full)";
    case GRANIKV_ERR_NO_COLD_SPACE: return "not enough free COLD slots";
    case GRANIKV_ERR_CUDA: return "CUDA runtime error";
    case GRANIKV_ERR_DEVICE_CHECK: return "device bounds check failed";
    case GRANIKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case GRANIKV_ERR_NO_DEVICE: return "context has no device resources";
    case GRANIKV_ERR_STATIC_WORKSPACE_TOO_SMALL:
      return "the plan needs more workspace than the library's built-in 16 MiB array";
    default: return "unknown status";
  }
}

int32_t granikv_version(void) { return 100; }

granikv_status granikv_create(const granikv_config* cfg, granikv_ctx** out) {
  if (!cfg || !out) return GRANIKV_ERR_INVALID;
  *out = nullptr;
  if (cfg->n_layers <= 0 || cfg->n_q <= 0 || cfg->n_kv <= 0 || cfg->n_q % cfg->n_kv)
    return GRANIKV_ERR_INVALID;
  if (cfg->head_dim <= 0 || cfg->head_dim % 32 || cfg->head_dim > 256) return GRANIKV_ERR_UNSUPPORTED;
  if (cfg->dtype != GRANIKV_DTYPE_F32 && cfg->dtype != GRANIKV_DTYPE_BF16) return GRANIKV_ERR_INVALID;
  if (cfg->n_slots <= 1 || cfg->n_slots > (int64_t)INT32_MAX) return GRANIKV_ERR_INVALID;
  double fp = cfg->hot_fraction == 0.0 ? 0.2 : cfg->hot_fraction;
  if (!(fp > 0.0 && fp < 1.0)) return GRANIKV_ERR_INVALID;
  if (cfg->max_slabs < 0 || cfg->max_batch < 0 || cfg->m_sat < 0) return GRANIKV_ERR_INVALID;

  granikv_ctx* c = new (std::nothrow) granikv_ctx();
  if (!c) return GRANIKV_ERR_INVALID;
  c->cfg = *cfg;
  c->cfg.hot_fraction = fp;
  if (c->cfg.max_slabs == 0) c->cfg.max_slabs = kDefaultMaxSlabs;
  if (c->cfg.max_batch == 0) c->cfg.max_batch = kDefaultMaxBatch;
  c->m_sat = cfg->m_sat ? cfg->m_sat : kDefaultMsat;
  c->g = cfg->n_q / cfg->n_kv;
  c->n_hot = (int64_t)std::floor(fp * (double)cfg->n_slots);
  c->n_cold = cfg->n_slots - c->n_hot;
  if (c->n_hot < 0 || c->n_cold <= 0) {
    delete c;
    return GRANIKV_ERR_INVALID;
  }
  if (c->n_hot > 0) c->free_ext.push_back({0, c->n_hot});
  c->slabs.resize(c->cfg.max_slabs);
  c->head = 0;
  c->tail = c->n_cold;
  c->cfg.k_pool = nullptr;
  c->cfg.v_pool = nullptr;
  c->cfg.cold_init_order = nullptr;
  if (cfg->k_pool && cfg->v_pool) {
    c->kpool.assign(cfg->k_pool, cfg->k_pool + cfg->n_layers);
    c->vpool.assign(cfg->v_pool, cfg->v_pool + cfg->n_layers);
  }

  if (!cfg->host_only) {
    if (!cfg->k_pool || !cfg->v_pool) {
      delete c;
      return GRANIKV_ERR_INVALID;
    }
    // the tensor-core kernels move pool rows with bulk copies, which need 16-byte alignment
    for (int32_t l = 0; l < cfg->n_layers; ++l)
      if (((uintptr_t)cfg->k_pool[l] | (uintptr_t)cfg->v_pool[l]) % 16) {
        delete c;
        return GRANIKV_ERR_INVALID;
      }
    std::vector<int32_t> init(c->n_cold);
    if (cfg->cold_init_order) {
      std::vector<char> seen(c->n_cold, 0);
      for (int64_t i = 0; i < c->n_cold; ++i) {
        int64_t v = cfg->cold_init_order[i];
        if (v < c->n_hot || v >= cfg->n_slots || seen[v - c->n_hot]) {
          delete c;
          return GRANIKV_ERR_INVALID;
        }
        seen[v - c->n_hot] = 1;
        init[i] = (int32_t)v;
      }
    } else {
      for (int64_t i = 0; i < c->n_cold; ++i) init[i] = (int32_t)(c->n_hot + i);
    }
    DeviceGuard dg(cfg->device);
    cudaError_t e = dg.ok ? cudaSuccess : cudaErrorInvalidDevice;
    cudaDeviceProp prop;
    if (e == cudaSuccess) e = cudaGetDeviceProperties(&prop, cfg->device);
    if (e == cudaSuccess) {
      c->num_sms = prop.multiProcessorCount;
      c->cc_major = prop.major;
      c->cc_minor = prop.minor;
    }
    if (e == cudaSuccess) e = cudaMalloc((void**)&c->d_ring, sizeof(int32_t) * c->n_cold);
    if (e == cudaSuccess) e = cudaMalloc((void**)&c->d_err, sizeof(int32_t) * 4);
    if (e == cudaSuccess) e = cudaMalloc((void**)&c->d_stage, sizeof(int32_t) * (c->cfg.max_batch + 1));
    if (e == cudaSuccess) e = cudaMalloc((void**)&c->d_ring_pos, sizeof(int64_t) * 2);
    if (e == cudaSuccess)
      e = cudaMemcpy(c->d_ring, init.data(), sizeof(int32_t) * c->n_cold, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(c->d_err, 0, sizeof(int32_t) * 4);
    if (e == cudaSuccess) {
      const int64_t pos[2] = {c->head, c->tail};
      e = cudaMemcpy(c->d_ring_pos, pos, sizeof(pos), cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->aux, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming);
    if (e == cudaSuccess && cfg->dtype == GRANIKV_DTYPE_BF16 && cfg->head_dim == 128 && c->cc_major == 10) {
      c->tmap_k.resize(cfg->n_layers);
      c->tmap_v.resize(cfg->n_layers);
      bool ok = true;
      for (int32_t l = 0; l < cfg->n_layers && ok; ++l) {
        ok = ((uintptr_t)c->kpool[l] % 16 == 0) && ((uintptr_t)c->vpool[l] % 16 == 0) &&
             encode_pool_map(&c->tmap_k[l], c->kpool[l], cfg->n_slots, cfg->n_kv) &&
             encode_pool_map(&c->tmap_v[l], c->vpool[l], cfg->n_slots, cfg->n_kv);
      }
      c->has_tmaps = ok;
    }
    if (e != cudaSuccess) {
      if (c->d_ring) cudaFree(c->d_ring);
      if (c->d_err) cudaFree(c->d_err);
      if (c->d_stage) cudaFree(c->d_stage);
      if (c->d_ring_pos) cudaFree(c->d_ring_pos);
      if (c->ev_fork) cudaEventDestroy(c->ev_fork);
      if (c->ev_join) cudaEventDestroy(c->ev_join);
      if (c->aux) cudaStreamDestroy(c->aux);
      delete c;
      return GRANIKV_ERR_CUDA;
    }
  }
  *out = c;
  return GRANIKV_OK;
}

granikv_status granikv_destroy(granikv_ctx* c) {
  if (!c) return GRANIKV_ERR_INVALID;
  if (c->own_plan) delete c->own_plan;
  if (!c->cfg.host_only) {
    DeviceGuard dg(c->cfg.device);
    if (c->d_ring) cudaFree(c->d_ring);
    if (c->d_err) cudaFree(c->d_err);
    if (c->d_stage) cudaFree(c->d_stage);
    if (c->d_ring_pos) cudaFree(c->d_ring_pos);
    if (c->ev_fork) cudaEventDestroy(c->ev_fork);
    if (c->ev_join) cudaEventDestroy(c->ev_join);
    if (c->aux) cudaStreamDestroy(c->aux);
  }
  delete c;
  return GRANIKV_OK;
}

// ---- HOT pool -------------------------------------------------------------------------------

granikv_status granikv_hot_alloc(granikv_ctx* c, int32_t L_p, int32_t* slab_id, int64_t* off) {
  if (!c || !slab_id || !off || L_p <= 0) return GRANIKV_ERR_INVALID;
  int32_t sid = -1;
  for (int32_t i = 0; i < (int32_t)c->slabs.size(); ++i)
    if (!c->slabs[i].live) {
      sid = i;
      break;
    }
  if (sid < 0) return GRANIKV_ERR_NO_HOT_SPACE;
  for (size_t i = 0; i < c->free_ext.size(); ++i) {
    Extent& e = c->free_ext[i];
    if (e.len >= L_p) {
      int64_t o = e.off;
      e.off += L_p;
      e.len -= L_p;
      if (e.len == 0) c->free_ext.erase(c->free_ext.begin() + i);
      c->slabs[sid].off = o;
      c->slabs[sid].len = L_p;
      c->slabs[sid].live = true;
      *slab_id = sid;
      *off = o;
      return GRANIKV_OK;
    }
  }
  return GRANIKV_ERR_NO_HOT_SPACE;
}

granikv_status granikv_hot_free(granikv_ctx* c, int32_t sid) {
  if (!c || sid < 0 || sid >= (int32_t)c->slabs.size() || !c->slabs[sid].live)
    return GRANIKV_ERR_INVALID;
  Slab& s = c->slabs[sid];
  Extent ne{s.off, s.len};
  s.live = false;
  auto it = std::lower_bound(c->free_ext.begin(), c->free_ext.end(), ne,
                             [](const Extent& a, const Extent& b) { return a.off < b.off; });
  it = c->free_ext.insert(it, ne);
  size_t i = it - c->free_ext.begin();
  if (i + 1 < c->free_ext.size() && c->free_ext[i].off + c->free_ext[i].len == c->free_ext[i + 1].off) {
    c->free_ext[i].len += c->free_ext[i + 1].len;
    c->free_ext.erase(c->free_ext.begin() + i + 1);
  }
  if (i > 0 && c->free_ext[i - 1].off + c->free_ext[i - 1].len == c->free_ext[i].off) {
    c->free_ext[i - 1].len += c->free_ext[i].len;
    c->free_ext.erase(c->free_ext.begin() + i);
  }
  return GRANIKV_OK;
}

granikv_status granikv_hot_info(granikv_ctx* c, int32_t sid, int64_t* off, int32_t* L_p) {
  if (!c || sid < 0 || sid >= (int32_t)c->slabs.size() || !c->slabs[sid].live)
    return GRANIKV_ERR_INVALID;
  if (off) *off = c->slabs[sid].off;
  if (L_p) *L_p = c->slabs[sid].len;
  return GRANIKV_OK;
}

granikv_status granikv_hot_stats(granikv_ctx* c, int64_t* n_hot, int64_t* largest) {
  if (!c) return GRANIKV_ERR_INVALID;
  if (n_hot) *n_hot = c->n_hot;
  if (largest) {
    int64_t m = 0;
    for (auto& e : c->free_ext) m = std::max(m, e.len);
    *largest = m;
  }
  return GRANIKV_OK;
}

granikv_status granikv_hot_fill(granikv_ctx* c, int32_t layer, int32_t sid, const void* k,
                                const void* v, granikv_stream_t stream) {
  if (!c || !k || !v || layer < 0 || layer >= c->cfg.n_layers) return GRANIKV_ERR_INVALID;
  if (sid < 0 || sid >= (int32_t)c->slabs.size() || !c->slabs[sid].live) return GRANIKV_ERR_INVALID;
  if (!has_device(c)) return GRANIKV_ERR_NO_DEVICE;
  DeviceGuard dg(c->cfg.device);
  size_t row = (size_t)c->cfg.n_kv * c->cfg.head_dim * elem_size(c->cfg.dtype);
  size_t off = (size_t)c->slabs[sid].off * row;
  size_t bytes = (size_t)c->slabs[sid].len * row;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync((char*)c->kpool[layer] + off, k, bytes, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync((char*)c->vpool[layer] + off, v, bytes, cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

// ---- COLD pool ------------------------------------------------------------------------------

granikv_status granikv_cold_alloc(granikv_ctx* c, const int32_t* n_new, int32_t B,
                                  int32_t* req_to_slot, int32_t* suffix_len, int32_t cap,
                                  int32_t* slots_out, granikv_stream_t stream) {
  if (!c || !n_new || B <= 0 || !req_to_slot || !suffix_len || cap <= 0) return GRANIKV_ERR_INVALID;
  if (B > c->cfg.max_batch) return GRANIKV_ERR_INVALID;
  if (!has_device(c)) return GRANIKV_ERR_NO_DEVICE;
  std::vector<int32_t> excl(B + 1);
  int64_t tot = 0;
  for (int32_t b = 0; b < B; ++b) {
    if (n_new[b] < 0 || n_new[b] > cap) return GRANIKV_ERR_INVALID;
    excl[b] = (int32_t)tot;
    tot += n_new[b];
  }
  if (tot > (int64_t)INT32_MAX) return GRANIKV_ERR_INVALID;
  excl[B] = (int32_t)tot;
  if (tot > c->tail - c->head) return GRANIKV_ERR_NO_COLD_SPACE;
  if (tot == 0) return GRANIKV_OK;
  DeviceGuard dg(c->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(c->d_stage, excl.data(), sizeof(int32_t) * (B + 1),
                                  cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = launch_cold_alloc(c->d_stage, B, c->d_ring, c->n_cold, c->head, req_to_slot, suffix_len,
                          cap, slots_out, c->d_ring_pos, c->d_err, s);
  if (e != cudaSuccess) return GRANIKV_ERR_CUDA;
  c->n_copies += 1;
  c->n_kernels += 1;
  c->head += tot;
  return GRANIKV_OK;
}

granikv_status granikv_cold_free(granikv_ctx* c, const int32_t* slots, int32_t n,
                                 granikv_stream_t stream) {
  if (!c || n < 0 || (n > 0 && !slots)) return GRANIKV_ERR_INVALID;
  if (!has_device(c)) return GRANIKV_ERR_NO_DEVICE;
  if ((c->tail - c->head) + n > c->n_cold) return GRANIKV_ERR_INVALID;
  if (n == 0) return GRANIKV_OK;
  DeviceGuard dg(c->cfg.device);
  cudaError_t e = launch_cold_free(slots, n, c->d_ring, c->n_cold, c->tail, c->n_hot,
                                   c->cfg.n_slots, c->checks, c->d_ring_pos, c->d_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return GRANIKV_ERR_CUDA;
  c->n_kernels += 1;
  c->tail += n;
  return GRANIKV_OK;
}

granikv_status granikv_cold_alloc_uniform(granikv_ctx* c, int32_t n, int32_t B, int32_t* req_to_slot,
                                          int32_t* suffix_len, int32_t cap, int32_t* slots_out,
                                          granikv_stream_t stream) {
  if (!c || n < 0 || B <= 0 || !req_to_slot || !suffix_len || cap <= 0 || n > cap) return GRANIKV_ERR_INVALID;
  if (B > c->cfg.max_batch) return GRANIKV_ERR_INVALID;
  if (!has_device(c)) return GRANIKV_ERR_NO_DEVICE;
  if (n == 0) return GRANIKV_OK;
  DeviceGuard dg(c->cfg.device);
  cudaError_t e = launch_cold_alloc_uniform(n, B, c->d_ring, c->n_cold, req_to_slot, suffix_len, cap, slots_out,
                                            c->d_ring_pos, c->d_err, (cudaStream_t)stream);
  if (e != cudaSuccess) return GRANIKV_ERR_CUDA;
  c->n_kernels += 1;
  c->head += (int64_t)n * B;  // as if it ran once; granikv_cold_sync reads the device's count
  return GRANIKV_OK;
}

granikv_status granikv_cold_sync(granikv_ctx* c, granikv_stream_t stream) {
  if (!c) return GRANIKV_ERR_INVALID;
  if (!has_device(c)) return GRANIKV_ERR_NO_DEVICE;
  DeviceGuard dg(c->cfg.device);
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  int64_t pos[2] = {0, 0};
  if (e == cudaSuccess) e = cudaMemcpy(pos, c->d_ring_pos, sizeof(pos), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return GRANIKV_ERR_CUDA;
  c->head = pos[0];
  c->tail = pos[1];
  return GRANIKV_OK;
}

granikv_status granikv_cold_free_count(granikv_ctx* c, int64_t* n_free) {
  if (!c || !n_free) return GRANIKV_ERR_INVALID;
  *n_free = c->tail - c->head;
  return GRANIKV_OK;
}

granikv_status granikv_cold_append(granikv_ctx* c, int32_t layer, const void* k_new,
                                   const void* v_new, const int32_t* slots, int32_t N,
                                   granikv_stream_t stream) {
  if (!c || layer < 0 || layer >= c->cfg.n_layers || N < 0) return GRANIKV_ERR_INVALID;
  if (N > 0 && (!k_new || !v_new || !slots)) return GRANIKV_ERR_INVALID;
  if (!has_device(c)) return GRANIKV_ERR_NO_DEVICE;
  if (N == 0) return GRANIKV_OK;
  DeviceGuard dg(c->cfg.device);
  cudaError_t e = launch_cold_append(c->cfg.dtype, k_new, v_new, slots, N, c->kpool[layer],
                                     c->vpool[layer], (int64_t)c->cfg.n_kv * c->cfg.head_dim,
                                     c->n_hot, c->cfg.n_slots, c->checks, c->d_err,
                                     (cudaStream_t)stream);
  if (e == cudaSuccess) c->n_kernels += 1;
  return cuda_status(e);
}

// ---- dispatch -------------------------------------------------------------------------------

granikv_status granikv_plan_create(granikv_ctx* c, granikv_plan** out) {
  if (!c || !out) return GRANIKV_ERR_INVALID;
  granikv_plan* p = new (std::nothrow) granikv_plan();
  if (!p) return GRANIKV_ERR_INVALID;
  p->ctx = c;
  p->uid = g_next_plan_uid.fetch_add(1);
  *out = p;
  return GRANIKV_OK;
}

granikv_status granikv_plan_destroy(granikv_plan* p) {
  if (!p) return GRANIKV_ERR_INVALID;
  delete p;
  return GRANIKV_OK;
}

granikv_status granikv_dispatch(granikv_ctx* c, const granikv_batch* bt, granikv_plan* p) {
  if (!c || !bt || !p || p->ctx != c) return GRANIKV_ERR_INVALID;
  const int32_t B = bt->B;
  if (B <= 0 || B > c->cfg.max_batch || !bt->slab_id || !bt->seq_len || bt->cap < 0)
    return GRANIKV_ERR_INVALID;
  p->valid = false;
  const int32_t g = c->g;
  const int32_t n_kv = c->cfg.n_kv;

  // 1. group requests by slab id, in order of first appearance; members in request order
  granikv_plan::Scratch& w = p->scratch;
  std::vector<int32_t>& grp_slab = w.grp_slab;
  std::vector<int32_t>& grp_count = w.grp_count;
  std::vector<int32_t>& req_group = w.req_group;
  int64_t T_all = 0;    // COLD tokens of the batch
  int64_t T_tiles = 0;  // their 16-token tiles, counted per request
  int64_t n_sreq = 0;   // requests with COLD tokens
  // the groups of the last dispatch stand if the batch has the same slab ids and each group's
  // slab is still the same live extent
  bool same_groups = w.groups_cached && (int32_t)w.cache_slab_id.size() == B &&
                     std::memcmp(w.cache_slab_id.data(), bt->slab_id, sizeof(int32_t) * (size_t)B) == 0;
  for (size_t i = 0; same_groups && i < grp_slab.size(); ++i) {
    const int32_t sid = grp_slab[i];
    same_groups = sid < (int32_t)c->slabs.size() && c->slabs[sid].live && c->slabs[sid].off == w.cache_slab[i].off &&
                  c->slabs[sid].len == w.cache_slab[i].len;
  }
  w.groups_cached = false;  // set again once this dispatch succeeds
  w.pitems_cached = w.pitems_cached && same_groups;
  if (same_groups) {
    for (int32_t b = 0; b < B; ++b) {
      const int32_t L = bt->seq_len[b];
      if (L < 0 || L > bt->cap || (L == 0 && bt->slab_id[b] < 0)) return GRANIKV_ERR_INVALID;
      T_all += L;
      T_tiles += (L + 15) / 16;
      n_sreq += L > 0 ? 1 : 0;
    }
  } else {
    w.pitems_cached = false;
    std::vector<int32_t>& slot_of_slab = w.slot_of_slab;
    if (slot_of_slab.size() != c->slabs.size()) slot_of_slab.assign(c->slabs.size(), -1);
    grp_slab.clear();
    grp_count.clear();
    struct ResetSlots {  // leave slot_of_slab all -1 again, whichever way this call returns
      std::vector<int32_t>& map;
      const std::vector<int32_t>& used;
      ~ResetSlots() {
        for (int32_t sid : used) map[sid] = -1;
      }
    } reset_slots{slot_of_slab, grp_slab};
    req_group.resize(B);
    for (int32_t b = 0; b < B; ++b) {
      int32_t sid = bt->slab_id[b];
      int32_t L = bt->seq_len[b];
      req_group[b] = -1;
      if (L < 0 || L > bt->cap) return GRANIKV_ERR_INVALID;
      T_all += L;
      T_tiles += (L + 15) / 16;
      n_sreq += L > 0 ? 1 : 0;
      if (sid < 0) {
        if (L == 0) return GRANIKV_ERR_INVALID;
        continue;
      }
      if (sid >= (int32_t)c->slabs.size() || !c->slabs[sid].live) return GRANIKV_ERR_INVALID;
      if (slot_of_slab[sid] < 0) {
        slot_of_slab[sid] = (int32_t)grp_slab.size();
        grp_slab.push_back(sid);
        grp_count.push_back(0);
      }
      req_group[b] = slot_of_slab[sid];
      grp_count[slot_of_slab[sid]]++;
    }
  }
  const int32_t G = (int32_t)grp_slab.size();

  // 2. backend per group: M_eff = B_g * n_q / n_kv, dense iff M_eff >= M_sat
  std::vector<DevGroup>& groups = w.groups;
  groups.assign(G, DevGroup{});
  p->info.assign(G, granikv_group_info{});
  std::vector<int32_t>& begin = w.begin;
  begin.assign(G + 1, 0);
  for (int32_t i = 0; i < G; ++i) begin[i + 1] = begin[i] + grp_count[i];
  for (int32_t i = 0; i < G; ++i) {
    DevGroup& dg = groups[i];
    const Slab& s = c->slabs[grp_slab[i]];
    int32_t m_eff = grp_count[i] * g;
    int32_t backend = c->forced != GRANIKV_BACKEND_AUTO
                          ? c->forced
                          : (m_eff >= c->m_sat ? GRANIKV_BACKEND_DENSE : GRANIKV_BACKEND_CASCADE);
    dg.slab_off = s.off;
    dg.L_p = s.len;
    dg.n_req = grp_count[i];
    dg.req_begin = begin[i];
    dg.backend = backend;
    dg.impl = prefix_impl_for(c, backend);
    dg.sub = dg.impl == kImplCascadeStream ? stream_sub_for(grp_count[i], g) : 0;
    dg.rows_per_cta = rows_per_cta_for(dg.impl, g, dg.sub);
    dg.row_blocks = (m_eff + dg.rows_per_cta - 1) / dg.rows_per_cta;
  }
  // Fused merge when every kernel of the step is a tensor-core kernel; then the suffix may run
  // next to the prefix on its own share of the SMs.
  const bool fast_suffix_pre = c->cfg.dtype == GRANIKV_DTYPE_BF16 && c->cfg.head_dim == 128 && g <= 8;
  bool fused = c->fused_merge && (fast_suffix_pre || T_all == 0);
  for (int32_t i = 0; i < G; ++i)
    if (groups[i].impl == kImplGeneric || groups[i].impl == kImplDenseTf32) fused = false;
  bool fast_all = fast_suffix_pre || T_all == 0;
  for (int32_t i = 0; i < G; ++i)
    if (groups[i].impl == kImplGeneric || groups[i].impl == kImplDenseTf32) fast_all = false;
  bool concurrent = fast_all && c->concurrent && G > 0 && T_all > 0;
  const bool split_sms = concurrent && c->prefix_share < 0.999f;
  const bool auto_share = split_sms && c->prefix_share <= 0.f;
  const int32_t prefix_sms =
      split_sms && !auto_share ? std::max(1, (int32_t)std::lround(c->prefix_share * c->num_sms)) : c->num_sms;
  int32_t suffix_sms = c->num_sms;  // set after the prefix pieces when the SMs are split
  bool read_ahead = false;          // the split's dense CTAs read ahead into L2 (see below)
  double tail_frac = 0.0;           // share of the suffix work the dense CTAs take after their piece

  // 3. prefix pieces: the smallest piece length (in tiles, one length for all groups) whose
  //    CTA count fits the target, pieces balanced to within one tile.  The tensor-core
  //    kernels run one CTA per SM, so their target is one wave over their SMs.
  int64_t target = 2LL * c->num_sms;
  for (int32_t i = 0; i < G; ++i)
    if (groups[i].impl != kImplGeneric) target = prefix_sms;
  {
    int64_t max_tiles = 1;
    for (int32_t i = 0; i < G; ++i) {
      const int64_t tile = tile_tokens_for(groups[i].impl, groups[i].sub);
      max_tiles = std::max<int64_t>(max_tiles, (groups[i].L_p + tile - 1) / tile);
    }
    auto ctas_for = [&](int64_t piece_tiles) {
      int64_t n = 0;
      for (int32_t i = 0; i < G; ++i) {
        const int64_t tile = tile_tokens_for(groups[i].impl, groups[i].sub);
        const int64_t t = (groups[i].L_p + tile - 1) / tile;
        n += ctas_per_piece(groups[i], n_kv) * ((t + piece_tiles - 1) / piece_tiles);
      }
      return n;
    };
    int64_t lo = 1, hi = max_tiles;  // smallest piece length with ctas_for <= target
    while (lo < hi) {
      const int64_t mid = (lo + hi) / 2;
      if (ctas_for(mid) <= target) hi = mid;
      else lo = mid + 1;
    }
    bool auto_found = false;
    if (auto_share) {
      // Automatic split: the piece length whose prefix time (one wave: the longest piece) and
      // suffix time (its work spread over the SMs the prefix CTAs leave) are most nearly equal,
      // i.e. the smallest max of the two.  Costs measured on GB300: a prefix CTA 5 us plus, per
      // 128-query-row block and token, 0.0078 us (dense) or 0.02 us (warp-MMA cascade), or per
      // token of a group of eight KV heads 0.09 us (streaming cascade, 4 KB a token); the suffix
      // 1.40 SM-us per 16 COLD tokens of one group of up to 8 KV heads.
      // The split is also weighed against running the two one after another on all SMs, with
      // the suffix then bound by the bandwidth HBM gives its random 2 KB row reads (about
      // 5.8 TB/s measured), and the step's bytes bounding either way at about 5.9 TB/s.
      const int64_t head_groups = (n_kv + 7) / 8;
      const double w_s = 1.40 * (double)head_groups * (double)T_tiles;
      const double suffix_bytes = 4.0 * n_kv * c->cfg.head_dim * (double)T_all;
      double prefix_bytes = 0.0;
      for (int32_t i = 0; i < G; ++i) prefix_bytes += 4.0 * n_kv * c->cfg.head_dim * (double)groups[i].L_p;
      auto prefix_time = [&](int64_t cand) {
        double t_p = 0.0;
        for (int32_t i = 0; i < G; ++i) {
          const int64_t tile = tile_tokens_for(groups[i].impl, groups[i].sub);
          const double per_token = groups[i].impl == kImplDenseTc ? 0.0078
                                   : groups[i].impl == kImplCascadeStream
                                       ? 0.09 * std::min(n_kv, stream_heads(groups[i].sub)) / 8.0
                                       : 0.02;
          const double fixed = groups[i].impl == kImplCascadeStream ? 3.0 : 5.0;
          t_p = std::max(t_p, fixed + per_token * (double)std::min<int64_t>(cand * tile, groups[i].L_p));
        }
        return t_p;
      };
      const double t_bytes = (prefix_bytes + suffix_bytes) / 5.9e6;  // us at 5.9 TB/s
      double best = 1e300;
      const int64_t lo_serial = lo;
      for (int64_t n = 1; n <= max_tiles; ++n) {
        const int64_t cand = (max_tiles + n - 1) / n;
        if (n > 1 && cand == (max_tiles + n - 2) / (n - 1)) continue;  // same length as n - 1
        const int64_t ctas = ctas_for(cand);
        if (ctas >= c->num_sms) break;  // one wave, and at least one SM for the suffix
        const double t = std::max({prefix_time(cand), w_s / (double)(c->num_sms - ctas), t_bytes});
        if (t < best) {
          best = t;
          lo = cand;
          auto_found = true;
        }
      }
      // read-ahead pays where the prefix side is estimated to end last and the suffix side
      // competes with it for HBM (suffix bytes at least the prefix's)
      if (auto_found)
        read_ahead = prefix_time(lo) > w_s / (double)(c->num_sms - ctas_for(lo)) && suffix_bytes >= prefix_bytes;
      // When the suffix side is estimated to end last and every prefix CTA is dense (one grid,
      // one KV-head group), the dense CTAs take suffix runs after their prefix piece: x SM-us of
      // suffix work such that both sides end together.  Qwen-2.5 shape, 16K prefix, B = 128:
      // the 80 dense CTAs ended 20 us before the 72 suffix CTAs without it.  The dense CTA's
      // set-up for its run (a few us) is left out: the prefix estimate runs about 6 us long on
      // that shape, which covers it; with 4 / 2 / 0 us set aside for it the call took 82.9 /
      // 81.0 / 80.3 us, and at 0 both sides end within 0.4 us of each other.
      bool all_dense = G > 0 && n_kv <= 8;
      for (int32_t i = 0; i < G; ++i) all_dense = all_dense && groups[i].impl == kImplDenseTc;
      if (auto_found && all_dense) {
        const double n_d = (double)ctas_for(lo), n_s = (double)c->num_sms - n_d;
        const double x = (w_s / n_s - prefix_time(lo)) / (1.0 / n_s + 1.0 / n_d);
        if (x > 0.0) tail_frac = x / w_s;
      }
      // serial: the suffix kernel starts only after the prefix kernel's last CTA (its tail and
      // the second kernel's ramp measured at about 5 us)
      const double t_serial =
          prefix_time(lo_serial) + std::max(w_s / (double)c->num_sms, suffix_bytes / 5.8e6) + 5.0;
      if (auto_found && t_serial < best) {
        lo = lo_serial;
        auto_found = false;
        concurrent = false;
        tail_frac = 0.0;
      }
    }
    for (int32_t i = 0; i < G; ++i) {
      DevGroup& dg = groups[i];
      const int64_t tile = tile_tokens_for(dg.impl, dg.sub);
      const int64_t t = (dg.L_p + tile - 1) / tile;
      const int64_t n_splits = (t + lo - 1) / lo;
      const int64_t base = t / n_splits;
      dg.n_splits = (int32_t)n_splits;
      dg.tile = (int32_t)tile;
      dg.split_len = (int32_t)(base * tile);
      dg.n_long = (int32_t)(t - base * n_splits);
      dg.q_b0 = -1;
      dg.causal = 0;
    }
    // Serial schedule, dense groups only (the dense kernel on all SMs by itself): when the
    // units do not divide into the SMs, the balanced one-wave pieces leave SMs idle (40 units of
    // the Qwen-2.5 shape: 3 pieces each, 120 CTAs on 152 SMs).  Pieces of a fixed length L with
    // a shorter remainder, launched longest first, put the remainders on the idle SMs and then
    // run them as a short second wave.  A greedy schedule of the pieces (longest first, each on
    // the SM that frees first; a CTA costs its tiles plus about 7 tiles of set-up and epilogue)
    // picks L, or keeps the balanced plan when that finishes first.  Only for groups of one
    // length (one shared prefix, or several of equal length): with prefixes of different
    // lengths the remainders come out of very different sizes, and measured on GB300 (eight
    // prefixes of 2K-16K) the second wave cost more than it saved.  The choice depends only on
    // the groups' tile counts, so it is memoised on them.
    w.grp_tail.assign(G, 0);
    bool all_dense = G > 0;
    for (int32_t i = 0; i < G; ++i)
      all_dense = all_dense && groups[i].impl == kImplDenseTc && groups[i].L_p == groups[0].L_p;
    if (!concurrent && all_dense) {
      constexpr int64_t kCtaFixedTiles = 7;
      std::vector<int64_t>& key = w.tail_key_now;
      key.assign({lo, (int64_t)c->num_sms});
      for (int32_t i = 0; i < G; ++i)
        key.insert(key.end(), {(groups[i].L_p + kDenseTile - 1) / kDenseTile, ctas_per_piece(groups[i], n_kv)});
      if (key != w.tail_key) {
        w.tail_key = key;
        std::vector<int64_t> lens;
        auto makespan = [&]() {
          std::sort(lens.begin(), lens.end(), std::greater<int64_t>());
          std::vector<int64_t>& heap = w.sim_heap;
          heap.assign((size_t)c->num_sms, 0);  // finish time of each SM (all 0: a valid min-heap)
          int64_t end = 0;
          for (const int64_t len : lens) {
            std::pop_heap(heap.begin(), heap.end(), std::greater<int64_t>());
            heap.back() += kCtaFixedTiles + len;
            end = std::max(end, heap.back());
            std::push_heap(heap.begin(), heap.end(), std::greater<int64_t>());
          }
          return end;
        };
        for (int32_t i = 0; i < G; ++i) {  // the balanced plan made above
          const DevGroup& dg = groups[i];
          const int64_t base = dg.split_len / kDenseTile;
          for (int32_t sp = 0; sp < dg.n_splits; ++sp)
            lens.insert(lens.end(), (size_t)ctas_per_piece(dg, n_kv), base + (sp < dg.n_long ? 1 : 0));
        }
        int64_t best = makespan(), best_len = 0;
        for (int64_t len = lo - 1; len >= std::max<int64_t>(1, lo - lo / 3); --len) {
          lens.clear();
          for (int32_t i = 0; i < G; ++i) {
            const int64_t t = (groups[i].L_p + kDenseTile - 1) / kDenseTile;
            const int64_t per = ctas_per_piece(groups[i], n_kv), pieces = (t + len - 1) / len;
            lens.insert(lens.end(), (size_t)(per * (pieces - 1)), len);
            lens.insert(lens.end(), (size_t)per, t - (pieces - 1) * len);
          }
          if ((int64_t)lens.size() > 2LL * c->num_sms) break;
          const int64_t m = makespan();
          if (m < best) {
            best = m;
            best_len = len;
          }
        }
        w.tail_len = best_len;
      }
      if (w.tail_len > 0) {
        for (int32_t i = 0; i < G; ++i) {
          DevGroup& dg = groups[i];
          const int64_t t = (dg.L_p + kDenseTile - 1) / kDenseTile;
          dg.n_splits = (int32_t)((t + w.tail_len - 1) / w.tail_len);
          dg.split_len = (int32_t)(w.tail_len * kDenseTile);
          dg.n_long = 0;
          w.grp_tail[i] = t % w.tail_len != 0 ? 1 : 0;
        }
      }
    }
    // the tensor-core prefix kernels hold one SM per CTA; the suffix gets every other SM (an
    // automatic split that found no piece length leaving the suffix an SM shares them all)
    if (split_sms && (!auto_share || auto_found))
      suffix_sms = (int32_t)std::max<int64_t>(1, (int64_t)c->num_sms - ctas_for(lo));
  }
  for (int32_t i = 0; i < G; ++i) {
    const DevGroup& dg = groups[i];
    granikv_group_info& gi = p->info[i];
    gi.slab_id = grp_slab[i];
    gi.n_requests = dg.n_req;
    gi.m_eff = dg.n_req * g;
    gi.backend = dg.backend;
    gi.L_p = dg.L_p;
    gi.n_splits = dg.n_splits;
    gi.slot_offset = dg.slab_off;
  }
  // 4. suffix: cut the concatenation of all requests' COLD tokens, in 16-token tiles counted
  //    per request (a request's last tile may be partial), into one run per token-CTA
  //    (stream-K); each request segment inside a run is one work item and record.  Cuts fall on
  //    tile boundaries of the request.  A segment costs its CTA about one tile on top of its
  //    tiles (measured on GB300, Llama-3.1-8B shape, 88 token-CTAs of 22-23 tiles: 0.54-0.76 us
  //    a segment against 0.6-0.7 us a tile; the segments of short requests also hold their
  //    recently appended tokens, whose slots are scattered), so each run ends where its tiles
  //    plus segments reach an equal share of what is left when it starts (cut_suffix_runs).
  static_assert(kSTile == 16, "the tile count above uses 16-token tiles");
  const int64_t T = T_tiles;
  const bool fast_suffix = c->cfg.dtype == GRANIKV_DTYPE_BF16 && c->cfg.head_dim == 128 && g <= 8;
  const int32_t suffix_impl = fast_suffix ? kImplSuffixMma : kImplGeneric;
  int32_t n_scta = 0;       // token-CTA runs
  int32_t n_tail = 0;       // of them, the last n_tail are run by the dense CTAs of one grid
  int64_t U = 0;            // tiles plus segment costs, with every cut counted as inside a request
  int64_t U_tail = 0;       // of U, the tail runs' share
  if (T > 0) {
    // one wave over the suffix's SMs, with at least kMinCtaTiles tiles per token-CTA (a CTA's
    // set-up and first-tile latency cost about as much as three tiles, and every CTA adds a
    // record per request it touches), unless a CTA would then stream more tokens than it can
    // stage slot ids for
    constexpr int64_t kMinCtaTiles = 4;
    constexpr int64_t kMaxCtaTiles = kSuffixMaxCtaTokens / kSTile;
    n_scta = (int32_t)std::min<int64_t>(suffix_sms, (T + kMinCtaTiles - 1) / kMinCtaTiles);
    n_scta = (int32_t)std::max<int64_t>(n_scta, (T + n_sreq + kMaxCtaTiles - 3) / (kMaxCtaTiles - 2));
    const int32_t n_dense_ctas = (int32_t)(c->num_sms - suffix_sms);
    if (tail_frac > 0.0 && n_scta == suffix_sms && n_dense_ctas > 0) {
      n_tail = n_dense_ctas;
      n_scta += n_tail;
    }
    U = T + kSegTiles * (n_sreq + n_scta - 1);
    U_tail = n_tail > 0 ? (int64_t)(tail_frac * (double)U) : 0;
    if (U_tail < 3 * (int64_t)n_tail) {  // under about two tiles a run: not worth a run's set-up
      n_scta -= n_tail;
      n_tail = 0;
      U_tail = 0;
      U = T + kSegTiles * (n_sreq + n_scta - 1);
    }
  }

  // 5. records and work items
  std::vector<int32_t>& group_req = w.group_req;
  if (!same_groups) {
    group_req.resize(begin[G]);
    std::vector<int32_t>& fill = w.fill;
    fill.assign(begin.begin(), begin.end() - 1);
    for (int32_t b = 0; b < B; ++b)
      if (req_group[b] >= 0) group_req[fill[req_group[b]]++] = b;
    w.grp_contig.assign(G, 0);
    for (int32_t i = 0; i < G; ++i) {
      bool contiguous = grp_count[i] > 0;
      for (int32_t k = 1; k < grp_count[i] && contiguous; ++k)
        contiguous = group_req[begin[i] + k] == group_req[begin[i]] + k;
      w.grp_contig[i] = contiguous ? 1 : 0;
    }
  }
  // dense groups whose requests are consecutive in the batch load their q rows by TMA boxes
  for (int32_t i = 0; i < G; ++i) {
    DevGroup& dg = groups[i];
    if (dg.impl == kImplDenseTc && kDenseRows % g == 0 && w.grp_contig[i]) dg.q_b0 = group_req[dg.req_begin];
  }
  // prefix items grouped by kernel; within a group the row blocks of one (KV head, piece)
  // are adjacent so they share the piece's K/V through L2
  std::vector<DevPrefixItem>& pitems = w.pitems;
  // the items depend on the groups' kernels and shapes only (and the KV heads)
  {
    std::vector<int32_t> key_now;
    key_now.reserve((size_t)G * 6 + 1);
    key_now.push_back(n_kv);
    for (int32_t i = 0; i < G; ++i) {
      const DevGroup& dg = groups[i];
      key_now.insert(key_now.end(), {dg.impl, dg.sub, dg.n_splits, dg.row_blocks, dg.split_len, dg.n_long, w.grp_tail[i]});
    }
    if (w.pitems_cached && key_now != w.pitems_key) w.pitems_cached = false;
    if (!w.pitems_cached) w.pitems_key.swap(key_now);
  }
  if (!w.pitems_cached) {
  pitems.clear();
  for (int32_t impl = 0; impl < kNumImpl; ++impl) {
    p->pitem_first[impl] = (int32_t)pitems.size();
    for (int32_t i = 0; i < G; ++i) {
      const DevGroup& dg = groups[i];
      if (dg.impl != impl) continue;
      const int32_t units = impl == kImplCascadeStream ? (int32_t)(ctas_per_piece(dg, n_kv) / dg.row_blocks) : n_kv;
      // a group whose last piece is a shorter remainder puts those pieces after all others
      // (longest first: they fill the SMs the long pieces leave, then run as a second wave)
      const int32_t s_end = w.grp_tail[i] ? dg.n_splits - 1 : dg.n_splits;
      for (int32_t j = 0; j < units; ++j)
        for (int32_t s = 0; s < s_end; ++s)
          for (int32_t rb = 0; rb < dg.row_blocks; ++rb) pitems.push_back({i, j, rb, s});
    }
    for (int32_t i = 0; i < G; ++i) {
      const DevGroup& dg = groups[i];
      if (dg.impl != impl || !w.grp_tail[i]) continue;
      for (int32_t j = 0; j < n_kv; ++j)
        for (int32_t rb = 0; rb < dg.row_blocks; ++rb) pitems.push_back({i, j, rb, dg.n_splits - 1});
    }
    p->pitem_count[impl] = (int32_t)pitems.size() - p->pitem_first[impl];
  }
  }


  // The device image: groups, group members, requests, prefix items, suffix items, each
  // token-CTA's first suffix item; each array at a 16-byte boundary, the padding between them
  // 0, the whole a multiple of 256 bytes.  The requests and suffix items are written in place
  // below (the suffix items' count, and so where the last array starts, is known at the end).
  p->off_groups = 0;
  p->off_group_req = align_up(sizeof(DevGroup) * G, 16);
  p->off_req = align_up(p->off_group_req + sizeof(int32_t) * group_req.size(), 16);
  p->off_pitems = align_up(p->off_req + sizeof(DevReq) * B, 16);
  p->off_sitems = align_up(p->off_pitems + sizeof(DevPrefixItem) * pitems.size(), 16);
  // at most one suffix item per request plus one per token-CTA boundary
  const size_t max_sitems = (size_t)B + n_scta + 1;
  p->blob.resize(align_up(p->off_sitems + sizeof(DevSuffixItem) * max_sitems + sizeof(int32_t) * (n_scta + 1), 256));
  unsigned char* const img = p->blob.data();
  DevReq* const reqs = reinterpret_cast<DevReq*>(img + p->off_req);
  DevSuffixItem* const si = reinterpret_cast<DevSuffixItem*>(img + p->off_sitems);
  std::vector<int32_t>& scta_begin = w.scta_begin;
  scta_begin.assign(n_scta + 1, 0);
  // the runs, each request's records and the suffix items
  std::vector<int32_t>& grp_np = w.grp_np;
  grp_np.resize((size_t)G + 1);
  grp_np[0] = 0;
  for (int32_t i = 0; i < G; ++i) grp_np[i + 1] = groups[i].n_splits;
  const SuffixCut cut = cut_suffix_runs(B, grp_np.data() + 1, req_group.data(), bt->seq_len, n_scta, n_tail, U,
                                        U_tail, reqs, si, scta_begin.data());
  const int32_t n_si = cut.n_items;
  const int32_t max_parts = cut.max_parts;
  const int64_t rec = cut.records;
  if (rec > (int64_t)INT32_MAX / 2) return GRANIKV_ERR_INVALID;
  // 6. the rest of the device image
  p->off_scta = align_up(p->off_sitems + sizeof(DevSuffixItem) * (size_t)n_si, 16);
  const size_t img_end = align_up(p->off_scta + sizeof(int32_t) * scta_begin.size(), 256);
  {
    struct Part {
      size_t off;
      const void* src;  // NULL: written in place above
      size_t bytes;
      size_t next;      // where the next array starts
    };
    const Part parts[] = {
        {p->off_groups, groups.data(), sizeof(DevGroup) * G, p->off_group_req},
        {p->off_group_req, group_req.data(), sizeof(int32_t) * group_req.size(), p->off_req},
        {p->off_req, nullptr, sizeof(DevReq) * B, p->off_pitems},
        {p->off_pitems, pitems.data(), sizeof(DevPrefixItem) * pitems.size(), p->off_sitems},
        {p->off_sitems, nullptr, sizeof(DevSuffixItem) * (size_t)n_si, p->off_scta},
        {p->off_scta, scta_begin.data(), sizeof(int32_t) * scta_begin.size(), img_end},
    };
    for (const Part& pt : parts) {
      if (pt.src && pt.bytes) std::memcpy(img + pt.off, pt.src, pt.bytes);
      std::memset(img + pt.off + pt.bytes, 0, pt.next - pt.off - pt.bytes);
    }
  }
  p->blob.resize(img_end);
  p->n_groups = G;
  p->n_pitems = (int32_t)pitems.size();
  p->n_sitems = n_si;
  p->B = B;
  p->n_records = (int32_t)rec;
  p->n_prefix_records = cut.prefix_records;
  p->n_scta = n_scta;
  p->n_tail = n_tail;
  p->suffix_impl = suffix_impl;
  {
    // the merge gives a row with many records (a cascade step over all SMs has one per L_p
    // piece) several warps, so that each loads its share in one batch (8, 8, 16 or 24 records
    // a warp for 1, 2, 4 or 8 warps).  That only pays while the rows alone leave the SMs short
    // of warps: past about 16 warps an SM, the rows' own loads hide each other's latency and the
    // extra warps' combine step is pure cost, so W halves until the grid is back under that.
    int32_t wpr = max_parts <= 8 ? 1 : max_parts <= 16 ? 2 : max_parts <= 64 ? 4 : 8;
    const int64_t rows = (int64_t)B * c->cfg.n_q;
    while (wpr > 1 && rows * wpr > 16LL * c->num_sms) wpr /= 2;
    p->merge_warps = wpr;
  }
  p->fused = fused && (T == 0 || suffix_impl == kImplSuffixMma);
  p->concurrent = concurrent;
  // The dense CTAs of a split whose prefix side is estimated to end last, next to a suffix side
  // that reads at least as many bytes, read two tiles ahead into L2: their per-tile chain keeps
  // few bytes in flight, and next to suffix CTAs that keep HBM busy they fall behind.  Measured
  // on GB300 (Llama-3.1-8B shape, 16K prefix, B = 64, a 32-layer step): 42.7 -> 40.9 us a call
  // with two tiles ahead, 41.0 / 41.1 / 41.4 us with three / four / five; on another GB300
  // 43.2 -> 43.0 / 46.1 us with six / eight (further ahead takes the suffix side's bandwidth).
  // Where the suffix side ends last (Qwen-2.5 shape) it does not help; next to a light suffix
  // side it costs (16K prefix, 256 COLD tokens a request: B = 1 17.7 -> 18.4 us, B = 8 18.9 ->
  // 19.8 us); and with the kernels one after another (eight prefixes) six tiles ahead cost 17 %.
  constexpr int32_t kAutoL2Ahead = 2;
  p->l2_ahead = c->l2_ahead >= 0 ? c->l2_ahead : (concurrent && read_ahead ? kAutoL2Ahead : 0);
  p->group_impl.resize(G);
  for (int32_t i = 0; i < G; ++i) p->group_impl[i] = groups[i].impl;
  // this dispatch succeeded: its groups and prefix items may serve the next one
  if (!same_groups) {  // (else they hold these values already)
    w.cache_slab_id.assign(bt->slab_id, bt->slab_id + B);
    w.cache_slab.resize(G);
    for (int32_t i = 0; i < G; ++i) w.cache_slab[i] = c->slabs[grp_slab[i]];
  }
  w.groups_cached = true;
  w.pitems_cached = true;
  p->version++;
  p->valid = true;
  return GRANIKV_OK;
}

granikv_status granikv_plan_num_groups(const granikv_plan* p, int32_t* n) {
  if (!p || !n || !p->valid) return GRANIKV_ERR_INVALID;
  *n = p->n_groups;
  return GRANIKV_OK;
}

granikv_status granikv_plan_group(const granikv_plan* p, int32_t i, granikv_group_info* out) {
  if (!p || !out || !p->valid || i < 0 || i >= p->n_groups) return GRANIKV_ERR_INVALID;
  *out = p->info[i];
  return GRANIKV_OK;
}

granikv_status granikv_plan_suffix_runs(const granikv_plan* p, int32_t* runs, int32_t* tail_runs) {
  if (!p || !p->valid) return GRANIKV_ERR_INVALID;
  if (runs) *runs = p->suffix_impl == kImplSuffixMma ? p->n_scta : p->n_sitems;
  if (tail_runs) *tail_runs = p->n_tail;
  return GRANIKV_OK;
}

granikv_status granikv_plan_dense_l2_ahead(const granikv_plan* p, int32_t* tiles) {
  if (!p || !p->valid || !tiles) return GRANIKV_ERR_INVALID;
  *tiles = p->l2_ahead;
  return GRANIKV_OK;
}

granikv_status granikv_plan_schedule(const granikv_plan* p, int32_t* concurrent, int32_t* prefix_ctas,
                                     int32_t* suffix_ctas) {
  if (!p || !p->valid) return GRANIKV_ERR_INVALID;
  if (concurrent) *concurrent = p->concurrent ? 1 : 0;
  if (prefix_ctas) *prefix_ctas = p->n_pitems;
  if (suffix_ctas) {
    const int32_t head_groups = (p->ctx->cfg.n_kv + 7) / 8;
    *suffix_ctas = p->suffix_impl == kImplSuffixMma ? (p->n_scta - p->n_tail) * head_groups : p->n_sitems;
  }
  return GRANIKV_OK;
}

namespace {
// Workspace bound that depends only on the batch size, the prefix pieces and the SM count, so a
// workspace sized once stays large enough while the suffixes grow step after step: the plan
// holds at most B + n_sm suffix segments (each token-CTA boundary adds at most one), and each
// request has one record per prefix piece and per suffix segment.
size_t workspace_bytes(const granikv_ctx* c, const granikv_plan* p) {
  const size_t n_cta = (size_t)std::max<int32_t>(c->num_sms, p->n_scta);
  const size_t max_sitems = (size_t)p->B + n_cta + 1;
  size_t blob = p->off_sitems + align_up(sizeof(DevSuffixItem) * max_sitems, 16) +
                align_up(sizeof(int32_t) * (n_cta + 1), 256);
  blob = std::max(blob, p->blob.size());
  const size_t max_records = (size_t)p->n_prefix_records + max_sitems;
  size_t off = align_up(blob, 256);
  off += align_up(sizeof(float) * max_records * c->cfg.n_q * c->cfg.head_dim, 256);
  off += align_up(sizeof(float) * max_records * c->cfg.n_q, 256);
  off += align_up(sizeof(int32_t) * (size_t)p->B * c->cfg.n_q, 256);  // tickets
  return off;
}
size_t records_offset(const granikv_ctx* c, const granikv_plan* p) {
  const size_t n_cta = (size_t)std::max<int32_t>(c->num_sms, p->n_scta);
  const size_t max_sitems = (size_t)p->B + n_cta + 1;
  size_t blob = p->off_sitems + align_up(sizeof(DevSuffixItem) * max_sitems, 16) +
                align_up(sizeof(int32_t) * (n_cta + 1), 256);
  blob = std::max(blob, p->blob.size());
  return align_up(blob, 256);
}
size_t lse_offset(const granikv_ctx* c, const granikv_plan* p) {
  const size_t n_cta = (size_t)std::max<int32_t>(c->num_sms, p->n_scta);
  const size_t max_records = (size_t)p->n_prefix_records + (size_t)p->B + n_cta + 1;
  return records_offset(c, p) + align_up(sizeof(float) * max_records * c->cfg.n_q * c->cfg.head_dim, 256);
}
size_t tickets_offset(const granikv_ctx* c, const granikv_plan* p) {
  const size_t n_cta = (size_t)std::max<int32_t>(c->num_sms, p->n_scta);
  const size_t max_records = (size_t)p->n_prefix_records + (size_t)p->B + n_cta + 1;
  return lse_offset(c, p) + align_up(sizeof(float) * max_records * c->cfg.n_q, 256);
}
}  // namespace

granikv_status granikv_plan_image(const granikv_plan* p, void* out, size_t cap, size_t* size) {
  if (!p || !size || !p->valid) return GRANIKV_ERR_INVALID;
  *size = p->blob.size();
  if (cap < p->blob.size() || (!out && !p->blob.empty())) return GRANIKV_ERR_INVALID;
  if (!p->blob.empty()) std::memcpy(out, p->blob.data(), p->blob.size());
  return GRANIKV_OK;
}

granikv_status granikv_workspace_size(granikv_ctx* c, const granikv_plan* p, size_t* bytes) {
  if (!c || !p || !bytes || !p->valid || p->ctx != c) return GRANIKV_ERR_INVALID;
  *bytes = workspace_bytes(c, p);
  return GRANIKV_OK;
}

granikv_status granikv_set_concurrency(granikv_ctx* c, int32_t on, float share) {
  if (!c || !(share >= 0.f && share <= 1.f)) return GRANIKV_ERR_INVALID;
  c->concurrent = on ? 1 : 0;
  c->prefix_share = share;
  return GRANIKV_OK;
}

granikv_status granikv_set_fused_merge(granikv_ctx* c, int32_t on) {
  if (!c) return GRANIKV_ERR_INVALID;
  c->fused_merge = on ? 1 : 0;
  return GRANIKV_OK;
}

granikv_status granikv_set_dense_l2_ahead(granikv_ctx* c, int32_t tiles) {
  if (!c || tiles < -1 || tiles > 64) return GRANIKV_ERR_INVALID;
  c->l2_ahead = tiles;
  return GRANIKV_OK;
}

granikv_status granikv_set_msat(granikv_ctx* c, int32_t m) {
  if (!c || m <= 0) return GRANIKV_ERR_INVALID;
  c->m_sat = m;
  return GRANIKV_OK;
}

granikv_status granikv_get_msat(granikv_ctx* c, int32_t* m) {
  if (!c || !m) return GRANIKV_ERR_INVALID;
  *m = c->m_sat;
  return GRANIKV_OK;
}

granikv_status granikv_force_backend(granikv_ctx* c, int32_t backend) {
  if (!c || backend < GRANIKV_BACKEND_AUTO || backend > GRANIKV_BACKEND_CASCADE)
    return GRANIKV_ERR_INVALID;
  c->forced = backend;
  return GRANIKV_OK;
}

// ---- decode attention -----------------------------------------------------------------------

}  // extern "C"

namespace {
// Decode attention of one layer; with k_new/v_new, each request's last COLD token is taken from
// them and written to its slot by the same launches (the fused COLD append).
granikv_status decode_attention_impl(granikv_ctx* c, int32_t layer, const void* q, const void* k_new,
                                     const void* v_new, const granikv_batch* bt, granikv_plan* p, void* o,
                                     float* lse, void* ws, size_t ws_bytes, granikv_stream_t stream) {
  if (!c || !bt || !q || !o || !lse || !ws) return GRANIKV_ERR_INVALID;
  if (layer < 0 || layer >= c->cfg.n_layers) return GRANIKV_ERR_INVALID;
  if (!has_device(c)) return GRANIKV_ERR_NO_DEVICE;
  if ((uintptr_t)ws % 256) return GRANIKV_ERR_INVALID;
  if (!bt->req_to_slot) return GRANIKV_ERR_INVALID;
  if (!p) {
    if (!c->own_plan) {
      granikv_status st = granikv_plan_create(c, &c->own_plan);
      if (st != GRANIKV_OK) return st;
    }
    p = c->own_plan;
    granikv_status st = granikv_dispatch(c, bt, p);
    if (st != GRANIKV_OK) return st;
  }
  if (!p->valid || p->ctx != c || p->B != bt->B) return GRANIKV_ERR_INVALID;
  if (ws_bytes < workspace_bytes(c, p)) return GRANIKV_ERR_INVALID;
  if (k_new) {
    // the suffix kernels take each request's newest token from k_new/v_new (the tensor-core one
    // with bulk copies, whose rows must start on 16-byte boundaries); every request needs a token
    if (!v_new || ((uintptr_t)k_new | (uintptr_t)v_new) % 16) return GRANIKV_ERR_INVALID;
    for (int32_t b = 0; b < bt->B; ++b)
      if (bt->seq_len[b] < 1) return GRANIKV_ERR_INVALID;
  }

  DeviceGuard dg(c->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  unsigned char* wsb = (unsigned char*)ws;
  int32_t* tickets = (int32_t*)(wsb + tickets_offset(c, p));
  const size_t tickets_bytes = sizeof(int32_t) * (size_t)p->B * c->cfg.n_q;
  if (!ws_holds(ws, p->uid, p->version)) {
    ws_forget(ws);  // a failed copy leaves the front unknown
    cudaError_t e = cudaMemcpyAsync(wsb, p->blob.data(), p->blob.size(), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && p->fused) e = cudaMemsetAsync(tickets, 0, tickets_bytes, s);
    if (e != cudaSuccess) return GRANIKV_ERR_CUDA;
    c->n_copies += 1;
    ws_record(ws, p->uid, p->version);
  }
  AttnParams a{};
  a.q = q;
  a.o = o;
  a.lse = lse;
  a.kpool = c->kpool[layer];
  a.vpool = c->vpool[layer];
  a.req_to_slot = bt->req_to_slot;
  a.n_slots = c->cfg.n_slots;
  a.n_hot = c->n_hot;
  a.cap = bt->cap;
  a.B = bt->B;
  a.n_q = c->cfg.n_q;
  a.n_kv = c->cfg.n_kv;
  a.d = c->cfg.head_dim;
  a.g = c->g;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->cfg.head_dim));
  a.groups = (const DevGroup*)(wsb + p->off_groups);
  a.group_req = (const int32_t*)(wsb + p->off_group_req);
  a.reqs = (const DevReq*)(wsb + p->off_req);
  a.pitems = (const DevPrefixItem*)(wsb + p->off_pitems);
  a.n_pitems = p->n_pitems;
  a.sitems = (const DevSuffixItem*)(wsb + p->off_sitems);
  a.n_sitems = p->n_sitems;
  a.scta_begin = (const int32_t*)(wsb + p->off_scta);
  a.n_scta = p->n_scta;
  a.rec_o = (float*)(wsb + records_offset(c, p));
  a.rec_lse = (float*)(wsb + lse_offset(c, p));
  a.n_records = p->n_records;
  a.err = c->d_err;
  a.checks = c->checks;
  a.tickets = tickets;
  a.fused_merge = p->fused ? 1 : 0;
  a.l2_ahead = p->l2_ahead;
  a.inject_stall = c->inject_stall;
  c->inject_stall = 0;
  a.live_len = bt->seq_len_dev;
  a.k_new = k_new;
  a.v_new = v_new;
  CUtensorMap tmq{};
  a.q_tma = 0;
  if (p->pitem_count[kImplDenseTc] > 0 && c->cfg.dtype == GRANIKV_DTYPE_BF16 && c->cfg.head_dim == 128)
    a.q_tma = encode_q_map(&tmq, q, bt->B, c->cfg.n_q, c->g) ? 1 : 0;
  c->last_tickets = tickets;
  c->last_tickets_bytes = tickets_bytes;

  cudaError_t e = cudaSuccess;
  auto launch_suffix = [&](cudaStream_t st, bool pdl) -> cudaError_t {
    if (p->n_sitems <= 0) return cudaSuccess;
    c->n_kernels += 1;
    return p->suffix_impl == kImplSuffixMma ? launch_suffix_mma(a, a.scta_begin, p->n_scta, st, pdl)
                                            : launch_suffix_generic(c->cfg.dtype, a, st);
  };
  // programmatic dependent launch only between kernels of this call on one stream, and for the
  // first prefix kernel (whose stream predecessor is whatever the caller enqueued last)
  auto launch_prefix = [&](cudaStream_t st) -> cudaError_t {
    cudaError_t r = cudaSuccess;
    if (p->pitem_count[kImplGeneric] > 0) {
      r = launch_prefix_generic(c->cfg.dtype, a, p->pitem_first[kImplGeneric], p->pitem_count[kImplGeneric], st);
      c->n_kernels += 1;
    }
    if (r == cudaSuccess && p->pitem_count[kImplDenseTf32] > 0) {
      r = launch_dense_tf32(a, p->pitem_first[kImplDenseTf32], p->pitem_count[kImplDenseTf32], st);
      c->n_kernels += 1;
    }
    if (r == cudaSuccess && p->pitem_count[kImplCascadeMma] > 0) {
      r = launch_cascade_mma(a, p->pitem_first[kImplCascadeMma], p->pitem_count[kImplCascadeMma], st);
      c->n_kernels += 1;
    }
    if (r == cudaSuccess && p->pitem_count[kImplCascadeStream] > 0) {
      // waits (griddepcontrol.wait) for its stream predecessor before reading q or the pools
      r = launch_cascade_stream(a, p->pitem_first[kImplCascadeStream], p->pitem_count[kImplCascadeStream], st, true);
      c->n_kernels += 1;
    }
    if (r == cudaSuccess && p->pitem_count[kImplDenseTc] > 0) {
      if (!c->has_tmaps) return cudaErrorNotSupported;
      const bool first = p->pitem_count[kImplGeneric] == 0 && p->pitem_count[kImplCascadeMma] == 0 &&
                         p->pitem_count[kImplCascadeStream] == 0 && p->pitem_count[kImplDenseTf32] == 0;
      r = launch_dense_tc(a, p->pitem_first[kImplDenseTc], p->pitem_count[kImplDenseTc], c->tmap_k[layer],
                          c->tmap_v[layer], tmq, st, first);
      c->n_kernels += 1;
    }
    return r;
  };
  auto launch_merge_k = [&](bool pdl) -> cudaError_t {
    c->n_kernels += 1;
    if (c->cfg.dtype == GRANIKV_DTYPE_BF16 && c->cfg.head_dim == 128) return launch_merge_rows(a, p->merge_warps, s, pdl);
    return launch_merge(c->cfg.dtype, a, s, pdl);
  };
  const int32_t n_dense = p->pitem_count[kImplDenseTc], n_casc = p->pitem_count[kImplCascadeStream];
  const bool one_launch = p->concurrent && p->n_pitems > 0 && n_dense + n_casc == p->n_pitems &&
                          (n_dense == 0 || c->has_tmaps) && p->suffix_impl == kImplSuffixMma && p->n_sitems > 0;
  if (one_launch) {
    // the prefix items (dense and streaming cascade) and the suffix token-CTAs side by side in
    // one grid, then the merge: both chained to their stream predecessor by programmatic
    // dependent launch
    const CUtensorMap& tk = c->has_tmaps ? c->tmap_k[layer] : tmq;
    const CUtensorMap& tv = c->has_tmaps ? c->tmap_v[layer] : tmq;
    // the last n_tail suffix runs go to dense CTAs 0.. after their prefix piece (a plan has
    // them only when every prefix item is dense, one per dense CTA); on any other launch path
    // every run is a suffix CTA of its own
    const int32_t n_tail = p->n_tail <= n_dense && n_casc == 0 ? p->n_tail : 0;
    e = launch_prefix_suffix_tc(a, p->pitem_first[kImplDenseTc], n_dense, p->pitem_first[kImplCascadeStream], n_casc,
                                tk, tv, tmq, a.scta_begin, p->n_scta - n_tail, n_tail, s, true);
    c->n_kernels += 1;
    if (e == cudaSuccess && !p->fused) e = launch_merge_k(true);
  } else if (p->concurrent) {
    // fork: the suffix kernel runs on the auxiliary stream next to the prefix kernel (enqueued
    // first, so the longer prefix work starts first); join before anything else on the stream
    e = cudaEventRecord(c->ev_fork, s);
    if (e == cudaSuccess) e = launch_prefix(s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->aux, c->ev_fork, 0);
    if (e == cudaSuccess) e = launch_suffix(c->aux, false);
    if (e == cudaSuccess) e = cudaEventRecord(c->ev_join, c->aux);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, c->ev_join, 0);
    if (e == cudaSuccess && !p->fused) e = launch_merge_k(false);
  } else {
    e = launch_prefix(s);
    // the suffix kernel follows a prefix kernel of this call, the merge the suffix kernel
    const bool after_prefix = p->n_pitems > 0 && n_dense + n_casc > 0;
    if (e == cudaSuccess) e = launch_suffix(s, after_prefix && p->suffix_impl == kImplSuffixMma);
    if (e == cudaSuccess && !p->fused) {
      // the merge's stream predecessor is this call's suffix kernel, or its prefix kernel when
      // the step has no COLD tokens; the merge waits (griddepcontrol.wait) before it reads a
      // record, so it may be launched as a dependent of either
      e = launch_merge_k(p->n_sitems > 0 || p->n_pitems > 0);
    }
  }
  if (e == cudaErrorNotSupported) return GRANIKV_ERR_UNSUPPORTED;
  return cuda_status(e);
}

}  // namespace

extern "C" {

granikv_status granikv_decode_attention(granikv_ctx* c, int32_t layer, const void* q,
                                        const granikv_batch* bt, granikv_plan* p, void* o,
                                        float* lse, void* ws, size_t ws_bytes,
                                        granikv_stream_t stream) {
  return decode_attention_impl(c, layer, q, nullptr, nullptr, bt, p, o, lse, ws, ws_bytes, stream);
}

granikv_status granikv_decode_attention_append(granikv_ctx* c, int32_t layer, const void* q, const void* k_new,
                                               const void* v_new, const granikv_batch* bt, granikv_plan* p,
                                               void* o, float* lse, void* ws, size_t ws_bytes,
                                               granikv_stream_t stream) {
  if (!k_new || !v_new) return GRANIKV_ERR_INVALID;
  return decode_attention_impl(c, layer, q, k_new, v_new, bt, p, o, lse, ws, ws_bytes, stream);
}

// ---- prefill of a HOT slab ------------------------------------------------------------------

namespace {
// Workspace of a prefill over L_p tokens: the plan image only (one causal group whose requests
// are the slab's tokens; each query row has one partial state, which the dense kernel writes
// out as the final o and lse, so there are no records and no merge).
struct PrefillLayout {
  size_t off_group_req, off_req, off_pitems, total;
  int32_t row_blocks;
};
PrefillLayout prefill_layout(const granikv_ctx* c, int32_t L_p) {
  PrefillLayout l{};
  const int64_t rows = (int64_t)L_p * c->g;
  l.row_blocks = (int32_t)((rows + kDenseRows - 1) / kDenseRows);
  size_t off = align_up(sizeof(DevGroup), 16);
  l.off_group_req = off;
  off = align_up(off + sizeof(int32_t) * (size_t)L_p, 16);
  l.off_req = off;
  off = align_up(off + sizeof(DevReq) * (size_t)L_p, 16);
  l.off_pitems = off;
  off = align_up(off + sizeof(DevPrefixItem) * (size_t)l.row_blocks * c->cfg.n_kv, 256);
  l.total = off;
  return l;
}
}  // namespace

granikv_status granikv_prefill_workspace_size(granikv_ctx* c, int32_t L_p, size_t* bytes) {
  if (!c || !bytes || L_p <= 0) return GRANIKV_ERR_INVALID;
  *bytes = prefill_layout(c, L_p).total;
  return GRANIKV_OK;
}

granikv_status granikv_prefill_attention(granikv_ctx* c, int32_t layer, int32_t sid, const void* k_new,
                                         const void* v_new, const void* q, void* o, float* lse, void* ws,
                                         size_t ws_bytes, granikv_stream_t stream) {
  if (!c || !q || !o || !lse || !ws) return GRANIKV_ERR_INVALID;
  if (layer < 0 || layer >= c->cfg.n_layers) return GRANIKV_ERR_INVALID;
  if (sid < 0 || sid >= (int32_t)c->slabs.size() || !c->slabs[sid].live) return GRANIKV_ERR_INVALID;
  if ((k_new == nullptr) != (v_new == nullptr)) return GRANIKV_ERR_INVALID;
  if ((uintptr_t)ws % 256) return GRANIKV_ERR_INVALID;
  if (!has_device(c)) return GRANIKV_ERR_NO_DEVICE;
  if (c->cfg.dtype != GRANIKV_DTYPE_BF16 || c->cfg.head_dim != 128 || !c->has_tmaps) return GRANIKV_ERR_UNSUPPORTED;
  const int32_t L_p = c->slabs[sid].len;
  const PrefillLayout lay = prefill_layout(c, L_p);
  if (ws_bytes < lay.total) return GRANIKV_ERR_INVALID;
  if (k_new) {
    granikv_status st = granikv_hot_fill(c, layer, sid, k_new, v_new, stream);
    if (st != GRANIKV_OK) return st;
  }
  DeviceGuard dg(c->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  const int32_t n_kv = c->cfg.n_kv, n_q = c->cfg.n_q;

  // plan image: one group (the slab), request b = token b, one record per token; the CTAs of
  // the longest rows (the last row blocks, which read the most keys) first
  DevGroup gr{};
  gr.slab_off = c->slabs[sid].off;
  gr.L_p = L_p;
  gr.n_req = L_p;
  gr.req_begin = 0;
  gr.n_splits = 1;
  gr.tile = kDenseTile;
  gr.split_len = (L_p + kDenseTile - 1) / kDenseTile * kDenseTile;
  gr.n_long = 0;
  gr.backend = GRANIKV_BACKEND_DENSE;
  gr.impl = kImplDenseTc;
  gr.rows_per_cta = kDenseRows;
  gr.row_blocks = lay.row_blocks;
  gr.q_b0 = 0;
  gr.causal = 1;
  std::vector<unsigned char>& blob = c->prefill_blob;
  blob.assign(lay.total, 0);
  std::memcpy(blob.data(), &gr, sizeof(DevGroup));
  int32_t* greq = reinterpret_cast<int32_t*>(blob.data() + lay.off_group_req);
  DevReq* reqs = reinterpret_cast<DevReq*>(blob.data() + lay.off_req);
  for (int32_t b = 0; b < L_p; ++b) {
    greq[b] = b;
    reqs[b] = DevReq{b, 1, 1, 0};
  }
  DevPrefixItem* items = reinterpret_cast<DevPrefixItem*>(blob.data() + lay.off_pitems);
  int32_t n_items = 0;
  for (int32_t rb = lay.row_blocks - 1; rb >= 0; --rb)
    for (int32_t j = 0; j < n_kv; ++j) items[n_items++] = DevPrefixItem{0, j, rb, 0};
  unsigned char* wsb = static_cast<unsigned char*>(ws);
  ws_record(ws, 0, 0);  // the front no longer holds a decode plan's image
  cudaError_t e = cudaMemcpyAsync(wsb, blob.data(), blob.size(), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return GRANIKV_ERR_CUDA;
  c->n_copies += 1;

  AttnParams a{};
  a.q = q;
  a.o = o;
  a.lse = lse;
  a.kpool = c->kpool[layer];
  a.vpool = c->vpool[layer];
  a.n_slots = c->cfg.n_slots;
  a.n_hot = c->n_hot;
  a.B = L_p;
  a.n_q = n_q;
  a.n_kv = n_kv;
  a.d = c->cfg.head_dim;
  a.g = c->g;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->cfg.head_dim));
  a.groups = (const DevGroup*)wsb;
  a.group_req = (const int32_t*)(wsb + lay.off_group_req);
  a.reqs = (const DevReq*)(wsb + lay.off_req);
  a.pitems = (const DevPrefixItem*)(wsb + lay.off_pitems);
  a.n_pitems = n_items;
  a.n_records = 0;
  a.err = c->d_err;
  a.checks = c->checks;
  CUtensorMap tmq{};
  a.q_tma = encode_q_map(&tmq, q, L_p, n_q, c->g) ? 1 : 0;
  e = launch_dense_tc(a, 0, n_items, c->tmap_k[layer], c->tmap_v[layer], tmq, s, true);
  c->n_kernels += 1;
  return cuda_status(e);
}

// ---- checks ---------------------------------------------------------------------------------

granikv_status granikv_set_checks(granikv_ctx* c, int32_t on) {
  if (!c) return GRANIKV_ERR_INVALID;
  c->checks = on ? 1 : 0;
  return GRANIKV_OK;
}

granikv_status granikv_inject_stall(granikv_ctx* c, int32_t on) {
  if (!c) return GRANIKV_ERR_INVALID;
  c->inject_stall = on ? 1 : 0;
  return GRANIKV_OK;
}

granikv_status granikv_sync_status(granikv_ctx* c, granikv_stream_t stream) {
  if (!c) return GRANIKV_ERR_INVALID;
  if (!has_device(c)) return GRANIKV_ERR_NO_DEVICE;
  DeviceGuard dg(c->cfg.device);
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return GRANIKV_ERR_CUDA;
  int32_t h = 0;
  e = cudaMemcpy(&h, c->d_err, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return GRANIKV_ERR_CUDA;
  if (h != 0) {
    cudaMemset(c->d_err, 0, sizeof(int32_t));
    // a failed call may have left row tickets part-way: start the next call from zero
    if (c->last_tickets) cudaMemset(c->last_tickets, 0, c->last_tickets_bytes);
    return GRANIKV_ERR_DEVICE_CHECK;
  }
  return GRANIKV_OK;
}

granikv_status granikv_launch_count(granikv_ctx* c, int64_t* kernels, int64_t* copies) {
  if (!c) return GRANIKV_ERR_INVALID;
  if (kernels) *kernels = c->n_kernels;
  if (copies) *copies = c->n_copies;
  return GRANIKV_OK;
}

}  // extern "C"

namespace granikv {

int32_t granikv_internal_device(const granikv_ctx* c, int* device) {
  if (!c || !device) return GRANIKV_ERR_INVALID;
  if (!has_device(c)) return GRANIKV_ERR_NO_DEVICE;
  *device = c->cfg.device;
  return GRANIKV_OK;
}

void granikv_internal_forget_workspace(const void* ws) { ws_forget(ws); }

void granikv_internal_hot_if_released(const granikv_ctx* c, const int32_t* slabs, int32_t n,
                                      int64_t* largest_free, int32_t* free_ids) {
  std::vector<Extent> ext = c->free_ext;
  int32_t ids = 0;
  for (const Slab& s : c->slabs) ids += s.live ? 0 : 1;
  for (int32_t i = 0; i < n; ++i) {
    const Slab& s = c->slabs[slabs[i]];
    ext.push_back({s.off, s.len});
    ids += 1;
  }
  std::sort(ext.begin(), ext.end(), [](const Extent& a, const Extent& b) { return a.off < b.off; });
  int64_t best = 0, run_off = -1, run_len = 0;
  for (const Extent& e : ext) {
    if (run_off >= 0 && run_off + run_len == e.off) {
      run_len += e.len;
    } else {
      run_off = e.off;
      run_len = e.len;
    }
    best = std::max(best, run_len);
  }
  *largest_free = best;
  *free_ids = ids;
}

}  // namespace granikv
