/*
 * granikv.h -- C ABI of libgranikv: decode-step attention over an asymmetric HOT/COLD KV cache.
 *
 * Source of every operation: "GraniKV: Asymmetric Granularity KV-Cache Paging for Multi-Agent
 * Systems with Long Shared Prefix" (arXiv:2608.15584).  Section names below refer to that
 * paper's summary page and card page.
 *
 * Conventions
 * -----------
 *  - Every call returns a granikv_status.  No C++ exception or abort crosses this boundary.
 *  - The caller owns every device buffer that holds data: the per-layer K/V pools, q, o, lse,
 *    the per-request token tables, the per-request lengths and the workspace.  Pointers marked
 *    "device" must be device (or managed) memory of the context's device; "host" pointers
 *    must be host memory.
 *  - The library owns the pool metadata: the HOT extent list and slab table (host), the COLD
 *    free ring (device, allocated by granikv_create), and a device error word.
 *  - Calls that take a cudaStream_t are stream-ordered and asynchronous.  Errors that only
 *    the device can see (bounds checks, see granikv_set_checks) are latched in the error word
 *    and reported by granikv_sync_status.
 *  - A context is not thread-safe; use one per host thread or serialise calls.
 *
 * KV layout
 * ---------
 *  Each layer has one K pool and one V pool, each [n_slots, n_kv, head_dim] of the context's
 *  dtype, row-major (slot stride n_kv*head_dim elements).  Slots [0, n_hot) form the HOT pool
 *  and [n_hot, n_slots) the COLD pool, n_hot = floor(hot_fraction * n_slots)
 *  ("Limitations", static HOT/COLD pool fraction f_p, default 0.2).  A slot id means the same
 *  token position in every layer's pools.
 */
#ifndef GRANIKV_H
#define GRANIKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* granikv_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef int32_t granikv_status;
enum {
  GRANIKV_OK = 0,
  GRANIKV_ERR_INVALID = 1,        /* bad argument or descriptor; nothing was changed        */
  GRANIKV_ERR_NO_HOT_SPACE = 2,   /* no free HOT extent can hold the prefix (or slab table full) */
  GRANIKV_ERR_NO_COLD_SPACE = 3,  /* fewer free COLD slots than asked; nothing was popped    */
  GRANIKV_ERR_CUDA = 4,           /* a CUDA runtime call failed                              */
  GRANIKV_ERR_DEVICE_CHECK = 5,   /* a kernel's bounds check failed (see granikv_set_checks) */
  GRANIKV_ERR_UNSUPPORTED = 6,    /* shape or dtype this build has no kernel for             */
  GRANIKV_ERR_NO_DEVICE = 7,      /* the call needs device resources the context lacks       */
  GRANIKV_ERR_STATIC_WORKSPACE_TOO_SMALL = 8 /* the plan needs more than the built-in workspace */
};

enum { GRANIKV_DTYPE_F32 = 0, GRANIKV_DTYPE_BF16 = 1 };

/* Prefix backends ("3 GraniKV", dual attention backends).  Kernels per shape: bf16 with
 * head_dim 128 -- dense on tcgen05 (kind::f16, TMA-fed), cascade as a bandwidth kernel over whole
 * slot rows (g <= 128); fp32 with head_dim 32, 64, 96 or 128 -- dense on tcgen05 (kind::tf32 in
 * split precision, fp32-accurate), cascade on CUDA cores; any other shape -- both on CUDA cores. */
enum {
  GRANIKV_BACKEND_AUTO = 0,     /* per-group dispatch on M_eff >= M_sat                    */
  GRANIKV_BACKEND_DENSE = 1,    /* batched-GEMM prefix backend (tensor cores)              */
  GRANIKV_BACKEND_CASCADE = 2   /* prefix read once per step, bandwidth-bound backend      */
};

typedef struct granikv_ctx granikv_ctx;
typedef struct granikv_plan granikv_plan;

typedef struct granikv_config {
  int32_t n_layers;
  int32_t n_q;        /* query heads                                   */
  int32_t n_kv;       /* KV heads; n_q % n_kv == 0                      */
  int32_t head_dim;   /* d                                             */
  int32_t dtype;      /* GRANIKV_DTYPE_*: pools, q and o                */
  int32_t device;     /* CUDA device ordinal                           */
  int64_t n_slots;    /* slots per pool                                */
  double hot_fraction;/* f_p in (0, 1); 0 selects the default 0.2       */
  void* const* k_pool;/* host array [n_layers] of device pointers, 16-byte aligned */
  void* const* v_pool;/* host array [n_layers] of device pointers, 16-byte aligned */
  const int32_t* cold_init_order; /* host [n_slots - n_hot]: initial COLD free-ring content, a
                                     permutation of [n_hot, n_slots); NULL = ascending order   */
  int32_t m_sat;      /* dense iff M_eff >= m_sat; 0 selects the built-in GB300 fit       */
  int32_t max_slabs;  /* slab table size; 0 selects 1024                                  */
  int32_t max_batch;  /* largest B of any call; 0 selects 4096                            */
  int32_t host_only;  /* 1: create no device resources (HOT pool and dispatch only)       */
} granikv_config;

/* One decode step's batch.  Request b attends over its HOT prefix slab (if slab_id[b] >= 0)
 * followed by the seq_len[b] tokens listed in req_to_slot[b, 0:seq_len[b]].  A prefix that is
 * not in HOT is simply the head of that list (the paged fallback).
 * seq_len_dev (optional) lets one plan serve several decode steps, as a CUDA graph replayed
 * step after step needs: the plan is made for seq_len (the lengths the requests may reach, e.g.
 * the current ones plus a headroom), and each attention call reads the lengths the requests
 * have now from seq_len_dev (device [B], e.g. the suffix_len array granikv_cold_alloc keeps) and
 * attends over req_to_slot[b, 0:min(seq_len[b], seq_len_dev[b])]. */
typedef struct granikv_batch {
  int32_t B;
  const int32_t* slab_id;     /* host [B]: HOT slab of request b, or -1                   */
  const int32_t* seq_len;     /* host [B]: tokens of request b in its COLD token table     */
  const int32_t* req_to_slot; /* device [B, cap] int32: COLD slot of each token, row-major */
  int32_t cap;                /* row stride of req_to_slot                                 */
  const int32_t* seq_len_dev; /* device [B] int32 or NULL: the tokens that exist now       */
} granikv_batch;

typedef struct granikv_group_info {
  int32_t slab_id;
  int32_t n_requests;
  int32_t m_eff;      /* n_requests * n_q / n_kv                        */
  int32_t backend;    /* GRANIKV_BACKEND_DENSE or GRANIKV_BACKEND_CASCADE */
  int32_t L_p;
  int32_t n_splits;   /* pieces the prefix is split into along L_p      */
  int64_t slot_offset;
} granikv_group_info;

/* Text for a status code (static storage). */
const char* granikv_status_string(granikv_status s);

/* Library version as major*10000 + minor*100 + patch. */
int32_t granikv_version(void);

/* Create a context.  Allocates the COLD free ring and a few small device buffers with
 * cudaMalloc on cfg->device (none when host_only).  The pools stay caller-owned.
 * "3 GraniKV", asymmetric KV-cache paging; "Limitations", static pool fraction. */
granikv_status granikv_create(const granikv_config* cfg, granikv_ctx** out);
granikv_status granikv_destroy(granikv_ctx* ctx);

/* ---- HOT pool ("B.10 Cross-pool admission and promotion policy"; "B.8 Multi-prefix
 * sensitivity": first-fit packing of mixed slab sizes; card page: one slab per prefix node).
 * Host only, no device access. ------------------------------------------------------------- */

/* Reserve a contiguous slab of L_p slots: the lowest-offset free extent that can hold it,
 * carved from its start.  Returns the lowest unused slab id and the slab's first slot.
 * GRANIKV_ERR_NO_HOT_SPACE if no extent is large enough or the slab table is full; the caller
 * then stores the prefix in COLD (admission fallback).  Existing slabs never move. */
granikv_status granikv_hot_alloc(granikv_ctx* ctx, int32_t L_p, int32_t* slab_id,
                                 int64_t* slot_offset);
/* Release a slab; its extent merges with free neighbours. */
granikv_status granikv_hot_free(granikv_ctx* ctx, int32_t slab_id);
/* Offset and length of a live slab. */
granikv_status granikv_hot_info(granikv_ctx* ctx, int32_t slab_id, int64_t* slot_offset,
                                int32_t* L_p);
/* Number of HOT slots, and the largest free extent. */
granikv_status granikv_hot_stats(granikv_ctx* ctx, int64_t* n_hot, int64_t* largest_free);
/* Copy a prefix's K/V ([L_p, n_kv, head_dim], device, contiguous) into a slab of one layer.
 * Stream-ordered device-to-device copies (granikv_prefill_attention does the same copy and then
 * the prefix's causal attention; the projection that produces K/V is outside the library). */
granikv_status granikv_hot_fill(granikv_ctx* ctx, int32_t layer, int32_t slab_id,
                                const void* k, const void* v, granikv_stream_t stream);

/* ---- COLD pool ("1 Introduction" and "3 GraniKV": a token-level pool, page size 1, for
 * suffix and decoded tokens; card page: a token-level free list). ------------------------- */

/* Pop n_new[b] slots for each request b from the free ring, in request order: request b gets
 * ring entries head + sum(n_new[0:b]) ..., appended to req_to_slot[b, suffix_len[b]:] and
 * suffix_len[b] += n_new[b].  The popped slots, in the same order, are also written to
 * slots_out (device [sum n_new], may be NULL) for granikv_cold_append.
 *   n_new:       host [B], each >= 0
 *   req_to_slot: device [B, cap] int32;  suffix_len: device [B] int32
 * All-or-nothing: GRANIKV_ERR_NO_COLD_SPACE (checked on the host, nothing popped) when fewer
 * slots are free than asked.  A row that would pass cap is a device check failure. */
granikv_status granikv_cold_alloc(granikv_ctx* ctx, const int32_t* n_new, int32_t B,
                                  int32_t* req_to_slot, int32_t* suffix_len, int32_t cap,
                                  int32_t* slots_out, granikv_stream_t stream);
/* Return n slots (device [n]) to the tail of the free ring, in the given order.
 * GRANIKV_ERR_INVALID if that would hold more than the pool's size. */
granikv_status granikv_cold_free(granikv_ctx* ctx, const int32_t* slots, int32_t n,
                                 granikv_stream_t stream);
/* Free COLD slots (host mirror of the ring's fill). */
granikv_status granikv_cold_free_count(granikv_ctx* ctx, int64_t* n_free);
/* granikv_cold_alloc with n_new[b] = n for every request b < B (decode steps: n = 1), safe to
 * capture in a CUDA graph and replay: the kernel reads the ring position from device memory,
 * checks there that n*B slots are free (otherwise it pops nothing and latches
 * GRANIKV_ERR_DEVICE_CHECK, reported by granikv_sync_status) and moves it; slots_out (device
 * [n*B], may be NULL) receives the slots in request order.  The host's copy of the ring
 * position is advanced as if the call ran once, so after capturing or replaying graphs that
 * contain it, call granikv_cold_sync before the next granikv_cold_alloc or granikv_cold_free. */
granikv_status granikv_cold_alloc_uniform(granikv_ctx* ctx, int32_t n, int32_t B, int32_t* req_to_slot,
                                          int32_t* suffix_len, int32_t cap, int32_t* slots_out,
                                          granikv_stream_t stream);
/* Synchronise the stream and take the host's copy of the COLD ring position from the device. */
granikv_status granikv_cold_sync(granikv_ctx* ctx, granikv_stream_t stream);
/* Scatter N new tokens' K/V ([N, n_kv, head_dim] each, device) into one layer's pools at
 * slots[i] (device [N]).  A slot outside [n_hot, n_slots) is a device check failure. */
granikv_status granikv_cold_append(granikv_ctx* ctx, int32_t layer, const void* k_new,
                                   const void* v_new, const int32_t* slots, int32_t N,
                                   granikv_stream_t stream);

/* ---- prefix index ("2 Related Work", prefix-aware serving: a radix tree over token-id
 * sequences with reference-counted nodes; card page: one HOT slab per radix-tree prefix node;
 * "B.10 Cross-pool admission and promotion policy": HOT first, COLD fallback, no demotion).
 * Host only, no device access; the HOT slabs come from the context's HOT pool.
 *
 * A prefix is used whole: a request reuses the deepest admitted prefix whose full token
 * sequence starts its own, and attends over all of it (L_p = its length).  Nested prefixes each
 * own a slab of their full length.  Prefix handles are never reused.  The LRU clock advances
 * on insert, on a match that takes a reference, on acquire and on release.  An index, like its
 * context, is not thread-safe. -------------------------------------------------------------- */

typedef struct granikv_index granikv_index;

typedef struct granikv_prefix_info {
  int32_t prefix_id;   /* handle (>= 0), or -1 when a match found nothing                */
  int32_t length;      /* L_p, tokens                                                     */
  int32_t slab_id;     /* HOT slab, or -1 when the prefix was placed in COLD              */
  int32_t refcount;    /* requests holding the prefix                                     */
  int64_t slot_offset; /* first HOT slot of the slab, or -1                               */
} granikv_prefix_info;

/* An empty index over ctx's HOT pool.  ctx must outlive the index.  Destroying the index
 * returns the slabs of its HOT prefixes to the pool (a COLD prefix's slots are the caller's). */
granikv_status granikv_index_create(granikv_ctx* ctx, granikv_index** out);
granikv_status granikv_index_destroy(granikv_index* idx);
/* Deepest admitted prefix of tokens (host [n]); out->prefix_id = -1 when none.  acquire = 1
 * takes a reference on the prefix found. */
granikv_status granikv_index_match(granikv_index* idx, const int32_t* tokens, int32_t n,
                                   int32_t acquire, granikv_prefix_info* out);
/* Admit tokens (host [n], n >= 1) as a prefix with refcount 0.  If exactly this sequence is
 * already admitted, that prefix is returned and nothing else changes.  Otherwise HOT first: a
 * first-fit slab of n slots.  If none is free, unreferenced HOT prefixes are evicted, least
 * recently used first, until the slab fits -- but only if evicting all of them would make it
 * fit; else nothing is evicted and the prefix is placed in COLD (slab_id = -1: the caller
 * stores its K/V in COLD slots).  Referenced prefixes never move or leave HOT.
 *   evicted: host [max_evicted] or NULL; receives the handles evicted, n_evicted their number
 *            (may be NULL).  GRANIKV_ERR_INVALID, with nothing changed, if evicted is given and
 *            more than max_evicted would go. */
granikv_status granikv_index_insert(granikv_index* idx, const int32_t* tokens, int32_t n,
                                    granikv_prefix_info* out, int32_t* evicted,
                                    int32_t max_evicted, int32_t* n_evicted);
/* Take or drop one reference.  GRANIKV_ERR_INVALID for an unknown handle, or a release of a
 * prefix nobody holds. */
granikv_status granikv_index_acquire(granikv_index* idx, int32_t prefix_id);
granikv_status granikv_index_release(granikv_index* idx, int32_t prefix_id);
/* Remove an unreferenced prefix; a HOT one's slab returns to the pool.  GRANIKV_ERR_INVALID for
 * an unknown or referenced handle. */
granikv_status granikv_index_remove(granikv_index* idx, int32_t prefix_id);
granikv_status granikv_index_info(granikv_index* idx, int32_t prefix_id, granikv_prefix_info* out);
/* Live prefixes, how many of them are in HOT, and tree nodes (root not counted: a node marks
 * where an admitted prefix ends or where two of them diverge). */
granikv_status granikv_index_stats(granikv_index* idx, int32_t* n_prefixes, int32_t* n_hot,
                                   int32_t* n_nodes);

/* ---- per-step dispatch ("3 GraniKV", per-step dispatch; "B.4 Per-Step Dispatch Trace";
 * "B.8": class-local dense batching).  Host only, no device access. ------------------------ */

granikv_status granikv_plan_create(granikv_ctx* ctx, granikv_plan** out);
granikv_status granikv_plan_destroy(granikv_plan* plan);
/* Group the batch's requests by HOT slab, compute M_eff = B_g * n_q / n_kv per group, choose
 * DENSE iff M_eff >= M_sat (unless a backend is forced), and lay out the step's work: prefix
 * splits, suffix chunks and partial-state records.  GRANIKV_ERR_INVALID for an unknown slab,
 * a request with neither prefix nor tokens, seq_len > cap, or B > max_batch.  The plan keeps
 * the dispatcher's working arrays, so dispatching into the same plan step after step allocates
 * host memory only while batches grow, and when a batch has the same slab ids as the plan's
 * last one (the same requests, lengths grown) its grouping and prefix work items are reused;
 * the plan is the same as a fresh dispatch of the batch would make.  A plan, like its context,
 * is used by one thread at a time. */
granikv_status granikv_dispatch(granikv_ctx* ctx, const granikv_batch* batch, granikv_plan* plan);
granikv_status granikv_plan_num_groups(const granikv_plan* plan, int32_t* n_groups);
granikv_status granikv_plan_group(const granikv_plan* plan, int32_t i, granikv_group_info* out);
/* How the plan runs: concurrent = 1 when the prefix and suffix work share the GPU side by side
 * (one grid, or two kernels on two streams), 0 when they run one after another; the number of
 * prefix CTAs and of suffix CTAs it launches. */
granikv_status granikv_plan_schedule(const granikv_plan* plan, int32_t* concurrent, int32_t* prefix_ctas,
                                     int32_t* suffix_ctas);
/* Diagnostics of the schedule (no counterpart in the paper).  The plan's suffix runs (token-CTA
 * work lists, one KV-head group's; the generic suffix kernel: its work items) and, of them, the
 * tail runs: when the step runs as one grid in which every prefix CTA is dense and the suffix
 * side is estimated to end last, the last tail_runs runs are taken by dense CTAs 0.. after
 * their prefix piece (granikv_plan_schedule counts the suffix CTAs launched, without them).
 * Either output pointer may be NULL.  GRANIKV_ERR_INVALID for a plan not yet dispatched. */
granikv_status granikv_plan_suffix_runs(const granikv_plan* plan, int32_t* runs, int32_t* tail_runs);
/* Diagnostics (no counterpart in the paper): the dense kernel's L2 read-ahead (in tiles, 0 for
 * none) the plan's launches use; see granikv_set_dense_l2_ahead.  GRANIKV_ERR_INVALID for a
 * NULL output or a plan not yet dispatched. */
granikv_status granikv_plan_dense_l2_ahead(const granikv_plan* plan, int32_t* tiles);
/* Diagnostics (no counterpart in the paper): copy the plan's device image -- the work list that
 * granikv_decode_attention copies to the front of the workspace -- into host memory.  *size
 * receives its length; nothing is copied when cap is smaller (then GRANIKV_ERR_INVALID). */
granikv_status granikv_plan_image(const granikv_plan* plan, void* out, size_t cap, size_t* size);
/* Workspace bytes granikv_decode_attention needs for this plan (256-byte aligned pointer). */
granikv_status granikv_workspace_size(granikv_ctx* ctx, const granikv_plan* plan, size_t* bytes);

/* Prefix/suffix concurrency of the tensor-core path: when on (the default), the prefix and
 * suffix work run side by side -- in one grid (dense prefix CTAs and suffix token-CTAs, one per
 * SM) when every prefix group is dense, else as two kernels, the suffix one on a library-owned
 * stream forked from and joined back into the caller's stream.  The automatic share (below) may
 * still pick the one-after-the-other plan when its estimate is lower (granikv_plan_schedule
 * tells which).  prefix_sm_share in (0, 1) splits the SMs: the prefix work list is sized
 * for that share and the suffix gets the SMs the prefix CTAs leave; 0 (the default) picks the
 * share from the step's estimated prefix and suffix work; 1 sizes both for all SMs, and the
 * suffix fills SMs as the prefix frees them.  When off, the prefix, suffix and merge kernels
 * run one after another on the caller's stream.  GRANIKV_ERR_INVALID for a share outside
 * [0, 1].  Takes effect at the next granikv_dispatch. */
granikv_status granikv_set_concurrency(granikv_ctx* ctx, int32_t on, float prefix_sm_share);

/* Merge strategy of the tensor-core path ("2 Related Work": partial states merged by
 * log-sum-exp).  0 (the default): a merge kernel runs after the prefix and suffix kernels.
 * 1: no merge kernel; every (request, head) row counts its producers with a ticket and the
 * producer that finishes last merges the row.  Takes effect at the next granikv_dispatch. */
granikv_status granikv_set_fused_merge(granikv_ctx* ctx, int32_t on);

/* Scheduling knob (no counterpart in the paper): L2 read-ahead of the dense tensor-core prefix
 * kernel.  When a CTA refills a slot of its shared-memory K (or V) ring with tile i of its
 * prefix piece, it also requests tile i + tiles into L2 (a bulk-tensor L2 prefetch: no data
 * moves to the SM, results are unchanged).  -1 (the default): two tiles when the step runs as
 * one grid whose prefix side is estimated to finish after its suffix side and whose suffix side
 * reads at least as many bytes, else none; 0: never; 1-64: that many tiles for every dense
 * decode launch.  GRANIKV_ERR_INVALID outside [-1, 64].  Takes effect at the next
 * granikv_dispatch. */
granikv_status granikv_set_dense_l2_ahead(granikv_ctx* ctx, int32_t tiles);

granikv_status granikv_set_msat(granikv_ctx* ctx, int32_t m_sat);
granikv_status granikv_get_msat(granikv_ctx* ctx, int32_t* m_sat);
granikv_status granikv_force_backend(granikv_ctx* ctx, int32_t backend);

/* ---- decode-step attention ("2 Related Work", prefix-suffix attention: prefix and suffix
 * partial attentions merged by log-sum-exp; "3 GraniKV", dual attention backends). -------- */

/* o[b, h, :] and lse[b, h] of softmax attention (scale 1/sqrt(head_dim), natural-log lse) of
 * query q[b, h, :] over request b's HOT prefix slab followed by its COLD tokens, using KV
 * head h / (n_q / n_kv) of layer `layer`.
 *   q: device [B, n_q, head_dim] (dtype);  o: device [B, n_q, head_dim] (dtype);
 *   lse: device [B, n_q] float32;  workspace: device, >= granikv_workspace_size bytes,
 *   256-byte aligned, not touched by the caller between calls that share a plan.
 * plan: from granikv_dispatch on this batch; NULL runs the dispatcher into the context's own
 * plan.  Its work list is copied into the workspace on first use with that workspace, so to
 * capture the call in a CUDA graph, make one call with that plan and workspace first: the
 * captured call then holds only the launches (see granikv_batch.seq_len_dev for replaying one
 * plan over several steps). */
granikv_status granikv_decode_attention(granikv_ctx* ctx, int32_t layer, const void* q,
                                        const granikv_batch* batch, granikv_plan* plan,
                                        void* o, float* lse, void* workspace, size_t ws_bytes,
                                        granikv_stream_t stream);

/* granikv_decode_attention with this step's COLD append fused in: row b of k_new and v_new
 * (device [B, n_kv, head_dim], 16-byte aligned) is the K and V of request b's newest token,
 * the last one of its COLD list (req_to_slot[b, n-1] with n = seq_len_dev[b] when given, else
 * seq_len[b]; its slot allocated already, e.g. by granikv_cold_alloc).  The call attends with
 * those rows and writes them to that slot of this layer's pools, so it equals granikv_cold_append
 * of the rows followed by granikv_decode_attention, one launch fewer.  GRANIKV_ERR_INVALID if a
 * request has no COLD token or k_new/v_new are not 16-byte aligned. */
granikv_status granikv_decode_attention_append(granikv_ctx* ctx, int32_t layer, const void* q,
                                               const void* k_new, const void* v_new,
                                               const granikv_batch* batch, granikv_plan* plan, void* o,
                                               float* lse, void* workspace, size_t ws_bytes,
                                               granikv_stream_t stream);
/* Decode attention without a caller workspace.  The paper has no counterpart: this is for
 * callers that cannot allocate device memory for a workspace, such as a serving engine that has
 * already reserved nearly all of the GPU's memory for its own pools and allocator, or a plain C
 * host that only holds pointers to buffers someone else owns.  It computes exactly what
 * granikv_decode_attention computes, using a workspace that lives in a file-scope device array
 * of the library (16 MiB per GPU, held by every GPU that loads the library until the process
 * exits).  It allocates nothing.
 *   plan:  required (from granikv_dispatch on this batch); no internal dispatch.
 *   q, o, lse, batch: as for granikv_decode_attention.
 * Errors: GRANIKV_ERR_STATIC_WORKSPACE_TOO_SMALL when granikv_workspace_size(plan) exceeds
 * 16 MiB (nothing is enqueued); otherwise as granikv_decode_attention.
 * The first call on each device looks up the array's device address (with that device made
 * current for the lookup).  All calls on a device
 * share the one array, and each call re-copies its work list and re-zeroes its merge tickets, so
 * calls that may overlap on the GPU (different streams, different threads) race and must be
 * ordered by the caller. */
granikv_status granikv_decode_attention_static(granikv_ctx* ctx, int32_t layer, const void* q,
                                               const granikv_batch* batch, granikv_plan* plan,
                                               void* o, float* lse, granikv_stream_t stream);

/* ---- prefill of a HOT slab ("2 Related Work", prefix-aware serving: a cached prefix skips
 * prefill for its matched tokens, so a prefix is prefilled once, when it is admitted; card
 * page: the HOT slab stores the prefix's K_p contiguously, which batched prefix kernels assume
 * and paged engines do not provide). ---------------------------------------------------- */

/* Causal self-attention of a HOT prefix's own L_p tokens over its slab, in one layer: query
 * token t (t < L_p) attends slab keys [0, t], with the softmax scale 1/sqrt(head_dim) and KV
 * head h / (n_q/n_kv) for query head h, as decode attention.
 *   k_new, v_new: device [L_p, n_kv, head_dim] or both NULL; when given they are first copied
 *                 into the slab (the prefill writes the contiguous K_p/V_p), stream-ordered
 *   q:   device [L_p, n_q, head_dim];  o: device [L_p, n_q, head_dim] (context dtype)
 *   lse: device [L_p, n_q] fp32, natural log
 *   ws:  device workspace of granikv_prefill_workspace_size(L_p) bytes, 256-byte aligned
 * L_p is the slab's length.  Runs on the tensor-core dense kernel alone (one CTA per 128 query
 * rows and KV head, keys up to the rows' diagonal, o and lse written directly).
 * GRANIKV_ERR_UNSUPPORTED unless the dtype is bf16 and head_dim is 128. */
granikv_status granikv_prefill_attention(granikv_ctx* ctx, int32_t layer, int32_t slab_id,
                                         const void* k_new, const void* v_new, const void* q, void* o,
                                         float* lse, void* workspace, size_t ws_bytes,
                                         granikv_stream_t stream);
granikv_status granikv_prefill_workspace_size(granikv_ctx* ctx, int32_t L_p, size_t* bytes);

/* ---- checks -------------------------------------------------------------------------- */

/* 1: kernels bounds-check slot ids, slab ranges and table rows, skip bad accesses and latch
 * GRANIKV_ERR_DEVICE_CHECK (no trap, no assert).  Default 1 for alloc/append, which are cheap;
 * the attention kernels check when on. */
granikv_status granikv_set_checks(granikv_ctx* ctx, int32_t on);
/* Test hook for the failure path (no counterpart in the paper): when on, the next
 * granikv_decode_attention call's first suffix token-CTA withholds the copies of its first
 * tile, so that CTA's consumers' bounded wait (2 s) expires.  The CTA then raises its abort
 * flag, waits for the copies it did issue, and exits; the call latches
 * GRANIKV_ERR_DEVICE_CHECK (reported by granikv_sync_status), and the context stays usable for
 * the next call.  Applies to one call of the bf16 tensor-core suffix path; 0 cancels it. */
granikv_status granikv_inject_stall(granikv_ctx* ctx, int32_t on);
/* Synchronise the stream and report (and clear) the device error word. */
granikv_status granikv_sync_status(granikv_ctx* ctx, granikv_stream_t stream);
/* Kernels (and host-to-device plan or offset copies) this context has enqueued since it was
 * created: the count a caller uses to attribute device work to the library. */
granikv_status granikv_launch_count(granikv_ctx* ctx, int64_t* kernels, int64_t* copies);

#ifdef __cplusplus
}
#endif
#endif /* GRANIKV_H */
