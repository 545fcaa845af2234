/*
 * ess.h - C ABI of the GB300 sparse-decode library with a host-resident
 * MLA latent cache.
 *
 * One decode layer of DSA-style sparse attention whose latent cache lives
 * in pinned host memory:
 *   (a1) lightning-indexer scores over the GPU-resident indexer cache,
 *   (a2) exact top-k, (a3) hit/miss resolution against the token->slot
 *   reverse index cache_slots and the miss union over MTP ways, (a4) LRU
 *   victim choice and state rewrite with copy triples, (a5) sparse
 *   absorbed-MLA attention whose row gather forks per row: hits from the
 *   HBM hot pool, misses straight from pinned host memory, (a6) a separate
 *   miss-staging copy, per-step counters, and the decode append of each
 *   step's new token (a device ring of two pages, written back to the host
 *   copy a page at a time).
 *
 * Sources (web pages on latent-cache offload for DSA sparse decode):
 *   [FO]  hwcomputing.csdn.net, analysis of FlashOffloading
 *         - "decode side (1)": cache_slots, the five-step steady-state flow,
 *           the MTP3 miss union, LIM and its worked example (Figure 4);
 *         - "decode side (2)": CopySFA, the gather that forks on hit/miss;
 *         - "architecture": one host master copy, paged by request, layer
 *           and token block behind a block table; a hot cache of C slots
 *           and two tail blocks for the new KV (Figure 2).
 *   [ESS] foosynaptic tech notes, "ESS: Latent-Cache Offload": the indexer
 *         cache stays on the GPU and scores every position; the latent
 *         entry is c^KV[512] + k^R[64]; a GPU sparse pool under LRU.
 *   [DEP] cloud.baidu.com deployment article, "monitoring": hit rate and
 *         link utilisation counters.
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device addresses; "pinned host" pointers come
 *     from cudaHostAlloc / cudaHostRegister and stay valid while bound.
 *   - The caller owns every buffer it passes, including the device
 *     workspace given to ess_pool_create.  The library owns only the opaque
 *     handle and never calls cudaMalloc.
 *   - Calls that take a stream are asynchronous on that stream.  Errors the
 *     host can detect are returned at once and nothing is launched.  Errors
 *     found on the device (bounds checks, capacity, a wait that timed out)
 *     are recorded in a device status word and returned by ess_pool_poll.
 *     No kernel traps or asserts.
 *   - A pool is not thread-safe.  Calls on one pool must be ordered on one
 *     stream (or ordered by the caller with events); they share scratch.
 *   - Layouts are row-major, the last index fastest.  B = batch, M = MTP
 *     ways, T = max_T, k = top-k, C = hot-pool slots per request, H_I =
 *     indexer heads, H = MLA heads, D = latent_dim + rope_dim = 576.
 */
#ifndef ESS_H
#define ESS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ess_pool ess_pool;
/* A cudaStream_t passed as an opaque pointer (NULL = the legacy stream). */
typedef void* ess_stream_t;

typedef enum {
  ESS_OK = 0,
  ESS_ERR_INVALID_ARG = 1,   /* bad pointer, size, layer or layout            */
  ESS_ERR_CAPACITY = 2,      /* the miss union cannot fit the C slots        */
  ESS_ERR_UNSUPPORTED = 3,   /* shape/dtype outside what the kernels handle  */
  ESS_ERR_OOM = 4,           /* the workspace is smaller than required       */
  ESS_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed            */
  ESS_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up           */
  ESS_ERR_DEVICE_CHECK = 7   /* a device-side bounds check failed            */
} ess_status;

enum { ESS_FP8_E4M3 = 0, ESS_BF16 = 1 };
/* FUSED: the attention kernel reads misses from host memory and writes them
 * to their pool slot in the same pass ([FO] "decode side (2)", CopySFA).
 * STAGED: a separate copy kernel moves the misses first ([FO] "decode side
 * (1)", step 5), then attention reads every row from the pool. */
enum { ESS_MISS_FUSED = 0, ESS_MISS_STAGED = 1 };

typedef struct {
  int32_t n_layers;    /* layers held by this pool                            */
  int32_t batch;       /* B requests                                          */
  int32_t max_T;       /* T: context capacity per request, a multiple of page */
                       /* and of 4                                            */
  int32_t C;           /* hot-pool slots per request and layer ([FO] C_b)     */
  int32_t page;        /* host page size in tokens (block-table granularity)  */
  int32_t k;           /* top-k per way ([FO]: k = 2048)                      */
  int32_t mtp;         /* M ways per step, 1..4 ([FO]: MTP3 = 4 ways), as far */
                       /* as one CTA's shared memory allows (see below)      */
  int32_t idx_heads;   /* H_I                                                 */
  int32_t idx_dim;     /* d_I; a key row must be 128 bytes                    */
  int32_t idx_dtype;   /* ESS_FP8_E4M3 (d_I = 128) or ESS_BF16 (d_I = 64)     */
  int32_t mla_heads;   /* H, 1..128                                           */
  int32_t latent_dim;  /* 512 ([ESS]: c^KV[512])                              */
  int32_t rope_dim;    /* 64  ([ESS]: k^R)                                    */
  float sm_scale;      /* softmax scale applied to q . row                   */
  int32_t miss_mode;   /* ESS_MISS_FUSED or ESS_MISS_STAGED                   */
} ess_config;

/* Counters accumulated per layer since the last read with reset ([DEP]
 * "monitoring": hit rate and link traffic). */
typedef struct {
  int64_t steps;        /* decode steps run on the layer (per request)     */
  int64_t hits;         /* selected rows found in the pool, summed over ways */
  int64_t misses;       /* selected rows not resident, summed over ways    */
  int64_t union_size;   /* |U|: distinct rows selected by any way          */
  int64_t miss_rows;    /* |Miss|: distinct rows moved from host           */
  int64_t miss_bytes;   /* miss_rows * D * 2                               */
  int64_t guided;       /* steps (per request) whose top-k read only the
                         * tokens the indexer flagged at or above the
                         * previous step's cut less one bin               */
  int64_t fine_cuts;    /* ways of those steps whose cut came from the
                         * indexer's fine histogram (8 more key bits)     */
} ess_stats;

/* Human-readable name of a status code (static storage). */
const char* ess_status_string(ess_status s);

/* Bytes of device workspace that ess_pool_create needs for cfg.
 * Covers, per layer: cache_slots [B][T] int32, slot_token [B][C] int32,
 * last_used [B][C] int32, step [B] int32, the hot pool [B][C][D] bf16, the
 * ring of appended rows [B][2 * page][D] bf16 and counters; plus scratch
 * shared by the layers (scores, selection lists, attention partials,
 * staging for ess_step_host).
 * A config whose kernels would need more shared memory per CTA than the GPU
 * has (227 KiB) is refused with ESS_ERR_UNSUPPORTED.  The indexer fits every
 * width up to 4 ways x 64 heads (its key ring shortens to make room for the
 * queries and one 16 KiB score histogram per way); the selection kernel's
 * per-CTA lists grow with min(max_T / 8, mtp * k), so 4 ways at k = 2048 fit
 * up to max_T = 32768 (the pages' MTP3 at the V3.2 shape) but not at 65536.
 * Errors: ESS_ERR_INVALID_ARG / ESS_ERR_UNSUPPORTED for a bad cfg. */
ess_status ess_pool_device_bytes(const ess_config* cfg, size_t* bytes);

/* Create a pool on the current CUDA device inside a caller-owned device
 * workspace (at least ess_pool_device_bytes, 256-byte aligned).  Every layer
 * starts empty (cache_slots = -1, slot_token = -1, last_used = -1, step 0):
 * the first step fills the pool from host memory ([FO] "decode side (1)",
 * first fill).  Initialisation is synchronous.  Requires
 * C >= min(mtp * k, max_T) so the miss union always fits. */
ess_status ess_pool_create(const ess_config* cfg, void* dev_workspace, size_t ws_bytes,
                           ess_pool** out);

/* Release the handle (the caller frees the workspace). */
ess_status ess_pool_destroy(ess_pool* pool);

/* Allocate pinned host memory for a latent cache, mapped into the device
 * address space (the kernels read miss rows from it directly) and usable from
 * every device.  The memory is zero-filled.  Release it with ess_host_free.
 * Errors: ESS_ERR_OOM (the allocation failed). */
ess_status ess_host_alloc(size_t bytes, void** out);

/* Free memory from ess_host_alloc. */
ess_status ess_host_free(void* ptr);

/* Bind the inputs of one layer ([FO] "architecture": host master copy
 * behind a block table; [ESS]: indexer cache resident on the GPU).
 *   host_latent  pinned host, [B][T][D] bf16, physical rows: logical token t
 *                of request b is row page_table[b][t / page] * page + t % page
 *   page_table   device int32 [B][T / page], or NULL for the identity map
 *   idx_keys     device [B][T][128 bytes]: e4m3 keys (d_I = 128) or bf16
 *                keys (d_I = 64)
 *   idx_scale    device float [B][T] per-token key scale, or NULL for 1.0
 *   T_host       host int32 [B], tokens per request, 0 <= T_b <= max_T
 * Buffers must stay valid while the layer is used.  The library changes them
 * only through ess_append, which writes rows t >= T_b of idx_keys, idx_scale
 * and (once a page of new tokens is complete) host_latent. */
ess_status ess_pool_bind_layer(ess_pool* pool, int layer, const void* host_latent,
                               const int32_t* page_table, const void* idx_keys,
                               const float* idx_scale, const int32_t* T_host);

/* ess_pool_bind_layer with the host master copy held as compact 656-byte
 * rows (the format of ess_compact_rows): 512 e4m3 latent values in four tiles
 * with power-of-two float32 scales, then the 64 RoPE values as bf16
 * ("ESS: Latent-Cache Offload", the ~656-byte FlashTrans + UVA transfers).
 *   host_compact  pinned host [B][T][656] bytes, physical rows through the
 *                 page table as for ess_pool_bind_layer
 * A miss moves 656 bytes over the host link instead of 1152: the gathers
 * (fused attention, staging, and the reload of ess_pool_set_state) widen the
 * row to bf16 on the way, exactly (a code times a power of two is a bf16
 * value), and the hot pool keeps bf16 rows, so hits and the attention
 * arithmetic are unchanged.  ess_append is refused (ESS_ERR_UNSUPPORTED) on
 * such a layer.  Errors as ess_pool_bind_layer. */
ess_status ess_pool_bind_layer_compact(ess_pool* pool, int layer, const void* host_compact,
                                       const int32_t* page_table, const void* idx_keys,
                                       const float* idx_scale, const int32_t* T_host);

/* Empty the hot pool of a layer again (asynchronous on stream). */
ess_status ess_pool_reset(ess_pool* pool, int layer, ess_stream_t stream);

/* Decode append: the newest token of every request joins the layer, so T_b
 * grows by one for each b ([FO] "architecture" and its Figure 2: besides the
 * hot cache the device keeps two tail blocks that take the new KV; the host
 * keeps the authoritative copy, paged behind the block table).
 *   latent_row  device bf16 [B][D], 16-byte aligned: the new token's c^KV|k^R
 *   key_row     device [B][128 bytes], 16-byte aligned: its indexer key, in
 *               the encoding of the bound idx_keys
 *   key_scale   device float [B]: its key scale; required when the layer
 *               was bound with idx_scale, ignored otherwise
 * Token t = T_b is written to row t of idx_keys (and idx_scale) and to a
 * device ring of two pages per request; when t completes a page, that page's
 * appended rows are written to their host_latent rows through the page table.
 * Until then (and for one more page) the gathers read them from the ring.  A
 * new token is not in the hot pool (cache_slots stays -1): the first step
 * that selects it loads it into a slot like any other miss.  Call it before
 * the step that should see the token.  Asynchronous on stream (one kernel).
 * Errors: ESS_ERR_CAPACITY, launching nothing, when a request is already at
 * max_T; ESS_ERR_INVALID_ARG for an unbound layer, a null or misaligned
 * row, or a missing key_scale; ESS_ERR_UNSUPPORTED on a layer bound with
 * compact rows. */
ess_status ess_append(ess_pool* pool, int layer, const void* latent_row, const void* key_row,
                      const float* key_scale, ess_stream_t stream);

/* (a1) Indexer scores ([ESS]: score all positions; formula
 * S[b][m][t] = fl32(scale[b][t] * sum_h w[b][m][h] * ReLU(q[b][m][h] . k[b][t]))).
 *   q_idx   device [B][M][H_I][128 bytes] (same encoding as the keys),
 *           16-byte aligned
 *   w       device float [B][M][H_I], 16-byte aligned (M * H_I a multiple of 4)
 *   scores  device float [B][M][T]; entries t >= T_b are not written */
ess_status ess_indexer_scores(ess_pool* pool, int layer, const void* q_idx, const float* w,
                              float* scores, ess_stream_t stream);

/* (a2)-(a4), (a8) Top-k, resolve, miss union and LRU update from given
 * scores ([FO] "decode side (1)", five-step flow and LIM outputs).
 *   scores      device float [B][M][T]
 * Outputs (device):
 *   topk_idx    int32 [B][M][k]: per way the min(k, T_b) selected tokens,
 *               misses first (ascending token), then hits (ascending token)
 *   topk_slot   int32 [B][M][k]: the slot of a hit, or ~slot (= -1 - slot)
 *               for a miss, naming the slot it is loaded into
 *   n_miss_way  int32 [B][M]: how many leading entries of way m are misses
 *   miss_tok    int32 [B][M*k]: the miss union Miss_b, ascending
 *   miss_slot   int32 [B][M*k]: the paired slot of each miss (copy triple:
 *               host row of miss_tok -> pool slot miss_slot, one row each)
 *   n_miss      int32 [B]: |Miss_b|
 * State: cache_slots, slot_token, last_used and step of the layer are
 * updated; entries past the selected count are left untouched.
 * Two kernels on stream: the selection (lists, miss union, victims) and the
 * LRU finishing kernel (the state rewrite and the next LRU order). */
ess_status ess_select_manage(ess_pool* pool, int layer, const float* scores,
                             int32_t* topk_idx, int32_t* topk_slot, int32_t* n_miss_way,
                             int32_t* miss_tok, int32_t* miss_slot, int32_t* n_miss,
                             ess_stream_t stream);

/* ess_select_manage for callers that cannot allocate device memory when they
 * call it: a serving engine that hands out all of its device memory at
 * start-up and has none left to give, or code on a thread where an allocation
 * would synchronise the device and stall decoding.  The pages have no
 * counterpart; this is a property of this library.
 * Same arguments, results and state updates as ess_select_manage, but the
 * selection's scratch (score histogram and victim list, about
 * B*M*(16 KiB + 4*k) bytes) lives in a fixed 2 MiB array compiled into the
 * library, which every GPU that loads the library keeps until the process
 * exits.  It calls no allocator.
 *   - Returns ESS_ERR_OOM, launching nothing, when the scratch needed exceeds
 *     the 2 MiB array, and ESS_ERR_INVALID_ARG when the current device is not
 *     the pool's (each device has its own copy of the array).
 *   - The first call on a device looks up the array's device address; make
 *     that first call before any stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (different
 *     streams, or several pools at once) race and must be ordered by the
 *     caller.  The histogram part is cleared at the start of every call. */
ess_status ess_select_manage_noalloc(ess_pool* pool, int layer, const float* scores,
                                     int32_t* topk_idx, int32_t* topk_slot, int32_t* n_miss_way,
                                     int32_t* miss_tok, int32_t* miss_slot, int32_t* n_miss,
                                     ess_stream_t stream);

/* (a1)-(a4) ess_indexer_scores followed by ess_select_manage, with the
 * scores kept in the pool's scratch ([FO] LIM: LI plus management).
 * Output arguments as in ess_select_manage. */
ess_status ess_indexer_topk(ess_pool* pool, int layer, const void* q_idx, const float* w,
                            int32_t* topk_idx, int32_t* topk_slot, int32_t* n_miss_way,
                            int32_t* miss_tok, int32_t* miss_slot, int32_t* n_miss,
                            ess_stream_t stream);

/* (a6) Copy the miss rows host -> pool slots ([FO] "decode side (1)", step
 * 5): for i < n_miss[b], host row of miss_tok[b][i] -> slot miss_slot[b][i].
 * Inputs are the device outputs of ess_select_manage. */
ess_status ess_stage_misses(ess_pool* pool, int layer, const int32_t* miss_tok,
                            const int32_t* miss_slot, const int32_t* n_miss,
                            ess_stream_t stream);

/* (a5) Sparse absorbed-MLA attention over the selected rows ([FO] "decode
 * side (2)": SFA/CopySFA; [ESS]: c^KV[512] + k^R[64]).
 *   q_mla      device bf16 [B][M][H][D]
 *   topk_idx, topk_slot: as produced by ess_select_manage
 *   out        device float [B][M][H][latent_dim]:
 *              softmax_s(sm_scale * q . row_s) @ row_s[:latent_dim]; zeros
 *              when nothing is selected
 * In FUSED mode a row with topk_slot < 0 is read from host memory and also
 * written to slot ~topk_slot; in STAGED mode every row is read from the pool
 * (run ess_stage_misses first). */
ess_status ess_sparse_mla_decode(ess_pool* pool, int layer, const void* q_mla,
                                 const int32_t* topk_idx, const int32_t* topk_slot, float* out,
                                 ess_stream_t stream);

/* (a1)-(a6) One decode step of one layer with every intermediate in the
 * pool's scratch: indexer, selection and management, (staging,) attention.
 *   q_idx, w  as in ess_indexer_scores;  q_mla, out as in
 *   ess_sparse_mla_decode.
 * Each kernel is launched as a programmatic dependent of the one before it on
 * the stream: its prologue overlaps the previous kernel, and it waits for that
 * kernel before touching memory.  With fused misses the attention kernel may
 * start while the selection still runs: each of its CTAs waits until the
 * selection CTAs of its own request have counted themselves done in a
 * per-request counter in the pool's scratch, then runs beside the LRU
 * finishing kernel and finishes only after it. */
ess_status ess_step(ess_pool* pool, int layer, const void* q_idx, const float* w,
                    const void* q_mla, float* out, ess_stream_t stream);

/* ess_step with measurement hooks: the same launches as ess_step, and
 * events[i] (each a cudaEvent_t, or NULL to skip) is recorded on stream
 * before the indexer (0), after the indexer (1), after selection and
 * staging (2) and after attention and merge (3).  A recorded event between two
 * kernels makes the second an ordinary launch (no early start). */
ess_status ess_step_profiled(ess_pool* pool, int layer, const void* q_idx, const float* w,
                             const void* q_mla, float* out, ess_stream_t stream,
                             void* const* events);

/* ess_step with HOST inputs and output.  Same layouts as ess_step.
 * When every buffer is pinned host memory mapped into the device address space
 * (ess_host_alloc, or cudaHostAlloc / cudaHostRegister on a system with unified
 * addressing), one more kernel at the head of the step reads the inputs over
 * the host link into device staging, and the merge kernel writes out_host
 * directly: no copy engine and no extra synchronisation inside the step.
 * Otherwise the inputs are copied to the staging and out back with
 * cudaMemcpyAsync on stream.  Either way the call is asynchronous on stream:
 * the caller keeps the inputs unchanged, and reads out_host, only after the
 * stream has passed the call. */
ess_status ess_step_host(ess_pool* pool, int layer, const void* q_idx_host,
                         const float* w_host, const void* q_mla_host, float* out_host,
                         ess_stream_t stream);

/* (a7) Layer-wise pipeline over two micro-batches (two pools with the same
 * config, e.g. the two halves of a batch): for layer l = 0..n_layers-1 each
 * pool runs ess_step on its own stream, so one micro-batch's selection and
 * staging overlap the other's attention ([ESS] layer-wise overlap).
 * Per-layer arrays are indexed [pool * n_layers + layer]. */
ess_status ess_pipeline_step(ess_pool* const* pools, int n_pools, int n_layers,
                             const void* const* q_idx, const float* const* w,
                             const void* const* q_mla, float* const* out,
                             const ess_stream_t* streams);

/* Copy the bookkeeping of one layer to host buffers (synchronous):
 * cache_slots [B][T], slot_token [B][C], last_used [B][C] int32, step [B]. */
ess_status ess_pool_get_state(ess_pool* pool, int layer, int32_t* cache_slots,
                              int32_t* slot_token, int32_t* last_used, int32_t* step);

/* Overwrite the bookkeeping of one layer from host buffers (synchronous):
 * resume from a saved state, or start from a full pool.  Any argument may be
 * NULL to keep that part.  The caller keeps it consistent (cache_slots and
 * slot_token inverse maps, last_used < step).  The LRU order is rebuilt from
 * last_used, and, when the layer is bound, the pool row of every resident
 * token (slot_token >= 0) is reloaded from the bound host copy, so that hits
 * read the right rows ([FO] "architecture": the host copy is the
 * authoritative one).  A resident token at or past T_b is reported by
 * ess_pool_poll as ESS_ERR_DEVICE_CHECK and its row is left as it was. */
ess_status ess_pool_set_state(ess_pool* pool, int layer, const int32_t* cache_slots,
                              const int32_t* slot_token, const int32_t* last_used,
                              const int32_t* step);

/* Gather rows of a pinned host array into device memory with 16-byte loads
 * issued by the GPU's own threads over the host link: the access pattern of
 * the miss path ([FO] "decode side (2)": misses are read from host memory
 * straight on chip).  Used to measure the link's sequential and random-row
 * rates, the host-link term of the layer's roofline.
 *   host_rows    pinned host [n_host_rows][row_bytes] (ess_host_alloc or any
 *                mapped pinned memory), 16-byte aligned
 *   row_bytes    a multiple of 16
 *   rows         device int64 [n_rows]: the host row of each output row, or
 *                NULL for rows 0..n_rows-1 (a sequential read)
 *   dst          device [n_rows][row_bytes], 16-byte aligned
 *   bad_row      device int32, or NULL: set to 1 by a row index outside
 *                [0, n_host_rows) (that row is skipped)
 * Errors: ESS_ERR_INVALID_ARG for a bad argument or memory that is not
 * pinned and mapped. */
ess_status ess_host_gather(const void* host_rows, int64_t n_host_rows, int32_t row_bytes,
                           const int64_t* rows, int64_t n_rows, void* dst, int32_t* bad_row,
                           ess_stream_t stream);

/* Copy the hot pool of one layer, [B][C][D] bf16, to a host buffer
 * (synchronous); rows of empty slots hold whatever was last written. */
ess_status ess_pool_get_rows(ess_pool* pool, int layer, void* rows_host);

/* Read (and optionally zero) the per-layer counters (synchronous). */
ess_status ess_pool_read_stats(ess_pool* pool, int layer, ess_stats* out, int reset);

/* Number of CUDA kernels the calls on this pool have launched since it was
 * created, counted on the host as each launch is enqueued (memsets and
 * copies are not kernels and are not counted). */
ess_status ess_pool_kernel_launches(const ess_pool* pool, int64_t* count);

/* Victim orders of ess_replay_misses. */
enum { ESS_EVICT_LRU = 0, ESS_EVICT_RANDOM = 1, ESS_EVICT_SCORE = 2, ESS_EVICT_LIM = 3 };

/* Victim order of the decode kernels for every layer of the pool (default
 * LRU).  The pages' decode ablation compares Random, LRU, Score and LIM on the
 * same access sequence ([FO] "evaluation", Figure 8); this makes the GPU path
 * run each of them.  Candidates are the slots whose token is not in the
 * step's miss union: empty slots first in slot order, then the resident ones
 * by last use (LRU), by a SplitMix64 draw keyed by (seed, request index b,
 * the layer's step counter) and the slot (Random), by the token's score this
 * step, the maximum over the ways (Score), or in slot order (LIM); ties go to
 * the lower slot, and the i-th miss (ascending token) takes the i-th
 * candidate, as in ess_replay_misses.  Orders other than LRU add one kernel
 * per selection.  Synchronous; switching back to LRU rebuilds its order from
 * last_used.
 * Errors: ESS_ERR_INVALID_ARG for an unknown policy. */
ess_status ess_pool_set_eviction(ess_pool* pool, int32_t policy, uint64_t seed);

/* Replay one request's trace of selections with an eviction policy and count
 * its misses ([FO] "evaluation": the decode ablation's offline simulator and
 * Figure 8, which replays the same top-k trace with Random, LRU, Score and
 * LIM eviction).  Host code only; ess_pool_set_eviction runs the same
 * orders in the decode kernels.
 *   offsets, tokens  the selections in CSR form: way m of step s selected
 *                    tokens[offsets[s*n_ways+m] .. offsets[s*n_ways+m+1])
 *   scores           host float [n_steps][n_ways][T], the ways' scores of every
 *                    token (ESS_EVICT_SCORE only; else may be NULL)
 *   T, C             tokens and hot-pool slots of the request
 *   policy           ESS_EVICT_*; seed and request key the Random draws
 * Each step: hits are stamped; the slots not holding a selected token are the
 * candidates, empty slots first in slot order, then resident ones by LRU
 * (last use), Random (a SplitMix64 draw per slot keyed by seed, request and
 * step), Score (the token's score this step, maximum over the ways) or LIM
 * (slot order), ties to the lower slot; the i-th miss in token order takes
 * the i-th candidate.
 * Outputs (host int32 [n_steps]): union_misses (distinct rows loaded) and
 * way_misses (selected tokens not resident before the step, summed over the
 * ways, as the page's figure counts them).
 * Errors: ESS_ERR_INVALID_ARG for bad arguments or a token outside [0, T);
 * ESS_ERR_CAPACITY when a step selects more than C distinct tokens. */
ess_status ess_replay_misses(int32_t n_steps, int32_t n_ways, const int64_t* offsets,
                             const int32_t* tokens, const float* scores, int32_t T, int32_t C,
                             int32_t policy, uint64_t seed, int64_t request,
                             int32_t* union_misses, int32_t* way_misses);

/* Encode latent rows as compact 656-byte rows ("ESS: Latent-Cache Offload",
 * the ~656-byte host transfers of its FlashTrans + UVA row and its 16.8% /
 * 83.2% indexer/latent byte split).  Layout (a reading; the page gives only
 * the size): bytes 0..511 the 512 latent values as e4m3 in four tiles of 128,
 * bytes 512..527 one little-endian float32 scale per tile, bytes 528..655 the
 * 64 RoPE values as bf16.  A tile's scale is the smallest power of two at or
 * above fl32(amax / 448) (1 for an all-zero tile), so every decoded value is
 * exact in bf16; a value's code is e4m3(x / scale), nearest with ties to the
 * even code, saturating at +-448, sign kept.
 *   rows_bf16  host bf16 [n_rows][576]
 *   out        host uint8 [n_rows][656]
 * Errors: ESS_ERR_INVALID_ARG for n_rows < 0 or a null buffer. */
ess_status ess_compact_rows(const uint16_t* rows_bf16, int64_t n_rows, uint8_t* out);

/* Binding table of the prefill layer schedule with whole-layer device
 * buffers ([FO] "prefill side": B0 pinned to layer 0, B1..B3 rotating through
 * a binding table, a buffer reused only after its layer's compute and
 * write-back, layer onload_layer_map[i] prefetched at layer i's scheduling
 * point).  Host code; it plans, ess_prefill_run moves the data.
 *   n_layers          L >= 1
 *   onload_layer_map  host int32 [L]: the layer (1..L-1) prefetched at layer
 *                     i's scheduling point, or -1; a layer no entry names is
 *                     loaded up front
 *   rotating          buffers besides B0 (the page uses 3)
 *   shared_copy       1 when loads and write-backs share one serial copy
 *                     stream (a layer's write-back is then issued after the
 *                     prefetch at its own scheduling point)
 * Outputs (host int32 [L]): buffer[l] (0 = B0, else 1..rotating, bound
 * round-robin in load order), load_at[l] (the scheduling point that issues
 * l's load, -1 for up front and for layer 0), reuse_after[l] (the layer whose
 * release l's load waits for, or -1).
 * Errors: ESS_ERR_INVALID_ARG for a bad argument, a layer loaded twice, or a
 * load that would wait for a layer whose write-back is not yet issued (the
 * buffer would still be held). */
ess_status ess_prefill_plan(int32_t n_layers, const int32_t* onload_layer_map, int32_t rotating,
                            int32_t shared_copy, int32_t* buffer, int32_t* load_at,
                            int32_t* reuse_after);

/* Per-layer compute of a prefill pass, called by ess_prefill_run on the
 * calling thread: enqueue the layer's work on `stream` (asynchronously); it
 * may read and update `buffer`, the device buffer that holds the layer's KV. */
typedef void (*ess_prefill_compute_fn)(void* user, int32_t layer, void* buffer,
                                       ess_stream_t stream);

/* One prefill pass over n_layers layers with whole-layer device buffers, run
 * by the schedule of ess_prefill_plan ([FO] "prefill side: four whole-layer
 * buffers hide the transfers", its five-step lifecycle and Figure 3):
 *   buffers      device [1 + rotating] buffers of layer_bytes each; buffers[0]
 *                (B0) holds layer 0 throughout and is neither loaded nor
 *                written back here; B1.. rotate over layers 1..L-1
 *   host_kv      pinned host [L] pointers, layer l's KV (layer_bytes each;
 *                host_kv[0] unused)
 *   compute      the caller's per-layer work, called in layer order
 *   wb_offset, wb_bytes  the byte range of a layer written back after its
 *                compute (e.g. the rows this pass produced)
 * Layer j is loaded (H2D on h2d_stream) up front, or at the scheduling point
 * of the layer that prefetches it, once the previous layer of its buffer has
 * been computed and written back; compute(i) waits for layer i's load; the
 * write-back (D2H on d2h_stream, or on h2d_stream when shared_copy) follows
 * compute(i) and releases the buffer.  Events carry every dependency, so the
 * copies overlap the computes of other layers.  Asynchronous: when
 * compute_stream has passed the call, every write-back is done.
 * Errors: ESS_ERR_INVALID_ARG for a bad argument or a schedule that
 * ess_prefill_plan refuses; ESS_ERR_CUDA when a CUDA call fails. */
ess_status ess_prefill_run(int32_t n_layers, const int32_t* onload_layer_map, int32_t rotating,
                           int32_t shared_copy, void* const* host_kv, size_t layer_bytes,
                           size_t wb_offset, size_t wb_bytes, void* const* buffers,
                           ess_prefill_compute_fn compute, void* user,
                           ess_stream_t compute_stream, ess_stream_t h2d_stream,
                           ess_stream_t d2h_stream);

/* Synchronise stream, return the first device-side error since the last
 * poll (ESS_OK if none) and clear it. */
ess_status ess_pool_poll(ess_pool* pool, ess_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ESS_H */
