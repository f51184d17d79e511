/*
 * okv: lookahead sparse KV staging and sparse decode attention on one GB300 (sm_103a).
 *
 * The operations follow OasisKV ("OasisKV: Scaling In-Decode KV Cache Beyond HBM with
 * Lookahead Sparse Prefetching", arXiv 2608.08097; summary page paperlayer.ai/abs/2608.08097v1):
 * the full KV cache stays off-GPU in host memory, HBM holds per-block key summaries and a
 * sparse working set of blocks, and a draft (lookahead) query stages the next step's blocks
 * ("4 System Design"). One library context serves one model on one GPU.
 *
 * Conventions
 *  - Every call returns an okv_status and never throws across the ABI. On failure,
 *    okv_last_error(ctx) holds a one-line reason.
 *  - "unit" = one (layer, request, kv head). "Kb" = budget_tokens / block_size slots per unit.
 *  - Device pointers are caller-owned device memory (e.g. torch tensors), contiguous, of the
 *    context's storage dtype unless stated. They must stay valid until the work enqueued on
 *    the given stream has finished.
 *  - `stream` arguments are cudaStream_t handles passed as void* (NULL = legacy default stream).
 *  - Calls are asynchronous unless their name starts with okv_read_ or is okv_sync.
 *  - A context is used from one host thread at a time.
 *  - Kernels never trap: an invalid index found on the device is recorded in a device error
 *    word and the access is skipped; okv_sync and the okv_read_* calls report it as
 *    OKV_EDEVICE.
 *
 * Host KV layout of one request (caller-owned, page-locked, e.g. from okv_host_alloc):
 *   [layers][kv_heads][capacity_blocks][2][block_size][head_dim], index 0 of the "2" axis is K,
 *   1 is V, storage dtype. One block of one unit (K and V of block_size tokens) is contiguous.
 */
#ifndef OKV_H
#define OKV_H

#include <stdint.h>

#if defined(__GNUC__)
#define OKV_API __attribute__((visibility("default")))
#else
#define OKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OKV_OK = 0,
  OKV_EINVAL = 1,   /* bad argument or unsupported shape */
  OKV_ENOMEM = 2,   /* device or page-locked host allocation failed */
  OKV_ECUDA = 3,    /* a CUDA runtime call failed */
  OKV_EDEVICE = 4,  /* a kernel recorded an invalid index in the device error word */
  OKV_ETIMEOUT = 5, /* okv_sync's deadline passed with work still running */
  OKV_ESTATE = 6    /* call not valid in the context's current state */
} okv_status;

enum { OKV_F32 = 0, OKV_BF16 = 1 };

typedef struct {
  int32_t layers;                 /* decoder layers */
  int32_t q_heads;                /* query heads; a multiple of kv_heads (GQA group g = q/kv) */
  int32_t kv_heads;               /* KV heads */
  int32_t head_dim;               /* d: a multiple of 32, at most 256 */
  int32_t block_size;             /* tokens per KV block (16) */
  int32_t budget_tokens;          /* KV budget per unit in tokens; Kb = budget/block_size slots */
  int32_t max_requests;           /* request ids are 0 .. max_requests-1 */
  int32_t max_blocks_per_request; /* largest context (in blocks) any request may reach; the
                                     selection keeps a unit's per-block arrays in one CTA's
                                     shared memory (6 bytes per block), which bounds it
                                     (about 37600 blocks, 600K tokens, at a 128-slot budget
                                     on GB300; okv_create says the limit) */
  float fetch_cap;                /* default fetch cap, a fraction of the budget (0.05) */
  int32_t dtype;                  /* OKV_F32 or OKV_BF16 storage for KV, queries, outputs */
} okv_config;

typedef struct okv_ctx okv_ctx;

/* Create a context on the current CUDA device. Allocates in HBM: block summaries
 * [layers][max_requests][kv_heads][max_blocks][2][head_dim], the slot pool
 * [layers][max_requests][kv_heads][Kb][2][block_size][head_dim], the per-unit tables, the
 * scoring coefficients and the device error word; creates its internal streams (two staging
 * lanes at the least priority, okv_step's attention stream at a middle priority, the gather's
 * copy stream and okv_step's append stream at the greatest). Environment variables read here
 * select measured alternatives: OKV_STAGE_LANES=1, OKV_STAGE_STREAM=caller,
 * OKV_STAGE_PRIORITY=high, OKV_ATTEND_PRIORITY=caller or high. EINVAL on an unsupported config,
 * ENOMEM if HBM is short. */
OKV_API okv_status okv_create(const okv_config* cfg, okv_ctx** out);
/* Waits for the context's work, frees everything it allocated. NULL is a no-op. */
OKV_API void okv_destroy(okv_ctx* ctx);
/* Reason for the last failure of a call on ctx ("" if none). */
OKV_API const char* okv_last_error(const okv_ctx* ctx);
OKV_API const char* okv_status_string(okv_status s);

/* Page-locked, device-mapped host memory for host KV buffers (cudaHostAlloc). The caller
 * frees it with okv_host_free. ENOMEM if the host cannot pin that much. */
OKV_API okv_status okv_host_alloc(int64_t bytes, void** out);
OKV_API okv_status okv_host_free(void* p);

/* Register request `req` whose full KV stays in host memory ("4 System Design": full KV in
 * CPU DRAM, compressed summaries in HBM). host_kv: page-locked buffer in the host KV layout
 * with capacity_blocks blocks per unit; the caller keeps it alive until okv_remove_request.
 * Builds the min/max summaries of the first n_tokens tokens of every layer by reading the
 * host buffer (or copies them from an active request registered with the same buffer and
 * length). The request's slot pool starts empty. EINVAL on bad ids/sizes or unpinned memory,
 * ESTATE if req is already active. */
OKV_API okv_status okv_add_request(okv_ctx* ctx, int32_t req, void* host_kv, int32_t capacity_blocks,
                           int32_t n_tokens, void* stream);
/* Register request `req` with admission-time partial staging ("4 System Design", last bullet:
 * the prefill side keeps each request's full KV cache in its host memory until the request
 * completes, and the decode side materialises only a demand-filled subset of it).
 *   full_kv:  the full copy, page-locked, host KV layout with capacity_blocks blocks per unit.
 *             It stands for the prefill side's memory; the caller keeps it alive until
 *             okv_remove_request.
 *   local_kv: the decode-side tier, page-locked, host KV layout with local_capacity_blocks
 *             entries per unit, [layers][kv_heads][local_capacity_blocks][2][block_size]
 *             [head_dim]; caller-owned, written by the library; NULL if local_capacity_blocks
 *             is 0. It may not overlap any active request's buffers.
 * Summaries are built from full_kv as in okv_add_request (the prefill side's work). Then every
 * fetch of a block by okv_stage reads the decode side's kept copy if it has one; a block fetched
 * for the first time is read from full_kv and kept in the next unused entry of its unit (entries
 * are taken in fetch order and never released before okv_remove_request); once a unit's entries
 * are used up, first-time blocks are read from full_kv without being kept. okv_append writes
 * full_kv and, if the block is kept, the kept copy. The okv_timing counters local_hits,
 * local_fills and full_reads count these fetches; okv_read_local returns the tables.
 * EINVAL: as okv_add_request, or local_capacity_blocks outside [0, capacity_blocks], or local_kv
 * unpinned, unaligned or overlapping; ESTATE if req is already active. */
OKV_API okv_status okv_add_request_partial(okv_ctx* ctx, int32_t req, void* full_kv, int32_t capacity_blocks,
                                           void* local_kv, int32_t local_capacity_blocks, int32_t n_tokens,
                                           void* stream);
/* Forget request `req` (its pool slots become free). Synchronises the internal streams. */
OKV_API okv_status okv_remove_request(okv_ctx* ctx, int32_t req);

/* Append one token per active request to `layer` ("2 Background": the cache must remain
 * available throughout generation). k_new, v_new: device [max_requests][kv_heads][head_dim];
 * rows of inactive requests are ignored. Writes the token into the host buffer, into the pool
 * slot if its block is resident, and updates the block's min/max summary; advances the
 * layer's length of each active request. Waits for the layer's previous staging. EINVAL if a
 * request is full or shares its host buffer with another active request. */
OKV_API okv_status okv_append(okv_ctx* ctx, int32_t layer, const void* k_new, const void* v_new,
                      void* stream);

/* Next-step prefetch from lookahead ("4 System Design": the per-layer background chain is
 * top-K prediction, KV selection and KV transfer). draft_q: device [max_requests][q_heads]
 * [head_dim], the draft query of every active request. Enqueued after the work already on
 * `stream`, on the context's internal streams:
 *   scores of every block from its summary, top-Kb blocks per unit (score desc, id asc),
 *   diff against the resident pool: admit at most C = max(1, floor(cap * Kb)) missing blocks
 *   per unit, evicting least-recently-selected unselected blocks, stamps = step,
 *   gather of the admitted blocks from host memory into their slots.
 * fetch_cap < 0 uses the config's cap. The scoring's coefficients are computed from the draft
 * on `stream` (per KV head and coordinate, the sums of the group's negative and of its positive
 * draft coordinates), so the caller may overwrite draft_q by work enqueued later on `stream`.
 * Returns once enqueued; okv_attend on the same layer waits for it. */
OKV_API okv_status okv_stage(okv_ctx* ctx, int32_t layer, const void* draft_q, int32_t step,
                     float fetch_cap, void* stream);

/* Sparse attention over the resident set ("4 System Design": attention runs over resident KV
 * in HBM). q: device [max_requests][q_heads][head_dim]; out: device, same shape and dtype.
 * For every active request and query head: softmax(q.k / sqrt(d)) v over every valid token of
 * every occupied slot of its unit (zeros if none). Waits on `stream` for the layer's last
 * staging. Rows of inactive requests are not written. */
OKV_API okv_status okv_attend(okv_ctx* ctx, int32_t layer, const void* q, void* out, void* stream);

/* Top-K prediction alone ("4 System Design": top-K prediction, the first link of the per-layer
 * chain) for any query, e.g. the true next query or the previous token's query, to measure how
 * well a draft predicts the blocks a step attends. query: device [max_requests][q_heads]
 * [head_dim]; counts: device [max_requests][kv_heads] int32; ids: device [max_requests]
 * [kv_heads][Kb] int32, the selected block ids in (score desc, id asc) order. The context's
 * selections, slot tables and pools are not changed. Ordered after the work on `stream`;
 * `stream` waits for the result. */
OKV_API okv_status okv_predict(okv_ctx* ctx, int32_t layer, const void* query, int32_t* counts, int32_t* ids,
                               void* stream);

/* Look-ahead attention ("4 System Design": normal and draft queries are computed together over
 * the resident KV): okv_attend for q -> out and, over the same resident set, for draft_q ->
 * draft_out (both device [max_requests][q_heads][head_dim]). When twice the GQA group fits the
 * tensor-core tile (2g <= 8) both are computed in one pass over K and V; otherwise the draft
 * heads take a second pass. */
OKV_API okv_status okv_attend_lookahead(okv_ctx* ctx, int32_t layer, const void* q, const void* draft_q,
                                        void* out, void* draft_out, void* stream);

/* One decode step over every layer, in layer order ("4 System Design": the foreground waits
 * only for each layer's transfer; the background chain of layer l overlaps the attention of the
 * later layers). The result is that of: for l = 0 .. layers-1: okv_append(l) if k_new is not NULL,
 * okv_attend(l), okv_stage(l, step). q, draft_q, out: device [layers][max_requests][q_heads]
 * [head_dim]; k_new, v_new: device [layers][max_requests][kv_heads][head_dim] or NULL.
 * Scheduling: the step's own work runs on the context's attention stream, which first waits
 * for the work enqueued on `stream` so far and which `stream` waits for at the end of the step
 * (with OKV_ATTEND_PRIORITY=caller, on `stream` itself). There the scoring coefficients of every
 * layer's draft are computed in one launch, up front, then the attentions run in layer order,
 * the attention of layer l waiting only for the append of layer l. Every layer's append is
 * enqueued up front on an internal stream, each after that layer's previous staging. The
 * inputs may be reused by work enqueued on `stream` after the call. Stops at the first failing check (before any work is
 * enqueued, for the append checks) and returns its status. */
OKV_API okv_status okv_step(okv_ctx* ctx, const void* q, const void* draft_q, void* out,
                            const void* k_new, const void* v_new, int32_t step, float fetch_cap,
                            void* stream);

/* Make `stream` wait (on the device, without blocking the host) for all work the context has
 * enqueued so far on its internal streams: the staging of every layer. */
OKV_API okv_status okv_join(okv_ctx* ctx, void* stream);

/* Wait (polling, up to timeout_ms; < 0 = no limit) for the context's internal streams and
 * check the device error word. ETIMEOUT with work still in flight, EDEVICE if a kernel
 * recorded an invalid index (the word is then cleared). */
OKV_API okv_status okv_sync(okv_ctx* ctx, int64_t timeout_ms);

/* ---- inspection: synchronise the internal streams, then copy to caller-owned host arrays.
 * The caller must first synchronise any stream it passed to okv_attend / okv_append /
 * okv_stage. ---- */

/* Summaries of one request: out [kv_heads][max_blocks_per_request][2][head_dim] storage. */
OKV_API okv_status okv_read_summaries(okv_ctx* ctx, int32_t layer, int32_t req, void* out);
/* Last selection of a layer: counts [max_requests][kv_heads]; ids and scores
 * [max_requests][kv_heads][Kb] (first counts[] entries valid). Either array may be NULL. */
OKV_API okv_status okv_read_selection(okv_ctx* ctx, int32_t layer, int32_t* counts, int32_t* ids,
                              float* scores);
/* Slot tables: slot_block [max_requests][kv_heads][Kb] (block id or -1), stamps (same shape). */
OKV_API okv_status okv_read_slot_table(okv_ctx* ctx, int32_t layer, int32_t* slot_block, int32_t* stamps);
/* Last fetch lists: counts [max_requests][kv_heads]; entries [max_requests][kv_heads][Kb][2]
 * as (block id, slot), in admission order. */
OKV_API okv_status okv_read_fetch_list(okv_ctx* ctx, int32_t layer, int32_t* counts, int32_t* entries);
/* Pool contents of one unit: out [Kb][2][block_size][head_dim] storage. */
OKV_API okv_status okv_read_pool(okv_ctx* ctx, int32_t layer, int32_t req, int32_t kv_head, void* out);
/* Current context length of every request at a layer: lengths [max_requests] (0 if inactive). */
OKV_API okv_status okv_read_lengths(okv_ctx* ctx, int32_t layer, int32_t* lengths);
/* Decode-side tiers of partially staged requests at a layer: local_used [max_requests][kv_heads]
 * (entries in use); local_of [max_requests][kv_heads][max_blocks_per_request] (kept entry of each
 * block or -1); routes [max_requests][kv_heads][Kb], one per entry of the last fetch list:
 * 2*e = read from kept entry e, 2*e + 1 = read from the full copy and kept in entry e, -1 = read
 * from the full copy only (always -1 for requests registered with okv_add_request). Rows of
 * other requests hold no meaning. Any array may be NULL. */
OKV_API okv_status okv_read_local(okv_ctx* ctx, int32_t layer, int32_t* local_used, int32_t* local_of,
                                  int32_t* routes);

/* ---- measurement ---- */

/* Kernel kinds of okv_timing: OKV_K_COEF is the scoring's coefficients of the draft queries
 * (okv_stage, okv_step and okv_predict compute them before the staging); OKV_K_COMBINE is unused. */
enum {
  OKV_K_SUMMARY = 0, OKV_K_SCORE_TOPK = 1, OKV_K_COEF = 2, OKV_K_GATHER = 3, OKV_K_ATTEND = 4,
  OKV_K_COMBINE = 5, OKV_K_APPEND = 6, OKV_K_COUNT = 7
};

typedef struct {
  double ms[OKV_K_COUNT];         /* summed device time of each kernel kind (CUDA events) */
  int64_t launches[OKV_K_COUNT];  /* kernel launches of each kind */
  int64_t fetched_blocks;         /* blocks gathered host -> HBM */
  int64_t attended_slots;         /* occupied slots read by attention launches */
  /* fetches of partially staged requests (okv_add_request_partial): */
  int64_t local_hits;             /* read from the decode side's kept copy */
  int64_t local_fills;            /* read from the full copy and kept */
  int64_t full_reads;             /* read from the full copy (local_fills included) */
} okv_timing;

/* Enable (1) or disable (0) per-launch CUDA-event timing; resets the totals. */
OKV_API okv_status okv_set_timing(okv_ctx* ctx, int32_t enable);
/* Synchronise and return the totals since okv_set_timing. */
OKV_API okv_status okv_read_timing(okv_ctx* ctx, okv_timing* out);
/* Kernel launches made by this context so far (all kinds), counted on the host. */
OKV_API int64_t okv_launch_count(const okv_ctx* ctx);

/* ---- allocation-free attention (no counterpart in the paper) ----
 *
 * Some callers cannot call cudaMalloc: code that runs where allocation is forbidden or must
 * not fail (a fixed memory budget handed over up front, an allocator they do not own, a
 * callback path that may not allocate). okv_attend_static gives them the sparse
 * attention of okv_attend without a context and without allocating anything: the caller
 * passes every input and output, and the kernels' only workspace (split partials, request ids,
 * an error word) is one fixed 16 MiB device array inside this library, which every GPU that
 * loads the library holds until the process exits.
 *
 *   pool:       device [n_requests][kv_heads][slots][2][block_size][head_dim] storage dtype,
 *               16-byte aligned (the layout of one layer of okv's slot pool)
 *   slot_block: device [n_requests][kv_heads][slots] int32, the block each slot holds or -1
 *   lengths:    device [n_requests] int32, each request's context length in tokens
 *   q, out:     device [n_requests][q_heads][head_dim] storage dtype
 * Every request 0 .. n_requests-1 attends: softmax(q.k / sqrt(d)) v over every valid token of
 * every occupied slot of its unit, zeros if none (the computation of okv_attend).
 *
 * Limits: n_requests <= 16384, and the split workspace the launch shape needs must fit in the
 * array (about 16 MiB of n_requests * kv_heads * split * g * (head_dim + 2) floats); beyond
 * them, and for shapes okv_create refuses, the call returns OKV_EINVAL without launching.
 * Every call resolves the array's device address on the current device
 * (cudaGetSymbolAddress). The first call in each CUDA context of a device (the first call on
 * the device, and the first after a cudaDeviceReset) also initialises the array's constant
 * part, synchronising that device. Calls then enqueue on
 * `stream`, which must belong to the current device (else OKV_EINVAL): two small clears of
 * the array (split counters, error word), then the attention kernels. All calls share the
 * array: calls whose work overlaps on the GPU (on different streams, or on different host
 * threads) race and must be serialised by the caller.
 * Failures the kernels record are not reported: this call has no context to report them
 * through. A slot whose block id fails the bounds check (outside the request's length) is
 * skipped, and a copy wait that gives up leaves the unit's output partial; the array's error
 * word holds the first such failure of the call until the next call clears it, and no call
 * reads it. */
OKV_API okv_status okv_attend_static(int32_t n_requests, int32_t q_heads, int32_t kv_heads,
                                     int32_t head_dim, int32_t block_size, int32_t slots,
                                     int32_t dtype, const void* pool, const int32_t* slot_block,
                                     const int32_t* lengths, const void* q, void* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif
