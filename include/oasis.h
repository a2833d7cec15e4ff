/*
 * oasis.h -- C ABI of the GB300 look-ahead sparse decode step (OasisKV).
 *
 * The step, per layer and per decode step t ([R] = "Pith review of OasisKV:
 * Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse Prefetching",
 * section "What carries the argument"; [V] = the pith.science verdict record
 * of arXiv 2608.08097, field "key_machinery"):
 *   a1  one shared paged-attention pass serves the normal query q and the
 *       speculative draft query qd (or D of them, oasis_config.num_drafts)
 *       of every request over the head-wise resident set of K blocks
 *       (B = 16 tokens each, GQA);
 *   a2  the draft query scores every logical block from per-block
 *       coordinate-wise min/max key summaries held in HBM with the upper bound
 *       sum_j sum_i max(qd_ji * min_i, qd_ji * max_i) (j over the KV head's
 *       query heads);
 *   a3  a head-wise top-K ranking of all logical blocks;
 *   a4  capped eviction: each admitted non-resident block is paired with the
 *       least-recently-selected resident block, at most
 *       C = floor(fetch_ratio * K) admissions per (request, KV head) per step
 *       ([S] = "OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead
 *       Sparse Prefetching" (agihunt.info summary), fetch-cap ablation);
 *   a5  the admitted blocks are gathered from pinned host memory into HBM on a
 *       side stream, overlapped with other work, and are used from step t+1
 *       on ([R] abstract: prefetched blocks land in HBM one step ahead of
 *       their use).
 *
 * Conventions
 *   - Every call returns an oasis_status.  No call aborts, prints or exits.
 *   - Device work is asynchronous on the caller's cudaStream_t (passed as
 *     void*, NULL = legacy default stream).  oasis_sync() waits for all work
 *     of the context and reports deferred device-side errors.
 *   - Ownership: every buffer is allocated by the caller and lent to the
 *     library for the life of the context; the library never frees it.  The
 *     library itself allocates only CUDA streams and events (and, with a
 *     remote tier, host threads and their queues).  oasis_query_sizes
 *     reports every buffer size.
 *   - Shapes: R requests, Hq query heads, Hkv KV heads (G = Hq/Hkv <= 4), head
 *     dim d = 128, block size B = 16, K resident blocks per (request, KV head),
 *     NBmax logical blocks of capacity per (request, KV head), C admissions per
 *     step, U = K + C pool units per (request, KV head).  Query head j reads KV
 *     head j / G.  One "unit" is the keys and values of one block of one KV
 *     head: [2][B][d] bf16 = 8 KiB.
 *   - Double-buffered state.  Step t reads table (t & 1) of res_ids / phys and
 *     ctx_len; its admission writes table ((t + 1) & 1).  Consecutive steps of
 *     one layer must therefore use consecutive t.  After step t the logical
 *     resident set is res_ids[(t + 1) & 1] and slot s holds pool unit
 *     phys[(t + 1) & 1][s].
 *   - Not thread-safe: one host thread drives a context at a time.
 *
 * Layouts (row-major, innermost last; "dev" = device memory, "pinned" =
 * page-locked host memory that the device can map):
 *   kv_pool    dev    [R][Hkv][U][2][B][d]      bf16   resident units + C spares
 *   summaries  dev    [R][Hkv][NBmax][2][d]     bf16   [0] = min row, [1] = max row
 *   host_kv    pinned [R][Hkv][NBmax][2][B][d]  bf16   full KV store ([0]=K,[1]=V)
 *   res_ids    dev    [2][R][Hkv][K]            int32  logical block per slot, -1 empty
 *   stamps     dev    [R][Hkv][K]               int32  step of last selection, -1 never
 *   phys       dev    [2][R][Hkv][U]            int32  pool unit per slot; [K..U) spares
 *   ctx_len    dev    [2][R]                    int32  tokens per request
 *   q          dev    [R][Hq][d]                bf16
 *   q_draft    dev    [D][R][Hq][d]             bf16   D = draft queries per step
 *   out        dev    [R][Hq][d]                bf16, or fp32 if cfg.out_fp32
 *   out_draft  dev    [D][R][Hq][d]             as out
 *   topk_ids   dev    [R][Hkv][K]               int32  rank order, -1 padded
 *   topk_scores dev   [R][Hkv][K]               fp32   (nullable)
 *   admit_ids, admit_slots, evict_ids  dev [R][Hkv][C] int32 (-1 padded)
 *   n_admit    dev    [R][Hkv]                  int32
 */
#ifndef OASIS_H
#define OASIS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define OASIS_API __attribute__((visibility("default")))
#else
#define OASIS_API
#endif

typedef enum {
  OASIS_OK = 0,
  OASIS_EINVAL = -1,   /* bad argument: null pointer, size, alignment, range */
  OASIS_ENOMEM = -2,   /* a host-side resource (stream/event/mapping) failed */
  OASIS_ECUDA = -3,    /* a CUDA runtime call failed; see oasis_last_error */
  OASIS_ETIMEOUT = -4, /* a bounded wait ran out (device or host side) */
  OASIS_ESTATE = -5,   /* call out of order (e.g. step before load) */
  OASIS_EDEVICE = -6   /* a kernel reported bad data (see oasis_sync) */
} oasis_status;

/* Device error word bits, reported by oasis_sync() as OASIS_EDEVICE. */
#define OASIS_DEVERR_BAD_BLOCK_ID 0x1u /* a block id >= NBmax or past context */
#define OASIS_DEVERR_TIMEOUT 0x2u      /* a kernel's bounded barrier wait expired */
#define OASIS_DEVERR_BAD_UNIT 0x4u     /* a pool unit index >= U */
#define OASIS_DEVERR_NOT_LOCAL 0x8u    /* remote tier: a block needed a local slot
                                          but the local tier was full */

typedef struct {
  int32_t num_layers;
  int32_t num_requests;  /* R */
  int32_t max_blocks;    /* NBmax, <= 131072 */
  int32_t num_q_heads;   /* Hq */
  int32_t num_kv_heads;  /* Hkv; Hq % Hkv == 0 and Hq / Hkv <= 4 */
  int32_t head_dim;      /* d; must be 128 */
  int32_t block_size;    /* B; must be 16 */
  int32_t topk;          /* K; 1..256 and K <= max_blocks */
  float fetch_ratio;     /* C = floor(fetch_ratio * K), 0 <= fetch_ratio <= 1 */
  float softmax_scale;   /* 0 -> 1/sqrt(d) */
  int32_t out_fp32;      /* attention outputs in fp32 (1) or bf16 (0) */
  int32_t device;        /* CUDA device ordinal */
  int32_t side_groups;   /* request groups oasis_step pipelines its side work
                            in (0 = one per 256 (request, KV head) pairs, <= 8) */
  int32_t schedule;      /* OASIS_SCHEDULE_*: how a step orders a1 */
  int32_t num_drafts;    /* D, draft queries per step: 0 or 1 = one, <= 3.
                            Several drafts (an option of the three-stream
                            pipeline) all read the one resident set in a1 and
                            their bounds add up in a2 like those of a group's
                            query heads; q_draft and out_draft hold D planes
                            of [R][Hq][d]. */
} oasis_config;

/* oasis_step schedules.  SCAN_FIRST: the attention of a step starts when the
 * step's scans are done, so the scans run alone and the host-link gathers
 * start early and overlap the attention.  CONCURRENT: the attention starts at
 * once, sharing HBM with the scans.  THREE_STREAMS: the pipeline as the pages
 * describe it ([R] *What carries the argument*: per layer, one background
 * stream each for ranking, selection and transfer): a stand-alone scan + top-K, a
 * stand-alone admission and the gathers on three streams, the attention
 * starting at once.  AUTO: SCAN_FIRST for every step call (measured on
 * GB300, 128 x 16K layer, scan-first against concurrent: oasis_step 3343-3346
 * against 2254-2866 layer-steps/s, oasis_step_host_async 3268-3279 against
 * 2784-2804, oasis_step_host 3070-3073 against 2546-2673).  Results are
 * identical. */
#define OASIS_SCHEDULE_SCAN_FIRST 0
#define OASIS_SCHEDULE_CONCURRENT 1
#define OASIS_SCHEDULE_THREE_STREAMS 2
#define OASIS_SCHEDULE_AUTO 3
/* EARLY_SCAN: the scan + top-K of step t runs on its own stream as soon as
 * its inputs exist, beside the previous step's attention, instead of after
 * the work already on `stream`; only the admission waits for that work (it
 * rewrites the table the previous attention read).  Contract: the draft
 * queries must be ready when oasis_step is called (oasis_step_host's host
 * buffers always are), and the summaries and context lengths may change
 * between steps only through this library's calls (build_summaries,
 * append_token, refresh_blocks, advance_context), which the early scan
 * follows, or with the device idle.  Results are identical.  Measured on
 * GB300 (128 x 16K layer): oasis_step 3456-3482 against 3336-3340
 * layer-steps/s scan-first, oasis_step_host 3267-3281 against 3070-3073,
 * oasis_step_host_async 3093-3100 against 3262-3269.  AUTO never picks it:
 * its contract is the caller's to keep. */
#define OASIS_SCHEDULE_EARLY_SCAN 4

typedef struct {
  size_t kv_pool_bytes;   /* per layer */
  size_t summaries_bytes; /* per layer */
  size_t host_kv_bytes;   /* per layer (pinned host) */
  size_t res_ids_bytes;   /* per layer, both tables */
  size_t stamps_bytes;    /* per layer */
  size_t phys_bytes;      /* per layer, both tables */
  size_t ctx_len_bytes;   /* once */
  size_t workspace_bytes; /* once, device, 256-byte aligned */
  int32_t fetch_cap;      /* C */
  int32_t units_per_head; /* U = K + C */
} oasis_sizes;

typedef struct {
  /* Arrays of num_layers pointers (the arrays themselves are copied at
   * oasis_init).  kv_pool, summaries and host_kv must be 16-byte aligned. */
  void* const* kv_pool;
  void* const* summaries;
  void* const* host_kv; /* pinned host pointers (cudaHostAlloc / registered) */
  int32_t* const* res_ids;
  int32_t* const* stamps;
  int32_t* const* phys;
  int32_t* ctx_len;     /* [2][R] */
  void* workspace;      /* workspace_bytes of device memory */
} oasis_buffers;

typedef struct oasis_ctx oasis_ctx;

/* NULL if cfg is supported, else a static message naming the first problem.
 * Pure host computation. */
OASIS_API const char* oasis_config_error(const oasis_config* cfg);

/* Sizes of every caller-owned buffer for cfg.  Pure host computation (needs
 * no GPU).  EINVAL on an unsupported configuration. */
OASIS_API int oasis_query_sizes(const oasis_config* cfg, oasis_sizes* out);

/* Validate cfg and bufs, map the host stores, build the TMA descriptors,
 * create the streams and events and load every kernel.  Buffers are not
 * initialised: call oasis_build_summaries and oasis_load_resident per layer
 * before its first step.  Errors: OASIS_EINVAL for a bad configuration, a
 * null or misaligned buffer (16 bytes; the workspace 256) or a host store
 * that is not page-locked memory mapped for the device; OASIS_ENOMEM if a
 * stream or event cannot be created; OASIS_ECUDA for a failed CUDA call.
 * *out is NULL on failure. */
OASIS_API int oasis_init(const oasis_config* cfg, const oasis_buffers* bufs,
                         oasis_ctx** out);

/* Wait for the context's work and release its streams, events and threads
 * (not the caller's buffers).  NULL is accepted. */
OASIS_API int oasis_destroy(oasis_ctx* ctx);

/* Message for the last failed call on ctx (never NULL). */
OASIS_API const char* oasis_last_error(const oasis_ctx* ctx);

/* Wait for all work of the device and return OASIS_EDEVICE if
 * a kernel raised a device error bit since the last oasis_sync (the bits are
 * then cleared; *device_bits receives them when non-NULL). */
OASIS_API int oasis_sync(oasis_ctx* ctx, uint32_t* device_bits);

/* Support (a0): per-block min/max key summaries of `layer` over the tokens
 * below ctx_len[table] ([R] *What carries the argument*: Quest-style
 * per-block min/max key summaries).  Reads the pinned host store through its device mapping. */
OASIS_API int oasis_build_summaries(oasis_ctx* ctx, int layer, int table,
                                    void* stream);

/* Support: take res_ids[first_step & 1] (written by the caller; ids distinct
 * per (r, h), -1 = empty) as the resident set at the start of step
 * first_step, set phys[first_step & 1] to the identity (slot s -> unit s,
 * spares K..U-1), set every stamp to -1 and copy the resident blocks from the
 * host store into the pool. */
OASIS_API int oasis_load_resident(oasis_ctx* ctx, int layer, int first_step,
                                  void* stream);

/* Support (resume from saved state): oasis_load_resident that keeps the
 * stamps the caller wrote into the stamps buffer.  The state of a layer
 * between steps is its caller-owned buffers: res_ids[t & 1], stamps and
 * ctx_len[t & 1] (plus, with a remote tier, its local map and tier); saving
 * them after step t - 1 and resuming with this call at first_step = t gives
 * the same results as continuing. */
OASIS_API int oasis_resume_resident(oasis_ctx* ctx, int layer, int first_step,
                                    void* stream);

/* a1: look-ahead attention ([R] *What carries the argument*, [V]
 * key_machinery: a single attention pass serves both the normal and the draft
 * token, reading one shared resident sparse set).  For every request r and
 * query head j, separately for q and each of the D draft planes of q_draft:
 * softmax(x . k / scale) . v over the valid tokens of the occupied slots of
 * KV head j / G in table (step & 1).  A block's valid tokens are those below
 * ctx_len[step & 1][r]; a head with no valid token outputs zeros. */
OASIS_API int oasis_lookahead_attn(oasis_ctx* ctx, int layer, int step,
                                   const void* q, const void* q_draft,
                                   void* out, void* out_draft, void* stream);

/* Dense anchor: full-context decode attention with the whole KV cache in HBM,
 * the dense baseline the pages compare against ([S] throughput table: dense
 * vLLM).  Same outputs as oasis_lookahead_attn, but over every block
 * b < ceil(ctx_len[table][r] / B) of the caller's dense cache
 * kv_dense [R][Hkv][NBmax][2][B][d] bf16 (device memory, 16-byte aligned;
 * the same layout as the host store).  Uses no resident table. */
OASIS_API int oasis_dense_attn(oasis_ctx* ctx, const void* kv_dense, int table,
                               const void* q, const void* q_draft, void* out,
                               void* out_draft, void* stream);

/* a2 + a3: summary scan and head-wise top-K ([R] *What carries the argument*:
 * the draft query ranks every logical block per KV head from the compressed
 * summaries alone, never touching the full keys).  For every (r, h) and every
 * logical block b < ceil(ctx_len[step & 1][r] / B):
 *   s[b] = sum_{e < D} sum_{j in group(h)} sum_i
 *            max(qd_eji * min_bi, qd_eji * max_bi)
 * then topk_ids = the first min(K, NB_r) blocks by (s desc, b asc), -1
 * padded; topk_scores (nullable) the matching s (fp32) or -inf. */
OASIS_API int oasis_score_topk(oasis_ctx* ctx, int layer, int step,
                               const void* q_draft, int32_t* topk_ids,
                               float* topk_scores, void* stream);

/* a4: capped least-recently-selected eviction ([R] *What carries the
 * argument*: every admitted block that is not resident replaces the resident
 * block selected least recently, under a per-step cap), per (r, h), from
 * table (step & 1) into table
 * ((step + 1) & 1):
 *   (i)   stamp = step for every slot whose block is in topk_ids;
 *   (ii)  M = blocks of topk_ids not resident, in rank order;
 *   (iii) E = slots whose block is not in topk_ids, ordered empty first, then
 *         by (stamp, block id, slot) ascending;
 *   (iv)  n = min(|M|, C);
 *   (v)   for i < n: evict_ids[i] = block of E[i]; slot E[i] takes M[i] with
 *         stamp = step; admit_ids[i] = M[i], admit_slots[i] = E[i]; the
 *         admitted block is assigned the spare pool unit phys[K + i] and the
 *         evicted unit becomes that spare.
 * topk_ids must hold distinct ids.  Output lists are -1 padded to C. */
OASIS_API int oasis_admit_evict(oasis_ctx* ctx, int layer, int step,
                                const int32_t* topk_ids, int32_t* admit_ids,
                                int32_t* admit_slots, int32_t* evict_ids,
                                int32_t* n_admit, void* stream);

/* a2 + a3 + a4 without caller scratch: oasis_score_topk followed by
 * oasis_admit_evict on `stream`, with the top-K list between the two held in
 * a fixed file-scope device array of the library (1 MiB: at most 262144 =
 * R x Hkv x K entries; a larger configuration is refused with OASIS_EINVAL
 * and a message) instead of a buffer the caller allocates.  The pages have
 * no counterpart: it exists for callers that cannot allocate device memory
 * where they issue the step (device memory fully committed to the KV pool
 * and summaries, or an allocator that may not be entered from the thread
 * driving the decode loop).  Outputs and table updates are those of the two
 * calls.  The scratch's device address is looked up once per device, with
 * that device current, on the first call: make that first call before any
 * stream capture.  The address is kept for the life of the process: after
 * cudaDeviceReset (or anything else that destroys the device's primary
 * context) it is stale, so do not call this entry point again in that
 * process.  Nothing in the scratch needs to start at zero.  The
 * scratch is shared by every context and layer in the process: two calls
 * whose work may overlap on the device (other streams, layers or contexts
 * without ordering between them) race on it, so order them (one stream, or
 * events). */
OASIS_API int oasis_score_admit_noalloc(oasis_ctx* ctx, int layer, int step,
                                        const void* q_draft, int32_t* admit_ids,
                                        int32_t* admit_slots, int32_t* evict_ids,
                                        int32_t* n_admit, void* stream);

/* a5: prefetch gather ([V] supporting_citations: a gather kernel reads the
 * selected blocks from pinned CPU memory through CUDA UVA).  For every (r, h) and i < n_admit: copy host
 * unit (r, h, admit_ids[i]) into pool unit phys[(step + 1) & 1][admit_slots[i]]
 * (byte copy of keys and values).  Those units are spares of table (step & 1),
 * so the copy may run while step `step`'s attention reads that table. */
OASIS_API int oasis_prefetch(oasis_ctx* ctx, int layer, int step,
                             const int32_t* admit_ids,
                             const int32_t* admit_slots,
                             const int32_t* n_admit, void* stream);

/* ------------------------------------------------------------------------
 * Miss stall (the other outcome of a look-ahead miss; [R] *What would settle
 * it*: a block the look-ahead did not bring is either dropped from attention
 * or fetched on demand, which stalls the step).  The look-ahead path above
 * drops; these calls stall.  Reading: a miss is a block of the step's own
 * normal query's top-K that is not resident when the step starts.  The step
 * ranks every block with the normal query (a2 + a3 with q as the one plane
 * of query vectors), admits every missing block of that top-K at once (a4's
 * rule, but uncapped and in place in table (step & 1): the admitted block is
 * written into the evicted slot's own pool unit), copies those units on the
 * critical path, and only then attends; the look-ahead part of the step
 * follows unchanged on the updated table.  Uncapped because a demand fetch
 * that stopped at C would still drop context.  Not available with a remote
 * tier (OASIS_ESTATE).  Demand lists are [R][Hkv][K] int32 (-1 padded) and
 * n_admit [R][Hkv].
 * ------------------------------------------------------------------------ */

/* a2 + a3 for the demand fetch: oasis_score_topk with the normal query q
 * ([R][Hq][d] bf16, one plane whatever num_drafts is) in place of the draft
 * queries.  topk_scores is nullable. */
OASIS_API int oasis_demand_topk(oasis_ctx* ctx, int layer, int step, const void* q,
                                int32_t* topk_ids, float* topk_scores, void* stream);

/* a4 for the demand fetch, per (r, h), in place in table (step & 1) and the
 * stamps: steps (i)-(v) of oasis_admit_evict with n = |M| (no cap); slot
 * E[i] takes M[i] and keeps its pool unit phys[step & 1][E[i]], which
 * oasis_fetch_demand then overwrites.  Every block of topk_ids is resident
 * afterwards.  topk_ids must hold distinct ids.  Lists [R][Hkv][K]. */
OASIS_API int oasis_admit_demand(oasis_ctx* ctx, int layer, int step, const int32_t* topk_ids,
                                 int32_t* admit_ids, int32_t* admit_slots,
                                 int32_t* evict_ids, int32_t* n_admit, void* stream);

/* a5 for the demand fetch: for every (r, h) and i < n_admit, copy host unit
 * (r, h, admit_ids[i]) into pool unit phys[step & 1][admit_slots[i]], one
 * warp per (r, h).  That unit belongs to table (step & 1): nothing may read
 * the table's pool concurrently (order the call before the step's
 * attention and after the layer's previous gathers). */
OASIS_API int oasis_fetch_demand(oasis_ctx* ctx, int layer, int step,
                                 const int32_t* admit_ids, const int32_t* admit_slots,
                                 const int32_t* n_admit, void* stream);

/* One miss-stall layer-step.  On `stream`: wait for this layer's previous
 * side work; the demand ranking and uncapped admission (fused, one kernel);
 * the demand gather; the attention (a1) of q and the draft queries over the
 * updated table (step & 1).  On the side streams, after the demand
 * admission: the look-ahead scan + top-K + capped admission (table
 * (step & 1) -> ((step + 1) & 1)) and its gathers, as in oasis_step.
 * cfg.schedule is not used (the order is fixed).  Outputs as oasis_step;
 * the demand lists are read with oasis_stall_lists, the look-ahead lists
 * with oasis_step_lists.  Steps of one layer may mix oasis_step and
 * oasis_step_stall (consecutive step numbers). */
OASIS_API int oasis_step_stall(oasis_ctx* ctx, int layer, int step, const void* q,
                               const void* q_draft, void* out, void* out_draft,
                               void* stream);

/* Pointers to the demand lists oasis_step_stall(layer, step) writes (any
 * output may be NULL), double-buffered by step parity like
 * oasis_step_lists: valid until the stall step step + 2 is issued. */
OASIS_API int oasis_stall_lists(oasis_ctx* ctx, int layer, int step, int32_t** topk_ids,
                                float** topk_scores, int32_t** admit_ids,
                                int32_t** admit_slots, int32_t** evict_ids,
                                int32_t** n_admit);

/* a1..a5 as one layer-step (a6; [R] *What carries the argument*: the
 * background work synchronises per layer).
 * Except in the scan-first schedule (the default), q_draft is first copied
 * (on `stream`) into a per-layer staging buffer; scan-first scans read it in
 * place, since `stream` waits for them before the attention.  Side work, on the context's two high-priority side streams, ordered after
 * everything already on `stream` (so after this layer's previous attention):
 * a2+a3 fused with a4 per request group, each group's a5 gather as soon as
 * its admissions exist; results go to the context's workspace lists.  On
 * `stream`: wait for this layer's previous side work (its admissions must be
 * in the pool), with OASIS_SCHEDULE_SCAN_FIRST also for this step's scans,
 * then a1.  Returns at once; q and q_draft may be reused once `stream`
 * passes the call.  The next oasis_step of the layer (or oasis_join) orders
 * the side work before its attention. */
OASIS_API int oasis_step(oasis_ctx* ctx, int layer, int step, const void* q,
                         const void* q_draft, void* out, void* out_draft,
                         void* stream);

/* Host-side bounded wait for this layer's outstanding side work (the last
 * oasis_step's scan, admission and gathers; with a remote tier also its
 * network transfers): polls an event until it completes (OASIS_OK) or
 * `timeout_ms` passes (OASIS_ETIMEOUT; the work keeps running and a later
 * wait may succeed).  OASIS_OK at once when no side work is outstanding. */
OASIS_API int oasis_wait(oasis_ctx* ctx, int layer, double timeout_ms);

/* Make `stream` wait for this layer's outstanding side work (event wait, no
 * host block). */
OASIS_API int oasis_join(oasis_ctx* ctx, int layer, void* stream);

/* oasis_step with host buffers: q/q_draft are copied from (pinned) host
 * memory into a workspace slot of the step's parity on the context's input
 * stream (after the slot's previous reader, step - 2, is done, so the copies
 * can overlap the previous step), `stream` waits for them, the step runs, and
 * out/out_draft are copied back to host memory on `stream`.  Everything is
 * complete when `stream` passes the call; host buffers must stay valid until
 * then. */
OASIS_API int oasis_step_host(oasis_ctx* ctx, int layer, int step,
                              const void* q_host, const void* q_draft_host,
                              void* out_host, void* out_draft_host,
                              void* stream);

/* oasis_step_host whose outputs go back on the context's own output stream
 * instead of `stream`: the copies of step t then overlap the following
 * steps.  The inputs are read as in oasis_step_host; out/out_draft are
 * complete once oasis_wait_outputs(layer, t) returns OASIS_OK (or the device
 * is synchronised), and must stay valid until then.  Outputs are
 * double-buffered by step parity: the attention of step t + 2 waits for the
 * copies of step t.  Nothing of the pages corresponds to this call; it is the
 * asynchronous form of the host-buffer step. */
OASIS_API int oasis_step_host_async(oasis_ctx* ctx, int layer, int step,
                                    const void* q_host, const void* q_draft_host,
                                    void* out_host, void* out_draft_host,
                                    void* stream);

/* Bounded host wait for the outputs of the host-buffer step `step` of
 * `layer` (oasis_step_host_async, or oasis_step_host) to be in host memory:
 * OASIS_OK, OASIS_ETIMEOUT after timeout_ms (>= 0), OASIS_ESTATE if the
 * layer's latest host steps do not include `step` (only the last two are
 * tracked, by parity). */
OASIS_API int oasis_wait_outputs(oasis_ctx* ctx, int layer, int step,
                                 double timeout_ms);

/* Pointers to the workspace lists that oasis_step(layer, step) writes
 * (topk_ids, topk_scores, admit_ids, admit_slots, evict_ids, n_admit; any
 * may be NULL).  The lists are double-buffered by step parity: those of step
 * t stay valid until oasis_step(layer, t + 2) is issued. */
OASIS_API int oasis_step_lists(oasis_ctx* ctx, int layer, int step,
                               int32_t** topk_ids, float** topk_scores,
                               int32_t** admit_ids, int32_t** admit_slots,
                               int32_t** evict_ids, int32_t** n_admit);

/* Support (a0, growing contexts): append one token per request to `layer`.
 * k_new, v_new: dev [R][Hkv][d] bf16.  The token goes to position
 * p = ctx_len[step & 1][r]: written into the host store (with a remote tier:
 * into the block's local slot, see below), folded into the tail block's
 * summary (a new block starts at min = max = key), and written into the
 * resident copy if block p / B is resident in table ((step + 1) & 1).  Runs
 * after the layer's side work of step `step`. */
OASIS_API int oasis_append_token(oasis_ctx* ctx, int layer, int step,
                                 const void* k_new, const void* v_new,
                                 void* stream);

/* Support: blocks the caller rewrote in `layer`'s host store before step
 * `step` (a workload whose hot blocks move between steps).  ids: dev
 * [R][Hkv][max_ids] int32, n_ids: dev [R][Hkv] int32; for every (r, h) and
 * i < n_ids, block ids[.., i] (< NBmax; -1 = skip) gets its summary rebuilt
 * over the tokens below ctx_len[step & 1][r] and, if it is resident in table
 * (step & 1), its pool unit rewritten from the host store.  Runs after the
 * layer's side work of step - 1.  Refused (OASIS_ESTATE) with a remote tier. */
OASIS_API int oasis_refresh_blocks(oasis_ctx* ctx, int layer, int step,
                                   const int32_t* ids, const int32_t* n_ids,
                                   int max_ids, void* stream);

/* ctx_len[(step + 1) & 1][r] = ctx_len[step & 1][r] + grow for every r. */
OASIS_API int oasis_advance_context(oasis_ctx* ctx, int step, int grow,
                                    void* stream);

/* ------------------------------------------------------------------------
 * Remote tier: emulation of prefill-decode disaggregation with remote partial
 * fetch ([R] abstract and *If this is right*: under disaggregation a request
 * is admitted to the decode node with a fraction of its KV, and the decode
 * node's host memory holds only part of the cache; [S] result table, PD row).
 *
 * Reading.  The full KV cache stays on the prefill side (the remote tier);
 * the decode side keeps a host tier of `capacity` local slots per (r, h).  A
 * block enters the local tier the first time the decode side needs it (the
 * initial resident set at oasis_load_resident, then every admitted block that
 * is not yet held) and stays there; the gather always copies from the local
 * tier into HBM.  Local slots are assigned in list order (admission rank
 * order) from 0 upwards.  Summaries are built from the remote store (they are
 * shipped with the request).  The network transfer remote -> local is done on
 * the host, as a NIC's DMA would be: a worker thread of the tier, told by the
 * stream (a 32-bit write after the slot assignment) that the lists are ready,
 * copies the listed units with a pool of `threads` host threads, optionally
 * throttled to `gbps`, and writes the transfer's number back; it moves no
 * data through the GPU.  The gather then runs in two launches on its stream:
 * the admitted units already held locally at once, beside the transfer, and
 * the units just fetched after a stream wait for that number.
 *
 * With a remote tier attached to a layer, host_kv (given to oasis_init) is the
 * remote store, pinned and mapped as before.  oasis_load_resident also brings
 * the block each request's context ends in (if it ends inside a block) to the
 * local tier, since decoding appends there; oasis_append_token then writes a
 * decoded token into its block's local slot, a block the token opens taking
 * the next free slot (OASIS_DEVERR_NOT_LOCAL if none is left), and never into
 * the remote store.  oasis_refresh_blocks is refused (OASIS_ESTATE).
 *
 * Layouts:
 *   local_tier pinned [R][Hkv][capacity][2][B][d]   bf16   local slots
 *   local_map  dev    [R][Hkv][NBmax] int32 (local slot of each block, -1 =
 *                     not held), then [R][Hkv] int32 (slots in use), then
 *                     [R][Hkv] int32 (slots in use before the last assignment)
 *   miss_lists pinned [R][Hkv] int32 n_miss, then [R][Hkv][M] int32 ids, then
 *                     [R][Hkv][M] int32 slots, M = max(K, C): the blocks the
 *                     last slot assignment of each (r, h) fetched, in order;
 *                     then (16-byte aligned) two uint32 sequence words the
 *                     stream and the tier's worker thread hand over with
 * ------------------------------------------------------------------------ */
typedef struct {
  int32_t capacity; /* local slots per (r, h): K <= capacity <= NBmax */
  float gbps;       /* emulated network bandwidth in 1e9 bytes/s; 0 = no throttle */
  int32_t threads;  /* host copy threads per transfer, 1..16 (0 = 4) */
} oasis_remote_config;

typedef struct {
  size_t local_tier_bytes; /* per layer, pinned host */
  size_t local_map_bytes;  /* per layer, device */
  size_t miss_lists_bytes; /* per layer, pinned host */
} oasis_remote_sizes;

OASIS_API int oasis_remote_query_sizes(const oasis_config* cfg,
                                       const oasis_remote_config* rcfg,
                                       oasis_remote_sizes* out);

/* Attach a remote tier to `layer` before its oasis_load_resident.  The
 * buffers are lent for the life of the context (16-byte aligned; local_tier
 * and miss_lists page-locked and mapped for the device).  Clears local_map
 * (every block not held, no slot in use); synchronises.  Errors: OASIS_EINVAL
 * on a bad size or pointer, OASIS_ESTATE once the layer is loaded. */
OASIS_API int oasis_remote_attach(oasis_ctx* ctx, int layer,
                                  const oasis_remote_config* rcfg,
                                  void* local_tier, int32_t* local_map,
                                  int32_t* miss_lists);

/* Totals of the layer's emulated network transfers since attach: units
 * (8 KiB each) moved remote -> local, transfers made, and seconds the
 * worker spent copying (throttle included); bad_entries counts list entries
 * the worker skipped as out of range, plus transfers it gave up waiting for
 * (0 unless something went wrong).
 * Read after oasis_sync for a settled value.  Any output may be NULL. */
OASIS_API int oasis_remote_stats(oasis_ctx* ctx, int layer, int64_t* units,
                                 int64_t* transfers, double* seconds,
                                 int64_t* bad_entries);

/* Time limit of the kernels' bounded barrier waits, in GPU clock cycles,
 * for the launches that follow (attention, scan).  cycles <= 0 restores the
 * default (2e9 cycles, about a second).  A wait that runs out sets
 * OASIS_DEVERR_TIMEOUT (reported by oasis_sync) and its kernel ends early
 * with undefined outputs; copies the kernel has already issued are still
 * waited for with the default limit before it exits.  Nothing of the pages
 * corresponds to this call: it lets a test take the timeout path on purpose
 * (a limit of a few cycles runs out before any copy lands). */
OASIS_API int oasis_set_wait_limit(oasis_ctx* ctx, long long cycles);

/* Kernel timing: when enabled, the step calls (oasis_step, oasis_step_stall)
 * and the stage calls record CUDA events around each of their kernels on the
 * stream that launches it. */
OASIS_API int oasis_profile_enable(oasis_ctx* ctx, int enable);

/* Kinds of timed launches, in this order: attention, summary scan (a2;
 * with OASIS_SCAN=fused in the environment the one-kernel scan + top-K +
 * admission), admit_evict, prefetch, demand scan (or a stand-alone demand
 * admission), demand gather, top-K ranking (a3, with the admission fused
 * into it in the step calls). */
#define OASIS_PROFILE_KINDS 7

/* Sum of kernel durations (ms) and launch counts since the last read, for
 * the first nkinds (1..OASIS_PROFILE_KINDS) kinds; start_ms_sum (nullable)
 * receives the summed start offsets of those launches from the start of
 * their step.  Launches of the other kinds are discarded.  Synchronises. */
OASIS_API int oasis_profile_read_n(oasis_ctx* ctx, int nkinds, double* ms_sum,
                                   int64_t* count, double* start_ms_sum);

/* oasis_profile_read_n with nkinds = 4. */
OASIS_API int oasis_profile_read(oasis_ctx* ctx, double* ms_sum4,
                                 int64_t* count4, double* start_ms_sum4);

#ifdef __cplusplus
}
#endif
#endif
