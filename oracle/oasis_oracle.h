/*
 * oasis_oracle.h -- plain, slow, sequential CPU restatement of OasisKV's
 * per-layer look-ahead sparse decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this code: only the test suite, the package smoke check and
 * the benchmark's CPU-baseline / reference arm use it.  It shares no code,
 * header, constant or helper with the CUDA library (include/oasis.h).
 *
 * Sources (page titles and sections):
 *   [R]  "Pith review of OasisKV: Scaling In-Decode KV Cache Beyond HBM with
 *         Lookahead Sparse Prefetching" (pith.science), section "What carries
 *         the argument"; "Assumptions & free parameters"; the abstract.
 *   [S]  "OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse
 *         Prefetching" (agihunt.info summary), the fetch-cap ablation paragraph.
 *   [V]  pith.science verdict record for arXiv 2608.08097, field
 *         "key_machinery".
 *
 * Arithmetic: bf16 inputs are held as raw uint16 bit patterns and widened to
 * double by a 16-bit shift; every sum is taken in double and rounded once.
 *
 * Layouts (row-major, innermost last):
 *   host_kv [R][Hkv][NBmax][2][B][d]  bf16   (index 0 = keys, 1 = values)
 *   summ    [R][Hkv][NBmax][2][d]     bf16   (index 0 = min row, 1 = max row)
 *   q       [R][Hq][d]                bf16   (normal queries)
 *   qd      [D][R][Hq][d]             bf16   (D >= 1 draft queries per step)
 *   res     [R][Hkv][K]               int32  (logical block id per slot, -1 = empty)
 *   stamp   [R][Hkv][K]               int32  (step of last selection, -1 = never)
 *   topk    [R][Hkv][K]               int32  (block ids in rank order, -1 pad)
 * Query head j reads KV head j / (Hq / Hkv).
 *
 * Every function returns 0 on success and -1 on an argument error.
 *
 * Parity pins: every function below is pinned by tests under tests/ against
 * closed forms, brute force or library routines (see test_oracle_pins.py).
 */
#ifndef OASIS_ORACLE_H
#define OASIS_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

/* Per-block coordinate-wise min/max of the keys over the block's valid tokens
 * ([R] *What carries the argument*: Quest-style compressed summaries, one
 * min and one max per coordinate and block).  Blocks b < ceil(ctx_len[r]/B) are written; others are
 * left untouched. */
int orc_summary_build(const uint16_t* host_kv, const int32_t* ctx_len, int R,
                      int Hkv, int NBmax, int B, int d, uint16_t* summ);

/* Sparse attention of one (request r, KV head h) over its resident blocks,
 * for the normal query and every draft query of each of the G query heads of
 * the group ([R] *What carries the argument*: one attention pass handles the
 * normal and the draft token, both reading the one resident block set; with
 * D > 1 drafts every draft reads that same set).
 * out[1 + D][G][d] (fp32): out[0] for q, out[1 + e] for draft e. */
int orc_attention_rh(const uint16_t* host_kv, const int32_t* ctx_len,
                     const int32_t* res, const uint16_t* q, const uint16_t* qd,
                     int D, int R, int Hq, int Hkv, int NBmax, int B, int d,
                     int K, double scale, int r, int h, float* out);

/* Summary score of every logical block b < ceil(ctx_len[r]/B) for one
 * (r, h): s[b] = sum over the drafts e, the group's query heads j and dims i
 * of max(qd[e][j][i]*min[b][i], qd[e][j][i]*max[b][i])  ([R] *What carries
 * the argument*: the draft query is scored against the summaries; several
 * drafts are read as further query vectors of the group, their bounds summed
 * like those of the group's heads).  scores[NBmax] (fp32, one rounding of a
 * double sum); entries b >= NB_r are set to -inf. */
int orc_score_rh(const uint16_t* summ, const int32_t* ctx_len,
                 const uint16_t* qd, int D, int R, int Hq, int Hkv, int NBmax,
                 int d, int B, int r, int h, float* scores);

/* Head-wise top-K of one (r, h): the first min(K, NB) block ids ordered by
 * (score descending, id ascending); the rest of topk[K] is -1
 * ([R] *What carries the argument*: every logical block is ranked per KV
 * head). */
int orc_topk_rh(const float* scores, int NB, int K, int32_t* topk);

/* Capped eviction for one (r, h) at step t ([R] *What carries the
 * argument*: each admitted non-resident block displaces the resident block
 * selected least recently; [S] fetch cap).  Updates res[K] and stamp[K] in place and
 * writes admit_ids/admit_slots/evict_ids[C] (-1 padded) and *n_admit. */
int orc_admit_evict_rh(int32_t* res, int32_t* stamp, const int32_t* topk,
                       int K, int C, int step, int32_t* admit_ids,
                       int32_t* admit_slots, int32_t* evict_ids,
                       int32_t* n_admit);

/* One whole layer-step for one (r, h): attention (on the resident set as it
 * stands at the start of the step) -> summary score -> top-K -> capped
 * eviction.  The prefetch needs no work on this logical view: the oracle
 * reads block contents straight from the host store.  scores_scratch needs
 * NBmax floats.  Outputs as in the functions above. */
int orc_step_rh(const uint16_t* host_kv, const uint16_t* summ,
                const int32_t* ctx_len, int32_t* res, int32_t* stamp,
                const uint16_t* q, const uint16_t* qd, int D, int R, int Hq,
                int Hkv, int NBmax, int B, int d, int K, int C, int step, double scale,
                int r, int h, float* attn_out, float* scores_scratch,
                int32_t* topk, int32_t* admit_ids, int32_t* admit_slots,
                int32_t* evict_ids, int32_t* n_admit);

/* Miss stall, the demand half, for one (r, h) at step t ([R] *What would
 * settle it*: a block the look-ahead did not bring is either dropped from
 * attention or fetched on demand, stalling the step).  The step's own normal
 * query q ([R][Hq][d], its G vectors of the group) scores every logical
 * block like a draft (orc_score_rh with one query plane), its top-K is taken
 * (orc_topk_rh) and every block of that top-K that is not resident is
 * admitted at once, without the fetch cap (orc_admit_evict_rh with C = K):
 * an on-demand fetch that stopped at the cap would still drop context.  The
 * least-recently-selected pairing and the stamps are those of the look-ahead
 * admission.  Afterwards every id of the top-K is resident.
 * scores[NBmax], topk[K]; admit_ids/admit_slots/evict_ids[K] (-1 padded). */
int orc_demand_rh(const uint16_t* summ, const int32_t* ctx_len, int32_t* res,
                  int32_t* stamp, const uint16_t* q, int R, int Hq, int Hkv,
                  int NBmax, int B, int d, int K, int step, int r, int h,
                  float* scores, int32_t* topk, int32_t* admit_ids,
                  int32_t* admit_slots, int32_t* evict_ids, int32_t* n_admit);

/* One miss-stall layer-step for one (r, h): orc_demand_rh (the demand
 * fetch, on the critical path), then orc_step_rh on the resulting table
 * (attention over a resident set that now holds the normal query's whole
 * top-K, then the look-ahead scan, top-K and capped admission of the draft
 * queries).  Outputs: the demand lists (dm_*: [K] each, scores NBmax) and
 * those of orc_step_rh. */
int orc_stall_step_rh(const uint16_t* host_kv, const uint16_t* summ,
                      const int32_t* ctx_len, int32_t* res, int32_t* stamp,
                      const uint16_t* q, const uint16_t* qd, int D, int R, int Hq,
                      int Hkv, int NBmax, int B, int d, int K, int C, int step,
                      double scale, int r, int h, float* dm_scores,
                      int32_t* dm_topk, int32_t* dm_admit_ids,
                      int32_t* dm_admit_slots, int32_t* dm_evict_ids,
                      int32_t* dm_n_admit, float* attn_out, float* scores_scratch,
                      int32_t* topk, int32_t* admit_ids, int32_t* admit_slots,
                      int32_t* evict_ids, int32_t* n_admit);

/* Remote-tier partial fetch for one (r, h) (emulated prefill-decode
 * disaggregation; [R] abstract: a request reaches the decode node with only
 * part of its KV and the decode node's host memory holds only part of the
 * cache; [S] result table, PD row).  The decode-side host tier has
 * `capacity` slots; local_map[NBmax] gives each block's slot (-1 = not held)
 * and *count the slots in use.  The ids ids[0..n) are visited in order; an id
 * < 0 is skipped; an id not yet held takes slot *count (then *count grows by
 * one) and is appended to miss_ids / miss_slots, *n_miss counting them.  When
 * no slot is left the id stays not held and the function reports 1 after
 * finishing the list; otherwise 0.  Ids are distinct and < NBmax. */
int orc_remote_fetch_rh(const int32_t* ids, int n, int32_t* local_map,
                        int32_t* count, int capacity, int NBmax,
                        int32_t* miss_ids, int32_t* miss_slots, int32_t* n_miss);

/* Append one decoded token to request r of one layer: write k_new/v_new
 * ([Hkv][d] each) at position pos = ctx_len[r] into the host store and fold
 * the key into the tail block's summary (a fresh block starts as min = max =
 * key).  ctx_len itself is not changed.  Requires pos < NBmax*B. */
int orc_append_token(uint16_t* host_kv, uint16_t* summ, const int32_t* ctx_len,
                     const uint16_t* k_new, const uint16_t* v_new, int R,
                     int Hkv, int NBmax, int B, int d, int r);

#ifdef __cplusplus
}
#endif
#endif
