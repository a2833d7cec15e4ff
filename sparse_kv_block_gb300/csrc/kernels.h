// kernels.h -- host-side launchers of the look-ahead sparse decode kernels.
// Plain C++ structs, no torch types; used by the C ABI in api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace oasis {

struct AttnArgs {
  const void* q;         // [R][Hq][d] bf16
  const void* qd;        // [D][R][Hq][d] bf16
  void* out;             // [R][Hq][d] bf16 or fp32
  void* outd;            // [D][R][Hq][d] bf16 or fp32
  const int32_t* res;    // [R][Hkv][K]  table of this step
  const int32_t* phys;   // [R][Hkv][U]  table of this step
  const int32_t* ctx_len;  // [R]        table of this step
  uint32_t* err;
  int R, Hq, Hkv, G, K, U, NBmax;
  int D;                 // draft queries per step, 1..3
  float scale_log2;      // softmax scale * log2(e)
  int out_fp32;
  // dense = 1: no resident table; every block b < ceil(ctx_len / B) of a pair
  // is read from unit pair * NBmax + b of a dense [R][Hkv][NBmax] cache.
  int dense;
  long long wait_limit;  // clock cycles a barrier wait may take (drains excepted)
};

// Pairs (request, KV head) are flattened as pair = r * Hkv + h; a launch
// covers pairs [pair0, pair0 + pairs).
struct AdmitArgs {
  const int32_t* topk;       // [R][Hkv][K]
  const int32_t* res_cur;    // [R][Hkv][K]
  int32_t* res_nxt;          // [R][Hkv][K]
  int32_t* stamps;           // [R][Hkv][K]
  const int32_t* phys_cur;   // [R][Hkv][U]
  int32_t* phys_nxt;         // [R][Hkv][U]
  int32_t* admit_ids;        // [R][Hkv][C]
  int32_t* admit_slots;      // [R][Hkv][C]
  int32_t* evict_ids;        // [R][Hkv][C]
  int32_t* n_admit;          // [R][Hkv]
  int R, Hkv, K, C, U, NBmax, step;
  int pair0, pairs;
  // in_place = 1 (the miss-stall demand fetch): res_nxt == res_cur and
  // phys_nxt == phys_cur; an admitted block goes into its slot's own pool
  // unit (no spare swap), so C may be up to K.
  int in_place;
};

struct ScoreArgs {
  const void* qd;        // [D][R][Hq][d] bf16
  const void* summ;      // [R][Hkv][NBmax][2][d] bf16
  const int32_t* ctx_len;  // [R]
  int32_t* topk_ids;     // [R][Hkv][K]
  float* topk_scores;    // [R][Hkv][K] or null
  uint32_t* err;
  int R, Hq, Hkv, G, K, NBmax;
  int D;                 // draft queries per step, 1..3 (their bounds add up)
  int pair0, pairs;
  int fuse_admit;        // run the capped eviction of each pair in the tail
  AdmitArgs admit;       // used when fuse_admit (its topk field is ignored)
  // scores_ws set: the scan writes every block's fp32 score to
  // scores_ws[pair][b] and a separate kernel ranks them (and admits, when
  // fused); null: one kernel ranks while it scans (no scratch).
  float* scores_ws;      // [R][Hkv][NBmax]
  long long wait_limit;  // clock cycles a barrier wait may take (drains excepted)
};

// Copies 8 KiB units host -> pool.  Item i of pair p = (r, h) reads block
// src_ids[p*items + i] (skipped if < 0 or i >= n_valid[p]) and writes pool
// unit phys[p*U + slot], slot = dst_slots ? dst_slots[p*items + i] : i.
struct GatherArgs {
  const void* host;          // device alias of the pinned store
  void* pool;
  const int32_t* src_ids;
  const int32_t* dst_slots;  // may be null
  const int32_t* n_valid;    // may be null
  const int32_t* phys;
  // Remote tier: when set, the host store is the local tier of src_units
  // slots per pair and block id b of pair p is read from slot
  // local_map[p*NBmax + b]; otherwise src_units = NBmax and slot = b.
  const int32_t* local_map;
  // phase 0: every item; 1: only items whose local slot < base[p] (held
  // before the last slot assignment); 2: only the others.
  const int32_t* base;
  int phase;
  uint32_t* err;
  int pair0, pairs, items, NBmax, U, src_units;
  // pair_major = 1: one warp per pair walks only that pair's n_valid items
  // (lists padded far beyond their use, such as the miss-stall demand
  // fetch); 0: one warp per (pair, item), the grid capped for the host link.
  int pair_major;
  // Item-major mode: CTAs at most (0: the launcher's default).
  int max_ctas;
};

// Remote tier slot assignment: item i of pair p names block
// ids[p*items + i] (skipped if < 0 or i >= n_valid[p]); every named block
// without a local slot gets slot count[p]++ (in item order) while
// count[p] < capacity, and is listed in miss_ids / miss_slots [p][M] with
// n_miss[p] entries; base[p] receives count[p] before the assignment.  The
// lists may live in mapped host memory.
struct RemoteArgs {
  const int32_t* ids;
  const int32_t* n_valid;    // may be null
  int32_t* local_map;        // [R][Hkv][NBmax]
  int32_t* count;            // [R][Hkv]
  int32_t* base;             // [R][Hkv]
  int32_t* n_miss;           // [R][Hkv]
  int32_t* miss_ids;         // [R][Hkv][M]
  int32_t* miss_slots;       // [R][Hkv][M]
  uint32_t* err;
  int pair0, pairs, items, NBmax, capacity, M;
};

struct SummaryArgs {
  const void* host;          // device alias of the pinned store
  void* summ;
  const int32_t* ctx_len;
  int R, Hkv, NBmax;
};

// Blocks the caller rewrote in the host store: for every pair p and
// i < n_ids[p], block ids[p*max_ids + i] gets its summary rebuilt (tokens
// below ctx_len[r]) and, if resident in (res, phys), its pool unit rewritten.
struct RefreshArgs {
  const void* host;          // device alias of the pinned store
  void* summ;
  void* pool;
  const int32_t* ids;        // [R][Hkv][max_ids]
  const int32_t* n_ids;      // [R][Hkv]
  const int32_t* ctx_len;    // [R]
  const int32_t* res;        // [R][Hkv][K]
  const int32_t* phys;       // [R][Hkv][U]
  uint32_t* err;
  int R, Hkv, NBmax, K, U, max_ids;
};

struct AppendArgs {
  const void* k_new;         // [R][Hkv][d]
  const void* v_new;
  void* host;                // device alias of the pinned store (or local tier)
  // Remote tier: the token goes to the block's local slot; a block that
  // starts with this token gets the next free slot (count[p]++ while below
  // capacity).  Null without a remote tier.
  int32_t* local_map;        // [R][Hkv][NBmax]
  int32_t* local_count;      // [R][Hkv]
  int capacity;
  void* summ;
  void* pool;
  const int32_t* ctx_len;    // the step's table
  const int32_t* res_nxt;
  const int32_t* phys_nxt;
  uint32_t* err;
  int R, Hkv, NBmax, K, U;
};

cudaError_t launch_attention(const AttnArgs& a, const CUtensorMap* pool_map,
                             cudaStream_t s);
// Scan + top-K (+ admission) in one kernel, no scratch used.
cudaError_t launch_score_topk(const ScoreArgs& a, cudaStream_t s);
// The same as two kernels: the scan writes every block's score to
// a.scores_ws, then the ranking (and admission) reads them back.  Used when
// scan_is_split(NBmax).
bool scan_is_split(int NBmax);
cudaError_t launch_scan_scores(const ScoreArgs& a, cudaStream_t s);
cudaError_t launch_topk_select(const ScoreArgs& a, cudaStream_t s);
cudaError_t launch_admit(const AdmitArgs& a, cudaStream_t s);
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s);
cudaError_t launch_remote_assign(const RemoteArgs& a, cudaStream_t s);
cudaError_t launch_init_tables(int32_t* phys, int32_t* stamps, int pairs,
                               int K, int U, cudaStream_t s);
cudaError_t launch_summary_build(const SummaryArgs& a, cudaStream_t s);
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);
cudaError_t launch_refresh(const RefreshArgs& a, cudaStream_t s);
// tail[p] = last block of request p / Hkv if its context ends inside a block,
// else -1 (the blocks a decode side appends into first).
cudaError_t launch_tail_blocks(const int32_t* ctx_len, int R, int Hkv, int32_t* tail,
                               cudaStream_t s);
cudaError_t launch_advance(const int32_t* cur, int32_t* nxt, int R, int grow,
                           cudaStream_t s);


// Load every kernel's code now (the runtime loads modules lazily on first
// launch, and a lazy load waits for work already queued on the device).
cudaError_t preload_attention_kernels();
cudaError_t preload_score_kernels();
cudaError_t preload_support_kernels();

// Largest NBmax the fused score + admit kernel can hold in shared memory.
constexpr int kMaxBlocksPerHead = 131072;

// oasis_score_admit_noalloc: entries of its file-scope top-K scratch, and the
// scratch's device address (looked up once per device, with that device
// current, on the first call).
constexpr size_t kNoAllocTopkEntries = 262144;
cudaError_t noalloc_topk_scratch(int device, int32_t** ptr);

}  // namespace oasis
