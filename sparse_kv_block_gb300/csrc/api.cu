// api.cu -- the C ABI (include/oasis.h): argument validation, the context,
// the side stream and its events, the TMA descriptors and step orchestration.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <functional>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <thread>
#include <tuple>
#include <vector>

#include "../../include/oasis.h"
#include "common.cuh"
#include "kernels.h"

using namespace oasis;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Remote tier (emulated prefill-decode disaggregation).  The transfer
// remote -> local tier of the blocks a slot assignment listed runs on the
// host, as a network adapter's DMA would: no GPU work.  A worker thread per
// tier takes the transfers in issue order; the GPU and the worker hand over
// through two sequence words in mapped host memory: the stream writes a
// transfer's number after its slot assignment (the worker then reads the
// lists) and waits, before gathering the fetched units, until the worker
// has written the number back.  (A CUDA host callback doing the copy was
// measured to hold up the issuing thread's CUDA calls for as long as the
// callback ran.)
struct RemoteStats {
  std::atomic<int64_t> units{0}, transfers{0}, bad{0}, nanos{0};
};

// Persistent host copy threads of one remote tier.  run(n, f) calls
// f(lo, hi) over [0, n) in chunks claimed from an atomic counter by the
// workers and the calling thread, and returns when all chunks are done.
class CopyPool {
 public:
  explicit CopyPool(int threads) {
    for (int i = 1; i < threads; ++i) th_.emplace_back([this] { loop(); });
  }
  ~CopyPool() {
    {
      std::lock_guard<std::mutex> g(m_);
      stop_ = true;
    }
    cv_.notify_all();
    for (auto& t : th_) t.join();
  }
  void run(size_t n, const std::function<void(size_t, size_t)>& f) {
    std::lock_guard<std::mutex> one(run_m_);
    if (th_.empty() || n <= kChunk) {
      f(0, n);
      return;
    }
    {
      std::lock_guard<std::mutex> g(m_);
      f_ = &f;
      n_ = n;
      next_ = 0;
      busy_ = th_.size();
      ++gen_;
    }
    cv_.notify_all();
    work();
    std::unique_lock<std::mutex> l(m_);
    done_.wait(l, [this] { return busy_ == 0; });
    f_ = nullptr;
  }

 private:
  static constexpr size_t kChunk = 8;  // units (64 KiB) per claim
  void work() {
    for (;;) {
      const size_t k = next_.fetch_add(kChunk);
      if (k >= n_) return;
      (*f_)(k, std::min(k + kChunk, n_));
    }
  }
  void loop() {
    uint64_t seen = 0;
    for (;;) {
      {
        std::unique_lock<std::mutex> l(m_);
        cv_.wait(l, [&] { return stop_ || gen_ != seen; });
        if (stop_) return;
        seen = gen_;
      }
      work();
      std::lock_guard<std::mutex> g(m_);
      if (--busy_ == 0) done_.notify_one();
    }
  }
  std::vector<std::thread> th_;
  std::mutex m_, run_m_;
  std::condition_variable cv_, done_;
  const std::function<void(size_t, size_t)>* f_ = nullptr;
  size_t n_ = 0;
  std::atomic<size_t> next_{0};
  size_t busy_ = 0;
  uint64_t gen_ = 0;
  bool stop_ = false;
};

struct RemoteJob {
  uint32_t seq = 0;                 // transfer number
  int pair0 = 0, pairs = 0;
};

// Driver entry points of the stream memory operations.
using PFN_WaitValue32 = CUresult(CUDAAPI*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
using PFN_WriteValue32 = CUresult(CUDAAPI*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
PFN_WaitValue32 get_wait_value32() {
  static PFN_WaitValue32 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &p, 11070, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_WaitValue32>(p);
    return static_cast<PFN_WaitValue32>(nullptr);
  }();
  return fn;
}
PFN_WriteValue32 get_write_value32() {
  static PFN_WriteValue32 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &p, 11070, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_WriteValue32>(p);
    return static_cast<PFN_WriteValue32>(nullptr);
  }();
  return fn;
}

// True when sequence word value v has reached s (wrap-around safe).
inline bool seq_reached(uint32_t v, uint32_t s) { return static_cast<int32_t>(v - s) >= 0; }

struct RemoteTier {
  int capacity = 0, M = 0, threads = 4, NBmax = 0, all_pairs = 0;
  double gbps = 0.0;
  const uint8_t* remote = nullptr; // the remote store, [pairs][NBmax] units
  uint8_t* local = nullptr;        // caller's pinned local tier
  void* local_dev = nullptr;       // its device mapping
  int32_t* map = nullptr;          // dev [pairs][NBmax]
  int32_t* count = nullptr;        // dev [pairs]: slots in use
  int32_t* base = nullptr;         // dev [pairs]: slots in use before the last assignment
  int32_t* lists = nullptr;        // caller's pinned miss lists
  int32_t* lists_dev = nullptr;    // their device mapping
  volatile uint32_t* assigned = nullptr;  // host view: last assignment done (GPU writes)
  volatile uint32_t* moved = nullptr;     // host view: last transfer done (worker writes)
  CUdeviceptr assigned_dev = 0, moved_dev = 0;
  uint32_t next_seq = 0;           // issue counter (API thread)
  RemoteStats stats;
  std::unique_ptr<CopyPool> pool;
  std::thread worker;
  std::mutex qm;
  std::condition_variable qcv;
  std::deque<RemoteJob> queue;
  bool stop = false;

  void start() { worker = std::thread([this] { run(); }); }
  void post(const RemoteJob& j) {
    {
      std::lock_guard<std::mutex> g(qm);
      queue.push_back(j);
    }
    qcv.notify_one();
  }
  ~RemoteTier() {
    {
      std::lock_guard<std::mutex> g(qm);
      stop = true;
    }
    qcv.notify_one();
    if (worker.joinable()) worker.join();
    if (moved) *moved = next_seq;  // nothing may wait on a transfer any more
  }

 private:
  // Transfers in issue order.  Waits (bounded, ~60 s) for the GPU to finish
  // the transfer's slot assignment, copies the listed units, holds the
  // throttle, then publishes the number; on a timeout it publishes without
  // copying and counts the lists as bad, so no stream waits forever.
  void run() {
    for (;;) {
      RemoteJob j;
      {
        std::unique_lock<std::mutex> l(qm);
        qcv.wait(l, [this] { return stop || !queue.empty(); });
        if (queue.empty()) return;
        j = queue.front();
        queue.pop_front();
      }
      const auto t0 = std::chrono::steady_clock::now();
      bool ready = true;
      for (int spin = 0; !seq_reached(*assigned, j.seq); ++spin) {
        if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(60)) {
          ready = false;
          break;
        }
        if (spin > 64) std::this_thread::sleep_for(std::chrono::microseconds(20));
      }
      std::atomic_thread_fence(std::memory_order_acquire);
      const auto t1 = std::chrono::steady_clock::now();
      size_t n = 0;
      int64_t bad = ready ? 0 : 1;
      if (ready) {
        const int32_t* n_miss = lists;
        const int32_t* ids = lists + all_pairs;
        const int32_t* slots = lists + all_pairs + static_cast<size_t>(all_pairs) * M;
        std::vector<std::pair<int, int>> items;
        for (int p = j.pair0; p < j.pair0 + j.pairs; ++p) {
          const int c = n_miss[p];
          if (c < 0 || c > M) {
            ++bad;
            continue;
          }
          for (int i = 0; i < c; ++i) {
            const size_t li = static_cast<size_t>(p) * M + i;
            if (ids[li] < 0 || ids[li] >= NBmax || slots[li] < 0 || slots[li] >= capacity) {
              ++bad;
              continue;
            }
            items.emplace_back(p, i);
          }
        }
        n = items.size();
        pool->run(n, [&](size_t lo, size_t hi) {
          for (size_t k = lo; k < hi; ++k) {
            const int p = items[k].first, i = items[k].second;
            const size_t li = static_cast<size_t>(p) * M + i;
            std::memcpy(local + (static_cast<size_t>(p) * capacity + slots[li]) * kUnitBytes,
                        remote + (static_cast<size_t>(p) * NBmax + ids[li]) * kUnitBytes,
                        kUnitBytes);
          }
        });
        if (gbps > 0.0) {
          const double sec = static_cast<double>(n) * kUnitBytes / (gbps * 1e9);
          std::this_thread::sleep_until(
              t1 + std::chrono::duration_cast<std::chrono::steady_clock::duration>(
                       std::chrono::duration<double>(sec)));
        }
      }
      const auto dt = std::chrono::steady_clock::now() - t1;
      std::atomic_thread_fence(std::memory_order_release);
      *moved = j.seq;
      stats.units += static_cast<int64_t>(n);
      stats.transfers += 1;
      stats.bad += bad;
      stats.nanos += std::chrono::duration_cast<std::chrono::nanoseconds>(dt).count();
    }
  }
};

struct LayerState {
  void* pool = nullptr;
  void* summ = nullptr;
  void* host = nullptr;      // caller's host pointer
  void* host_dev = nullptr;  // its device mapping
  int32_t* res = nullptr;    // [2][R][Hkv][K]
  int32_t* stamps = nullptr;
  int32_t* phys = nullptr;   // [2][R][Hkv][U]
  CUtensorMap pool_map;
  // Workspace lists of oasis_step, double-buffered by step parity: the
  // gathers of step t read lists[t & 1] while the admission of step t + 1
  // may already write lists[(t + 1) & 1].
  struct Lists {
    int32_t* topk_ids = nullptr;
    float* topk_scores = nullptr;
    int32_t* admit_ids = nullptr;
    int32_t* admit_slots = nullptr;
    int32_t* evict_ids = nullptr;
    int32_t* n_admit = nullptr;
  } lists[2];
  // Block scores of the split scan by step parity: every scan of step t
  // (look-ahead, demand, stage call) uses scores[t & 1].  The scans of one
  // step run one after the other; step t + 2's scans follow step t's.
  float* scan_scores[2] = {nullptr, nullptr};
  // Miss-stall demand lists (oasis_step_stall), by step parity; the
  // admission lists are [R][Hkv][K] (the demand fetch is not capped).
  Lists dm[2];
  // oasis_step_host's input staging, by step parity: the copies of step
  // t + 1 run on the context's input stream while step t computes.
  void* q_stage[2] = {nullptr, nullptr};
  void* qd_stage[2] = {nullptr, nullptr};
  cudaEvent_t ev_in[2] = {nullptr, nullptr};          // inputs of the slot copied
  cudaEvent_t ev_stage_free[2] = {nullptr, nullptr};  // last reader of the slot done
  bool stage_used[2] = {false, false};
  // Attention outputs of host-buffer steps, by step parity; with
  // oasis_step_host_async they are copied back on the context's output
  // stream, so a slot is reused only after its copy (step - 2) is done.
  void* out_stage[2] = {nullptr, nullptr};
  void* outd_stage[2] = {nullptr, nullptr};
  cudaEvent_t ev_attn_done = nullptr;                // the latest host step's attention
  cudaEvent_t ev_out_done[2] = {nullptr, nullptr};   // a slot's outputs are in host memory
  bool out_pending[2] = {false, false};
  int out_step[2] = {-1, -1};
  void* qd_ring[2] = {nullptr, nullptr};  // staged draft queries, by step parity
  cudaEvent_t ev_start = nullptr;
  cudaEvent_t ev_demand_done = nullptr;  // a stall step's demand admission written
  cudaEvent_t ev_side_done = nullptr;
  cudaEvent_t ev_scan_done = nullptr;
  // Early-scan schedule: the draft queries staged on the scan stream; the
  // admissions of a step parity done (the next scan of that parity rewrites
  // the top-K lists they read).
  cudaEvent_t ev_qd_copied = nullptr;
  cudaEvent_t ev_admitted[2] = {nullptr, nullptr};
  bool admitted_pending[2] = {false, false};
  // The library's last write of this layer's summaries (build, append,
  // refresh), which an early scan must follow.
  cudaEvent_t ev_mut = nullptr;
  bool mut_pending = false;
  std::vector<cudaEvent_t> ev_group;  // one per side-work request group
  std::vector<cudaEvent_t> ev_group2; // admissions done (three-stream schedule)
  bool side_pending = false;
  bool loaded = false;
  std::unique_ptr<RemoteTier> remote;
};

struct ProfPair {
  cudaEvent_t a, b;
  int kind;
  int start;  // index of the step-start event this launch belongs to
};

struct WsLayout {
  size_t err, per_layer;
  size_t topk_ids, topk_scores, admit_ids, admit_slots, evict_ids, n_admit;
  size_t q_stage, qd_stage, q_stage1, qd_stage1, out_stage, outd_stage, qd_ring0, qd_ring1;
  size_t out_stage1, outd_stage1;
  size_t dm_topk_ids, dm_topk_scores, dm_admit_ids, dm_admit_slots, dm_evict_ids, dm_n_admit;
  size_t scan_scores;
  size_t total;
};

// The device address of page-locked host memory (cudaHostAlloc'd or
// registered), or null.  Pageable memory is refused even where the device
// could reach it through the system's address translation: the gathers need
// memory that stays resident.
void* mapped_host(const void* p) {
  cudaPointerAttributes at{};
  void* d = nullptr;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess || at.type != cudaMemoryTypeHost ||
      cudaHostGetDevicePointer(&d, const_cast<void*>(p), 0) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return d;
}

int fetch_cap(const oasis_config& c) {
  return static_cast<int>(std::floor(static_cast<double>(c.fetch_ratio) * c.topk + 1e-9));
}

// Draft queries per step (0 in the config means one).
int num_drafts(const oasis_config& c) { return c.num_drafts > 0 ? c.num_drafts : 1; }

WsLayout ws_layout(const oasis_config& c) {
  WsLayout w{};
  const size_t pairs = static_cast<size_t>(c.num_requests) * c.num_kv_heads;
  const size_t C = static_cast<size_t>(fetch_cap(c));
  const size_t qbytes = static_cast<size_t>(c.num_requests) * c.num_q_heads * c.head_dim * 2;
  const size_t obytes = qbytes * (c.out_fp32 ? 2 : 1);
  const size_t D = static_cast<size_t>(num_drafts(c));
  w.err = 0;
  size_t o = kAlign;
  // each list twice (step parity 0 and 1), the copies adjacent
  w.topk_ids = o;    o += 2 * align_up(pairs * c.topk * 4);
  w.topk_scores = o; o += 2 * align_up(pairs * c.topk * 4);
  w.admit_ids = o;   o += 2 * align_up(pairs * (C ? C : 1) * 4);
  w.admit_slots = o; o += 2 * align_up(pairs * (C ? C : 1) * 4);
  w.evict_ids = o;   o += 2 * align_up(pairs * (C ? C : 1) * 4);
  w.n_admit = o;     o += 2 * align_up(pairs * 4);
  w.q_stage = o;     o += align_up(qbytes);
  w.qd_stage = o;    o += align_up(D * qbytes);
  w.q_stage1 = o;    o += align_up(qbytes);
  w.qd_stage1 = o;   o += align_up(D * qbytes);
  w.out_stage = o;   o += align_up(obytes);
  w.outd_stage = o;  o += align_up(D * obytes);
  w.out_stage1 = o;  o += align_up(obytes);
  w.outd_stage1 = o; o += align_up(D * obytes);
  w.qd_ring0 = o;    o += align_up(D * qbytes);
  w.qd_ring1 = o;    o += align_up(D * qbytes);
  // miss-stall demand lists, [R][Hkv][K] each, both step parities
  w.dm_topk_ids = o;    o += 2 * align_up(pairs * c.topk * 4);
  w.dm_topk_scores = o; o += 2 * align_up(pairs * c.topk * 4);
  w.dm_admit_ids = o;   o += 2 * align_up(pairs * c.topk * 4);
  w.dm_admit_slots = o; o += 2 * align_up(pairs * c.topk * 4);
  w.dm_evict_ids = o;   o += 2 * align_up(pairs * c.topk * 4);
  w.dm_n_admit = o;     o += 2 * align_up(pairs * 4);
  // block scores of the split scan, both step parities
  w.scan_scores = o;    o += 2 * align_up(pairs * static_cast<size_t>(c.max_blocks) * 4);
  w.per_layer = o - kAlign;
  w.total = kAlign + w.per_layer * static_cast<size_t>(c.num_layers);
  return w;
}

const char* config_error(const oasis_config* c) {
  if (!c) return "config is NULL";
  if (c->num_layers <= 0) return "num_layers must be > 0";
  if (c->num_requests <= 0) return "num_requests must be > 0";
  if (c->max_blocks <= 0) return "max_blocks must be > 0";
  if (c->num_kv_heads <= 0 || c->num_q_heads <= 0) return "head counts must be > 0";
  if (c->num_q_heads % c->num_kv_heads != 0) return "num_q_heads must be a multiple of num_kv_heads";
  if (c->num_q_heads / c->num_kv_heads > kMaxGroup) return "query heads per KV head must be <= 4";
  if (c->head_dim != kHeadDim) return "head_dim must be 128";
  if (c->block_size != kBlock) return "block_size must be 16";
  if (c->topk <= 0 || c->topk > kMaxTopK) return "topk must be in 1..256";
  if (c->topk > c->max_blocks) return "topk must be <= max_blocks";
  if (!(c->fetch_ratio >= 0.f && c->fetch_ratio <= 1.f)) return "fetch_ratio must be in [0, 1]";
  if (!(c->softmax_scale >= 0.f) || std::isinf(c->softmax_scale)) return "softmax_scale must be finite and >= 0";
  if (c->device < 0) return "device must be >= 0";
  if (c->max_blocks > kMaxBlocksPerHead) return "max_blocks must be <= 131072";
  if (c->side_groups < 0 || c->side_groups > 64) return "side_groups must be in 0..64";
  if (c->num_drafts < 0 || c->num_drafts > kMaxDrafts) return "num_drafts must be in 0..3";
  if (c->schedule != OASIS_SCHEDULE_SCAN_FIRST && c->schedule != OASIS_SCHEDULE_CONCURRENT &&
      c->schedule != OASIS_SCHEDULE_THREE_STREAMS && c->schedule != OASIS_SCHEDULE_AUTO &&
      c->schedule != OASIS_SCHEDULE_EARLY_SCAN)
    return "schedule must be one of OASIS_SCHEDULE_*";
  const double units = static_cast<double>(c->num_requests) * c->num_kv_heads *
                       (c->topk + fetch_cap(*c)) * 2 * kBlock;
  if (units >= 2147483647.0) return "pool too large for a 32-bit TMA row coordinate";
  if (static_cast<double>(c->num_requests) * c->num_kv_heads * c->max_blocks >= 2147483647.0)
    return "num_requests * num_kv_heads * max_blocks must fit in int32";
  return nullptr;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

struct oasis_ctx {
  oasis_config cfg{};
  int G = 0, C = 0, U = 0;
  int D = 1;  // draft queries per step
  int groups = 1;  // request groups the side work is pipelined in
  float scale_log2 = 0.f;
  long long wait_limit = kWaitLimitCycles;  // oasis_set_wait_limit
  std::vector<LayerState> layers;
  int32_t* ctx_len = nullptr;
  uint8_t* ws = nullptr;
  uint32_t* err = nullptr;
  WsLayout wl{};
  cudaStream_t side = nullptr;   // scan + top-K + admission
  cudaStream_t side2 = nullptr;  // host -> HBM gathers
  cudaStream_t side3 = nullptr;  // admissions (three-stream) or scans (early scan)
  cudaEvent_t ev_ctx_mut = nullptr;  // the library's last write of ctx_len
  bool ctx_mut_pending = false;
  cudaStream_t io = nullptr;     // oasis_step_host input copies
  cudaStream_t io_out = nullptr; // oasis_step_host_async output copies
  std::string last_error;
  bool prof = false;
  std::vector<ProfPair> prof_pool;
  size_t prof_used = 0;
  std::vector<cudaEvent_t> prof_starts;
  size_t prof_starts_used = 0;

  int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    last_error = buf;
    return code;
  }
  int cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return OASIS_OK;
    return fail(OASIS_ECUDA, "%s: %s", what, cudaGetErrorString(e));
  }
  int32_t* res_tab(int l, int step) const {
    const size_t n = static_cast<size_t>(cfg.num_requests) * cfg.num_kv_heads * cfg.topk;
    return layers[l].res + (step & 1) * n;
  }
  int32_t* phys_tab(int l, int step) const {
    const size_t n = static_cast<size_t>(cfg.num_requests) * cfg.num_kv_heads * U;
    return layers[l].phys + (step & 1) * n;
  }
  int32_t* ctx_tab(int step) const { return ctx_len + (step & 1) * cfg.num_requests; }
  int set_device() { return cuda(cudaSetDevice(cfg.device), "cudaSetDevice"); }

  // Profiling: a timing event at the start of each step, and an event pair
  // around each launch of `kind` (0 attention, 1 score_topk, 2 admit, 3 gather).
  void prof_step_start(cudaStream_t s) {
    if (!prof) return;
    if (prof_starts_used == prof_starts.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return;
      prof_starts.push_back(e);
    }
    cudaEventRecord(prof_starts[prof_starts_used++], s);
  }
  cudaEvent_t* prof_begin(int kind, cudaStream_t s) {
    if (!prof) return nullptr;
    if (prof_used == prof_pool.size()) {
      ProfPair p{};
      if (cudaEventCreate(&p.a) != cudaSuccess) return nullptr;
      if (cudaEventCreate(&p.b) != cudaSuccess) {
        cudaEventDestroy(p.a);
        return nullptr;
      }
      prof_pool.push_back(p);
    }
    ProfPair& p = prof_pool[prof_used++];
    p.kind = kind;
    p.start = static_cast<int>(prof_starts_used) - 1;
    cudaEventRecord(p.a, s);
    return &p.b;
  }
  void prof_end(cudaEvent_t* e, cudaStream_t s) {
    if (e) cudaEventRecord(*e, s);
  }
};

namespace {

// NVTX range for the host-side issue of one call (visible in a timeline
// profiler; without one attached the calls return at once).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

int check_layer(oasis_ctx* ctx, int layer) {
  if (!ctx) return OASIS_EINVAL;
  if (layer < 0 || layer >= ctx->cfg.num_layers)
    return ctx->fail(OASIS_EINVAL, "layer %d out of range [0, %d)", layer, ctx->cfg.num_layers);
  return OASIS_OK;
}

int run_attention(oasis_ctx* ctx, int layer, int step, const void* q, const void* qd,
                  void* out, void* outd, cudaStream_t s) {
  LayerState& L = ctx->layers[layer];
  AttnArgs a{};
  a.q = q;
  a.qd = qd;
  a.out = out;
  a.outd = outd;
  a.res = ctx->res_tab(layer, step);
  a.phys = ctx->phys_tab(layer, step);
  a.ctx_len = ctx->ctx_tab(step);
  a.err = ctx->err;
  a.R = ctx->cfg.num_requests;
  a.Hq = ctx->cfg.num_q_heads;
  a.Hkv = ctx->cfg.num_kv_heads;
  a.G = ctx->G;
  a.D = ctx->D;
  a.K = ctx->cfg.topk;
  a.U = ctx->U;
  a.NBmax = ctx->cfg.max_blocks;
  a.scale_log2 = ctx->scale_log2;
  a.out_fp32 = ctx->cfg.out_fp32;
  a.wait_limit = ctx->wait_limit;
  cudaEvent_t* pe = ctx->prof_begin(0, s);
  cudaError_t e = launch_attention(a, &L.pool_map, s);
  ctx->prof_end(pe, s);
  return ctx->cuda(e, "attention launch");
}

AdmitArgs admit_args(oasis_ctx* ctx, int layer, int step, const int32_t* topk, int32_t* aid,
                     int32_t* aslot, int32_t* evid, int32_t* nadm) {
  AdmitArgs a{};
  a.topk = topk;
  a.res_cur = ctx->res_tab(layer, step);
  a.res_nxt = ctx->res_tab(layer, step + 1);
  a.stamps = ctx->layers[layer].stamps;
  a.phys_cur = ctx->phys_tab(layer, step);
  a.phys_nxt = ctx->phys_tab(layer, step + 1);
  a.admit_ids = aid;
  a.admit_slots = aslot;
  a.evict_ids = evid;
  a.n_admit = nadm;
  a.R = ctx->cfg.num_requests;
  a.Hkv = ctx->cfg.num_kv_heads;
  a.K = ctx->cfg.topk;
  a.C = ctx->C;
  a.U = ctx->U;
  a.NBmax = ctx->cfg.max_blocks;
  a.step = step;
  a.pair0 = 0;
  a.pairs = a.R * a.Hkv;
  return a;
}

// The miss-stall demand admission: the same rule, uncapped (C = K), in place
// in table (step & 1).
AdmitArgs demand_admit_args(oasis_ctx* ctx, int layer, int step, const int32_t* topk,
                            int32_t* aid, int32_t* aslot, int32_t* evid, int32_t* nadm) {
  AdmitArgs a = admit_args(ctx, layer, step, topk, aid, aslot, evid, nadm);
  a.res_nxt = ctx->res_tab(layer, step);
  a.phys_nxt = ctx->phys_tab(layer, step);
  a.C = ctx->cfg.topk;
  a.in_place = 1;
  return a;
}

// Scan arguments of all pairs: `x` holds `planes` planes of [R][Hq][d]
// query vectors (the D draft queries, or the one normal query).
ScoreArgs score_args(oasis_ctx* ctx, int layer, int step, const void* x, int planes,
                     int32_t* ids, float* scores) {
  ScoreArgs a{};
  a.qd = x;
  a.summ = ctx->layers[layer].summ;
  a.ctx_len = ctx->ctx_tab(step);
  a.topk_ids = ids;
  a.topk_scores = scores;
  a.err = ctx->err;
  a.R = ctx->cfg.num_requests;
  a.Hq = ctx->cfg.num_q_heads;
  a.Hkv = ctx->cfg.num_kv_heads;
  a.G = ctx->G;
  a.D = planes;
  a.K = ctx->cfg.topk;
  a.NBmax = ctx->cfg.max_blocks;
  a.pair0 = 0;
  a.pairs = a.R * a.Hkv;
  a.scores_ws = ctx->layers[layer].scan_scores[step & 1];
  a.wait_limit = ctx->wait_limit;
  return a;
}

// Launch a scan + ranking: split (scan, then ranking and fused admission,
// timed as profile kinds scan_kind and 6) or as one kernel (longer contexts,
// or OASIS_SCAN=fused; timed as scan_kind).  `scanned`, when given, is recorded on `s` once the
// scan is done: work that needs only that (it reads HBM beside the scan)
// may start while the ranking runs.
int launch_scan_timed(oasis_ctx* ctx, const ScoreArgs& a, cudaStream_t s, int scan_kind,
                      cudaEvent_t scanned) {
  if (scan_is_split(a.NBmax)) {
    cudaEvent_t* pe = ctx->prof_begin(scan_kind, s);
    cudaError_t e = launch_scan_scores(a, s);
    ctx->prof_end(pe, s);
    if (int rc = ctx->cuda(e, "scan launch")) return rc;
    if (scanned) {
      if (int rc = ctx->cuda(cudaEventRecord(scanned, s), "record scan")) return rc;
    }
    pe = ctx->prof_begin(6, s);
    e = launch_topk_select(a, s);
    ctx->prof_end(pe, s);
    return ctx->cuda(e, "top-k launch");
  }
  cudaEvent_t* pe = ctx->prof_begin(scan_kind, s);
  cudaError_t e = launch_score_topk(a, s);
  ctx->prof_end(pe, s);
  if (int rc = ctx->cuda(e, "score_topk launch")) return rc;
  if (scanned) return ctx->cuda(cudaEventRecord(scanned, s), "record scan");
  return OASIS_OK;
}

// Miss stall: scan + top-K of every pair with the step's normal query; with
// `fused` also the uncapped in-place admission into the layer's demand
// lists of this step's parity.
int run_demand_score(oasis_ctx* ctx, int layer, int step, const void* q, int32_t* ids,
                     float* scores, cudaStream_t s, bool fused) {
  LayerState& L = ctx->layers[layer];
  ScoreArgs a = score_args(ctx, layer, step, q, 1, ids, scores);
  a.fuse_admit = fused ? 1 : 0;
  if (fused) {
    const LayerState::Lists& Dm = L.dm[step & 1];
    a.admit = demand_admit_args(ctx, layer, step, nullptr, Dm.admit_ids, Dm.admit_slots,
                                Dm.evict_ids, Dm.n_admit);
  }
  return launch_scan_timed(ctx, a, s, 4, nullptr);
}

// Scan + top-K of pairs [pair0, pair0 + pairs); with `fused` also their
// capped eviction into the layer's workspace lists.
int run_score(oasis_ctx* ctx, int layer, int step, const void* qd, int32_t* ids,
              float* scores, cudaStream_t s, int pair0 = 0, int pairs = -1,
              bool fused = false, cudaEvent_t scanned = nullptr) {
  LayerState& L = ctx->layers[layer];
  ScoreArgs a = score_args(ctx, layer, step, qd, ctx->D, ids, scores);
  a.pair0 = pair0;
  if (pairs >= 0) a.pairs = pairs;
  a.fuse_admit = fused ? 1 : 0;
  if (fused)
    a.admit = admit_args(ctx, layer, step, nullptr, L.lists[step & 1].admit_ids,
                         L.lists[step & 1].admit_slots, L.lists[step & 1].evict_ids,
                         L.lists[step & 1].n_admit);
  return launch_scan_timed(ctx, a, s, 1, scanned);
}

int run_admit(oasis_ctx* ctx, int layer, int step, const int32_t* topk, int32_t* aid,
              int32_t* aslot, int32_t* evid, int32_t* nadm, cudaStream_t s, int pair0 = 0,
              int pairs = -1) {
  AdmitArgs a = admit_args(ctx, layer, step, topk, aid, aslot, evid, nadm);
  a.pair0 = pair0;
  if (pairs >= 0) a.pairs = pairs;
  cudaEvent_t* pe = ctx->prof_begin(2, s);
  cudaError_t e = launch_admit(a, s);
  ctx->prof_end(pe, s);
  return ctx->cuda(e, "admit_evict launch");
}

// Remote tier: assign local slots to the listed blocks not yet held (on
// `s`), then hand the transfer remote -> local to the tier's worker thread.
int run_remote_fetch(oasis_ctx* ctx, int layer, const int32_t* ids, const int32_t* n_valid,
                     int items, int pair0, int pairs, cudaStream_t s) {
  LayerState& L = ctx->layers[layer];
  RemoteTier& T = *L.remote;
  const int all = ctx->cfg.num_requests * ctx->cfg.num_kv_heads;
  RemoteArgs r{};
  r.ids = ids;
  r.n_valid = n_valid;
  r.local_map = T.map;
  r.count = T.count;
  r.base = T.base;
  r.n_miss = T.lists_dev;
  r.miss_ids = T.lists_dev + all;
  r.miss_slots = T.lists_dev + all + static_cast<size_t>(all) * T.M;
  r.err = ctx->err;
  r.pair0 = pair0;
  r.pairs = pairs;
  r.items = items;
  r.NBmax = ctx->cfg.max_blocks;
  r.capacity = T.capacity;
  r.M = T.M;
  if (int rc = ctx->cuda(launch_remote_assign(r, s), "remote slot assignment launch")) return rc;
  // The stream publishes the transfer number once the assignment is done
  // (with a memory barrier, so the lists are visible); the worker copies.
  const uint32_t seq = ++T.next_seq;
  auto write = get_write_value32();
  if (!write) return ctx->fail(OASIS_ECUDA, "cuStreamWriteValue32 unavailable");
  if (write(s, T.assigned_dev, seq, 0) != CUDA_SUCCESS)
    return ctx->fail(OASIS_ECUDA, "remote: stream write of the assignment number failed");
  RemoteJob j;
  j.seq = seq;
  j.pair0 = pair0;
  j.pairs = pairs;
  T.post(j);
  return OASIS_OK;
}

// Make `s` wait until the tier's worker has finished the latest transfer.
int wait_remote(oasis_ctx* ctx, const RemoteTier& T, cudaStream_t s) {
  auto wait = get_wait_value32();
  if (!wait) return ctx->fail(OASIS_ECUDA, "cuStreamWaitValue32 unavailable");
  if (wait(s, T.moved_dev, T.next_seq, CU_STREAM_WAIT_VALUE_GEQ) != CUDA_SUCCESS)
    return ctx->fail(OASIS_ECUDA, "remote: stream wait for the transfer failed");
  return OASIS_OK;
}

// With a remote tier the gather runs in two launches: the units already held
// in the local tier (slot < base) at once, beside the network transfer, and
// the units this assignment fetched (slot >= base) after it.
int launch_gather_split(oasis_ctx* ctx, const LayerState& L, GatherArgs g, cudaStream_t s) {
  if (!L.remote) {
    g.phase = 0;
    return ctx->cuda(launch_gather(g, s), "gather launch");
  }
  g.phase = 1;
  if (int rc = ctx->cuda(launch_gather(g, s), "gather launch (held units)")) return rc;
  if (int rc = wait_remote(ctx, *L.remote, s)) return rc;
  g.phase = 2;
  return ctx->cuda(launch_gather(g, s), "gather launch (fetched units)");
}

void gather_source(const oasis_ctx* ctx, const LayerState& L, GatherArgs& g) {
  if (L.remote) {
    g.host = L.remote->local_dev;
    g.local_map = L.remote->map;
    g.base = L.remote->base;
    g.src_units = L.remote->capacity;
  } else {
    g.host = L.host_dev;
    g.local_map = nullptr;
    g.src_units = ctx->cfg.max_blocks;
  }
}

int run_prefetch(oasis_ctx* ctx, int layer, int step, const int32_t* aid,
                 const int32_t* aslot, const int32_t* nadm, cudaStream_t s, int pair0 = 0,
                 int pairs = -1) {
  if (ctx->C == 0) return OASIS_OK;
  LayerState& L = ctx->layers[layer];
  if (pairs < 0) pairs = ctx->cfg.num_requests * ctx->cfg.num_kv_heads;
  if (L.remote) {
    if (int rc = run_remote_fetch(ctx, layer, aid, nadm, ctx->C, pair0, pairs, s)) return rc;
  }
  GatherArgs g{};
  gather_source(ctx, L, g);
  g.pool = L.pool;
  g.src_ids = aid;
  g.dst_slots = aslot;
  g.n_valid = nadm;
  g.phys = ctx->phys_tab(layer, step + 1);
  g.err = ctx->err;
  g.pair0 = pair0;
  g.pairs = pairs;
  g.items = ctx->C;
  g.NBmax = ctx->cfg.max_blocks;
  g.U = ctx->U;
  // A one-layer context's gathers must land within one step (the next
  // attention of the layer follows at once), so they get a few more units
  // in flight; with several layers they have the other layers' time, and
  // fewer in flight slow the HBM kernels beside them less, the fewer the
  // more a step's admissions leave the link idle.  Measured on GB300: 128 x
  // 16K layer (6144 units a step) 44 CTAs 3342 / end to end 3286-3289
  // layer-steps/s against 40: 3337-3338 / 3260-3261; 32-layer 64 x 32K loop
  // (3072 units a layer-step) 20 / 24 / 40 / 44 CTAs: 3837-3932 / 4105-4149
  // / 3981-4006 / 3716; 36-layer 90 x 16K loop (4320 units) 32 / 40 / 48:
  // 3548 / 3736 / 3636.
  const long long units = static_cast<long long>(pairs) * ctx->C;
  g.max_ctas = ctx->cfg.num_layers == 1 ? 44 : units <= 3072 ? 24 : 0;
  cudaEvent_t* pe = ctx->prof_begin(3, s);
  const int rc = launch_gather_split(ctx, L, g, s);
  ctx->prof_end(pe, s);
  return rc;
}

// Miss stall: copy the demand-admitted units into their slots' own pool
// units of table (step & 1), one warp per pair.
int run_demand_gather(oasis_ctx* ctx, int layer, int step, const int32_t* aid,
                      const int32_t* aslot, const int32_t* nadm, cudaStream_t s) {
  LayerState& L = ctx->layers[layer];
  GatherArgs g{};
  gather_source(ctx, L, g);
  g.pool = L.pool;
  g.src_ids = aid;
  g.dst_slots = aslot;
  g.n_valid = nadm;
  g.phys = ctx->phys_tab(layer, step);
  g.err = ctx->err;
  g.pair0 = 0;
  g.pairs = ctx->cfg.num_requests * ctx->cfg.num_kv_heads;
  g.items = ctx->cfg.topk;
  g.NBmax = ctx->cfg.max_blocks;
  g.U = ctx->U;
  g.pair_major = 1;
  cudaEvent_t* pe = ctx->prof_begin(5, s);
  cudaError_t e = launch_gather(g, s);
  ctx->prof_end(pe, s);
  return ctx->cuda(e, "demand gather launch");
}

}  // namespace

extern "C" {

OASIS_API const char* oasis_config_error(const oasis_config* cfg) { return config_error(cfg); }

OASIS_API int oasis_query_sizes(const oasis_config* cfg, oasis_sizes* out) {
  if (!out || config_error(cfg)) return OASIS_EINVAL;
  const size_t R = cfg->num_requests, H = cfg->num_kv_heads, K = cfg->topk;
  const size_t NB = cfg->max_blocks;
  const int C = fetch_cap(*cfg);
  const size_t U = K + C;
  out->kv_pool_bytes = R * H * U * kUnitBytes;
  out->summaries_bytes = R * H * NB * kSummBytes;
  out->host_kv_bytes = R * H * NB * kUnitBytes;
  out->res_ids_bytes = 2 * R * H * K * 4;
  out->stamps_bytes = R * H * K * 4;
  out->phys_bytes = 2 * R * H * U * 4;
  out->ctx_len_bytes = 2 * R * 4;
  out->workspace_bytes = ws_layout(*cfg).total;
  out->fetch_cap = C;
  out->units_per_head = static_cast<int32_t>(U);
  return OASIS_OK;
}

OASIS_API int oasis_init(const oasis_config* cfg, const oasis_buffers* bufs,
                         oasis_ctx** out) {
  if (!out) return OASIS_EINVAL;
  *out = nullptr;
  if (config_error(cfg) || !bufs) return OASIS_EINVAL;
  const int L = cfg->num_layers;
  if (!bufs->kv_pool || !bufs->summaries || !bufs->host_kv || !bufs->res_ids ||
      !bufs->stamps || !bufs->phys || !bufs->ctx_len || !bufs->workspace)
    return OASIS_EINVAL;
  if ((reinterpret_cast<uintptr_t>(bufs->workspace) & (kAlign - 1)) != 0) return OASIS_EINVAL;
  for (int l = 0; l < L; ++l) {
    if (!bufs->kv_pool[l] || !bufs->summaries[l] || !bufs->host_kv[l] || !bufs->res_ids[l] ||
        !bufs->stamps[l] || !bufs->phys[l])
      return OASIS_EINVAL;
    if (!aligned16(bufs->kv_pool[l]) || !aligned16(bufs->summaries[l]) ||
        !aligned16(bufs->host_kv[l]) || !aligned16(bufs->res_ids[l]) ||
        !aligned16(bufs->stamps[l]) || !aligned16(bufs->phys[l]))
      return OASIS_EINVAL;
  }

  oasis_ctx* c = new (std::nothrow) oasis_ctx();
  if (!c) return OASIS_ENOMEM;
  c->cfg = *cfg;
  c->G = cfg->num_q_heads / cfg->num_kv_heads;
  c->D = num_drafts(*cfg);
  c->C = fetch_cap(*cfg);
  c->U = cfg->topk + c->C;
  const double scale = cfg->softmax_scale > 0.f ? cfg->softmax_scale : 1.0 / std::sqrt(128.0);
  c->scale_log2 = static_cast<float>(scale * 1.4426950408889634);
  c->ctx_len = bufs->ctx_len;
  c->ws = static_cast<uint8_t*>(bufs->workspace);
  c->wl = ws_layout(*cfg);
  c->err = reinterpret_cast<uint32_t*>(c->ws + c->wl.err);
  c->layers.resize(L);

  auto bail = [&](int code) {
    oasis_destroy(c);
    return code;
  };
  if (cudaSetDevice(cfg->device) != cudaSuccess) return bail(OASIS_ECUDA);
  int lo = 0, hi = 0;
  if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess) return bail(OASIS_ECUDA);
  if (cudaStreamCreateWithPriority(&c->side, cudaStreamNonBlocking, hi) != cudaSuccess ||
      cudaStreamCreateWithPriority(&c->side2, cudaStreamNonBlocking, hi) != cudaSuccess ||
      cudaStreamCreateWithPriority(&c->side3, cudaStreamNonBlocking, hi) != cudaSuccess ||
      cudaStreamCreateWithPriority(&c->io, cudaStreamNonBlocking, hi) != cudaSuccess ||
      cudaStreamCreateWithPriority(&c->io_out, cudaStreamNonBlocking, hi) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev_ctx_mut, cudaEventDisableTiming) != cudaSuccess)
    return bail(OASIS_ENOMEM);
  {
    const int pairs = cfg->num_requests * cfg->num_kv_heads;
    // Default: one group.  Measured on GB300 (128 x 16K layer): smaller
    // groups start the gathers earlier but each launch covers too few SMs and
    // the scan slows by more than the link gains.
    c->groups = cfg->side_groups > 0 ? cfg->side_groups : 1;
    if (c->groups > pairs) c->groups = pairs;
    if (c->groups < 1) c->groups = 1;
  }
  auto encode = get_encode();
  if (!encode) return bail(OASIS_ECUDA);
  // Load all kernels up front: a kernel's first launch otherwise loads its
  // module lazily, and that load waits for the work already queued on the
  // device (measured: a first oasis_step issued while a throttled remote
  // transfer was pending blocked the calling thread for the transfer's
  // 130 ms).
  if (preload_attention_kernels() != cudaSuccess || preload_score_kernels() != cudaSuccess ||
      preload_support_kernels() != cudaSuccess)
    return bail(OASIS_ECUDA);

  const size_t R = cfg->num_requests, H = cfg->num_kv_heads;
  for (int l = 0; l < L; ++l) {
    LayerState& S = c->layers[l];
    S.pool = bufs->kv_pool[l];
    S.summ = bufs->summaries[l];
    S.host = bufs->host_kv[l];
    S.res = bufs->res_ids[l];
    S.stamps = bufs->stamps[l];
    S.phys = bufs->phys[l];
    void* dptr = mapped_host(S.host);
    if (!dptr) {
      c->last_error = "host_kv is not page-locked host memory mapped for the device";
      return bail(OASIS_EINVAL);
    }
    S.host_dev = dptr;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim),
                                static_cast<cuuint64_t>(R * H * c->U * 2 * kBlock)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim * 2)};
    const cuuint32_t box[2] = {64, 2 * kBlock};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&S.pool_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, S.pool, dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return bail(OASIS_ECUDA);
    // WsLayout offsets place layer 0's lists right after the error word.
    uint8_t* w = c->ws + kAlign + static_cast<size_t>(l) * c->wl.per_layer;
    const size_t b0 = kAlign;
    {
      const size_t pairs = R * H;
      const size_t tk = align_up(pairs * cfg->topk * 4);
      const size_t ad = align_up(pairs * (c->C ? c->C : 1) * 4);
      const size_t na = align_up(pairs * 4);
      for (int p = 0; p < 2; ++p) {
        auto& Lp = S.lists[p];
        Lp.topk_ids = reinterpret_cast<int32_t*>(w + (c->wl.topk_ids - b0) + p * tk);
        Lp.topk_scores = reinterpret_cast<float*>(w + (c->wl.topk_scores - b0) + p * tk);
        Lp.admit_ids = reinterpret_cast<int32_t*>(w + (c->wl.admit_ids - b0) + p * ad);
        Lp.admit_slots = reinterpret_cast<int32_t*>(w + (c->wl.admit_slots - b0) + p * ad);
        Lp.evict_ids = reinterpret_cast<int32_t*>(w + (c->wl.evict_ids - b0) + p * ad);
        Lp.n_admit = reinterpret_cast<int32_t*>(w + (c->wl.n_admit - b0) + p * na);
        auto& Dp = S.dm[p];
        Dp.topk_ids = reinterpret_cast<int32_t*>(w + (c->wl.dm_topk_ids - b0) + p * tk);
        Dp.topk_scores = reinterpret_cast<float*>(w + (c->wl.dm_topk_scores - b0) + p * tk);
        Dp.admit_ids = reinterpret_cast<int32_t*>(w + (c->wl.dm_admit_ids - b0) + p * tk);
        Dp.admit_slots = reinterpret_cast<int32_t*>(w + (c->wl.dm_admit_slots - b0) + p * tk);
        Dp.evict_ids = reinterpret_cast<int32_t*>(w + (c->wl.dm_evict_ids - b0) + p * tk);
        Dp.n_admit = reinterpret_cast<int32_t*>(w + (c->wl.dm_n_admit - b0) + p * na);
        const size_t sb = align_up(pairs * static_cast<size_t>(cfg->max_blocks) * 4);
        S.scan_scores[p] = reinterpret_cast<float*>(w + (c->wl.scan_scores - b0) + p * sb);
      }
    }
    S.q_stage[0] = w + (c->wl.q_stage - b0);
    S.qd_stage[0] = w + (c->wl.qd_stage - b0);
    S.q_stage[1] = w + (c->wl.q_stage1 - b0);
    S.qd_stage[1] = w + (c->wl.qd_stage1 - b0);
    for (int k = 0; k < 2; ++k)
      if (cudaEventCreateWithFlags(&S.ev_in[k], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&S.ev_stage_free[k], cudaEventDisableTiming) != cudaSuccess)
        return bail(OASIS_ENOMEM);
    S.qd_ring[0] = w + (c->wl.qd_ring0 - b0);
    S.qd_ring[1] = w + (c->wl.qd_ring1 - b0);
    S.out_stage[0] = w + (c->wl.out_stage - b0);
    S.outd_stage[0] = w + (c->wl.outd_stage - b0);
    S.out_stage[1] = w + (c->wl.out_stage1 - b0);
    S.outd_stage[1] = w + (c->wl.outd_stage1 - b0);
    if (cudaEventCreateWithFlags(&S.ev_start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&S.ev_demand_done, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&S.ev_side_done, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&S.ev_scan_done, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&S.ev_qd_copied, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&S.ev_admitted[0], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&S.ev_admitted[1], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&S.ev_mut, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&S.ev_attn_done, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&S.ev_out_done[0], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&S.ev_out_done[1], cudaEventDisableTiming) != cudaSuccess)
      return bail(OASIS_ENOMEM);
    S.ev_group.assign(c->groups, nullptr);
    S.ev_group2.assign(c->groups, nullptr);
    for (auto& e : S.ev_group)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
        return bail(OASIS_ENOMEM);
    for (auto& e : S.ev_group2)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
        return bail(OASIS_ENOMEM);
  }
  if (cudaMemsetAsync(c->err, 0, sizeof(uint32_t), c->side) != cudaSuccess ||
      cudaStreamSynchronize(c->side) != cudaSuccess)
    return bail(OASIS_ECUDA);
  *out = c;
  return OASIS_OK;
}

OASIS_API int oasis_destroy(oasis_ctx* ctx) {
  if (!ctx) return OASIS_OK;
  cudaSetDevice(ctx->cfg.device);
  if (ctx->side) cudaStreamSynchronize(ctx->side);
  if (ctx->side2) cudaStreamSynchronize(ctx->side2);
  if (ctx->side3) cudaStreamSynchronize(ctx->side3);
  if (ctx->io) cudaStreamSynchronize(ctx->io);
  if (ctx->io_out) cudaStreamSynchronize(ctx->io_out);
  // A remote tier's transfers may sit on a caller's stream.
  for (auto& L : ctx->layers)
    if (L.remote) {
      cudaDeviceSynchronize();
      break;
    }
  for (auto& L : ctx->layers) {
    for (auto& e : L.ev_group)
      if (e) cudaEventDestroy(e);
    for (auto& e : L.ev_group2)
      if (e) cudaEventDestroy(e);
    if (L.ev_start) cudaEventDestroy(L.ev_start);
    if (L.ev_demand_done) cudaEventDestroy(L.ev_demand_done);
    if (L.ev_side_done) cudaEventDestroy(L.ev_side_done);
    if (L.ev_scan_done) cudaEventDestroy(L.ev_scan_done);
    if (L.ev_qd_copied) cudaEventDestroy(L.ev_qd_copied);
    if (L.ev_mut) cudaEventDestroy(L.ev_mut);
    if (L.ev_attn_done) cudaEventDestroy(L.ev_attn_done);
    for (int k = 0; k < 2; ++k) {
      if (L.ev_out_done[k]) cudaEventDestroy(L.ev_out_done[k]);
      if (L.ev_admitted[k]) cudaEventDestroy(L.ev_admitted[k]);
      if (L.ev_in[k]) cudaEventDestroy(L.ev_in[k]);
      if (L.ev_stage_free[k]) cudaEventDestroy(L.ev_stage_free[k]);
    }
  }
  for (auto& p : ctx->prof_pool) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  for (auto& e : ctx->prof_starts) cudaEventDestroy(e);
  if (ctx->side) cudaStreamDestroy(ctx->side);
  if (ctx->side2) cudaStreamDestroy(ctx->side2);
  if (ctx->side3) cudaStreamDestroy(ctx->side3);
  if (ctx->ev_ctx_mut) cudaEventDestroy(ctx->ev_ctx_mut);
  if (ctx->io) cudaStreamDestroy(ctx->io);
  if (ctx->io_out) cudaStreamDestroy(ctx->io_out);
  ctx->layers.clear();  // remote tiers: worker and copy threads joined
  delete ctx;
  return OASIS_OK;
}

OASIS_API const char* oasis_last_error(const oasis_ctx* ctx) {
  if (!ctx) return "null context";
  return ctx->last_error.c_str();
}

OASIS_API int oasis_sync(oasis_ctx* ctx, uint32_t* device_bits) {
  if (!ctx) return OASIS_EINVAL;
  if (int rc = ctx->set_device()) return rc;
  if (int rc = ctx->cuda(cudaDeviceSynchronize(), "cudaDeviceSynchronize")) return rc;
  uint32_t bits = 0;
  if (int rc = ctx->cuda(cudaMemcpy(&bits, ctx->err, sizeof bits, cudaMemcpyDeviceToHost),
                         "read device error word"))
    return rc;
  if (device_bits) *device_bits = bits;
  if (bits) {
    if (int rc = ctx->cuda(cudaMemset(ctx->err, 0, sizeof bits), "clear device error word"))
      return rc;
    return ctx->fail(OASIS_EDEVICE, "device error bits 0x%x", bits);
  }
  return OASIS_OK;
}

namespace {
// A library call wrote this layer's summaries on `s`: an early scan issued
// later waits for it (the other schedules follow the caller's stream).
int note_summary_write(oasis_ctx* ctx, LayerState& L, cudaStream_t s) {
  if (int rc = ctx->cuda(cudaEventRecord(L.ev_mut, s), "record summary write")) return rc;
  L.mut_pending = true;
  return OASIS_OK;
}
}  // namespace

OASIS_API int oasis_build_summaries(oasis_ctx* ctx, int layer, int table, void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (int rc = ctx->set_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerState& L = ctx->layers[layer];
  // A scan of an earlier step may still read the summaries.
  if (L.side_pending) {
    if (int rc = ctx->cuda(cudaStreamWaitEvent(s, L.ev_side_done, 0), "wait side")) return rc;
  }
  SummaryArgs a{};
  a.host = L.host_dev;
  a.summ = L.summ;
  a.ctx_len = ctx->ctx_tab(table);
  a.R = ctx->cfg.num_requests;
  a.Hkv = ctx->cfg.num_kv_heads;
  a.NBmax = ctx->cfg.max_blocks;
  if (int rc = ctx->cuda(launch_summary_build(a, s), "summary_build launch")) return rc;
  return note_summary_write(ctx, L, s);
}

namespace {
// Resident set res_ids[first_step & 1] into the pool, phys[first_step & 1]
// reset to the identity; stamps reset to -1 unless keep_stamps.
int load_resident(oasis_ctx* ctx, int layer, int first_step, bool keep_stamps, void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (first_step < 0) return ctx->fail(OASIS_EINVAL, "first_step must be >= 0");
  if (int rc = ctx->set_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerState& L = ctx->layers[layer];
  if (L.side_pending) {
    if (int rc = ctx->cuda(cudaStreamWaitEvent(s, L.ev_side_done, 0), "wait side")) return rc;
  }
  const int pairs = ctx->cfg.num_requests * ctx->cfg.num_kv_heads;
  if (int rc = ctx->cuda(launch_init_tables(ctx->phys_tab(layer, first_step),
                                            keep_stamps ? nullptr : L.stamps, pairs,
                                            ctx->cfg.topk, ctx->U, s),
                         "init tables launch"))
    return rc;
  if (L.remote) {
    if (int rc = run_remote_fetch(ctx, layer, ctx->res_tab(layer, first_step), nullptr,
                                  ctx->cfg.topk, 0, pairs, s))
      return rc;
  }
  GatherArgs g{};
  gather_source(ctx, L, g);
  g.pool = L.pool;
  g.src_ids = ctx->res_tab(layer, first_step);
  g.dst_slots = nullptr;
  g.n_valid = nullptr;
  g.phys = ctx->phys_tab(layer, first_step);
  g.err = ctx->err;
  g.pair0 = 0;
  g.pairs = pairs;
  g.items = ctx->cfg.topk;
  g.NBmax = ctx->cfg.max_blocks;
  g.U = ctx->U;
  if (int rc = launch_gather_split(ctx, L, g, s)) return rc;
  if (L.remote) {
    // The block each request's context ends in (decoding appends there
    // first) also travels to the local tier; the list borrows a workspace
    // buffer no step uses yet.
    int32_t* tail = L.lists[1].topk_ids;
    if (int rc = ctx->cuda(launch_tail_blocks(ctx->ctx_tab(first_step), ctx->cfg.num_requests,
                                              ctx->cfg.num_kv_heads, tail, s),
                           "tail blocks launch"))
      return rc;
    if (int rc = run_remote_fetch(ctx, layer, tail, nullptr, 1, 0, pairs, s)) return rc;
    if (int rc = wait_remote(ctx, *L.remote, s)) return rc;
  }
  L.loaded = true;
  L.side_pending = false;
  return OASIS_OK;
}

}  // namespace

OASIS_API int oasis_load_resident(oasis_ctx* ctx, int layer, int first_step, void* stream) {
  return load_resident(ctx, layer, first_step, false, stream);
}

OASIS_API int oasis_resume_resident(oasis_ctx* ctx, int layer, int first_step, void* stream) {
  return load_resident(ctx, layer, first_step, true, stream);
}

OASIS_API int oasis_lookahead_attn(oasis_ctx* ctx, int layer, int step, const void* q,
                                   const void* q_draft, void* out, void* out_draft,
                                   void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || !q || !q_draft || !out || !out_draft)
    return ctx->fail(OASIS_EINVAL, "attention: bad step or null pointer");
  if (int rc = ctx->set_device()) return rc;
  return run_attention(ctx, layer, step, q, q_draft, out, out_draft,
                       static_cast<cudaStream_t>(stream));
}

OASIS_API int oasis_dense_attn(oasis_ctx* ctx, const void* kv_dense, int table, const void* q,
                               const void* q_draft, void* out, void* out_draft,
                               void* stream) {
  if (!ctx) return OASIS_EINVAL;
  if (table < 0 || !kv_dense || !q || !q_draft || !out || !out_draft)
    return ctx->fail(OASIS_EINVAL, "dense_attn: bad table or null pointer");
  if (!aligned16(kv_dense)) return ctx->fail(OASIS_EINVAL, "dense_attn: kv_dense not 16-byte aligned");
  const double rows = static_cast<double>(ctx->cfg.num_requests) * ctx->cfg.num_kv_heads *
                      ctx->cfg.max_blocks * 2 * kBlock;
  if (rows >= 2147483647.0)
    return ctx->fail(OASIS_EINVAL, "dense_attn: cache too large for a 32-bit TMA row coordinate");
  if (int rc = ctx->set_device()) return rc;
  auto encode = get_encode();
  if (!encode) return ctx->fail(OASIS_ECUDA, "cuTensorMapEncodeTiled unavailable");
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim * 2)};
  const cuuint32_t box[2] = {64, 2 * kBlock};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_dense), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return ctx->fail(OASIS_ECUDA, "dense_attn: tensor map encode failed");
  AttnArgs a{};
  a.q = q;
  a.qd = q_draft;
  a.out = out;
  a.outd = out_draft;
  a.ctx_len = ctx->ctx_tab(table);
  a.err = ctx->err;
  a.R = ctx->cfg.num_requests;
  a.Hq = ctx->cfg.num_q_heads;
  a.Hkv = ctx->cfg.num_kv_heads;
  a.G = ctx->G;
  a.D = ctx->D;
  a.NBmax = ctx->cfg.max_blocks;
  a.scale_log2 = ctx->scale_log2;
  a.out_fp32 = ctx->cfg.out_fp32;
  a.dense = 1;
  a.wait_limit = ctx->wait_limit;
  return ctx->cuda(launch_attention(a, &map, static_cast<cudaStream_t>(stream)),
                   "dense attention launch");
}

OASIS_API int oasis_score_topk(oasis_ctx* ctx, int layer, int step, const void* q_draft,
                               int32_t* topk_ids, float* topk_scores, void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || !q_draft || !topk_ids)
    return ctx->fail(OASIS_EINVAL, "score_topk: bad step or null pointer");
  if (int rc = ctx->set_device()) return rc;
  return run_score(ctx, layer, step, q_draft, topk_ids, topk_scores,
                   static_cast<cudaStream_t>(stream));
}

OASIS_API int oasis_admit_evict(oasis_ctx* ctx, int layer, int step, const int32_t* topk_ids,
                                int32_t* admit_ids, int32_t* admit_slots, int32_t* evict_ids,
                                int32_t* n_admit, void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || step > (1 << 30) || !topk_ids || !admit_ids || !admit_slots || !evict_ids ||
      !n_admit)
    return ctx->fail(OASIS_EINVAL, "admit_evict: bad step or null pointer");
  if (int rc = ctx->set_device()) return rc;
  return run_admit(ctx, layer, step, topk_ids, admit_ids, admit_slots, evict_ids, n_admit,
                   static_cast<cudaStream_t>(stream));
}

OASIS_API int oasis_score_admit_noalloc(oasis_ctx* ctx, int layer, int step,
                                        const void* q_draft, int32_t* admit_ids,
                                        int32_t* admit_slots, int32_t* evict_ids,
                                        int32_t* n_admit, void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || step > (1 << 30) || !q_draft || !admit_ids || !admit_slots || !evict_ids ||
      !n_admit)
    return ctx->fail(OASIS_EINVAL, "score_admit_noalloc: bad step or null pointer");
  const size_t need = static_cast<size_t>(ctx->cfg.num_requests) * ctx->cfg.num_kv_heads *
                      ctx->cfg.topk;
  if (need > kNoAllocTopkEntries)
    return ctx->fail(OASIS_EINVAL,
                     "score_admit_noalloc: the top-K lists need %zu entries, the fixed "
                     "scratch holds %zu (1 MiB); use oasis_score_topk + oasis_admit_evict",
                     need, kNoAllocTopkEntries);
  if (int rc = ctx->set_device()) return rc;
  int32_t* topk = nullptr;
  if (int rc = ctx->cuda(noalloc_topk_scratch(ctx->cfg.device, &topk), "scratch address"))
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = run_score(ctx, layer, step, q_draft, topk, nullptr, s)) return rc;
  return run_admit(ctx, layer, step, topk, admit_ids, admit_slots, evict_ids, n_admit, s);
}

OASIS_API int oasis_prefetch(oasis_ctx* ctx, int layer, int step, const int32_t* admit_ids,
                             const int32_t* admit_slots, const int32_t* n_admit,
                             void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || !admit_ids || !admit_slots || !n_admit)
    return ctx->fail(OASIS_EINVAL, "prefetch: bad step or null pointer");
  if (int rc = ctx->set_device()) return rc;
  return run_prefetch(ctx, layer, step, admit_ids, admit_slots, n_admit,
                      static_cast<cudaStream_t>(stream));
}

OASIS_API int oasis_demand_topk(oasis_ctx* ctx, int layer, int step, const void* q,
                                int32_t* topk_ids, float* topk_scores, void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || !q || !topk_ids)
    return ctx->fail(OASIS_EINVAL, "demand_topk: bad step or null pointer");
  if (int rc = ctx->set_device()) return rc;
  return run_demand_score(ctx, layer, step, q, topk_ids, topk_scores,
                          static_cast<cudaStream_t>(stream), false);
}

OASIS_API int oasis_admit_demand(oasis_ctx* ctx, int layer, int step, const int32_t* topk_ids,
                                 int32_t* admit_ids, int32_t* admit_slots, int32_t* evict_ids,
                                 int32_t* n_admit, void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || step > (1 << 30) || !topk_ids || !admit_ids || !admit_slots || !evict_ids ||
      !n_admit)
    return ctx->fail(OASIS_EINVAL, "admit_demand: bad step or null pointer");
  if (ctx->layers[layer].remote)
    return ctx->fail(OASIS_ESTATE, "admit_demand: the miss stall has no remote tier");
  if (int rc = ctx->set_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const AdmitArgs a = demand_admit_args(ctx, layer, step, topk_ids, admit_ids, admit_slots,
                                        evict_ids, n_admit);
  cudaEvent_t* pe = ctx->prof_begin(4, s);
  cudaError_t e = launch_admit(a, s);
  ctx->prof_end(pe, s);
  return ctx->cuda(e, "demand admission launch");
}

OASIS_API int oasis_fetch_demand(oasis_ctx* ctx, int layer, int step, const int32_t* admit_ids,
                                 const int32_t* admit_slots, const int32_t* n_admit,
                                 void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || !admit_ids || !admit_slots || !n_admit)
    return ctx->fail(OASIS_EINVAL, "fetch_demand: bad step or null pointer");
  if (ctx->layers[layer].remote)
    return ctx->fail(OASIS_ESTATE, "fetch_demand: the miss stall has no remote tier");
  if (int rc = ctx->set_device()) return rc;
  return run_demand_gather(ctx, layer, step, admit_ids, admit_slots, n_admit,
                           static_cast<cudaStream_t>(stream));
}

OASIS_API int oasis_step_stall(oasis_ctx* ctx, int layer, int step, const void* q,
                               const void* q_draft, void* out, void* out_draft, void* stream) {
  NvtxRange nvtx("oasis_step_stall");
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || step > (1 << 30) || !q || !q_draft || !out || !out_draft)
    return ctx->fail(OASIS_EINVAL, "step_stall: bad step or null pointer");
  LayerState& L = ctx->layers[layer];
  if (!L.loaded) return ctx->fail(OASIS_ESTATE, "layer %d: oasis_load_resident first", layer);
  if (L.remote) return ctx->fail(OASIS_ESTATE, "step_stall: the miss stall has no remote tier");
  if (int rc = ctx->set_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The look-ahead side work reads the draft queries from the layer's
  // staging buffer, so the caller may reuse its buffer once `stream` passes.
  void* qd_copy = L.qd_ring[step & 1];
  const size_t qbytes = static_cast<size_t>(ctx->D) * ctx->cfg.num_requests *
                        ctx->cfg.num_q_heads * kHeadDim * 2;
  if (int rc = ctx->cuda(cudaMemcpyAsync(qd_copy, q_draft, qbytes, cudaMemcpyDeviceToDevice, s),
                         "stage q_draft"))
    return rc;
  // The demand admission rewrites table (step & 1), which the layer's
  // previous look-ahead admission wrote, and the demand gather may overwrite
  // a unit that admission's gather filled: both wait for that side work.
  if (L.side_pending) {
    if (int rc = ctx->cuda(cudaStreamWaitEvent(s, L.ev_side_done, 0), "wait side")) return rc;
  }
  ctx->prof_step_start(s);
  const LayerState::Lists& Dm = L.dm[step & 1];
  if (int rc = run_demand_score(ctx, layer, step, q, Dm.topk_ids, Dm.topk_scores, s, true))
    return rc;
  // Look-ahead side work on the table the demand fetch left: the scan +
  // top-K + capped admission per request group on `side`, each group's
  // gather on `side2` (into spare units, which the attention does not read).
  if (int rc = ctx->cuda(cudaEventRecord(L.ev_demand_done, s), "record demand")) return rc;
  if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side, L.ev_demand_done, 0), "side wait"))
    return rc;
  if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side2, L.ev_demand_done, 0), "side2 wait"))
    return rc;
  const int pairs = ctx->cfg.num_requests * ctx->cfg.num_kv_heads;
  const LayerState::Lists& Ls = L.lists[step & 1];
  for (int g = 0; g < ctx->groups; ++g) {
    const int p0 = static_cast<int>(static_cast<long long>(pairs) * g / ctx->groups);
    const int p1 = static_cast<int>(static_cast<long long>(pairs) * (g + 1) / ctx->groups);
    if (int rc = run_score(ctx, layer, step, qd_copy, Ls.topk_ids, Ls.topk_scores, ctx->side, p0,
                           p1 - p0, true))
      return rc;
    if (int rc = ctx->cuda(cudaEventRecord(L.ev_group[g], ctx->side), "record group")) return rc;
    if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side2, L.ev_group[g], 0), "group wait"))
      return rc;
    if (ctx->C > 0) {
      if (int rc = run_prefetch(ctx, layer, step, Ls.admit_ids, Ls.admit_slots, Ls.n_admit,
                                ctx->side2, p0, p1 - p0))
        return rc;
    }
  }
  if (int rc = ctx->cuda(cudaEventRecord(L.ev_admitted[step & 1], ctx->side), "record admitted"))
    return rc;
  L.admitted_pending[step & 1] = true;
  // The stall: the demand units land before the attention reads the table.
  if (int rc = run_demand_gather(ctx, layer, step, Dm.admit_ids, Dm.admit_slots, Dm.n_admit, s))
    return rc;
  if (int rc = run_attention(ctx, layer, step, q, q_draft, out, out_draft, s)) return rc;
  if (int rc = ctx->cuda(cudaEventRecord(L.ev_side_done, ctx->side2), "record side")) return rc;
  L.side_pending = true;
  return OASIS_OK;
}

OASIS_API int oasis_stall_lists(oasis_ctx* ctx, int layer, int step, int32_t** topk_ids,
                                float** topk_scores, int32_t** admit_ids, int32_t** admit_slots,
                                int32_t** evict_ids, int32_t** n_admit) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0) return ctx->fail(OASIS_EINVAL, "stall_lists: bad step");
  const LayerState::Lists& Dm = ctx->layers[layer].dm[step & 1];
  if (topk_ids) *topk_ids = Dm.topk_ids;
  if (topk_scores) *topk_scores = Dm.topk_scores;
  if (admit_ids) *admit_ids = Dm.admit_ids;
  if (admit_slots) *admit_slots = Dm.admit_slots;
  if (evict_ids) *evict_ids = Dm.evict_ids;
  if (n_admit) *n_admit = Dm.n_admit;
  return OASIS_OK;
}

namespace {
int step_impl(oasis_ctx* ctx, int layer, int step, const void* q, const void* q_draft, void* out,
              void* out_draft, void* stream, int schedule, cudaEvent_t inputs_ready);
}  // namespace

OASIS_API int oasis_step(oasis_ctx* ctx, int layer, int step, const void* q,
                         const void* q_draft, void* out, void* out_draft, void* stream) {
  NvtxRange nvtx("oasis_step");
  if (!ctx) return OASIS_EINVAL;
  const int sched = ctx->cfg.schedule == OASIS_SCHEDULE_AUTO ? OASIS_SCHEDULE_SCAN_FIRST
                                                              : ctx->cfg.schedule;
  return step_impl(ctx, layer, step, q, q_draft, out, out_draft, stream, sched, nullptr);
}

namespace {
// inputs_ready: with the early-scan schedule, the event after which the draft
// queries may be read (null: they are ready when the call is made).
int step_impl(oasis_ctx* ctx, int layer, int step, const void* q, const void* q_draft, void* out,
              void* out_draft, void* stream, int schedule, cudaEvent_t inputs_ready) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || step > (1 << 30) || !q || !q_draft || !out || !out_draft)
    return ctx->fail(OASIS_EINVAL, "step: bad step or null pointer");
  LayerState& L = ctx->layers[layer];
  if (!L.loaded) return ctx->fail(OASIS_ESTATE, "layer %d: oasis_load_resident first", layer);
  if (int rc = ctx->set_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool early = schedule == OASIS_SCHEDULE_EARLY_SCAN;
  // The side work reads the draft query from a per-layer double buffer, so
  // the caller may reuse its buffer as soon as `stream` passes this call.
  // Scan-first needs no copy: `stream` passes the call only after the
  // attention, which waits for the last scan, the only reader of q_draft on
  // the side streams.
  const bool stage_qd = schedule != OASIS_SCHEDULE_SCAN_FIRST;
  void* qd_copy = L.qd_ring[step & 1];
  const void* qd_scan = stage_qd ? qd_copy : q_draft;
  const size_t qbytes = static_cast<size_t>(ctx->D) * ctx->cfg.num_requests *
                        ctx->cfg.num_q_heads * kHeadDim * 2;
  if (early) {
    // Early scan: the scans run on their own stream as soon as the draft
    // queries, the summaries and the context lengths they read exist, not
    // after the work already on `stream` (the previous attention).  They
    // write only this step's top-K lists, whose previous readers (the
    // admissions two steps back) must be done.
    cudaStream_t sc = ctx->side3;
    if (inputs_ready) {
      if (int rc = ctx->cuda(cudaStreamWaitEvent(sc, inputs_ready, 0), "scan wait inputs"))
        return rc;
    }
    if (L.mut_pending) {
      if (int rc = ctx->cuda(cudaStreamWaitEvent(sc, L.ev_mut, 0), "scan wait summaries"))
        return rc;
    }
    if (ctx->ctx_mut_pending) {
      if (int rc = ctx->cuda(cudaStreamWaitEvent(sc, ctx->ev_ctx_mut, 0), "scan wait ctx_len"))
        return rc;
    }
    if (L.admitted_pending[step & 1]) {
      if (int rc = ctx->cuda(cudaStreamWaitEvent(sc, L.ev_admitted[step & 1], 0),
                             "scan wait lists"))
        return rc;
    }
    if (int rc = ctx->cuda(cudaMemcpyAsync(qd_copy, q_draft, qbytes, cudaMemcpyDeviceToDevice,
                                           sc), "stage q_draft"))
      return rc;
    if (int rc = ctx->cuda(cudaEventRecord(L.ev_qd_copied, sc), "record q_draft staged"))
      return rc;
  } else if (stage_qd) {
    if (int rc = ctx->cuda(cudaMemcpyAsync(qd_copy, q_draft, qbytes, cudaMemcpyDeviceToDevice, s),
                           "stage q_draft"))
      return rc;
  }
  // Start of this step's side work: everything earlier on `stream`, which
  // includes the previous step's attention of this layer.  That is all the
  // scan and the admission need (the admission rewrites the table the
  // previous attention read, and its gathers write units that attention
  // read), so the scan may overlap the previous step's gathers.
  if (int rc = ctx->cuda(cudaEventRecord(L.ev_start, s), "record start")) return rc;
  ctx->prof_step_start(s);
  if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side, L.ev_start, 0), "side wait")) return rc;
  if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side2, L.ev_start, 0), "side2 wait")) return rc;
  // This step's attention needs the previous step's admissions in the pool.
  if (L.side_pending) {
    if (int rc = ctx->cuda(cudaStreamWaitEvent(s, L.ev_side_done, 0), "wait side")) return rc;
  }
  // Request group g: scan + top-K + admission on `side`, then its gather on
  // `side2` as soon as the group's admissions exist.
  const int pairs = ctx->cfg.num_requests * ctx->cfg.num_kv_heads;
  for (int g = 0; g < ctx->groups; ++g) {
    const int p0 = static_cast<int>(static_cast<long long>(pairs) * g / ctx->groups);
    const int p1 = static_cast<int>(static_cast<long long>(pairs) * (g + 1) / ctx->groups);
    const LayerState::Lists& Ls = L.lists[step & 1];
    if (early) {
      // Scan + top-K on side3 (already running ahead); the group's
      // admission on `side` after the step start and the group's scan; its
      // gather on side2.
      if (int rc = run_score(ctx, layer, step, qd_scan, Ls.topk_ids, Ls.topk_scores, ctx->side3,
                             p0, p1 - p0, false))
        return rc;
      if (int rc = ctx->cuda(cudaEventRecord(L.ev_group2[g], ctx->side3), "record top-k"))
        return rc;
      if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side, L.ev_group2[g], 0), "wait top-k"))
        return rc;
      if (int rc = run_admit(ctx, layer, step, Ls.topk_ids, Ls.admit_ids, Ls.admit_slots,
                             Ls.evict_ids, Ls.n_admit, ctx->side, p0, p1 - p0))
        return rc;
      if (int rc = ctx->cuda(cudaEventRecord(L.ev_group[g], ctx->side), "record group"))
        return rc;
      if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side2, L.ev_group[g], 0), "group wait"))
        return rc;
      if (ctx->C > 0) {
        if (int rc = run_prefetch(ctx, layer, step, Ls.admit_ids, Ls.admit_slots, Ls.n_admit,
                                  ctx->side2, p0, p1 - p0))
          return rc;
      }
      continue;
    }
    if (schedule == OASIS_SCHEDULE_THREE_STREAMS) {
      // The pages' pipeline: top-K prediction, KV selection and KV transfer
      // on three streams, each stage of a group ordered by an event.
      if (int rc = run_score(ctx, layer, step, qd_scan, Ls.topk_ids, Ls.topk_scores, ctx->side,
                             p0, p1 - p0, false))
        return rc;
      if (int rc = ctx->cuda(cudaEventRecord(L.ev_group2[g], ctx->side), "record top-k"))
        return rc;
      if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side3, L.ev_group2[g], 0), "wait top-k"))
        return rc;
      if (int rc = run_admit(ctx, layer, step, Ls.topk_ids, Ls.admit_ids, Ls.admit_slots,
                             Ls.evict_ids, Ls.n_admit, ctx->side3, p0, p1 - p0))
        return rc;
      if (int rc = ctx->cuda(cudaEventRecord(L.ev_group[g], ctx->side3), "record group"))
        return rc;
      if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side2, L.ev_group[g], 0), "group wait"))
        return rc;
      if (ctx->C > 0) {
        if (int rc = run_prefetch(ctx, layer, step, Ls.admit_ids, Ls.admit_slots, Ls.n_admit,
                                  ctx->side2, p0, p1 - p0))
          return rc;
      }
      continue;
    }
    // Scan-first: the attention waits for the last group's scan (the
    // ranking and admission after it overlap the attention).
    cudaEvent_t scanned =
        schedule == OASIS_SCHEDULE_SCAN_FIRST && g == ctx->groups - 1 ? L.ev_scan_done : nullptr;
    if (int rc = run_score(ctx, layer, step, qd_scan, Ls.topk_ids, Ls.topk_scores, ctx->side, p0,
                           p1 - p0, true, scanned))
      return rc;
    if (ctx->C > 0) {
      if (int rc = ctx->cuda(cudaEventRecord(L.ev_group[g], ctx->side), "record group"))
        return rc;
      if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side2, L.ev_group[g], 0), "group wait"))
        return rc;
      if (int rc = run_prefetch(ctx, layer, step, Ls.admit_ids, Ls.admit_slots, Ls.n_admit,
                                ctx->side2, p0, p1 - p0))
        return rc;
    }
  }
  if (ctx->C == 0) {
    if (int rc = ctx->cuda(cudaEventRecord(L.ev_group[0], ctx->side), "record group")) return rc;
    if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->side2, L.ev_group[0], 0), "group wait"))
      return rc;
  }
  if (early) {
    if (int rc = ctx->cuda(cudaEventRecord(L.ev_admitted[step & 1], ctx->side), "record admitted"))
      return rc;
    L.admitted_pending[step & 1] = true;
    // The caller may reuse q_draft once `stream` passes this call.
    if (int rc = ctx->cuda(cudaStreamWaitEvent(s, L.ev_qd_copied, 0), "wait q_draft staged"))
      return rc;
  }
  if (schedule == OASIS_SCHEDULE_SCAN_FIRST) {
    // The scan gets the whole HBM bandwidth and the SMs first, so the
    // gathers (host-link bound) start as early as possible; the attention
    // then overlaps the ranking, the admission and the gathers, which write
    // only spare units.  (ev_scan_done was recorded after the last group's
    // scan above.)
    if (int rc = ctx->cuda(cudaStreamWaitEvent(s, L.ev_scan_done, 0), "wait scan")) return rc;
  }
  if (int rc = run_attention(ctx, layer, step, q, q_draft, out, out_draft, s)) return rc;
  if (int rc = ctx->cuda(cudaEventRecord(L.ev_side_done, ctx->side2), "record side")) return rc;
  L.side_pending = true;
  return OASIS_OK;
}

}  // namespace

OASIS_API int oasis_wait(oasis_ctx* ctx, int layer, double timeout_ms) {
  NvtxRange nvtx("oasis_wait");
  if (int rc = check_layer(ctx, layer)) return rc;
  if (!(timeout_ms >= 0.0)) return ctx->fail(OASIS_EINVAL, "wait: timeout must be >= 0");
  if (int rc = ctx->set_device()) return rc;
  LayerState& L = ctx->layers[layer];
  if (!L.side_pending) return OASIS_OK;
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t e = cudaEventQuery(L.ev_side_done);
    if (e == cudaSuccess) return OASIS_OK;
    if (e != cudaErrorNotReady) return ctx->cuda(e, "wait: event query");
    const double ms =
        std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    if (ms >= timeout_ms)
      return ctx->fail(OASIS_ETIMEOUT, "wait: layer %d side work not done after %.1f ms", layer,
                       timeout_ms);
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

OASIS_API int oasis_join(oasis_ctx* ctx, int layer, void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (int rc = ctx->set_device()) return rc;
  LayerState& L = ctx->layers[layer];
  if (!L.side_pending) return OASIS_OK;
  return ctx->cuda(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), L.ev_side_done, 0),
                   "join");
}

namespace {
// The schedule AUTO picks for the host-buffer steps.
constexpr int kHostAuto = OASIS_SCHEDULE_SCAN_FIRST;

// Host-buffer step.  async = false: outputs copied back on `stream`
// (complete when `stream` passes the call); true: on the output stream,
// complete when oasis_wait_outputs(layer, step) says so.
int step_host_impl(oasis_ctx* ctx, int layer, int step, const void* q_host,
                   const void* q_draft_host, void* out_host, void* out_draft_host, void* stream,
                   bool async) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (!q_host || !q_draft_host || !out_host || !out_draft_host)
    return ctx->fail(OASIS_EINVAL, "step_host: null pointer");
  LayerState& L = ctx->layers[layer];
  if (!L.loaded) return ctx->fail(OASIS_ESTATE, "layer %d: oasis_load_resident first", layer);
  if (int rc = ctx->set_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Inputs go to the staging slot of this step's parity on the input stream,
  // as soon as the slot's last readers are done (step - 2's attention, and
  // its q_draft copy or scan-first scans, which `stream` passed before that
  // attention), so they usually land while the previous step still
  // computes; `stream` waits for them before the step.
  const int slot = step & 1;
  const size_t qb = static_cast<size_t>(ctx->cfg.num_requests) * ctx->cfg.num_q_heads * kHeadDim * 2;
  const size_t ob = qb * (ctx->cfg.out_fp32 ? 2 : 1);
  if (L.stage_used[slot]) {
    if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->io, L.ev_stage_free[slot], 0), "wait stage"))
      return rc;
  }
  if (int rc = ctx->cuda(cudaMemcpyAsync(L.q_stage[slot], q_host, qb, cudaMemcpyHostToDevice,
                                         ctx->io), "h2d q"))
    return rc;
  if (int rc = ctx->cuda(cudaMemcpyAsync(L.qd_stage[slot], q_draft_host, ctx->D * qb,
                                         cudaMemcpyHostToDevice, ctx->io), "h2d q_draft"))
    return rc;
  if (int rc = ctx->cuda(cudaEventRecord(L.ev_in[slot], ctx->io), "record inputs")) return rc;
  if (int rc = ctx->cuda(cudaStreamWaitEvent(s, L.ev_in[slot], 0), "wait inputs")) return rc;
  // The output slot's previous copy back (step - 2, on the output stream)
  // must be done before this step's attention rewrites it.
  if (L.out_pending[slot]) {
    if (int rc = ctx->cuda(cudaStreamWaitEvent(s, L.ev_out_done[slot], 0), "wait output slot"))
      return rc;
  }
  // AUTO: scan-first, as for oasis_step, with the outputs copied back on
  // `stream` too (measured end to end since the scan-first scans read the
  // draft queries in place: 3070-3073 against 2683-2703 layer-steps/s with
  // the attention starting at once).
  const int sched = ctx->cfg.schedule != OASIS_SCHEDULE_AUTO ? ctx->cfg.schedule
                                                             : kHostAuto;
  if (int rc = step_impl(ctx, layer, step, L.q_stage[slot], L.qd_stage[slot], L.out_stage[slot],
                         L.outd_stage[slot], stream, sched, L.ev_in[slot]))
    return rc;
  if (int rc = ctx->cuda(cudaEventRecord(L.ev_stage_free[slot], s), "record stage")) return rc;
  L.stage_used[slot] = true;
  // The outputs go back with copies: the attention writing the mapped host
  // buffers itself was slower end to end (2871 against 2935 layer-steps/s).
  cudaStream_t so = s;
  if (async) {
    if (int rc = ctx->cuda(cudaEventRecord(L.ev_attn_done, s), "record attention")) return rc;
    if (int rc = ctx->cuda(cudaStreamWaitEvent(ctx->io_out, L.ev_attn_done, 0), "out wait"))
      return rc;
    so = ctx->io_out;
  }
  if (int rc = ctx->cuda(cudaMemcpyAsync(out_host, L.out_stage[slot], ob, cudaMemcpyDeviceToHost,
                                         so), "d2h out"))
    return rc;
  if (int rc = ctx->cuda(cudaMemcpyAsync(out_draft_host, L.outd_stage[slot], ctx->D * ob,
                                         cudaMemcpyDeviceToHost, so), "d2h out_draft"))
    return rc;
  if (int rc = ctx->cuda(cudaEventRecord(L.ev_out_done[slot], so), "record outputs")) return rc;
  L.out_step[slot] = step;
  // Only copies on the output stream need a wait before the slot's next use;
  // those on `stream` are ordered before it anyway.
  L.out_pending[slot] = async;
  return OASIS_OK;
}
}  // namespace

OASIS_API int oasis_step_host(oasis_ctx* ctx, int layer, int step, const void* q_host,
                              const void* q_draft_host, void* out_host, void* out_draft_host,
                              void* stream) {
  return step_host_impl(ctx, layer, step, q_host, q_draft_host, out_host, out_draft_host, stream,
                        false);
}

OASIS_API int oasis_step_host_async(oasis_ctx* ctx, int layer, int step, const void* q_host,
                                    const void* q_draft_host, void* out_host,
                                    void* out_draft_host, void* stream) {
  return step_host_impl(ctx, layer, step, q_host, q_draft_host, out_host, out_draft_host, stream,
                        true);
}

OASIS_API int oasis_wait_outputs(oasis_ctx* ctx, int layer, int step, double timeout_ms) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || !(timeout_ms >= 0.0))
    return ctx->fail(OASIS_EINVAL, "wait_outputs: bad step or timeout");
  if (int rc = ctx->set_device()) return rc;
  LayerState& L = ctx->layers[layer];
  const int slot = step & 1;
  if (L.out_step[slot] != step)
    return ctx->fail(OASIS_ESTATE, "wait_outputs: layer %d holds no outputs of step %d", layer,
                     step);
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t e = cudaEventQuery(L.ev_out_done[slot]);
    if (e == cudaSuccess) return OASIS_OK;
    if (e != cudaErrorNotReady) return ctx->cuda(e, "wait_outputs: event query");
    const double ms =
        std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    if (ms >= timeout_ms)
      return ctx->fail(OASIS_ETIMEOUT, "wait_outputs: layer %d step %d not done after %.1f ms",
                       layer, step, timeout_ms);
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

OASIS_API int oasis_step_lists(oasis_ctx* ctx, int layer, int step, int32_t** topk_ids,
                               float** topk_scores, int32_t** admit_ids, int32_t** admit_slots,
                               int32_t** evict_ids, int32_t** n_admit) {
  if (int rc = check_layer(ctx, layer)) return rc;
  LayerState& L = ctx->layers[layer];
  if (step < 0) return ctx->fail(OASIS_EINVAL, "step_lists: bad step");
  const LayerState::Lists& Ls = L.lists[step & 1];
  if (topk_ids) *topk_ids = Ls.topk_ids;
  if (topk_scores) *topk_scores = Ls.topk_scores;
  if (admit_ids) *admit_ids = Ls.admit_ids;
  if (admit_slots) *admit_slots = Ls.admit_slots;
  if (evict_ids) *evict_ids = Ls.evict_ids;
  if (n_admit) *n_admit = Ls.n_admit;
  return OASIS_OK;
}

OASIS_API int oasis_append_token(oasis_ctx* ctx, int layer, int step, const void* k_new,
                                 const void* v_new, void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || !k_new || !v_new) return ctx->fail(OASIS_EINVAL, "append: bad argument");
  if (int rc = ctx->set_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerState& L = ctx->layers[layer];
  // The token may land in a block this layer's side work is copying.
  if (L.side_pending) {
    if (int rc = ctx->cuda(cudaStreamWaitEvent(s, L.ev_side_done, 0), "wait side")) return rc;
  }
  AppendArgs a{};
  a.k_new = k_new;
  a.v_new = v_new;
  a.host = L.remote ? L.remote->local_dev : L.host_dev;
  a.local_map = L.remote ? L.remote->map : nullptr;
  a.local_count = L.remote ? L.remote->count : nullptr;
  a.capacity = L.remote ? L.remote->capacity : 0;
  a.summ = L.summ;
  a.pool = L.pool;
  a.ctx_len = ctx->ctx_tab(step);
  a.res_nxt = ctx->res_tab(layer, step + 1);
  a.phys_nxt = ctx->phys_tab(layer, step + 1);
  a.err = ctx->err;
  a.R = ctx->cfg.num_requests;
  a.Hkv = ctx->cfg.num_kv_heads;
  a.NBmax = ctx->cfg.max_blocks;
  a.K = ctx->cfg.topk;
  a.U = ctx->U;
  if (int rc = ctx->cuda(launch_append(a, s), "append launch")) return rc;
  return note_summary_write(ctx, L, s);
}

OASIS_API int oasis_refresh_blocks(oasis_ctx* ctx, int layer, int step, const int32_t* ids,
                                   const int32_t* n_ids, int max_ids, void* stream) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (step < 0 || !ids || !n_ids || max_ids < 0)
    return ctx->fail(OASIS_EINVAL, "refresh: bad argument");
  if (int rc = ctx->set_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerState& L = ctx->layers[layer];
  if (L.remote)
    return ctx->fail(OASIS_ESTATE, "refresh: layer %d has a remote tier attached", layer);
  // The previous step's gathers write units of table (step & 1).
  if (L.side_pending) {
    if (int rc = ctx->cuda(cudaStreamWaitEvent(s, L.ev_side_done, 0), "wait side")) return rc;
  }
  RefreshArgs a{};
  a.host = L.host_dev;
  a.summ = L.summ;
  a.pool = L.pool;
  a.ids = ids;
  a.n_ids = n_ids;
  a.ctx_len = ctx->ctx_tab(step);
  a.res = ctx->res_tab(layer, step);
  a.phys = ctx->phys_tab(layer, step);
  a.err = ctx->err;
  a.R = ctx->cfg.num_requests;
  a.Hkv = ctx->cfg.num_kv_heads;
  a.NBmax = ctx->cfg.max_blocks;
  a.K = ctx->cfg.topk;
  a.U = ctx->U;
  a.max_ids = max_ids;
  if (int rc = ctx->cuda(launch_refresh(a, s), "refresh launch")) return rc;
  return note_summary_write(ctx, L, s);
}

OASIS_API int oasis_advance_context(oasis_ctx* ctx, int step, int grow, void* stream) {
  if (!ctx) return OASIS_EINVAL;
  if (step < 0 || grow < 0) return ctx->fail(OASIS_EINVAL, "advance: bad argument");
  if (int rc = ctx->set_device()) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = ctx->cuda(launch_advance(ctx->ctx_tab(step), ctx->ctx_tab(step + 1),
                                        ctx->cfg.num_requests, grow, s),
                         "advance launch"))
    return rc;
  // An early scan of a later step reads the new table: it waits for this.
  if (int rc = ctx->cuda(cudaEventRecord(ctx->ev_ctx_mut, s), "record ctx write")) return rc;
  ctx->ctx_mut_pending = true;
  return OASIS_OK;
}

namespace {
const char* remote_config_error(const oasis_config* cfg, const oasis_remote_config* r) {
  if (!r) return "remote config is NULL";
  if (r->capacity < cfg->topk || r->capacity > cfg->max_blocks)
    return "remote capacity must be in [K, NBmax]";
  if (!(r->gbps >= 0.f) || std::isinf(r->gbps)) return "remote gbps must be finite and >= 0";
  if (r->threads < 0 || r->threads > 16) return "remote threads must be in 0..16";
  return nullptr;
}
}  // namespace

OASIS_API int oasis_remote_query_sizes(const oasis_config* cfg, const oasis_remote_config* rcfg,
                                       oasis_remote_sizes* out) {
  if (!out || config_error(cfg) || remote_config_error(cfg, rcfg)) return OASIS_EINVAL;
  const size_t pairs = static_cast<size_t>(cfg->num_requests) * cfg->num_kv_heads;
  const size_t M = std::max(cfg->topk, fetch_cap(*cfg));
  out->local_tier_bytes = pairs * rcfg->capacity * kUnitBytes;
  out->local_map_bytes = (pairs * cfg->max_blocks + 2 * pairs) * 4;
  // the lists, then two 32-bit sequence words (16-byte aligned)
  out->miss_lists_bytes = ((pairs + 2 * pairs * M) * 4 + 15) / 16 * 16 + 16;
  return OASIS_OK;
}

OASIS_API int oasis_remote_attach(oasis_ctx* ctx, int layer, const oasis_remote_config* rcfg,
                                  void* local_tier, int32_t* local_map, int32_t* miss_lists) {
  if (int rc = check_layer(ctx, layer)) return rc;
  if (const char* e = remote_config_error(&ctx->cfg, rcfg))
    return ctx->fail(OASIS_EINVAL, "remote_attach: %s", e);
  if (!local_tier || !local_map || !miss_lists || !aligned16(local_tier) ||
      !aligned16(local_map) || !aligned16(miss_lists))
    return ctx->fail(OASIS_EINVAL, "remote_attach: null or misaligned buffer");
  LayerState& L = ctx->layers[layer];
  if (L.loaded || L.remote)
    return ctx->fail(OASIS_ESTATE, "remote_attach: layer %d already loaded or attached", layer);
  if (int rc = ctx->set_device()) return rc;
  std::unique_ptr<RemoteTier> T(new (std::nothrow) RemoteTier());
  if (!T) return ctx->fail(OASIS_ENOMEM, "remote tier");
  T->capacity = rcfg->capacity;
  T->M = std::max(ctx->cfg.topk, ctx->C);
  T->threads = rcfg->threads > 0 ? rcfg->threads : 4;
  T->gbps = rcfg->gbps;
  T->local = static_cast<uint8_t*>(local_tier);
  T->lists = miss_lists;
  void* d = mapped_host(local_tier);
  if (!d)
    return ctx->fail(OASIS_EINVAL, "remote_attach: local_tier is not mapped page-locked memory");
  T->local_dev = d;
  d = mapped_host(miss_lists);
  if (!d)
    return ctx->fail(OASIS_EINVAL, "remote_attach: miss_lists is not mapped page-locked memory");
  T->lists_dev = static_cast<int32_t*>(d);
  const size_t pairs = static_cast<size_t>(ctx->cfg.num_requests) * ctx->cfg.num_kv_heads;
  T->map = local_map;
  T->count = local_map + pairs * ctx->cfg.max_blocks;
  T->base = T->count + pairs;
  if (!get_wait_value32() || !get_write_value32())
    return ctx->fail(OASIS_ECUDA, "remote_attach: stream memory operations unavailable");
  {
    const size_t words = ((pairs + 2 * pairs * static_cast<size_t>(T->M)) * 4 + 15) / 16 * 16;
    uint8_t* hb = reinterpret_cast<uint8_t*>(miss_lists) + words;
    uint8_t* db = reinterpret_cast<uint8_t*>(T->lists_dev) + words;
    T->assigned = reinterpret_cast<volatile uint32_t*>(hb);
    T->moved = reinterpret_cast<volatile uint32_t*>(hb + 4);
    T->assigned_dev = reinterpret_cast<CUdeviceptr>(db);
    T->moved_dev = reinterpret_cast<CUdeviceptr>(db + 4);
    *T->assigned = 0;
    *T->moved = 0;
  }
  T->remote = static_cast<const uint8_t*>(L.host);
  T->NBmax = ctx->cfg.max_blocks;
  T->all_pairs = static_cast<int>(pairs);
  T->pool.reset(new (std::nothrow) CopyPool(T->threads));
  if (!T->pool) return ctx->fail(OASIS_ENOMEM, "remote_attach: copy threads");
  T->start();
  if (int rc = ctx->cuda(cudaMemsetAsync(T->map, 0xff, pairs * ctx->cfg.max_blocks * 4, ctx->side2),
                         "clear local map"))
    return rc;
  if (int rc = ctx->cuda(cudaMemsetAsync(T->count, 0, 2 * pairs * 4, ctx->side2), "clear slot counts"))
    return rc;
  if (int rc = ctx->cuda(cudaStreamSynchronize(ctx->side2), "remote attach sync")) return rc;
  std::memset(miss_lists, 0, pairs * 4);
  L.remote = std::move(T);
  return OASIS_OK;
}

OASIS_API int oasis_remote_stats(oasis_ctx* ctx, int layer, int64_t* units, int64_t* transfers,
                                 double* seconds, int64_t* bad_entries) {
  if (int rc = check_layer(ctx, layer)) return rc;
  const LayerState& L = ctx->layers[layer];
  if (!L.remote) return ctx->fail(OASIS_ESTATE, "remote_stats: layer %d has no remote tier", layer);
  const RemoteStats& S = L.remote->stats;
  if (units) *units = S.units.load();
  if (transfers) *transfers = S.transfers.load();
  if (seconds) *seconds = static_cast<double>(S.nanos.load()) * 1e-9;
  if (bad_entries) *bad_entries = S.bad.load();
  return OASIS_OK;
}

OASIS_API int oasis_set_wait_limit(oasis_ctx* ctx, long long cycles) {
  if (!ctx) return OASIS_EINVAL;
  ctx->wait_limit = cycles > 0 ? cycles : kWaitLimitCycles;
  return OASIS_OK;
}

OASIS_API int oasis_profile_enable(oasis_ctx* ctx, int enable) {
  if (!ctx) return OASIS_EINVAL;
  ctx->prof = enable != 0;
  ctx->prof_used = 0;
  ctx->prof_starts_used = 0;
  return OASIS_OK;
}

OASIS_API int oasis_profile_read_n(oasis_ctx* ctx, int nkinds, double* ms_sum, int64_t* count,
                                   double* start_ms_sum) {
  if (!ctx || !ms_sum || !count || nkinds < 1 || nkinds > OASIS_PROFILE_KINDS)
    return OASIS_EINVAL;
  if (int rc = ctx->set_device()) return rc;
  if (int rc = ctx->cuda(cudaDeviceSynchronize(), "cudaDeviceSynchronize")) return rc;
  for (int k = 0; k < nkinds; ++k) {
    ms_sum[k] = 0.0;
    count[k] = 0;
    if (start_ms_sum) start_ms_sum[k] = 0.0;
  }
  for (size_t i = 0; i < ctx->prof_used; ++i) {
    const ProfPair& p = ctx->prof_pool[i];
    float ms = 0.f;
    if (p.kind < nkinds && cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
      ms_sum[p.kind] += ms;
      count[p.kind] += 1;
      float off = 0.f;
      if (start_ms_sum && p.start >= 0 &&
          cudaEventElapsedTime(&off, ctx->prof_starts[p.start], p.a) == cudaSuccess)
        start_ms_sum[p.kind] += off;
    }
  }
  ctx->prof_used = 0;
  ctx->prof_starts_used = 0;
  return OASIS_OK;
}

OASIS_API int oasis_profile_read(oasis_ctx* ctx, double* ms_sum4, int64_t* count4,
                                 double* start_ms_sum4) {
  return oasis_profile_read_n(ctx, 4, ms_sum4, count4, start_ms_sum4);
}

}  // extern "C"
