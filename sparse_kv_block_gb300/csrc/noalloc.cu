// noalloc.cu -- the fixed device scratch of oasis_score_admit_noalloc.
//
// That entry point runs the summary scan + top-K kernel and then the capped
// eviction kernel with the top-K list between them held here, in a
// file-scope device array, instead of in memory the caller allocates.  It
// serves callers that cannot allocate device memory at the point where they
// issue a step: an embedding whose device memory is fully committed to the
// KV pool and summaries (the caller of the stage-level calls otherwise has
// to allocate the R x Hkv x K top-K buffer between oasis_score_topk and
// oasis_admit_evict), or one whose allocator may not be entered from the
// thread that drives the decode loop.
#include <mutex>

#include "kernels.h"

namespace oasis {
namespace {

// 1 MiB: the top-K lists of up to 262144 (request, KV head, slot) entries,
// e.g. 128 requests x 8 KV heads x K = 256.  Nothing in it needs to start at
// zero: the scan kernel writes every entry of every pair (ids or -1) before
// the admission kernel, later on the same stream, reads them.
__device__ __align__(256) int32_t g_topk_scratch[kNoAllocTopkEntries];

constexpr int kMaxDevices = 64;

}  // namespace

cudaError_t noalloc_topk_scratch(int device, int32_t** ptr) {
  // One symbol lookup per device, made with that device current.
  static std::mutex m;
  static int32_t* cache[kMaxDevices] = {};
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(m);
  if (!cache[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess) return e;
    cache[device] = static_cast<int32_t*>(p);
  }
  *ptr = cache[device];
  return cudaSuccess;
}

}  // namespace oasis
