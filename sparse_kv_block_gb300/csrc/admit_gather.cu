// admit_gather.cu -- capped eviction (a4), prefetch gather (a5) and the
// support kernels: table initialisation, summary build and token append.
#include "common.cuh"
#include "kernels.h"

namespace oasis {
namespace {

// ------------------------------------------------------------------ a4
// Capped least-recently-selected eviction, one warp per (request, KV head)
// ("Pith review of OasisKV", section "What carries the argument": a
// capped-eviction policy pairs each admitted nonresident block with a
// least-recently-selected resident block so per-step traffic is bounded).
// Reading of the pages: (i) stamp re-selected residents with the step;
// (ii) missing top-K blocks in rank order; (iii) candidates = unselected
// slots, empty first, then (stamp, block id, slot) ascending; (iv) at most C;
// (v) pair the i-th missing block with the i-th candidate.  The admitted
// block takes spare pool unit K+i; the evicted unit becomes that spare, so
// the copy never touches a unit the current table still references.
constexpr int kAdmitWarps = 4;

struct AdmitSmem {
  int topk[kMaxTopK];
  int res[kMaxTopK];
  int stamp[kMaxTopK];
  int phys[2 * kMaxTopK];
  unsigned char in_t[kMaxTopK];
  unsigned char is_res[kMaxTopK];
  int missing[kMaxTopK];
  int evslot[kMaxTopK];
};

__global__ void __launch_bounds__(kAdmitWarps * 32) admit_kernel(const AdmitArgs a) {
  __shared__ AdmitSmem sm_all[kAdmitWarps];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x * kAdmitWarps + warp;
  if (pair >= a.R * a.Hkv) return;  // warp-uniform; no block barrier follows
  AdmitSmem& S = sm_all[warp];
  const int K = a.K, C = a.C, U = a.U;
  const size_t ok_ = static_cast<size_t>(pair) * K;
  const size_t ou = static_cast<size_t>(pair) * U;

  for (int s = lane; s < K; s += 32) {
    S.topk[s] = a.topk[ok_ + s];
    S.res[s] = a.res_cur[ok_ + s];
    S.stamp[s] = a.stamps[ok_ + s];
  }
  for (int u = lane; u < U; u += 32) S.phys[u] = a.phys_cur[ou + u];
  __syncwarp();

  // Membership both ways (K x K compares; K <= 256).
  for (int s = lane; s < K; s += 32) {
    const int id = S.res[s];
    bool f = false;
    if (id >= 0)
      for (int i = 0; i < K; ++i) f |= (S.topk[i] == id);
    S.in_t[s] = f;
    if (f) S.stamp[s] = a.step;
    const int b = S.topk[s];
    bool rr = false;
    if (b >= 0)
      for (int i = 0; i < K; ++i) rr |= (S.res[i] == b);
    S.is_res[s] = rr;
  }
  __syncwarp();

  // (ii) missing blocks in rank order (ballot compaction).
  int n_missing = 0;
  for (int c = 0; c < K; c += 32) {
    const int i = c + lane;
    const bool m = i < K && S.topk[i] >= 0 && !S.is_res[i];
    const unsigned bal = __ballot_sync(0xffffffffu, m);
    if (m) S.missing[n_missing + __popc(bal & ((1u << lane) - 1u))] = S.topk[i];
    n_missing += __popc(bal);
  }
  const int n = min(n_missing, C);

  // (iii) rank of each eviction candidate under (nonempty, stamp, id, slot).
  for (int s = lane; s < K; s += 32) {
    if (S.in_t[s]) continue;
    const int ne = S.res[s] >= 0, st = S.stamp[s], id = S.res[s];
    int rank = 0;
    for (int s2 = 0; s2 < K; ++s2) {
      if (S.in_t[s2] || s2 == s) continue;
      const int ne2 = S.res[s2] >= 0, st2 = S.stamp[s2], id2 = S.res[s2];
      const bool less = ne2 != ne ? ne2 < ne
                                  : st2 != st ? st2 < st : id2 != id ? id2 < id : s2 < s;
      rank += less;
    }
    if (rank < n) S.evslot[rank] = s;
  }
  __syncwarp();

  // (v) outputs and the next tables.
  for (int i = lane; i < C; i += 32) {
    const size_t oc = static_cast<size_t>(pair) * C + i;
    if (i < n) {
      const int s = S.evslot[i];
      a.admit_ids[oc] = S.missing[i];
      a.admit_slots[oc] = s;
      a.evict_ids[oc] = S.res[s];
    } else {
      a.admit_ids[oc] = -1;
      a.admit_slots[oc] = -1;
      a.evict_ids[oc] = -1;
    }
  }
  if (lane == 0) a.n_admit[pair] = n;
  __syncwarp();
  // Each admission i: slot E[i] takes block M[i] and spare unit K+i; the
  // evicted unit moves to spare position K+i.  Lanes own distinct i, and the
  // evicted slots are distinct, so the updates do not collide.
  for (int i = lane; i < n; i += 32) {
    const int s = S.evslot[i];
    const int unit_old = S.phys[s];
    const int unit_new = S.phys[K + i];
    S.res[s] = S.missing[i];
    S.stamp[s] = a.step;
    S.phys[s] = unit_new;
    S.phys[K + i] = unit_old;
  }
  __syncwarp();
  for (int s = lane; s < K; s += 32) {
    a.res_nxt[ok_ + s] = S.res[s];
    a.stamps[ok_ + s] = S.stamp[s];
  }
  for (int u = lane; u < U; u += 32) a.phys_nxt[ou + u] = S.phys[u];
}

// ------------------------------------------------------------------ a5
// Gather of 8 KiB units from the pinned host store (read through its device
// mapping over the host link) into pool units, one warp per unit; every lane
// issues all 16 of its 16-byte loads before storing, so each warp keeps a
// whole unit in flight.
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const GatherArgs a) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * (kGatherThreads / 32);
  const long long total = static_cast<long long>(a.pairs) * a.items;
  for (long long it = blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5); it < total;
       it += nwarps) {
    const int pair = static_cast<int>(it / a.items);
    const int i = static_cast<int>(it - static_cast<long long>(pair) * a.items);
    if (a.n_valid && i >= a.n_valid[pair]) continue;
    const int id = a.src_ids[it];
    if (id < 0) continue;
    const int slot = a.dst_slots ? a.dst_slots[it] : i;
    const int unit = (slot >= 0 && slot < a.U) ? a.phys[static_cast<size_t>(pair) * a.U + slot] : -1;
    if (id >= a.NBmax) {
      if (lane == 0) raise_error(a.err, kErrBadBlock);
      continue;
    }
    if (unit < 0 || unit >= a.U) {
      if (lane == 0) raise_error(a.err, kErrBadUnit);
      continue;
    }
    const uint4* src = static_cast<const uint4*>(a.host) +
                       (static_cast<size_t>(pair) * a.NBmax + id) * (kUnitBytes / 16);
    uint4* dst = static_cast<uint4*>(a.pool) +
                 (static_cast<size_t>(pair) * a.U + unit) * (kUnitBytes / 16);
    uint4 v[kUnitBytes / 16 / 32];
#pragma unroll
    for (int j = 0; j < kUnitBytes / 16 / 32; ++j) v[j] = __ldcs(src + j * 32 + lane);
#pragma unroll
    for (int j = 0; j < kUnitBytes / 16 / 32; ++j) dst[j * 32 + lane] = v[j];
  }
}

__global__ void init_tables_kernel(int32_t* phys, int32_t* stamps, int pairs, int K,
                                   int U) {
  const long long n = static_cast<long long>(pairs) * U;
  for (long long i = blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    phys[i] = static_cast<int32_t>(i % U);
  }
  const long long m = static_cast<long long>(pairs) * K;
  for (long long i = blockIdx.x * blockDim.x + threadIdx.x; i < m;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    stamps[i] = -1;
  }
}

// ------------------------------------------------------------------ a0
// Per-block coordinate-wise min/max of the keys over the valid tokens, one
// warp per (request, KV head, block); lanes 0-15 take even tokens, 16-31 odd
// tokens, 8 dims per lane; bf16 min/max are exact.
__global__ void summary_build_kernel(const SummaryArgs a) {
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  const long long total = static_cast<long long>(a.R) * a.Hkv * a.NBmax;
  for (long long it = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); it < total;
       it += warps) {
    const int b = static_cast<int>(it % a.NBmax);
    const int pair = static_cast<int>(it / a.NBmax);
    const int r = pair / a.Hkv;
    const int ctx = a.ctx_len[r];
    const int valid = min(kBlock, ctx - b * kBlock);
    if (valid <= 0) continue;
    const uint4* keys = static_cast<const uint4*>(a.host) +
                        static_cast<size_t>(it) * (kUnitBytes / 16);  // K rows first
    const int dch = lane & 15;
    __nv_bfloat162 mn[4], mx[4];
    const __nv_bfloat162 pinf = __floats2bfloat162_rn(INFINITY, INFINITY);
    const __nv_bfloat162 ninf = __floats2bfloat162_rn(-INFINITY, -INFINITY);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mn[i] = pinf;
      mx[i] = ninf;
    }
    for (int tkn = lane >> 4; tkn < valid; tkn += 2) {
      const uint4 v = keys[tkn * (kHeadDim / 8) + dch];
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mn[i] = __hmin2(mn[i], p[i]);
        mx[i] = __hmax2(mx[i], p[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t mnb = *reinterpret_cast<uint32_t*>(&mn[i]);
      uint32_t mxb = *reinterpret_cast<uint32_t*>(&mx[i]);
      mnb = __shfl_xor_sync(0xffffffffu, mnb, 16);
      mxb = __shfl_xor_sync(0xffffffffu, mxb, 16);
      mn[i] = __hmin2(mn[i], *reinterpret_cast<__nv_bfloat162*>(&mnb));
      mx[i] = __hmax2(mx[i], *reinterpret_cast<__nv_bfloat162*>(&mxb));
    }
    uint4 outv;
    __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(&outv);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = (lane < 16) ? mn[i] : mx[i];
    uint4* dst = static_cast<uint4*>(a.summ) + static_cast<size_t>(it) * (kSummBytes / 16);
    dst[(lane >> 4) * (kHeadDim / 8) + dch] = outv;
  }
}

// One warp per (request, KV head): write the new token into the host store,
// fold its key into the tail summary and patch the resident copy.
__global__ void append_kernel(const AppendArgs a) {
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (pair >= a.R * a.Hkv) return;
  const int r = pair / a.Hkv;
  const int pos = a.ctx_len[r];
  if (pos < 0 || pos >= a.NBmax * kBlock) {
    if (lane == 0) raise_error(a.err, kErrBadBlock);
    return;
  }
  const int b = pos / kBlock, tk = pos % kBlock;
  const int kvsel = lane >> 4;  // 0: key, 1: value
  const int dch = lane & 15;
  const uint4 v = (kvsel ? static_cast<const uint4*>(a.v_new)
                         : static_cast<const uint4*>(a.k_new))[static_cast<size_t>(pair) * 16 + dch];
  const size_t unit_host = static_cast<size_t>(pair) * a.NBmax + b;
  uint4* hrow = static_cast<uint4*>(a.host) + unit_host * (kUnitBytes / 16) +
                (kvsel * kBlock + tk) * (kHeadDim / 8) + dch;
  *hrow = v;
  if (kvsel == 0) {
    uint4* srow = static_cast<uint4*>(a.summ) + unit_host * (kSummBytes / 16);
    uint4 mn = srow[dch], mx = srow[16 + dch];
    if (tk == 0) {
      mn = v;
      mx = v;
    } else {
      __nv_bfloat162* pn = reinterpret_cast<__nv_bfloat162*>(&mn);
      __nv_bfloat162* px = reinterpret_cast<__nv_bfloat162*>(&mx);
      const __nv_bfloat162* pv = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        pn[i] = __hmin2(pn[i], pv[i]);
        px[i] = __hmax2(px[i], pv[i]);
      }
    }
    srow[dch] = mn;
    srow[16 + dch] = mx;
  }
  // Resident copy of block b in the next table, if any.
  int slot = -1;
  for (int c = 0; c < a.K; c += 32) {
    const int s = c + lane;
    const bool hit = s < a.K && a.res_nxt[static_cast<size_t>(pair) * a.K + s] == b;
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    if (bal && slot < 0) slot = c + __ffs(bal) - 1;
  }
  if (slot >= 0) {
    const int unit = a.phys_nxt[static_cast<size_t>(pair) * a.U + slot];
    if (unit < 0 || unit >= a.U) {
      if (lane == 0) raise_error(a.err, kErrBadUnit);
      return;
    }
    uint4* prow = static_cast<uint4*>(a.pool) +
                  (static_cast<size_t>(pair) * a.U + unit) * (kUnitBytes / 16) +
                  (kvsel * kBlock + tk) * (kHeadDim / 8) + dch;
    *prow = v;
  }
}

__global__ void advance_kernel(const int32_t* cur, int32_t* nxt, int R, int grow) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < R; i += gridDim.x * blockDim.x)
    nxt[i] = cur[i] + grow;
}

int sm_count() {
  static int cached_dev = -1, cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev != cached_dev) {
    if (cudaDeviceGetAttribute(&cached, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      cached = 152;
    cached_dev = dev;
  }
  return cached;
}

}  // namespace

cudaError_t launch_admit(const AdmitArgs& a, cudaStream_t s) {
  const int pairs = a.R * a.Hkv;
  if (pairs == 0) return cudaSuccess;
  admit_kernel<<<(pairs + kAdmitWarps - 1) / kAdmitWarps, kAdmitWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s) {
  const long long total = static_cast<long long>(a.pairs) * a.items;
  if (total == 0) return cudaSuccess;
  const long long warps_needed = total;
  long long grid = (warps_needed + (kGatherThreads / 32) - 1) / (kGatherThreads / 32);
  const long long cap = 2LL * sm_count();
  if (grid > cap) grid = cap;
  gather_kernel<<<static_cast<int>(grid), kGatherThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_init_tables(int32_t* phys, int32_t* stamps, int pairs, int K,
                               int U, cudaStream_t s) {
  if (pairs == 0) return cudaSuccess;
  init_tables_kernel<<<sm_count(), 256, 0, s>>>(phys, stamps, pairs, K, U);
  return cudaGetLastError();
}

cudaError_t launch_summary_build(const SummaryArgs& a, cudaStream_t s) {
  if (a.R * a.Hkv * a.NBmax == 0) return cudaSuccess;
  summary_build_kernel<<<8 * sm_count(), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  const int pairs = a.R * a.Hkv;
  if (pairs == 0) return cudaSuccess;
  append_kernel<<<(pairs + 3) / 4, 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_advance(const int32_t* cur, int32_t* nxt, int R, int grow,
                           cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  advance_kernel<<<(R + 255) / 256, 256, 0, s>>>(cur, nxt, R, grow);
  return cudaGetLastError();
}

}  // namespace oasis
