// admit_gather.cu -- capped eviction (a4), prefetch gather (a5) and the
// support kernels: table initialisation, summary build and token append.
#include <cstdlib>

#include "admit.cuh"
#include "common.cuh"
#include "kernels.h"

namespace oasis {
namespace {

// ------------------------------------------------------------------ a4
// Stand-alone capped eviction: one warp per (request, KV head), the list
// read from global memory (the fused score kernel runs the same admit_warp
// on its own top-K list).
constexpr int kAdmitWarps = 4;

template <int KPL>
__global__ void __launch_bounds__(kAdmitWarps * 32) admit_kernel(const AdmitArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int local = blockIdx.x * kAdmitWarps + warp;
  if (local >= a.pairs) return;  // warp-uniform; no block barrier follows
  const int pair = a.pair0 + local;
  uint8_t* mine = smem + warp * admit_warp_smem_bytes(a.NBmax);
  AdmitWarpSmem& S = *reinterpret_cast<AdmitWarpSmem*>(mine);
  for (int s = lane; s < a.K; s += 32) S.topk[s] = a.topk[static_cast<size_t>(pair) * a.K + s];
  __syncwarp();
  admit_warp<KPL>(a, pair, S, reinterpret_cast<uint32_t*>(mine + sizeof(AdmitWarpSmem)));
}

template <int KPL>
cudaError_t launch_admit_kpl(const AdmitArgs& a, cudaStream_t s) {
  const size_t smem = kAdmitWarps * admit_warp_smem_bytes(a.NBmax);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(admit_kernel<KPL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  admit_kernel<KPL><<<(a.pairs + kAdmitWarps - 1) / kAdmitWarps, kAdmitWarps * 32, smem, s>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ a5
// Gather of 8 KiB units from the pinned host store (read through its device
// mapping over the host link) into pool units, one warp per unit; every lane
// issues all 16 of its 16-byte loads before storing, so each warp keeps a
// whole unit in flight.  The grid is kept small: at most kGatherCtas CTAs of
// 4 warps, 1.25 MiB of host reads in flight.  Measured on GB300 (pinned H2D
// ~210 GB/s): 16 / 32 / 64 / 96 CTAs move 131 / 174 / 199 / 206 GB/s, while a
// concurrent HBM-streaming kernel slows by 1 / 9 / 35 / 48 %: the host reads
// in flight compete with HBM traffic in the memory system.  In the 128 x 16K
// layer-step 24 / 32 / 40 / 48 / 64 CTAs give 3040 / 3036 / 3066 / 2980 /
// 2787 layer-steps/s: 40 moves the units in time (266 us of a 326 us step)
// while slowing the attention least.  The caller may ask for another cap
// (GatherArgs::max_ctas), as the step does for a one-layer context.
constexpr int kGatherThreads = 128;
constexpr int kGatherCtas = 40;

// Copy item i of `pair` (one warp; skipped items and bad entries return).
__device__ __forceinline__ void gather_item(const GatherArgs& a, int pair, int i, int lane) {
  const long long it = static_cast<long long>(pair) * a.items + i;
  const int id = a.src_ids[it];
  if (id < 0) return;
  const int slot = a.dst_slots ? a.dst_slots[it] : i;
  const int unit = (slot >= 0 && slot < a.U) ? a.phys[static_cast<size_t>(pair) * a.U + slot] : -1;
  if (id >= a.NBmax) {
    if (lane == 0) raise_error(a.err, kErrBadBlock);
    return;
  }
  if (unit < 0 || unit >= a.U) {
    if (lane == 0) raise_error(a.err, kErrBadUnit);
    return;
  }
  const int src_slot = a.local_map ? a.local_map[static_cast<size_t>(pair) * a.NBmax + id] : id;
  if (src_slot < 0 || src_slot >= a.src_units) {
    if (lane == 0 && a.phase != 2) raise_error(a.err, kErrNotLocal);
    return;
  }
  if (a.phase != 0 && (a.phase == 1) == (src_slot >= a.base[pair])) return;
  const uint4* src = static_cast<const uint4*>(a.host) +
                     (static_cast<size_t>(pair) * a.src_units + src_slot) * (kUnitBytes / 16);
  uint4* dst = static_cast<uint4*>(a.pool) +
               (static_cast<size_t>(pair) * a.U + unit) * (kUnitBytes / 16);
  uint4 v[kUnitBytes / 16 / 32];
#pragma unroll
  for (int j = 0; j < kUnitBytes / 16 / 32; ++j) v[j] = __ldcs(src + j * 32 + lane);
#pragma unroll
  for (int j = 0; j < kUnitBytes / 16 / 32; ++j) dst[j * 32 + lane] = v[j];
}

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const GatherArgs a) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * (kGatherThreads / 32);
  const long long w0 = blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5);
  if (a.pair_major) {
    for (long long lp = w0; lp < a.pairs; lp += nwarps) {
      const int pair = a.pair0 + static_cast<int>(lp);
      const int n = a.n_valid ? min(a.n_valid[pair], a.items) : a.items;
      for (int i = 0; i < n; ++i) gather_item(a, pair, i, lane);
    }
    return;
  }
  const long long total = static_cast<long long>(a.pairs) * a.items;
  for (long long lt = w0; lt < total; lt += nwarps) {
    const int local = static_cast<int>(lt / a.items);
    const int i = static_cast<int>(lt - static_cast<long long>(local) * a.items);
    const int pair = a.pair0 + local;
    if (a.n_valid && i >= a.n_valid[pair]) continue;
    gather_item(a, pair, i, lane);
  }
}

// Remote tier slot assignment, one warp per pair: 32 items at a time, the
// blocks that need a slot found by ballot and numbered by their rank among
// them, so slots follow item order exactly as a sequential loop would give.
constexpr int kRemoteWarps = 4;

__global__ void __launch_bounds__(kRemoteWarps * 32) remote_assign_kernel(const RemoteArgs a) {
  const int lane = threadIdx.x & 31;
  const int local = blockIdx.x * kRemoteWarps + (threadIdx.x >> 5);
  if (local >= a.pairs) return;  // warp-uniform
  const int pair = a.pair0 + local;
  const size_t base_map = static_cast<size_t>(pair) * a.NBmax;
  int count = a.count[pair];
  if (lane == 0) a.base[pair] = count;
  int n = a.items;
  if (a.n_valid) n = min(max(a.n_valid[pair], 0), a.items);
  int nm = 0;
  for (int b = 0; b < n; b += 32) {
    const int i = b + lane;
    const int id = i < n ? a.ids[static_cast<size_t>(pair) * a.items + i] : -1;
    bool need = false;
    if (id >= a.NBmax) {
      raise_error(a.err, kErrBadBlock);
    } else if (id >= 0) {
      need = a.local_map[base_map + id] < 0;
    }
    const unsigned ball = __ballot_sync(0xffffffffu, need);
    const int rank = __popc(ball & ((1u << lane) - 1u));
    const int room = max(a.capacity - count, 0);
    if (need) {
      if (rank < room) {
        const int slot = count + rank;
        a.local_map[base_map + id] = slot;
        a.miss_ids[static_cast<size_t>(pair) * a.M + nm + rank] = id;
        a.miss_slots[static_cast<size_t>(pair) * a.M + nm + rank] = slot;
      } else {
        raise_error(a.err, kErrNotLocal);
      }
    }
    const int got = min(__popc(ball), room);
    count += got;
    nm += got;
  }
  if (lane == 0) {
    a.count[pair] = count;
    a.n_miss[pair] = nm;
  }
}

__global__ void init_tables_kernel(int32_t* phys, int32_t* stamps, int pairs, int K,
                                   int U) {
  const long long n = static_cast<long long>(pairs) * U;
  for (long long i = blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    phys[i] = static_cast<int32_t>(i % U);
  }
  if (!stamps) return;  // resume: the caller's stamps stay
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
// Min/max of one block's keys over its `valid` tokens by one warp: lanes
// 0-15 take even tokens, 16-31 odd tokens, 8 dims per lane; the min row is
// written by lanes 0-15 and the max row by lanes 16-31.
__device__ __forceinline__ void warp_block_summary(const uint4* keys, int valid, uint4* dst,
                                                   int lane) {
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
  dst[(lane >> 4) * (kHeadDim / 8) + dch] = outv;
}

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
    warp_block_summary(keys, valid, static_cast<uint4*>(a.summ) +
                                        static_cast<size_t>(it) * (kSummBytes / 16),
                       lane);
  }
}

// Blocks rewritten in the host store: one warp per listed (pair, block)
// rebuilds the block's summary and, when the block is resident in the given
// table, copies the new contents into its pool unit.
__global__ void refresh_kernel(const RefreshArgs a) {
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  const long long total = static_cast<long long>(a.R) * a.Hkv * a.max_ids;
  for (long long it = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); it < total;
       it += warps) {
    const int pair = static_cast<int>(it / a.max_ids);
    const int i = static_cast<int>(it - static_cast<long long>(pair) * a.max_ids);
    if (i >= a.n_ids[pair]) continue;
    const int b = a.ids[it];
    if (b < 0) continue;
    if (b >= a.NBmax) {
      if (lane == 0) raise_error(a.err, kErrBadBlock);
      continue;
    }
    const int r = pair / a.Hkv;
    const int valid = min(kBlock, a.ctx_len[r] - b * kBlock);
    const size_t blk = static_cast<size_t>(pair) * a.NBmax + b;
    const uint4* src = static_cast<const uint4*>(a.host) + blk * (kUnitBytes / 16);
    if (valid > 0)
      warp_block_summary(src, valid, static_cast<uint4*>(a.summ) + blk * (kSummBytes / 16), lane);
    int slot = -1;
    for (int s0 = 0; s0 < a.K && slot < 0; s0 += 32) {
      const int s = s0 + lane;
      const unsigned hit = __ballot_sync(0xffffffffu, s < a.K && a.res[static_cast<size_t>(pair) * a.K + s] == b);
      if (hit) slot = s0 + __ffs(hit) - 1;
    }
    if (slot < 0) continue;
    const int unit = a.phys[static_cast<size_t>(pair) * a.U + slot];
    if (unit < 0 || unit >= a.U) {
      if (lane == 0) raise_error(a.err, kErrBadUnit);
      continue;
    }
    uint4* dst = static_cast<uint4*>(a.pool) + (static_cast<size_t>(pair) * a.U + unit) * (kUnitBytes / 16);
    uint4 v[kUnitBytes / 16 / 32];
#pragma unroll
    for (int j = 0; j < kUnitBytes / 16 / 32; ++j) v[j] = src[j * 32 + lane];
#pragma unroll
    for (int j = 0; j < kUnitBytes / 16 / 32; ++j) dst[j * 32 + lane] = v[j];
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
  size_t unit_store = unit_host;
  if (a.local_map) {
    // The decode side's copy of block b: its local slot, or a fresh slot for
    // a block this token opens.  One warp per pair: no other writer.
    int slot = a.local_map[unit_host];
    if (slot < 0 && tk == 0) {
      const int c = a.local_count[pair];
      if (c < a.capacity) {
        slot = c;
        __syncwarp();
        if (lane == 0) {
          a.local_count[pair] = c + 1;
          a.local_map[unit_host] = c;
        }
      }
    }
    if (slot < 0) {
      if (lane == 0) raise_error(a.err, kErrNotLocal);
      return;
    }
    unit_store = static_cast<size_t>(pair) * a.capacity + slot;
  }
  uint4* hrow = static_cast<uint4*>(a.host) + unit_store * (kUnitBytes / 16) +
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
  if (a.pairs <= 0) return cudaSuccess;
  if (a.K <= 32) return launch_admit_kpl<1>(a, s);
  if (a.K <= 64) return launch_admit_kpl<2>(a, s);
  if (a.K <= 128) return launch_admit_kpl<4>(a, s);
  return launch_admit_kpl<8>(a, s);
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s) {
  const long long total = static_cast<long long>(a.pairs) * a.items;
  if (total == 0) return cudaSuccess;
  if (a.pair_major) {
    // One warp per pair, every pair in one pass (at most kPairMajorCtas CTAs).
    constexpr long long kPairMajorCtas = 1024;
    long long grid = (a.pairs + (kGatherThreads / 32) - 1) / (kGatherThreads / 32);
    if (grid > kPairMajorCtas) grid = kPairMajorCtas;
    gather_kernel<<<static_cast<int>(grid), kGatherThreads, 0, s>>>(a);
    return cudaGetLastError();
  }
  const long long warps_needed = total;
  long long grid = (warps_needed + (kGatherThreads / 32) - 1) / (kGatherThreads / 32);
  static const int forced = [] {
    // Tuning override of the gather's CTA count (units in flight / 4).
    const char* e = std::getenv("OASIS_GATHER_CTAS");
    const int v = e ? std::atoi(e) : 0;
    return v > 0 ? v : 0;
  }();
  const int cap = forced > 0 ? forced : a.max_ctas > 0 ? a.max_ctas : kGatherCtas;
  if (grid > cap) grid = cap;
  gather_kernel<<<static_cast<int>(grid), kGatherThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_remote_assign(const RemoteArgs& a, cudaStream_t s) {
  if (a.pairs <= 0) return cudaSuccess;
  remote_assign_kernel<<<(a.pairs + kRemoteWarps - 1) / kRemoteWarps, kRemoteWarps * 32, 0, s>>>(a);
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

cudaError_t launch_refresh(const RefreshArgs& a, cudaStream_t s) {
  const long long total = static_cast<long long>(a.R) * a.Hkv * a.max_ids;
  if (total == 0) return cudaSuccess;
  long long grid = (total + 7) / 8;
  if (grid > 8 * sm_count()) grid = 8 * sm_count();
  refresh_kernel<<<static_cast<int>(grid), 256, 0, s>>>(a);
  return cudaGetLastError();
}

__global__ void tail_blocks_kernel(const int32_t* ctx_len, int R, int Hkv, int32_t* tail) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= R * Hkv) return;
  const int c = ctx_len[p / Hkv];
  tail[p] = (c > 0 && c % kBlock != 0) ? c / kBlock : -1;
}

cudaError_t launch_tail_blocks(const int32_t* ctx_len, int R, int Hkv, int32_t* tail,
                               cudaStream_t s) {
  const int pairs = R * Hkv;
  if (pairs == 0) return cudaSuccess;
  tail_blocks_kernel<<<(pairs + 255) / 256, 256, 0, s>>>(ctx_len, R, Hkv, tail);
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

cudaError_t preload_support_kernels() {
  cudaFuncAttributes at;
  const void* fns[] = {
      reinterpret_cast<const void*>(admit_kernel<1>), reinterpret_cast<const void*>(admit_kernel<2>),
      reinterpret_cast<const void*>(admit_kernel<4>), reinterpret_cast<const void*>(admit_kernel<8>),
      reinterpret_cast<const void*>(gather_kernel),
      reinterpret_cast<const void*>(remote_assign_kernel),
      reinterpret_cast<const void*>(init_tables_kernel),
      reinterpret_cast<const void*>(summary_build_kernel),
      reinterpret_cast<const void*>(refresh_kernel), reinterpret_cast<const void*>(append_kernel),
      reinterpret_cast<const void*>(advance_kernel),
      reinterpret_cast<const void*>(tail_blocks_kernel)};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncGetAttributes(&at, f);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace oasis
