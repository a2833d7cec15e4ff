// scan.cu -- summary scan and head-wise top-K (steps a2 + a3) as one
// persistent, dynamically scheduled stream, with the capped eviction (a4)
// fused into the pair's selection.
//
// The draft query scores every logical block of its request from the
// per-block min/max key summaries and the blocks are ranked head-wise
// ("Pith review of OasisKV", section "What carries the argument": the draft
// query is scored against Quest-style per-block minima and maxima of the
// keys, and every logical block is ranked per KV head from those summaries
// alone).  Score of block b for KV head h, summed over the group's query
// heads j and the step's draft queries e:
//   s[b] = sum_e sum_j sum_i max(qd_eji * mn_bi, qd_eji * mx_bi)
//        = sum_i W+_i * mx_bi + W-_i * mn_bi,
// W+ = sum max(qd, 0), W- = sum min(qd, 0) (mn <= mx), one length-256 dot
// product per 512-byte summary row pair: the scan is a pure HBM stream.
//
// GB300 mapping.  The work is cut into items of item_blocks consecutive
// blocks of one (request, KV head) pair.  A grid of as many CTAs as fit on
// the GPU at once pulls items from a global atomic queue, so the stream has
// no wave boundaries and CTAs that start late (SMs still busy with other
// kernels) simply take fewer items.  Per CTA, a producer warp streams each
// item's summary rows through an NST-deep ring of 1-D bulk copies (4 blocks
// per consumer warp per stage, with the item's pair and block range beside
// each stage); CW consumer warps score 4 blocks each per stage (one 16-byte
// load per lane per block, packed fp32x2 multiply-adds, transposed shuffle
// reduction) and write the fp32 scores to a per-pair row of scratch (4 bytes
// per 512 read).  The CTA that finishes the last item of a pair (a counter
// per pair, release/acquire through fences) ranks that pair while the other
// CTAs keep streaming: its consumer warps read the pair's scores back from
// L2, each sorts KP = 32*KPL of them at a time with a warp bitonic network
// over 64-bit keys (order-preserving score bits above the complemented block
// id, so ties break to the lower id) folding them into a running top-KP, the
// warps' lists are merged in a tree, and warp 0 writes the top-K and, when
// fused, runs the pair's capped eviction.  Only the last pairs' rankings
// are left for the end of the kernel, instead of one ranking tail per CTA
// per wave.
#include <cstdlib>

#include "admit.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sortnet.cuh"

namespace oasis {
namespace {

constexpr int kItemStages = 8;   // stages per item: 8 x 32 blocks = 256 blocks (128 KiB)

// Shared memory: the ring, per-stage descriptors, the barriers, a broadcast
// word, and a region that holds either the warps' key lists (tree merge) or
// the fused admission's scratch.  Same arithmetic on host and device.
template <int KPL, int CW, int NST>
struct StreamLayout {
  static constexpr int KP = 32 * KPL;
  static constexpr int kChunk = 4 * CW;                     // blocks per stage
  static constexpr int kStageBytes = kChunk * kSummBytes;
  static constexpr int kRing = NST * kStageBytes;
  static constexpr int kMeta = kRing;                       // int4 per stage
  static constexpr int kBars = kMeta + NST * 16;            // full[NST], empty[NST], sync
  static constexpr int kFlag = kBars + (2 * NST + 1) * 8;
  static constexpr int kUnion = (kFlag + 16 + 127) / 128 * 128;
  __host__ __device__ static size_t union_bytes(int NBmax) {
    const size_t keys = static_cast<size_t>(CW) * KP * 8;
    const size_t adm = admit_warp_smem_bytes(NBmax);
    return keys > adm ? keys : adm;
  }
  __host__ __device__ static int total(int NBmax) {
    return static_cast<int>(kUnion + union_bytes(NBmax) + 128);
  }
};

constexpr int kFlagLast = 1;

template <int KPL, int CW, int NST>
__global__ void __launch_bounds__((CW + 1) * 32, NST >= 3 ? 3 : 4)
    scan_kernel(const ScoreArgs a) {
  using L = StreamLayout<KPL, CW, NST>;
  constexpr int KP = L::KP;
  constexpr int kChunk = L::kChunk;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  int4* meta = reinterpret_cast<int4*>(smem + L::kMeta);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* empty = full + NST;
  uint64_t* csync_bar = empty + NST;   // the consumer warps' own barrier
  int* flag_s = reinterpret_cast<int*>(smem + L::kFlag);
  uint8_t* uni = smem + L::kUnion;
  uint64_t* keybuf = reinterpret_cast<uint64_t*>(uni);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int item_blocks = kItemStages * kChunk;
  const int ipp = (a.NBmax + item_blocks - 1) / item_blocks;   // items per pair
  const int total_items = a.pairs * ipp;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], CW);
    }
    mbar_init(csync_bar, CW);
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == CW) {
    // ---------------- producer: pull items, stream their summary rows
    if (lane == 0) {
      int c = 0;
      bool ok = true;
      // Stage c: wait until its previous occupant has been consumed, publish
      // the descriptor, then the bytes (or a bare arrival for no bytes).
      auto emit = [&](int pair, int b0, int nblk, int flags) {
        const int st = c % NST;
        if (c >= NST) ok = mbar_wait(&empty[st], ((c / NST) - 1) & 1);
        if (!ok) return;
        meta[st] = make_int4(pair, b0, nblk, flags);
        const uint32_t bytes = static_cast<uint32_t>(nblk) * kSummBytes;
        mbar_arrive_expect_tx(&full[st], bytes);
        if (bytes) {
          const uint8_t* src = static_cast<const uint8_t*>(a.summ) +
                               (static_cast<size_t>(pair) * a.NBmax + b0) * kSummBytes;
          bulk_g2s(ring + st * L::kStageBytes, src, bytes, &full[st]);
        }
        ++c;
      };
      while (ok) {
        const int item = static_cast<int>(atomicAdd(&a.queue[0], 1u));
        if (item >= total_items) break;
        const int lp = item / ipp;
        const int it = item - lp * ipp;
        const int pair = a.pair0 + lp;
        const int r = pair / a.Hkv;
        const int ctx = a.ctx_len[r];
        int nb = ctx > 0 ? (ctx + kBlock - 1) / kBlock : 0;
        if (nb > a.NBmax) {
          raise_error(a.err, kErrBadBlock);
          nb = a.NBmax;
        }
        const int b1 = min(it * item_blocks + item_blocks, nb);
        int b0 = it * item_blocks;
        if (b0 >= b1) {
          emit(pair, b0, 0, kFlagLast);   // nothing to read: completion only
          continue;
        }
        for (; b0 < b1 && ok; b0 += kChunk) {
          const int nblk = min(kChunk, b1 - b0);
          emit(pair, b0, nblk, b0 + kChunk >= b1 ? kFlagLast : 0);
        }
      }
      if (ok) emit(-1, 0, 0, 0);          // end of the stream for the consumers
      if (!ok) raise_error(a.err, kErrTimeout);
      // Drain: the latest phase issued on each stage must have landed before
      // the CTA may exit (a no-op on the normal path).
      for (int cc = max(0, c - NST); cc < c; ++cc)
        (void)mbar_wait(&full[cc % NST], (cc / NST) & 1);
    }
    __syncwarp();
  } else {
    // ---------------- consumers
    const int row = lane >> 4;            // lanes 0-15: min row, 16-31: max row
    const int d0 = (lane & 15) * 8;
    const size_t plane = static_cast<size_t>(a.R) * a.Hq * kHeadDim;
    uint64_t w2[4] = {0ull, 0ull, 0ull, 0ull};
    int cur_pair = -1;
    bool ok = true;
    // Barrier of the CW consumer warps (the producer does not take part),
    // with a bounded wait: if one warp has left the loop on a failed wait,
    // the others fail here too instead of waiting for it.  Each warp counts
    // the phases it has passed; all pass the same sequence of barriers.
    uint32_t sync_phase = 0;
    auto csync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(csync_bar);
      const bool done = __all_sync(0xffffffffu, mbar_wait(csync_bar, sync_phase & 1u));
      ++sync_phase;
      return done;
    };
    for (int c = 0;; ++c) {
      const int st = c % NST;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (c / NST) & 1));
      if (!ok) break;
      const int4 m = meta[st];
      const int pair = m.x;
      if (pair < 0) break;
      if (pair != cur_pair) {
        // The pair's weights: every draft plane's group vectors folded into
        // W- (min row) and W+ (max row), 8 dims per lane.
        const int r = pair / a.Hkv, h = pair - r * a.Hkv;
        float w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0.f;
        for (int e = 0; e < a.D; ++e) {
          const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.qd) + e * plane +
                                    (static_cast<size_t>(r) * a.Hq + h * a.G) * kHeadDim + d0;
          for (int gi = 0; gi < a.G; ++gi) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(qg + gi * kHeadDim));
            const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float lo = bf16lo(wd[i]), hi = bf16hi(wd[i]);
              w[2 * i] += row ? fmaxf(lo, 0.f) : fminf(lo, 0.f);
              w[2 * i + 1] += row ? fmaxf(hi, 0.f) : fminf(hi, 0.f);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) w2[i] = f2pack(w[2 * i], w[2 * i + 1]);
        cur_pair = pair;
      }
      const int nblk = m.z;
      const uint8_t* stage = ring + st * L::kStageBytes;
      float v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = warp * 4 + q;
        float acc = 0.f;
        if (j < nblk) {
          const uint4 u = *reinterpret_cast<const uint4*>(stage + j * kSummBytes + lane * 16);
          uint64_t acc2 = 0ull;
          acc2 = ffma2(w2[0], f2pack(bf16lo(u.x), bf16hi(u.x)), acc2);
          acc2 = ffma2(w2[1], f2pack(bf16lo(u.y), bf16hi(u.y)), acc2);
          acc2 = ffma2(w2[2], f2pack(bf16lo(u.z), bf16hi(u.z)), acc2);
          acc2 = ffma2(w2[3], f2pack(bf16lo(u.w), bf16hi(u.w)), acc2);
          acc = f2sum(acc2);
        }
        v[q] = acc;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      // Transposed reduction of 4 values over 32 lanes: 6 shuffles; lane
      // 8q' then holds block warp*4 + q' with q' = (lane>>4)*2 + ((lane>>3)&1).
      const bool b4 = lane & 16, b3 = lane & 8;
      float k0 = b4 ? v[2] : v[0], k1 = b4 ? v[3] : v[1];
      const float s0 = b4 ? v[0] : v[2], s1 = b4 ? v[1] : v[3];
      k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
      k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
      float x = b3 ? k1 : k0;
      x += __shfl_xor_sync(0xffffffffu, b3 ? k0 : k1, 8);
      x += __shfl_xor_sync(0xffffffffu, x, 4);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      const int q = ((lane >> 4) << 1) | ((lane >> 3) & 1);
      if ((lane & 7) == 0 && warp * 4 + q < nblk)
        a.scores_ws[static_cast<size_t>(pair) * a.NBmax + m.y + warp * 4 + q] = x;

      if (!(m.w & kFlagLast)) continue;
      // ---- end of an item: publish its scores, count it for the pair
      __threadfence();
      if (!(ok = csync())) break;
      if (threadIdx.x == 0) {
        const int old = atomicAdd(&a.done[pair], 1);
        const int last = old == ipp - 1;
        if (last) {
          a.done[pair] = 0;
          __threadfence();   // acquire side: the other CTAs' scores are visible
        }
        *flag_s = last;
      }
      if (!(ok = csync())) break;
      if (!*flag_s) continue;

      // ---- this CTA ranks the pair: fold KP scores at a time per warp
      const int r = pair / a.Hkv;
      const int ctx = a.ctx_len[r];
      int nb = ctx > 0 ? (ctx + kBlock - 1) / kBlock : 0;
      if (nb > a.NBmax) nb = a.NBmax;
      const float* sp = a.scores_ws + static_cast<size_t>(pair) * a.NBmax;
      uint64_t top[KPL];
#pragma unroll
      for (int i = 0; i < KPL; ++i) top[i] = 0ull;
      bool have_top = false;
      for (int base = warp * KP; base < nb; base += CW * KP) {
        uint64_t nk[KPL];
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
          const int e = base + i * 32 + lane;
          nk[i] = e < nb ? (static_cast<uint64_t>(float_key(__ldcg(sp + e))) << 32) |
                               static_cast<uint32_t>(~e)
                         : 0ull;
        }
        if (have_top) {
          bitonic_sort<KPL>(nk, false);
          merge_top<KPL>(top, nk);
        } else {
          bitonic_sort<KPL>(nk, true);
#pragma unroll
          for (int i = 0; i < KPL; ++i) top[i] = nk[i];
          have_top = true;
        }
      }
      // tree merge of the consumer warps' lists
#pragma unroll 1
      for (int sz = 1; sz < CW && ok; sz <<= 1) {
        if (!(ok = csync())) break;
        if ((warp % (2 * sz)) == sz) {
#pragma unroll
          for (int i = 0; i < KPL; ++i) keybuf[warp * KP + i * 32 + lane] = top[i];
        }
        if (!(ok = csync())) break;
        if ((warp % (2 * sz)) == 0) {
          const uint64_t* p = keybuf + (warp + sz) * KP;
          uint64_t nk[KPL];
#pragma unroll
          for (int i = 0; i < KPL; ++i) nk[i] = p[KP - 1 - (i * 32 + lane)];
          merge_top<KPL>(top, nk);
        }
      }
      if (!ok) break;
      if (warp == 0) {
        // The key lists are no longer read: the region takes the admission.
        AdmitWarpSmem& S = *reinterpret_cast<AdmitWarpSmem*>(uni);
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
          const int e = i * 32 + lane;
          if (e < a.K) {
            const uint64_t key = top[i];
            const int id = key == 0ull ? -1 : static_cast<int>(~static_cast<uint32_t>(key));
            a.topk_ids[static_cast<size_t>(pair) * a.K + e] = id;
            if (a.topk_scores)
              a.topk_scores[static_cast<size_t>(pair) * a.K + e] =
                  key == 0ull ? -INFINITY : key_float(static_cast<uint32_t>(key >> 32));
            S.topk[e] = id;
          }
        }
        if (a.fuse_admit) {
          __syncwarp();
          admit_warp<KPL>(a.admit, pair, S,
                          reinterpret_cast<uint32_t*>(uni + sizeof(AdmitWarpSmem)));
        }
      }
    }
    if (!ok && lane == 0) raise_error(a.err, kErrTimeout);
  }

  // ---------------- the last CTA to leave resets the queue and the counters
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&a.queue[1], 1u);
    if (old == gridDim.x - 1) {
      for (int p = 0; p < a.pairs; ++p) a.done[a.pair0 + p] = 0;
      a.queue[0] = 0u;
      a.queue[1] = 0u;
      __threadfence();
    }
  }
}

template <int KPL, int CW, int NST>
cudaError_t configure(int smem) {
  static int configured_device = -1;
  static int configured_smem = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev || smem > configured_smem) {
    e = cudaFuncSetAttribute(scan_kernel<KPL, CW, NST>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
    configured_smem = smem;
  }
  return cudaSuccess;
}

// CTAs of the kernel resident on the whole GPU at once (cached per device
// and NBmax).
template <int KPL, int CW, int NST>
int resident_ctas(int NBmax) {
  static int cached_dev = -1, cached_nb = -1, cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev == cached_dev && NBmax == cached_nb) return cached;
  const int smem = StreamLayout<KPL, CW, NST>::total(NBmax);
  int sms = 0, per = 0;
  if (configure<KPL, CW, NST>(smem) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, scan_kernel<KPL, CW, NST>,
                                                    (CW + 1) * 32, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cached_dev = dev;
  cached_nb = NBmax;
  cached = per * sms;
  return cached;
}

template <int KPL, int CW, int NST>
cudaError_t launch_stream(const ScoreArgs& a, cudaStream_t s) {
  using L = StreamLayout<KPL, CW, NST>;
  const int smem = L::total(a.NBmax);
  cudaError_t e = configure<KPL, CW, NST>(smem);
  if (e != cudaSuccess) return e;
  const int item_blocks = kItemStages * L::kChunk;
  const long long items =
      static_cast<long long>(a.pairs) * ((a.NBmax + item_blocks - 1) / item_blocks);
  int grid = resident_ctas<KPL, CW, NST>(a.NBmax);
  if (grid <= 0) grid = 152;
  if (items < grid) grid = static_cast<int>(items);
  scan_kernel<KPL, CW, NST><<<grid, (CW + 1) * 32, smem, s>>>(a);
  return cudaGetLastError();
}

// Ring depth: 2 stages of 16 KiB (4 CTAs per SM) unless OASIS_SCAN_STAGES=3
// asks for 3 (48 KiB in flight per CTA, 3 CTAs per SM).
int ring_stages() {
  static const int v = [] {
    const char* e = std::getenv("OASIS_SCAN_STAGES");
    return (e && std::atoi(e) == 3) ? 3 : 2;
  }();
  return v;
}

template <int KPL>
cudaError_t launch_kpl(const ScoreArgs& a, cudaStream_t s) {
  return ring_stages() == 3 ? launch_stream<KPL, 8, 3>(a, s) : launch_stream<KPL, 8, 2>(a, s);
}

}  // namespace

cudaError_t launch_scan_stream(const ScoreArgs& a, cudaStream_t s) {
  if (a.pairs <= 0) return cudaSuccess;
  if (a.K <= 32) return launch_kpl<1>(a, s);
  if (a.K <= 64) return launch_kpl<2>(a, s);
  if (a.K <= 128) return launch_kpl<4>(a, s);
  return launch_kpl<8>(a, s);
}

cudaError_t preload_stream_kernels() {
  cudaFuncAttributes at;
  const void* fns[] = {reinterpret_cast<const void*>(scan_kernel<1, 8, 2>),
                       reinterpret_cast<const void*>(scan_kernel<2, 8, 2>),
                       reinterpret_cast<const void*>(scan_kernel<4, 8, 2>),
                       reinterpret_cast<const void*>(scan_kernel<8, 8, 2>),
                       reinterpret_cast<const void*>(scan_kernel<1, 8, 3>),
                       reinterpret_cast<const void*>(scan_kernel<2, 8, 3>),
                       reinterpret_cast<const void*>(scan_kernel<4, 8, 3>),
                       reinterpret_cast<const void*>(scan_kernel<8, 8, 3>)};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncGetAttributes(&at, f);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace oasis
