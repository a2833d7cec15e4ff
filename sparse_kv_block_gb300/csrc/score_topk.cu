// score_topk.cu -- summary scan and head-wise top-K (steps a2 + a3).
//
// The draft query scores every logical block of its request from the
// per-block min/max key summaries and the blocks are ranked head-wise
// ("Pith review of OasisKV", section "What carries the argument": the draft
// query is scored against Quest-style per-block minima and maxima of the
// keys, and every logical block is ranked per KV head from those summaries
// alone; the full keys are never read).
//
// Score of block b for KV head h (group = the G query heads of h; with D
// draft queries per step, every draft's G vectors count as group members):
//   s[b] = sum_e sum_j sum_i max(qd_eji * mn_bi, qd_eji * mx_bi).
// Because mn <= mx, max(x*mn, x*mx) = max(x,0)*mx + min(x,0)*mn, so the sum
// over the group (and the drafts) folds into one dot product of length 2d
// with the weights W+ = sum_j max(qd_j, 0) (on the max row) and
// W- = sum_j min(qd_j, 0) (on the min row): more drafts cost no scan time.
// Each block then costs 256 multiply-adds on 512 bytes: the scan is a pure
// HBM stream.
//
// GB300 mapping.  One CTA per (request, KV head): a producer warp streams the
// request's contiguous summary rows through a 2-deep ring of stages (4
// blocks per consumer warp, 2 KiB) with 1-D bulk copies; CW consumer warps
// each score 4 blocks per stage (one 16-byte load per lane per block, packed
// fp32x2 multiply-adds, transposed shuffle reduction), keep a running top-KP
// list in registers (each filled buffer of KP keys bitonic-sorted, then
// merged in; with CW = 8 every 32-key run of a buffer is sorted as soon as
// it exists, while the stream runs), and finally merge their lists in a
// tree.  Shared memory is sized from the actual NBmax (the fused admission
// reuses the ring).  Two variants: CW = 8 (16 KiB stages, ~41 KB, 4 CTAs per
// SM) and CW = 4 (8 KiB stages, ~21 KB and 48 registers per thread, 8 CTAs
// per SM); the launcher picks one by wave quantisation (see scan_warps).
// Alone on the 128 x 16K layer CW = 4 is faster (92.5 vs 95 us) but inside
// the step, beside the host-link gather, CW = 8 is (118-120 vs 129 us).
// Keys are 64-bit: order-preserving score bits above the complemented block
// id, so ties break to the lower id and all keys are distinct.
#include <cstdlib>
#include <string>

#include "admit.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sortnet.cuh"

namespace oasis {
namespace {

constexpr int kStages = 2;                   // ring depth

// The pair's scan weights, 8 dims per lane: lanes 0-15 hold W- (min row),
// 16-31 W+ (max row); every draft plane adds its group's vectors to them.
// As fp32 pairs for the packed fp32x2 multiply-add.
__device__ __forceinline__ void pair_weights(const ScoreArgs& a, int r, int h, int lane,
                                             uint64_t (&w2)[4]) {
  const int row = lane >> 4;
  const int d0 = (lane & 15) * 8;
  float w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = 0.f;
  const size_t plane = static_cast<size_t>(a.R) * a.Hq * kHeadDim;
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
}

// Partial scores (per lane) of this warp's 4 blocks of a staged chunk: one
// 16-byte load per lane per block; blocks j >= nblk give 0.
__device__ __forceinline__ void stage_partials(const uint8_t* stage, int warp, int lane,
                                               int nblk, const uint64_t (&w2)[4],
                                               float (&v)[4]) {
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
}

// Transposed reduction of the 4 partials over 32 lanes (6 shuffles): lane
// 8q' returns the score of block warp*4 + q' with
// q' = (lane>>4)*2 + ((lane>>3)&1).
__device__ __forceinline__ float reduce4(const float (&v)[4], int lane) {
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
  return x;
}

// Producer of one pair's summary rows: chunk c of kChunk blocks into stage
// c % kStages of the ring, after the stage's previous chunk was consumed
// (kCW arrivals on empty).  Returns false if a wait ran out; drains its own
// copies before returning either way.
template <int kChunk>
__device__ bool produce_pair(const uint8_t* src, int nb, uint8_t* ring, uint64_t* full,
                             uint64_t* empty, long long limit) {
  constexpr int kChunkBytes = kChunk * kSummBytes;
  const int nchunks = (nb + kChunk - 1) / kChunk;
  int c = 0;
  bool ok = true;
  for (; c < nchunks && ok; ++c) {
    const int st = c % kStages;
    if (c >= kStages) ok = mbar_wait(&empty[st], ((c / kStages) - 1) & 1, limit);
    if (!ok) break;
    const int nblk = min(kChunk, nb - c * kChunk);
    const uint32_t bytes = static_cast<uint32_t>(nblk) * kSummBytes;
    mbar_arrive_expect_tx(&full[st], bytes);
    bulk_g2s(ring + st * kChunkBytes, src + static_cast<size_t>(c) * kChunkBytes, bytes,
             &full[st]);
  }
  // Drain: the latest phase issued on each stage must have landed before
  // the CTA may exit (a no-op on the normal path).
  for (int cc = max(0, c - kStages); cc < c; ++cc)
    (void)mbar_wait(&full[cc % kStages], (cc / kStages) & 1);
  return ok;
}

// Shared memory: the ring of kStages stages (reused by the fused admission
// once every stage has been consumed, so at least the admission's scratch
// for this NBmax), the stage barriers, and the per-warp key buffers.  The
// same arithmetic runs on the host (launch size) and in the kernel.
template <int KPL, int CW>
struct Layout {
  static constexpr int KP = 32 * KPL;
  static constexpr int kChunk = 4 * CW;                    // blocks per stage
  static constexpr int kChunkBytes = kChunk * kSummBytes;  // 2 KiB per warp
  __host__ __device__ static int bars(int NBmax) {
    const size_t ring = static_cast<size_t>(kStages) * kChunkBytes;
    const size_t adm = admit_warp_smem_bytes(NBmax);
    return static_cast<int>(((ring > adm ? ring : adm) + 127) / 128 * 128);
  }
  __host__ __device__ static int keys(int NBmax) { return bars(NBmax) + 64; }  // [CW][KP] u64
  __host__ __device__ static int total(int NBmax) { return keys(NBmax) + CW * KP * 8 + 128; }
};

// The launch bounds pin the occupancy the 8-warp variants are sized for: 4
// CTAs per SM (K <= 128) and 3 (K > 128); the 4-warp variants reach 8 and 5
// unbounded.
template <int KPL, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, CW == 4 ? 0 : (KPL <= 4 ? 4 : 3))
    score_topk_kernel(const ScoreArgs a) {
  using L = Layout<KPL, CW>;
  constexpr int KP = L::KP;
  constexpr int kCW = CW;
  constexpr int kChunk = L::kChunk;
  constexpr int kChunkBytes = L::kChunkBytes;
  constexpr bool kRunsEarly = CW == 8;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bars(a.NBmax));
  uint64_t* empty = full + kStages;
  uint64_t* keybuf = reinterpret_cast<uint64_t*>(smem + L::keys(a.NBmax));

  const int pair = a.pair0 + blockIdx.x;
  const int r = pair / a.Hkv;
  const int h = pair - r * a.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ctx = a.ctx_len[r];
  int nb = ctx > 0 ? (ctx + kBlock - 1) / kBlock : 0;
  if (nb > a.NBmax) {
    if (threadIdx.x == 0) raise_error(a.err, kErrBadBlock);
    nb = a.NBmax;
  }
  const int nchunks = (nb + kChunk - 1) / kChunk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCW);
    }
    fence_barrier_init();
  }
  __syncthreads();

  uint64_t top[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) top[i] = 0ull;

  if (warp == kCW) {
    // ---------------- producer: stream this (r, h)'s summary rows
    if (lane == 0) {
      const uint8_t* src = static_cast<const uint8_t*>(a.summ) +
                           static_cast<size_t>(pair) * a.NBmax * kSummBytes;
      int c = 0;
      bool ok = true;
      for (; c < nchunks && ok; ++c) {
        const int st = c % kStages;
        if (c >= kStages) ok = mbar_wait(&empty[st], ((c / kStages) - 1) & 1, a.wait_limit);
        if (!ok) break;
        const int nblk = min(kChunk, nb - c * kChunk);
        const uint32_t bytes = static_cast<uint32_t>(nblk) * kSummBytes;
        mbar_arrive_expect_tx(&full[st], bytes);
        bulk_g2s(ring + st * kChunkBytes,
                 src + static_cast<size_t>(c) * kChunkBytes, bytes, &full[st]);
      }
      if (!ok) raise_error(a.err, kErrTimeout);
      // Drain: the latest phase issued on each stage must have landed before
      // the CTA may exit (a no-op on the normal path).
      for (int cc = max(0, c - kStages); cc < c; ++cc)
        (void)mbar_wait(&full[cc % kStages], (cc / kStages) & 1);
    }
    __syncwarp();
  } else {
    // ---------------- consumers: score, then keep a running top-KP
    // Lane weights: lanes 0-15 cover the min row, 16-31 the max row, 8 dims each.
    const int row = lane >> 4;
    const int d0 = (lane & 15) * 8;
    float w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0.f;
    // Every draft plane adds its group's vectors to the same two weights.
    const size_t plane = static_cast<size_t>(a.R) * a.Hq * kHeadDim;
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
    // Weights as fp32 pairs for the packed fp32x2 multiply-add.
    uint64_t w2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w2[i] = f2pack(w[2 * i], w[2 * i + 1]);
    uint64_t* mybuf = keybuf + warp * KP;
    int cnt = 0;
    bool have_top = false;  // false while `top` still holds only empty keys
    // The buffer's keys as sorted 32-key runs (run i = keys i*32 .. i*32+31),
    // nrun of them complete.  With 8 consumer warps each run is sorted as
    // soon as its 32 keys exist (the sorts then overlap the stream: 94.2
    // against 97.9 us alone on 1024 pairs); with 4, whose warps each see
    // twice the keys, the whole buffer is sorted when full (92.5 against
    // 96.9 us the other way).
    uint64_t run[KPL];
    int nrun = 0;
    // Run i of a buffer sorted in the direction the bitonic network over the
    // whole buffer gives it (descending for even i when the buffer is sorted
    // descending), so finishing the network needs only the merges of size
    // 64 and up.
    auto sort_run = [&](uint64_t& x, int i, bool desc) {
      uint64_t one[1] = {x};
      bitonic_sort<1>(one, ((i & 1) == 0) == desc);
      x = one[0];
    };
    // A full (or final, zero-padded) unsorted buffer: sort it and fold it
    // into `top` (the first buffer becomes `top`, later ones are merged).
    auto fold_buffer = [&](uint64_t(&nk)[KPL]) {
      if (have_top) {
        bitonic_sort<KPL>(nk, false);
        merge_top<KPL>(top, nk);
      } else {
        bitonic_sort<KPL>(nk, true);
#pragma unroll
        for (int i = 0; i < KPL; ++i) top[i] = nk[i];
        have_top = true;
      }
    };
    // The same for a buffer already held as sorted runs: finish its network.
    auto finish_buffer = [&]() {
      if (have_top) {
        bitonic_finish<KPL>(run, false);
        merge_top<KPL>(top, run);
      } else {
        bitonic_finish<KPL>(run, true);
#pragma unroll
        for (int i = 0; i < KPL; ++i) top[i] = run[i];
        have_top = true;
      }
    };
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int st = c % kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (c / kStages) & 1, a.wait_limit));
      if (!ok) break;
      const int nblk = min(kChunk, nb - c * kChunk);
      const uint8_t* stage = ring + st * kChunkBytes;
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
      // Transposed reduction of 4 values over 32 lanes: 6 shuffles.
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
      // lane 8q' holds block warp*4 + q' with q' = (lane>>4)*2 + ((lane>>3)&1)
      const int q = ((lane >> 4) << 1) | ((lane >> 3) & 1);
      const int nv = max(0, min(4, nblk - warp * 4));
      if ((lane & 7) == 0 && q < nv) {
        const uint32_t b = static_cast<uint32_t>(c * kChunk + warp * 4 + q);
        mybuf[cnt + q] = (static_cast<uint64_t>(float_key(x)) << 32) | (~b);
      }
      cnt += nv;
      if constexpr (kRunsEarly) {
        // Every 32 keys are sorted as soon as they exist, while the stream
        // still runs, into the run their place in the buffer's bitonic
        // network calls for; a full buffer then needs only the network's
        // last merges.
        if (cnt >= 32 * (nrun + 1)) {
          __syncwarp();
          uint64_t x = mybuf[nrun * 32 + lane];
          __syncwarp();
          sort_run(x, nrun, !have_top);
#pragma unroll
          for (int i = 0; i < KPL; ++i)
            if (i == nrun) run[i] = x;
          ++nrun;
        }
        if (nrun == KPL) {
          finish_buffer();
          cnt = 0;
          nrun = 0;
        }
      } else if (cnt == KP) {
        __syncwarp();
        uint64_t nk[KPL];
#pragma unroll
        for (int i = 0; i < KPL; ++i) nk[i] = mybuf[i * 32 + lane];
        __syncwarp();
        fold_buffer(nk);
        cnt = 0;
      }
    }
    if (!ok && lane == 0) raise_error(a.err, kErrTimeout);
    if (cnt > 0) {
      if constexpr (kRunsEarly) {
        // The runs not sorted yet (zero keys pad the partial one), then the
        // rest of the network.
        __syncwarp();
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
          if (i >= nrun) {
            const int e = i * 32 + lane;
            run[i] = e < cnt ? mybuf[e] : 0ull;
            sort_run(run[i], i, !have_top);
          }
        }
        __syncwarp();
        finish_buffer();
      } else {
        __syncwarp();
        uint64_t nk[KPL];
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
          const int e = i * 32 + lane;
          nk[i] = e < cnt ? mybuf[e] : 0ull;
        }
        __syncwarp();
        fold_buffer(nk);
      }
    }
  }

  // ---------------- tree merge of the consumer warps' lists
#pragma unroll 1
  for (int sz = 1; sz < kCW; sz <<= 1) {
    __syncthreads();
    if (warp < kCW && (warp % (2 * sz)) == sz) {
#pragma unroll
      for (int i = 0; i < KPL; ++i) keybuf[warp * KP + i * 32 + lane] = top[i];
    }
    __syncthreads();
    if (warp < kCW && (warp % (2 * sz)) == 0) {
      const uint64_t* p = keybuf + (warp + sz) * KP;
      uint64_t nk[KPL];
#pragma unroll
      for (int i = 0; i < KPL; ++i) nk[i] = p[KP - 1 - (i * 32 + lane)];
      merge_top<KPL>(top, nk);
    }
  }

  if (warp == 0) {
    // The ring is idle now (every bulk copy has landed and been consumed).
    AdmitWarpSmem& S = *reinterpret_cast<AdmitWarpSmem*>(ring);
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
                      reinterpret_cast<uint32_t*>(ring + sizeof(AdmitWarpSmem)));
    }
  }
}

// ------------------------------------------------------------ split scan
// Step a2 alone: one CTA per (request, KV head) streams the pair's summary
// rows through the same producer and ring as the fused kernel and writes
// every block's fp32 score to scores_ws[pair][b] (4 bytes per 512 read).
// Nothing is ranked here, so each CTA ends with its stream: no sort or merge
// tail holds its slot while HBM idles.
template <int CW>
__global__ void __launch_bounds__((CW + 1) * 32, CW == 4 ? 0 : 4)
    scan_kernel(const ScoreArgs a) {
  constexpr int kChunk = 4 * CW;
  constexpr int kChunkBytes = kChunk * kSummBytes;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kChunkBytes);
  uint64_t* empty = full + kStages;

  const int pair = a.pair0 + blockIdx.x;
  const int r = pair / a.Hkv;
  const int h = pair - r * a.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ctx = a.ctx_len[r];
  int nb = ctx > 0 ? (ctx + kBlock - 1) / kBlock : 0;
  if (nb > a.NBmax) {
    if (threadIdx.x == 0) raise_error(a.err, kErrBadBlock);
    nb = a.NBmax;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], CW);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == CW) {
    const uint8_t* src = static_cast<const uint8_t*>(a.summ) +
                         static_cast<size_t>(pair) * a.NBmax * kSummBytes;
    if (lane == 0 && !produce_pair<kChunk>(src, nb, ring, full, empty, a.wait_limit))
      raise_error(a.err, kErrTimeout);
    return;  // no block barrier follows
  }
  uint64_t w2[4];
  pair_weights(a, r, h, lane, w2);
  float* out = a.scores_ws + static_cast<size_t>(pair) * a.NBmax;
  const int nchunks = (nb + kChunk - 1) / kChunk;
  const int q = ((lane >> 4) << 1) | ((lane >> 3) & 1);
  for (int c = 0; c < nchunks; ++c) {
    const int st = c % kStages;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (c / kStages) & 1, a.wait_limit))) {
      if (lane == 0) raise_error(a.err, kErrTimeout);
      break;
    }
    const int nblk = min(kChunk, nb - c * kChunk);
    float v[4];
    stage_partials(ring + st * kChunkBytes, warp, lane, nblk, w2, v);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    const float x = reduce4(v, lane);
    if ((lane & 7) == 0 && warp * 4 + q < nblk) out[c * kChunk + warp * 4 + q] = x;
  }
}

// Steps a3 (and a4 when fused) of the split scan: one CTA of kSelThreads
// threads per pair ranks the pair's block scores (written by scan_kernel
// just before).  A block's rank key is its order-preserving score bits
// (larger is better); equal scores rank the lower block id first.  A radix
// selection finds the K-th largest score key, most significant digit first:
// the first digit starts at the highest bit on which the pair's keys differ
// (the bits above it are shared by all of them), and each pass builds a
// 256-bin histogram of the next (up to) 8 bits over the keys that still
// match the prefix chosen so far and picks the bin that holds the K-th key,
// until that bin holds exactly the keys still wanted.  Every key above the
// final prefix, and every key in its bin, is in the top-K; if after the last
// bit more keys share the K-th score than are wanted, the lowest block ids
// among them are taken (ranked in block-id order).  The winners (score key
// above the complemented block id) are sorted by a bitonic network spread
// over the CTA's warps (shuffles within a warp, shared memory across warps)
// and written, and warp 0 then runs the pair's capped eviction.  Each thread
// holds NPT keys in registers (kSelThreads * NPT >= NBmax); with NPT = 0
// every pass reads the scores again, from a copy in shared memory up to
// kSelStageMax blocks, else from global memory.
constexpr int kSelThreads = 128;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelStageMax = 8192;

__host__ __device__ inline bool select_stages(int NBmax) {
  return NBmax > kSelThreads * 8 && NBmax <= kSelStageMax;
}

template <int KPL>
__host__ __device__ inline size_t select_smem_bytes(int NBmax) {
  // histogram, control words, winners, staged scores; the admission's
  // scratch reuses the region once the winners are sorted
  const size_t rank = 1024 + 64 + static_cast<size_t>(32) * KPL * 8 +
                      (select_stages(NBmax) ? static_cast<size_t>(NBmax) * 4 : 0);
  const size_t adm = admit_warp_smem_bytes(NBmax);
  return ((rank > adm ? rank : adm) + 15) & ~static_cast<size_t>(15);
}

template <int KPL, int NPT>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const ScoreArgs a) {
  constexpr int P = 32 * KPL;                        // sorted list length (>= K)
  constexpr int kHeld = P > kSelThreads ? P / kSelThreads : 1;
  constexpr int kRegs = NPT > 0 ? NPT : 1;
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);           // [256]
  int* ctl = reinterpret_cast<int*>(smem + 1024);               // [16]
  uint64_t* buf = reinterpret_cast<uint64_t*>(smem + 1024 + 64);  // [P]
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const unsigned lt = (1u << lane) - 1u;
  const int pair = a.pair0 + blockIdx.x;
  const int r = pair / a.Hkv;
  const int ctx = a.ctx_len[r];
  int nb = ctx > 0 ? (ctx + kBlock - 1) / kBlock : 0;
  if (nb > a.NBmax) nb = a.NBmax;  // reported by the scan
  const float* sp = a.scores_ws + static_cast<size_t>(pair) * a.NBmax;

  uint32_t ureg[kRegs];
  if constexpr (NPT > 0) {
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int e = j * kSelThreads + tid;
      ureg[j] = e < nb ? float_key(sp[e]) : 0u;
    }
  } else if (select_stages(a.NBmax)) {
    float* staged = reinterpret_cast<float*>(smem + 1024 + 64 + P * 8);
    for (int e = tid; e < nb; e += kSelThreads) staged[e] = sp[e];
    __syncthreads();
    sp = staged;
  }
  // f(score key, block id, valid) for slot j of every thread, j ascending:
  // the same trip count in every thread (barriers may sit inside f).
  const int nslots = (nb + kSelThreads - 1) / kSelThreads;
  auto for_each_slot = [&](auto&& f) {
    if constexpr (NPT > 0) {
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int e = j * kSelThreads + tid;
        f(ureg[j], e, e < nb);
      }
    } else {
      for (int j = 0; j < nslots; ++j) {
        const int e = j * kSelThreads + tid;
        f(e < nb ? float_key(sp[e]) : 0u, e, e < nb);
      }
    }
  };

  // ---- the bits every key shares, then radix passes below them
  uint32_t any = 0u, all = ~0u;
  for_each_slot([&](uint32_t u, int, bool v) {
    if (v) {
      any |= u;
      all &= u;
    }
  });
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    any |= __shfl_xor_sync(0xffffffffu, any, off);
    all &= __shfl_xor_sync(0xffffffffu, all, off);
  }
  if (lane == 0) {
    ctl[8 + warp] = static_cast<int>(any);
    ctl[12 + warp] = static_cast<int>(all);
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    any |= static_cast<uint32_t>(ctl[8 + w]);
    all &= static_cast<uint32_t>(ctl[12 + w]);
  }
  const uint32_t diff = any ^ all;
  const int hb = diff ? 31 - __clz(diff) : -1;   // -1: every key equal
  uint32_t mask = hb < 0 ? ~0u : (hb >= 31 ? 0u : ~((2u << hb) - 1u));
  uint32_t prefix = all & mask;
  int need = min(a.K, nb);
  int in_bin = nb;   // keys matching the prefix
  if (need > 0 && need < nb) {
    for (int hi = hb; hi >= 0 && in_bin != need;) {
      const int lo = hi >= 7 ? hi - 7 : 0;
      const uint32_t dmask = (2u << (hi - lo)) - 1u;
      hist[tid] = 0u;
      hist[tid + kSelThreads] = 0u;
      __syncthreads();
      for_each_slot([&](uint32_t u, int, bool v) {
        if (v && (u & mask) == prefix) atomicAdd(&hist[(u >> lo) & dmask], 1u);
      });
      __syncthreads();
      if (warp == 0) {
        // Lane l owns bins 8l .. 8l+7: keys in higher bins than a lane's are
        // the suffix sum over the lanes above it.
        uint32_t c[8];
        uint32_t total = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          c[k] = hist[lane * 8 + k];
          total += c[k];
        }
        uint32_t incl = total;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t x = __shfl_down_sync(0xffffffffu, incl, off);
          if (lane + off < 32) incl += x;
        }
        uint32_t cum = incl - total;
#pragma unroll
        for (int k = 7; k >= 0; --k) {
          if (static_cast<int>(cum) < need && need <= static_cast<int>(cum + c[k])) {
            ctl[0] = lane * 8 + k;
            ctl[1] = need - static_cast<int>(cum);
            ctl[2] = static_cast<int>(c[k]);
          }
          cum += c[k];
        }
      }
      __syncthreads();
      prefix |= static_cast<uint32_t>(ctl[0]) << lo;
      mask |= dmask << lo;
      need = ctl[1];
      in_bin = ctl[2];
      hi = lo - 1;
    }
  }
  // ---- compaction of the winners: keys above the prefix, and those in its
  // bin (all of them, or the `need` lowest ids when more share the K-th
  // score than are wanted)
  const bool ties = in_bin > need;
  if (tid == 0) ctl[3] = 0;
  __syncthreads();
  auto put = [&](uint32_t u, int e) {
    const int pos = atomicAdd(&ctl[3], 1);
    if (pos < P)
      buf[pos] = (static_cast<uint64_t>(u) << 32) |
                 static_cast<uint32_t>(~static_cast<uint32_t>(e));
  };
  if (!ties) {
    for_each_slot([&](uint32_t u, int e, bool v) {
      if (v && (u & mask) >= prefix) put(u, e);
    });
  } else {
    // Only when the K-th score is shared (the mask covers every bit):
    // equal keys are ranked in block-id order, one slot of every thread at
    // a time.
    int taken = 0;
    for_each_slot([&](uint32_t u, int e, bool v) {
      if (v && (u & mask) > prefix) put(u, e);
      const bool eq = v && (u & mask) == prefix;
      const unsigned b = __ballot_sync(0xffffffffu, eq);
      if (lane == 0) ctl[4 + warp] = __popc(b);
      __syncthreads();
      int before = taken + __popc(b & lt);
      for (int w = 0; w < warp; ++w) before += ctl[4 + w];
      if (eq && before < need) put(u, e);
      for (int w = 0; w < kSelWarps; ++w) taken += ctl[4 + w];
      __syncthreads();
    });
  }
  __syncthreads();
  const int n = min(ctl[3], P);

  // ---- bitonic sort of the P winner slots, descending: element
  // e = i * kSelThreads + tid sits in x[i]; partners closer than 32 are
  // swapped by shuffles, farther ones through shared memory, and within a
  // thread when they are kSelThreads apart.
  uint64_t x[kHeld];
#pragma unroll
  for (int i = 0; i < kHeld; ++i) {
    const int e = i * kSelThreads + tid;
    x[i] = (e < P && e < n) ? buf[e] : 0ull;
  }
  __syncthreads();
#pragma unroll
  for (int size = 2; size <= P; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      uint64_t y[kHeld];
      if (j < 32) {
#pragma unroll
        for (int i = 0; i < kHeld; ++i) y[i] = __shfl_xor_sync(0xffffffffu, x[i], j);
      } else if (j < kSelThreads) {
#pragma unroll
        for (int i = 0; i < kHeld; ++i) {
          const int e = i * kSelThreads + tid;
          if (e < P) buf[e] = x[i];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kHeld; ++i) {
          const int e = i * kSelThreads + tid;
          y[i] = e < P ? buf[e ^ j] : 0ull;
        }
        __syncthreads();
      } else {
#pragma unroll
        for (int i = 0; i < kHeld; ++i) y[i] = x[i ^ (j / kSelThreads)];
      }
#pragma unroll
      for (int i = 0; i < kHeld; ++i) {
        const int e = i * kSelThreads + tid;
        const bool d = (e & size) == 0;          // this block sorted descending
        const bool lower = (e & j) == 0;
        const bool take_max = lower == d;
        x[i] = take_max ? (x[i] > y[i] ? x[i] : y[i]) : (x[i] < y[i] ? x[i] : y[i]);
      }
    }
  }
  // ---- outputs; the region takes the admission's scratch
  AdmitWarpSmem& S = *reinterpret_cast<AdmitWarpSmem*>(smem);
#pragma unroll
  for (int i = 0; i < kHeld; ++i) {
    const int e = i * kSelThreads + tid;
    if (e < a.K) {
      const uint64_t key = x[i];
      const int id = key == 0ull ? -1 : static_cast<int>(~static_cast<uint32_t>(key));
      a.topk_ids[static_cast<size_t>(pair) * a.K + e] = id;
      if (a.topk_scores)
        a.topk_scores[static_cast<size_t>(pair) * a.K + e] =
            key == 0ull ? -INFINITY : key_float(static_cast<uint32_t>(key >> 32));
      S.topk[e] = id;
    }
  }
  if (!a.fuse_admit) return;
  __syncthreads();
  if (warp == 0)
    admit_warp<KPL>(a.admit, pair, S, reinterpret_cast<uint32_t*>(smem + sizeof(AdmitWarpSmem)));
}

// Raise the kernel's dynamic shared memory limit to `smem` (once per device
// and size).
template <int KPL, int CW>
cudaError_t configure(int smem) {
  static int configured_device = -1;
  static int configured_smem = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev || smem > configured_smem) {
    e = cudaFuncSetAttribute(score_topk_kernel<KPL, CW>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
    configured_smem = smem;
  }
  return cudaSuccess;
}

template <int KPL, int CW>
cudaError_t launch_kpl_cw(const ScoreArgs& a, cudaStream_t s) {
  if (a.pairs <= 0) return cudaSuccess;
  const int smem = Layout<KPL, CW>::total(a.NBmax);
  cudaError_t e = configure<KPL, CW>(smem);
  if (e != cudaSuccess) return e;
  score_topk_kernel<KPL, CW><<<a.pairs, (CW + 1) * 32, smem, s>>>(a);
  return cudaGetLastError();
}

// CTAs of a variant resident on the whole GPU at once (0 if unknown).
template <int KPL, int CW>
int grid_slots(int NBmax) {
  const int smem = Layout<KPL, CW>::total(NBmax);
  int dev = 0, sms = 0, per = 0;
  if (configure<KPL, CW>(smem) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, score_topk_kernel<KPL, CW>,
                                                    (CW + 1) * 32, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per * sms;
}

// Consumer warps per CTA, chosen by wave quantisation of the one-CTA-per-pair
// grid.  8 warps (twice the bytes in flight per CTA) unless that grid needs a
// second wave that would run less than half full while the 4-warp grid fits
// in one: measured on GB300, 720 pairs (36-layer loop, 90 requests): 4 warps
// 3657 against 3392 layer-steps/s (scan 91 vs 109 us); 1024 pairs (last
// 8-warp wave 68 % full): 8 warps 3108 against 2872; 512 pairs of 2048
// blocks (one wave either way): 8 warps 3685 against 3630.
// OASIS_SCAN_WARPS=4 or 8 forces a variant.
template <int KPL>
int scan_warps(int pairs, int NBmax) {
  static const int forced = [] {
    const char* e = std::getenv("OASIS_SCAN_WARPS");
    const int v = e ? std::atoi(e) : 0;
    return (v == 4 || v == 8) ? v : 0;
  }();
  if (forced) return forced;
  static int cached_dev = -1, cached_nb = -1, s8 = 0, s4 = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 8;
  if (dev != cached_dev || NBmax != cached_nb) {
    s8 = grid_slots<KPL, 8>(NBmax);
    s4 = grid_slots<KPL, 4>(NBmax);
    cached_dev = dev;
    cached_nb = NBmax;
  }
  if (s8 > 0 && s4 > 0 && pairs > s8 && pairs <= s4) {
    const int last = pairs % s8;  // CTAs of the 8-warp grid's last wave
    if (last != 0 && 2 * last < s8) return 4;
  }
  return 8;
}

template <int KPL>
cudaError_t launch_kpl(const ScoreArgs& a, cudaStream_t s) {
  return scan_warps<KPL>(a.pairs, a.NBmax) == 4 ? launch_kpl_cw<KPL, 4>(a, s)
                                                : launch_kpl_cw<KPL, 8>(a, s);
}

template <int CW>
constexpr int scan_smem_bytes() {
  return kStages * 4 * CW * kSummBytes + 64;
}

// CTAs of scan_kernel<CW> resident on the whole GPU at once (0 if unknown).
template <int CW>
int scan_slots() {
  int dev = 0, sms = 0, per = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, scan_kernel<CW>, (CW + 1) * 32,
                                                    scan_smem_bytes<CW>()) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per * sms;
}

// Consumer warps of the split scan, by wave quantisation as for the fused
// kernel: 8 unless its one-CTA-per-pair grid needs a second wave less than
// half full while the 4-warp grid fits in one.  OASIS_SCAN_WARPS forces one.
int split_scan_warps(int pairs) {
  static const int forced = [] {
    const char* e = std::getenv("OASIS_SCAN_WARPS");
    const int v = e ? std::atoi(e) : 0;
    return (v == 4 || v == 8) ? v : 0;
  }();
  if (forced) return forced;
  static int cached_dev = -1, s8 = 0, s4 = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 8;
  if (dev != cached_dev) {
    s8 = scan_slots<8>();
    s4 = scan_slots<4>();
    cached_dev = dev;
  }
  if (s8 > 0 && s4 > 0 && pairs > s8 && pairs <= s4) {
    const int last = pairs % s8;
    if (last != 0 && 2 * last < s8) return 4;
  }
  return 8;
}

template <int KPL, int NPT>
cudaError_t launch_select_npt(const ScoreArgs& a, cudaStream_t s) {
  const size_t smem = select_smem_bytes<KPL>(a.NBmax);
  if (smem > 48 * 1024) {
    static int configured_device = -1;
    static size_t configured_smem = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != configured_device || smem > configured_smem) {
      e = cudaFuncSetAttribute(select_kernel<KPL, NPT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      configured_device = dev;
      configured_smem = smem;
    }
  }
  select_kernel<KPL, NPT><<<a.pairs, kSelThreads, smem, s>>>(a);
  return cudaGetLastError();
}

// Keys per thread: the smallest of 1, 2, 4, 8 that holds NBmax blocks, else
// 0 (scores read again per pass).
template <int KPL>
cudaError_t launch_select_kpl(const ScoreArgs& a, cudaStream_t s) {
  const int per = (a.NBmax + kSelThreads - 1) / kSelThreads;
  if (per <= 1) return launch_select_npt<KPL, 1>(a, s);
  if (per <= 2) return launch_select_npt<KPL, 2>(a, s);
  if (per <= 4) return launch_select_npt<KPL, 4>(a, s);
  if (per <= 8) return launch_select_npt<KPL, 8>(a, s);
  return launch_select_npt<KPL, 0>(a, s);
}

}  // namespace

// Split (scan, then ranking) while the ranking keeps a pair's keys in
// registers (NBmax <= kSelThreads * 8 = 1024 blocks); one kernel for longer
// contexts, whose stream amortises the in-kernel ranking and whose separate
// ranking would compete longer with the attention beside it.  Measured on
// GB300, alternating on one box: 128 x 16K layer split 2935 / 3003 against
// fused 2862 / 2876 layer-steps/s (profiled passes; end to end 3137 / 3092
// against 3063 / 3078); 32-layer loop of 64 x 32K contexts (2064 blocks)
// split 3670 / 3595 against fused 3897 / 3879.  OASIS_SCAN=split or
// OASIS_SCAN=fused forces one form.
bool scan_is_split(int NBmax) {
  static const int forced = [] {
    const char* e = std::getenv("OASIS_SCAN");
    if (!e) return 0;
    if (std::string(e) == "fused") return 1;
    if (std::string(e) == "split") return 2;
    return 0;
  }();
  if (forced) return forced == 2;
  return NBmax <= kSelThreads * 8;
}

cudaError_t launch_scan_scores(const ScoreArgs& a, cudaStream_t s) {
  if (a.pairs <= 0) return cudaSuccess;
  if (split_scan_warps(a.pairs) == 4) {
    scan_kernel<4><<<a.pairs, 5 * 32, scan_smem_bytes<4>(), s>>>(a);
  } else {
    scan_kernel<8><<<a.pairs, 9 * 32, scan_smem_bytes<8>(), s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_topk_select(const ScoreArgs& a, cudaStream_t s) {
  if (a.pairs <= 0) return cudaSuccess;
  if (a.K <= 32) return launch_select_kpl<1>(a, s);
  if (a.K <= 64) return launch_select_kpl<2>(a, s);
  if (a.K <= 128) return launch_select_kpl<4>(a, s);
  return launch_select_kpl<8>(a, s);
}

cudaError_t launch_score_topk(const ScoreArgs& a, cudaStream_t s) {
  if (a.K <= 32) return launch_kpl<1>(a, s);
  if (a.K <= 64) return launch_kpl<2>(a, s);
  if (a.K <= 128) return launch_kpl<4>(a, s);
  return launch_kpl<8>(a, s);
}

cudaError_t preload_score_kernels() {
  cudaFuncAttributes at;
  const void* fns[] = {
      reinterpret_cast<const void*>(score_topk_kernel<1, 8>),
      reinterpret_cast<const void*>(score_topk_kernel<2, 8>),
      reinterpret_cast<const void*>(score_topk_kernel<4, 8>),
      reinterpret_cast<const void*>(score_topk_kernel<8, 8>),
      reinterpret_cast<const void*>(score_topk_kernel<1, 4>),
      reinterpret_cast<const void*>(score_topk_kernel<2, 4>),
      reinterpret_cast<const void*>(score_topk_kernel<4, 4>),
      reinterpret_cast<const void*>(score_topk_kernel<8, 4>),
      reinterpret_cast<const void*>(scan_kernel<8>),
      reinterpret_cast<const void*>(scan_kernel<4>),
      reinterpret_cast<const void*>(select_kernel<1, 1>),
      reinterpret_cast<const void*>(select_kernel<4, 8>),
      reinterpret_cast<const void*>(select_kernel<4, 0>),
      reinterpret_cast<const void*>(select_kernel<8, 8>)};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncGetAttributes(&at, f);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace oasis
