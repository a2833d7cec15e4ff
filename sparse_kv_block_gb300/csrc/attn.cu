// attn.cu -- look-ahead attention (step a1).
//
// One shared pass serves the normal and the draft query of every query head
// of a KV head over that head's resident blocks ("Pith review of OasisKV",
// section "What carries the argument": a single attention kernel handles both
// tokens of a decode step, reading one resident block set for the two).
//
// GB300 mapping.  One CTA per (request, KV head); four warps, each streaming
// its own share of the resident units through a private two-deep ring of
// 8 KiB shared-memory stages filled by TMA tensor copies (128-byte swizzle,
// so ldmatrix reads are bank-conflict free).  The contraction per 16-token
// unit is tiny (16 tokens x 8 query vectors x 128 dims), so it runs on
// mma.sync m16n8k16 with the tokens as M and the 2 x G <= 8 query vectors as
// N: S^T = K_unit * Q^T, online softmax over tokens, then O^T += V^T * P^T
// with P^T moved into the B-operand layout by movmatrix.  With several draft
// queries per step the (1 + D) x G query vectors take two such 8-column
// tiles (kNT = 2), reading each staged unit once for all of them.  The
// kernel is bound by HBM reads of the resident units (8 KiB per unit).
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"

namespace oasis {
namespace {

constexpr int kStages = 2;
constexpr int kStageBytes = kUnitBytes;            // 8 KiB: [half][32 rows][128 B]

// Shared memory of a CTA of W warps: W private rings, barriers, unit list.
template <int W>
struct AttnLayout {
  // The merge space ([W][16][128] fp32 partial outputs at most) reuses the
  // ring, so the ring must hold it.
  static_assert(W * kStages * kStageBytes >= W * 16 * 128 * 4 + 2 * W * 16 * 4,
                "merge space exceeds the ring");
  static constexpr int kRingBytes = W * kStages * kStageBytes;
  static constexpr int kBarOffset = kRingBytes;
  static constexpr int kListOffset = kBarOffset + 256;
  static constexpr int kCountOffset = kListOffset + kMaxTopK * 8;
  static constexpr int kSmemBytes = kCountOffset + 16 + 1024;  // + alignment slack
};

struct UnitRef {
  int unit;   // global pool unit index (pair * U + phys slot unit)
  int valid;  // valid tokens, 1..16
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t s = smem_u32(p);
  return p + ((1024u - (s & 1023u)) & 1023u);
}

// Byte offset of (row, 16-byte chunk) inside one 64-column half of a stage,
// as written by a TMA copy with 128-byte swizzle into a 1024-aligned buffer.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// kNT tiles of 8 query columns: column n = which * 4 + gi, which 0 = the
// normal query, 1 + e = draft e; gi = query head within the group.
// Register caps: three CTAs of this kernel fill an SM's shared memory, and
// the host-link gather of the same step must still find registers for one of
// its 128-thread CTAs (80 registers per thread) beside them.  Two tiles need
// up to 166 registers uncapped (3 x 128 x 166 fills the whole register file,
// which held the gathers back: 2538 against 3101 layer-steps/s at D = 2); at
// 144 there is no spill and 3 x 128 x 144 + 128 x 80 = 65536.
template <int kWarps, int kNT>
__global__ void __maxnreg__(kNT == 2 ? 144 : 96)
    attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap pool_map) {
  using Lay = AttnLayout<kWarps>;
  constexpr int kThreads = kWarps * 32;
  constexpr int kCols = 8 * kNT;
  constexpr int kBarOffset = Lay::kBarOffset;
  constexpr int kListOffset = Lay::kListOffset;
  constexpr int kCountOffset = Lay::kCountOffset;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kBarOffset);
  UnitRef* list = reinterpret_cast<UnitRef*>(base + kListOffset);
  int* count_s = reinterpret_cast<int*>(base + kCountOffset);

  const int pair = blockIdx.x;
  const int r = pair / a.Hkv;
  const int h = pair - r * a.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ctx = a.ctx_len[r];

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWarps * kStages; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
    prefetch_tensormap(&pool_map);
  }
  if (a.dense) {
    if (threadIdx.x == 0) {
      int nb = ctx > 0 ? (ctx + kBlock - 1) / kBlock : 0;
      if (nb > a.NBmax) {
        raise_error(a.err, kErrBadBlock);
        nb = a.NBmax;
      }
      *count_s = nb;
    }
  } else if (warp == 0) {
    // Compact the occupied slots (in slot order) into the unit list.
    const int32_t* res = a.res + static_cast<size_t>(pair) * a.K;
    const int32_t* phys = a.phys + static_cast<size_t>(pair) * a.U;
    int n = 0;
    for (int c = 0; c < a.K; c += 32) {
      const int s = c + lane;
      bool ok = false;
      int unit = 0, valid = 0;
      if (s < a.K) {
        const int id = res[s];
        if (id >= 0) {
          valid = min(kBlock, ctx - id * kBlock);
          unit = phys[s];
          if (id >= a.NBmax || valid <= 0) {
            raise_error(a.err, kErrBadBlock);
          } else if (unit < 0 || unit >= a.U) {
            raise_error(a.err, kErrBadUnit);
          } else {
            ok = true;
          }
        }
      }
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      if (ok) {
        UnitRef u;
        u.unit = pair * a.U + unit;
        u.valid = valid;
        list[n + __popc(bal & ((1u << lane) - 1u))] = u;
      }
      n += __popc(bal);
    }
    if (lane == 0) *count_s = n;
  }

  // B fragments of Q^T (d x 8 query vectors) per column tile; this lane
  // loads column g of each tile.
  const int g = lane >> 2;
  const int t = lane & 3;
  const size_t plane = static_cast<size_t>(a.R) * a.Hq * kHeadDim;
  uint32_t qf[kNT][8][2];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    const int which = nt * 2 + (g >> 2), gi = g & 3;
    if (gi < a.G && which <= a.D) {
      const __nv_bfloat16* base_q = which == 0
          ? static_cast<const __nv_bfloat16*>(a.q)
          : static_cast<const __nv_bfloat16*>(a.qd) + (which - 1) * plane;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(
          base_q + (static_cast<size_t>(r) * a.Hq + h * a.G + gi) * kHeadDim);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qf[nt][kk][0] = __ldg(src + 8 * kk + t);
        qf[nt][kk][1] = __ldg(src + 8 * kk + 4 + t);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) qf[nt][kk][0] = qf[nt][kk][1] = 0u;
    }
  }
  __syncthreads();

  const int n_units = *count_s;
  const int my_count = n_units > warp ? (n_units - warp + kWarps - 1) / kWarps : 0;
  uint8_t* my_ring = base + warp * kStages * kStageBytes;
  uint64_t* my_bars = bars + warp * kStages;

  // The k-th unit of this warp: a pool unit from the compacted list, or in
  // dense mode block `idx` of the pair's dense cache row.
  auto unit_row = [&](int k) {
    const int idx = warp + k * kWarps;
    return a.dense ? pair * a.NBmax + idx : list[idx].unit;
  };
  auto unit_valid = [&](int k) {
    const int idx = warp + k * kWarps;
    return a.dense ? min(kBlock, ctx - idx * kBlock) : list[idx].valid;
  };
  auto issue = [&](int k) {
    const int st = k % kStages;
    const int y = unit_row(k) * (2 * kBlock);
    uint8_t* dst = my_ring + st * kStageBytes;
    mbar_arrive_expect_tx(&my_bars[st], kStageBytes);
    tma_load_2d(dst, &pool_map, 0, y, &my_bars[st]);
    tma_load_2d(dst + kStageBytes / 2, &pool_map, 64, y, &my_bars[st]);
  };
  if (lane == 0) {
    for (int k = 0; k < kStages && k < my_count; ++k) issue(k);
  }

  // Per-lane ldmatrix row/chunk constants.
  const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;  // K rows (tokens)
  const int kch = lane >> 4;
  const int vrow = kBlock + (lane & 7) + ((lane >> 4) & 1) * 8;  // V rows
  const int vch = (lane >> 3) & 1;

  // Per column tile: O^T accumulators, running max and sum of columns 2t, 2t+1.
  float o[kNT][8][4];
  float m0[kNT], m1[kNT], l0[kNT], l1[kNT];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
    m0[nt] = m1[nt] = -INFINITY;
    l0[nt] = l1[nt] = 0.f;
  }
  const float sc = a.scale_log2;

  int k = 0;
  bool failed = false;
  for (; k < my_count; ++k) {
    const int st = k % kStages;
    const bool ok =
        __all_sync(0xffffffffu, mbar_wait(&my_bars[st], (k / kStages) & 1, a.wait_limit));
    if (!ok) {
      failed = true;
      break;
    }
    const int valid = unit_valid(k);
    uint8_t* stage = my_ring + st * kStageBytes;
    const uint32_t sb = smem_u32(stage);

    // S^T (16 tokens x 8 queries) = K_unit (16 x 128) * Q^T (128 x 8), per
    // column tile; each K fragment is loaded once for all tiles.
    float s[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int half = kk >> 2;
      const int chunk = (kk & 3) * 2 + kch;
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sb + half * (kStageBytes / 2) + swz(krow, chunk), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
        mma_bf16_16816(s[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
    }

    // Online softmax over tokens (rows g, g+8) per query column (2t, 2t+1).
    uint32_t b0[kNT], b1[kNT];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      float x0 = s[nt][0] * sc, x1 = s[nt][1] * sc, x2 = s[nt][2] * sc, x3 = s[nt][3] * sc;
      if (g >= valid) x0 = x1 = -INFINITY;
      if (g + 8 >= valid) x2 = x3 = -INFINITY;
      float t0 = fmaxf(x0, x2), t1 = fmaxf(x1, x3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, off));
        t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, off));
      }
      const float mn0 = fmaxf(m0[nt], t0), mn1 = fmaxf(m1[nt], t1);
      const float al0 = exp2f(m0[nt] - mn0), al1 = exp2f(m1[nt] - mn1);
      m0[nt] = mn0;
      m1[nt] = mn1;
      const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
      const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
      l0[nt] = l0[nt] * al0 + p0 + p2;
      l1[nt] = l1[nt] * al1 + p1 + p3;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[nt][mt][0] *= al0;
        o[nt][mt][1] *= al1;
        o[nt][mt][2] *= al0;
        o[nt][mt][3] *= al1;
      }
      b0[nt] = movmatrix_t(pack_bf16x2(p0, p1));
      b1[nt] = movmatrix_t(pack_bf16x2(p2, p3));
    }

    if (valid < kBlock) {
      // Zero the value rows past the context so that 0 * garbage stays 0.
      const int nchunks = (kBlock - valid) * 16;
      for (int j = lane; j < nchunks; j += 32) {
        const int row = kBlock + valid + (j >> 4);
        const int half = (j >> 3) & 1;
        *reinterpret_cast<uint4*>(stage + half * (kStageBytes / 2) + row * 128 +
                                  ((j & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }

    // O^T (128 dims x 8 queries) += V^T (128 x 16 tokens) * P^T (16 x 8)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int half = mt >> 2;
      const int chunk = (mt & 3) * 2 + vch;
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(sb + half * (kStageBytes / 2) + swz(vrow, chunk), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) mma_bf16_16816(o[nt][mt], a0, a1, a2, a3, b0[nt], b1[nt]);
    }
    __syncwarp();
    if (lane == 0 && k + kStages < my_count) issue(k + kStages);
  }
  if (failed) {
    if (lane == 0) raise_error(a.err, kErrTimeout);
    // Drain this warp's copies still in flight before the ring is reused.
    for (int kk = k; kk < my_count && kk < k + kStages; ++kk)
      (void)mbar_wait(&my_bars[kk % kStages], (kk / kStages) & 1);
  }

  // Row sums: reduce over the 8 lanes that share t.
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0[nt] += __shfl_xor_sync(0xffffffffu, l0[nt], off);
      l1[nt] += __shfl_xor_sync(0xffffffffu, l1[nt], off);
    }
  }

  __syncthreads();  // every ring slot has been consumed: reuse as merge space
  float* mo = reinterpret_cast<float*>(base);           // [kWarps][kCols][128]
  float* mm = mo + kWarps * kCols * kHeadDim;           // [kWarps][kCols]
  float* ml = mm + kWarps * kCols;                      // [kWarps][kCols]
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    const int c0 = warp * kCols + nt * 8 + 2 * t;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d0 = mt * 16 + g;
      mo[c0 * kHeadDim + d0] = o[nt][mt][0];
      mo[(c0 + 1) * kHeadDim + d0] = o[nt][mt][1];
      mo[c0 * kHeadDim + d0 + 8] = o[nt][mt][2];
      mo[(c0 + 1) * kHeadDim + d0 + 8] = o[nt][mt][3];
    }
    if (g == 0) {
      mm[c0] = m0[nt];
      mm[c0 + 1] = m1[nt];
      ml[c0] = l0[nt];
      ml[c0 + 1] = l1[nt];
    }
  }
  __syncthreads();

  for (int e = threadIdx.x; e < kCols * kHeadDim; e += kThreads) {
    const int n = e >> 7;
    const int dd = e & (kHeadDim - 1);
    const int which = n >> 2, gi = n & 3;
    if (gi >= a.G || which > a.D) continue;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, mm[w * kCols + n]);
    float acc = 0.f, den = 0.f;
    if (mx > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(mm[w * kCols + n] - mx);
        acc += f * mo[(w * kCols + n) * kHeadDim + dd];
        den += f * ml[w * kCols + n];
      }
    }
    const float v = den > 0.f ? acc / den : 0.f;
    const size_t idx = (which ? (which - 1) * plane : 0) +
                       (static_cast<size_t>(r) * a.Hq + h * a.G + gi) * kHeadDim + dd;
    void* dst = which ? a.outd : a.out;
    if (a.out_fp32)
      static_cast<float*>(dst)[idx] = v;
    else
      static_cast<__nv_bfloat16*>(dst)[idx] = __float2bfloat16_rn(v);
  }
}

}  // namespace

namespace {

template <int W, int NT>
cudaError_t configure_attn() {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(attn_kernel<W, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AttnLayout<W>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return cudaSuccess;
}

// Warps per CTA: 4 (3 CTAs per SM).  A 3-warp variant (4 CTAs per SM, the
// same bytes in flight per SM) fills the last wave of some grids better and
// is faster alone there (64 requests x 8 heads: 86.6 against 96.6 us), but
// measured inside the decode loops it was not (32-layer, 64-request loop:
// 3692 / 3636 against 3822 / 3731 layer-steps/s; 128 requests: equal), so it
// is only a tuning override: OASIS_ATTN_WARPS=3.
int attn_warps() {
  static const int forced = [] {
    const char* e = std::getenv("OASIS_ATTN_WARPS");
    return (e && std::atoi(e) == 3) ? 3 : 4;
  }();
  return forced;
}

template <int W, int NT>
cudaError_t launch_w(const AttnArgs& a, const CUtensorMap* pool_map, int grid, cudaStream_t s) {
  cudaError_t e = configure_attn<W, NT>();
  if (e != cudaSuccess) return e;
  attn_kernel<W, NT><<<grid, W * 32, AttnLayout<W>::kSmemBytes, s>>>(a, *pool_map);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, const CUtensorMap* pool_map,
                             cudaStream_t s) {
  const int grid = a.R * a.Hkv;
  if (grid == 0) return cudaSuccess;
  if (a.D < 1 || a.D > kMaxDrafts) return cudaErrorInvalidValue;
  if (a.D > 1)  // 12 or 16 query columns: two tiles
    return attn_warps() == 3 ? launch_w<3, 2>(a, pool_map, grid, s)
                             : launch_w<4, 2>(a, pool_map, grid, s);
  return attn_warps() == 3 ? launch_w<3, 1>(a, pool_map, grid, s)
                           : launch_w<4, 1>(a, pool_map, grid, s);
}

cudaError_t preload_attention_kernels() {
  cudaFuncAttributes at;
  const void* fns[] = {reinterpret_cast<const void*>(attn_kernel<4, 1>),
                       reinterpret_cast<const void*>(attn_kernel<3, 1>),
                       reinterpret_cast<const void*>(attn_kernel<4, 2>),
                       reinterpret_cast<const void*>(attn_kernel<3, 2>)};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncGetAttributes(&at, f);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace oasis
