// admit.cuh -- capped least-recently-selected eviction of one
// (request, KV head) by one warp (step a4), shared by the stand-alone admit
// kernel and the tail of the fused score + top-K + admit kernel.
//
// "Pith review of OasisKV", section "What carries the argument": eviction is
// capped, and every block admitted from outside the resident set replaces
// the resident block selected least recently, which bounds the traffic of a
// step.
// Reading of the pages: (i) stamp re-selected residents with the step;
// (ii) missing top-K blocks in rank order; (iii) eviction candidates = slots
// whose block is not selected, empty first, then (stamp, block id, slot)
// ascending; (iv) at most C admissions; (v) the i-th missing block replaces
// the i-th candidate.  The admitted block takes spare pool unit K+i and the
// evicted unit becomes that spare, so the gather never writes a unit that
// the current table still references.  The miss-stall demand fetch runs the
// same steps in place (in_place, C = K): its gather completes on the
// critical path before any reader of the table, so the admitted block is
// written into the evicted slot's own unit.
//
// Membership is tested with two NBmax-bit bitmaps in shared memory; the
// eviction order is that of 64-bit keys
//   [63] occupied | [62:32] stamp+1 | [31:8] block id+1 | [7:0] slot
// (selected slots get the all-ones key and come last), the n first found by
// repeated warp minima when n is small, else by a bitonic sort.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "sortnet.cuh"

namespace oasis {

// Up to this many admissions the eviction order is found by repeated warp
// minima instead of a full sort of the K slot keys.
constexpr int kArgminRounds = 8;

struct AdmitWarpSmem {
  int topk[kMaxTopK];
  int res[kMaxTopK];
  int stamp[kMaxTopK];
  int phys[2 * kMaxTopK];
  int missing[kMaxTopK];
  int evslot[kMaxTopK];
  unsigned char in_t[kMaxTopK];
};

__host__ __device__ inline int bitmap_words(int nb) { return (nb + 31) >> 5; }

// Shared bytes one warp needs: the struct plus two bitmaps, 16-byte rounded.
__host__ __device__ inline size_t admit_warp_smem_bytes(int NBmax) {
  return (sizeof(AdmitWarpSmem) + 2 * 4 * static_cast<size_t>(bitmap_words(NBmax)) + 15) &
         ~static_cast<size_t>(15);
}

// Precondition: S.topk[0..K) holds this pair's top-K list (rank order, -1
// padded) and the warp has synchronised.  bm points at 2*bitmap_words(NBmax)
// words of this warp's shared memory.
template <int KPL>
__device__ void admit_warp(const AdmitArgs& a, int pair, AdmitWarpSmem& S, uint32_t* bm) {
  const int lane = threadIdx.x & 31;
  const int K = a.K, C = a.C, U = a.U, NB = a.NBmax;
  const int nw = bitmap_words(NB);
  uint32_t* bmT = bm;
  uint32_t* bmR = bm + nw;
  const size_t ok = static_cast<size_t>(pair) * K;
  const size_t ou = static_cast<size_t>(pair) * U;

  for (int s = lane; s < K; s += 32) {
    S.res[s] = a.res_cur[ok + s];
    S.stamp[s] = a.stamps[ok + s];
  }
  for (int u = lane; u < U; u += 32) S.phys[u] = a.phys_cur[ou + u];
  for (int w = lane; w < 2 * nw; w += 32) bm[w] = 0u;
  __syncwarp();
  for (int s = lane; s < K; s += 32) {
    const int b = S.topk[s];
    if (b >= 0 && b < NB) atomicOr(&bmT[b >> 5], 1u << (b & 31));
    const int id = S.res[s];
    if (id >= 0 && id < NB) atomicOr(&bmR[id >> 5], 1u << (id & 31));
  }
  __syncwarp();

  // (i) re-selected residents take the step as their stamp.
  for (int s = lane; s < K; s += 32) {
    const int id = S.res[s];
    const bool f = id >= 0 && id < NB && ((bmT[id >> 5] >> (id & 31)) & 1u);
    S.in_t[s] = f;
    if (f) S.stamp[s] = a.step;
  }
  // (ii) missing blocks in rank order.
  int n_missing = 0;
  for (int c = 0; c < K; c += 32) {
    const int i = c + lane;
    const int b = i < K ? S.topk[i] : -1;
    const bool m = b >= 0 && b < NB && !((bmR[b >> 5] >> (b & 31)) & 1u);
    const unsigned bal = __ballot_sync(0xffffffffu, m);
    if (m) S.missing[n_missing + __popc(bal & ((1u << lane) - 1u))] = b;
    n_missing += __popc(bal);
  }
  const int n = min(n_missing, C);
  __syncwarp();

  // (iii) eviction order.
  uint64_t key[KPL];
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int s = i * 32 + lane;
    if (s < K && !S.in_t[s]) {
      const uint64_t occ = S.res[s] >= 0 ? 1ull : 0ull;
      key[i] = (occ << 63) | (static_cast<uint64_t>(static_cast<uint32_t>(S.stamp[s] + 1)) << 32) |
               (static_cast<uint64_t>(static_cast<uint32_t>(S.res[s] + 1) & 0xffffffu) << 8) |
               static_cast<uint64_t>(s);
    } else {
      key[i] = ~0ull;
    }
  }
  if (n <= kArgminRounds) {
    // Few admissions: the n smallest keys by repeated warp minima (keys are
    // distinct: the slot sits in the low byte).
    for (int e = 0; e < n; ++e) {
      uint64_t m = key[0];
#pragma unroll
      for (int i = 1; i < KPL; ++i) m = key[i] < m ? key[i] : m;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, m, off);
        m = o < m ? o : m;
      }
      if (lane == 0) S.evslot[e] = static_cast<int>(m & 0xffu);
#pragma unroll
      for (int i = 0; i < KPL; ++i)
        if (key[i] == m) key[i] = ~0ull;
    }
  } else {
    bitonic_sort<KPL>(key, false);
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int e = i * 32 + lane;
      if (e < n) S.evslot[e] = static_cast<int>(key[i] & 0xffu);
    }
  }
  __syncwarp();

  // (iv, v) outputs and the next tables.
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
  for (int i = lane; i < n; i += 32) {
    const int s = S.evslot[i];
    S.res[s] = S.missing[i];
    S.stamp[s] = a.step;
    if (!a.in_place) {
      const int unit_old = S.phys[s];
      S.phys[s] = S.phys[K + i];
      S.phys[K + i] = unit_old;
    }
  }
  __syncwarp();
  for (int s = lane; s < K; s += 32) {
    a.res_nxt[ok + s] = S.res[s];
    a.stamps[ok + s] = S.stamp[s];
  }
  for (int u = lane; u < U; u += 32) a.phys_nxt[ou + u] = S.phys[u];
}

}  // namespace oasis
