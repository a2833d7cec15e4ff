// sortnet.cuh -- warp-level bitonic networks over 64-bit keys held in
// registers: key e = i*32 + lane lives in x[i] of lane `lane` (E = 32*KPL keys).
#pragma once

#include <stdint.h>

namespace oasis {

// One compare-exchange stage: partner e ^ j; the block of `size` keys that
// holds e is ordered descending when ((e & size) == 0) == desc.
template <int KPL>
__device__ __forceinline__ void bitonic_stage(uint64_t (&x)[KPL], int size, int j,
                                              bool desc) {
  const int lane = threadIdx.x & 31;
  if (j >= 32) {
    const int jr = j >> 5;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      if ((i & jr) == 0) {
        const int p = i | jr;
        const int e = i * 32 + lane;
        const bool d = ((e & size) == 0) == desc;
        const uint64_t lo = x[i], hi = x[p];
        const bool sw = d ? (lo < hi) : (lo > hi);
        x[i] = sw ? hi : lo;
        x[p] = sw ? lo : hi;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int e = i * 32 + lane;
      const uint64_t y = __shfl_xor_sync(0xffffffffu, x[i], j);
      const bool lower = (lane & j) == 0;
      const bool d = ((e & size) == 0) == desc;
      const bool take_max = (lower == d);
      x[i] = take_max ? (x[i] > y ? x[i] : y) : (x[i] < y ? x[i] : y);
    }
  }
}

// Full sort of the E keys, descending if `desc`, else ascending.
template <int KPL>
__device__ __forceinline__ void bitonic_sort(uint64_t (&x)[KPL], bool desc) {
  constexpr int E = 32 * KPL;
#pragma unroll
  for (int size = 2; size <= E; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) bitonic_stage<KPL>(x, size, j, desc);
  }
}

// The stages of bitonic_sort of size 64 and up: x holds KPL runs of 32 keys,
// run i already sorted descending iff ((i & 1) == 0) == desc.
template <int KPL>
__device__ __forceinline__ void bitonic_finish(uint64_t (&x)[KPL], bool desc) {
  constexpr int E = 32 * KPL;
#pragma unroll
  for (int size = 64; size <= E; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) bitonic_stage<KPL>(x, size, j, desc);
  }
}

// a (descending) <- the top E keys of a and b, descending; b must be ascending.
template <int KPL>
__device__ __forceinline__ void merge_top(uint64_t (&a)[KPL], const uint64_t (&b)[KPL]) {
  constexpr int E = 32 * KPL;
#pragma unroll
  for (int i = 0; i < KPL; ++i) a[i] = a[i] > b[i] ? a[i] : b[i];
#pragma unroll
  for (int j = E >> 1; j > 0; j >>= 1) bitonic_stage<KPL>(a, E, j, true);
}

}  // namespace oasis
