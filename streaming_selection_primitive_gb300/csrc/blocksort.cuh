// Shared-memory sort of up to 8192 keys by one CTA of 1024 threads.
#pragma once

#include "common.cuh"

namespace profk {

// Descending bitonic sort of 1024*E keys held in shared memory by a block of
// 1024 threads.  Thread t of warp w holds keys w*32E + r*32 + lane
// (r = 0..E-1) in registers: compare-exchange partners closer than 32E are
// in the same warp (a shuffle for distance < 32, a register pair otherwise);
// only the wider stages go through shared memory, with one barrier each.
template <int E>
__device__ __forceinline__ void block_sort_desc(unsigned long long* s) {
  constexpr int T = 1024;
  constexpr int P = T * E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = warp * 32 * E;
  unsigned long long v[E];
#pragma unroll
  for (int r = 0; r < E; ++r) v[r] = s[seg + r * 32 + lane];
  for (int size = 2; size <= P; size <<= 1) {
    int j = size >> 1;
    if (j >= 32 * E) {
#pragma unroll
      for (int r = 0; r < E; ++r) s[seg + r * 32 + lane] = v[r];
      __syncthreads();
      for (; j >= 32 * E; j >>= 1) {
        for (int i = threadIdx.x; i < P; i += T) {
          const int l = i ^ j;
          if (l > i) {
            const unsigned long long a = s[i], b = s[l];
            const bool desc = (i & size) == 0;
            if (desc ? (a < b) : (a > b)) {
              s[i] = b;
              s[l] = a;
            }
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int r = 0; r < E; ++r) v[r] = s[seg + r * 32 + lane];
      __syncthreads();
    }
    // Partner in the same lane, register r ^ (jj / 32) (distances 32E/2 .. 32).
#pragma unroll
    for (int m = E / 2; m >= 1; m >>= 1) {
      const int jj = 32 * m;
      if (jj < size) {
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const int r2 = r ^ m;
          if (r2 > r) {
            const int i = seg + r * 32 + lane;
            const bool desc = (i & size) == 0;
            const unsigned long long a = v[r], b = v[r2];
            if (desc ? (a < b) : (a > b)) {
              v[r] = b;
              v[r2] = a;
            }
          }
        }
      }
    }
    // Partner in lane ^ jj, same register (distances 16 .. 1).
#pragma unroll
    for (int jj = 16; jj >= 1; jj >>= 1) {
      if (jj < size) {
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const int i = seg + r * 32 + lane;
          const bool desc = (i & size) == 0;
          const unsigned long long o = __shfl_xor_sync(FULL_MASK, v[r], jj);
          const bool lower = (lane & jj) == 0;
          v[r] = (desc == lower) ? (v[r] > o ? v[r] : o) : (v[r] < o ? v[r] : o);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < E; ++r) s[seg + r * 32 + lane] = v[r];
  __syncthreads();
}

}  // namespace profk
