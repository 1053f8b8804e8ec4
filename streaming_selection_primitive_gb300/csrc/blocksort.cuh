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

// Descending sort of 32 E keys (E = 1, 2, 4 or 8) by one warp, E in each
// lane's registers: key lane * E + r is v[r].  The bitonic network's
// partners closer than E are other registers of the same lane (an exchange),
// the rest other lanes (shuffles).  With the lane-major layout only the
// partner distances E .. 16E cross lanes: 15 shuffle passes for any E,
// against 30 for 256 keys with key r * 32 + lane.
template <int E>
__device__ __forceinline__ void warp_sort_desc(unsigned long long (&v)[E]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32 * E; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j >= 1; j >>= 1) {
      if (j < E) {
        // The block's direction: from the register for blocks inside a lane,
        // else from the lane.
        const bool lane_desc = (lane & (size >= E ? size / E : 0)) == 0;
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const int r2 = r ^ j;
          if (r2 > r) {
            const bool desc = size < E ? (r & size) == 0 : lane_desc;
            const unsigned long long a = v[r], b = v[r2];
            if (desc ? (a < b) : (a > b)) {
              v[r] = b;
              v[r2] = a;
            }
          }
        }
      } else {
        const int jl = j / E;  // partner lane distance
        const bool lower = (lane & jl) == 0;
        const bool desc = (lane & (size / E)) == 0;  // size >= 2E: the block's direction depends on the lane only
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const unsigned long long o = __shfl_xor_sync(FULL_MASK, v[r], jl);
          v[r] = (desc == lower) ? (v[r] > o ? v[r] : o) : (v[r] < o ? v[r] : o);
        }
      }
    }
  }
}

__device__ __forceinline__ void warp_sort256_desc(unsigned long long (&v)[8]) { warp_sort_desc<8>(v); }

// Shared-memory slot of key i in the buffers of block_merge_sort_desc: the
// low four bits of i XORed with the next four.  A 64-bit key spans two of the
// 32 banks, so 16 consecutive keys fill them once; with the swizzle, threads
// that read or write keys 4 or 8 apart (the merge rounds' pattern, each thread
// taking consecutive outputs) spread over all banks instead of piling onto
// two or four of them (an 8- or 16-way conflict), and consecutive keys stay
// conflict-free.  The map permutes each aligned group of 256 keys.
__device__ __forceinline__ int mswz(int i) { return i ^ ((i >> 4) & 15); }

// Descending sort of P keys (P a multiple of 256, at most 256 x the warps of
// the block) by a block of 1024 threads, key i stored at s[mswz(i)]: every
// warp sorts one run of 256 in registers, then runs are merged pairwise
// (merge path: each thread finds where its P / 1024 outputs start by a binary
// search, then merges them), alternating between s and t (P keys each, the
// same layout).  Keys must be distinct.  Returns the buffer that holds the
// result (key i at mswz(i)); ends with a block barrier.
__device__ __forceinline__ unsigned long long* block_merge_sort_desc(unsigned long long* s, unsigned long long* t,
                                                                     int P) {
  constexpr int T = 1024;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp * 256 < P) {
    unsigned long long v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) v[r] = s[mswz(warp * 256 + lane * 8 + r)];
    warp_sort256_desc(v);
#pragma unroll
    for (int r = 0; r < 8; ++r) s[mswz(warp * 256 + lane * 8 + r)] = v[r];
  }
  __syncthreads();
  // Outputs per thread and round: a power of two, so that no thread's run of
  // outputs crosses the boundary of a merged pair (pairs are 512 or more long).
  int per = 1;
  while (per * T < P) per <<= 1;
  for (int w = 256; w < P; w <<= 1) {
    const int p0 = threadIdx.x * per;
    if (p0 < P) {
      const int base = p0 / (2 * w) * (2 * w);  // this pair's first position
      const int na = w < P - base ? w : P - base;
      const int nb = P - base - na < w ? P - base - na : w;
      auto A = [&](int q) { return s[mswz(base + q)]; };
      auto B = [&](int q) { return s[mswz(base + na + q)]; };
      const int off = p0 - base;
      int lo = off > nb ? off - nb : 0, hi = off < na ? off : na;
      while (lo < hi) {  // how many of the first `off` outputs come from A
        const int mid = (lo + hi) >> 1;
        if (A(mid) > B(off - mid - 1))
          lo = mid + 1;
        else
          hi = mid;
      }
      int i = lo, j = off - lo;
      const int end = p0 + per < base + na + nb ? p0 + per : base + na + nb;
      // The heads of both runs are kept in registers: one shared load per output.
      unsigned long long ha = i < na ? A(i) : 0ull, hb = j < nb ? B(j) : 0ull;
      for (int p = p0; p < end; ++p) {
        const bool takeA = j >= nb || (i < na && ha > hb);
        if (takeA) {
          t[mswz(p)] = ha;
          ++i;
          ha = i < na ? A(i) : 0ull;
        } else {
          t[mswz(p)] = hb;
          ++j;
          hb = j < nb ? B(j) : 0ull;
        }
      }
    }
    __syncthreads();
    unsigned long long* x = s;
    s = t;
    t = x;
  }
  return s;
}

}  // namespace profk
