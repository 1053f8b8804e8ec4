// Step 3 of Prof-K, the filter pass ("Prof-K: Probabilistic One-Pass Filtering
// for Efficient Top-k Selection", Section 3, stage 3, and Appendix C "The
// Filter Kernel"): stream x once, count R = |{x_i >= tau}| exactly and append
// the passers to a buffer of capacity M.
//
// GB300 design.  The pass is a pure HBM read stream, so the kernel keeps as
// many 16-byte loads in flight as the memory system wants and does almost
// nothing else on the common path, with no block-wide barrier anywhere:
//  * persistent grid of resident CTAs; every warp strides on its own over
//    warp tiles of 32 lanes x U float4 (4U values per lane), issuing U
//    independent 128-bit non-allocating loads per lane;
//  * fast path: a NaN-propagating max over the lane's 4U values, one compare
//    against tau and one warp vote;
//  * slow path (some lane holds a passer or a NaN): per-element >= / > / NaN
//    tests into a 64-bit lane mask and a warp scan of the passer counts; the
//    passers go to the warp's private staging area in shared memory (128
//    keys).  A full stage is flushed with ONE atomicAdd on the row's counter,
//    whose old value is the slot of the first flushed key, so dense inputs
//    (large k) do not serialize on the counter.  Stores are masked to M and
//    the counter keeps counting, as in the pages' kernel.  Once a warp sees
//    the counter pass M it counts the rest in a register (no more atomics,
//    no stores), so inputs that overflow the buffer cost no atomics either;
//  * R_gt, the NaN count and those late passers are per-lane registers,
//    reduced once per row per warp.
// A passer (v, i) is stored as the 64-bit key (ord(v) << 32) | ~i, the order
// the refinement sorts by.
#include "kernels.h"

namespace profk {
namespace {

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ float comp(const float4& v, int c) {
  return c == 0 ? v.x : (c == 1 ? v.y : (c == 2 ? v.z : v.w));
}

__device__ __forceinline__ void flush_row(RowState& S, unsigned long long& gt, unsigned long long& nan,
                                          unsigned long long& late) {
  unsigned long long g = gt, q = nan;
  for (int o = 16; o; o >>= 1) {
    g += __shfl_down_sync(FULL_MASK, g, o);
    q += __shfl_down_sync(FULL_MASK, q, o);
  }
  if ((threadIdx.x & 31) == 0) {
    if (g) atomicAdd(&S.R_gt, g);
    if (q) atomicAdd(&S.nan, q);
    if (late) atomicAdd(&S.R_ge, late);
  }
  gt = 0;
  nan = 0;
  late = 0;
}

constexpr int STAGE = 128;  // staged passer keys per warp

// Moves a warp's staged keys into the buffer with one reservation.
__device__ __forceinline__ void flush_stage(RowState& S, unsigned long long* stage, int& stage_n,
                                            unsigned long long* br, int64_t M, bool& over) {
  if (stage_n == 0) return;
  const int lane = threadIdx.x & 31;
  unsigned long long gbase = 0;
  if (lane == 0) gbase = atomicAdd(&S.R_ge, static_cast<unsigned long long>(stage_n));
  gbase = __shfl_sync(FULL_MASK, gbase, 0);
  __syncwarp();
  for (int j = lane; j < stage_n; j += 32)
    if (gbase + j < static_cast<unsigned long long>(M)) br[gbase + j] = stage[j];
  if (gbase + stage_n > static_cast<unsigned long long>(M)) over = true;
  stage_n = 0;
  __syncwarp();
}

template <int T, int U>
__global__ void __launch_bounds__(T) k_filter(FilterArgs a) {
  pdl_wait();
  static_assert(4 * U <= 64, "at most 64 elements per lane");
  constexpr int64_t WT = 32 * 4 * U;  // elements per warp tile
  __shared__ unsigned long long s_stage[T / 32][STAGE];
  unsigned long long* stage = s_stage[threadIdx.x >> 5];
  int stage_n = 0;  // warp-uniform
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (T / 32);
  const int64_t tiles_per_row = (a.n + WT - 1) / WT;
  const int64_t total = tiles_per_row * a.nrows;
  int cur = -1;
  int row = 0;
  float tau = 0.f;
  bool over = false;  // this warp saw the row's counter pass M
  const float* xr = nullptr;
  unsigned long long* br = nullptr;
  unsigned long long gt = 0, nan = 0, late = 0;
  for (int64_t tile = static_cast<int64_t>(blockIdx.x) * (T / 32) + (threadIdx.x >> 5); tile < total;
       tile += nwarps) {
    const int ri = static_cast<int>(tile / tiles_per_row);
    const int64_t base = (tile - static_cast<int64_t>(ri) * tiles_per_row) * WT;
    if (ri != cur) {
      if (cur >= 0) {
        flush_stage(a.st[row], stage, stage_n, br, a.M, over);
        flush_row(a.st[row], gt, nan, late);
      }
      cur = ri;
      row = a.rows ? a.rows[ri] : ri;
      tau = key_to_float(a.st[row].tau_key);
      xr = a.x + static_cast<int64_t>(row) * a.ld;
      br = a.buf + static_cast<int64_t>(row) * a.M;
      over = false;
    }
    float4 v[U];
    uint64_t valid = ~0ull;
    if (base + WT <= a.n) {
      const float4* p = reinterpret_cast<const float4*>(xr + base) + lane;
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = ld_stream(p + u * 32);
    } else {
      valid = 0;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t i = base + (static_cast<int64_t>(u) * 32 + lane) * 4 + c;
          const bool ok = i < a.n;
          f[c] = ok ? xr[i] : -INFINITY;
          valid |= static_cast<uint64_t>(ok) << (u * 4 + c);
        }
        v[u] = make_float4(f[0], f[1], f[2], f[3]);
      }
    }
    float mu[U];
#pragma unroll
    for (int u = 0; u < U; ++u) mu[u] = max_nan(max_nan(v[u].x, v[u].y), max_nan(v[u].z, v[u].w));
    float m = mu[0];
#pragma unroll
    for (int u = 1; u < U; ++u) m = max_nan(m, mu[u]);
    // Masked lanes hold -inf; they reach the slow path only when tau is -inf,
    // and `valid` keeps them out of every count there.
    const bool hit = !(m < tau);
    if (!__any_sync(FULL_MASK, hit)) continue;
    uint64_t ge = 0;
    if (hit) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (mu[u] < tau) continue;  // no passer and no NaN among these four
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int e = u * 4 + c;
          const float f = comp(v[u], c);
          const bool ok = (valid >> e) & 1ull;
          ge |= static_cast<uint64_t>(ok && f >= tau) << e;
          gt += (ok && f > tau);
          nan += (ok && f != f);
        }
      }
    }
    const unsigned cnt = __popcll(ge);
    unsigned incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned tot = __shfl_sync(FULL_MASK, incl, 31);
    if (tot == 0) continue;
    if (over) {
      if (lane == 0) late += tot;
      continue;
    }
    if (tot <= STAGE) {
      if (stage_n + static_cast<int>(tot) > STAGE) {
        flush_stage(a.st[row], stage, stage_n, br, a.M, over);
        if (over) {
          if (lane == 0) late += tot;
          continue;
        }
      }
      if (cnt) {
        int pos = stage_n + static_cast<int>(incl - cnt);
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int e = u * 4 + c;
            if ((ge >> e) & 1ull) {
              const int64_t idx = base + (static_cast<int64_t>(u) * 32 + lane) * 4 + c;
              stage[pos++] = cand_key(comp(v[u], c), static_cast<uint32_t>(idx));
            }
          }
        }
      }
      stage_n += static_cast<int>(tot);
      __syncwarp();
      continue;
    }
    // More passers in this tile than a stage holds: reserve for the tile alone.
    unsigned long long gbase = 0;
    if (lane == 0) gbase = atomicAdd(&a.st[row].R_ge, static_cast<unsigned long long>(tot));
    gbase = __shfl_sync(FULL_MASK, gbase, 0);
    if (gbase + tot > static_cast<unsigned long long>(a.M)) over = true;
    if (cnt && gbase < static_cast<unsigned long long>(a.M)) {
      unsigned long long pos = gbase + incl - cnt;
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int e = u * 4 + c;
          if ((ge >> e) & 1ull) {
            if (pos < static_cast<unsigned long long>(a.M)) {
              const int64_t idx = base + (static_cast<int64_t>(u) * 32 + lane) * 4 + c;
              br[pos] = cand_key(comp(v[u], c), static_cast<uint32_t>(idx));
            }
            ++pos;
          }
        }
      }
    }
  }
  if (cur >= 0) {
    flush_stage(a.st[row], stage, stage_n, br, a.M, over);
    flush_row(a.st[row], gt, nan, late);
  }
}

// Launch shape: threads per CTA and 16-byte loads per lane per warp tile.
#ifndef PROFK_FILTER_THREADS
#define PROFK_FILTER_THREADS 256
#endif
#ifndef PROFK_FILTER_VEC
#define PROFK_FILTER_VEC 8
#endif
constexpr int FT = PROFK_FILTER_THREADS;
constexpr int FU = PROFK_FILTER_VEC;

}  // namespace

int filter_default_grid(int sms) {
  int per = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_filter<FT, FU>, FT, 0);
  if (per < 1) per = 1;
  return sms * per;
}

void launch_filter(const FilterArgs& a, cudaStream_t stream) {
  const int64_t WT = 32 * 4 * FU;
  const int64_t warp_tiles = ((a.n + WT - 1) / WT) * a.nrows;
  const int64_t ctas = (warp_tiles + FT / 32 - 1) / (FT / 32);
  int grid = a.grid;
  if (ctas < grid) grid = static_cast<int>(ctas);
  if (grid < 1) grid = 1;
  launch_kernel(k_filter<FT, FU>, grid, FT, 0, stream, a);
}

}  // namespace profk
