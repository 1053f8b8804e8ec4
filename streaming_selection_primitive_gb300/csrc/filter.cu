// Step 3 of Prof-K, the filter pass ("Prof-K: Probabilistic One-Pass Filtering
// for Efficient Top-k Selection", Section 3, stage 3, and Appendix C "The
// Filter Kernel"): stream x once, count R = |{x_i >= tau}| exactly and append
// the passers to a buffer of capacity M, one atomic reservation per block.
//
// GB300 design.  The pass is a pure HBM read stream, so the kernel is built to
// keep as many 16-byte loads in flight as the memory system wants and to do
// almost nothing else on the common path:
//  * persistent grid of resident CTAs striding over tiles of THREADS*4*U
//    floats; each thread issues U independent 128-bit non-allocating loads;
//  * fast path: one NaN-propagating max over the thread's 4U values and a
//    single compare against tau (a NaN or a passer sends the block to the slow
//    path, NaNs are then counted and reported);
//  * slow path (any passer in the tile): per-element >= / > / NaN tests, a warp
//    scan of the passer counts, one shared scan of the warp totals and ONE
//    global atomicAdd per tile on the row's R counter, whose old value is the
//    slot of the tile's first passer.  Stores are masked to M, the counter
//    keeps counting past it, exactly as the pages' kernel does;
//  * R_gt and the NaN count are per-thread registers reduced once per row.
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

template <int T>
__device__ __forceinline__ void flush_row(RowState& S, unsigned long long& gt, unsigned long long& nan) {
  unsigned long long g = gt, q = nan;
  for (int o = 16; o; o >>= 1) {
    g += __shfl_down_sync(FULL_MASK, g, o);
    q += __shfl_down_sync(FULL_MASK, q, o);
  }
  if ((threadIdx.x & 31) == 0) {
    if (g) atomicAdd(&S.R_gt, g);
    if (q) atomicAdd(&S.nan, q);
  }
  gt = 0;
  nan = 0;
}

// Processes one tile whose values sit in v[] (U float4 per thread).  `valid`
// marks real elements (all of them except in a row's last, partial tile).
template <int T, int U>
__device__ __forceinline__ void tile_slow(const float4 (&v)[U], uint64_t valid, bool hit, float tau, int64_t base,
                                          RowState& S, unsigned long long* buf, int64_t M, unsigned long long& gt,
                                          unsigned long long& nan, unsigned* s_warp, unsigned long long* s_gbase) {
  constexpr int NW = T / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t ge = 0;
  if (hit) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
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
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned w = lane < NW ? s_warp[lane] : 0u;
    unsigned wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(FULL_MASK, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < NW) s_warp[lane] = wi - w;
    const unsigned total = __shfl_sync(FULL_MASK, wi, 31);
    if (lane == 0) *s_gbase = total ? atomicAdd(&S.R_ge, static_cast<unsigned long long>(total)) : 0ull;
  }
  __syncthreads();
  if (cnt) {
    unsigned long long pos = *s_gbase + s_warp[warp] + incl - cnt;
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = u * 4 + c;
        if ((ge >> e) & 1ull) {
          if (pos < static_cast<unsigned long long>(M)) {
            const int64_t idx = base + (static_cast<int64_t>(u) * T + threadIdx.x) * 4 + c;
            buf[pos] = cand_key(comp(v[u], c), static_cast<uint32_t>(idx));
          }
          ++pos;
        }
      }
    }
  }
}

template <int T, int U>
__global__ void __launch_bounds__(T) k_filter(FilterArgs a) {
  static_assert(4 * U <= 64, "at most 64 elements per thread");
  constexpr int64_t TILE = static_cast<int64_t>(T) * 4 * U;
  __shared__ unsigned s_warp[T / 32];
  __shared__ unsigned long long s_gbase;
  const int64_t tiles_per_row = (a.n + TILE - 1) / TILE;
  const int64_t total = tiles_per_row * a.nrows;
  int cur = -1;
  int row = 0;
  float tau = 0.f;
  const float* xr = nullptr;
  unsigned long long* br = nullptr;
  unsigned long long gt = 0, nan = 0;
  for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const int ri = static_cast<int>(tile / tiles_per_row);
    const int64_t base = (tile - static_cast<int64_t>(ri) * tiles_per_row) * TILE;
    if (ri != cur) {
      if (cur >= 0) flush_row<T>(a.st[row], gt, nan);
      cur = ri;
      row = a.rows ? a.rows[ri] : ri;
      tau = key_to_float(a.st[row].tau_key);
      xr = a.x + static_cast<int64_t>(row) * a.ld;
      br = a.buf + static_cast<int64_t>(row) * a.M;
    }
    float4 v[U];
    uint64_t valid = ~0ull;
    if (base + TILE <= a.n) {
      const float4* p = reinterpret_cast<const float4*>(xr + base) + threadIdx.x;
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = ld_stream(p + u * T);
    } else {
      valid = 0;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t i = base + (static_cast<int64_t>(u) * T + threadIdx.x) * 4 + c;
          const bool ok = i < a.n;
          f[c] = ok ? xr[i] : -INFINITY;
          valid |= static_cast<uint64_t>(ok) << (u * 4 + c);
        }
        v[u] = make_float4(f[0], f[1], f[2], f[3]);
      }
    }
    float m = max_nan(max_nan(v[0].x, v[0].y), max_nan(v[0].z, v[0].w));
#pragma unroll
    for (int u = 1; u < U; ++u) m = max_nan(m, max_nan(max_nan(v[u].x, v[u].y), max_nan(v[u].z, v[u].w)));
    // Masked lanes hold -inf; they can reach the slow path only when tau is
    // -inf, and `valid` keeps them out of every count there.
    const bool hit = !(m < tau);
    if (__syncthreads_or(hit)) tile_slow<T, U>(v, valid, hit, tau, base, a.st[row], br, a.M, gt, nan, s_warp, &s_gbase);
  }
  if (cur >= 0) flush_row<T>(a.st[row], gt, nan);
}

constexpr int FT = 256;
constexpr int FU = 16;

}  // namespace

int filter_default_grid(int sms) {
  int per = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_filter<FT, FU>, FT, 0);
  if (per < 1) per = 1;
  return sms * per;
}

void launch_filter(const FilterArgs& a, cudaStream_t stream) {
  const int64_t TILE = static_cast<int64_t>(FT) * 4 * FU;
  const int64_t tiles = ((a.n + TILE - 1) / TILE) * a.nrows;
  int grid = a.grid;
  if (tiles < grid) grid = static_cast<int>(tiles);
  if (grid < 1) grid = 1;
  ++launch_count();
  k_filter<FT, FU><<<grid, FT, 0, stream>>>(a);
}

}  // namespace profk
