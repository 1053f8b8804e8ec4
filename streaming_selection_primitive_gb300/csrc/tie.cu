// The tie exit of the run-time check (an addition that keeps the output
// exact; it sits in the check of "Prof-K: Probabilistic One-Pass Filtering
// for Efficient Top-k Selection", Section 3, stage 4).  When the filter finds
// R > M elements >= tau but only R_gt < k elements > tau, tau is exactly the
// k-th largest value, and the top-k is every x > tau plus the need = k - R_gt
// lowest-index copies of tau.
//
//  1. `k_tie_count`, one streaming pass like the filter's (persistent grid,
//     warp tiles of 128-bit loads): every x > tau is appended to the row's
//     output keys (fewer than k of them), and the copies of tau are counted
//     per block of 2^TIE_BLOCK_LOG2 elements (one atomic per warp tile that has any);
//  2. `k_tie_cut`, one CTA per row: the exclusive prefix of the block counts
//     and the block in which the running count of tau reaches `need` (the
//     scan stops there);
//  3. `k_tie_take`, CTAs striding over the blocks up to that one: a block's
//     copies of tau in index order (one block-wide scan of its 16K
//     elements), the first `need` of the row written after the x > tau keys.
// Only the blocks up to the cut that hold copies of tau are read a second time.
//
// After a filter pass that ran with its tie bookkeeping, step 1 is not a
// pass over the input: the filter has counted the copies of tau per block
// and appended every x > tau that its full buffer dropped, so
//  1'. `k_tie_gather` adds the buffer's own x > tau to those, and the cut
//      checks that they are R_gt in all.
#include "kernels.h"

namespace profk {

struct TieCtl {
  unsigned gt_count;       // x > tau appended so far
  unsigned pad;
  long long cut;           // last block that holds a taken copy of tau
  unsigned long long need;
};

namespace {

constexpr int TC_THREADS = 256;
constexpr int TC_U = 8;                        // float4 per lane per warp tile
constexpr int64_t TC_WT = 32 * 4 * TC_U;       // elements per warp tile
constexpr int TT_THREADS = 256;
constexpr int TT_F4 = 16;                      // float4 per thread per segment
constexpr int64_t TT_SEG = TT_THREADS * TT_F4 * 4;  // 16K elements

__device__ __forceinline__ float4 ld_stream4(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float comp(const float4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

__global__ void __launch_bounds__(TC_THREADS) k_tie_count(TieArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (TC_THREADS / 32);
  const int64_t tiles_per_row = (a.n + TC_WT - 1) / TC_WT;
  const int64_t total = tiles_per_row * a.nrows;
  for (int64_t tile = static_cast<int64_t>(blockIdx.x) * (TC_THREADS / 32) + (threadIdx.x >> 5); tile < total;
       tile += nwarps) {
    const int ri = static_cast<int>(tile / tiles_per_row);
    const int row = a.rows ? a.rows[ri] : ri;
    const int64_t base = (tile - static_cast<int64_t>(ri) * tiles_per_row) * TC_WT;
    const float tau = key_to_float(a.st[row].tau_key);
    const float* xr = a.x + static_cast<int64_t>(row) * a.ld;
    float4 v[TC_U];
    if (base + TC_WT <= a.n) {
      const float4* p = reinterpret_cast<const float4*>(xr + base) + lane;
#pragma unroll
      for (int u = 0; u < TC_U; ++u) v[u] = ld_stream4(p + u * 32);
    } else {
#pragma unroll
      for (int u = 0; u < TC_U; ++u) {
        float f[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t i = base + (static_cast<int64_t>(u) * 32 + lane) * 4 + c;
          f[c] = i < a.n ? xr[i] : __int_as_float(0x7fc00000);  // NaN: neither == nor > tau
        }
        v[u] = make_float4(f[0], f[1], f[2], f[3]);
      }
    }
    unsigned eq = 0, gt = 0;
#pragma unroll
    for (int u = 0; u < TC_U; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        eq += comp(v[u], c) == tau;
        gt += comp(v[u], c) > tau;
      }
    unsigned eq_w = eq;
    for (int o = 16; o >= 1; o >>= 1) eq_w += __shfl_xor_sync(FULL_MASK, eq_w, o);
    if (lane == 0 && eq_w) atomicAdd(a.block_eq + static_cast<int64_t>(row) * a.nblocks + (base >> TIE_BLOCK_LOG2), eq_w);
    if (__any_sync(FULL_MASK, gt != 0)) {
      // The x > tau of the tile go after the row's earlier ones (any order:
      // they are all in the top-k and are sorted at the end).
      unsigned incl = gt;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += t;
      }
      unsigned b0 = 0;
      if (lane == 31) b0 = atomicAdd(&a.ctl[row].gt_count, incl);
      b0 = __shfl_sync(FULL_MASK, b0, 31);
      unsigned pos = b0 + incl - gt;
      unsigned long long* out = a.sel + static_cast<int64_t>(row) * a.kstride;
#pragma unroll
      for (int u = 0; u < TC_U; ++u)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float f = comp(v[u], c);
          if (f > tau) {
            const uint32_t idx = static_cast<uint32_t>(base + (static_cast<int64_t>(u) * 32 + lane) * 4 + c);
            if (pos < static_cast<unsigned long long>(a.k)) out[pos] = cand_key(f, idx);
            ++pos;
          }
        }
    }
  }
}

// The buffer's keys above tau (its first min(R_ge, M) entries), appended to
// the row's tie list after those the filter appended: CTAs (blockIdx.x) take
// strided runs of the buffer of row blockIdx.y, one atomic per warp and run.
constexpr int TG_THREADS = 256;

__global__ void __launch_bounds__(TG_THREADS) k_tie_gather(TieArgs a, const unsigned long long* buf, int64_t M) {
  pdl_trigger();
  pdl_wait();
  const int row = launch_row(a.rows);
  RowState& S = a.st[row];
  const uint32_t tkey = S.tau_key;
  const int64_t len = S.R_ge < static_cast<unsigned long long>(M) ? static_cast<int64_t>(S.R_ge) : M;
  const unsigned long long* br = buf + static_cast<int64_t>(row) * M;
  unsigned long long* out = a.sel + static_cast<int64_t>(row) * a.kstride;
  const int lane = threadIdx.x & 31;
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * TG_THREADS; i0 < len;
       i0 += static_cast<int64_t>(gridDim.x) * TG_THREADS) {  // uniform across the warp
    const int64_t i = i0 + threadIdx.x;
    const unsigned long long key = i < len ? br[i] : 0ull;
    const bool take = i < len && static_cast<uint32_t>(key >> 32) > tkey;
    const unsigned m = __ballot_sync(FULL_MASK, take);
    if (m == 0) continue;
    const int lead = __ffs(m) - 1;
    unsigned b0 = 0;
    if (lane == lead) b0 = atomicAdd(&S.tie_gt, static_cast<unsigned>(__popc(m)));
    b0 = __shfl_sync(FULL_MASK, b0, lead);
    if (take) {
      const unsigned pos = b0 + __popc(m & ((1u << lane) - 1u));
      if (pos < static_cast<unsigned long long>(a.k)) out[pos] = key;
    }
  }
}

// One CTA per row: exclusive prefix of the block counts, and the cut.  With
// check_gt, the tie list must hold exactly the R_gt keys above tau (the
// filter's appended ones and the buffer's); a row where it does not is
// marked with a device error (never expected: a broken invariant).
__global__ void __launch_bounds__(1024) k_tie_cut(TieArgs a, bool check_gt) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned long long sw[33];
  __shared__ long long s_cut;
  const int row = a.rows ? a.rows[blockIdx.x] : static_cast<int>(blockIdx.x);
  RowState& S = a.st[row];
  const unsigned long long need = static_cast<unsigned long long>(a.k) - S.R_gt;
  const unsigned* be = a.block_eq + static_cast<int64_t>(row) * a.nblocks;
  unsigned long long* bp = a.block_pre + static_cast<int64_t>(row) * a.nblocks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_cut = a.nblocks - 1;
  unsigned long long carry = 0;
  for (int64_t b0 = 0; b0 < a.nblocks; b0 += 1024) {
    const int64_t b = b0 + threadIdx.x;
    const unsigned long long v = b < a.nblocks ? be[b] : 0ull;
    unsigned long long incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) sw[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const unsigned long long w = sw[lane];
      unsigned long long wi = w;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(FULL_MASK, wi, o);
        if (lane >= o) wi += t;
      }
      sw[lane] = wi - w;
      if (lane == 31) sw[32] = wi;
    }
    __syncthreads();
    const unsigned long long excl = carry + sw[warp] + incl - v;
    if (b < a.nblocks) {
      bp[b] = excl;
      if (excl < need && need <= excl + v) atomicMin(&s_cut, static_cast<long long>(b));
    }
    carry += sw[32];
    __syncthreads();
    if (carry >= need) break;  // the cut is known; later blocks are not taken
  }
  if (threadIdx.x == 0) {
    a.ctl[row].cut = s_cut;
    a.ctl[row].need = need;
    S.skip = 0;  // the refinement enqueued before the check voided this row
    if (check_gt && static_cast<unsigned long long>(atomicAdd(&S.tie_gt, 0u)) != S.R_gt) atomicOr(&S.error, 32u);
  }
}

// Block blk of a row: its copies of tau in index order, those of rank < need
// written after the row's x > tau keys (all threads of the CTA call it).
__device__ __forceinline__ void tie_take_block(const TieArgs& a, int row, int64_t blk, unsigned long long* sw) {
  // A block without copies of tau has nothing to take: only the blocks that
  // hold copies are read (for distinct values, one block however far the cut).
  if (a.block_eq[static_cast<int64_t>(row) * a.nblocks + blk] == 0) return;
  const TieCtl& c = a.ctl[row];
  RowState& S = a.st[row];
  const float tau = key_to_float(S.tau_key);
  const unsigned long long need = c.need, gt = S.R_gt;
  const float* xr = a.x + static_cast<int64_t>(row) * a.ld;
  unsigned long long* out = a.sel + static_cast<int64_t>(row) * a.kstride;
  const int64_t b_lo = blk << TIE_BLOCK_LOG2;
  const int64_t b_hi = b_lo + (int64_t(1) << TIE_BLOCK_LOG2) < a.n ? b_lo + (int64_t(1) << TIE_BLOCK_LOG2) : a.n;
  unsigned long long run = a.block_pre[static_cast<int64_t>(row) * a.nblocks + blk];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t s0 = b_lo; s0 < b_hi && run < need; s0 += TT_SEG) {
    // Thread t takes the contiguous elements [s0 + 64 t, s0 + 64 t + 64).
    const int64_t e0 = s0 + static_cast<int64_t>(threadIdx.x) * (TT_F4 * 4);
    uint64_t m = 0;
    if (e0 + TT_F4 * 4 <= b_hi) {
      const float4* p = reinterpret_cast<const float4*>(xr + e0);
#pragma unroll
      for (int q = 0; q < TT_F4; ++q) {
        const float4 v = ld_stream4(p + q);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) m |= static_cast<uint64_t>(comp(v, cc) == tau) << (q * 4 + cc);
      }
    } else {
      for (int q = 0; q < TT_F4 * 4; ++q)
        if (e0 + q < b_hi) m |= static_cast<uint64_t>(xr[e0 + q] == tau) << q;
    }
    const unsigned long long v = static_cast<unsigned long long>(__popcll(m));
    unsigned long long incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) sw[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const unsigned long long w = lane < TT_THREADS / 32 ? sw[lane] : 0ull;
      unsigned long long wi = w;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(FULL_MASK, wi, o);
        if (lane >= o) wi += t;
      }
      if (lane < TT_THREADS / 32) sw[lane] = wi - w;
      if (lane == 31) sw[TT_THREADS / 32] = wi;
    }
    __syncthreads();
    unsigned long long r = run + sw[warp] + incl - v;
    while (m && r < need) {
      const int q = __ffsll(static_cast<long long>(m)) - 1;
      m &= m - 1;
      out[gt + r] = cand_key(tau, static_cast<uint32_t>(e0 + q));
      ++r;
    }
    run += sw[TT_THREADS / 32];
    __syncthreads();
  }
}

// CTAs striding over the blocks (blockIdx.x, ...) of a row (blockIdx.y) up
// to the cut: a block's copies of tau in index order, those of rank < need
// written after the row's x > tau keys.
__global__ void __launch_bounds__(TT_THREADS) k_tie_take(TieArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned long long sw[TT_THREADS / 32 + 1];
  const int row = launch_row(a.rows);
  const TieCtl& c = a.ctl[row];
  const int64_t cut = c.cut;
  for (int64_t blk = blockIdx.x; blk <= cut; blk += gridDim.x) tie_take_block(a, row, blk, sw);
}

}  // namespace

// CTAs of the take per row: the blocks, at most two per SM (they stride).
unsigned take_ctas(int64_t nblocks) {
  const int64_t cap = 2 * static_cast<int64_t>(sms());
  return static_cast<unsigned>(nblocks < cap ? (nblocks > 0 ? nblocks : 1) : cap);
}

int64_t tie_blocks(int64_t n) { return (n + (int64_t(1) << TIE_BLOCK_LOG2) - 1) >> TIE_BLOCK_LOG2; }

size_t tie_ctl_bytes() { return sizeof(TieCtl); }

cudaError_t launch_tie_take(const TieArgs& a, int filter_grid, cudaStream_t stream) {
  // The counters start at zero: the per-row control blocks and block counts.
  cudaError_t e = cudaMemsetAsync(a.ctl, 0, sizeof(TieCtl) * a.total_rows, stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(a.block_eq, 0, sizeof(unsigned) * a.nblocks * a.total_rows, stream);
  if (e != cudaSuccess) return e;
  const int64_t warp_tiles = ((a.n + TC_WT - 1) / TC_WT) * a.nrows;
  int64_t ctas = (warp_tiles + TC_THREADS / 32 - 1) / (TC_THREADS / 32);
  if (ctas > filter_grid) ctas = filter_grid;
  if (ctas < 1) ctas = 1;
  launch_kernel(k_tie_count, dim3(static_cast<unsigned>(ctas)), TC_THREADS, 0, stream, a);
  launch_kernel(k_tie_cut, dim3(static_cast<unsigned>(a.nrows)), 1024, 0, stream, a, false);
  launch_kernel(k_tie_take, dim3(take_ctas(a.nblocks), static_cast<unsigned>(a.nrows)), TT_THREADS, 0, stream, a);
  return cudaGetLastError();
}

cudaError_t launch_tie_after_filter(const TieArgs& a, const unsigned long long* buf, int64_t M,
                                    cudaStream_t stream) {
  int64_t runs = (M + TG_THREADS - 1) / TG_THREADS;  // one key per thread: one round of atomics
  if (runs > 1024) runs = 1024;
  if (runs < 1) runs = 1;
  launch_kernel(k_tie_gather, dim3(static_cast<unsigned>(runs), static_cast<unsigned>(a.nrows)), TG_THREADS, 0,
                stream, a, buf, M);
  launch_kernel(k_tie_cut, dim3(static_cast<unsigned>(a.nrows)), 1024, 0, stream, a, true);
  launch_kernel(k_tie_take, dim3(take_ctas(a.nblocks), static_cast<unsigned>(a.nrows)), TT_THREADS, 0, stream, a);
  return cudaGetLastError();
}

}  // namespace profk
