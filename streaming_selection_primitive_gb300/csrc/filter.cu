// Step 3 of Prof-K, the filter pass ("Prof-K: Probabilistic One-Pass Filtering
// for Efficient Top-k Selection", Section 3, stage 3, and Appendix C "The
// Filter Kernel"): stream x once, count R = |{x_i >= tau}| exactly and append
// the passers to a buffer of capacity M.
//
// GB300 design.  The pass is a pure HBM read stream, so the kernel keeps as
// many 16-byte loads in flight as the memory system wants and does almost
// nothing else on the common path, with no block-wide barrier after the
// start (where each CTA gathers its rows' tau into shared memory):
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
//    the counter pass M it only counts the rest, per lane (no mask, scan,
//    atomic or store), so inputs that overflow the buffer, such as heavily
//    tied ones whose check takes the tie exit, stream at full rate;
//  * NaNs are counted only on a lane whose maximum is NaN;
//  * R_gt, the NaN count and those late passers are per-lane registers,
//    reduced once per row per warp.
// A passer (v, i) is stored as the 64-bit key (ord(v) << 32) | ~i, the order
// the refinement sorts by.  Each store of passers also ORs their
// ord(v) ^ ord(tau) into the row's vdiff word (one warp reduction and one
// atomic per flush), which tells the refinement the high bits that every
// stored value shares with tau.
//
// Two loops over the tiles.  The plain one is all of the above.  With the
// tie exit's bookkeeping requested, the rows whose sample held tau more than
// once (a heavily tied top, the case in which the check may take the tie
// exit) go to a second loop.  That loop also counts the copies of tau per
// block of 2^TIE_BLOCK_LOG2 elements and appends to the row's tie list every
// x > tau that the full buffer drops.  The tie exit then needs no second
// pass over those rows.  Each loop skips the other's rows whole; keeping the
// bookkeeping out of the plain loop keeps its registers, and its speed, those
// of a kernel without it.
#include <type_traits>

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
  unsigned long long g = gt, q = nan, l = late;
  for (int o = 16; o; o >>= 1) {
    g += __shfl_down_sync(FULL_MASK, g, o);
    q += __shfl_down_sync(FULL_MASK, q, o);
    l += __shfl_down_sync(FULL_MASK, l, o);
  }
  if ((threadIdx.x & 31) == 0) {
    if (g) atomicAdd(&S.R_gt, g);
    if (q) atomicAdd(&S.nan, q);
    if (l) atomicAdd(&S.R_ge, l);
  }
  gt = 0;
  nan = 0;
  late = 0;
}

constexpr int STAGE = 128;  // staged passer keys per warp

// The L2 prefetch before tau (prefetch_first_tiles): about this many MB of
// the tiles that the warps take first, every PF_STRIDE-th of a warp's tiles.
#ifndef PROFK_FILTER_PREFETCH_MB
#define PROFK_FILTER_PREFETCH_MB 64
#endif
#ifndef PROFK_FILTER_PREFETCH_STRIDE
#define PROFK_FILTER_PREFETCH_STRIDE 2
#endif
constexpr int PF_STRIDE = PROFK_FILTER_PREFETCH_STRIDE;

// A lane's mask over its 4U elements of a warp tile: 32 bits when they fit
// (U <= 8, the shipped shape), else 64.
template <int U>
using LaneMask = std::conditional_t<(4 * U <= 32), uint32_t, uint64_t>;

__device__ __forceinline__ unsigned popc_mask(uint32_t m) { return static_cast<unsigned>(__popc(m)); }
__device__ __forceinline__ unsigned popc_mask(uint64_t m) { return static_cast<unsigned>(__popcll(m)); }

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Tie list of a row (the x > tau that the full buffer drops): one key per
// lane whose `take` is set, appended at the row's cursor with one atomic per
// warp.  All 32 lanes call it.
__device__ __forceinline__ void tie_append_one(RowState& S, unsigned long long* tl, int64_t k, bool take,
                                               unsigned long long key) {
  const unsigned m = __ballot_sync(FULL_MASK, take);
  if (m == 0) return;
  const int lane = threadIdx.x & 31, lead = __ffs(m) - 1;
  unsigned b0 = 0;
  if (lane == lead) b0 = atomicAdd(&S.tie_gt, static_cast<unsigned>(__popc(m)));
  b0 = __shfl_sync(FULL_MASK, b0, lead);
  if (take) {
    const unsigned pos = b0 + __popc(m & ((1u << lane) - 1u));
    if (pos < static_cast<unsigned long long>(k)) tl[pos] = key;
  }
}

// The same for the elements of a warp tile that bit e of each lane's mask m
// selects (element e is component e % 4 of the lane's float4 v[e / 4]).
template <int U>
__device__ __forceinline__ void tie_append_tile(RowState& S, unsigned long long* tl, int64_t k, LaneMask<U> m,
                                                const float4 (&v)[U], int64_t base) {
  if (!__any_sync(FULL_MASK, m != 0)) return;
  const int lane = threadIdx.x & 31;
  const unsigned c = popc_mask(m);
  unsigned incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += t;
  }
  unsigned b0 = 0;
  if (lane == 31) b0 = atomicAdd(&S.tie_gt, incl);
  b0 = __shfl_sync(FULL_MASK, b0, 31);
  unsigned long long pos = b0 + incl - c;
#pragma unroll
  for (int u = 0; u < U; ++u) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if ((m >> (u * 4 + q)) & 1u) {
        if (pos < static_cast<unsigned long long>(k)) {
          const int64_t idx = base + (static_cast<int64_t>(u) * 32 + lane) * 4 + q;
          tl[pos] = cand_key(comp(v[u], q), static_cast<uint32_t>(idx));
        }
        ++pos;
      }
    }
  }
}

// Moves a warp's staged keys into the buffer with one reservation; with the
// tie bookkeeping (TIE), the keys above tau (key tkey) that fall beyond M go
// to the tie list tl.  Without it the staged keys above tau are counted here
// into the lane's gt (the plain loop does not count them per tile).
template <bool TIE>
__device__ __forceinline__ void flush_stage(RowState& S, unsigned long long* stage, int& stage_n,
                                            unsigned long long* br, int64_t M, bool& over, unsigned long long* tl,
                                            int64_t k, uint32_t tkey, unsigned long long& gt) {
  if (stage_n == 0) return;
  const int lane = threadIdx.x & 31;
  unsigned long long gbase = 0;
  if (lane == 0) gbase = atomicAdd(&S.R_ge, static_cast<unsigned long long>(stage_n));
  gbase = __shfl_sync(FULL_MASK, gbase, 0);
  __syncwarp();
  uint32_t dv = 0;  // the bits where these values differ from tau's
  for (int j = lane; j < stage_n; j += 32) {
    const unsigned long long key = stage[j];
    if (gbase + j < static_cast<unsigned long long>(M)) br[gbase + j] = key;
    dv |= static_cast<uint32_t>(key >> 32) ^ tkey;
    if constexpr (!TIE) gt += static_cast<uint32_t>(key >> 32) > tkey;
  }
  dv = __reduce_or_sync(FULL_MASK, dv);
  if (lane == 0 && dv != 0u) atomicOr(&S.vdiff, dv);
  if (gbase + stage_n > static_cast<unsigned long long>(M)) {
    over = true;
    if constexpr (TIE) {
      for (int j0 = 0; j0 < stage_n; j0 += 32) {
        const int j = j0 + lane;
        const unsigned long long key = j < stage_n ? stage[j] : 0ull;
        tie_append_one(S, tl, k, j < stage_n && gbase + j >= static_cast<unsigned long long>(M) &&
                                     static_cast<uint32_t>(key >> 32) > tkey,
                       key);
      }
    }
  }
  stage_n = 0;
  __syncwarp();
}

// What a warp needs at each change of row, in one word: ord(tau) (bits
// 0-31), whether the row's sample held tau twice or more (bit 32: the
// bookkeeping loop's row), whether an earlier attempt settled it (bit 33) and
// the storage row (bits 34-63).  The kernel gathers the words of its rows
// into shared memory once per CTA (one round trip), so that a row change
// costs a shared-memory read rather than two dependent L2 loads; with many
// rows a warp changes row every few tiles.
constexpr int INFO_ROWS = 4096;  // rows whose words are cached (32 KB)

__device__ __forceinline__ unsigned long long row_info(const FilterArgs& a, int ri) {
  const int r = a.rows ? a.rows[ri] : ri;
  const RowState& S = a.st[r];
  return static_cast<unsigned long long>(S.tau_key) | (static_cast<unsigned long long>(S.tau_copies >= 2) << 32) |
         (static_cast<unsigned long long>(settled_before(S, a.attempt)) << 33) |
         (static_cast<unsigned long long>(r) << 34);
}

// The pass over the rows this loop takes: with the tie bookkeeping on
// (a.block_eq), the rows whose sample holds tau more than once (a heavily
// tied top, RowState::tau_copies >= 2) go to the TIE loop and the others to
// the plain one; with it off the plain loop takes every row.  A row of the
// other loop is skipped whole.
template <int T, int U, bool TIE, bool UNAL>
__device__ __forceinline__ void filter_rows(const FilterArgs& a, unsigned long long* stage,
                                            const unsigned long long* info, int cached) {
  static_assert(!(TIE && UNAL), "the tie bookkeeping counts per aligned block");
  static_assert(4 * U <= 64, "at most 64 elements per lane");
  constexpr int64_t WT = 32 * 4 * U;  // elements per warp tile
  int stage_n = 0;  // warp-uniform
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (T / 32);
  // A row's warp tiles cover positions 0 .. n + head of the row counted from
  // the 16-byte boundary at or before it (head: the 0-3 elements between;
  // always 0 when every row is aligned); element e of the row is position
  // e + head.
  const int64_t tiles_per_row = (a.n + (UNAL ? 3 : 0) + WT - 1) / WT;
  const int64_t total = tiles_per_row * a.nrows;
  int cur = -1;
  bool active = false;  // the row `row` is this loop's and has state to flush
  int row = 0;
  float tau = 0.f;
  bool over = false;  // this warp saw the row's counter pass M
  const float* xr = nullptr;  // the row's position 0 (head elements before the row)
  int64_t head = 0;
  unsigned long long* br = nullptr;
  unsigned long long* tl = nullptr;  // the row's tie list (with the tie bookkeeping)
  unsigned* beq = nullptr;           // the row's per-block counts of tau
  uint32_t tkey = 0;
  unsigned long long gt = 0, nan = 0, late = 0;
  // The warps' tiles.  One row: warp w takes tiles w, w + nwarps, ...
  // (the whole grid sweeps the row front to back).  Several rows: each warp
  // takes one contiguous range of tiles (the rows in order), so that it
  // changes row at most a few times however short the rows are (measured:
  // 256 rows of 2^22, 0.719 -> 0.605 ms; a single 2^30 row sweeps 2.6 %
  // faster with the strided order).
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * (T / 32) + (threadIdx.x >> 5);
  const bool one = a.nrows == 1;
  const int tpr = static_cast<int>(tiles_per_row);  // at most 2^22 + 1
  const int step = one ? static_cast<int>(nwarps) : 1;
  int64_t left;  // tiles still to take
  int ri, tir;   // the tile's row (index in the launch) and its index in that row
  if (one) {
    left = wid < total ? (total - wid + nwarps - 1) / nwarps : 0;
    ri = 0;
    tir = static_cast<int>(wid);
  } else {
    const int64_t per = (total + nwarps - 1) / nwarps;
    const int64_t t0 = wid * per < total ? wid * per : total;
    left = (t0 + per < total ? t0 + per : total) - t0;
    ri = static_cast<int>(t0 / tiles_per_row);
    tir = static_cast<int>(t0 - static_cast<int64_t>(ri) * tiles_per_row);
  }
  for (; left > 0; --left, tir += step) {
    if (tir >= tpr) {  // several rows only: on into the next row
      ++ri;
      tir = 0;
    }
    const int64_t base = static_cast<int64_t>(tir) * WT;
    if (ri != cur) {
      if (active) {
        flush_stage<TIE>(a.st[row], stage, stage_n, br, a.M, over, tl, a.k, tkey, gt);
        flush_row(a.st[row], gt, nan, late);
        active = false;
      }
      cur = ri;
      const unsigned long long w = ri < cached ? info[ri] : row_info(a, ri);
      if ((a.block_eq && static_cast<bool>((w >> 32) & 1ull) != TIE) || ((w >> 33) & 1ull)) {
        // The other loop's row, or one that an earlier attempt settled: on
        // to the next row (the loop's step moves past this row's last tile).
        if (one) break;
        left -= tpr - 1 - tir;
        tir = tpr - 1;
        continue;
      }
      row = static_cast<int>(w >> 34);
      active = true;
      tkey = static_cast<uint32_t>(w);
      tau = key_to_float(tkey);
      xr = a.x + static_cast<int64_t>(row) * a.ld;
      if constexpr (UNAL) {
        head = static_cast<int64_t>((reinterpret_cast<uintptr_t>(xr) >> 2) & 3u);
        xr -= head;  // never read below the row: positions < head are masked
      }
      br = a.buf + static_cast<int64_t>(row) * a.M;
      if constexpr (TIE) {
        tl = a.tie_keys + static_cast<int64_t>(row) * a.tie_stride;
        beq = a.block_eq + static_cast<int64_t>(row) * a.nblocks;
      }
      over = false;
    }
    // The bookkeeping loop's rows are heavily tied, and other warps fill the
    // buffer long before this warp's own stage would tell it so: the row's
    // counter is read with the tile (its latency hidden by the tile's loads).
    unsigned long long rge = 0;
    if constexpr (TIE) {
      if (!over && lane == 0) rge = ld_relaxed_u64(&a.st[row].R_ge);
    }
    float4 v[U];
    using LM = LaneMask<U>;
    LM valid = ~LM(0);
    // A full tile holds only the row's elements; the row's element index of
    // the tile's position 0 is ebase.
    auto full_tile = [&]() { return UNAL ? base >= head && base + WT <= a.n + head : base + WT <= a.n; };
    const int64_t ebase = UNAL ? base - head : base;
    if (full_tile()) {
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
          const bool ok = UNAL ? i >= head && i < a.n + head : i < a.n;
          f[c] = ok ? xr[i] : -INFINITY;
          valid |= static_cast<LM>(ok) << (u * 4 + c);
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
    if (hit && m != m) {  // a NaN among the lane's values (the max propagates it)
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float f = comp(v[u], c);
          nan += (((valid >> (u * 4 + c)) & 1u) && f != f);
        }
    }
    // Copies of tau in this tile (per lane), added to the block's counter.
    auto count_ties = [&](unsigned eq) {
      if constexpr (TIE) {
        if (__any_sync(FULL_MASK, eq != 0)) {
          unsigned w = eq;
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) w += __shfl_xor_sync(FULL_MASK, w, o);
          if (lane == 0 && w) atomicAdd(beq + (ebase >> TIE_BLOCK_LOG2), w);  // aligned rows: ebase = base
        }
      }
    };
    // Per lane: the elements >= tau and those > tau (the rest of ge are
    // copies of tau); ok: element e of the lane is in the row.
    auto masks = [&](LM& ge, LM& gtm) {
      ge = 0;
      gtm = 0;
      if (!hit) return;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (mu[u] < tau) continue;  // no passer and no NaN among these four
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int e = u * 4 + c;
          const float f = comp(v[u], c);
          const bool ok = (valid >> e) & 1u;
          ge |= static_cast<LM>(ok && f >= tau) << e;
          gtm |= static_cast<LM>(ok && f > tau) << e;
        }
      }
    };
    // The elements >= tau alone (the plain loop counts the x > tau among the
    // staged keys when it flushes them).
    auto ge_mask = [&]() {
      LM ge = 0;
      if (!hit) return ge;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (mu[u] < tau) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int e = u * 4 + c;
          ge |= static_cast<LM>(((valid >> e) & 1u) && comp(v[u], c) >= tau) << e;
        }
      }
      return ge;
    };
    auto gt_count = [&]() {
      LM ge, gtm;
      masks(ge, gtm);
      return popc_mask(gtm);
    };
    if constexpr (TIE) {
      if (!over && __shfl_sync(FULL_MASK, rge, 0) >= static_cast<unsigned long long>(a.M)) over = true;
    }
    if (over) {
      // The row's buffer is full: only the counts are left (per lane), and
      // with the bookkeeping the x > tau (those rarely exist when the tie exit
      // applies).  A full tile is counted without masks or branches.
      unsigned cge = 0, cgt = 0;
      if (full_tile()) {
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float f = comp(v[u], c);
            cge += f >= tau;
            cgt += f > tau;
          }
      } else {
        LM ge, gtm;
        masks(ge, gtm);
        cge = popc_mask(ge);
        cgt = popc_mask(gtm);
      }
      late += cge;
      gt += cgt;
      count_ties(cge - cgt);
      if constexpr (TIE) {
        if (__any_sync(FULL_MASK, cgt != 0)) {
          LM ge, gtm;
          masks(ge, gtm);
          tie_append_tile<U>(a.st[row], tl, a.k, gtm, v, ebase);
        }
      }
      continue;
    }
    LM ge, gtm = 0;
    if constexpr (TIE) {
      masks(ge, gtm);
      gt += popc_mask(gtm);
      count_ties(popc_mask(ge) - popc_mask(gtm));
    } else {
      ge = ge_mask();
    }
    // With the tie bookkeeping: this tile's x > tau that the buffer does not
    // keep, appended to the row's tie list at the end of the tile.
    LM dropm = 0;
    {
      // The lane's passers go after those of the lanes below it: with at
      // most one per lane (the usual case, even for large k) two ballots
      // give every lane its place, otherwise a warp scan of the counts.
      const unsigned cnt = popc_mask(ge);
      const unsigned some = __ballot_sync(FULL_MASK, cnt != 0);
      unsigned excl, tot;
      if (!__any_sync(FULL_MASK, cnt > 1)) {
        excl = static_cast<unsigned>(__popc(some & ((1u << lane) - 1u)));
        tot = static_cast<unsigned>(__popc(some));
      } else {
        unsigned incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned t = __shfl_up_sync(FULL_MASK, incl, o);
          if (lane >= o) incl += t;
        }
        excl = incl - cnt;
        tot = __shfl_sync(FULL_MASK, incl, 31);
      }
      if (tot != 0 && tot <= STAGE) {
        if (stage_n + static_cast<int>(tot) > STAGE)
          flush_stage<TIE>(a.st[row], stage, stage_n, br, a.M, over, tl, a.k, tkey, gt);
        if (over) {  // the flush filled the buffer: this tile's passers are only counted
          if (lane == 0) late += tot;
          if constexpr (TIE)
            dropm = gtm;
          else
            gt += gt_count();
        } else {
          if (cnt) {
            // Each group's passers in turn (usually one): the component by
            // its bit, then the key.
            int pos = stage_n + static_cast<int>(excl);
#pragma unroll
            for (int u = 0; u < U; ++u) {
              unsigned nib = static_cast<unsigned>(ge >> (u * 4)) & 15u;
              while (nib) {
                const int c = __ffs(nib) - 1;
                nib &= nib - 1u;
                const int64_t idx = ebase + (static_cast<int64_t>(u) * 32 + lane) * 4 + c;
                stage[pos++] = cand_key(comp(v[u], c), static_cast<uint32_t>(idx));
              }
            }
          }
          stage_n += static_cast<int>(tot);
          __syncwarp();
        }
      } else if (tot > STAGE) {
        // More passers in this tile than a stage holds: reserve for the tile alone.
        unsigned long long gbase = 0;
        if (lane == 0) gbase = atomicAdd(&a.st[row].R_ge, static_cast<unsigned long long>(tot));
        gbase = __shfl_sync(FULL_MASK, gbase, 0);
        if constexpr (!TIE) gt += gt_count();
        if (gbase + tot > static_cast<unsigned long long>(a.M)) over = true;
        unsigned long long pos = gbase + excl;
        uint32_t dv = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int e = u * 4 + c;
            if ((ge >> e) & 1u) {
              dv |= ord_key(comp(v[u], c)) ^ tkey;
              if (pos < static_cast<unsigned long long>(a.M)) {
                const int64_t idx = ebase + (static_cast<int64_t>(u) * 32 + lane) * 4 + c;
                br[pos] = cand_key(comp(v[u], c), static_cast<uint32_t>(idx));
              } else if constexpr (TIE) {
                dropm |= gtm & (LM(1) << e);
              }
              ++pos;
            }
          }
        }
        dv = __reduce_or_sync(FULL_MASK, dv);
        if (lane == 0 && dv != 0u) atomicOr(&a.st[row].vdiff, dv);
      }
    }
    if constexpr (TIE) tie_append_tile<U>(a.st[row], tl, a.k, dropm, v, ebase);
  }
  if (active) {
    flush_stage<TIE>(a.st[row], stage, stage_n, br, a.M, over, tl, a.k, tkey, gt);
    flush_row(a.st[row], gt, nan, late);
  }
}

__device__ __forceinline__ void prefetch_l2(const char* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Before tau is known.  With programmatic dependent launch the filter's
// first CTAs become resident beside the sampler, whose work is a chain of
// dependent steps that leaves HBM nearly idle; those CTAs (the first
// pf_ctas) ask L2 for pf_tiles warp tiles of every warp of the grid, one
// bulk prefetch per tile: every PF_STRIDE-th of the tiles filter_rows hands
// the warp first, so that in the pass's first rounds each warp alternates a
// tile on chip with one from HBM and HBM stays busy.  A prefetch is a hint:
// nothing waits for it, and it covers only the row's own elements (rounded
// inward to 16 bytes).  Measured on 2^26 inputs: 3-5 us less per call.
template <int T, int U, bool UNAL>
__device__ __forceinline__ void prefetch_first_tiles(const FilterArgs& a) {
  constexpr int64_t WT = 32 * 4 * U;
  const int64_t C = a.pf_ctas;
  if (static_cast<int64_t>(blockIdx.x) >= C) return;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (T / 32);
  const int64_t tpr = (a.n + (UNAL ? 3 : 0) + WT - 1) / WT;
  const int64_t total = tpr * a.nrows;
  const int64_t per = (total + nwarps - 1) / nwarps;
  const int64_t F = a.pf_tiles;
  const int64_t w0 = blockIdx.x * nwarps / C, w1 = (blockIdx.x + 1) * nwarps / C;
  const int64_t items = (w1 - w0) * F;
  for (int64_t it = threadIdx.x; it < items; it += T) {
    const int64_t w = w0 + it / F, f = it % F;
    int64_t tile;
    if (a.nrows == 1) {
      tile = w + f * PF_STRIDE * nwarps;
    } else {
      if (f * PF_STRIDE >= per) continue;
      tile = w * per + f * PF_STRIDE;
    }
    if (tile >= total) continue;
    const int64_t ri = tile / tpr, tir = tile - ri * tpr;
    const int r = a.rows ? a.rows[ri] : static_cast<int>(ri);
    const uintptr_t row0 = reinterpret_cast<uintptr_t>(a.x + static_cast<int64_t>(r) * a.ld);
    const uintptr_t row1 = row0 + static_cast<uintptr_t>(a.n) * 4u;
    const uintptr_t head = UNAL ? ((row0 >> 2) & 3u) : 0u;
    uintptr_t lo = row0 - head * 4u + static_cast<uintptr_t>(tir) * WT * 4u;
    uintptr_t hi = lo + WT * 4u;
    const uintptr_t first = (row0 + 15u) & ~uintptr_t(15), last = row1 & ~uintptr_t(15);
    if (lo < first) lo = first;
    if (hi > last) hi = last;
    if (hi > lo) prefetch_l2(reinterpret_cast<const char*>(lo), static_cast<unsigned>(hi - lo));
  }
}

// UNAL: some row is off the 16-byte grid (its own instantiation, so that the
// aligned kernel's code is that of a kernel without the head).
template <int T, int U, bool UNAL>
__global__ void __launch_bounds__(T, 3) k_filter(FilterArgs a) {
  if (a.pf_tiles) prefetch_first_tiles<T, U, UNAL>(a);
  pdl_wait();
  __shared__ unsigned long long s_stage[T / 32][STAGE];
  extern __shared__ unsigned long long s_info[];  // the first `cached` rows' words (row_info)
  const int cached = a.nrows < INFO_ROWS ? a.nrows : INFO_ROWS;
  for (int i = threadIdx.x; i < cached; i += T) s_info[i] = row_info(a, i);
  __syncthreads();
  unsigned long long* stage = s_stage[threadIdx.x >> 5];
  filter_rows<T, U, false, UNAL>(a, stage, s_info, cached);
  if constexpr (!UNAL) {
    if (a.block_eq) filter_rows<T, U, true, false>(a, stage, s_info, cached);
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
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_filter<FT, FU, false>, FT, 0);
  if (per < 1) per = 1;
  return sms * per;
}

void launch_filter(const FilterArgs& args, cudaStream_t stream) {
  FilterArgs a = args;
  // Some row off the 16-byte grid: x itself, or a row stride that is not a
  // multiple of 4 elements whenever a row other than the first can be among
  // those listed (several rows, or a row list, which may hold one later row).
  const bool unaligned = (reinterpret_cast<uintptr_t>(a.x) & 15u) != 0 ||
                         ((a.ld & 3) != 0 && (a.nrows > 1 || a.rows != nullptr));
  if (unaligned) a.block_eq = nullptr;  // the tie bookkeeping counts per aligned block
  const int64_t WT = 32 * 4 * FU;
  const int64_t warp_tiles = ((a.n + (unaligned ? 3 : 0) + WT - 1) / WT) * a.nrows;
  const int64_t ctas = (warp_tiles + FT / 32 - 1) / (FT / 32);
  int grid = a.grid;
  if (ctas < grid) grid = static_cast<int>(ctas);
  if (grid < 1) grid = 1;
  // The L2 prefetch before tau (prefetch_first_tiles): the first CTAs, one
  // per SM (those that fit beside the sampler's), warm about
  // PROFK_FILTER_PREFETCH_MB of the tiles that every warp takes first
  // (every PF_STRIDE-th of them).
  const int64_t nwarps = static_cast<int64_t>(grid) * (FT / 32);
  const int64_t per_warp = (warp_tiles + nwarps - 1) / nwarps;
  int64_t pf = (static_cast<int64_t>(PROFK_FILTER_PREFETCH_MB) << 20) / (nwarps * WT * 4);
  if (pf > (per_warp + PF_STRIDE - 1) / PF_STRIDE) pf = (per_warp + PF_STRIDE - 1) / PF_STRIDE;
  a.pf_tiles = static_cast<int>(pf);
  a.pf_ctas = sms() < grid ? sms() : grid;
  const size_t info = sizeof(unsigned long long) * static_cast<size_t>(a.nrows < INFO_ROWS ? a.nrows : INFO_ROWS);
  if (unaligned)
    launch_kernel(k_filter<FT, FU, true>, grid, FT, info, stream, a);
  else
    launch_kernel(k_filter<FT, FU, false>, grid, FT, info, stream, a);
}

}  // namespace profk
