// Exact selection machinery shared by Prof-K's steps 2 and 4 and by the exact
// fallback ("Prof-K: Probabilistic One-Pass Filtering for Efficient Top-k
// Selection", Section 3, stages 2 and 4).
//
// * Radix selection of the r-th largest key, most significant digit first:
//   one launch per 11/11/10-bit digit.  Every block histograms the keys that
//   match the prefix resolved so far; the last block to finish (a ticket
//   counter, no spin-wait) picks the digit that holds rank r, narrows the
//   prefix and clears the histogram for the next launch.  Composite
//   (value, index) keys are distinct, so six digits give the exact k-th key;
//   the selection stops early once a whole bucket falls inside the top-k.
// * Compaction of the keys >= the selected threshold (exactly k of them).
// * Bitonic sort of the k keys (descending) and emission of values/indices.
#include <algorithm>

#include "kernels.h"
#include "blocksort.cuh"

namespace profk {
namespace {

constexpr int SEL_THREADS = 512;
constexpr int SMALL_SORT_MAX = 8192;    // keys sorted by one CTA in shared memory
constexpr int CHUNK = 8192;             // shared-memory chunk of the multi-CTA sort
constexpr int SORT_THREADS = 1024;

struct SrcSample {
  static constexpr bool kFloat = false;
  const uint32_t* k;
  int64_t stride, len;
  __device__ int64_t length(const RowState&) const { return len; }
  __device__ uint64_t key(int row, int64_t i) const {
    return static_cast<uint64_t>(k[row * stride + i]) << 32;
  }
};

struct SrcInput {
  static constexpr bool kFloat = true;
  const float* x;
  int64_t ld, n;
  bool vec4;  // every row starts on a 16-byte boundary (x aligned; ld % 4 == 0 or one row)
  __device__ int64_t length(const RowState&) const { return n; }
  __device__ uint64_t key(int row, int64_t i) const {
    return cand_key(x[row * ld + i], static_cast<uint32_t>(i));
  }
};

struct SrcBuffer {
  static constexpr bool kFloat = false;
  const unsigned long long* b;
  int64_t stride, cap;
  __device__ int64_t length(const RowState& s) const {
    return s.R_ge < static_cast<unsigned long long>(cap) ? static_cast<int64_t>(s.R_ge) : cap;
  }
  __device__ uint64_t key(int row, int64_t i) const { return b[row * stride + i]; }
};

__global__ void k_sel_init(RowState* st, const int* rows, unsigned long long rank) {
  pdl_trigger();
  pdl_wait();
  const int row = rows ? rows[blockIdx.x] : static_cast<int>(blockIdx.x);
  RowState& S = st[row];
  for (int b = threadIdx.x; b < HIST_BINS; b += blockDim.x) S.hist[b] = 0;
  if (threadIdx.x == 0) {
    S.sel_prefix = 0;
    S.sel_rank = rank;
    S.sel_above = 0;
    S.sel_bucket = 0;
    S.sel_thresh = 0;
    S.sel_nan = 0;
    S.sel_bits = 0;
    S.sel_done = 0;
    S.done_blocks = 0;
    S.compact_count = 0;
    S.skip = 0;
  }
}

__global__ void k_tie_init(RowState* st, const int* rows, unsigned long long k) {
  pdl_trigger();
  pdl_wait();
  const int row = rows ? rows[blockIdx.x] : static_cast<int>(blockIdx.x);
  RowState& S = st[row];
  for (int b = threadIdx.x; b < HIST_BINS; b += blockDim.x) S.hist[b] = 0;
  if (threadIdx.x == 0) {
    S.sel_prefix = S.tau_key;
    S.sel_above = S.R_gt;
    S.sel_rank = k - S.R_gt;  // 1 <= rank because R_gt < k on this path
    S.sel_bucket = 0;
    S.sel_thresh = 0;
    S.sel_nan = 0;
    S.sel_bits = 32;
    S.sel_done = 0;
    S.done_blocks = 0;
    S.compact_count = 0;
    S.skip = 0;
  }
}

__global__ void k_store_tau(RowState* st, const int* rows) {
  pdl_trigger();
  pdl_wait();
  const int row = rows ? rows[blockIdx.x] : static_cast<int>(blockIdx.x);
  if (threadIdx.x == 0) st[row].tau_key = static_cast<uint32_t>(st[row].sel_prefix);
}

// Block-wide exclusive scan of one u64 per thread (thread order).
__device__ __forceinline__ unsigned long long block_excl_scan(unsigned long long v, unsigned long long* sw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned long long incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sw[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = lane < nw ? sw[lane] : 0ull;
    unsigned long long wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(FULL_MASK, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < nw) sw[lane] = wi - w;
  }
  __syncthreads();
  return sw[warp] + incl - v;
}

template <class Src>
__global__ void __launch_bounds__(SEL_THREADS) k_radix_pass(Src src, RowState* st, const int* rows, int shift,
                                                           int width, int final_shift, int value_only,
                                                           int count_nan) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned h[HIST_BINS];
  __shared__ unsigned long long sw[32];
  __shared__ unsigned s_nan;
  __shared__ int s_last;
  const int row = launch_row(rows);
  RowState& S = st[row];
  if (S.sel_done) return;
  const unsigned long long prefix = S.sel_prefix;
  const int bits = S.sel_bits;
  const int hi_shift = shift + width;
  const unsigned nb = 1u << width;
  for (unsigned b = threadIdx.x; b < nb; b += blockDim.x) h[b] = 0;
  if (threadIdx.x == 0) s_nan = 0;
  __syncthreads();
  const int64_t len = src.length(S);
  const int lane = threadIdx.x & 31;
  unsigned nan_local = 0;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  auto count_key = [&](uint64_t key, bool valid) {
    if (Src::kFloat && count_nan && valid && key_is_nan(static_cast<uint32_t>(key >> 32))) ++nan_local;
    const bool match = valid && (bits == 0 || (key >> hi_shift) == prefix);
    hist_add(h, static_cast<uint32_t>(key >> shift) & (nb - 1), match);
  };
  int64_t head = 0;  // elements counted by the vector loop
  if constexpr (Src::kFloat) {
    if (src.vec4) {
    // A 16-byte aligned input row as float4, four of them per lane loaded
    // together; the tail (and unaligned rows) element by element below.
    const float4* x4 = reinterpret_cast<const float4*>(src.x + static_cast<int64_t>(row) * src.ld);
    const int64_t n4 = len / 4;
    constexpr int VU = 4;
    for (int64_t w0 = static_cast<int64_t>(blockIdx.x) * blockDim.x * VU + (threadIdx.x & ~31) * VU; w0 < n4;
         w0 += step * VU) {
      float4 v[VU];
#pragma unroll
      for (int u = 0; u < VU; ++u) {
        const int64_t q = w0 + u * 32 + lane;
        v[u] = q < n4 ? __ldcs(x4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < VU; ++u) {
        const int64_t q = w0 + u * 32 + lane;
        const bool valid = q < n4;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float f = c == 0 ? v[u].x : c == 1 ? v[u].y : c == 2 ? v[u].z : v[u].w;
          count_key(cand_key(f, static_cast<uint32_t>(4 * q + c)), valid);
        }
      }
    }
    head = n4 * 4;
    }
  }
  for (int64_t w0 = head + static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); w0 < len;
       w0 += step) {
    const int64_t i = w0 + lane;
    const bool valid = i < len;
    count_key(valid ? src.key(row, i) : 0ull, valid);
  }
  if (nan_local) atomicAdd(&s_nan, nan_local);
  __syncthreads();
  for (unsigned b = threadIdx.x; b < nb; b += blockDim.x)
    if (h[b]) atomicAdd(&S.hist[b], h[b]);
  if (threadIdx.x == 0 && s_nan) atomicAdd(&S.sel_nan, static_cast<unsigned long long>(s_nan));
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&S.done_blocks, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (unsigned b = threadIdx.x; b < nb; b += blockDim.x) h[b] = __ldcg(&S.hist[b]);
  __syncthreads();
  // Thread t owns `per` consecutive bins counted down from the top digit.
  const int per = (nb + blockDim.x - 1) / blockDim.x;
  const int top = static_cast<int>(nb) - 1 - static_cast<int>(threadIdx.x) * per;
  unsigned long long local = 0;
  for (int q = 0; q < per; ++q)
    if (top - q >= 0) local += h[top - q];
  const unsigned long long rank = S.sel_rank;  // read before any thread updates it
  const unsigned long long excl = block_excl_scan(local, sw);
  if (excl < rank && rank <= excl + local) {
    unsigned long long acc = excl;
    for (int q = 0; q < per; ++q) {
      const int b = top - q;
      if (b < 0) break;
      const unsigned long long c = h[b];
      if (rank <= acc + c) {
        const unsigned long long np = (prefix << width) | static_cast<unsigned long long>(b);
        S.sel_above += acc;
        S.sel_rank = rank - acc;
        S.sel_prefix = np;
        S.sel_bits = bits + width;
        S.sel_bucket = c;
        if (shift == final_shift || (!value_only && c == rank - acc)) {
          S.sel_done = 1;
          S.sel_thresh = np << shift;
          if (value_only) {  // the threshold of step 2, and how many keys hold it
            S.tau_key = static_cast<uint32_t>(np);
            S.tau_copies = static_cast<unsigned>(c < 0xffffffffull ? c : 0xffffffffull);
          }
        }
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
  for (unsigned b = threadIdx.x; b < nb; b += blockDim.x) S.hist[b] = 0;
  if (threadIdx.x == 0) {
    if (S.sel_bits == bits) {  // no digit was chosen
      atomicOr(&S.error, 4u);
      S.sel_done = 1;
      S.sel_thresh = ~0ull;
    }
    S.done_blocks = 0;
  }
}

template <class Src>
__global__ void __launch_bounds__(SEL_THREADS) k_compact(Src src, RowState* st, const int* rows,
                                                        unsigned long long* out, int64_t out_stride, int64_t k) {
  pdl_trigger();
  pdl_wait();
  const int row = launch_row(rows);
  RowState& S = st[row];
  if (!S.sel_done || S.skip) return;
  const unsigned long long thresh = S.sel_thresh;
  const int64_t len = src.length(S);
  const int lane = threadIdx.x & 31;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t w0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); w0 < len; w0 += step) {
    const int64_t i = w0 + lane;
    const bool valid = i < len;
    const uint64_t key = valid ? src.key(row, i) : 0ull;
    const bool sel = valid && key >= thresh;
    const unsigned m = __ballot_sync(FULL_MASK, sel);
    if (m) {
      unsigned base = 0;
      if (lane == 0) base = atomicAdd(&S.compact_count, static_cast<unsigned>(__popc(m)));
      base = __shfl_sync(FULL_MASK, base, 0);
      if (sel) {
        const unsigned pos = base + __popc(m & ((1u << lane) - 1u));
        if (pos < static_cast<unsigned long long>(k)) out[row * out_stride + pos] = key;
      }
    }
  }
}

// Writes output j of a row.  The index is checked against the row length so
// that a selection that went wrong can never read outside x; such an entry is
// written as (NaN, -1), which no valid result contains.
__device__ __forceinline__ void emit_one(const unsigned long long key, int row, int64_t j, int64_t k, const float* x,
                                         int64_t ld, int64_t n, float* out_vals, int64_t* out_idx) {
  const uint32_t idx = cand_index(key);
  if (static_cast<int64_t>(idx) < n) {
    out_idx[row * k + j] = static_cast<int64_t>(idx);
    out_vals[row * k + j] = x[row * ld + idx];
  } else {
    out_idx[row * k + j] = -1;
    out_vals[row * k + j] = __int_as_float(0x7fc00000);
  }
}

// One CTA per row: load k keys, pad to P (>= 1024) with 0 (below every real
// key), sort descending in shared memory (registers and shuffles for the
// closer compare-exchange partners), emit.  gt_first: keys [R_gt, k) of the
// row are copies of one value in ascending index order, below every key of
// [0, R_gt) (the tie step's layout), so only a prefix that covers the first
// R_gt keys is sorted (none when R_gt <= 1): its other keys are the largest
// of the ordered copies, and every key after it is smaller.
__global__ void __launch_bounds__(SORT_THREADS) k_sort_small(const unsigned long long* keys, int64_t key_stride,
                                                            int64_t k, int P, const int* rows, const float* x,
                                                            int64_t ld, int64_t n, float* out_vals,
                                                            int64_t* out_idx, const RowState* st, bool gt_first) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ unsigned long long s[];
  const int row = rows ? rows[blockIdx.x] : static_cast<int>(blockIdx.x);
  if (st && st[row].skip) return;
  const unsigned long long* kr = keys + row * key_stride;
  const int64_t count = gt_first && st ? static_cast<int64_t>(st[row].R_gt < static_cast<unsigned long long>(k)
                                                                   ? st[row].R_gt
                                                                   : static_cast<unsigned long long>(k))
                                       : k;
  int Ps = SORT_THREADS;  // the sorted prefix: a power of two >= 1024, <= P
  while (Ps < count) Ps <<= 1;
  for (int i = threadIdx.x; i < P; i += blockDim.x) s[i] = i < k ? kr[i] : 0ull;
  __syncthreads();
  if (count > 1) {
    switch (Ps / SORT_THREADS) {
      case 1: block_sort_desc<1>(s); break;
      case 2: block_sort_desc<2>(s); break;
      case 4: block_sort_desc<4>(s); break;
      default: block_sort_desc<8>(s); break;
    }
  }
  for (int j = threadIdx.x; j < k; j += blockDim.x) emit_one(s[j], row, j, k, x, ld, n, out_vals, out_idx);
}

// Multi-CTA bitonic sort (descending) of rows of P = 2^m keys.
__global__ void __launch_bounds__(SORT_THREADS) k_pad(unsigned long long* keys, int64_t key_stride, int64_t k,
                                                      int64_t P, const int* rows) {
  pdl_trigger();
  pdl_wait();
  const int row = launch_row(rows);
  for (int64_t i = k + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < P;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    keys[row * key_stride + i] = 0ull;
}

// Stages size <= `upto` (all j < CHUNK) of one CHUNK-key chunk in shared memory,
// starting at stage `from` (2 for a full local sort, or one merge stage).
__global__ void __launch_bounds__(SORT_THREADS) k_bitonic_chunk(unsigned long long* keys, int64_t key_stride,
                                                                int from, int64_t upto, const int* rows) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ unsigned long long s[];
  const int row = launch_row(rows);
  unsigned long long* kr = keys + row * key_stride + static_cast<int64_t>(blockIdx.x) * CHUNK;
  const int64_t g0 = static_cast<int64_t>(blockIdx.x) * CHUNK;
  for (int i = threadIdx.x; i < CHUNK; i += blockDim.x) s[i] = kr[i];
  __syncthreads();
  for (int64_t size = from; size <= upto; size <<= 1) {
    int64_t j = size >> 1;
    if (j >= CHUNK) j = CHUNK >> 1;
    for (; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < CHUNK; i += blockDim.x) {
        const int l = i ^ static_cast<int>(j);
        if (l > i) {
          const unsigned long long a = s[i], b = s[l];
          const bool desc = ((g0 + i) & size) == 0;
          if (desc ? (a < b) : (a > b)) {
            s[i] = b;
            s[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < CHUNK; i += blockDim.x) kr[i] = s[i];
}

__global__ void __launch_bounds__(SORT_THREADS) k_bitonic_global(unsigned long long* keys, int64_t key_stride,
                                                                 int64_t P, int64_t size, int64_t j, const int* rows) {
  pdl_trigger();
  pdl_wait();
  const int row = launch_row(rows);
  unsigned long long* kr = keys + row * key_stride;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < P;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t l = i ^ j;
    if (l > i) {
      const unsigned long long a = kr[i], b = kr[l];
      const bool desc = (i & size) == 0;
      if (desc ? (a < b) : (a > b)) {
        kr[i] = b;
        kr[l] = a;
      }
    }
  }
}

__global__ void __launch_bounds__(SORT_THREADS) k_emit(const unsigned long long* keys, int64_t key_stride, int64_t k,
                                                       const int* rows, const float* x, int64_t ld, int64_t n,
                                                       float* out_vals, int64_t* out_idx, const RowState* st) {
  pdl_trigger();
  pdl_wait();
  const int row = launch_row(rows);
  if (st && st[row].skip) return;
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < k;
       j += static_cast<int64_t>(gridDim.x) * blockDim.x)
    emit_one(keys[row * key_stride + j], row, j, k, x, ld, n, out_vals, out_idx);
}

// ---------------------------------------------------------------------------
// Step 4 in one CTA per row.  The candidates (R <= M keys) are read from L2;
// 11/11/10/11/11/10-bit MSD passes narrow the bucket that holds the k-th
// largest key.  As soon as the keys above the bucket plus the bucket itself
// fit the gather budget (at least 2k, at most ONE_OUT keys), all of them are
// gathered into shared memory, sorted descending there, and the first k are
// emitted.  The kernel is enqueued before the host has checked k <= R <= M;
// a row that fails the check is marked skip and its outputs are not touched.
constexpr int ONE_THREADS = 1024;
constexpr int ONE_OUT = 8192;    // keys gathered into shared memory (64 KB)
constexpr int ONE_MAX_K = 8192;
constexpr int64_t ONE_MAX_M = 1 << 19;

__global__ void __launch_bounds__(ONE_THREADS) k_refine_one(RefineOneArgs a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ unsigned long long s_out[];  // ONE_OUT keys
  __shared__ unsigned h[HIST_BINS];
  __shared__ unsigned long long sw[32];
  __shared__ int s_digit;
  __shared__ unsigned long long s_above, s_count;
  __shared__ unsigned s_cursor;
  const int row = a.rows ? a.rows[blockIdx.x] : static_cast<int>(blockIdx.x);
  RowState& S = a.st[row];
  const int tid = threadIdx.x;
  const unsigned long long R = S.R_ge;
  const unsigned long long k = static_cast<unsigned long long>(a.k);
  if (!(k <= R && R <= static_cast<unsigned long long>(a.M))) {
    if (tid == 0) S.skip = 1;
    return;  // block-uniform
  }
  if (tid == 0) {
    S.skip = 0;
    s_cursor = 0;
  }
  const unsigned long long* keys = a.buf + static_cast<int64_t>(row) * a.M;
  const int64_t len = static_cast<int64_t>(R);
  const unsigned long long budget = k * 2 < 2048 ? 2048 : (k * 2 > ONE_OUT ? ONE_OUT : k * 2);
  unsigned long long prefix = 0, want = k, thresh = 0, total = k;
  int bits = 0;
  const int shifts[6] = {53, 42, 32, 21, 10, 0}, widths[6] = {11, 11, 10, 11, 11, 10};
#pragma unroll 1
  for (int p = 0; p < 6; ++p) {
    const int shift = shifts[p], width = widths[p];
    const int nb = 1 << width, hs = shift + width;
    for (int b = tid; b < nb; b += ONE_THREADS) h[b] = 0;
    if (tid == 0) {
      s_digit = 0;
      s_above = 0;
      s_count = 0;
    }
    __syncthreads();
    for (int64_t base = 0; base < len; base += 8 * ONE_THREADS) {
      unsigned long long kk[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t i = base + static_cast<int64_t>(j) * ONE_THREADS + tid;
        kk[j] = i < len ? __ldcg(keys + i) : 0ull;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t i = base + static_cast<int64_t>(j) * ONE_THREADS + tid;
        const bool m = i < len && (bits == 0 || (kk[j] >> hs) == prefix);
        hist_add(h, static_cast<uint32_t>(kk[j] >> shift) & (nb - 1), m);
      }
    }
    __syncthreads();
    // Bins counted down from the top: thread t owns nb / 1024 of them.
    const int per = nb / ONE_THREADS;
    const int top = nb - 1 - tid * per;
    unsigned long long local = 0;
    for (int q = 0; q < per; ++q) local += h[top - q];
    const unsigned long long excl = block_excl_scan(local, sw);
    if (excl < want && want <= excl + local) {
      unsigned long long acc = excl;
      for (int q = 0; q < per; ++q) {
        const unsigned long long c = h[top - q];
        if (want <= acc + c) {
          s_digit = top - q;
          s_above = acc;
          s_count = c;
          break;
        }
        acc += c;
      }
    }
    __syncthreads();
    prefix = (prefix << width) | static_cast<unsigned long long>(s_digit);
    want -= s_above;
    bits += width;
    const unsigned long long above_all = k - want;  // keys above the bucket, all in the top-k
    if (s_count == want || shift == 0) {  // the whole bucket is in the top-k: keys >= its bound are exactly k
      thresh = prefix << shift;
      total = k;
      break;
    }
    if (above_all + s_count <= budget) {  // gather the whole bucket and finish in shared memory
      thresh = prefix << shift;
      total = above_all + s_count;
      break;
    }
    __syncthreads();
  }
  // Gather every key >= thresh (exactly `total` of them).
  for (int64_t base = 0; base < len; base += 8 * ONE_THREADS) {
    unsigned long long kk[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t i = base + static_cast<int64_t>(j) * ONE_THREADS + tid;
      kk[j] = i < len ? __ldcg(keys + i) : 0ull;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t i = base + static_cast<int64_t>(j) * ONE_THREADS + tid;
      const bool sel = i < len && kk[j] >= thresh;
      const unsigned m = __ballot_sync(FULL_MASK, sel);
      if (m) {
        unsigned pos0 = 0;
        if ((tid & 31) == 0) pos0 = atomicAdd(&s_cursor, static_cast<unsigned>(__popc(m)));
        pos0 = __shfl_sync(FULL_MASK, pos0, 0);
        if (sel) {
          const unsigned pos = pos0 + __popc(m & ((1u << (tid & 31)) - 1u));
          if (pos < ONE_OUT) s_out[pos] = kk[j];
        }
      }
    }
  }
  __syncthreads();
  const int cnt = static_cast<int>(total < ONE_OUT ? total : ONE_OUT);
  int P = ONE_THREADS;
  while (P < cnt) P <<= 1;
  for (int i = cnt + tid; i < P; i += ONE_THREADS) s_out[i] = 0ull;  // below every real key
  __syncthreads();
  switch (P / ONE_THREADS) {
    case 1: block_sort_desc<1>(s_out); break;
    case 2: block_sort_desc<2>(s_out); break;
    case 4: block_sort_desc<4>(s_out); break;
    default: block_sort_desc<8>(s_out); break;
  }
  for (int j = tid; j < static_cast<int>(a.k); j += ONE_THREADS)
    emit_one(s_out[j], row, j, a.k, a.x, a.ld, a.n, a.out_vals, a.out_idx);
}

int64_t next_pow2(int64_t v) {
  int64_t p = 1;
  while (p < v) p <<= 1;
  return p;
}

unsigned blocks_for(int64_t len, int threads, int cap) {
  int64_t b = (len + threads * 4 - 1) / (threads * 4);
  if (b < 1) b = 1;
  if (b > cap) b = cap;
  return static_cast<unsigned>(b);
}

}  // namespace

int sms() {
  static int count[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!count[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    count[dev] = v > 0 ? v : 1;
  }
  return count[dev];
}

namespace {


// Whether every row of a selection over the input starts on a 16-byte boundary.
bool input_vec4(const SelectArgs& a) {
  return (reinterpret_cast<uintptr_t>(a.base) & 15u) == 0 && (a.nrows == 1 && !a.rows ? true : (a.stride & 3) == 0);
}

template <class Src>
void run_passes(const Src& src, const SelectArgs& a, bool value_only, int first_pass, cudaStream_t stream) {
  // Digits of the 64-bit key from the top: 11, 11, 10 | 11, 11, 10 bits.
  static const int shifts[6] = {53, 42, 32, 21, 10, 0};
  static const int widths[6] = {11, 11, 10, 11, 11, 10};
  const int last = value_only ? 2 : 5;
  const int final_shift = shifts[last];
  const unsigned bx = blocks_for(a.len, SEL_THREADS, 4 * sms());
  for (int p = first_pass; p <= last; ++p) {
    launch_kernel(k_radix_pass<Src>, dim3(bx, a.nrows), SEL_THREADS, 0, stream, src, a.st, a.rows, shifts[p], widths[p],
                                                                     final_shift, value_only ? 1 : 0, p == 0);
  }
}

}  // namespace

void launch_select(const SelectArgs& a, uint64_t init_rank, bool value_only, int first_pass, cudaStream_t stream) {
  if (init_rank > 0) {
    launch_kernel(k_sel_init, a.nrows, 256, 0, stream, a.st, a.rows, init_rank);
  }
  switch (a.src) {
    case KeySource::SampleKeys:
      run_passes(SrcSample{static_cast<const uint32_t*>(a.base), a.stride, a.len}, a, value_only, first_pass, stream);
      break;
    case KeySource::Input:
      run_passes(SrcInput{static_cast<const float*>(a.base), a.stride, a.len, input_vec4(a)}, a, value_only, first_pass, stream);
      break;
    case KeySource::Buffer:
      run_passes(SrcBuffer{static_cast<const unsigned long long*>(a.base), a.stride, a.len}, a, value_only,
                 first_pass, stream);
      break;
  }
}

void launch_store_tau(int nrows, const int* rows, RowState* st, cudaStream_t stream) {
  launch_kernel(k_store_tau, nrows, 32, 0, stream, st, rows);
}

void launch_tie_init(int nrows, const int* rows, RowState* st, int64_t k, cudaStream_t stream) {
  launch_kernel(k_tie_init, nrows, 256, 0, stream, st, rows, static_cast<unsigned long long>(k));
}

void launch_compact(const SelectArgs& a, uint64_t* out, int64_t out_stride, int64_t k, cudaStream_t stream) {
  const unsigned bx = blocks_for(a.len, SEL_THREADS, 4 * sms());
  unsigned long long* o = reinterpret_cast<unsigned long long*>(out);
  switch (a.src) {
    case KeySource::SampleKeys:
      launch_kernel(k_compact<SrcSample>, dim3(bx, a.nrows), SEL_THREADS, 0, stream,
          SrcSample{static_cast<const uint32_t*>(a.base), a.stride, a.len}, a.st, a.rows, o, out_stride, k);
      break;
    case KeySource::Input:
      launch_kernel(k_compact<SrcInput>, dim3(bx, a.nrows), SEL_THREADS, 0, stream,
          SrcInput{static_cast<const float*>(a.base), a.stride, a.len, input_vec4(a)}, a.st, a.rows, o, out_stride, k);
      break;
    case KeySource::Buffer:
      launch_kernel(k_compact<SrcBuffer>, dim3(bx, a.nrows), SEL_THREADS, 0, stream,
          SrcBuffer{static_cast<const unsigned long long*>(a.base), a.stride, a.len}, a.st, a.rows, o, out_stride,
          k);
      break;
  }
}

void launch_refine_one(const RefineOneArgs& a, cudaStream_t stream) {
  const size_t smem = sizeof(unsigned long long) * ONE_OUT;
  cudaFuncSetAttribute(k_refine_one, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  launch_kernel(k_refine_one, a.nrows, ONE_THREADS, smem, stream, a);
}

int64_t refine_one_max_k() { return ONE_MAX_K; }
int64_t refine_one_max_m() { return ONE_MAX_M; }

int64_t sort_stride(int64_t k) { return k > SMALL_SORT_MAX ? next_pow2(k) : k; }

int64_t small_sort_max() { return SMALL_SORT_MAX; }

void launch_sort_emit(uint64_t* keys_u, int64_t key_stride, int64_t k, int nrows, const int* rows, const float* x,
                      int64_t ld, int64_t n, float* out_vals, int64_t* out_idx, cudaStream_t stream,
                      RowState* st, void* scratch, int64_t total_rows, bool gt_first) {
  if (k > SMALL_SORT_MAX && scratch) {
    RadixSortArgs ra{reinterpret_cast<unsigned long long*>(keys_u), key_stride, k,
                     st ? SortCount::KUnlessSkip : SortCount::All, nrows, rows, total_rows > 0 ? total_rows : nrows,
                     scratch, false, x, ld, n, out_vals, out_idx, st};
    launch_radix_sort(ra, stream);
    return;
  }
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(keys_u);
  if (k <= SMALL_SORT_MAX) {
    cudaFuncSetAttribute(k_sort_small, cudaFuncAttributeMaxDynamicSharedMemorySize, SMALL_SORT_MAX * 8);
    const int P = static_cast<int>(std::max<int64_t>(next_pow2(k), SORT_THREADS));
    launch_kernel(k_sort_small, nrows, SORT_THREADS, P * 8, stream, keys, key_stride, k, P, rows, x, ld, n, out_vals, out_idx,
                  st, gt_first && st != nullptr);
    return;
  }
  const int64_t P = next_pow2(k);  // >= 2 * CHUNK here
  cudaFuncSetAttribute(k_bitonic_chunk, cudaFuncAttributeMaxDynamicSharedMemorySize, CHUNK * 8);
  const unsigned padb = static_cast<unsigned>(std::min<int64_t>((P - k + SORT_THREADS - 1) / SORT_THREADS + 1, 1024));
  launch_kernel(k_pad, dim3(padb, nrows), SORT_THREADS, 0, stream, keys, key_stride, k, P, rows);
  const unsigned chunks = static_cast<unsigned>(P / CHUNK);
  launch_kernel(k_bitonic_chunk, dim3(chunks, nrows), SORT_THREADS, CHUNK * 8, stream, keys, key_stride, 2, CHUNK, rows);
  const unsigned gb = static_cast<unsigned>(std::min<int64_t>(P / 2 / SORT_THREADS + 1, 4096));
  for (int64_t size = 2 * CHUNK; size <= P; size <<= 1) {
    for (int64_t j = size >> 1; j >= CHUNK; j >>= 1) {
      launch_kernel(k_bitonic_global, dim3(gb, nrows), SORT_THREADS, 0, stream, keys, key_stride, P, size, j, rows);
    }
    launch_kernel(k_bitonic_chunk, dim3(chunks, nrows), SORT_THREADS, CHUNK * 8, stream, keys, key_stride,
                                                                             static_cast<int>(size), size, rows);
  }
  const unsigned eb = static_cast<unsigned>(std::min<int64_t>((k + SORT_THREADS - 1) / SORT_THREADS, 1024));
  launch_kernel(k_emit, dim3(eb, nrows), SORT_THREADS, 0, stream, keys, key_stride, k, rows, x, ld, n, out_vals, out_idx, st);
}

}  // namespace profk
