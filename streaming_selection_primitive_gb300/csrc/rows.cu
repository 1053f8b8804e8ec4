// Exact top-k of short rows, one CTA per row: the exact selection over the
// full input ("Prof-K: Probabilistic One-Pass Filtering for Efficient Top-k
// Selection", Section 3, stage 4, the fallback) for calls whose rows are small
// enough that a row fits one SM's share of the bandwidth, such as the batched
// shapes of Appendix E.2 (up to 1024 rows of 2^16 - 2^22 elements).
//
// A CTA takes rows in turn.  Keys are the 64-bit (ord(v) << 32) | ~i, so the
// k largest keys are the k largest values with ties to the lower index.  Per
// row, the method's own filter idea inside one CTA:
//  1. a threshold tau from a small sample of the row (positions from a hash,
//     values into shared memory; tau = a sample order statistic chosen so
//     that k <= R <= RX_CAP is very likely, R = #{x >= tau});
//  2. one pass over the row appends every key with value >= tau to a list
//     in shared memory and counts R exactly;
//  3. if k <= R <= RX_CAP the k-th largest key T of the list is found by
//     digit passes on the list alone (11, 11, 10 bits of the value, then of
//     the index); otherwise (a sample that missed, or heavy ties) the same
//     digit passes run over the row until the keys at or above the chosen
//     bucket fit the list, and one more pass lists them;
//  4. the k keys >= T are compacted and placed in order: by counting the
//     larger keys (k <= 512), else by a bitonic sort.
// The sample only decides the speed: every output is checked by the exact
// count R, as in the method.  Histograms aggregate each warp's equal digits
// with ballots (a digit of float keys is often shared by most of a warp).
// No global atomics, no grid-wide step: each row is one CTA's work.
#include <algorithm>
#include <cmath>

#include "kernels.h"

namespace profk {
namespace {

constexpr int RX_THREADS = 512;
constexpr int RX_CAP = 8192;     // keys listed in shared memory (64 KB, dynamic)
constexpr int RX_MAX_K = 2048;
constexpr int RX_U = 8;          // float4 loads in flight per thread
constexpr int RX_COUNT_K = RX_THREADS;  // up to this k, keys are placed by counting
constexpr int RX_SAMPLE_MIN = 1024, RX_SAMPLE_MAX = 16384;  // the sample fills at most the list's space
constexpr int64_t RX_MAX_N = 1 << 20;  // rows up to this length keep a sample of 1/64

// Digit p of a key, from the top: 11, 11, 10 bits of the value, then of ~i.
__device__ __forceinline__ int rx_width(int p) { return (p == 2 || p == 5) ? 10 : 11; }
__device__ __forceinline__ int rx_shift(int p) { return 64 - 11 * (p + 1) + (p >= 2 ? 1 : 0) + (p >= 5 ? 1 : 0); }
// The pass that follows `bits` resolved bits.
__device__ __forceinline__ int rx_pass_of(int bits) {
  return bits == 0 ? 0 : bits == 11 ? 1 : bits == 22 ? 2 : bits == 32 ? 3 : bits == 43 ? 4 : 5;
}

// Histogram increment by a whole warp (all 32 lanes call it): the lanes with
// the same digit are found with one ballot per digit bit, and the lowest of
// them adds their count, so equal digits cost one shared-memory atomic.
__device__ __forceinline__ void rx_hist_add(unsigned* h, uint32_t digit, bool valid, int width) {
  unsigned peers = __ballot_sync(FULL_MASK, valid);
  if (peers == 0u) return;
#pragma unroll
  for (int b = 0; b < 11; ++b) {
    if (b < width) {
      const bool bit = (digit >> b) & 1u;
      const unsigned bal = __ballot_sync(FULL_MASK, bit);
      peers &= bit ? bal : ~bal;
    }
  }
  if (valid && static_cast<int>(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(h + digit, __popc(peers));
}

// Appends key to list (capacity RX_CAP) when s; *cursor counts every append.
__device__ __forceinline__ void rx_append(unsigned long long* list, unsigned* cursor, unsigned long long key,
                                          bool s) {
  const unsigned m = __ballot_sync(FULL_MASK, s);
  if (m) {
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(m) - 1;
    unsigned base = 0;
    if (lane == leader) base = atomicAdd(cursor, static_cast<unsigned>(__popc(m)));
    base = __shfl_sync(FULL_MASK, base, leader);
    if (s) {
      const unsigned pos = base + __popc(m & ((1u << lane) - 1u));
      if (pos < static_cast<unsigned>(RX_CAP)) list[pos] = key;
    }
  }
}

// Sample position j of a row: a splitmix64 hash of (row, j) scaled to [0, n).
__device__ __forceinline__ uint32_t rx_sample_pos(int row, int j, uint64_t n) {
  uint64_t z = (static_cast<uint64_t>(row) << 32 | static_cast<uint32_t>(j)) + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return static_cast<uint32_t>(((z >> 32) * n) >> 32);
}

// Every element of a row through f(value, index, valid), on every thread the
// same number of times (f may be warp-collective): RX_U float4 loads per
// thread in flight, then a scalar tail.
template <class F>
__device__ __forceinline__ void rx_scan_row(const float* xr, int64_t n, F&& f) {
  const int tid = threadIdx.x;
  const int64_t n4 = n >> 2;
  const float4* x4 = reinterpret_cast<const float4*>(xr);
  for (int64_t b = 0; b < n4; b += static_cast<int64_t>(RX_THREADS) * RX_U) {
    float4 v[RX_U];
#pragma unroll
    for (int u = 0; u < RX_U; ++u) {
      const int64_t q = b + u * RX_THREADS + tid;
      v[u] = q < n4 ? __ldg(x4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < RX_U; ++u) {
      const int64_t q = b + u * RX_THREADS + tid;
      const bool ok = q < n4;
      f(v[u].x, 4 * q, ok);
      f(v[u].y, 4 * q + 1, ok);
      f(v[u].z, 4 * q + 2, ok);
      f(v[u].w, 4 * q + 3, ok);
    }
  }
  if ((n4 << 2) < n) {  // at most 3 elements
    const int64_t i = (n4 << 2) + tid;
    const bool ok = i < n;
    f(ok ? xr[i] : 0.f, i, ok);
  }
}

// Digit choice after a histogram pass: the bin (counted down from the top)
// that holds the want-th largest counted key.  Thread t owns nb / 512 bins.
struct RxPick {
  unsigned digit;
  unsigned long long above;  // counted keys in higher bins
  unsigned long long count;  // keys in the chosen bin
};

__device__ __forceinline__ RxPick rx_pick(const unsigned* h, unsigned nb, unsigned long long want,
                                          unsigned long long* sw, RxPick* s_pick) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = static_cast<int>(nb) / RX_THREADS;  // 4 or 2
  const int top = static_cast<int>(nb) - 1 - tid * per;
  unsigned hv[4] = {0u, 0u, 0u, 0u};
  unsigned long long local = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q < per) {
      hv[q] = h[top - q];
      local += hv[q];
    }
  }
  unsigned long long incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sw[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = lane < RX_THREADS / 32 ? sw[lane] : 0ull;
    unsigned long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(FULL_MASK, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < RX_THREADS / 32) sw[lane] = wi - w;
  }
  __syncthreads();
  const unsigned long long excl = sw[warp] + incl - local;
  if (excl < want && want <= excl + local) {
    unsigned long long acc = excl;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q < per && want <= acc + hv[q]) {
        s_pick->digit = static_cast<unsigned>(top - q);
        s_pick->above = acc;
        s_pick->count = hv[q];
        break;
      }
      acc += hv[q];
    }
  }
  __syncthreads();
  const RxPick r = *s_pick;
  __syncthreads();
  return r;
}

// Descending bitonic sort of P (a power of two, <= RX_CAP) keys in shared
// memory by the whole CTA.
__device__ __forceinline__ void rx_bitonic_desc(unsigned long long* s, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int j = size >> 1; j >= 1; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += RX_THREADS) {
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
  }
}

__device__ __forceinline__ void rx_emit(unsigned long long key, int row, int64_t j, int64_t k, const float* xr,
                                        int64_t n, float* out_vals, int64_t* out_idx) {
  const uint32_t idx = cand_index(key);
  if (static_cast<int64_t>(idx) < n) {
    out_idx[row * k + j] = static_cast<int64_t>(idx);
    out_vals[row * k + j] = xr[idx];
  } else {  // never for a correct selection; keeps reads inside the row
    out_idx[row * k + j] = -1;
    out_vals[row * k + j] = __int_as_float(0x7fc00000);
  }
}

__global__ void __launch_bounds__(RX_THREADS, 2) k_rows_exact(RowsExactArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned h[HIST_BINS];
  __shared__ unsigned long long sw[32];
  __shared__ RxPick s_pick;
  __shared__ unsigned s_cursor, s_nan;
  extern __shared__ unsigned long long list[];  // RX_CAP keys; the sample's values before that
  uint32_t* skey = reinterpret_cast<uint32_t*>(list);
  const int tid = threadIdx.x, lane = tid & 31;
  const unsigned long long k = static_cast<unsigned long long>(a.k);
  const uint64_t n = static_cast<uint64_t>(a.n);
  for (int g = blockIdx.x; g < a.nrows; g += gridDim.x) {
    const int row = a.rows ? a.rows[g] : g;
    const float* xr = a.x + static_cast<int64_t>(row) * a.ld;

    // 1. tau (as an order key) from a sample; 0 (every key) for short rows.
    uint32_t tau = 0u;
    if (n > static_cast<uint64_t>(RX_CAP)) {
      int SS = RX_SAMPLE_MIN;
      while (SS < RX_SAMPLE_MAX && static_cast<uint64_t>(SS) * 64 < n) SS <<= 1;
      const float f = static_cast<float>(SS) / static_cast<float>(n);
      const float kf = static_cast<float>(k) * f;
      // Rank t in the sample.  R < k needs t or more sampled keys above the
      // k-th largest (about Poisson(k f) of them); R > RX_CAP needs fewer than
      // t at or above the RX_CAP-th (about Poisson(RX_CAP f), f >= 1/64 for
      // rows up to RX_MAX_N).  t = k f + 4 sqrt(k f) + 9 keeps both rare.
      const int t = static_cast<int>(ceilf(kf + 4.f * sqrtf(kf) + 8.f)) + 1;
      if (t <= SS) {
        for (int j0 = 0; j0 < SS; j0 += 4 * RX_THREADS) {
          float v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = j0 + u * RX_THREADS + tid;
            v[u] = j < SS ? xr[rx_sample_pos(row, j, n)] : 0.f;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = j0 + u * RX_THREADS + tid;
            if (j < SS) skey[j] = ord_key(v[u]);
          }
        }
        __syncthreads();
        // The t-th largest sample key: 11/11/10-bit passes.
        uint32_t pre = 0u;
        unsigned long long w = static_cast<unsigned long long>(t);
        int pb = 0;
        for (int p = 0; p < 3; ++p) {
          const int width = p == 2 ? 10 : 11;
          const int shift = 32 - pb - width;
          const unsigned nb = 1u << width;
          for (unsigned b = tid; b < nb; b += RX_THREADS) h[b] = 0u;
          __syncthreads();
          for (int j0 = 0; j0 < SS; j0 += RX_THREADS) {
            const int j = j0 + tid;
            const uint32_t key = j < SS ? skey[j] : 0u;
            const bool m = j < SS && (pb == 0 || (key >> (32 - pb)) == pre);
            rx_hist_add(h, (key >> shift) & (nb - 1), m, width);
          }
          __syncthreads();
          const RxPick pk = rx_pick(h, nb, w, sw, &s_pick);
          pre = (pre << width) | pk.digit;
          pb += width;
          w -= pk.above;
        }
        tau = pre;
      }
    }

    // 2. The pass over the row: keys with value >= tau into the list, R exact.
    if (tid == 0) {
      s_cursor = 0u;
      s_nan = 0u;
    }
    __syncthreads();
    unsigned nan_local = 0;
    rx_scan_row(xr, a.n, [&](float v, int64_t i, bool ok) {
      const uint32_t kv = ord_key(v);
      nan_local += ok && key_is_nan(kv);
      rx_append(list, &s_cursor, (static_cast<unsigned long long>(kv) << 32) | static_cast<uint32_t>(~i),
                ok && kv >= tau);
    });
    nan_local = __reduce_add_sync(FULL_MASK, nan_local);
    if (lane == 0 && nan_local) atomicAdd(&s_nan, nan_local);
    __syncthreads();
    if (tid == 0) a.st[row].sel_nan = s_nan;
    const unsigned R = s_cursor;

    // Selection state: the k-th largest key lies in the bucket of keys whose
    // top `bits` bits equal `prefix`; `above` keys are above the bucket.
    unsigned long long prefix = 0, want = k, above = 0, cnt = R;
    int bits = 0;
    if (R < k || R > static_cast<unsigned>(RX_CAP)) {
      // 3'. Digit passes over the row until the keys at or above the bucket
      //     fit the list, then those keys into the list.
      for (int p = 0; p < 6; ++p) {
        const int shift = rx_shift(p), width = rx_width(p);
        const unsigned nb = 1u << width;
        for (unsigned b = tid; b < nb; b += RX_THREADS) h[b] = 0u;
        __syncthreads();
        rx_scan_row(xr, a.n, [&](float v, int64_t i, bool ok) {
          const unsigned long long key = cand_key(v, static_cast<uint32_t>(i));
          const bool m = ok && (bits == 0 || (key >> (64 - bits)) == prefix);
          rx_hist_add(h, static_cast<uint32_t>(key >> shift) & (nb - 1), m, width);
        });
        __syncthreads();
        const RxPick pk = rx_pick(h, nb, want, sw, &s_pick);
        prefix = (prefix << width) | pk.digit;
        bits += width;
        above += pk.above;
        want -= pk.above;
        cnt = pk.count;
        if (above + cnt <= static_cast<unsigned long long>(RX_CAP)) break;
      }
      const unsigned long long lb = bits >= 64 ? prefix : prefix << (64 - bits);
      if (tid == 0) s_cursor = 0u;
      __syncthreads();
      rx_scan_row(xr, a.n, [&](float v, int64_t i, bool ok) {
        const unsigned long long key = cand_key(v, static_cast<uint32_t>(i));
        rx_append(list, &s_cursor, key, ok && key >= lb);
      });
      __syncthreads();
    }
    const int L = s_cursor < static_cast<unsigned>(RX_CAP) ? static_cast<int>(s_cursor) : RX_CAP;

    // 3. The k-th largest key T inside the list: digit passes on the list
    //    alone, until the bucket is taken whole or fully resolved.
    while (bits < 64 && cnt != want) {
      const int p = rx_pass_of(bits);
      const int shift = rx_shift(p), width = rx_width(p);
      const unsigned nb = 1u << width;
      for (unsigned b = tid; b < nb; b += RX_THREADS) h[b] = 0u;
      __syncthreads();
      for (int j0 = 0; j0 < L; j0 += RX_THREADS) {
        const int j = j0 + tid;
        const unsigned long long key = j < L ? list[j] : 0ull;
        const bool m = j < L && (bits == 0 || (key >> (64 - bits)) == prefix);
        rx_hist_add(h, static_cast<uint32_t>(key >> shift) & (nb - 1), m, width);
      }
      __syncthreads();
      const RxPick pk = rx_pick(h, nb, want, sw, &s_pick);
      prefix = (prefix << width) | pk.digit;
      bits += width;
      above += pk.above;
      want -= pk.above;
      cnt = pk.count;
    }
    const unsigned long long T = bits == 0 ? 0ull : bits >= 64 ? prefix : prefix << (64 - bits);

    // 4. The k keys >= T to the front of the list, one block of 512 at a time
    //    (a block's keys are read before any is written, and the compacted
    //    positions never pass the block being read).
    if (tid == 0) s_cursor = 0u;
    __syncthreads();
    for (int j0 = 0; j0 < L; j0 += RX_THREADS) {
      const int j = j0 + tid;
      const unsigned long long key = j < L ? list[j] : 0ull;
      __syncthreads();
      rx_append(list, &s_cursor, key, j < L && key >= T);
      __syncthreads();
    }
    const int kk = static_cast<int>(k);
    // Placement: key j goes to the count of larger keys among the k.
    if (kk <= RX_COUNT_K) {
      if (tid < kk) {
        const unsigned long long e = list[tid];
        int rank = 0;
        for (int j = 0; j < kk; ++j) rank += list[j] > e;
        rx_emit(e, row, rank, a.k, xr, a.n, a.out_vals, a.out_idx);
      }
    } else {
      int P = RX_COUNT_K;
      while (P < kk) P <<= 1;
      for (int j = kk + tid; j < P; j += RX_THREADS) list[j] = 0ull;  // below every key
      __syncthreads();
      rx_bitonic_desc(list, P);
      for (int j = tid; j < kk; j += RX_THREADS) rx_emit(list[j], row, j, a.k, xr, a.n, a.out_vals, a.out_idx);
    }
    __syncthreads();  // the list and histogram are reused by the next row
  }
}

}  // namespace

int64_t rows_exact_max_k() { return RX_MAX_K; }

bool rows_exact_suits(int64_t nrows, int64_t n, int64_t k) {
  if (k > RX_MAX_K || n > RX_MAX_N) return false;
  // Measured on GB300: a CTA alone on its SM streams its row at about
  // 18 GB/s, two CTAs sharing an SM at about 8 GB/s each, plus about 15 us
  // of sampling and shared-memory work per row; the multi-CTA selection
  // takes up to six passes over all rows at about 1.5 TB/s plus ~60 us of
  // launches.  Both in microseconds.
  const double bytes = 4.0 * static_cast<double>(n);
  const double s = static_cast<double>(sms());
  const double rows_us = nrows <= s ? bytes / 18e3 + 15.0
                                    : std::ceil(static_cast<double>(nrows) / (2.0 * s)) * (bytes / 8e3 + 15.0);
  const double multi_us = 6.0 * bytes * static_cast<double>(nrows) / 1.5e6 + 60.0;
  return rows_us < multi_us;
}

void launch_rows_exact(const RowsExactArgs& a, cudaStream_t stream) {
  const int64_t G = std::min<int64_t>(a.nrows, 2ll * sms());
  constexpr int smem = RX_CAP * static_cast<int>(sizeof(unsigned long long));
  cudaFuncSetAttribute(k_rows_exact, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  launch_kernel(k_rows_exact, static_cast<unsigned>(G), RX_THREADS, smem, stream, a);
}

}  // namespace profk
