// Descending sort of the k selected 64-bit keys when k is too large for one
// CTA (Prof-K step 4 and the exact path, "Prof-K: Probabilistic One-Pass
// Filtering for Efficient Top-k Selection", Section 3, stage 4).
//
// Stable least-significant-digit radix sort, 8-bit digits, on the complement
// of the key (ascending order of ~key = descending order of key):
//  * one pre-pass histograms all eight digit positions at once; a digit
//    position where every key has the same digit is skipped on the device
//    (the sign and exponent bytes of a top-k usually are), and the
//    ping-pong buffer of every remaining pass is fixed by the same kernel;
//  * per pass, three kernels: per-tile digit counts, an exclusive scan of the
//    counts in (digit, tile) order, and a stable scatter in which a tile of
//    4096 keys is ranked in four rounds of 1024 keys (warp match for equal
//    digits, shared per-warp digit counts scanned across warps).
// No block waits on another block.
#include "kernels.h"

namespace profk {
namespace {

constexpr int RS_THREADS = 1024;
constexpr int RS_TILE = 4096;  // keys per tile (4 rounds of 1024)
constexpr int RS_WARPS = RS_THREADS / 32;

__device__ __forceinline__ unsigned digit_of(unsigned long long key, int pass) {
  return static_cast<unsigned>((~key) >> (8 * pass)) & 255u;
}

// Per-row sort control, in the workspace (zeroed by the host).
struct SortCtl {
  unsigned hist[8][256];
  int src_of_pass[8];  // 0: keys -> tmp, 1: tmp -> keys, -1: pass skipped
  int final_in_tmp;
  int pad[7];
};

__global__ void __launch_bounds__(RS_THREADS) k_rs_hist(const unsigned long long* keys, int64_t key_stride,
                                                       int64_t k, const int* rows, SortCtl* ctl,
                                                       const RowState* st) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned h[8][256];
  const int row = launch_row(rows);
  if (st && st[row].skip) return;
  for (int i = threadIdx.x; i < 8 * 256; i += RS_THREADS) (&h[0][0])[i] = 0;
  __syncthreads();
  const unsigned long long* kr = keys + row * key_stride;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * RS_THREADS + threadIdx.x; i < k;
       i += static_cast<int64_t>(gridDim.x) * RS_THREADS) {
    const unsigned long long key = kr[i];
#pragma unroll
    for (int p = 0; p < 8; ++p) atomicAdd(&h[p][digit_of(key, p)], 1u);
  }
  __syncthreads();
  SortCtl& c = ctl[row];
  for (int i = threadIdx.x; i < 8 * 256; i += RS_THREADS)
    if ((&h[0][0])[i]) atomicAdd(&c.hist[0][0] + i, (&h[0][0])[i]);
}

// Which passes run, and from which buffer.
__global__ void k_rs_plan(int64_t k, const int* rows, SortCtl* ctl, const RowState* st) {
  pdl_trigger();
  pdl_wait();
  const int row = rows ? rows[blockIdx.x] : static_cast<int>(blockIdx.x);
  if (st && st[row].skip) return;
  SortCtl& c = ctl[row];
  __shared__ int trivial[8];
  if (threadIdx.x < 8) trivial[threadIdx.x] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x)
    if (static_cast<int64_t>((&c.hist[0][0])[i]) == k) trivial[i / 256] = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    int in_tmp = 0;
    for (int p = 0; p < 8; ++p) {
      if (trivial[p]) {
        c.src_of_pass[p] = -1;
      } else {
        c.src_of_pass[p] = in_tmp;
        in_tmp ^= 1;
      }
    }
    c.final_in_tmp = in_tmp;
  }
}

// counts[row][digit * ntiles + tile]
__global__ void __launch_bounds__(RS_THREADS) k_rs_count(const unsigned long long* keys, unsigned long long* tmp,
                                                        int64_t key_stride, int64_t k, const int* rows,
                                                        const SortCtl* ctl, unsigned* counts, int pass,
                                                        const RowState* st) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned h[256];
  const int row = launch_row(rows);
  if (st && st[row].skip) return;
  const int src = ctl[row].src_of_pass[pass];
  if (src < 0) return;
  const unsigned long long* in = (src ? tmp : keys) + row * key_stride;
  const int ntiles = gridDim.x;
  for (int i = threadIdx.x; i < 256; i += RS_THREADS) h[i] = 0;
  __syncthreads();
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * RS_TILE;
  for (int r = 0; r < RS_TILE / RS_THREADS; ++r) {
    const int64_t i = t0 + r * RS_THREADS + threadIdx.x;
    if (i < k) atomicAdd(&h[digit_of(in[i], pass)], 1u);
  }
  __syncthreads();
  unsigned* cr = counts + static_cast<int64_t>(row) * 256 * ntiles;
  for (int d = threadIdx.x; d < 256; d += RS_THREADS) cr[static_cast<int64_t>(d) * ntiles + blockIdx.x] = h[d];
}

// Exclusive scan of one row's 256 * ntiles counts (one block per row).
__global__ void __launch_bounds__(RS_THREADS) k_rs_scan(unsigned* counts, int ntiles, const int* rows,
                                                       const SortCtl* ctl, int pass, const RowState* st) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned s_w[RS_WARPS];
  __shared__ unsigned s_carry;
  const int row = rows ? rows[blockIdx.x] : static_cast<int>(blockIdx.x);
  if (st && st[row].skip) return;
  if (ctl[row].src_of_pass[pass] < 0) return;
  unsigned* cr = counts + static_cast<int64_t>(row) * 256 * ntiles;
  const int64_t total = static_cast<int64_t>(256) * ntiles;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < total; base += RS_THREADS) {
    const int64_t i = base + threadIdx.x;
    const unsigned v = i < total ? cr[i] : 0u;
    unsigned incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const unsigned w = s_w[lane];
      unsigned wi = w;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(FULL_MASK, wi, o);
        if (lane >= o) wi += t;
      }
      s_w[lane] = wi - w;
    }
    __syncthreads();
    const unsigned carry = s_carry;
    if (i < total) cr[i] = carry + s_w[warp] + incl - v;
    __syncthreads();
    if (threadIdx.x == RS_THREADS - 1) s_carry = carry + s_w[warp] + incl;
    __syncthreads();
  }
}

// Stable scatter of one tile.
__global__ void __launch_bounds__(RS_THREADS) k_rs_scatter(unsigned long long* keys, unsigned long long* tmp,
                                                          int64_t key_stride, int64_t k, const int* rows,
                                                          const SortCtl* ctl, const unsigned* counts, int pass,
                                                          const RowState* st) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned short s_wc[RS_WARPS][256];  // per-warp digit counts of a round
  __shared__ unsigned s_base[256];                // running tile offset per digit
  const int row = launch_row(rows);
  if (st && st[row].skip) return;
  const int src = ctl[row].src_of_pass[pass];
  if (src < 0) return;
  const unsigned long long* in = (src ? tmp : keys) + row * key_stride;
  unsigned long long* out = (src ? keys : tmp) + row * key_stride;
  const int ntiles = gridDim.x;
  const unsigned* cr = counts + static_cast<int64_t>(row) * 256 * ntiles;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int d = threadIdx.x; d < 256; d += RS_THREADS) s_base[d] = cr[static_cast<int64_t>(d) * ntiles + blockIdx.x];
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * RS_TILE;
  for (int r = 0; r < RS_TILE / RS_THREADS; ++r) {
    const int64_t i = t0 + r * RS_THREADS + threadIdx.x;  // tile order = input order
    const bool valid = i < k;
    const unsigned long long key = valid ? in[i] : 0ull;
    const unsigned d = valid ? digit_of(key, pass) : 256u;  // 256: no digit
    for (int j = threadIdx.x; j < RS_WARPS * 256; j += RS_THREADS) (&s_wc[0][0])[j] = 0;
    __syncthreads();
    const unsigned act = __ballot_sync(FULL_MASK, valid);
    unsigned peers = 0, below = 0;
    if (valid) {
      peers = __match_any_sync(act, d);
      below = __popc(peers & ((1u << lane) - 1u));
      if (below == 0) s_wc[warp][d] = static_cast<unsigned short>(__popc(peers));
    }
    __syncthreads();
    // Per digit: exclusive scan of the warp counts over the warps, added to
    // the running base; threads 0..255 own one digit each.
    unsigned round_total = 0;
    if (threadIdx.x < 256) {
      unsigned acc = 0;
      for (int w = 0; w < RS_WARPS; ++w) {
        const unsigned c = s_wc[w][threadIdx.x];
        s_wc[w][threadIdx.x] = static_cast<unsigned short>(acc);
        acc += c;
      }
      round_total = acc;
    }
    __syncthreads();
    if (valid) out[s_base[d] + s_wc[warp][d] + below] = key;
    __syncthreads();
    if (threadIdx.x < 256) s_base[threadIdx.x] += round_total;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(RS_THREADS) k_rs_emit(const unsigned long long* keys,
                                                       const unsigned long long* tmp, int64_t key_stride, int64_t k,
                                                       const int* rows, const SortCtl* ctl, const float* x,
                                                       int64_t ld, int64_t n, float* out_vals, int64_t* out_idx,
                                                       const RowState* st) {
  pdl_trigger();
  pdl_wait();
  const int row = launch_row(rows);
  if (st && st[row].skip) return;
  const unsigned long long* sorted = (ctl[row].final_in_tmp ? tmp : keys) + row * key_stride;
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * RS_THREADS + threadIdx.x; j < k;
       j += static_cast<int64_t>(gridDim.x) * RS_THREADS) {
    const uint32_t idx = cand_index(sorted[j]);
    const int64_t o = static_cast<int64_t>(row) * k + j;
    if (static_cast<int64_t>(idx) < n) {
      out_idx[o] = static_cast<int64_t>(idx);
      out_vals[o] = x[static_cast<int64_t>(row) * ld + idx];
    } else {
      out_idx[o] = -1;
      out_vals[o] = __int_as_float(0x7fc00000);
    }
  }
}

}  // namespace

size_t radix_sort_scratch_bytes(int64_t k, int64_t key_stride, int64_t rows) {
  const int64_t ntiles = (k + RS_TILE - 1) / RS_TILE;
  const size_t tmp = sizeof(unsigned long long) * key_stride * rows;
  const size_t counts = sizeof(unsigned) * 256 * ntiles * rows;
  const size_t ctl = sizeof(SortCtl) * rows;
  return ((tmp + 255) & ~size_t(255)) + ((counts + 255) & ~size_t(255)) + ((ctl + 255) & ~size_t(255));
}

cudaError_t launch_radix_sort_emit(uint64_t* keys_u, int64_t key_stride, int64_t k, int nrows, const int* rows,
                                   void* scratch, int64_t total_rows, const float* x, int64_t ld, int64_t n,
                                   float* out_vals, int64_t* out_idx, cudaStream_t stream, const RowState* st) {
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(keys_u);
  const int64_t ntiles = (k + RS_TILE - 1) / RS_TILE;
  char* p = static_cast<char*>(scratch);
  // Scratch regions are indexed by row number, so they are sized for all
  // `total_rows` rows of the call (a row list may hold any of them).
  const size_t tmp_bytes = sizeof(unsigned long long) * key_stride * total_rows;
  unsigned long long* tmp = reinterpret_cast<unsigned long long*>(p);
  p += (tmp_bytes + 255) & ~size_t(255);
  unsigned* counts = reinterpret_cast<unsigned*>(p);
  p += (sizeof(unsigned) * 256 * ntiles * total_rows + 255) & ~size_t(255);
  SortCtl* ctl = reinterpret_cast<SortCtl*>(p);
  cudaError_t e = cudaMemsetAsync(ctl, 0, sizeof(SortCtl) * total_rows, stream);
  if (e != cudaSuccess) return e;
  const unsigned hb = static_cast<unsigned>(ntiles < 256 ? ntiles : 256);
  launch_kernel(k_rs_hist, dim3(hb, nrows), RS_THREADS, 0, stream, keys, key_stride, k, rows, ctl, st);
  launch_kernel(k_rs_plan, dim3(nrows), 256, 0, stream, k, rows, ctl, st);
  for (int pass = 0; pass < 8; ++pass) {
    launch_kernel(k_rs_count, dim3(static_cast<unsigned>(ntiles), nrows), RS_THREADS, 0, stream, keys, tmp,
                  key_stride, k, rows, ctl, counts, pass, st);
    launch_kernel(k_rs_scan, dim3(nrows), RS_THREADS, 0, stream, counts, static_cast<int>(ntiles), rows, ctl, pass,
                  st);
    launch_kernel(k_rs_scatter, dim3(static_cast<unsigned>(ntiles), nrows), RS_THREADS, 0, stream, keys, tmp,
                  key_stride, k, rows, ctl, counts, pass, st);
  }
  const unsigned eb = static_cast<unsigned>((k + RS_THREADS - 1) / RS_THREADS < 1024 ? (k + RS_THREADS - 1) / RS_THREADS
                                                                                    : 1024);
  return launch_kernel(k_rs_emit, dim3(eb, nrows), RS_THREADS, 0, stream, keys, tmp, key_stride, k, rows, ctl, x, ld,
                       n, out_vals, out_idx, st);
}

}  // namespace profk
