// Step 1 of Prof-K: uniform sampling of S indices without replacement and the
// gather of their values ("Prof-K: Probabilistic One-Pass Filtering for
// Efficient Top-k Selection", Section 3, stage 1).
//
// The sample is the first S distinct values of a counter-based draw stream
// (Philox4x64-10 words mapped to [0, n) by Lemire's method), in order of first
// appearance.  Rejecting repeats while drawing i.i.d. uniform indices gives a
// uniform S-subset, which is what the analysis of Section 4 assumes.
//
// GPU form: D >= S draws are generated in parallel and inserted into an
// open-addressing hash table that keeps, for every drawn value, the smallest
// draw position (atomicMin).  A draw is a first occurrence iff the table holds
// its own position; an ordered compaction of the first occurrences (block
// counts + in-block scan) yields the first S distinct draws in draw order.
// The result does not depend on D as long as the first D draws hold S
// distinct values; the count is reported so that the host can grow D.
#include "kernels.h"

namespace profk {
namespace {

constexpr unsigned long long EMPTY_SLOT = ~0ull;
constexpr int MARK_THREADS = 1024;

__device__ __forceinline__ uint64_t hash_slot(uint32_t u, int log2H) {
  return (static_cast<uint64_t>(u) * 0x9E3779B97F4A7C15ull) >> (64 - log2H);
}

__global__ void __launch_bounds__(256) k_sample_draw(SampleArgs a, int64_t key_row0) {
  pdl_trigger();
  pdl_wait();
  // One draw per thread: the four lanes that share a Philox block each
  // compute it (cheap arithmetic) and keep their own word, so every hash
  // insertion proceeds in parallel.
  const int row = launch_row(a.rows);
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= a.D) return;
  const uint64_t H = 1ull << a.log2H;
  unsigned long long* table = a.table + static_cast<int64_t>(row) * H;
  const uint64_t k0 = a.seed, k1 = static_cast<uint64_t>(row + key_row0);
  const uint64_t q = static_cast<uint64_t>(i >> 2);
  const int e = static_cast<int>(i & 3);
  uint64_t w[4] = {q, static_cast<uint64_t>(a.attempt), 0ull, 0ull};
  philox4x64_10(w, k0, k1);
  uint64_t u;
  if (!lemire64(w[e], a.n, &u)) {
    bool ok = false;
    for (uint64_t j = 1; j <= 64 && !ok; ++j) {
      uint64_t c[4] = {q, static_cast<uint64_t>(a.attempt), j, 0ull};
      philox4x64_10(c, k0, k1);
      ok = lemire64(c[e], a.n, &u);
    }
    if (!ok) {  // probability below (n / 2^64)^64: record, never hang
      atomicOr(&a.st[row].error, 1u);
      u = 0;
    }
  }
  const uint32_t u32 = static_cast<uint32_t>(u);
  a.draws[static_cast<int64_t>(row) * a.D + i] = u32;
  const unsigned long long entry = (static_cast<unsigned long long>(u32) << 32) | static_cast<uint32_t>(i);
  uint64_t slot = hash_slot(u32, a.log2H);
  for (uint64_t probe = 0; probe < H; ++probe) {
    const unsigned long long prev = atomicCAS(table + slot, EMPTY_SLOT, entry);
    if (prev == EMPTY_SLOT) return;
    if (static_cast<uint32_t>(prev >> 32) == u32) {
      atomicMin(table + slot, entry);
      return;
    }
    slot = (slot + 1) & (H - 1);
  }
  atomicOr(&a.st[row].error, 2u);
}

__device__ __forceinline__ uint32_t first_position(const unsigned long long* table, int log2H, uint32_t u) {
  const uint64_t H = 1ull << log2H;
  uint64_t slot = hash_slot(u, log2H);
  for (uint64_t probe = 0; probe < H; ++probe) {
    const unsigned long long v = table[slot];
    if (v == EMPTY_SLOT) break;
    if (static_cast<uint32_t>(v >> 32) == u) return static_cast<uint32_t>(v);
    slot = (slot + 1) & (H - 1);
  }
  return 0xffffffffu;
}

__global__ void __launch_bounds__(MARK_THREADS) k_sample_mark(SampleArgs a) {
  pdl_trigger();
  pdl_wait();
  const int row = launch_row(a.rows);
  const int64_t i = static_cast<int64_t>(blockIdx.x) * MARK_THREADS + threadIdx.x;
  const unsigned long long* table = a.table + (static_cast<int64_t>(row) << a.log2H);
  bool first = false;
  if (i < a.D) {
    const uint32_t u = a.draws[static_cast<int64_t>(row) * a.D + i];
    first = first_position(table, a.log2H, u) == static_cast<uint32_t>(i);
  }
  const int cnt = __syncthreads_count(first);
  if (threadIdx.x == 0) a.blockcnt[static_cast<int64_t>(row) * gridDim.x + blockIdx.x] = cnt;
}

// Last block of the compaction: the first radix pass of the tau selection
// (step 2) over the row's S sample keys is complete in the 2048-bin histogram
// of their top 11 bits; pick the bin that holds the t-th largest key and leave
// the selection state at "11 bits resolved" for the two remaining passes.
// Nothing is selected when fewer than S distinct draws were found (the host
// then grows D and the attempt runs again).
__device__ __noinline__ void tau_first_digit(const SampleArgs& a, int row) {
  constexpr int NW = MARK_THREADS / 32;
  __shared__ unsigned long long s_scan[NW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  RowState& S = a.st[row];
  const uint32_t* bc = a.blockcnt + static_cast<int64_t>(row) * gridDim.x;
  unsigned long long total = 0;
  for (unsigned b = lane; b < gridDim.x; b += 32) total += __ldcg(bc + b);
  for (int o = 16; o; o >>= 1) total += __shfl_xor_sync(FULL_MASK, total, o);
  // Thread t owns bins 2047 - 2t and 2046 - 2t (descending order).
  const int top = HIST_BINS - 1 - 2 * tid;
  const unsigned c0 = __ldcg(S.hist + top), c1 = __ldcg(S.hist + top - 1);
  const unsigned long long v = static_cast<unsigned long long>(c0) + c1;
  unsigned long long incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = lane < NW ? s_scan[lane] : 0ull;
    unsigned long long wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(FULL_MASK, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < NW) s_scan[lane] = wi - w;
  }
  __syncthreads();
  const unsigned long long excl = s_scan[warp] + incl - v;
  const unsigned long long want = a.t;
  if (total >= static_cast<unsigned long long>(a.S) && excl < want && want <= excl + v) {
    const bool in0 = want <= excl + c0;
    const unsigned d = in0 ? static_cast<unsigned>(top) : static_cast<unsigned>(top - 1);
    S.sel_prefix = d;
    S.sel_above = in0 ? excl : excl + c0;
    S.sel_rank = want - (in0 ? excl : excl + c0);
    S.sel_bucket = in0 ? c0 : c1;
    S.sel_bits = HIST_BITS;
  }
  __syncthreads();
  S.hist[top] = 0;
  S.hist[top - 1] = 0;
  if (tid == 0) S.done_blocks = 0;
}

__global__ void __launch_bounds__(MARK_THREADS) k_sample_compact(SampleArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int NW = MARK_THREADS / 32;
  __shared__ unsigned s_warp[NW];
  __shared__ unsigned long long s_base;
  const int row = launch_row(a.rows);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t* bc = a.blockcnt + static_cast<int64_t>(row) * gridDim.x;
  if (warp == 0) {
    // Prefix over the earlier blocks; block 0 also publishes the total.
    unsigned long long before = 0, total = 0;
    for (unsigned b = lane; b < gridDim.x; b += 32) {
      const unsigned c = bc[b];
      total += c;
      if (b < blockIdx.x) before += c;
    }
    for (int o = 16; o; o >>= 1) {
      before += __shfl_down_sync(FULL_MASK, before, o);
      total += __shfl_down_sync(FULL_MASK, total, o);
    }
    if (lane == 0) {
      s_base = before;
      if (blockIdx.x == 0) a.st[row].distinct = static_cast<unsigned>(total < 0xffffffffull ? total : 0xffffffffull);
    }
  }
  const int64_t i = static_cast<int64_t>(blockIdx.x) * MARK_THREADS + threadIdx.x;
  const unsigned long long* table = a.table + (static_cast<int64_t>(row) << a.log2H);
  uint32_t u = 0;
  bool first = false;
  if (i < a.D) {
    u = a.draws[static_cast<int64_t>(row) * a.D + i];
    first = first_position(table, a.log2H, u) == static_cast<uint32_t>(i);
  }
  const unsigned bal = __ballot_sync(FULL_MASK, first);
  if (lane == 0) s_warp[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    const unsigned v = lane < NW ? s_warp[lane] : 0u;
    unsigned incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane < NW) s_warp[lane] = incl - v;
  }
  __syncthreads();
  bool has = false;
  uint32_t key = 0;
  if (first) {
    const unsigned long long rank = s_base + s_warp[warp] + __popc(bal & ((1u << lane) - 1u));
    if (rank < static_cast<unsigned long long>(a.S)) {
      const int64_t o = static_cast<int64_t>(row) * a.S + static_cast<int64_t>(rank);
      key = ord_key(a.x[static_cast<int64_t>(row) * a.ld + u]);
      a.sidx[o] = u;
      a.skeys[o] = key;
      has = true;
    }
  }
  if (!a.tau_pass1) return;
  // First pass of step 2 fused: the keys' top 11 bits go to the row's
  // histogram (block-local first, then one atomic per non-empty bin); the
  // last block to finish picks the digit.
  __shared__ unsigned s_h[HIST_BINS];
  for (int b = threadIdx.x; b < HIST_BINS; b += MARK_THREADS) s_h[b] = 0;
  __syncthreads();
  hist_add(s_h, key >> (32 - HIST_BITS), has);
  __syncthreads();
  RowState& S = a.st[row];
  for (int b = threadIdx.x; b < HIST_BINS; b += MARK_THREADS)
    if (s_h[b]) atomicAdd(S.hist + b, s_h[b]);
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (threadIdx.x == 0) s_last = atomicAdd(&S.done_blocks, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  tau_first_digit(a, row);
}

}  // namespace

void launch_sample_rows(const SampleArgs& a, int64_t key_row0, cudaStream_t stream) {
  const int64_t blocks = (a.D + 255) / 256;
  launch_kernel(k_sample_draw, dim3(static_cast<unsigned>(blocks), a.nrows), 256, 0, stream, a, key_row0);
  const unsigned nb = static_cast<unsigned>((a.D + MARK_THREADS - 1) / MARK_THREADS);
  launch_kernel(k_sample_mark, dim3(nb, a.nrows), MARK_THREADS, 0, stream, a);
  launch_kernel(k_sample_compact, dim3(nb, a.nrows), MARK_THREADS, 0, stream, a);
}

void launch_sample(const SampleArgs& a, cudaStream_t stream) { launch_sample_rows(a, 0, stream); }

}  // namespace profk
