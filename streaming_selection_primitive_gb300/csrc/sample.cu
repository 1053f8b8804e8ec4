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

// Draw i of a row's stream: word i % 4 of Philox block (i / 4, attempt, 0, 0)
// under key (seed, key row), mapped to [0, n) by Lemire's method; a word
// that Lemire rejects is replaced by the same word of blocks (i / 4, attempt,
// j, 0), j = 1, 2, ...  (Each thread computes the whole block and keeps one
// word: cheap arithmetic, and every draw proceeds in parallel.)
__device__ __forceinline__ uint32_t draw_value(const SampleArgs& a, int row, uint64_t key_row, int64_t i) {
  const uint64_t k0 = a.seed, k1 = key_row;
  const uint64_t q = static_cast<uint64_t>(i >> 2);
  const int e = static_cast<int>(i & 3);
  // (word e picked with selects: a dynamic index would put the block in local memory)
  auto word = [e](const uint64_t (&v)[4]) { return e == 0 ? v[0] : e == 1 ? v[1] : e == 2 ? v[2] : v[3]; };
  uint64_t w[4] = {q, static_cast<uint64_t>(a.attempt), 0ull, 0ull};
  philox4x64_10(w, k0, k1);
  uint64_t u;
  if (!lemire64(word(w), a.n, &u)) {
    bool ok = false;
    for (uint64_t j = 1; j <= 64 && !ok; ++j) {
      uint64_t c[4] = {q, static_cast<uint64_t>(a.attempt), j, 0ull};
      philox4x64_10(c, k0, k1);
      ok = lemire64(word(c), a.n, &u);
    }
    if (!ok) {  // probability below (n / 2^64)^64: record, never hang
      atomicOr(&a.st[row].error, 1u);
      u = 0;
    }
  }
  return static_cast<uint32_t>(u);
}

// Linear probing, PROBE_SPAN slots per step: the slots of a step are loaded
// together, so that a long cluster costs a few round trips rather than one
// per slot.  Slots only ever go from empty to holding a value u, and only
// the draw part of a held entry changes later (atomicMin for the same u), so
// a load that shows another value is final, and a load that shows an empty
// slot is checked by the compare-and-swap that claims it.
constexpr int PROBE_SPAN = 4;

__device__ __forceinline__ unsigned long long ld_slot(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Insertion of (value u, draw i), keeping the smallest draw of u, in two
// steps so that a thread can have several insertions in flight: the
// compare-and-swap on the home slot, then (with its result) the rest.
__device__ __forceinline__ unsigned long long table_entry(uint32_t u, int64_t i) {
  return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(i);
}

__device__ __forceinline__ unsigned long long table_try_home(unsigned long long* table, int log2H, uint32_t u,
                                                             int64_t i) {
  return atomicCAS(table + hash_slot(u, log2H), EMPTY_SLOT, table_entry(u, i));
}

// Returns the slot that holds u (values never move once placed).
__device__ __forceinline__ uint64_t table_finish(const SampleArgs& a, int row, unsigned long long* table, uint32_t u,
                                                 int64_t i, unsigned long long prev) {
  const uint64_t H = 1ull << a.log2H;
  const unsigned long long entry = table_entry(u, i);
  uint64_t slot = hash_slot(u, a.log2H);
  if (prev == EMPTY_SLOT) return slot;
  if (static_cast<uint32_t>(prev >> 32) == u) {
    atomicMin(table + slot, entry);
    return slot;
  }
  slot = (slot + 1) & (H - 1);
  for (uint64_t seen = 1; seen < H;) {
    unsigned long long v[PROBE_SPAN];
#pragma unroll
    for (int q = 0; q < PROBE_SPAN; ++q) v[q] = ld_slot(table + ((slot + q) & (H - 1)));
    int adv = PROBE_SPAN;
#pragma unroll
    for (int q = 0; q < PROBE_SPAN; ++q) {
      if (adv != PROBE_SPAN) continue;  // an earlier slot of this step decided
      const uint64_t sq = (slot + q) & (H - 1);
      if (v[q] == EMPTY_SLOT) {
        prev = atomicCAS(table + sq, EMPTY_SLOT, entry);
        if (prev == EMPTY_SLOT) return sq;
        if (static_cast<uint32_t>(prev >> 32) == u) {
          atomicMin(table + sq, entry);
          return sq;
        }
        adv = q + 1;  // taken by another value: continue after it
      } else if (static_cast<uint32_t>(v[q] >> 32) == u) {
        atomicMin(table + sq, entry);
        return sq;
      }
    }
    slot = (slot + adv) & (H - 1);
    seen += adv;
  }
  atomicOr(&a.st[row].error, 2u);
  return 0;
}

__device__ __forceinline__ void table_insert(const SampleArgs& a, int row, unsigned long long* table, uint32_t u,
                                             int64_t i) {
  table_finish(a, row, table, u, i, table_try_home(table, a.log2H, u, i));
}

__global__ void __launch_bounds__(256) k_sample_draw(SampleArgs a, int64_t key_row0) {
  pdl_trigger();
  pdl_wait();
  const int row = launch_row(a.rows);
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= a.D) return;
  unsigned long long* table = a.table + (static_cast<int64_t>(row) << a.log2H);
  const uint32_t u = draw_value(a, row, static_cast<uint64_t>(row + key_row0), i);
  a.draws[static_cast<int64_t>(row) * a.D + i] = u;
  table_insert(a, row, table, u, i);
}

// Smallest draw of u (the table is complete): PROBE_SPAN slots per step.
__device__ __forceinline__ uint32_t first_position(const unsigned long long* table, int log2H, uint32_t u) {
  const uint64_t H = 1ull << log2H;
  uint64_t slot = hash_slot(u, log2H);
  for (uint64_t seen = 0; seen < H; seen += PROBE_SPAN) {
    unsigned long long v[PROBE_SPAN];
#pragma unroll
    for (int q = 0; q < PROBE_SPAN; ++q) v[q] = __ldcg(table + ((slot + q) & (H - 1)));
#pragma unroll
    for (int q = 0; q < PROBE_SPAN; ++q) {
      if (v[q] == EMPTY_SLOT) return 0xffffffffu;
      if (static_cast<uint32_t>(v[q] >> 32) == u) return static_cast<uint32_t>(v[q]);
    }
    slot = (slot + PROBE_SPAN) & (H - 1);
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

// ---------------------------------------------------------------------------
// Steps 1 and 2 in one persistent kernel (the main path): one 512-thread CTA
// per SM and contiguous chunk of the draw positions, all CTAs of the launch
// resident together (chunks x rows <= the SM count) so that they can meet at
// grid barriers (bounded waits on a per-row arrival counter).
//  a. every CTA draws its chunk and inserts it into the row's hash table;
//     barrier;
//  b. first occurrences are marked; a CTA publishes its count and adds up
//     the counts of the earlier chunks (a look-back: each is published
//     before its CTA waits for anything), which places its first occurrences
//     in draw order; those of rank < S are the sample: their values are
//     gathered and their keys kept (and stored, with the indices);
//  c. tau = the t-th largest sample key, by 11/11/10-bit MSD passes whose
//     chunk histograms meet in global atomics; after each pass's barrier
//     every CTA reads the same totals and takes the same digit.  Once the
//     bucket that holds tau has at most 512 keys, they are listed and the
//     first CTA finds the rank among them directly.
// The first CTA leaves tau in RowState::tau_key and the last the number of
// distinct draws in RowState::distinct (below S, the host grows D).

constexpr int ST_THREADS = 512;
constexpr int ST_HELD = 2;                      // rounds of draws whose keys stay in registers
constexpr int ST_WAIT_POLLS = 1 << 22;          // bound on one wait (a poll is an L2 round trip)
constexpr unsigned ST_ERR_WAIT = 8u;            // RowState::error bit of a wait that ran out
constexpr unsigned long long CNT_READY = 1ull << 63;
constexpr int TAU_GATHER = ST_THREADS;  // a tau bucket this small is finished by one CTA

}  // namespace

// Per-row control block, zeroed at the start of every attempt.
struct SampleCtl {
  unsigned hist[3][HIST_BINS];        // tau pass histograms, summed over the chunks
  unsigned long long count[256];      // first occurrences per chunk | CNT_READY
  uint32_t bucket[TAU_GATHER];        // the sample keys of tau's final bucket
  unsigned bucket_n;
  unsigned bar;                       // grid-barrier arrivals
  unsigned pad[62];
};
static_assert(sizeof(SampleCtl) % 16 == 0, "SampleCtl is zeroed with 16-byte stores");

namespace {

__device__ __forceinline__ unsigned st_ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long st_ld_relaxed(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_st_relaxed(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Every CTA of the row arrives (a release: the CTA's writes, ordered before
// it by the block barrier, become visible with it), then waits until all
// have (acquire loads of the arrival count).
__device__ __forceinline__ void st_grid_sync(unsigned* bar, unsigned target, int* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
    for (int poll = 0; st_ld_acquire(bar) < target; ++poll) {
      if (poll >= ST_WAIT_POLLS) {
        *err = 1;
        break;
      }
    }
  }
  __syncthreads();
}

// Block-wide sum and exclusive scan (thread order) of one value per thread.
__device__ __forceinline__ unsigned long long st_excl_scan(unsigned long long v, unsigned long long* sw,
                                                           unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sw[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = lane < ST_THREADS / 32 ? sw[lane] : 0ull;
    unsigned long long wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(FULL_MASK, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < ST_THREADS / 32) sw[lane] = wi - w;
    if (lane == 31) sw[32] = wi;
  }
  __syncthreads();
  const unsigned long long r = sw[warp] + incl - v;
  *total = sw[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(ST_THREADS, 1) k_sample_tau(SampleArgs a, SampleCtl* ctl) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned h[HIST_BINS];
  __shared__ unsigned long long sw[33];
  __shared__ int s_err;
  __shared__ unsigned s_digit;
  __shared__ unsigned long long s_above, s_count, s_base;
  __shared__ uint32_t s_list[TAU_GATHER];
  __shared__ uint32_t s_tau;
  const int row = launch_row(a.rows);
  RowState& S = a.st[row];
  SampleCtl& c = ctl[row];
  const int tid = threadIdx.x;
  if (tid == 0) s_err = 0;
  const int64_t G = gridDim.x, chunk = blockIdx.x;
  const int64_t Dc = (((a.D + G - 1) / G) + 31) & ~int64_t(31);
  const int64_t lo = chunk * Dc < a.D ? chunk * Dc : a.D;
  const int64_t hi = lo + Dc < a.D ? lo + Dc : a.D;
  const int rounds = static_cast<int>((hi - lo + ST_THREADS - 1) / ST_THREADS);
  unsigned long long* table = a.table + (static_cast<int64_t>(row) << a.log2H);
  unsigned target = 0;

  // a. Draw and insert.
  // Rounds j < ST_HELD keep their draws (and later keys) in registers; the
  // loops over them are unrolled so that the arrays stay there.
  // Their values are gathered at once (used only if the draw is a member),
  // so that the gather's latency overlaps the insertions.
  // Both rounds' loads and home-slot swaps are issued before any result is
  // waited for.
  uint32_t uh[ST_HELD] = {0u, 0u};
  float vh[ST_HELD] = {0.f, 0.f};
  unsigned long long ph[ST_HELD] = {EMPTY_SLOT, EMPTY_SLOT};
  uint64_t sh[ST_HELD] = {0, 0};  // the slot that holds each held draw's value
#pragma unroll
  for (int j = 0; j < ST_HELD; ++j) {
    const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
    if (j < rounds && i < hi) uh[j] = draw_value(a, row, static_cast<uint64_t>(row), i);
  }
#pragma unroll
  for (int j = 0; j < ST_HELD; ++j) {
    const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
    if (j < rounds && i < hi) {
      vh[j] = a.x[static_cast<int64_t>(row) * a.ld + uh[j]];
      ph[j] = table_try_home(table, a.log2H, uh[j], i);
    }
  }
#pragma unroll
  for (int j = 0; j < ST_HELD; ++j) {
    const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
    if (j < rounds && i < hi) sh[j] = table_finish(a, row, table, uh[j], i, ph[j]);
  }
  for (int j = ST_HELD; j < rounds; ++j) {
    const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
    if (i < hi) table_insert(a, row, table, draw_value(a, row, static_cast<uint64_t>(row), i), i);
  }
  st_grid_sync(&c.bar, target += static_cast<unsigned>(G), &s_err);

  // b. First occurrences, their count and their place in draw order.
  bool first_h[ST_HELD] = {false, false};
  unsigned long long cnt = 0;
#pragma unroll
  for (int j = 0; j < ST_HELD; ++j) {
    if (j < rounds) {
      const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
      // The table is complete: the slot's draw is the smallest draw of u.
      first_h[j] = i < hi && static_cast<uint32_t>(__ldcg(table + sh[j])) == static_cast<uint32_t>(i);
      cnt += __syncthreads_count(first_h[j]);
    }
  }
  for (int j = ST_HELD; j < rounds; ++j) {
    const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
    const bool f = i < hi && first_position(table, a.log2H, draw_value(a, row, static_cast<uint64_t>(row), i)) ==
                                 static_cast<uint32_t>(i);
    cnt += __syncthreads_count(f);
  }
  if (tid == 0) st_st_relaxed(&c.count[chunk], CNT_READY | cnt);
  {
    unsigned long long before = 0;
    if (tid < chunk) {
      unsigned long long v = st_ld_relaxed(&c.count[tid]);
      for (int poll = 0; !(v & CNT_READY); ++poll) {
        if (poll >= ST_WAIT_POLLS) {
          s_err = 1;
          v = CNT_READY;
          break;
        }
        v = st_ld_relaxed(&c.count[tid]);
      }
      before = v & ~CNT_READY;
    }
    for (int o = 16; o >= 1; o >>= 1) before += __shfl_xor_sync(FULL_MASK, before, o);
    if ((tid & 31) == 0) sw[tid >> 5] = before;
    __syncthreads();
    if (tid == 0) {
      unsigned long long b = 0;
      for (int w = 0; w < ST_THREADS / 32; ++w) b += sw[w];
      s_base = b;
      if (chunk == G - 1) S.distinct = static_cast<unsigned>(b + cnt < 0xffffffffull ? b + cnt : 0xffffffffull);
    }
    __syncthreads();
  }
  // Sample members: keys kept for the held rounds; all are stored.
  uint32_t kh[ST_HELD] = {0u, 0u};
  bool mh[ST_HELD] = {false, false};
  unsigned long long run = s_base;
#pragma unroll
  for (int j = 0; j < ST_HELD; ++j) {
    if (j < rounds) {
      unsigned long long tot;
      const unsigned long long rank = run + st_excl_scan(first_h[j] ? 1ull : 0ull, sw, &tot);
      run += tot;
      if (first_h[j] && rank < static_cast<unsigned long long>(a.S)) {
        const int64_t o = static_cast<int64_t>(row) * a.S + static_cast<int64_t>(rank);
        kh[j] = ord_key(vh[j]);
        mh[j] = true;
        a.sidx[o] = uh[j];
        a.skeys[o] = kh[j];
      }
    }
  }
  for (int j = ST_HELD; j < rounds; ++j) {
    const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
    uint32_t u = 0;
    bool f = false;
    if (i < hi) {
      u = draw_value(a, row, static_cast<uint64_t>(row), i);
      f = first_position(table, a.log2H, u) == static_cast<uint32_t>(i);
    }
    unsigned long long tot;
    const unsigned long long rank = run + st_excl_scan(f ? 1ull : 0ull, sw, &tot);
    run += tot;
    if (f && rank < static_cast<unsigned long long>(a.S)) {
      const int64_t o = static_cast<int64_t>(row) * a.S + static_cast<int64_t>(rank);
      a.sidx[o] = u;
      a.skeys[o] = ord_key(a.x[static_cast<int64_t>(row) * a.ld + u]);
    }
  }
  // The chunk's members are the sample ranks [m0, m1).
  const int64_t m0 = s_base < static_cast<unsigned long long>(a.S) ? static_cast<int64_t>(s_base) : a.S;
  const int64_t m1 = s_base + cnt < static_cast<unsigned long long>(a.S) ? static_cast<int64_t>(s_base + cnt) : a.S;
  const bool held = rounds <= ST_HELD;
  __syncthreads();

  // c. tau: the t-th largest sample key.
  unsigned long long prefix = 0, want = a.t;
  int bits = 0;
#pragma unroll 1
  for (int p = 0; p < 3; ++p) {
    const int width = p == 2 ? 10 : 11;
    const int shift = 32 - 11 * (p + 1) + (p == 2 ? 1 : 0);  // 21, 10, 0
    const unsigned nb = 1u << width;
    for (unsigned b = tid; b < nb; b += ST_THREADS) h[b] = 0;
    __syncthreads();
    if (held) {
#pragma unroll
      for (int j = 0; j < ST_HELD; ++j) {
        const bool m = mh[j] && (bits == 0 || (static_cast<unsigned long long>(kh[j]) >> (shift + width)) == prefix);
        hist_add(h, (kh[j] >> shift) & (nb - 1), m);
      }
    } else {
      for (int64_t r0 = m0; r0 < m0 + (((m1 - m0) + 31) & ~int64_t(31)); r0 += ST_THREADS) {
        const int64_t r = r0 + tid;
        const bool v = r < m1;
        const uint32_t key = v ? __ldcg(a.skeys + static_cast<int64_t>(row) * a.S + r) : 0u;
        const bool m = v && (bits == 0 || (static_cast<unsigned long long>(key) >> (shift + width)) == prefix);
        hist_add(h, (key >> shift) & (nb - 1), m);
      }
    }
    __syncthreads();
    for (unsigned b = tid; b < nb; b += ST_THREADS)
      if (h[b]) atomicAdd(&c.hist[p][b], h[b]);
    st_grid_sync(&c.bar, target += static_cast<unsigned>(G), &s_err);
    // Bins counted down from the top: thread t owns nb / 512 of them.
    if (tid == 0) {
      s_digit = 0;
      s_above = 0;
      s_count = 0;
    }
    const int per = static_cast<int>(nb) / ST_THREADS;
    const int top = static_cast<int>(nb) - 1 - tid * per;
    unsigned hv[4] = {0u, 0u, 0u, 0u};
    unsigned long long local = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q < per) {
        hv[q] = __ldcg(&c.hist[p][top - q]);
        local += hv[q];
      }
    }
    unsigned long long tot;
    const unsigned long long excl = st_excl_scan(local, sw, &tot);
    if (excl < want && want <= excl + local) {
      unsigned long long acc = excl;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q < per && want <= acc + hv[q]) {
          s_digit = static_cast<unsigned>(top - q);
          s_above = acc;
          s_count = hv[q];
          break;
        }
        acc += hv[q];
      }
    }
    __syncthreads();
    prefix = (prefix << width) | s_digit;
    want -= s_above;
    bits += width;
    const unsigned long long bucket_n = s_count;
    __syncthreads();
    if (p < 2 && bucket_n <= TAU_GATHER) {
      // The bucket's sample keys go to one list; the first CTA ranks them.
      auto put = [&](uint32_t key) {
        if ((static_cast<unsigned long long>(key) >> (32 - bits)) == prefix) {
          const unsigned pos = atomicAdd(&c.bucket_n, 1u);
          if (pos < TAU_GATHER) c.bucket[pos] = key;
        }
      };
      if (held) {
#pragma unroll
        for (int j = 0; j < ST_HELD; ++j)
          if (mh[j]) put(kh[j]);
      } else {
        for (int64_t r = m0 + tid; r < m1; r += ST_THREADS) put(__ldcg(a.skeys + static_cast<int64_t>(row) * a.S + r));
      }
      st_grid_sync(&c.bar, target += static_cast<unsigned>(G), &s_err);
      if (chunk == 0) {
        const int nl = static_cast<int>(bucket_n);
        if (tid < nl) s_list[tid] = __ldcg(&c.bucket[tid]);
        if (tid == 0) s_tau = 0;
        __syncthreads();
        if (tid < nl) {
          // The want-th largest: fewer than want keys above it, want or
          // more at or above it.
          const uint32_t e = s_list[tid];
          unsigned gt = 0, eq = 0;
          for (int j = 0; j < nl; ++j) {
            gt += s_list[j] > e;
            eq += s_list[j] == e;
          }
          if (gt < want && want <= gt + eq) s_tau = e;
        }
        __syncthreads();
        prefix = s_tau;
      }
      break;
    }
  }
  if (tid == 0) {
    if (chunk == 0) {
      S.tau_key = static_cast<uint32_t>(prefix);
      S.sel_prefix = prefix;
      S.sel_bits = 32;
      S.sel_done = 1;
    }
    if (s_err) atomicOr(&S.error, ST_ERR_WAIT);
  }
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

size_t sample_tau_ctl_bytes() { return sizeof(SampleCtl); }

namespace {
// Chunks per row: all CTAs (chunks x rows) resident at once, one per SM, at
// most 256 (the control block's count slots), no chunk shorter than 512.
int64_t sample_tau_chunks(int64_t D, int nrows) {
  int64_t G = sms() / (nrows > 0 ? nrows : 1);
  const int64_t by_len = (D + ST_THREADS - 1) / ST_THREADS;
  if (G > by_len) G = by_len;
  if (G > 256) G = 256;
  return G < 1 ? 1 : G;
}
}  // namespace

bool sample_tau_fits(int64_t D, int nrows) {
  const int64_t G = sample_tau_chunks(D, nrows);
  const int64_t Dc = (((D + G - 1) / G) + 31) & ~int64_t(31);
  return Dc <= static_cast<int64_t>(ST_HELD) * ST_THREADS;
}

cudaError_t launch_sample_tau(const SampleArgs& a, void* ctl, cudaStream_t stream) {
  const int64_t G = sample_tau_chunks(a.D, a.nrows);
  launch_kernel(k_sample_tau, dim3(static_cast<unsigned>(G), static_cast<unsigned>(a.nrows)), ST_THREADS, 0, stream,
                a, static_cast<SampleCtl*>(ctl));
  return cudaGetLastError();
}

}  // namespace profk
