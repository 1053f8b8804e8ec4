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
constexpr unsigned long long CNT_READY = 1ull << 63;
constexpr int TAU_GATHER = ST_THREADS;  // a tau bucket this small is finished by one CTA
constexpr int ST_QB = 2;                // wide form: quads per thread in flight
constexpr int ST_WIDE_ROUNDS = 24;      // wide form: at most this many rounds of 512 quads
constexpr int64_t ST_WIDE_MAX = static_cast<int64_t>(ST_WIDE_ROUNDS) * 4 * ST_THREADS;  // draws per chunk
constexpr uint32_t NOT_FIRST = 0xffffffffu;  // a repeated draw (values are below n < 2^32)

}  // namespace

// Per-row control block, zeroed at the start of every attempt.
struct SampleCtl {
  unsigned hist[3][HIST_BINS];        // tau pass histograms, summed over the chunks
  unsigned long long count[256];      // first occurrences per chunk | CNT_READY
  uint32_t bucket[TAU_GATHER];        // the sample keys of tau's final bucket
  unsigned bucket_n;
  unsigned bar;                       // grid-barrier arrivals
  unsigned abort;                     // set by a CTA whose wait gave up
  unsigned pad[61];
};
static_assert(sizeof(SampleCtl) % 16 == 0, "SampleCtl is zeroed with 16-byte stores");

namespace {

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
// have (acquire loads of the arrival count).  A wait that ends without them
// (bounded, see wait_count) sets *err, which every thread reads afterwards.
__device__ __forceinline__ void st_grid_sync(SampleCtl& c, unsigned target, int* err, int limit) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&c.bar) : "memory");
    if (!wait_count(&c.bar, target, &c.abort, limit)) *err = 1;
  }
  __syncthreads();
}

// After a wait that gave up, the CTA reports it and leaves without writing
// anything else (s_err is block-uniform here: read after a block barrier).
#define ST_LEAVE_IF_GAVE_UP()                 \
  if (s_err) {                                \
    if (tid == 0) atomicOr(&S.error, ERR_WAIT); \
    return;                                   \
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

// Draws 4q .. 4q + 3 of a row's stream, all four words of one Philox block
// (the same values as draw_value; a word that Lemire rejects takes the
// replacement path, out of line since it is rare).
__device__ __noinline__ uint32_t draw_value_slow(const SampleArgs& a, int row, uint64_t key_row, int64_t i) {
  return draw_value(a, row, key_row, i);
}

__device__ __forceinline__ void draw_quad(const SampleArgs& a, int row, uint64_t key_row, int64_t q,
                                          uint32_t (&u)[4]) {
  uint64_t w[4] = {static_cast<uint64_t>(q), static_cast<uint64_t>(a.attempt), 0ull, 0ull};
  philox4x64_10(w, a.seed, key_row);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    uint64_t v;
    u[e] = lemire64(w[e], a.n, &v) ? static_cast<uint32_t>(v) : draw_value_slow(a, row, key_row, 4 * q + e);
  }
}

// WIDE: the launch's chunks are longer than the registers hold (the host
// knows from the chunk length); each form is its own, smaller, kernel.
template <bool WIDE>
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
  __shared__ unsigned s_copies;
  __shared__ unsigned s_wcnt[ST_WIDE_ROUNDS * (ST_THREADS / 32)];
  extern __shared__ uint4 st_dyn[];
  const int row = launch_row(a.rows);
  RowState& S = a.st[row];
  SampleCtl& c = ctl[row];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_err = 0;
  const int limit = wait_limit(a.wait);
  const int64_t G = gridDim.x, chunk = blockIdx.x;
  const int64_t Dc = (((a.D + G - 1) / G) + 31) & ~int64_t(31);
  const int64_t lo = chunk * Dc < a.D ? chunk * Dc : a.D;
  const int64_t hi = lo + Dc < a.D ? lo + Dc : a.D;
  unsigned long long* table = a.table + (static_cast<int64_t>(row) << a.log2H);
  const float* xr = a.x + static_cast<int64_t>(row) * a.ld;
  const int64_t orow = static_cast<int64_t>(row) * a.S;
  const uint64_t key_row = static_cast<uint64_t>(row + a.key_row0);
  unsigned target = 0;
  // Held form: at most ST_HELD draws per thread, kept in registers.  Wide
  // form (launched with dynamic shared memory): the chunk's draws in quads,
  // thread t taking quads t, t + 512, ...; per quad one 16-byte shared-memory
  // entry that holds in turn the four draws' table slots, their values (or
  // NOT_FIRST), then the members' keys, and four membership bits.
  const bool wide = WIDE;  // the held form needs every chunk within ST_HELD x ST_THREADS
  const int nq = static_cast<int>((hi - lo + 3) / 4);
  const int nm = (nq + ST_THREADS - 1) / ST_THREADS;  // rounds of quads
  uint4* W4 = st_dyn;
  unsigned* mbits = reinterpret_cast<unsigned*>(st_dyn + Dc / 4);

  // a. Draw and insert.
  uint32_t uh[ST_HELD] = {0u, 0u};
  float vh[ST_HELD] = {0.f, 0.f};
  uint64_t sh[ST_HELD] = {0, 0};  // the slot that holds each held draw's value
  if (!wide) {
    // Both draws' value loads and home-slot swaps are issued before any
    // result is waited for (the values are used only if the draw is a
    // member, so the gather's latency overlaps the insertions).
    unsigned long long ph[ST_HELD] = {EMPTY_SLOT, EMPTY_SLOT};
#pragma unroll
    for (int j = 0; j < ST_HELD; ++j) {
      const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
      if (i < hi) uh[j] = draw_value(a, row, key_row, i);
    }
#pragma unroll
    for (int j = 0; j < ST_HELD; ++j) {
      const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
      if (i < hi) {
        vh[j] = xr[uh[j]];
        ph[j] = table_try_home(table, a.log2H, uh[j], i);
      }
    }
#pragma unroll
    for (int j = 0; j < ST_HELD; ++j) {
      const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
      if (i < hi) sh[j] = table_finish(a, row, table, uh[j], i, ph[j]);
    }
  } else {
    for (int w = tid; w < Dc / 32; w += ST_THREADS) mbits[w] = 0u;
    // ST_QB rounds at a time: 4 x ST_QB swaps in flight per thread.
    for (int m0 = 0; m0 < nm; m0 += ST_QB) {
      uint32_t u[ST_QB][4];
      unsigned long long p[ST_QB][4];
#pragma unroll
      for (int b = 0; b < ST_QB; ++b) {
        const int q = tid + (m0 + b) * ST_THREADS;
        if (q < nq) draw_quad(a, row, key_row, lo / 4 + q, u[b]);
      }
#pragma unroll
      for (int b = 0; b < ST_QB; ++b) {
        const int q = tid + (m0 + b) * ST_THREADS;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t i = lo + 4 * static_cast<int64_t>(q) + e;
          if (q < nq && i < hi) p[b][e] = table_try_home(table, a.log2H, u[b][e], i);
        }
      }
#pragma unroll
      for (int b = 0; b < ST_QB; ++b) {
        const int q = tid + (m0 + b) * ST_THREADS;
        if (q < nq) {
          uint32_t s[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int64_t i = lo + 4 * static_cast<int64_t>(q) + e;
            if (i < hi) s[e] = static_cast<uint32_t>(table_finish(a, row, table, u[b][e], i, p[b][e]));
          }
          W4[q] = make_uint4(s[0], s[1], s[2], s[3]);
        }
      }
    }
  }
  st_grid_sync(c, (target += static_cast<unsigned>(G)) + a.wait.skew, &s_err, limit);
  ST_LEAVE_IF_GAVE_UP();

  // b. First occurrences (the table is complete: a slot's draw is the
  // smallest draw of its value), their count and their place in draw order.
  bool first_h[ST_HELD] = {false, false};
  unsigned long long cnt = 0;
  if (!wide) {
#pragma unroll
    for (int j = 0; j < ST_HELD; ++j) {
      const int64_t i = lo + static_cast<int64_t>(j) * ST_THREADS + tid;
      first_h[j] = i < hi && static_cast<uint32_t>(__ldcg(table + sh[j])) == static_cast<uint32_t>(i);
      cnt += __syncthreads_count(first_h[j]);
    }
  } else {
    // Per quad: the four slots' entries (loaded ST_QB quads at a time); the
    // entry carries the value, so the quad's entry becomes the values of its
    // first occurrences.  Per (round, warp): the count of first occurrences.
    for (int m0 = 0; m0 < nm; m0 += ST_QB) {
      unsigned long long ent[ST_QB][4];
#pragma unroll
      for (int b = 0; b < ST_QB; ++b) {
        const int q = tid + (m0 + b) * ST_THREADS;
        if (q < nq) {
          const uint4 s = W4[q];
          const uint32_t sl[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            ent[b][e] = lo + 4 * static_cast<int64_t>(q) + e < hi ? __ldcg(table + sl[e]) : 0ull;
        }
      }
#pragma unroll
      for (int b = 0; b < ST_QB; ++b) {
        if (m0 + b >= nm) break;  // uniform across the block
        const int q = tid + (m0 + b) * ST_THREADS;
        uint32_t o[4] = {NOT_FIRST, NOT_FIRST, NOT_FIRST, NOT_FIRST};
        unsigned f = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t i = lo + 4 * static_cast<int64_t>(q) + e;
          if (q < nq && i < hi && static_cast<uint32_t>(ent[b][e]) == static_cast<uint32_t>(i)) {
            o[e] = static_cast<uint32_t>(ent[b][e] >> 32);
            ++f;
          }
        }
        if (q < nq) W4[q] = make_uint4(o[0], o[1], o[2], o[3]);
        const unsigned wsum = __reduce_add_sync(FULL_MASK, f);
        if (lane == 0) s_wcnt[(m0 + b) * (ST_THREADS / 32) + warp] = wsum;
      }
    }
    __syncthreads();
    // Exclusive prefix over (round, warp) in draw order; the total is the
    // chunk's count.
    const int E = nm * (ST_THREADS / 32);
    const unsigned v = tid < E ? s_wcnt[tid] : 0u;
    unsigned long long tot;
    const unsigned long long ex = st_excl_scan(v, sw, &tot);
    if (tid < E) s_wcnt[tid] = static_cast<unsigned>(ex);
    cnt = tot;
  }
  if (tid == 0) st_st_relaxed(&c.count[chunk], CNT_READY | cnt);
  {
    unsigned long long before = 0;
    if (tid < chunk) {
      unsigned long long v = st_ld_relaxed(&c.count[tid]);
      for (int poll = 0; !(v & CNT_READY); ++poll) {
        if (wait_should_stop(poll, limit, &c.abort)) {
          s_err = 1;
          v = CNT_READY;
          break;
        }
        v = st_ld_relaxed(&c.count[tid]);
      }
      before = v & ~CNT_READY;
    }
    for (int o = 16; o >= 1; o >>= 1) before += __shfl_xor_sync(FULL_MASK, before, o);
    if (lane == 0) sw[warp] = before;
    __syncthreads();
    ST_LEAVE_IF_GAVE_UP();
    if (tid == 0) {
      unsigned long long b = 0;
      for (int w = 0; w < ST_THREADS / 32; ++w) b += sw[w];
      s_base = b;
      if (chunk == G - 1) S.distinct = static_cast<unsigned>(b + cnt < 0xffffffffull ? b + cnt : 0xffffffffull);
    }
    __syncthreads();
  }
  // Sample members (first occurrences of rank < S): indices and keys stored;
  // the keys also kept (registers, or the quad's shared-memory entry).
  uint32_t kh[ST_HELD] = {0u, 0u};
  bool mh[ST_HELD] = {false, false};
  const unsigned long long Su = static_cast<unsigned long long>(a.S);
  if (!wide) {
    unsigned long long run = s_base;
#pragma unroll
    for (int j = 0; j < ST_HELD; ++j) {
      unsigned long long tot;
      const unsigned long long rank = run + st_excl_scan(first_h[j] ? 1ull : 0ull, sw, &tot);
      run += tot;
      if (first_h[j] && rank < Su) {
        const int64_t o = orow + static_cast<int64_t>(rank);
        kh[j] = ord_key(vh[j]);
        mh[j] = true;
        a.sidx[o] = uh[j];
        a.skeys[o] = kh[j];
      }
    }
  } else {
    // A quad's first rank: the chunk's base, the (round, warp) prefix and the
    // first occurrences of the warp's earlier lanes; values gathered ST_QB
    // quads at a time.
    for (int m0 = 0; m0 < nm; m0 += ST_QB) {
      uint32_t uq[ST_QB][4];
      float v[ST_QB][4];
      unsigned long long r0[ST_QB];
      unsigned fl[ST_QB];
#pragma unroll
      for (int b = 0; b < ST_QB; ++b) {  // every round of the group, also those past nm
        fl[b] = 0u;
        r0[b] = 0ull;
      }
#pragma unroll
      for (int b = 0; b < ST_QB; ++b) {
        if (m0 + b >= nm) break;  // uniform across the block
        const int q = tid + (m0 + b) * ST_THREADS;
        const uint4 e4 = q < nq ? W4[q] : make_uint4(NOT_FIRST, NOT_FIRST, NOT_FIRST, NOT_FIRST);
        uq[b][0] = e4.x;
        uq[b][1] = e4.y;
        uq[b][2] = e4.z;
        uq[b][3] = e4.w;
        unsigned f = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) f |= (uq[b][e] != NOT_FIRST ? 1u : 0u) << e;
        const unsigned cq = __popc(f);
        unsigned incl = cq;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned t = __shfl_up_sync(FULL_MASK, incl, o);
          if (lane >= o) incl += t;
        }
        r0[b] = s_base + s_wcnt[(m0 + b) * (ST_THREADS / 32) + warp] + (incl - cq);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool mem = ((f >> e) & 1u) && r0[b] + __popc(f & ((1u << e) - 1u)) < Su;
          if (mem) {
            fl[b] |= 1u << e;
            v[b][e] = xr[uq[b][e]];
          }
        }
      }
#pragma unroll
      for (int b = 0; b < ST_QB; ++b) {
        if (m0 + b >= nm || fl[b] == 0u) continue;
        const int q = tid + (m0 + b) * ST_THREADS;
        unsigned long long r = r0[b];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if ((fl[b] >> e) & 1u) {
            const uint32_t key = ord_key(v[b][e]);
            a.sidx[orow + static_cast<int64_t>(r)] = uq[b][e];
            a.skeys[orow + static_cast<int64_t>(r)] = key;
            uq[b][e] = key;
            ++r;
          }
        }
        W4[q] = make_uint4(uq[b][0], uq[b][1], uq[b][2], uq[b][3]);
        atomicOr(&mbits[q >> 3], fl[b] << ((q & 7) * 4));
      }
    }
  }
  __syncthreads();

  // Every member key of this CTA through fn(key, is_member) on every thread,
  // the same number of times (fn may be warp-collective).
  auto each_key = [&](auto&& fn) {
    if (!wide) {
#pragma unroll
      for (int j = 0; j < ST_HELD; ++j) fn(kh[j], mh[j]);
    } else {
      for (int m = 0; m < nm; ++m) {
        const int q = tid + m * ST_THREADS;
        uint4 k4 = make_uint4(0u, 0u, 0u, 0u);
        unsigned f = 0u;
        if (q < nq) {
          k4 = W4[q];
          f = (mbits[q >> 3] >> ((q & 7) * 4)) & 15u;
        }
        fn(k4.x, (f & 1u) != 0u);
        fn(k4.y, (f & 2u) != 0u);
        fn(k4.z, (f & 4u) != 0u);
        fn(k4.w, (f & 8u) != 0u);
      }
    }
  };

  // c. tau: the t-th largest sample key (and its copies among them).
  unsigned long long prefix = 0, want = a.t, copies = 0;
  int bits = 0;
#pragma unroll 1
  for (int p = 0; p < 3; ++p) {
    const int width = p == 2 ? 10 : 11;
    const int shift = 32 - 11 * (p + 1) + (p == 2 ? 1 : 0);  // 21, 10, 0
    const unsigned nb = 1u << width;
    for (unsigned b = tid; b < nb; b += ST_THREADS) h[b] = 0;
    __syncthreads();
    each_key([&](uint32_t key, bool mem) {
      const bool m = mem && (bits == 0 || (static_cast<unsigned long long>(key) >> (shift + width)) == prefix);
      hist_add(h, (key >> shift) & (nb - 1), m);
    });
    __syncthreads();
    for (unsigned b = tid; b < nb; b += ST_THREADS)
      if (h[b]) atomicAdd(&c.hist[p][b], h[b]);
    st_grid_sync(c, target += static_cast<unsigned>(G), &s_err, limit);
    ST_LEAVE_IF_GAVE_UP();
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
    copies = bucket_n;  // after the last pass: the keys equal to tau
    __syncthreads();
    if (p < 2 && bucket_n <= TAU_GATHER) {
      // The bucket's sample keys go to one list; the first CTA ranks them.
      each_key([&](uint32_t key, bool mem) {
        if (mem && (static_cast<unsigned long long>(key) >> (32 - bits)) == prefix) {
          const unsigned pos = atomicAdd(&c.bucket_n, 1u);
          if (pos < TAU_GATHER) c.bucket[pos] = key;
        }
      });
      st_grid_sync(c, target += static_cast<unsigned>(G), &s_err, limit);
      ST_LEAVE_IF_GAVE_UP();
      if (chunk == 0) {
        const int nl = static_cast<int>(bucket_n);
        if (tid < nl) s_list[tid] = __ldcg(&c.bucket[tid]);
        if (tid == 0) {
          s_tau = 0;
          s_copies = 0;
        }
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
          if (gt < want && want <= gt + eq) {
            s_tau = e;
            s_copies = eq;
          }
        }
        __syncthreads();
        prefix = s_tau;
        copies = s_copies;
      }
      break;
    }
  }
  if (tid == 0) {
    if (chunk == 0) {
      S.tau_key = static_cast<uint32_t>(prefix);
      S.tau_copies = static_cast<unsigned>(copies < 0xffffffffull ? copies : 0xffffffffull);
      S.sel_prefix = prefix;
      S.sel_bits = 32;
      S.sel_done = 1;
    }
  }
}
#undef ST_LEAVE_IF_GAVE_UP

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

// Dynamic shared memory of the wide form: a 16-byte entry per quad and four
// membership bits per quad.
size_t sample_tau_wide_smem(int64_t Dc) { return static_cast<size_t>(Dc) * 4 + static_cast<size_t>(Dc) / 8; }

int64_t sample_tau_chunk_len(int64_t D, int nrows) {
  const int64_t G = sample_tau_chunks(D, nrows);
  return (((D + G - 1) / G) + 31) & ~int64_t(31);
}
}  // namespace

bool sample_tau_fits(int64_t D, int nrows, uint64_t n) {
  const int64_t Dc = sample_tau_chunk_len(D, nrows);
  if (Dc <= static_cast<int64_t>(ST_HELD) * ST_THREADS) return true;
  return Dc <= ST_WIDE_MAX && n < (1ull << 32);
}

cudaError_t launch_sample_tau(const SampleArgs& a, void* ctl, cudaStream_t stream) {
  const int64_t G = sample_tau_chunks(a.D, a.nrows);
  const int64_t Dc = sample_tau_chunk_len(a.D, a.nrows);
  if (Dc > static_cast<int64_t>(ST_HELD) * ST_THREADS) {
    if (Dc > ST_WIDE_MAX || a.n >= (1ull << 32)) return cudaErrorInvalidValue;
    cudaFuncSetAttribute(k_sample_tau<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(sample_tau_wide_smem(ST_WIDE_MAX)));
    launch_kernel(k_sample_tau<true>, dim3(static_cast<unsigned>(G), static_cast<unsigned>(a.nrows)), ST_THREADS,
                  sample_tau_wide_smem(Dc), stream, a, static_cast<SampleCtl*>(ctl));
  } else {
    launch_kernel(k_sample_tau<false>, dim3(static_cast<unsigned>(G), static_cast<unsigned>(a.nrows)), ST_THREADS, 0,
                  stream, a, static_cast<SampleCtl*>(ctl));
  }
  return cudaGetLastError();
}

}  // namespace profk
