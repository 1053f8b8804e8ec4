// Step 1 of Prof-K: uniform sampling of S indices without replacement and the
// gather of their values ("Prof-K: Probabilistic One-Pass Filtering for
// Efficient Top-k Selection", Section 3, stage 1), and, in the persistent
// form, step 2: tau, the t-th largest sampled value (stage 2).
//
// The sample is pi(0), ..., pi(S-1), where pi is a keyed pseudo-random
// permutation of [0, n).  pi is a twelve-round Feistel network on [0, 2^b),
// b = max(2, ceil(log2 n)): round i splits the state into its high part L
// and its low w bits R (w = floor(b/2) in round 0, then the widths
// alternate) and maps it to (R << (b - w)) | (L xor f_i(R) mod 2^(b - w)),
// with f_i(R) = mix(R xor K_i), mix the SplitMix64 output function (Steele,
// Lea and Flood, OOPSLA 2014) and K_0 .. K_11 the words of the
// Philox4x64-10 blocks (q, attempt, 0, 0), q = 0, 1, 2, under the key
// (seed, row).  A value at or above n is encrypted again until it falls
// below n (cycle-walking: Black and Rogaway, "Ciphers with arbitrary finite
// domains"), which makes pi a permutation of [0, n).  The S indices are
// therefore distinct by construction and each is computed on its own: no
// table of drawn values, no repeat removal, no ordering across threads.
//
// Three forms:
//  * k_sample_draw (one thread per sample position, all rows of a launch):
//    the sample and its keys, optionally with the first 11-bit pass of the
//    tau selection fused (the last block picks the digit; launch_select
//    finishes);
//  * k_sample_lists (t <= TAU_CAND, rows too many for the persistent form):
//    CTAs of 256 threads take up to 2048 positions of one row and publish
//    lists of their t largest keys; a CTA that finds every list of its row
//    published selects tau among them, with no CTA waiting for another;
//  * k_sample_tau (the main path, one 512-thread CTA per SM and contiguous
//    chunk of at most 1024 sample positions, all CTAs of the launch resident
//    together): the sample, then tau.  For t <= TAU_CAND (8) every CTA
//    selects its own t largest keys (rounds of block maxima) and lists them;
//    one CTA waits for every list (a bounded wait) and selects tau among
//    them: the t-th largest of the sample is among the t largest of its own
//    chunk.  For larger t, 11/11/10-bit MSD passes whose chunk histograms
//    meet in global atomics, every CTA taking the same digit after each
//    pass's barrier.
#include <atomic>
#include <chrono>

#include <unistd.h>

#include "kernels.h"

namespace profk {
namespace {

constexpr int FEISTEL_ROUNDS = 12;
constexpr int WALK_MAX = 1024;       // cycle-walking steps (each ends below n with probability > 1/2)
constexpr int DRAW_THREADS = 1024;   // k_sample_draw
constexpr int ST_THREADS = 512;      // k_sample_tau
constexpr int ST_HELD = 2;           // sample positions per thread (keys kept in registers)
// Largest t of the candidate-list selection (whose selections take rounds of
// maxima).  For larger t the grid passes measured faster: at t = 93 the
// candidate lists held G t ~ 12K keys for one CTA to select among (2^30,
// k = 2^19: sampling stage 36.5 us against 23.5 us with the passes).
constexpr int TAU_CAND = 8;
constexpr int SMALL_T = TAU_CAND;
constexpr int TAU_GATHER = ST_THREADS;  // a tau bucket this small is finished by one CTA (t > TAU_CAND)
constexpr int MAX_CHUNKS = 256;

// A sampled value.  The positions are spread over the whole row, so no two
// share a cache line: the load bypasses L1, whose misses fill whole lines,
// and asks L2 for the one 32-byte sector that holds the value.
__device__ __forceinline__ float gather_one(const float* p) { return __ldcg(p); }

// b = max(2, ceil(log2 n)): the Feistel network permutes [0, 2^b), 2^b >= n.
__device__ __forceinline__ int domain_bits(uint64_t n) { return n <= 4 ? 2 : 64 - __clzll(n - 1); }

// The round keys of a row and attempt, computed by threads 0-2 of the block
// into K (shared memory); the caller synchronizes the block before use.
__device__ __forceinline__ void round_keys(uint64_t seed, uint64_t key_row, uint64_t attempt, uint64_t* K) {
  const int q = threadIdx.x;
  if (q < FEISTEL_ROUNDS / 4) {
    uint64_t c[4] = {static_cast<uint64_t>(q), attempt, 0ull, 0ull};
    philox4x64_10(c, seed, key_row);
#pragma unroll
    for (int e = 0; e < 4; ++e) K[4 * q + e] = c[e];
  }
}

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// One pass of the network.  Rows hold at most 2^32 elements, so b <= 32: the
// state and both halves (at most 16 bits each) are 32-bit words, and only the
// round function works on 64 bits.
__device__ __forceinline__ uint32_t feistel(uint32_t x, int b, const uint64_t* K) {
  int w = b >> 1;
#pragma unroll
  for (int i = 0; i < FEISTEL_ROUNDS; ++i) {
    const int wl = b - w;
    const uint32_t right = x & ((1u << w) - 1u);
    const uint32_t left = x >> w;
    const uint32_t f = static_cast<uint32_t>(mix64(static_cast<uint64_t>(right) ^ K[i]));
    x = (right << wl) | (left ^ (f & ((1u << wl) - 1u)));
    w = wl;
  }
  return x;
}

// pi(j) for positions x[0..H) of one thread (each below n), computed
// together so that their Philox chains interleave; a position whose walk[h]
// is false on entry is left alone.  Returns false if some walk did not end
// within WALK_MAX steps (only a broken network could; its index is then 0).
template <int H>
__device__ __forceinline__ bool permute(uint64_t (&x)[H], bool (&walk)[H], uint64_t n, int b, const uint64_t* K) {
  for (int s = 0; s < WALK_MAX; ++s) {
    bool any = false;
#pragma unroll
    for (int h = 0; h < H; ++h) any |= walk[h];
    if (!any) return true;
#pragma unroll
    for (int h = 0; h < H; ++h) {
      const uint64_t y = feistel(static_cast<uint32_t>(x[h]), b, K);
      if (walk[h]) {
        x[h] = y;
        walk[h] = y >= n;
      }
    }
  }
  bool ok = true;
#pragma unroll
  for (int h = 0; h < H; ++h) {
    if (walk[h]) {
      x[h] = 0;
      ok = false;
    }
  }
  return ok;
}

// Block-wide exclusive scan (thread order) of one u64 per thread; *total is
// the block's sum.  sw holds 33 words of shared memory.
template <int NT>
__device__ __forceinline__ unsigned long long excl_scan_block(unsigned long long v, unsigned long long* sw,
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
    const unsigned long long w = lane < NT / 32 ? sw[lane] : 0ull;
    unsigned long long wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(FULL_MASK, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < NT / 32) sw[lane] = wi - w;
    if (lane == 31) sw[32] = wi;
  }
  __syncthreads();
  const unsigned long long r = sw[warp] + incl - v;
  *total = sw[32];
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------------------
// The step-by-step form.

// Last block of k_sample_draw: the first radix pass of the tau selection
// (step 2) over the row's S sample keys is complete in the 2048-bin histogram
// of their top 11 bits; pick the bin that holds the t-th largest key and
// leave the selection state at "11 bits resolved" for the two remaining
// passes (launch_select with first_pass = 1).
__device__ __noinline__ void tau_first_digit(const SampleArgs& a, int row) {
  constexpr int NW = DRAW_THREADS / 32;
  __shared__ unsigned long long s_scan[NW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  RowState& S = a.st[row];
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
  if (excl < want && want <= excl + v) {
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

__global__ void __launch_bounds__(DRAW_THREADS) k_sample_draw(SampleArgs a, int64_t key_row0) {
  pdl_trigger();
  pdl_wait();
  const int row = launch_row(a.rows);
  RowState& S = a.st[row];
  __shared__ uint64_t s_keys[FEISTEL_ROUNDS];
  round_keys(a.seed, static_cast<uint64_t>(row + key_row0), static_cast<uint64_t>(a.attempt), s_keys);
  __syncthreads();
  const int64_t j = static_cast<int64_t>(blockIdx.x) * DRAW_THREADS + threadIdx.x;
  const bool has = j < a.S;
  uint32_t key = 0;
  if (has) {
    uint64_t x[1] = {static_cast<uint64_t>(j)};
    bool walk[1] = {true};
    if (!permute<1>(x, walk, a.n, domain_bits(a.n), s_keys)) atomicOr(&S.error, 1u);
    const uint32_t u = static_cast<uint32_t>(x[0]);
    key = ord_key(gather_one(a.x + static_cast<int64_t>(row) * a.ld + u));
    const int64_t o = static_cast<int64_t>(row) * a.S + j;
    a.sidx[o] = u;
    a.skeys[o] = key;
  }
  if (j == 0) S.distinct = static_cast<unsigned>(a.S < 0xffffffffll ? a.S : 0xffffffffll);
  if (!a.tau_pass1) return;
  // First pass of step 2 fused: the keys' top 11 bits go to the row's
  // histogram (block-local first, then one atomic per non-empty bin); the
  // last block to finish picks the digit.
  __shared__ unsigned s_h[HIST_BINS];
  for (int b = threadIdx.x; b < HIST_BINS; b += DRAW_THREADS) s_h[b] = 0;
  __syncthreads();
  hist_add(s_h, key >> (32 - HIST_BITS), has);
  __syncthreads();
  for (int b = threadIdx.x; b < HIST_BINS; b += DRAW_THREADS)
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

// ---------------------------------------------------------------------------
// The persistent form.

// Per-row control block, zeroed at the start of every attempt.
struct SampleCtl {
  unsigned hist[3][HIST_BINS];  // tau pass histograms, summed over the chunks (t > TAU_CAND)
  uint32_t bucket[TAU_GATHER];  // the sample keys of tau's final bucket (t > TAU_CAND)
  unsigned bucket_n;
  unsigned bar;                 // grid-barrier arrivals (t > TAU_CAND)
  unsigned abort;               // set by a CTA whose wait gave up
  unsigned pad[61];
};
static_assert(sizeof(SampleCtl) % 16 == 0, "SampleCtl is zeroed with 16-byte stores");

// Per-row candidate lists of the selection for t <= TAU_CAND (written whole
// by every launch, so not zeroed): chunk c's t largest keys at key[c t ..],
// its t-th largest key with the number of its copies the list leaves out,
// and its flag: (epoch << 1) | (a walk of the chunk did not end), written
// once the list is complete.  The launch's epoch is unique to it (a process
// nonce and a launch counter), so a flag left by an earlier launch, or any
// other content of fresh memory, does not read as written.
struct SampleCand {
  uint32_t key[MAX_CHUNKS * TAU_CAND];
  uint32_t kth[MAX_CHUNKS];
  uint32_t extra[MAX_CHUNKS];
  unsigned long long flag[MAX_CHUNKS];
};

namespace {

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
#define ST_LEAVE_IF_GAVE_UP()                   \
  if (s_err) {                                  \
    if (tid == 0) atomicOr(&S.error, ERR_WAIT); \
    return;                                     \
  }

// Shared memory of the selections (the passes of the t > TAU_CAND path, and
// the rounds of maxima below).
struct SelSmem {
  unsigned h[HIST_BINS];
  unsigned long long sw[33];
  unsigned digit;
  unsigned long long above, count;
  unsigned wmax[ST_THREADS / 32], wcnt[ST_THREADS / 32];
};

// The want-th largest of the keys that each_key(fn) presents (fn(key,
// valid), called the same number of times on every thread), for a small
// want: rounds of "the largest key below the previous round's, and its
// copies", a block maximum and a block count each, until the copies reach
// the rank left (at most want rounds).  Returns the key; *above = keys
// strictly larger, *eq = keys equal to it.  The block must hold at least
// want valid keys.
template <int NT = ST_THREADS, class EachKey>
__device__ __forceinline__ uint32_t block_select_small(EachKey each_key, unsigned long long want, SelSmem& sm,
                                                       unsigned long long* above, unsigned long long* eq) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long want0 = want;
  uint32_t bound = 0xffffffffu;  // keys at or above it are taken (all keys remain in the first round)
  bool first = true;
  uint32_t result = 0;
  for (int r = 0; r < SMALL_T; ++r) {
    uint32_t m = 0;
    each_key([&](uint32_t key, bool v) {
      if (v && (first || key < bound) && key > m) m = key;
    });
    m = __reduce_max_sync(FULL_MASK, m);
    if (lane == 0) sm.wmax[warp] = m;
    __syncthreads();
    m = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) m = sm.wmax[w] > m ? sm.wmax[w] : m;
    unsigned c = 0;
    each_key([&](uint32_t key, bool v) { c += (v && (first || key < bound) && key == m) ? 1u : 0u; });
    c = __reduce_add_sync(FULL_MASK, c);
    if (lane == 0) sm.wcnt[warp] = c;
    __syncthreads();
    unsigned long long cnt = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) cnt += sm.wcnt[w];
    __syncthreads();  // wmax and wcnt are rewritten by the next round
    result = m;
    *eq = cnt;
    if (cnt >= want) break;
    want -= cnt;
    bound = m;
    first = false;
  }
  *above = want0 - want;
  return result;
}

// The attempt's set-up (see SampleArgs::zero_ctl), done by the sampler in
// place of a reset kernel: the first CTA of the row zeroes the row state,
// every CTA its share of the refinement's control block and of the tie
// step's block counts.  The kernels that use them come later on the stream;
// the CTA that writes tau does so after chunk 0 has published its list.
template <int NT>
__device__ __forceinline__ void attempt_setup(const SampleArgs& a, RowState& S, int row, int64_t chunk, int64_t G) {
  const int tid = threadIdx.x;
  const int64_t gt = chunk * NT + tid, gs = G * NT;
  if (a.zero_ctl) {
    ulonglong2* zc = reinterpret_cast<ulonglong2*>(a.zero_ctl + static_cast<int64_t>(row) * a.zero_words);
    for (int64_t i = gt; i < a.zero_words / 2; i += gs) zc[i] = make_ulonglong2(0ull, 0ull);
  }
  if (a.zero_eq) {
    unsigned* ze = a.zero_eq + static_cast<int64_t>(row) * a.zero_nb;
    for (int64_t i = gt; i < a.zero_nb; i += gs) ze[i] = 0u;
  }
  if (chunk == 0) {
    for (int b = tid; b < HIST_BINS; b += NT) S.hist[b] = 0u;
    if (tid == 0) {
      S.R_ge = 0;
      S.R_gt = 0;
      S.nan = 0;
      S.error = 0;
      S.sel_rank = a.t;
      S.sel_above = 0;
      S.sel_bucket = 0;
      S.sel_thresh = 0;
      S.sel_nan = 0;
      S.done_blocks = 0;
      S.compact_count = 0;
      S.skip = 0;
      S.tie_gt = 0;
      S.settled = 0;
      S.vdiff = 0;
    }
  }
}

template <bool CAND>
__global__ void __launch_bounds__(ST_THREADS, 1) k_sample_tau(SampleArgs a, SampleCtl* ctl, SampleCand* cands,
                                                             unsigned long long epoch) {
  pdl_trigger();
  // The first attempt of the candidate lists' form computes its first
  // position (shared memory and registers only) before it waits for the
  // preceding kernel, and reads or writes global memory only after.  Later
  // attempts first read what earlier ones settled; the passes' form follows
  // a reset kernel of its own attempt.
  const bool early = CAND && a.attempt == 0;
  if (!early) pdl_wait();
  extern __shared__ uint32_t s_cand[];  // CAND: the G t candidates, in the first CTA
  __shared__ SelSmem sm;
  __shared__ int s_err, s_fail;
  __shared__ unsigned s_pos;
  __shared__ uint64_t s_keys[FEISTEL_ROUNDS];
  const int row = launch_row(a.rows);
  RowState& S = a.st[row];
  SampleCtl& c = ctl[row];
  const int tid = threadIdx.x;
  const int64_t G = gridDim.x, chunk = blockIdx.x;
  if (settled_before(S, a.attempt)) return;  // every CTA of the row leaves: nothing is waited for
  if (tid == 0) {
    s_err = 0;
    s_fail = 0;
    s_pos = 0;
  }
  round_keys(a.seed, static_cast<uint64_t>(row + a.key_row0), static_cast<uint64_t>(a.attempt), s_keys);
  __syncthreads();
  const int limit = wait_limit(a.wait);
  const int64_t Cn = (((a.S + G - 1) / G) + 31) & ~int64_t(31);
  const int64_t lo = chunk * Cn < a.S ? chunk * Cn : a.S;
  const int64_t hi = lo + Cn < a.S ? lo + Cn : a.S;
  const float* xr = a.x + static_cast<int64_t>(row) * a.ld;
  const int64_t orow = static_cast<int64_t>(row) * a.S;

  // a. The chunk's sample positions, their values and keys (each position's
  // gather is in flight while the next position is computed; the first
  // position is computed before the wait, then the attempt's set-up).
  uint64_t xs[ST_HELD];
  bool mh[ST_HELD];
  float vh[ST_HELD];
  bool ok = true;
#pragma unroll
  for (int h = 0; h < ST_HELD; ++h) {
    const int64_t j = lo + static_cast<int64_t>(h) * ST_THREADS + tid;
    uint64_t x1[1] = {static_cast<uint64_t>(j)};
    bool w1[1] = {j < hi};
    mh[h] = w1[0];
    ok &= permute<1>(x1, w1, a.n, domain_bits(a.n), s_keys);
    if (h == 0) {
      if (early) pdl_wait();
      if constexpr (CAND) attempt_setup<ST_THREADS>(a, S, row, chunk, G);
    }
    xs[h] = x1[0];
    vh[h] = mh[h] ? gather_one(xr + x1[0]) : 0.f;
  }
  // A walk that did not end: reported through the chunk's flag (the
  // candidate lists' form, whose first CTA owns the error word) or the error
  // word (the passes' form).
  if (!ok) s_fail = 1;
  uint32_t kh[ST_HELD];
#pragma unroll
  for (int h = 0; h < ST_HELD; ++h) kh[h] = ord_key(vh[h]);
  // The sample and RowState::distinct.  Called by every thread.
  auto publish_sample = [&]() {
#pragma unroll
    for (int h = 0; h < ST_HELD; ++h) {
      if (mh[h] && a.store_sample) {
        const int64_t o = orow + lo + static_cast<int64_t>(h) * ST_THREADS + tid;
        a.sidx[o] = static_cast<uint32_t>(xs[h]);
        a.skeys[o] = kh[h];
      }
    }
    if (chunk == 0 && tid == 0) S.distinct = static_cast<unsigned>(a.S < 0xffffffffll ? a.S : 0xffffffffll);
    if constexpr (!CAND) {
      __syncthreads();
      if (tid == 0 && s_fail) atomicOr(&S.error, 1u);
    }
  };
  auto each_key = [&](auto&& fn) {
#pragma unroll
    for (int h = 0; h < ST_HELD; ++h) fn(kh[h], mh[h]);
  };
  const unsigned long long t = a.t;

  if constexpr (CAND) {
    // b. This chunk's t largest keys: those above its t-th largest K, and
    // copies of K to make t (or all its keys, padded with zero keys, when
    // it has fewer than t), then its arrival.
    SampleCand& cd = cands[row];
    const int64_t cnt = hi - lo;
    const bool short_chunk = cnt < static_cast<int64_t>(t);
    uint32_t K = 0;
    unsigned long long above = 0, eq = 0;
    if (!short_chunk)
      K = block_select_small(each_key, t, sm, &above, &eq);
    else
      above = static_cast<unsigned long long>(cnt);  // every key goes to the list
    publish_sample();
    uint32_t* mine = cd.key + chunk * static_cast<int64_t>(t);
#pragma unroll
    for (int h = 0; h < ST_HELD; ++h) {
      if (mh[h] && (short_chunk || kh[h] > K)) mine[atomicAdd(&s_pos, 1u)] = kh[h];
    }
    for (unsigned long long q = above + tid; q < t; q += ST_THREADS) mine[q] = short_chunk ? 0u : K;
    if (tid == 0) {
      cd.kth[chunk] = K;
      cd.extra[chunk] = short_chunk ? 0u : static_cast<unsigned>(eq - (t - above));
    }
    __syncthreads();
    if (tid == 0) {
      const unsigned long long f = (epoch << 1) | (s_fail ? 1ull : 0ull);
      asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(&cd.flag[chunk]), "l"(f) : "memory");
    }
    if (chunk != 0) return;
    // c. The first CTA waits for every list (thread c for chunk c's flag,
    // bounded), then selects tau among the G t candidates.  The copies of
    // tau in the sample are the listed ones plus those left out by the
    // chunks whose t-th largest is tau (a chunk's t-th largest is at most
    // tau, and below it every copy of tau is listed).
    (void)c;
    const int64_t nflags = G + a.wait.skew;  // a test setting waits for a flag no chunk writes
    for (int64_t ch = tid; ch < nflags; ch += ST_THREADS) {
      unsigned long long f;
      for (int poll = 0;; ++poll) {
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(f) : "l"(&cd.flag[ch]) : "memory");
        if ((f >> 1) == epoch) break;
        if (poll >= limit) {
          s_err = 1;
          break;
        }
      }
      if ((f >> 1) == epoch && (f & 1ull)) s_fail = 1;
    }
    __syncthreads();
    ST_LEAVE_IF_GAVE_UP();
    if (tid == 0 && s_fail) atomicOr(&S.error, 1u);
    // The lists into shared memory, eight independent loads per thread in
    // flight at a time, then the selection there.
    const int64_t total = G * static_cast<int64_t>(t);
    for (int64_t base = 0; base < total; base += 8 * ST_THREADS) {
      uint32_t v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t e = base + i * ST_THREADS + tid;
        v[i] = e < total ? __ldcg(cd.key + e) : 0u;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t e = base + i * ST_THREADS + tid;
        if (e < total) s_cand[e] = v[i];
      }
    }
    __syncthreads();
    const int per = static_cast<int>((total + ST_THREADS - 1) / ST_THREADS);
    auto each_cand = [&](auto&& fn) {
      for (int q = 0; q < per; ++q) {
        const int64_t e = static_cast<int64_t>(q) * ST_THREADS + tid;
        const bool v = e < total;
        fn(v ? s_cand[e] : 0u, v);
      }
    };
    unsigned long long cabove = 0, ceq = 0;
    const uint32_t tau = block_select_small(each_cand, t, sm, &cabove, &ceq);
    unsigned long long more = 0;
    for (int64_t ch = tid; ch < G; ch += ST_THREADS)
      if (__ldcg(&cd.kth[ch]) == tau) more += __ldcg(&cd.extra[ch]);
    unsigned long long tot;
    excl_scan_block<ST_THREADS>(more, sm.sw, &tot);
    if (tid == 0) {
      const unsigned long long copies = ceq + tot;
      S.tau_key = tau;
      S.tau_copies = static_cast<unsigned>(copies < 0xffffffffull ? copies : 0xffffffffull);
      S.sel_prefix = tau;
      S.sel_bits = 32;
      S.sel_done = 1;
    }
  } else {
    // b'. tau = the t-th largest sample key (and its copies among them) by
    // 11/11/10-bit passes whose chunk histograms meet in global atomics.
    publish_sample();
    unsigned long long prefix = 0, want = t, copies = 0;
    int bits = 0;
    unsigned target = 0;
    __shared__ uint32_t s_list[TAU_GATHER];
    __shared__ uint32_t s_tau;
    __shared__ unsigned s_copies;
#pragma unroll 1
    for (int p = 0; p < 3; ++p) {
      const int width = p == 2 ? 10 : 11;
      const int shift = 32 - 11 * (p + 1) + (p == 2 ? 1 : 0);  // 21, 10, 0
      const unsigned nb = 1u << width;
      for (unsigned b = tid; b < nb; b += ST_THREADS) sm.h[b] = 0;
      __syncthreads();
      each_key([&](uint32_t key, bool mem) {
        const bool m = mem && (bits == 0 || (static_cast<unsigned long long>(key) >> (shift + width)) == prefix);
        hist_add(sm.h, (key >> shift) & (nb - 1), m);
      });
      __syncthreads();
      for (unsigned b = tid; b < nb; b += ST_THREADS)
        if (sm.h[b]) atomicAdd(&c.hist[p][b], sm.h[b]);
      st_grid_sync(c, (target += static_cast<unsigned>(G)) + (p == 0 ? a.wait.skew : 0u), &s_err, limit);
      ST_LEAVE_IF_GAVE_UP();
      // Bins counted down from the top: thread t owns nb / 512 of them.
      if (tid == 0) {
        sm.digit = 0;
        sm.above = 0;
        sm.count = 0;
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
      const unsigned long long excl = excl_scan_block<ST_THREADS>(local, sm.sw, &tot);
      if (excl < want && want <= excl + local) {
        unsigned long long acc = excl;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q < per && want <= acc + hv[q]) {
            sm.digit = static_cast<unsigned>(top - q);
            sm.above = acc;
            sm.count = hv[q];
            break;
          }
          acc += hv[q];
        }
      }
      __syncthreads();
      prefix = (prefix << width) | sm.digit;
      want -= sm.above;
      bits += width;
      const unsigned long long bucket_n = sm.count;
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
            unsigned gt = 0, eqn = 0;
            for (int jj = 0; jj < nl; ++jj) {
              gt += s_list[jj] > e;
              eqn += s_list[jj] == e;
            }
            if (gt < want && want <= gt + eqn) {
              s_tau = e;
              s_copies = eqn;
            }
          }
          __syncthreads();
          prefix = s_tau;
          copies = s_copies;
        }
        break;
      }
    }
    if (tid == 0 && chunk == 0) {
      S.tau_key = static_cast<uint32_t>(prefix);
      S.tau_copies = static_cast<unsigned>(copies < 0xffffffffull ? copies : 0xffffffffull);
      S.sel_prefix = prefix;
      S.sel_bits = 32;
      S.sel_done = 1;
    }
  }
}
#undef ST_LEAVE_IF_GAVE_UP

// ---------------------------------------------------------------------------
// The lists form (t <= TAU_CAND, any number of rows).  A CTA of LS_THREADS
// threads takes LS_THREADS x H consecutive sample positions of one row
// (thread tid: positions lo + h LS_THREADS + tid), lists its t largest keys
// as the persistent form's chunks do, and publishes the list with a flag
// stamped with the launch's epoch (unique to the launch, so the flags need
// no zeroing).  It then reads the row's flags: a CTA that finds every chunk
// published selects tau among the lists.  No CTA waits for another.
//
// Selections of a few largest keys go warp by warp (reductions inside the
// warp, no block barrier), then one warp merges the warps' lists: the t
// largest of a set are among the union of the t largest of its parts.
constexpr int LS_THREADS = 256;
constexpr int LS_WARPS = LS_THREADS / 32;
constexpr int LS_MAX_H = 8;

// The want-th largest of the keys that each_key(fn) presents to the warp
// (fn(key, valid), called the same number of times on every lane): rounds
// of "the largest key below the previous round's, and its copies", at most
// want rounds.  *above = keys strictly larger, *eq = keys equal to it.  The
// warp must hold at least want valid keys.
template <class EachKey>
__device__ __forceinline__ uint32_t warp_select_small(EachKey each_key, unsigned want, unsigned* above,
                                                      unsigned* eq) {
  const unsigned want0 = want;
  uint32_t bound = 0xffffffffu, result = 0;
  bool first = true;
  unsigned cnt = 0;
  for (int r = 0; r < SMALL_T; ++r) {
    uint32_t m = 0;
    each_key([&](uint32_t key, bool v) {
      if (v && (first || key < bound) && key > m) m = key;
    });
    m = __reduce_max_sync(FULL_MASK, m);
    unsigned c = 0;
    each_key([&](uint32_t key, bool v) { c += (v && (first || key < bound) && key == m) ? 1u : 0u; });
    cnt = __reduce_add_sync(FULL_MASK, c);
    result = m;
    if (cnt >= want) break;
    want -= cnt;
    bound = m;
    first = false;
  }
  *above = want0 - want;
  *eq = cnt;
  return result;
}

// The t largest keys of a warp's keys into out[0, t): those above the t-th
// largest Kw, in lane order, then copies of Kw (a warp with fewer than t
// keys lists them all, padded with zero keys, and Kw = 0).  Returns Kw;
// *extra = the copies of Kw that the list leaves out.
template <class EachKey>
__device__ __forceinline__ uint32_t warp_list_t(EachKey each_key, unsigned t, uint32_t* out, unsigned* extra) {
  const int lane = threadIdx.x & 31;
  unsigned vc = 0;
  each_key([&](uint32_t, bool v) { vc += v ? 1u : 0u; });
  vc = __reduce_add_sync(FULL_MASK, vc);
  const bool few = vc < t;
  uint32_t K = 0;
  unsigned above = vc, eq = 0;
  if (!few) K = warp_select_small(each_key, t, &above, &eq);
  unsigned pos = 0;
  each_key([&](uint32_t key, bool v) {
    const bool take = v && (few || key > K);
    const unsigned m = __ballot_sync(FULL_MASK, take);
    if (take) out[pos + __popc(m & ((1u << lane) - 1u))] = key;
    pos += __popc(m);
  });
  for (unsigned q = above + lane; q < t; q += 32) out[q] = K;
  *extra = few ? 0u : eq - (t - above);
  return K;
}

struct ListsSmem {
  uint32_t key[LS_WARPS * TAU_CAND];  // each warp's t largest
  uint32_t kth[LS_WARPS];
  unsigned extra[LS_WARPS];
};

// The t largest keys of the block (each warp's keys presented by each_key),
// listed by warp 0 into out[0, t).  Returns the block's t-th largest K to
// warp 0, with *extra = the block's copies of K that the list leaves out.
// The block must hold at least t keys.  Ends with warp 0 alone (the other
// warps return 0 and must not use the list before a block barrier).
template <class EachKey>
__device__ __forceinline__ uint32_t block_list_t(EachKey each_key, unsigned t, ListsSmem& sm, uint32_t* out,
                                                 unsigned* extra) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned ex;
  const uint32_t Kw = warp_list_t(each_key, t, sm.key + warp * t, &ex);
  if (lane == 0) {
    sm.kth[warp] = Kw;
    sm.extra[warp] = ex;
  }
  __syncthreads();
  if (warp != 0) return 0;
  const unsigned total = LS_WARPS * t;
  auto each_cand = [&](auto&& fn) {
#pragma unroll
    for (int q = 0; q < (LS_WARPS * TAU_CAND + 31) / 32; ++q) {
      const unsigned e = q * 32 + lane;
      const bool v = e < total;
      fn(v ? sm.key[e] : 0u, v);
    }
  };
  unsigned cex;
  const uint32_t K = warp_list_t(each_cand, t, out, &cex);
  // The copies of K outside the candidates: a warp whose t-th largest is
  // above K cannot exist (its t keys would all be above K), and one whose
  // t-th largest is below K listed all its copies of K.
  unsigned more = (lane < LS_WARPS && sm.kth[lane] == K) ? sm.extra[lane] : 0u;
  more = __reduce_add_sync(FULL_MASK, more);
  *extra = cex + more;
  return K;
}

template <int H>
__global__ void __launch_bounds__(LS_THREADS) k_sample_lists(SampleArgs a, SampleCand* cands,
                                                            unsigned long long epoch) {
  pdl_trigger();
  // As in k_sample_tau: the first attempt computes its first positions
  // before it waits for the preceding kernel.
  const bool early = a.attempt == 0;
  if (!early) pdl_wait();
  __shared__ ListsSmem sm;
  __shared__ uint64_t s_keys[FEISTEL_ROUNDS];
  __shared__ uint32_t s_cand[MAX_CHUNKS * TAU_CAND];  // a finishing CTA: every list of the row
  __shared__ uint32_t s_final[TAU_CAND];
  __shared__ unsigned s_pos;
  __shared__ int s_fail;
  const int row = launch_row(a.rows);
  RowState& S = a.st[row];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t G = gridDim.x, chunk = blockIdx.x;
  if (settled_before(S, a.attempt)) return;  // every CTA of the row leaves before publishing
  if (tid == 0) {
    s_pos = 0;
    s_fail = 0;
  }
  round_keys(a.seed, static_cast<uint64_t>(row + a.key_row0), static_cast<uint64_t>(a.attempt), s_keys);
  __syncthreads();
  const int64_t lo = chunk * (static_cast<int64_t>(LS_THREADS) * H);
  const float* xr = a.x + static_cast<int64_t>(row) * a.ld;
  const int64_t orow = static_cast<int64_t>(row) * a.S;
  const int b = domain_bits(a.n);
  // The positions in two halves: the first half's gathers are in flight
  // while the second half's indices are computed.
  constexpr int H1 = H > 1 ? H / 2 : 1, H2 = H - H1;
  uint64_t xs[H];
  bool mh[H];
  float vh[H];
  bool ok = true;
  {
    uint64_t x1[H1];
    bool w1[H1];
#pragma unroll
    for (int h = 0; h < H1; ++h) {
      const int64_t j = lo + static_cast<int64_t>(h) * LS_THREADS + tid;
      x1[h] = static_cast<uint64_t>(j);
      w1[h] = mh[h] = j < a.S;
    }
    ok &= permute<H1>(x1, w1, a.n, b, s_keys);
    if (early) pdl_wait();
    attempt_setup<LS_THREADS>(a, S, row, chunk, G);
#pragma unroll
    for (int h = 0; h < H1; ++h) {
      xs[h] = x1[h];
      vh[h] = mh[h] ? gather_one(xr + x1[h]) : 0.f;
    }
  }
  if constexpr (H2 > 0) {
    uint64_t x2[H2 > 0 ? H2 : 1];
    bool w2[H2 > 0 ? H2 : 1];
#pragma unroll
    for (int h = 0; h < H2; ++h) {
      const int64_t j = lo + static_cast<int64_t>(H1 + h) * LS_THREADS + tid;
      x2[h] = static_cast<uint64_t>(j);
      w2[h] = mh[H1 + h] = j < a.S;
    }
    ok &= permute<H2>(x2, w2, a.n, b, s_keys);
#pragma unroll
    for (int h = 0; h < H2; ++h) {
      xs[H1 + h] = x2[h];
      vh[H1 + h] = mh[H1 + h] ? gather_one(xr + x2[h]) : 0.f;
    }
  }
  if (!ok) s_fail = 1;
  uint32_t kh[H];
#pragma unroll
  for (int h = 0; h < H; ++h) {
    kh[h] = ord_key(vh[h]);
    if (mh[h] && a.store_sample) {
      const int64_t o = orow + lo + static_cast<int64_t>(h) * LS_THREADS + tid;
      a.sidx[o] = static_cast<uint32_t>(xs[h]);
      a.skeys[o] = kh[h];
    }
  }
  if (chunk == 0 && tid == 0) S.distinct = static_cast<unsigned>(a.S < 0xffffffffll ? a.S : 0xffffffffll);
  auto each_key = [&](auto&& fn) {
#pragma unroll
    for (int h = 0; h < H; ++h) fn(kh[h], mh[h]);
  };
  const unsigned t = static_cast<unsigned>(a.t);
  SampleCand& cd = cands[row];
  uint32_t* mine = cd.key + chunk * static_cast<int64_t>(t);
  // The chunk's t largest keys (all of them, padded with zero keys, when it
  // has fewer than t).
  const int64_t cnt = (a.S - lo < static_cast<int64_t>(LS_THREADS) * H) ? a.S - lo : static_cast<int64_t>(LS_THREADS) * H;
  if (cnt < static_cast<int64_t>(t)) {
#pragma unroll
    for (int h = 0; h < H; ++h)
      if (mh[h]) mine[atomicAdd(&s_pos, 1u)] = kh[h];
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      for (unsigned q = static_cast<unsigned>(cnt); q < t; ++q) mine[q] = 0u;
      cd.kth[chunk] = 0u;
      cd.extra[chunk] = 0u;
    }
  } else {
    unsigned ex;
    const uint32_t K = block_list_t(each_key, t, sm, mine, &ex);
    if (tid == 0) {
      cd.kth[chunk] = K;
      cd.extra[chunk] = ex;
    }
  }
  // Publication: the chunk's flag, (epoch << 1) | (a walk did not end),
  // stored with release semantics once its list is written (by warp 0, or by
  // every thread before the block barrier above).  Then every CTA reads the
  // row's flags; one that finds them all of this launch finishes the row.
  // The fences between each CTA's flag store and its reads make sure that
  // the last CTA to publish finds every flag; two CTAs that both do finish
  // the row compute the same tau and write the same words.
  if (warp == 0) {
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      const unsigned long long f = (epoch << 1) | (s_fail ? 1ull : 0ull);
      asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(&cd.flag[chunk]), "l"(f) : "memory");
      __threadfence();
    }
  }
  __syncthreads();
  __threadfence();
  bool mine_ok = true;
  for (int64_t ch = tid; ch < G; ch += LS_THREADS) {
    unsigned long long f;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(f) : "l"(&cd.flag[ch]) : "memory");
    if ((f >> 1) != epoch) mine_ok = false;
    else if (f & 1ull) s_fail = 1;
  }
  if (!__syncthreads_and(mine_ok)) return;
  // A CTA that finishes the row: tau among the G t candidates.  The copies
  // of tau in the sample are those among the candidates plus those left out
  // by the chunks whose t-th largest is tau.
  const int total = static_cast<int>(G) * static_cast<int>(t);
  for (int e = tid; e < total; e += LS_THREADS) s_cand[e] = __ldcg(cd.key + e);
  __syncthreads();
  // Warp w takes candidates w, w + LS_WARPS, ... (at most MAX_CHUNKS TAU_CAND / LS_THREADS a lane).
  auto each_cand = [&](auto&& fn) {
#pragma unroll
    for (int q = 0; q < MAX_CHUNKS * TAU_CAND / LS_THREADS; ++q) {
      const int e = (q * 32 + lane) * LS_WARPS + warp;
      const bool v = e < total;
      fn(v ? s_cand[e] : 0u, v);
    }
  };
  unsigned cex;
  const uint32_t tau = block_list_t(each_cand, t, sm, s_final, &cex);
  if (warp != 0) return;
  unsigned more = 0;
  for (int64_t ch = lane; ch < G; ch += 32)
    if (__ldcg(&cd.kth[ch]) == tau) more += __ldcg(&cd.extra[ch]);
  more = __reduce_add_sync(FULL_MASK, more);
  __syncwarp();  // s_final, written by the warp's lanes
  if (lane == 0) {
    if (s_fail) atomicOr(&S.error, 1u);
    // t listed keys are at or above tau; those equal to it, plus the copies
    // left out of the candidates and out of the chunks' lists.
    unsigned eq_listed = 0;
    for (unsigned q = 0; q < t; ++q) eq_listed += s_final[q] == tau;
    const unsigned long long copies = static_cast<unsigned long long>(eq_listed) + cex + more;
    S.tau_key = tau;
    S.tau_copies = static_cast<unsigned>(copies < 0xffffffffull ? copies : 0xffffffffull);
    S.sel_prefix = tau;
    S.sel_bits = 32;
    S.sel_done = 1;
  }
}

// Chunks per row: all CTAs (chunks x rows) resident at once, one per SM, at
// most MAX_CHUNKS, at least ST_THREADS sample positions per chunk.
int64_t sample_tau_chunks(int64_t S, int nrows) {
  int64_t G = sms() / (nrows > 0 ? nrows : 1);
  const int64_t by_len = (S + ST_THREADS - 1) / ST_THREADS;
  if (G > by_len) G = by_len;
  if (G > MAX_CHUNKS) G = MAX_CHUNKS;
  return G < 1 ? 1 : G;
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// Epochs of the candidate lists' flags: a nonce drawn once per process (the
// clock and the process id, mixed) in the high 31 bits, a launch counter in
// the low 32.  Never 0.
unsigned long long next_epoch() {
  static const unsigned long long nonce = [] {
    unsigned long long z = static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count()) ^
                           (static_cast<unsigned long long>(getpid()) << 40);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return (z ^ (z >> 31)) & 0x7FFFFFFFull;
  }();
  static std::atomic<unsigned long long> count{0};
  return (nonce << 32) | ((count.fetch_add(1) + 1) & 0xFFFFFFFFull);
}

}  // namespace

int64_t sample_tau_setup_max_t() { return TAU_CAND; }

void launch_sample_rows(const SampleArgs& a, int64_t key_row0, cudaStream_t stream) {
  const int64_t blocks = (a.S + DRAW_THREADS - 1) / DRAW_THREADS;
  launch_kernel(k_sample_draw, dim3(static_cast<unsigned>(blocks), a.nrows), DRAW_THREADS, 0, stream, a, key_row0);
}

void launch_sample(const SampleArgs& a, cudaStream_t stream) { launch_sample_rows(a, 0, stream); }

size_t sample_tau_ctl_bytes() { return sizeof(SampleCtl); }

size_t sample_tau_scratch_bytes(int64_t rows) {
  return align256(sizeof(SampleCtl) * rows) + sizeof(SampleCand) * rows;
}

bool sample_tau_fits(int64_t S, int nrows) {
  const int64_t G = sample_tau_chunks(S, nrows);
  const int64_t Cn = (((S + G - 1) / G) + 31) & ~int64_t(31);
  return Cn <= static_cast<int64_t>(ST_HELD) * ST_THREADS;
}

cudaError_t launch_sample_tau(const SampleArgs& a, void* scratch, int64_t total_rows, cudaStream_t stream) {
  if (!sample_tau_fits(a.S, a.nrows)) return cudaErrorInvalidValue;
  const int64_t G = sample_tau_chunks(a.S, a.nrows);
  SampleCtl* ctl = static_cast<SampleCtl*>(scratch);
  SampleCand* cand =
      reinterpret_cast<SampleCand*>(static_cast<char*>(scratch) + align256(sizeof(SampleCtl) * total_rows));
  const dim3 grid(static_cast<unsigned>(G), static_cast<unsigned>(a.nrows));
  if (a.t <= static_cast<unsigned long long>(TAU_CAND)) {
    const size_t smem = sizeof(uint32_t) * static_cast<size_t>(G) * a.t;  // at most 8 KB
    launch_kernel(k_sample_tau<true>, grid, ST_THREADS, smem, stream, a, ctl, cand, next_epoch());
  } else {
    launch_kernel(k_sample_tau<false>, grid, ST_THREADS, 0, stream, a, ctl, cand, 0ull);
  }
  return cudaGetLastError();
}

bool sample_lists_fits(int64_t S, unsigned long long t) {
  return t >= 1 && t <= static_cast<unsigned long long>(TAU_CAND) &&
         (S + LS_THREADS * LS_MAX_H - 1) / (LS_THREADS * LS_MAX_H) <= MAX_CHUNKS;
}

cudaError_t launch_sample_lists(const SampleArgs& a, void* scratch, int64_t total_rows, cudaStream_t stream) {
  if (!sample_lists_fits(a.S, a.t)) return cudaErrorInvalidValue;
  SampleCand* cand =
      reinterpret_cast<SampleCand*>(static_cast<char*>(scratch) + align256(sizeof(SampleCtl) * total_rows));
  // Positions per thread: the fewest that keep the launch within about four
  // CTAs per SM (one wave), at most LS_MAX_H, and within MAX_CHUNKS chunks.
  const int64_t wave = 4 * static_cast<int64_t>(sms());
  int h = 1;
  auto chunks = [&](int hh) { return (a.S + LS_THREADS * hh - 1) / (LS_THREADS * hh); };
  while (h < LS_MAX_H && (chunks(h) > MAX_CHUNKS || chunks(h) * a.nrows > wave)) h *= 2;
  const dim3 grid(static_cast<unsigned>(chunks(h)), static_cast<unsigned>(a.nrows));
  const unsigned long long ep = next_epoch();
  switch (h) {
    case 1: launch_kernel(k_sample_lists<1>, grid, LS_THREADS, 0, stream, a, cand, ep); break;
    case 2: launch_kernel(k_sample_lists<2>, grid, LS_THREADS, 0, stream, a, cand, ep); break;
    case 4: launch_kernel(k_sample_lists<4>, grid, LS_THREADS, 0, stream, a, cand, ep); break;
    default: launch_kernel(k_sample_lists<8>, grid, LS_THREADS, 0, stream, a, cand, ep); break;
  }
  return cudaGetLastError();
}

}  // namespace profk
