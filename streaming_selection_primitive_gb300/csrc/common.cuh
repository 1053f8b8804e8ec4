// Shared device definitions of the Prof-K library (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace profk {

constexpr unsigned FULL_MASK = 0xffffffffu;
constexpr int HIST_BITS = 11;
constexpr int HIST_BINS = 1 << HIST_BITS;  // 2048-bin radix histograms

// ---------------------------------------------------------------------------
// Order keys.  ord(v) maps a float to a uint32 whose unsigned order is the
// IEEE order of the values, with -0.0 folded onto +0.0 so that they compare
// equal.  A candidate (v, i) is the 64-bit key (ord(v) << 32) | ~i: larger key
// = larger value, and for equal values the lower index.  NaN maps above
// ord(+inf) (positive NaN) or below ord(-inf) (negative NaN).
__host__ __device__ __forceinline__ uint32_t ord_key(float v) {
#ifdef __CUDA_ARCH__
  uint32_t b = __float_as_uint(v);
#else
  uint32_t b;
  __builtin_memcpy(&b, &v, 4);
#endif
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__host__ __device__ __forceinline__ float key_to_float(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
#ifdef __CUDA_ARCH__
  return __uint_as_float(b);
#else
  float v;
  __builtin_memcpy(&v, &b, 4);
  return v;
#endif
}

constexpr uint32_t KEY_POS_INF = 0xff800000u;  // ord(+inf)
constexpr uint32_t KEY_NEG_INF = 0x007fffffu;  // ord(-inf)

__host__ __device__ __forceinline__ bool key_is_nan(uint32_t k) {
  return k > KEY_POS_INF || k < KEY_NEG_INF;
}

__device__ __forceinline__ uint64_t cand_key(float v, uint32_t idx) {
  return (static_cast<uint64_t>(ord_key(v)) << 32) | static_cast<uint32_t>(~idx);
}

__device__ __forceinline__ uint32_t cand_index(uint64_t key) {
  return ~static_cast<uint32_t>(key & 0xffffffffull);
}

// ---------------------------------------------------------------------------
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds; each round
// multiplies counter words 0 and 2 by two odd constants (128-bit products)
// and mixes with words 1, 3 and the key; the key is bumped by two Weyl
// constants between rounds.
constexpr uint64_t PHILOX_M0 = 0xD2E7470EE14C6C93ull;
constexpr uint64_t PHILOX_M1 = 0xCA5A826395121157ull;
constexpr uint64_t PHILOX_W0 = 0x9E3779B97F4A7C15ull;
constexpr uint64_t PHILOX_W1 = 0xBB67AE8584CAA73Bull;

__device__ __forceinline__ void philox4x64_10(uint64_t c[4], uint64_t k0, uint64_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    const uint64_t lo0 = PHILOX_M0 * c[0], hi0 = __umul64hi(PHILOX_M0, c[0]);
    const uint64_t lo1 = PHILOX_M1 * c[2], hi1 = __umul64hi(PHILOX_M1, c[2]);
    const uint64_t n0 = hi1 ^ c[1] ^ k0;
    const uint64_t n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// ---------------------------------------------------------------------------
// Per-row device state of one call.  Zeroed by the host before use.
struct RowState {
  // Filter counters of the current attempt.  R_ge is also the slot cursor
  // of the candidate buffer: it counts every passer, stores stop at M.
  unsigned long long R_ge;
  unsigned long long R_gt;
  unsigned long long nan;
  // The first attempt's counts, kept for the statistics when later attempts
  // run before the host reads the row (written by attempt 0's refinement).
  unsigned long long R_first;
  unsigned long long R_gt_first;
  // Sampling.
  unsigned int distinct;  // distinct draws among the D examined
  unsigned int tau_key;   // ord(tau)
  // Radix selection of the r-th largest key (r = 1 is the maximum).
  unsigned long long sel_prefix;  // resolved high bits (right-aligned)
  unsigned long long sel_rank;    // rank still to find inside the prefix bucket
  unsigned long long sel_above;   // keys strictly above the prefix bucket
  unsigned long long sel_bucket;  // population of the last chosen bucket
  unsigned long long sel_thresh;  // final threshold key (valid when sel_done)
  unsigned long long sel_nan;     // NaN keys seen by the first pass (float sources)
  int sel_bits;                   // number of resolved high bits
  int sel_done;                   // 1 once the threshold is known
  unsigned int done_blocks;       // last-block-done ticket
  unsigned int compact_count;     // output cursor of the compaction
  unsigned int error;             // nonzero: a device-side check failed
  unsigned int skip;              // 1: this row's refinement is void (its attempt failed the check)
  unsigned int tie_gt;            // x > tau appended to the tie list by the filter
  unsigned int tau_copies;        // copies of tau among the sample keys (2 or more: a tied top)
  // 1 + the attempt whose check settled the row (it passed, or takes the tie
  // exit, or met a NaN or an error), 0 while it is open.  The kernels of a
  // later attempt leave a settled row alone.
  unsigned int settled;
  unsigned int tau_first;         // ord(tau) of the first attempt
  unsigned int hist[HIST_BINS];
  // OR of ord(x) ^ ord(tau) over the filter's passers: every passer's value
  // key agrees with tau's above the highest set bit (0: all equal tau).
  unsigned int vdiff;
};

// Whether an attempt before `attempt` settled the row: the kernels of this
// attempt then leave it alone.  Every CTA of the row reads the same value
// (only a refinement writes it, and those of earlier attempts have finished),
// so the test is row-uniform.
__device__ __forceinline__ bool settled_before(const RowState& S, int attempt) {
  if (attempt == 0) return false;
  const unsigned s = __ldcg(&S.settled);
  return s != 0u && s <= static_cast<unsigned>(attempt);
}

// The run-time check of `attempt` for the row, taken on the device by its
// refinement (one thread): the row is settled when k <= R <= M, or when the
// tie exit takes it (R > M and R_gt < k, with the tie exit on), or when a
// NaN or an error was counted; otherwise the next attempt redraws it.  The
// host reads the same counts and takes the same decision.  Attempt 0 also
// keeps its counts for the statistics.
__device__ __forceinline__ void settle_row(RowState& S, int attempt, unsigned long long k, unsigned long long M,
                                           bool tie_exit) {
  const unsigned long long R = __ldcg(&S.R_ge), Rt = __ldcg(&S.R_gt);
  const bool pass = k <= R && R <= M;
  const bool tie = tie_exit && R > M && Rt < k;
  if (pass || tie || __ldcg(&S.nan) != 0ull || __ldcg(&S.error) != 0u) S.settled = static_cast<unsigned>(attempt) + 1u;
  if (attempt == 0) {
    S.R_first = R;
    S.R_gt_first = Rt;
    S.tau_first = __ldcg(&S.tau_key);
  }
}

// ---------------------------------------------------------------------------
// Bounded waits of the persistent kernels (grid barriers and look-backs).
// A wait gives up after a bounded number of polls, or as soon as another CTA
// of the same row has given up (the row's abort word, in the kernel's control
// block, zero at launch).  A CTA that gives up sets the abort word, reports
// ERR_WAIT in RowState::error and leaves the kernel without writing any more
// data; the kernels after it skip a row whose error word is set, so the
// host sees PROFK_ERR_DEVICE_TIMEOUT and the outputs are left alone.
constexpr int WAIT_POLLS = 1 << 22;   // default bound on one wait (a poll is an L2 round trip: seconds in all)
constexpr int WAIT_ABORT_EVERY = 32;  // polls between two reads of the abort word
constexpr unsigned ERR_WAIT = 8u;     // RowState::error bit of a wait that gave up

// Test setting of a kernel's waits: `skew` extra arrivals awaited at its
// first grid barrier (which then can never be met) and a shorter bound
// `polls` (0: WAIT_POLLS).  Both zero on every ordinary call.
struct WaitCfg {
  unsigned skew = 0;
  int polls = 0;
};

__device__ __forceinline__ int wait_limit(const WaitCfg& w) { return w.polls > 0 ? w.polls : WAIT_POLLS; }

__device__ __forceinline__ unsigned wait_ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ bool wait_aborted(const unsigned* abort_word) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(abort_word) : "memory");
  return v != 0u;
}

__device__ __forceinline__ void wait_give_up(unsigned* abort_word) { atomicExch(abort_word, 1u); }

// Whether poll number `poll` of a wait should end it: the bound was reached
// (the wait gives up, setting the abort word) or, every WAIT_ABORT_EVERY
// polls, another CTA of the row has given up.
__device__ __forceinline__ bool wait_should_stop(int poll, int limit, unsigned* abort_word) {
  if (poll >= limit) {
    wait_give_up(abort_word);
    return true;
  }
  return poll % WAIT_ABORT_EVERY == WAIT_ABORT_EVERY - 1 && wait_aborted(abort_word);
}

// One thread waits (acquire loads) until *count reaches target.  Returns
// false if the wait ended without it.
__device__ __forceinline__ bool wait_count(const unsigned* count, unsigned target, unsigned* abort_word, int limit) {
  for (int poll = 0; wait_ld_acquire(count) < target; ++poll)
    if (wait_should_stop(poll, limit, abort_word)) return false;
  return true;
}

// Row of a launch: identity unless a row list is given.
__device__ __forceinline__ int launch_row(const int* rows) {
  return rows ? rows[blockIdx.y] : static_cast<int>(blockIdx.y);
}

// Histogram increment by a whole warp (all 32 lanes call it).  Lanes with
// nothing to count cost one vote; when every counting lane hits the same bin
// (a heavily tied input) the warp adds once; otherwise each lane adds its own.
__device__ __forceinline__ void hist_add(unsigned int* h, uint32_t bin, bool valid) {
  const unsigned act = __ballot_sync(FULL_MASK, valid);
  if (act == 0) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(act) - 1;
  const uint32_t b0 = __shfl_sync(FULL_MASK, bin, leader);
  if (__all_sync(FULL_MASK, !valid || bin == b0)) {
    if (lane == leader) atomicAdd(h + b0, static_cast<unsigned>(__popc(act)));
  } else if (valid) {
    atomicAdd(h + bin, 1u);
  }
}

}  // namespace profk
