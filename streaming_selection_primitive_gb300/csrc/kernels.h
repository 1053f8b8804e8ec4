// Host-side launchers of the Prof-K kernels (internal interface).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "common.cuh"

namespace profk {

// Kernels launched by the calling host thread since it started (the library's
// own kernels only); profk_stats reports the difference over one call.
inline int64_t& launch_count() {
  thread_local int64_t count = 0;
  return count;
}

// Programmatic dependent launch.  Every kernel of the library starts with
// pdl_wait() (griddepcontrol.wait: returns once the preceding kernel on the
// stream has completed and its memory is visible; a no-op for an ordinary
// launch).  Small kernels call pdl_trigger() first, so that the next kernel
// can be launched while they run.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

bool pdl_enabled();  // PROFK_OPT_PDL

// Launches a library kernel on `stream`, with the programmatic-serialization
// attribute when PDL is enabled, and counts it.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 Args&&... args) {
  ++launch_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Where a radix selection reads its keys from.
enum class KeySource : int {
  SampleKeys = 0,  // uint32 order keys of the sample, value-only selection
  Input = 1,       // float input row, composite (value, index) keys
  Buffer = 2,      // candidate buffer of composite keys, length min(R_ge, M)
};

struct SelectArgs {
  KeySource src;
  const void* base;   // sample keys / input / buffer
  int64_t stride;     // row stride in elements of `base`
  int64_t len;        // elements per row (Buffer: capacity M; length from R_ge)
  int nrows;          // rows in this launch
  const int* rows;    // device row list, or nullptr for rows 0..nrows-1
  RowState* st;       // per-row state (indexed by row)
};

// Sampling (sample.cu): the sample of each listed row is pi(0), ..., pi(S-1)
// for the keyed permutation pi of [0, n) that sample.cu defines (a Feistel
// network with Philox rounds, cycle-walked into [0, n)), key (seed, storage
// row + key_row0) and the attempt number.
struct SampleArgs {
  const float* x;
  int64_t ld;           // row stride of x
  uint64_t n;           // row length, at most 2^32
  int64_t S;            // sample size, 1 <= S <= n
  uint64_t seed;
  int attempt;
  int nrows;
  const int* rows;
  RowState* st;
  uint32_t* sidx;   // rows x S (out): the indices in sample order
  uint32_t* skeys;  // rows x S (out): their order keys
  // Optional: the first 11-bit pass of the tau selection (step 2, rank t)
  // fused into the sampling kernel; the selection state must have been reset
  // (RowState::hist zero, done_blocks 0).  The two remaining passes are
  // launch_select(..., first_pass = 1).
  bool tau_pass1 = false;
  unsigned long long t = 0;
  int64_t key_row0 = 0;
  WaitCfg wait{};  // launch_sample_tau: test setting of its waits
  // launch_sample_tau for t <= sample_tau_setup_max_t(): the attempt's set-up
  // done by the sampler itself, in place of a reset kernel: the row state
  // (counters, error word, selection state, histogram), the refinement's
  // control block (zero_words 8-byte words per row, an even number) and
  // the tie step's block counts (zero_nb per row) are zeroed.
  unsigned long long* zero_ctl = nullptr;
  int zero_words = 0;
  unsigned* zero_eq = nullptr;
  int64_t zero_nb = 0;
  // Whether the persistent and the lists forms store sidx and skeys (the
  // step-by-step form always does: its tau selection reads skeys); the main
  // path needs neither.
  bool store_sample = true;
};
// One thread per sample position: indices, keys and RowState::distinct (= S).
void launch_sample(const SampleArgs& a, cudaStream_t stream);
// Same, with Philox key word 1 = storage row + key_row0 (a single stored row
// can then reproduce any row's sample).
void launch_sample_rows(const SampleArgs& a, int64_t key_row0, cudaStream_t stream);
// Steps 1 and 2 of the main path in one persistent kernel: the sample
// (RowState::distinct; sidx and skeys when store_sample) and tau
// (RowState::tau_key, tau_copies; rank a.t) of each listed row.  `scratch` holds sample_tau_scratch_bytes(
// total_rows): first the per-row control blocks (sample_tau_ctl_bytes()
// each, indexed by row, zero at launch), then candidate lists that need no
// initialisation.  Rows that an attempt before a.attempt settled
// (settled_before) are left alone.
size_t sample_tau_ctl_bytes();
size_t sample_tau_scratch_bytes(int64_t rows);
cudaError_t launch_sample_tau(const SampleArgs& a, void* scratch, int64_t total_rows, cudaStream_t stream);
// Whether launch_sample_tau takes these rows: each CTA's chunk of the sample
// (S split over the row's share of the SMs) held in registers, at most 1024
// positions; otherwise the step-by-step kernels (launch_sample with
// tau_pass1, then launch_select).
bool sample_tau_fits(int64_t S, int nrows);
// Largest t for which launch_sample_tau also does the attempt's set-up (and
// needs no zeroed control block of its own).
int64_t sample_tau_setup_max_t();
// The lists form of steps 1 and 2, for t <= sample_tau_setup_max_t() and any
// number of rows: CTAs of 256 threads take up to 2048 consecutive sample
// positions of one row each and publish lists of their t largest keys; a CTA
// that finds every list of its row published selects tau among them.  No
// CTA waits for another, so the launch needs no co-residency.  It does the
// attempt's set-up like the persistent form (SampleArgs::zero_ctl) and uses
// the same scratch (sample_tau_scratch_bytes), whose lists need no
// initialisation.  Rows that an earlier attempt settled are left alone.
bool sample_lists_fits(int64_t S, unsigned long long t);
cudaError_t launch_sample_lists(const SampleArgs& a, void* scratch, int64_t total_rows, cudaStream_t stream);

// Exact top-k of short rows, one CTA per row (rows.cu): outputs of each listed
// row (or rows 0 .. nrows-1) sorted, RowState::sel_nan set to the row's NaN
// count.  Needs k <= rows_exact_max_k(), n < 2^32 and 16-byte aligned rows.
struct RowsExactArgs {
  const float* x;
  int64_t ld;
  int64_t n;
  int64_t k;
  int nrows;
  const int* rows;
  RowState* st;
  float* out_vals;
  int64_t* out_idx;
};
int64_t rows_exact_max_k();
// Whether the one-CTA-per-row selection is expected to beat the multi-CTA one.
bool rows_exact_suits(int64_t nrows, int64_t n, int64_t k);
void launch_rows_exact(const RowsExactArgs& a, cudaStream_t stream);

// Radix selection of the rank-th largest key per row.  init_rank > 0 resets the
// state of each row first; otherwise the state is taken as it is (tie path).
void launch_select(const SelectArgs& a, uint64_t init_rank, bool value_only, int first_pass,
                   cudaStream_t stream);
// Resolved value key of the tau selection into RowState::tau_key.
void launch_store_tau(int nrows, const int* rows, RowState* st, cudaStream_t stream);
// Tie path: set the state to "value ord(tau) resolved, rank k - R_gt left".
void launch_tie_init(int nrows, const int* rows, RowState* st, int64_t k, cudaStream_t stream);

// Tie exit (tie.cu): the k outputs of each listed row (R > M, R_gt < k) into
// `sel` (every x > tau, then the k - R_gt lowest-index copies of tau), ready
// for launch_sort_emit; also clears RowState::skip of those rows.
struct TieCtl;
// Counting blocks of the tie step: 2^TIE_BLOCK_LOG2 elements (one segment of
// the take, so that the blocks up to the cut are taken in parallel).
constexpr int TIE_BLOCK_LOG2 = 14;

struct TieArgs {
  const float* x;
  int64_t ld;
  int64_t n;
  int nrows;
  const int* rows;
  RowState* st;
  unsigned long long* sel;  // rows x kstride output keys
  int64_t kstride;
  int64_t k;
  unsigned* block_eq;             // rows x nblocks: copies of tau per block of 2^TIE_BLOCK_LOG2 elements
  unsigned long long* block_pre;  // rows x nblocks: their exclusive prefix
  int64_t nblocks;                // tie_blocks(n)
  TieCtl* ctl;                    // rows x tie_ctl_bytes()
  int64_t total_rows;             // rows the arrays are sized for
};
int64_t tie_blocks(int64_t n);
size_t tie_ctl_bytes();
// The tie step after a selection of tau = v_k that left RowState::R_gt = the
// count of x > v_k (the exact path): one counting pass over the rows, then
// the cut and the take.
cudaError_t launch_tie_take(const TieArgs& a, int filter_grid, cudaStream_t stream);
// The tie exit after a filter pass run with its tie bookkeeping (block_eq
// and the appended x > tau already filled): the buffer's x > tau join the
// appended ones, then the cut and the take.  buf: the filter's buffer, M its
// capacity per row.
cudaError_t launch_tie_after_filter(const TieArgs& a, const unsigned long long* buf, int64_t M,
                                    cudaStream_t stream);

// Writes the k keys >= the selected threshold into out (row stride out_stride).
void launch_compact(const SelectArgs& a, uint64_t* out, int64_t out_stride, int64_t k,
                    cudaStream_t stream);

// Sorts each row's k keys descending (in place in `keys`, row stride
// key_stride >= next_pow2(k)) and writes values (read from x) and indices.
// Rows whose state says skip are left untouched when st is given.  For
// k > 8192 the keys are radix-sorted when `scratch` (radix_sort_scratch_bytes
// of key_stride for all `total_rows` rows of the call) is given, else
// bitonic-sorted in place (key_stride must then be next_pow2(k)).
// gt_first (with st, k <= 8192): each row's keys [R_gt, k) are copies of one
// value in ascending index order, below the keys [0, R_gt) (the tie step's
// layout), and only the latter are sorted.
void launch_sort_emit(uint64_t* keys, int64_t key_stride, int64_t k, int nrows, const int* rows,
                      const float* x, int64_t ld, int64_t n, float* out_vals, int64_t* out_idx,
                      cudaStream_t stream, RowState* st = nullptr, void* scratch = nullptr,
                      int64_t total_rows = 0, bool gt_first = false);
// Large-row sort and emission (sort.cu).  Which keys a row sorts:
enum class SortCount {
  All,          // k keys, every listed row
  KUnlessSkip,  // k keys, rows whose RowState::skip is clear
  FromState,    // RowState::R_ge keys, rows with k <= R_ge <= key_stride
};
struct RadixSortArgs {
  unsigned long long* keys;  // rows x key_stride; permuted in place
  int64_t key_stride;        // also the most keys a row may hold
  int64_t k;                 // outputs per row: the k largest, descending
  SortCount mode;
  int nrows;
  const int* rows;     // row list, or nullptr for 0..nrows-1
  int64_t total_rows;  // rows the scratch is sized for (rows are indexed by number)
  void* scratch;       // radix_sort_scratch_bytes(key_stride, total_rows)
  bool ctl_zeroed;     // the control block (radix_sort_ctl) is already zero
  const float* x;
  int64_t ld;
  int64_t n;
  float* out_vals;
  int64_t* out_idx;
  RowState* st;  // skip / count source, and where a timed-out wait is reported
  WaitCfg wait{};  // test setting of its waits
  // FromState: the attempt this refinement belongs to (rows settled by an
  // earlier one are left alone; see settle_row) and whether the call's tie
  // exit is on.
  int attempt = 0;
  bool tie_exit = false;
};
size_t radix_sort_scratch_bytes(int64_t key_stride, int64_t rows);
void* radix_sort_ctl(void* scratch, int64_t key_stride, int64_t rows);  // per-row control blocks
size_t radix_sort_ctl_bytes();                                          // one row's control block
cudaError_t launch_radix_sort(const RadixSortArgs& a, cudaStream_t stream);
int sms();  // SMs of the current device
int64_t small_sort_max();
int64_t sort_stride(int64_t k);  // key_stride the sort needs for k keys

// Step 4 in one CTA per row for k <= refine_one_max_k() (select.cu): radix
// selection over the candidate keys read from L2, early gather of the top
// bucket, shared-memory sort and emission.  A row whose count fails
// k <= R <= M is marked skip and left alone.
struct RefineOneArgs {
  const unsigned long long* buf;  // rows x M candidate keys
  int64_t M;
  int nrows;
  const int* rows;
  RowState* st;
  int64_t k;
  const float* x;
  int64_t ld;
  int64_t n;
  float* out_vals;
  int64_t* out_idx;
  WaitCfg wait{};  // launch_refine_grid: test setting of its waits
  // launch_refine_grid: the attempt this refinement belongs to (rows settled
  // by an earlier one are left alone; see settle_row) and whether the call's
  // tie exit is on.
  int attempt = 0;
  bool tie_exit = false;
  // launch_refine_grid: the bits of the filter's RowState::vdiff it trusts
  // (all but in the test of its prefix check).
  uint32_t vdiff_keep = 0xFFFFFFFFu;
};
void launch_refine_one(const RefineOneArgs& a, cudaStream_t stream);
int64_t refine_one_max_k();
int64_t refine_one_max_m();

// Step 4 on the filter path for k <= refine_grid_max_k() and M <=
// refine_grid_max_m() (refine.cu): the same result as launch_refine_one, by
// one CTA per SM with grid barriers.  `scratch` holds
// refine_grid_scratch_bytes(total_rows); its control blocks (refine_grid_ctl,
// refine_grid_ctl_bytes each, indexed by row) must be zero at launch.
using RefineGridArgs = RefineOneArgs;
size_t refine_grid_scratch_bytes(int64_t rows);
void* refine_grid_ctl(void* scratch);
size_t refine_grid_ctl_bytes();
int64_t refine_grid_max_k();
int64_t refine_grid_max_m();
cudaError_t launch_refine_grid(const RefineGridArgs& a, void* scratch, int64_t total_rows, cudaStream_t stream);

// Filter pass.
struct FilterArgs {
  const float* x;
  int64_t ld;
  int64_t n;
  int64_t M;
  int nrows;
  const int* rows;
  RowState* st;
  unsigned long long* buf;  // rows x M
  int grid;                 // persistent CTAs
  // Bookkeeping for the tie exit (off when block_eq is null): the copies of
  // tau per block of 2^TIE_BLOCK_LOG2 elements (rows x nblocks, zero at
  // launch), and every x > tau that the full buffer drops, appended to the
  // row's tie list (row stride tie_stride) from RowState::tie_gt on (stores
  // beyond k are dropped; the count goes on).  The x > tau of the buffer and
  // those appended are then all of them.
  unsigned* block_eq = nullptr;
  int64_t nblocks = 0;
  unsigned long long* tie_keys = nullptr;
  int64_t tie_stride = 0;
  int64_t k = 0;
  int attempt = 0;  // rows settled by an earlier attempt are left alone (settled_before)
  // Set by launch_filter: the CTAs that warm L2 with the first tiles of every
  // warp before tau is known, and how many tiles per warp.
  int pf_ctas = 0;
  int pf_tiles = 0;
};
// The filter pass over the listed rows.  x must be 4-byte aligned.  When some
// row does not start on a 16-byte boundary (x 4-byte aligned only, or a row
// stride that is not a multiple of 4), a kernel instantiation of its own
// starts each row's warp tiles at the boundary at or before the row, and the
// row's first and last tiles take the masked path (element loads of the
// row's own elements only); the tie bookkeeping, which counts per aligned
// block, is then dropped.
void launch_filter(const FilterArgs& a, cudaStream_t stream);
int filter_default_grid(int sms);

// Merge of the per-segment top-k lists of a row split into segments
// (segments.cu).  List s (s < lists - 1) holds list_len entries at
// vals/idx + s * list_len, the last list last_len <= list_len entries after
// them; each is sorted in the library order with indices relative to its
// segment, which starts at s * seg_len in the row.  Writes the row's top k.
struct MergeSegmentsArgs {
  const float* vals;
  const int64_t* idx;
  int lists;
  int64_t list_len, last_len, seg_len, k;
  float* out_vals;
  int64_t* out_idx;
};
void launch_merge_segments(const MergeSegmentsArgs& a, cudaStream_t stream);

}  // namespace profk
