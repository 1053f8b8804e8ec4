// Host-side launchers of the Prof-K kernels (internal interface).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace profk {

// Kernels launched by the calling host thread since it started (the library's
// own kernels only); profk_stats reports the difference over one call.
inline int64_t& launch_count() {
  thread_local int64_t count = 0;
  return count;
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

// Sampling: draws, first-occurrence marking and ordered compaction.
struct SampleArgs {
  const float* x;
  int64_t ld;           // row stride of x
  uint64_t n;           // row length
  int64_t S;
  int64_t D;            // draws examined (multiple of 4)
  int log2H;            // hash table of 2^log2H slots per row
  uint64_t seed;
  int attempt;
  int nrows;
  const int* rows;
  RowState* st;
  unsigned long long* table;  // rows x 2^log2H, filled with ~0 by the host
  uint32_t* draws;            // rows x D
  uint32_t* blockcnt;         // rows x ceil(D / 1024)
  uint32_t* sidx;             // rows x S (out)
  uint32_t* skeys;            // rows x S (out)
};
void launch_sample(const SampleArgs& a, cudaStream_t stream);
// Same, with Philox key word 1 = storage row + key_row0 (a single stored row
// can then reproduce any row's stream).
void launch_sample_rows(const SampleArgs& a, int64_t key_row0, cudaStream_t stream);

// Radix selection of the rank-th largest key per row.  init_rank > 0 resets the
// state of each row first; otherwise the state is taken as it is (tie path).
void launch_select(const SelectArgs& a, uint64_t init_rank, bool value_only, int first_pass,
                   cudaStream_t stream);
// Resolved value key of the tau selection into RowState::tau_key.
void launch_store_tau(int nrows, const int* rows, RowState* st, cudaStream_t stream);
// Refinement set-up straight after the filter: rows whose count fails
// k <= R <= M are marked void on the device (their refinement writes nothing).
void launch_refine_init(int nrows, const int* rows, RowState* st, int64_t k, int64_t M, cudaStream_t stream);
// Tie path: set the state to "value ord(tau) resolved, rank k - R_gt left".
void launch_tie_init(int nrows, const int* rows, RowState* st, int64_t k, cudaStream_t stream);

// Writes the k keys >= the selected threshold into out (row stride out_stride).
void launch_compact(const SelectArgs& a, uint64_t* out, int64_t out_stride, int64_t k,
                    cudaStream_t stream);

// Sorts each row's k keys descending (in place in `keys`, row stride
// key_stride >= next_pow2(k)) and writes values (read from x) and indices.
// Rows whose state says skip are left untouched when st is given.
void launch_sort_emit(uint64_t* keys, int64_t key_stride, int64_t k, int nrows, const int* rows,
                      const float* x, int64_t ld, int64_t n, float* out_vals, int64_t* out_idx,
                      cudaStream_t stream, const RowState* st = nullptr);
int64_t sort_stride(int64_t k);  // key_stride the sort needs for k keys

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
};
void launch_filter(const FilterArgs& a, cudaStream_t stream);
int filter_default_grid(int sms);

}  // namespace profk
