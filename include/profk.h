/*
 * profk.h -- Prof-K exact top-k selection for NVIDIA GB300 (sm_103a).
 *
 * Prof-K ("Prof-K: Probabilistic One-Pass Filtering for Efficient Top-k
 * Selection") returns the k largest entries of a vector with their indices.
 * It draws a uniform sample of S indices without replacement, takes the t-th
 * largest sampled value as a threshold tau, streams the input once keeping
 * every x_i >= tau in a buffer of capacity M while counting them exactly (R),
 * and selects the exact top-k from the buffer.  When the run-time check
 * k <= R <= M fails it redraws, and after a fixed number of attempts it runs
 * an exact selection over the whole input, so the result is always exact
 * (paper, Section 3 "The Prof-K Algorithm" and Section 4 "Failure Modes").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Order.  Values descending under IEEE-754 comparison (-0.0 == +0.0, +-inf
 *   are ordinary values); equal values by ascending index.  The pages assume
 *   distinct values (Section 4 "Notation and Conventions"); this tie rule is
 *   the library's reading.  Returned values keep their original bits.
 * NaN.  An input containing NaN is rejected with PROFK_ERR_NAN; the output
 *   buffers are then unspecified.
 * Pointers.  x, out_vals, out_idx and every array documented as "device" are
 *   device pointers owned by the caller; x is only read.  stats is a host
 *   pointer and may be NULL.
 * Indices.  int64, relative to the row (0 .. n-1).  n < 2^40.
 * Streams.  All device work is ordered on `stream` (0 = legacy default).
 *   profk_topk / profk_topk_batched synchronize `stream` once per filter
 *   attempt to read the exact count R (the pages' run-time check); outputs
 *   are complete once `stream` is synchronized after the call returns, and
 *   *stats is complete when the call returns.
 * Workspace.  The library allocates its workspace stream-ordered from a
 *   memory pool it owns (cudaMallocAsync) and returns it before the call
 *   returns; its size is O(M + S) per row, never O(n) (stats->aux_bytes).
 * Errors.  Every entry point returns PROFK_OK (0) or a negative
 *   profk_status; no exception crosses the ABI and there is no CPU fallback.
 * Threads.  Calls from several host threads are safe; profk_set_option
 *   changes process-wide settings and should not race with running calls.
 */
#ifndef PROFK_H_
#define PROFK_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum profk_status {
  PROFK_OK = 0,
  PROFK_ERR_INVALID = -1,        /* an argument is out of range or NULL */
  PROFK_ERR_CUDA = -2,           /* a CUDA call failed (stats->cuda_error has the code), or a
                                    device-side consistency check of the library's own state failed
                                    (cuda_error 0; never expected) */
  PROFK_ERR_NAN = -3,            /* the input holds a NaN */
  PROFK_ERR_UNSUPPORTED = -4,    /* e.g. n >= 2^40, or x not 4-byte aligned */
  PROFK_ERR_DEVICE_TIMEOUT = -5, /* a bounded device-side wait gave up */
  PROFK_ERR_SCRATCH = -6         /* the problem needs more than the fixed scratch or the caller's workspace */
} profk_status;

/* How a row's result was produced. */
typedef enum profk_path {
  PROFK_PATH_FILTER = 0,    /* sample -> threshold -> filter -> refine (k <= R <= M) */
  PROFK_PATH_TIE = 1,       /* R > M but R_gt < k: tau is the k-th largest value; the
                               library emits x > tau plus the lowest-index copies of tau */
  PROFK_PATH_FALLBACK = 2,  /* every attempt failed: exact selection over the row */
  PROFK_PATH_EXACT = 3      /* no sampling (S > n/8, or t = S or M = n: k too close
                               to n for the budget): exact selection */
} profk_path;

/* Per-row report.  Counts of attempts that did not run are -1. */
typedef struct profk_stats {
  int64_t S, t, M;           /* sample size, threshold rank, buffer capacity */
  int64_t R_first;           /* |{x >= tau}| of the first attempt */
  int64_t R_gt_first;        /* |{x >  tau}| of the first attempt */
  int64_t R_final;           /* the same counts for the last attempt */
  int64_t R_gt_final;
  float tau_first;           /* threshold of the first attempt */
  float tau_final;
  int32_t attempts;          /* filter passes run for this row (0 on the exact path) */
  int32_t path;              /* a profk_path */
  int32_t draw_doublings;    /* always 0: the sample has no repeats to redraw (see profk_sample) */
  int32_t cuda_error;        /* cudaError_t of the failing call, else 0 */
  uint64_t aux_bytes;        /* device workspace of the whole call, bytes */
  float filter_ms;           /* device time of the first filter pass over all rows when
                                PROFK_OPT_TIMING is on, else -1 */
  int32_t launches;          /* kernels the whole call launched (all rows) */
} profk_stats;

/* ---- the method -------------------------------------------------------- */

/* Exact top-k of one row x[0..n) (problem statement: paper Section 3).
 *   x         device, n floats, 4-byte aligned (else PROFK_ERR_UNSUPPORTED).
 *             The filter reads 16-byte blocks; a row that does not start on
 *             a 16-byte boundary (a tensor slice such as x + 1) takes its
 *             first and last elements with element loads, and its tie exit
 *             (if any) by radix selection over the row instead of the
 *             vectorised tie step.  The result is the same.
 *   n         1 <= n < 2^40.  A row longer than 2^32 elements (the paper's
 *             Table 4 goes to 4.3e9) is split into P = ceil(n / 2^32)
 *             contiguous segments of equal length rounded up to a multiple
 *             of 4, the last one possibly shorter; each segment's exact
 *             top-min(k, length) is selected as a row of the batched call
 *             with the budget eps / P, and the P sorted lists are merged by
 *             value and global index.  The result is the row's exact top-k;
 *             the call then runs synchronously, and its stats describe the
 *             segments together: S, t, M and tau of the first segment, the
 *             counts R summed over segments (-1 if any is -1), attempts and
 *             path the largest over segments, aux_bytes the workspace of the
 *             largest segment call plus the merge's 12 bytes per candidate.
 *             PROFK_OPT_MAX_SEGMENT lowers the 2^32 split point (for tests).
 *   k         1 <= k <= n
 *   eps       failure budget of one attempt, 0 < eps < 1, split eps/2 + eps/2
 *             between recall failure and overflow (Theorem 4's default split)
 *   seed      seeds every sample; the same (x, k, eps, seed) reproduces the
 *             same samples, counts and stats
 *   out_vals  device, k floats, sorted in the library order
 *   out_idx   device, k int64 indices into x
 */
int profk_topk(const float* x, int64_t n, int64_t k, double eps, uint64_t seed,
               float* out_vals, int64_t* out_idx, cudaStream_t stream,
               profk_stats* stats);

/* Exact top-k of each of `rows` rows; row r is x[r*ld .. r*ld + n).  The
 * paper applies the procedure to each batch element (Section 3) with a
 * per-row threshold, buffer and counter (Appendix C "The Filter Kernel").
 * Each row gets the budget eps / rows, so one attempt of the whole call fails
 * with probability <= eps (union bound, Appendix E.2).  Rows that fail the
 * check are redrawn alone.
 *   ld        row stride in elements, ld >= n (any value: rows off the
 *             16-byte grid are handled as profk_topk describes)
 *   out_vals  device, rows*k floats, row-major (row r at r*k)
 *   out_idx   device, rows*k int64, row-relative indices
 *   stats     host array of `rows` entries, or NULL
 */
int profk_topk_batched(const float* x, int64_t rows, int64_t n, int64_t ld, int64_t k,
                       double eps, uint64_t seed, float* out_vals, int64_t* out_idx,
                       cudaStream_t stream, profk_stats* stats);

/* Asynchronous form of profk_topk / profk_topk_batched.  The call enqueues
 * the first attempt (sampling, filter, the refinement and a kernel that
 * writes the run-time check's counts into pinned host memory) on `stream`
 * and returns at once with *call set; profk_wait(call, stats) then completes
 * it: it waits for those counts (not for the stream), and if every row
 * passed the check the outputs are final and stream-ordered; otherwise (a
 * redraw, the tie exit, the fallback, a NaN) it continues synchronously from
 * that first attempt, in the call's workspace, with the same result and
 * statistics as profk_topk.  Calls
 * with non-default options (forced parameters, timing, no attempts), those
 * routed to the exact path, and those made while a caller workspace is set
 * run synchronously at submission instead.  Each call owns its workspace, so
 * several may be in flight; every call must be passed to profk_wait exactly
 * once, which also frees it.  Submission returns PROFK_ERR_INVALID /
 * PROFK_ERR_UNSUPPORTED as profk_topk does (with *call NULL) and PROFK_OK
 * otherwise; the call's own status is profk_wait's return value. */
typedef struct profk_call profk_call;
int profk_topk_async(const float* x, int64_t n, int64_t k, double eps, uint64_t seed,
                     float* out_vals, int64_t* out_idx, cudaStream_t stream, profk_call** call);
int profk_topk_batched_async(const float* x, int64_t rows, int64_t n, int64_t ld, int64_t k,
                             double eps, uint64_t seed, float* out_vals, int64_t* out_idx,
                             cudaStream_t stream, profk_call** call);
int profk_wait(profk_call* call, profk_stats* stats /* array[rows] or NULL */);

/* Parameters (S, t, M) for one row of length n at budget eps.
 *   mode PROFK_PARAMS_DEFAULT: S from the older version's Theorem 5,
 *     S* = (z log2(k) / 2)^(2/3) (k(n-k))^(1/3) with z = 2 Phi^{-1}(1-eps/2),
 *     rounded and clamped to [32768, 131072] (its Algorithm 1, the sample-size step);
 *     t and M from the corrected Algorithm 1 (Eq 10 or 11, then Eq 12) with
 *     z = Phi^{-1}(1-eps/2); then 1 <= t <= S and k <= M <= n.
 *   mode PROFK_PARAMS_OLD: the older Algorithm 1 literally (Eq 6 t,
 *     Corollary 4 M, and t = 1 when (k/n) S < -ln(eps/2)).
 *   mode PROFK_PARAMS_EXACT: S as in the default mode; t and M the exact
 *     optimum of Theorem 4 (corrected version) for that S, with the budget
 *     split eps/2 + eps/2: t - 1 is the (1 - eps/2)-quantile of the
 *     hypergeometric count of the top k - 1 in the sample, M the smallest M
 *     with Pr(at most t - 1 of the top M are sampled) <= eps/2.
 *   mode PROFK_PARAMS_CORRECTED: the corrected Algorithm 1 throughout: S
 *     from its sample-size steps (Proposition 7, Appendix E.1),
 *     S = clip(floor(max(S1, S2)), 2^14, 2^18) with
 *     S1 = (z/r)^(2/3) (k n)^(1/3), S2 = ((z^2 + 1/2) n / r)^(1/2),
 *     z = Phi^{-1}(1-eps/2); S = 2^14 when r is infinite or k/n > 2^-10;
 *     then S <= n/128.  The cost ratio r(k) has the paper's form
 *     1/r = a log2(k) + b for k > 2^7 (infinite below), with a = 0.0033 and
 *     b = 0.41 fitted on a GB300 by the paper's procedure
 *     (streaming_selection_primitive_gb300/calibrate.py).  t and M as in
 *     the default mode.
 * Pure host arithmetic (fp64), no device work. */
#define PROFK_PARAMS_DEFAULT 0
#define PROFK_PARAMS_OLD 1
#define PROFK_PARAMS_EXACT 2
#define PROFK_PARAMS_CORRECTED 3
int profk_params(int64_t n, int64_t k, double eps, int mode,
                 int64_t* S, int64_t* t, int64_t* M);

/* Device bytes one call of profk_topk_batched(rows, n, k, eps) allocates at
 * most (profk_topk is rows = 1).  0 on invalid arguments. */
size_t profk_workspace_size(int64_t rows, int64_t n, int64_t k, double eps);

/* Caller-owned workspace for this host thread's later profk_topk and
 * profk_topk_batched calls (the step entry points below keep allocating).
 * dev_ptr: device memory of `bytes` bytes on the device of those calls,
 * 256-byte aligned; the library uses it instead of its memory pool and never
 * frees it.  A call that needs more than `bytes` (profk_workspace_size gives
 * the need) returns PROFK_ERR_SCRATCH without producing output.  The buffer
 * is used in stream order, so calls on different streams must not have it in
 * flight at the same time.  dev_ptr = NULL or bytes = 0 returns to the pool.
 * Returns PROFK_OK, or PROFK_ERR_INVALID for a misaligned pointer. */
int profk_set_workspace(void* dev_ptr, size_t bytes);

/* Process-wide options (defaults in brackets). */
typedef enum profk_option {
  PROFK_OPT_PARAM_MODE = 0,    /* PROFK_PARAMS_DEFAULT [0], _OLD, _EXACT or _CORRECTED */
  PROFK_OPT_MAX_ATTEMPTS = 1,  /* filter attempts before the exact fallback [6]; 0 = fallback at once */
  PROFK_OPT_TIE_EXIT = 2,      /* take PROFK_PATH_TIE when R > M and R_gt < k [1] */
  PROFK_OPT_FORCE_S = 3,       /* >0 overrides S (and disables the exact-path routing) [0] */
  PROFK_OPT_FORCE_T = 4,       /* >0 overrides t [0] */
  PROFK_OPT_FORCE_M = 5,       /* >0 overrides M [0] */
  PROFK_OPT_TIMING = 6,        /* record stats.filter_ms with CUDA events [0] */
  PROFK_OPT_FILTER_CTAS_PER_SM = 7, /* persistent filter grid = SMs x this; 0 = auto [0] */
  PROFK_OPT_PDL = 8,           /* launch kernels with programmatic dependent launch [1] */
  PROFK_OPT_MAX_SEGMENT = 9,   /* rows longer than this are split into segments (see profk_topk);
                                  a multiple of 4, >= 2^16; 0 = 2^32 [0] */
  PROFK_OPT_SAMPLER = 10,      /* kernels of steps 1-2 (sample and tau): PROFK_SAMPLER_AUTO [0],
                                  _GRID, _STEPS or _LISTS (GRID and LISTS fall back to the
                                  automatic choice where they cannot take the problem) */
  PROFK_OPT_WAIT_TEST = 11,    /* test of the path taken when a bounded device wait runs out [0]:
                                  PROFK_WAIT_TEST_SAMPLER, _REFINE or _SORT makes the first grid barrier
                                  of that persistent kernel (the sampler's grid form, the grid
                                  refinement for k <= 8192, the buffer sort above) wait for one CTA
                                  more than the launch has, with a bound of 4096 polls instead of
                                  2^22.  Every CTA of the row then gives up, writes nothing more, and
                                  the call returns PROFK_ERR_DEVICE_TIMEOUT with its outputs untouched;
                                  the next call is unaffected */
  PROFK_OPT_SPECULATIVE = 12,  /* redraws enqueued on the device [0]: 0 .. 8 attempts enqueued right
                                  after the first one, before the host reads the run-time check.  Each
                                  is attempt a of every row (the same sample, tau and result as the
                                  host-driven attempt a), and its kernels leave alone every row that an
                                  earlier attempt settled (its check passed, or it takes the tie exit,
                                  or it met a NaN or an error): a row that fails the check is redrawn
                                  without a host round trip, and the host reads the report once, after
                                  the last of them (profk_wait, for the asynchronous calls).  Results and
                                  statistics are those of the option's default.  Capped at
                                  PROFK_OPT_MAX_ATTEMPTS - 1; taken only where the grid form of the
                                  sampler takes the rows (see PROFK_OPT_SAMPLER) and
                                  PROFK_OPT_TIMING is off.  A call whose rows all pass the first check
                                  pays the empty attempts' launches (a few microseconds each) */
  PROFK_OPT_PREFIX_TEST = 13,  /* test of the grid refinement's prefix check [0]: v in 1 .. 33 makes the
                                  refinement (k <= 8192) trust only the low v - 1 bits of the filter's
                                  record of the bits in which its passers' values differ from tau, so
                                  that it takes a longer prefix as shared by every candidate than the
                                  candidates share; its first pass finds a key outside that prefix and
                                  every CTA of the row starts the passes again from the key's top bit.
                                  Results and statistics are those of the default */
  PROFK_OPT__COUNT = 14
} profk_option;
#define PROFK_WAIT_TEST_OFF 0
#define PROFK_WAIT_TEST_SAMPLER 1
#define PROFK_WAIT_TEST_REFINE 2
#define PROFK_WAIT_TEST_SORT 3
/* Forms of the sampling kernels (PROFK_OPT_SAMPLER); all give the same
 * sample and tau.  GRID: one persistent kernel (all CTAs resident), each CTA
 * taking up to 1024 sample positions; tau from per-CTA candidate lists that
 * one CTA waits for (t <= 8) or from passes whose CTAs meet at grid
 * barriers (larger t).  LISTS (t <= 8): CTAs of up to 2048 positions of one
 * row, each publishing a list of its t largest sampled values; a CTA that
 * finds every list of its row published selects tau among them, and no CTA
 * waits for another; taken for t <= 8 when the rows' shares of the SMs are
 * too small for GRID.
 * STEPS: one thread per sample position, then a radix selection of tau; the
 * remaining cases.  A form that cannot take the problem falls back to the
 * automatic choice. */
#define PROFK_SAMPLER_AUTO 0
#define PROFK_SAMPLER_GRID 1
#define PROFK_SAMPLER_STEPS 2
#define PROFK_SAMPLER_LISTS 3
int profk_set_option(int option, int64_t value);
int64_t profk_get_option(int option);

/* Stage times (ms) of the first filter attempt of this host thread's last
 * profk_topk / profk_topk_batched call made with PROFK_OPT_TIMING on, from
 * CUDA events on the call's stream: out[0] sampling, out[1] threshold
 * selection, out[2] filter, out[3] refinement (enqueued before the check),
 * out[4] read-back of the counts; out[5] is the host wall time of the whole
 * call.  Writes min(count, 6) values (-1 where not measured) and returns that
 * number, or PROFK_ERR_INVALID. */
int profk_last_stage_ms(float* out, int count);

/* Static description of a status code. */
const char* profk_strerror(int code);

/* ---- the individual steps (for testing and composition) ---------------- */

/* Step 1, sampling (paper Section 3, stage 1: a uniform sample of S indices
 * without replacement).  The sample is pi(0), ..., pi(S-1) for a keyed
 * pseudo-random permutation pi of [0, n):
 *   round keys K_0 .. K_11: the words of Philox4x64-10 blocks with counters
 *     (q, attempt, 0, 0), q = 0, 1, 2, under the key (seed, row), in order;
 *   E: a twelve-round Feistel network on [0, 2^b), b = max(2, ceil(log2 n)):
 *     round i splits the state into its high part L and its low w bits R
 *     (w = floor(b/2) in round 0, then the widths alternate) and maps it to
 *     (R << (b - w)) | (L xor (mix(R xor K_i) mod 2^(b - w))), mix being the
 *     SplitMix64 output function (z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *     z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31, mod 2^64);
 *   pi(j): E applied to j, then again while the value is >= n.
 * The S indices are distinct by construction.  Writes out_sidx[0..S)
 * (device int64, in that order) and out_vals[0..S) = x[out_sidx] (device
 * float).  Requires 1 <= S <= n <= 2^32. */
int profk_sample(const float* x, int64_t n, int64_t S, uint64_t seed, int64_t row,
                 int32_t attempt, int64_t* out_sidx, float* out_vals, cudaStream_t stream);

/* Step 2, threshold (Section 3, stage 2): *out_tau (device float) = the t-th
 * largest of vals[0..S) (device), 1 <= t <= S.  A zero is returned as +0.0. */
int profk_threshold(const float* vals, int64_t S, int64_t t, float* out_tau,
                    cudaStream_t stream);

/* Step 3, filter (Section 3, stage 3; Appendix C): one pass over x[0..n)
 * (device, 4-byte aligned) counting out_counts[0] = R = |{x_i >= tau}|,
 * out_counts[1] = |{x_i > tau}|, out_counts[2] = |{x_i is NaN}| (device
 * uint64[3]), and storing min(R, M) passers into out_keys[0..M) (device) in
 * an unspecified order.  A passer (v, i) is stored as the 64-bit key
 *   (ord(v) << 32) | (0xFFFFFFFF - i),
 * ord(v) = bits(v) ^ 0x80000000 for v >= +0.0 (with -0.0 read as +0.0) and
 * ~bits(v) for v < 0, so that keys compare like the library order. */
int profk_filter(const float* x, int64_t n, float tau, int64_t M, uint64_t* out_keys,
                 uint64_t* out_counts, cudaStream_t stream);

/* Step 4, refinement (Section 3, stage 4): exact top-k of the R keys
 * keys[0..R) (device, the profk_filter encoding, distinct), 1 <= k <= R;
 * values are read back from x[0..n) (device) at the decoded indices.  A key
 * whose index is >= n yields the output entry (NaN, -1) instead of a read. */
int profk_refine(const uint64_t* keys, int64_t R, int64_t k, const float* x, int64_t n,
                 float* out_vals, int64_t* out_idx, cudaStream_t stream);

/* Exact top-k over the whole row without sampling (the fallback of Section 3,
 * stage 4): multi-pass radix selection of the k-th largest key, compaction
 * and sort.  Returns PROFK_ERR_NAN if x holds a NaN (synchronizes stream). */
int profk_exact(const float* x, int64_t n, int64_t k, float* out_vals, int64_t* out_idx,
                cudaStream_t stream);

/* ---- calls that allocate nothing --------------------------------------- */

/* Bytes of the fixed device scratch array behind profk_topk_noalloc.  Every
 * GPU that loads the library holds this much device memory until exit. */
#define PROFK_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Exact top-k of one row, with the arguments and the exact result of
 * profk_topk, but without allocating anything: no cudaMalloc/cudaMallocAsync,
 * no pinned host buffer, no pool.  The paper has no counterpart to this entry
 * point; it exists for callers that must not allocate on the call path (a
 * latency-bounded serving loop, a plugin whose host owns all device memory
 * through its own allocator, a process whose pool already holds nearly all
 * of the GPU).  The workspace is a static device array of
 * PROFK_NOALLOC_SCRATCH_BYTES reserved when the library is loaded.  The call
 * runs the step-by-step kernels (sampler, radix selections, sorts without
 * scratch), not the persistent ones of profk_topk, and synchronizes `stream`
 * once per attempt and once at the end.
 *   Limits: n <= 2^32 (longer rows return PROFK_ERR_UNSUPPORTED) and x
 *     4-byte aligned (else PROFK_ERR_UNSUPPORTED).  The array must hold, at
 *     the parameters (S, t, M) that profk_params gives, each part rounded up
 *     to 256 bytes: the row state (8.4 KB); on the sampling route 4S bytes of
 *     sample indices, 4S bytes of sample keys and 8M bytes of candidate
 *     buffer; and 8 K bytes of selected keys, K = k for k <= 8192, else the
 *     power of two >= k.  A problem that needs more returns
 *     PROFK_ERR_SCRATCH before any device work (n = 2^30 with k = 2^19
 *     needs about 14 MB).
 *   Errors: as profk_topk, including PROFK_ERR_CUDA / PROFK_ERR_DEVICE_TIMEOUT
 *     when a device-side check of any step fails.
 *   Statistics: S, t, M, the counts, tau, attempts and path as profk_topk;
 *     aux_bytes is 0 (nothing was allocated); launches counts this call's
 *     kernels, which differ from profk_topk's.
 *   Sharing: every call on a device uses the same array and finds the
 *     previous call's contents there (it clears what must start at zero);
 *     calls whose GPU work overlaps on one device race and must be ordered
 *     by the caller (one stream, or serialized).
 *   Set-up: the first call on a device looks up the array's device address
 *     with that device current and caches it; make that first call before any
 *     stream capture.
 *   Options honoured: PROFK_OPT_PARAM_MODE, PROFK_OPT_MAX_ATTEMPTS,
 *     PROFK_OPT_TIE_EXIT. */
int profk_topk_noalloc(const float* x, int64_t n, int64_t k, double eps, uint64_t seed,
                       float* out_vals, int64_t* out_idx, cudaStream_t stream,
                       profk_stats* stats);

#ifdef __cplusplus
}
#endif

#endif /* PROFK_H_ */
