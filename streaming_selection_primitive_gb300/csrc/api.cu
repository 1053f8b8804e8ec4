// C-ABI of the Prof-K library and the host control of the method
// ("Prof-K: Probabilistic One-Pass Filtering for Efficient Top-k Selection",
// Section 3 "The Prof-K Algorithm": sample -> threshold -> filter -> check ->
// refine, redraw on failure, exact fallback after a fixed number of attempts).
//
// The host does what the pages' host does: it computes (S, t, M) once per
// configuration (memoized, Section 4 "Fast Approximate Parameter
// Computation"), launches the steps on the caller's stream, and reads the
// exact counts back after the filter (the run-time check, Appendix D "Cost of
// the Run-Time Check").  All arithmetic on the data happens in the kernels.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstddef>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/profk.h"
#include "kernels.h"
#include "params.h"

namespace profk {
namespace {

// ---------------------------------------------------------------------------
// Options.
std::atomic<int64_t> g_opt[PROFK_OPT__COUNT] = {
    {PROFK_PARAMS_DEFAULT}, {6}, {1}, {0}, {0}, {0}, {0}, {0}, {1}, {0}, {PROFK_SAMPLER_AUTO}, {PROFK_WAIT_TEST_OFF}, {0},
    {0}};

// PROFK_OPT_WAIT_TEST: the wait setting of the persistent kernel it names
// (one arrival more than the launch has at its first grid barrier, and a
// short bound), the default setting for every other kernel.
WaitCfg wait_cfg_for(int64_t kernel) {
  const int64_t t = g_opt[PROFK_OPT_WAIT_TEST].load();
  if (t == PROFK_WAIT_TEST_OFF || t != kernel) return WaitCfg{};
  WaitCfg w;
  w.skew = 1u;
  w.polls = 1 << 12;
  return w;
}

// Longest row handled as one (PROFK_OPT_MAX_SEGMENT; 0 = 2^32, the reach of a
// candidate key's 32-bit index field).  Longer rows are split into segments.
int64_t max_segment() {
  const int64_t v = g_opt[PROFK_OPT_MAX_SEGMENT].load();
  return v > 0 ? v : (int64_t(1) << 32);
}

// Rows up to 2^40 elements, split into at most this many segments.
constexpr int64_t MAX_ROW = int64_t(1) << 40;
constexpr int64_t MAX_SEGMENTS = 4096;

// A row of n > max_segment() elements as P segments: the first main_rows of
// seg_len elements (a multiple of 4, so every segment stays 16-byte aligned),
// then, unless all are equal (main_rows == P), a shorter last one of tail_len.
struct SegmentPlan {
  int64_t P = 1, seg_len = 0, tail_len = 0, main_rows = 0;
};

SegmentPlan plan_segments(int64_t n, int64_t max_seg) {
  SegmentPlan p;
  p.P = (n + max_seg - 1) / max_seg;
  const int64_t per = (n + p.P - 1) / p.P;
  p.seg_len = (per + 3) & ~int64_t(3);
  p.tail_len = n - (p.P - 1) * p.seg_len;
  p.main_rows = p.tail_len == p.seg_len ? p.P : p.P - 1;
  return p;
}

// ---------------------------------------------------------------------------
// Memoized parameters per (n, k, eps, mode).
Params cached_params(int64_t n, int64_t k, double eps, int mode) {
  static std::mutex mu;
  static std::map<std::tuple<int64_t, int64_t, double, int>, Params> cache;
  const auto key = std::make_tuple(n, k, eps, mode);
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const Params p = compute_params(n, k, eps, mode);
  std::lock_guard<std::mutex> g(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = p;
  return p;
}

// ---------------------------------------------------------------------------
// Device memory: one stream-ordered pool per device, owned by the library.
cudaError_t pool_for_current_device(cudaMemPool_t* out) {
  static std::mutex mu;
  static std::map<int, cudaMemPool_t> pools;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(mu);
  auto it = pools.find(dev);
  if (it != pools.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  cudaMemPoolProps props;
  std::memset(&props, 0, sizeof(props));
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  cudaMemPool_t pool;
  e = cudaMemPoolCreate(&pool, &props);
  if (e != cudaSuccess) return e;
  uint64_t keep = ~0ull;
  cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
  pools[dev] = pool;
  *out = pool;
  return cudaSuccess;
}

// Small pinned host scratch per host thread (row lists and count read-back).
struct Pinned {
  void* p = nullptr;
  size_t cap = 0;
};
thread_local Pinned t_pinned;

cudaError_t pinned(size_t bytes, void** out) {
  if (t_pinned.cap < bytes) {
    if (t_pinned.p) cudaFreeHost(t_pinned.p);
    t_pinned.p = nullptr;
    t_pinned.cap = 0;
    const size_t cap = std::max<size_t>(bytes, 1 << 16);
    cudaError_t e = cudaHostAlloc(&t_pinned.p, cap, cudaHostAllocDefault);
    if (e != cudaSuccess) return e;
    t_pinned.cap = cap;
  }
  *out = t_pinned.p;
  return cudaSuccess;
}

// Stage timing (PROFK_OPT_TIMING): events at the stage boundaries of the
// first attempt, and the stage times of this thread's last timed call.
struct Events {
  cudaEvent_t e[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
};
thread_local Events t_events;
thread_local float t_stage_ms[6] = {-1.f, -1.f, -1.f, -1.f, -1.f, -1.f};

// ---------------------------------------------------------------------------
// Small kernels of the control flow.
// Start of an attempt for the listed rows: counters to zero and the
// selection state ready for tau (rank t).  The control blocks of each row's
// sampling (sample_ctl, sample_words 8-byte words per row) and refinement
// (sort_ctl, ctl_words) are zeroed too.  A row that an earlier attempt
// settled is left alone.
__global__ void k_attempt_reset(const int* rows, RowState* st, unsigned long long t, unsigned long long* sort_ctl,
                                int ctl_words, unsigned long long* sample_ctl, int sample_words, unsigned* block_eq,
                                int64_t nblocks, int attempt) {
  pdl_trigger();
  pdl_wait();
  const int row = launch_row(rows);
  if (settled_before(st[row], attempt)) return;
  // 16-byte stores, grid-strided over the row's CTAs: the control blocks (an
  // even number of words each) to zero.
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t gstride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (sort_ctl) {
    ulonglong2* sc = reinterpret_cast<ulonglong2*>(sort_ctl + static_cast<int64_t>(row) * ctl_words);
    for (int64_t i = gtid; i < ctl_words / 2; i += gstride) sc[i] = make_ulonglong2(0ull, 0ull);
  }
  ulonglong2* pc = reinterpret_cast<ulonglong2*>(sample_ctl + static_cast<int64_t>(row) * sample_words);
  for (int64_t i = gtid; i < sample_words / 2; i += gstride) pc[i] = make_ulonglong2(0ull, 0ull);
  RowState& S = st[row];
  for (int64_t b = gtid; b < HIST_BINS; b += gstride) S.hist[b] = 0;
  if (block_eq) {
    unsigned* be = block_eq + static_cast<int64_t>(row) * nblocks;
    for (int64_t b = gtid; b < nblocks; b += gstride) be[b] = 0u;
  }
  if (gtid == 0) {
    S.R_ge = 0;
    S.R_gt = 0;
    S.nan = 0;
    S.distinct = 0;
    S.error = 0;
    S.sel_prefix = 0;
    S.sel_rank = t;
    S.sel_above = 0;
    S.sel_bucket = 0;
    S.sel_thresh = 0;
    S.sel_nan = 0;
    S.sel_bits = 0;
    S.sel_done = 0;
    S.done_blocks = 0;
    S.compact_count = 0;
    S.skip = 0;
    S.tie_gt = 0;
    S.tau_copies = 0;
    S.settled = 0;
    S.vdiff = 0;
  }
}

__global__ void k_set_tau(RowState* st, float tau) {
  pdl_trigger();
  pdl_wait();
  st->tau_key = ord_key(tau);
  st->vdiff = 0;
  st->R_ge = 0;
  st->R_gt = 0;
  st->nan = 0;
}

__global__ void k_set_count(RowState* st, unsigned long long R) {
  pdl_trigger();
  pdl_wait(); st->R_ge = R; }

__global__ void k_vals_to_keys(const float* v, int64_t S, uint32_t* keys) {
  pdl_trigger();
  pdl_wait();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < S;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    keys[i] = ord_key(v[i]);
}

__global__ void k_tau_out(const RowState* st, float* out) {
  pdl_trigger();
  pdl_wait(); *out = key_to_float(st->tau_key); }

__global__ void k_sample_out(const uint32_t* sidx, int64_t S, const float* x, int64_t* out_sidx, float* out_vals) {
  pdl_trigger();
  pdl_wait();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < S;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t u = sidx[i];
    out_sidx[i] = static_cast<int64_t>(u);
    out_vals[i] = x[u];
  }
}

// ---------------------------------------------------------------------------
// Workspace layout.
size_t align_up(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct Layout {
  int64_t rows = 0, n = 0, k = 0, S = 0, M = 0, kstride = 0;
  bool sampling = false;
  bool radix_refine = false;  // step 4 on the filter buffer by the radix sort
  size_t off_state = 0, off_lists = 0, off_sidx = 0, off_skeys = 0, off_buf = 0, off_sel = 0, off_sort = 0,
         off_refine = 0, off_sctl = 0, off_tie = 0, total = 0;
};

Layout make_layout(int64_t rows, int64_t n, int64_t k, int64_t S, int64_t M, bool sampling) {
  Layout L;
  L.rows = rows;
  L.n = n;
  L.k = k;
  L.S = S;
  L.M = M;
  L.sampling = sampling;
  L.kstride = sort_stride(k);
  size_t off = 0;
  L.off_state = off;
  off = align_up(off + sizeof(RowState) * rows);
  L.off_lists = off;
  off = align_up(off + sizeof(int) * rows * 4);
  if (sampling) {
    L.off_sidx = off;
    off = align_up(off + sizeof(uint32_t) * rows * S);
    L.off_skeys = off;
    off = align_up(off + sizeof(uint32_t) * rows * S);
    L.off_buf = off;
    off = align_up(off + sizeof(unsigned long long) * rows * M);
    L.off_sctl = off;
    off = align_up(off + sample_tau_scratch_bytes(rows));
  }
  L.off_sel = off;
  off = align_up(off + sizeof(unsigned long long) * rows * L.kstride);
  L.off_sort = off;
  // Radix-sort scratch, for whichever of its two uses this call can have: the
  // filter buffer (row stride M) and the k selected keys (row stride kstride).
  L.radix_refine = sampling && !(k <= refine_grid_max_k() && M <= refine_grid_max_m());
  size_t sort_bytes = 0;
  if (k > small_sort_max()) sort_bytes = radix_sort_scratch_bytes(L.kstride, rows);
  if (L.radix_refine) sort_bytes = std::max(sort_bytes, radix_sort_scratch_bytes(M, rows));
  off = align_up(off + sort_bytes);
  L.off_refine = off;
  if (sampling && !L.radix_refine) off = align_up(off + refine_grid_scratch_bytes(rows));
  L.off_tie = off;  // tie exit and exact path: control blocks, block counts and their prefixes
  off = align_up(off + align_up(tie_ctl_bytes() * rows) + align_up(sizeof(unsigned) * tie_blocks(n) * rows) +
                 sizeof(unsigned long long) * tie_blocks(n) * rows);
  L.total = off;
  return L;
}

template <class T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

// Per-row counters read back after each filter pass (the head of RowState).
constexpr size_t REPORT_BYTES = offsetof(RowState, hist);
static_assert(REPORT_BYTES % 4 == 0, "the report is copied in 4-byte words");

// The check's report written straight into pinned host memory: the heads of
// the first `rows` row states, then (after a system-scope fence) the call's
// sequence number in *flag, which the host waits for.  One CTA; used for up
// to REPORT_ROWS_MAPPED rows.
constexpr int64_t REPORT_ROWS_MAPPED = 64;

__global__ void __launch_bounds__(256) k_report(const RowState* st, int rows, unsigned* rep,
                                                unsigned long long* flag, unsigned long long seq) {
  pdl_trigger();
  pdl_wait();
  constexpr int W = static_cast<int>(REPORT_BYTES / 4);
  for (int i = threadIdx.x; i < rows * W; i += blockDim.x) {
    const unsigned* src = reinterpret_cast<const unsigned*>(st + i / W);
    *reinterpret_cast<volatile unsigned*>(rep + i) = __ldcg(src + i % W);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence_system();
    *reinterpret_cast<volatile unsigned long long*>(flag) = seq;
  }
}

thread_local unsigned long long t_report_seq = 0;

// The host buffers of the reports are reused from call to call, and where a
// call's flag word lies depends on its row count: an earlier call's report
// (a count, a rank, a key) may hold any value there, the new call's sequence
// number included.  So the word is cleared before the kernel that writes it
// is enqueued (sequence numbers start at 1).
void clear_flag(unsigned long long* flag) {
  *reinterpret_cast<volatile unsigned long long*>(flag) = 0ull;
  std::atomic_thread_fence(std::memory_order_seq_cst);
}

// Waits for the report of sequence number `seq`.  A stream that fails or
// finishes without it (or a wait of more than 10 s) ends the wait with the
// stream synchronized, so that its error, if any, is returned.
cudaError_t wait_report(const volatile unsigned long long* flag, unsigned long long seq, cudaStream_t stream) {
  const auto t0 = std::chrono::steady_clock::now();
  for (uint64_t spin = 0;; ++spin) {
    if (*flag == seq) {
      std::atomic_thread_fence(std::memory_order_acquire);
      return cudaSuccess;
    }
    if ((spin & 1023) == 1023) {
      const cudaError_t q = cudaStreamQuery(stream);
      const bool late = std::chrono::steady_clock::now() - t0 > std::chrono::seconds(10);
      if ((q != cudaErrorNotReady && *flag != seq) || late) {
        const cudaError_t e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return e;
        return *flag == seq ? cudaSuccess : cudaErrorUnknown;
      }
    }
  }
}

struct Call {
  cudaStream_t stream;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  bool ws_user = false;  // the caller's workspace (profk_set_workspace): never freed
  cudaError_t err = cudaSuccess;
  int status = PROFK_OK;
};

// A failed CUDA call ends the call with PROFK_ERR_CUDA, unless a more specific
// status was already set.
#define PK_CHECK(expr)                                  \
  do {                                                  \
    cudaError_t e_ = (expr);                            \
    if (e_ != cudaSuccess) {                            \
      c.err = e_;                                       \
      if (c.status == PROFK_OK) c.status = PROFK_ERR_CUDA; \
      goto done;                                        \
    }                                                   \
  } while (0)

// Caller-owned workspace of this host thread (profk_set_workspace).
thread_local void* t_user_ws = nullptr;
thread_local size_t t_user_ws_bytes = 0;

// The workspace of a call: the caller's, when one is set and `allow_user`
// (the whole-call entry points), else a stream-ordered pool allocation.
cudaError_t ws_alloc(Call& c, size_t bytes, bool allow_user = false) {
  if (allow_user && t_user_ws) {
    if (bytes > t_user_ws_bytes) {
      c.status = PROFK_ERR_SCRATCH;
      return cudaErrorMemoryAllocation;
    }
    c.ws = t_user_ws;
    c.ws_bytes = bytes;
    c.ws_user = true;
    return cudaSuccess;
  }
  c.ws_user = false;
  cudaMemPool_t pool;
  cudaError_t e = pool_for_current_device(&pool);
  if (e != cudaSuccess) return e;
  e = cudaMallocFromPoolAsync(&c.ws, bytes, pool, c.stream);
  if (e == cudaSuccess) c.ws_bytes = bytes;
  return e;
}

void ws_free(Call& c) {
  if (c.ws && !c.ws_user) cudaFreeAsync(c.ws, c.stream);
  c.ws = nullptr;
}

// Copies a row list into list slot `slot` of the workspace (through the
// pinned scratch at `hbuf`); *dev_out is nullptr for the list 0..rows-1.
cudaError_t upload_rows(const Layout& L, void* ws, void* hbuf, int slot, const std::vector<int>& rows,
                        cudaStream_t stream, int** dev_out) {
  bool identity = static_cast<int64_t>(rows.size()) == L.rows;
  for (size_t i = 0; identity && i < rows.size(); ++i) identity = rows[i] == static_cast<int>(i);
  *dev_out = nullptr;
  if (identity) return cudaSuccess;
  int* hs = static_cast<int*>(hbuf) + slot * L.rows;
  std::copy(rows.begin(), rows.end(), hs);
  int* d = at<int>(ws, L.off_lists) + slot * L.rows;
  *dev_out = d;
  return cudaMemcpyAsync(d, hs, sizeof(int) * rows.size(), cudaMemcpyHostToDevice, stream);
}

__global__ void k_exact_to_tie(RowState* st, const int* rows) {
  pdl_trigger();
  pdl_wait();
  const int row = rows ? rows[blockIdx.x] : static_cast<int>(blockIdx.x);
  if (threadIdx.x == 0) st[row].R_gt = st[row].sel_above;  // |{x > v_k}|, below k
}

int filter_grid(int64_t ctas_per_sm);

// Whether every row starts on a 16-byte boundary.
bool rows_aligned(const float* x, int64_t rows, int64_t ld) {
  return (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (rows == 1 || (ld & 3) == 0);
}

// Rows from which the exact path goes through the value selection and the
// tie step (measured: 430 vs 668 us at n = 2^26; below 2^25 the selection of
// the 64-bit keys, which stops as soon as its bucket is exactly the rest of
// the top k, is faster: 51 vs 78 us at 2^18, 154 vs 212 us at 2^24).
constexpr int64_t EXACT_TIE_MIN_N = int64_t(1) << 25;

// Exact selection over whole rows (fallback / exact path).  Many short rows:
// one CTA per row.  Long rows: the k-th largest VALUE v_k by three radix
// passes over the row's value keys (11, 11 and 10 bits), which also count
// the x > v_k; then the tie step takes every x > v_k and the lowest-index
// copies of v_k (one streaming pass, then a re-read of the blocks that hold
// copies up to the last one taken), and the k keys are sorted: four reads of
// the row and those blocks.  Other rows: the radix selection of the 64-bit
// (value, index) keys, a compaction and the sort.
void launch_exact(const Layout& L, void* ws, const float* x, int64_t ld, int nrows, const int* rows,
                  float* out_vals, int64_t* out_idx, cudaStream_t stream) {
  RowState* st = at<RowState>(ws, L.off_state);
  const bool aligned = (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (L.rows == 1 || (ld & 3) == 0);
  if (aligned && rows_exact_suits(nrows, L.n, L.k)) {
    launch_rows_exact(RowsExactArgs{x, ld, L.n, L.k, nrows, rows, st, out_vals, out_idx}, stream);
    return;
  }
  unsigned long long* sel = at<unsigned long long>(ws, L.off_sel);
  SelectArgs a{KeySource::Input, x, ld, L.n, nrows, rows, st};
  if (aligned && L.n >= EXACT_TIE_MIN_N) {
    launch_select(a, static_cast<uint64_t>(L.k), true, 0, stream);  // value only; leaves tau_key = v_k
    launch_kernel(k_exact_to_tie, nrows, 32, 0, stream, st, rows);
    char* tw = at<char>(ws, L.off_tie);
    const int64_t nb = tie_blocks(L.n);
    TieArgs ta{x, ld, L.n, nrows, rows, st, sel, L.kstride, L.k,
               reinterpret_cast<unsigned*>(tw + align_up(tie_ctl_bytes() * L.rows)),
               reinterpret_cast<unsigned long long*>(tw + align_up(tie_ctl_bytes() * L.rows) +
                                                     align_up(sizeof(unsigned) * nb * L.rows)),
               nb, reinterpret_cast<TieCtl*>(tw), L.rows};
    launch_tie_take(ta, filter_grid(0), stream);
    launch_sort_emit(reinterpret_cast<uint64_t*>(sel), L.kstride, L.k, nrows, rows, x, ld, L.n, out_vals, out_idx,
                     stream, st, at<char>(ws, L.off_sort), L.rows, true);
    return;
  }
  launch_select(a, static_cast<uint64_t>(L.k), false, 0, stream);
  launch_compact(a, reinterpret_cast<uint64_t*>(sel), L.kstride, L.k, stream);
  launch_sort_emit(reinterpret_cast<uint64_t*>(sel), L.kstride, L.k, nrows, rows, x, ld, L.n, out_vals, out_idx, stream,
                   st, at<char>(ws, L.off_sort), L.rows);
}

// SM count and the filter's persistent grid, cached per device.
struct DeviceInfo {
  int sms = 0;
  int filter_grid = 0;
};
DeviceInfo g_dev[64];
std::mutex g_dev_mu;

int filter_grid(int64_t ctas_per_sm) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  std::lock_guard<std::mutex> g(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.sms) {
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (d.sms <= 0) d.sms = 1;
    d.filter_grid = filter_default_grid(d.sms);
  }
  return ctas_per_sm > 0 ? static_cast<int>(d.sms * ctas_per_sm) : d.filter_grid;
}

void fill_stats_params(profk_stats* s, const Params& P) {
  std::memset(s, 0, sizeof(*s));
  s->S = P.S;
  s->t = P.t;
  s->M = P.M;
  s->R_first = s->R_gt_first = s->R_final = s->R_gt_final = -1;
  s->filter_ms = -1.f;
}


// Kernels of steps 1-2 for ng rows of S sample positions each and tau of
// rank t: the form PROFK_OPT_SAMPLER asks for where it takes the problem;
// otherwise the persistent grid kernel where its CTAs' shares of the sample
// fit their registers, else the lists kernel for t <= 8, else the
// step-by-step ones.
enum class Sampler { Grid, Lists, Steps };

Sampler choose_sampler(int64_t S, int64_t ng, unsigned long long t) {
  const int64_t opt = g_opt[PROFK_OPT_SAMPLER].load();
  if (opt == PROFK_SAMPLER_STEPS) return Sampler::Steps;
  const bool lists = sample_lists_fits(S, t);
  if (opt == PROFK_SAMPLER_LISTS && lists) return Sampler::Lists;
  if (sample_tau_fits(S, static_cast<int>(ng))) return Sampler::Grid;
  return lists ? Sampler::Lists : Sampler::Steps;
}

// Attempts enqueued after the first attempt of all `rows`, before the host
// reads the check (PROFK_OPT_SPECULATIVE): within max_attempts, and only where
// the grid or the lists sampler takes the rows (the step-by-step kernels do
// not leave settled rows alone).
int speculative_attempts(const Params& P, int64_t rows, int max_attempts) {
  const int64_t want = g_opt[PROFK_OPT_SPECULATIVE].load();
  if (want <= 0 || max_attempts <= 1 || choose_sampler(P.S, rows, P.t) == Sampler::Steps) return 0;
  return static_cast<int>(std::min<int64_t>(want, max_attempts - 1));
}

// One attempt of the listed rows (gl, ng of them; all rows when gl is null):
// reset, sampling and tau, filter, and the refinement, which is enqueued
// before the host has seen the counts (a row whose count fails the check is
// voided on the device and left untouched, so the host round trip of the
// check is off the critical path of the likely successful attempt).  ev:
// stage events e[1..4] (e[0] is the caller's), or nullptr.  The refinement
// also records the check's outcome in the row state (settle_row, with the
// call's tie_exit), and every kernel of an attempt a > 0 leaves alone the
// rows that an earlier one settled, so that attempts can follow one another
// on the stream before the host has read any report.
cudaError_t enqueue_attempt(const Layout& L, void* ws, const Params& P, int a, int ng, const int* gl, int64_t rows,
                            const float* x, int64_t ld, int64_t n, int64_t k, uint64_t seed, int64_t cps,
                            float* out_vals, int64_t* out_idx, cudaStream_t stream, cudaEvent_t* ev,
                            bool tie_book, bool tie_exit) {
  RowState* st = at<RowState>(ws, L.off_state);
  const Sampler form = choose_sampler(P.S, ng, P.t);
  // Reset CTAs per row: a few 16-byte stores per thread of 256.
  constexpr unsigned rb = 8;
  // The refinement's control blocks start every attempt at zero.
  unsigned long long* ref_ctl =
      L.radix_refine ? static_cast<unsigned long long*>(radix_sort_ctl(at<char>(ws, L.off_sort), P.M, rows))
                     : static_cast<unsigned long long*>(refine_grid_ctl(at<char>(ws, L.off_refine)));
  const int ref_words = static_cast<int>((L.radix_refine ? radix_sort_ctl_bytes() : refine_grid_ctl_bytes()) / 8);
  // tie_book (the call's tie exit is on): the filter keeps the tie step's
  // per-block counts of tau and the x > tau that its full buffer drops (in
  // the selection keys), which the tie exit then uses instead of a pass.
  const int64_t nb = tie_blocks(n);
  unsigned* block_eq = tie_book ? reinterpret_cast<unsigned*>(at<char>(ws, L.off_tie) +
                                                              align_up(tie_ctl_bytes() * rows))
                                : nullptr;
  // The candidate-list forms of the sampler (t <= 8: the grid kernel's and
  // the lists kernel) do the attempt's set-up themselves; the other forms get
  // the reset kernel first.
  const bool fused_setup =
      form == Sampler::Lists || (form == Sampler::Grid && P.t <= static_cast<uint64_t>(sample_tau_setup_max_t()));
  if (!fused_setup)
    launch_kernel(k_attempt_reset, dim3(rb, ng), 256, 0, stream, gl, st, static_cast<unsigned long long>(P.t), ref_ctl,
                  ref_words, at<unsigned long long>(ws, L.off_sctl), static_cast<int>(sample_tau_ctl_bytes() / 8),
                  block_eq, nb, a);
  // Sampling and tau: one persistent kernel (its stage time is reported as
  // the sampling's, the threshold stage then being empty), or, when many rows
  // share the SMs, the step-by-step kernels with the first radix pass of tau
  // fused into the sampler's last one.
  SampleArgs sa{x, ld, static_cast<uint64_t>(n), P.S, seed, a, ng, gl, st, at<uint32_t>(ws, L.off_sidx),
                at<uint32_t>(ws, L.off_skeys), false, static_cast<unsigned long long>(P.t)};
  sa.wait = wait_cfg_for(PROFK_WAIT_TEST_SAMPLER);
  if (fused_setup) {
    sa.zero_ctl = ref_ctl;
    sa.zero_words = ref_words;
    sa.zero_eq = block_eq;
    sa.zero_nb = nb;
  }
  cudaError_t e = cudaSuccess;
  if (form != Sampler::Steps) {
    sa.store_sample = false;  // nothing after this step reads the sample
    e = form == Sampler::Grid ? launch_sample_tau(sa, at<char>(ws, L.off_sctl), rows, stream)
                              : launch_sample_lists(sa, at<char>(ws, L.off_sctl), rows, stream);
    if (e != cudaSuccess) return e;
    if (ev) cudaEventRecord(ev[1], stream);
  } else {
    sa.tau_pass1 = true;
    launch_sample(sa, stream);
    if (ev) cudaEventRecord(ev[1], stream);
    SelectArgs ta{KeySource::SampleKeys, at<uint32_t>(ws, L.off_skeys), P.S, P.S, ng, gl, st};
    launch_select(ta, 0, true, 1, stream);  // its last pass stores tau
  }
  if (ev) cudaEventRecord(ev[2], stream);
  FilterArgs fa{x, ld, n, P.M, ng, gl, st, at<unsigned long long>(ws, L.off_buf), filter_grid(cps), block_eq, nb,
                tie_book ? at<unsigned long long>(ws, L.off_sel) : nullptr, L.kstride, k, a};
  launch_filter(fa, stream);
  if (ev) cudaEventRecord(ev[3], stream);
  if (!L.radix_refine) {
    RefineGridArgs ga{at<unsigned long long>(ws, L.off_buf), P.M, ng, gl, st, k, x, ld, n, out_vals, out_idx};
    ga.wait = wait_cfg_for(PROFK_WAIT_TEST_REFINE);
    const int64_t pt = g_opt[PROFK_OPT_PREFIX_TEST].load();
    if (pt > 0) ga.vdiff_keep = pt > 32 ? 0xFFFFFFFFu : (1u << (pt - 1)) - 1u;
    ga.attempt = a;
    ga.tie_exit = tie_exit;
    e = launch_refine_grid(ga, at<char>(ws, L.off_refine), rows, stream);
  } else {
    // The whole buffer (R <= M keys) is sorted and its first k emitted.
    RadixSortArgs ra{at<unsigned long long>(ws, L.off_buf), P.M, k, SortCount::FromState, ng, gl, rows,
                     at<char>(ws, L.off_sort), true, x, ld, n, out_vals, out_idx, st};
    ra.wait = wait_cfg_for(PROFK_WAIT_TEST_SORT);
    ra.attempt = a;
    ra.tie_exit = tie_exit;
    e = launch_radix_sort(ra, stream);
  }
  if (e != cudaSuccess) return e;
  if (ev) cudaEventRecord(ev[4], stream);
  return cudaGetLastError();
}

// The check's report of the first `rows` row states into `rep` (pinned):
// written by k_report followed by the sequence number in *flag (up to
// REPORT_ROWS_MAPPED rows), else copied (the caller then synchronizes).
cudaError_t enqueue_report(const RowState* st, int64_t rows, char* rep, unsigned long long* flag,
                           unsigned long long seq, cudaStream_t stream) {
  if (rows <= REPORT_ROWS_MAPPED) {
    launch_kernel(k_report, 1, 256, 0, stream, st, static_cast<int>(rows), reinterpret_cast<unsigned*>(rep), flag,
                  seq);
    return cudaGetLastError();
  }
  return cudaMemcpy2DAsync(rep, REPORT_BYTES, st, sizeof(RowState), REPORT_BYTES, rows, cudaMemcpyDeviceToHost,
                           stream);
}

// The state an asynchronous call hands to the synchronous loop when its first
// attempt (and the speculative ones after it) did not clear the check: the
// workspace they used (its layout is run_topk's for the same arguments), the
// parameters and the report (the heads of every row's state).  The loop
// continues from there instead of repeating the attempts.
struct Resume {
  void* ws = nullptr;
  size_t ws_bytes = 0;
  const char* report = nullptr;
  Params P{};
  int64_t launches = 0;  // kernels the first attempt launched
  bool tie_exit = true;  // PROFK_OPT_TIE_EXIT when the first attempt was enqueued
  int extra = 0;         // attempts enqueued after the first (speculative_attempts)
};

int run_topk(const float* x, int64_t rows, int64_t n, int64_t ld, int64_t k, double eps, uint64_t seed,
             float* out_vals, int64_t* out_idx, cudaStream_t stream, profk_stats* stats,
             const Resume* resume = nullptr);

// Rows longer than max_segment(): each row is split into segments (see
// plan_segments), the segments' exact top-k lists are selected by the batched
// path (budget eps / (rows P) per segment), and merged into the row's top k
// by k_merge_segments.  Rows are handled one after the other.
int run_long_rows(const float* x, int64_t rows, int64_t n, int64_t ld, int64_t k, double eps, uint64_t seed,
                  float* out_vals, int64_t* out_idx, cudaStream_t stream, profk_stats* stats) {
  const SegmentPlan sp = plan_segments(n, max_segment());
  if (sp.P > MAX_SEGMENTS || sp.tail_len < 1) return PROFK_ERR_UNSUPPORTED;
  const int64_t k_main = std::min(k, sp.seg_len);
  const bool has_tail = sp.main_rows < sp.P;
  const int64_t k_tail = has_tail ? std::min(k, sp.tail_len) : 0;
  const int64_t cand = sp.main_rows * k_main + k_tail;
  const size_t val_bytes = align_up(sizeof(float) * cand);
  const size_t temp = val_bytes + align_up(sizeof(int64_t) * cand);
  const double eps_seg = eps / static_cast<double>(rows) / static_cast<double>(sp.P);
  const int64_t launches0 = launch_count();
  std::vector<profk_stats> sub(static_cast<size_t>(sp.P));
  int status = PROFK_OK;
  if (stats)
    for (int64_t r = 0; r < rows; ++r) fill_stats_params(&stats[r], Params{0, 0, 0});
  // The candidate lists: from the caller's workspace (its last `temp` bytes,
  // the segment calls using the rest) or from the library's pool.
  void* const user_ws = t_user_ws;
  const size_t user_bytes = t_user_ws_bytes;
  char* tbuf = nullptr;
  cudaMemPool_t pool = nullptr;
  cudaError_t ce = cudaSuccess;
  if (user_ws) {
    if (user_bytes < temp) return PROFK_ERR_SCRATCH;
    tbuf = static_cast<char*>(user_ws) + ((user_bytes - temp) & ~static_cast<size_t>(255));
    t_user_ws_bytes = (user_bytes - temp) & ~static_cast<size_t>(255);
  } else {
    ce = pool_for_current_device(&pool);
    if (ce == cudaSuccess) ce = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&tbuf), temp, pool, stream);
    if (ce != cudaSuccess) {
      if (stats)
        for (int64_t r = 0; r < rows; ++r) {
          std::memset(&stats[r], 0, sizeof(profk_stats));
          stats[r].cuda_error = static_cast<int32_t>(ce);
        }
      return PROFK_ERR_CUDA;
    }
  }
  float* tv = reinterpret_cast<float*>(tbuf);
  int64_t* ti = reinterpret_cast<int64_t*>(tbuf + val_bytes);
  uint64_t aux = 0;
  for (int64_t r = 0; r < rows && status == PROFK_OK; ++r) {
    const float* xr = x + r * ld;
    status = run_topk(xr, sp.main_rows, sp.seg_len, sp.seg_len, k_main, eps_seg * static_cast<double>(sp.main_rows),
                      seed, tv, ti, stream, sub.data());
    if (status == PROFK_OK && has_tail)
      status = run_topk(xr + sp.main_rows * sp.seg_len, 1, sp.tail_len, sp.tail_len, k_tail, eps_seg, seed,
                        tv + sp.main_rows * k_main, ti + sp.main_rows * k_main, stream, &sub[sp.P - 1]);
    if (status == PROFK_OK) {
      launch_merge_segments(MergeSegmentsArgs{tv, ti, static_cast<int>(sp.P), k_main, has_tail ? k_tail : k_main,
                                              sp.seg_len, k, out_vals + r * k, out_idx + r * k},
                            stream);
      ce = cudaGetLastError();
      if (ce != cudaSuccess) status = PROFK_ERR_CUDA;
    }
    if (stats) {
      profk_stats& o = stats[r];
      o = sub[0];
      o.attempts = 0;
      o.path = 0;
      o.draw_doublings = 0;
      o.cuda_error = static_cast<int32_t>(ce);
      int64_t* const sums[4] = {&o.R_first, &o.R_gt_first, &o.R_final, &o.R_gt_final};
      for (auto* p : sums) *p = 0;
      for (const profk_stats& q : sub) {
        const int64_t vals[4] = {q.R_first, q.R_gt_first, q.R_final, q.R_gt_final};
        for (int j = 0; j < 4; ++j) *sums[j] = (*sums[j] < 0 || vals[j] < 0) ? -1 : *sums[j] + vals[j];
        o.attempts = std::max(o.attempts, q.attempts);
        o.path = std::max(o.path, q.path);
        o.draw_doublings += q.draw_doublings;
        if (!o.cuda_error) o.cuda_error = q.cuda_error;
        aux = std::max<uint64_t>(aux, q.aux_bytes);
      }
    }
  }
  if (user_ws)
    t_user_ws_bytes = user_bytes;
  else
    cudaFreeAsync(tbuf, stream);
  if (stats)
    for (int64_t r = 0; r < rows; ++r) {
      stats[r].aux_bytes = aux + temp;
      stats[r].launches = static_cast<int32_t>(launch_count() - launches0);
    }
  return status;
}

int run_topk(const float* x, int64_t rows, int64_t n, int64_t ld, int64_t k, double eps, uint64_t seed,
             float* out_vals, int64_t* out_idx, cudaStream_t stream, profk_stats* stats, const Resume* resume) {
  if (!x || !out_vals || !out_idx) return PROFK_ERR_INVALID;
  if (rows < 1 || n < 1 || k < 1 || k > n || ld < n || !(eps > 0.0 && eps < 1.0)) return PROFK_ERR_INVALID;
  if (rows > (1 << 20)) return PROFK_ERR_INVALID;
  if (n >= MAX_ROW) return PROFK_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) & 3) != 0) return PROFK_ERR_UNSUPPORTED;  // not a float pointer
  if (n > max_segment()) return run_long_rows(x, rows, n, ld, k, eps, seed, out_vals, out_idx, stream, stats);

  const int mode = static_cast<int>(g_opt[PROFK_OPT_PARAM_MODE].load());
  const int max_attempts = static_cast<int>(std::max<int64_t>(0, g_opt[PROFK_OPT_MAX_ATTEMPTS].load()));
  // The first attempt's tie bookkeeping decides for a resumed call.
  const bool tie_exit = resume ? resume->tie_exit : g_opt[PROFK_OPT_TIE_EXIT].load() != 0;
  // Rows that all start on a 16-byte boundary take the vectorised tie step
  // (and the filter's bookkeeping for it); others the selection-based one.
  const bool aligned_rows = rows_aligned(x, rows, ld);
  const int64_t fS = g_opt[PROFK_OPT_FORCE_S].load(), ft = g_opt[PROFK_OPT_FORCE_T].load(),
                fM = g_opt[PROFK_OPT_FORCE_M].load();
  const bool timing = g_opt[PROFK_OPT_TIMING].load() != 0;
  const int64_t cps = g_opt[PROFK_OPT_FILTER_CTAS_PER_SM].load();

  const double eps_row = eps / static_cast<double>(rows);
  Params P = cached_params(n, k, eps_row, mode);
  const bool forced = fS > 0 || ft > 0 || fM > 0;
  if (fS > 0) {
    P.S = std::min<int64_t>(fS, std::max<int64_t>(1, n / 2));
    P.t = std::min<int64_t>(std::max<int64_t>(threshold_rank_fast(n, k, P.S, eps_row), 1), P.S);
    P.M = std::min<int64_t>(std::max<int64_t>(buffer_capacity_fast(n, P.S, P.t, eps_row), k), n);
  }
  if (ft > 0) P.t = std::min<int64_t>(ft, P.S);
  if (fM > 0) P.M = std::min<int64_t>(std::max<int64_t>(fM, k), n);
  if (forced && 2 * P.S > n) return PROFK_ERR_INVALID;
  if (resume) P = resume->P;

  const bool sampling = resume || forced ? true : uses_filter(P, n, k, rows);
  std::vector<profk_stats> st_host(static_cast<size_t>(rows));
  for (auto& s : st_host) fill_stats_params(&s, P);

  Call c;
  c.stream = stream;
  const int64_t launches0 = launch_count();
  const auto wall0 = std::chrono::steady_clock::now();
  const Layout L = make_layout(rows, n, k, P.S, P.M, sampling);
  std::vector<int> pending, fallback, attempt(static_cast<size_t>(rows), 0);
  bool exact_ran = false, tie_ran = false, first_filter = true, resume_used = false;
  float filter_ms = -1.f;
  void* hbuf = nullptr;
  RowState* st = nullptr;

  if (resume) {  // the first attempt's workspace, freed at the end like our own
    c.ws = resume->ws;
    c.ws_bytes = resume->ws_bytes;
    c.ws_user = false;
  } else {
    PK_CHECK(ws_alloc(c, L.total, true));
  }
  st = at<RowState>(c.ws, L.off_state);
  // The sampling path starts every attempt with k_attempt_reset, which
  // initialises the state of its rows; the exact path needs zeroed state,
  // and so does the fallback when no attempt is allowed (max_attempts 0):
  // no reset then runs before it, and the workspace may hold anything.
  if (!sampling || max_attempts == 0) PK_CHECK(cudaMemsetAsync(st, 0, sizeof(RowState) * rows, stream));
  PK_CHECK(pinned(sizeof(int) * rows * 4 + REPORT_BYTES * rows + 512, &hbuf));

  if (!sampling) {
    for (int64_t r = 0; r < rows; ++r) st_host[r].path = PROFK_PATH_EXACT;
    launch_exact(L, c.ws, x, ld, static_cast<int>(rows), nullptr, out_vals, out_idx, stream);
    PK_CHECK(cudaGetLastError());
    exact_ran = true;
  } else {
    for (int64_t r = 0; r < rows; ++r) pending.push_back(static_cast<int>(r));
  }

  while (!pending.empty()) {
    // Rows advance in groups that share an attempt number (the draw stream of
    // an attempt is keyed by it).
    int a = attempt[pending[0]];
    for (int r : pending) a = std::min(a, attempt[r]);
    std::vector<int> group, next;
    for (int r : pending) (attempt[r] == a ? group : next).push_back(r);
    if (a >= max_attempts) {
      for (int r : group) fallback.push_back(r);
      pending = next;
      continue;
    }
    const int ng = static_cast<int>(group.size());
    int* gl = nullptr;
    // The first attempt of all rows already ran (asynchronous call): take its report.
    const bool resumed = resume && !resume_used && a == 0 && static_cast<int64_t>(ng) == rows;
    if (!resumed) PK_CHECK(upload_rows(L, c.ws, hbuf, 0, group, stream, &gl));
    // Attempts a+1 .. a+extra, enqueued after attempt a of all rows before
    // the report is read: a row's report is then that of the attempt that
    // settled it (RowState::settled), or of the last one.
    int extra = 0;
    {
      const bool time_it = timing && first_filter && !resumed;
      if (time_it) {
        if (!t_events.e[0])
          for (auto& ev : t_events.e) PK_CHECK(cudaEventCreate(&ev));
        PK_CHECK(cudaEventRecord(t_events.e[0], stream));
      }
      char* rep = static_cast<char*>(hbuf) + sizeof(int) * rows * 4;
      if (resumed) {
        std::memcpy(rep, resume->report, REPORT_BYTES * rows);
        resume_used = true;
        extra = resume->extra;
      } else {
      PK_CHECK(enqueue_attempt(L, c.ws, P, a, ng, gl, rows, x, ld, n, k, seed, cps, out_vals, out_idx, stream,
                               time_it ? t_events.e : nullptr, tie_exit && aligned_rows, tie_exit));
      if (time_it) PK_CHECK(cudaEventRecord(t_events.e[4], stream));
      if (a == 0 && static_cast<int64_t>(ng) == rows && !timing) extra = speculative_attempts(P, rows, max_attempts);
      for (int q = 1; q <= extra; ++q)
        PK_CHECK(enqueue_attempt(L, c.ws, P, q, ng, gl, rows, x, ld, n, k, seed, cps, out_vals, out_idx, stream,
                                 nullptr, tie_exit && aligned_rows, tie_exit));
      PK_CHECK(cudaGetLastError());
      // Run-time check: read the exact counts of every row (written into
      // pinned memory by a kernel and waited for, or copied and synchronized
      // for many rows).
      {
        unsigned long long* flag =
            reinterpret_cast<unsigned long long*>(align_up(reinterpret_cast<uintptr_t>(rep + REPORT_BYTES * rows)));
        const unsigned long long seq = ++t_report_seq;
        clear_flag(flag);
        PK_CHECK(enqueue_report(st, rows, rep, flag, seq, stream));
        if (time_it) PK_CHECK(cudaEventRecord(t_events.e[5], stream));
        if (rows <= REPORT_ROWS_MAPPED) {
          PK_CHECK(wait_report(flag, seq, stream));
          if (time_it) PK_CHECK(cudaEventSynchronize(t_events.e[5]));
        } else {
          PK_CHECK(cudaStreamSynchronize(stream));
        }
      }
      }
      if (time_it) {
        PK_CHECK(cudaEventElapsedTime(&filter_ms, t_events.e[2], t_events.e[3]));
        for (int q = 0; q < 5; ++q) PK_CHECK(cudaEventElapsedTime(&t_stage_ms[q], t_events.e[q], t_events.e[q + 1]));
        first_filter = false;
      }
      std::vector<int> tie, tie_count;  // tie exit rows with the filter's bookkeeping, and without
      for (int r : group) {
        const char* h = rep + REPORT_BYTES * r;
        unsigned long long Rg = 0, Rt = 0, nanc = 0;
        unsigned distinct = 0, tau_key = 0, errf = 0, copies = 0, settled = 0;
        std::memcpy(&settled, h + offsetof(RowState, settled), 4);
        std::memcpy(&copies, h + offsetof(RowState, tau_copies), 4);
        std::memcpy(&Rg, h + offsetof(RowState, R_ge), 8);
        std::memcpy(&Rt, h + offsetof(RowState, R_gt), 8);
        std::memcpy(&nanc, h + offsetof(RowState, nan), 8);
        std::memcpy(&distinct, h + offsetof(RowState, distinct), 4);
        std::memcpy(&tau_key, h + offsetof(RowState, tau_key), 4);
        std::memcpy(&errf, h + offsetof(RowState, error), 4);
        if (nanc > 0) {
          c.status = PROFK_ERR_NAN;
          goto done;
        }
        if (errf) {
          c.status = (errf & 8u) ? PROFK_ERR_DEVICE_TIMEOUT : PROFK_ERR_CUDA;
          goto done;
        }
        if (static_cast<int64_t>(distinct) != P.S) {  // the sampler always reports S (a consistency check)
          c.status = PROFK_ERR_CUDA;
          goto done;
        }
        profk_stats& s = st_host[r];
        const int ar = extra == 0 ? a : (settled ? static_cast<int>(settled) - 1 : a + extra);  // the report's attempt
        s.attempts = ar + 1;
        const float tau = key_to_float(tau_key);
        if (a == 0) {
          // Attempt 0's counts: the report's own, or the copy that attempt
          // kept when later ones ran before the report was read.
          unsigned long long R1 = Rg, Rt1 = Rt;
          unsigned tau1 = tau_key;
          if (extra > 0) {
            std::memcpy(&R1, h + offsetof(RowState, R_first), 8);
            std::memcpy(&Rt1, h + offsetof(RowState, R_gt_first), 8);
            std::memcpy(&tau1, h + offsetof(RowState, tau_first), 4);
          }
          s.R_first = static_cast<int64_t>(R1);
          s.R_gt_first = static_cast<int64_t>(Rt1);
          s.tau_first = key_to_float(tau1);
        }
        s.R_final = static_cast<int64_t>(Rg);
        s.R_gt_final = static_cast<int64_t>(Rt);
        s.tau_final = tau;
        const bool pass = static_cast<uint64_t>(k) <= Rg && Rg <= static_cast<uint64_t>(P.M);
        const bool tie_row = !pass && tie_exit && Rg > static_cast<uint64_t>(P.M) && Rt < static_cast<uint64_t>(k);
        // The device took the same decision (settle_row): a mismatch is a fault.
        if (extra > 0 && (settled != 0) != (pass || tie_row)) {
          c.status = PROFK_ERR_CUDA;
          goto done;
        }
        if (pass) {
          s.path = PROFK_PATH_FILTER;  // refined on the device already
        } else if (tie_row) {
          s.path = PROFK_PATH_TIE;
          // The filter kept the tie step's counts for the rows whose sample
          // held tau more than once (aligned rows); the others need the
          // counting pass (or, unaligned, the selection-based step).
          (copies >= 2 && aligned_rows ? tie : tie_count).push_back(r);
        } else {
          attempt[r] = ar + 1;
          next.push_back(r);
        }
      }
      // The rows with the filter's bookkeeping first: the counting pass of
      // the others starts by clearing every row's block counts.
      for (int pass = 0; pass < 2; ++pass) {
        const std::vector<int>& tr = pass == 0 ? tie : tie_count;
        if (tr.empty()) continue;
        tie_ran = true;
        int* tl = nullptr;
        PK_CHECK(upload_rows(L, c.ws, hbuf, pass == 0 ? 2 : 1, tr, stream, &tl));
        uint64_t* sel = at<uint64_t>(c.ws, L.off_sel);
        char* tw = at<char>(c.ws, L.off_tie);
        const int64_t nb = tie_blocks(n);
        TieArgs ta{x, ld, n, static_cast<int>(tr.size()), tl, st, reinterpret_cast<unsigned long long*>(sel),
                   L.kstride, k, reinterpret_cast<unsigned*>(tw + align_up(tie_ctl_bytes() * rows)),
                   reinterpret_cast<unsigned long long*>(tw + align_up(tie_ctl_bytes() * rows) +
                                                         align_up(sizeof(unsigned) * nb * rows)),
                   nb, reinterpret_cast<TieCtl*>(tw), rows};
        if (!aligned_rows) {
          // Rows off the 16-byte grid: the selection passes over the rows'
          // (value, index) keys below the resolved value ord(tau) (element
          // loads), the k selected keys compacted, then sorted.  The rows'
          // state is marked skip by the refinement, so the sort takes the
          // listed rows whole.
          launch_tie_init(static_cast<int>(tr.size()), tl, st, k, stream);
          SelectArgs ia{KeySource::Input, x, ld, n, static_cast<int>(tr.size()), tl, st};
          launch_select(ia, 0, false, 3, stream);
          launch_compact(ia, sel, L.kstride, k, stream);
          launch_sort_emit(sel, L.kstride, k, static_cast<int>(tr.size()), tl, x, ld, n, out_vals, out_idx, stream,
                           nullptr, at<char>(c.ws, L.off_sort), L.rows);
          continue;
        }
        if (pass == 0)
          PK_CHECK(launch_tie_after_filter(ta, at<unsigned long long>(c.ws, L.off_buf), P.M, stream));
        else
          PK_CHECK(launch_tie_take(ta, filter_grid(cps), stream));
        launch_sort_emit(sel, L.kstride, k, static_cast<int>(tr.size()), tl, x, ld, n, out_vals, out_idx, stream, st,
                         at<char>(c.ws, L.off_sort), L.rows, true);
      }
      PK_CHECK(cudaGetLastError());
    }
    pending = next;
  }

  if (!fallback.empty()) {
    int* fl = nullptr;
    PK_CHECK(upload_rows(L, c.ws, hbuf, 3, fallback, stream, &fl));
    for (int r : fallback) st_host[r].path = PROFK_PATH_FALLBACK;
    launch_exact(L, c.ws, x, ld, static_cast<int>(fallback.size()), fl, out_vals, out_idx, stream);
    PK_CHECK(cudaGetLastError());
    exact_ran = true;
  }
  if (exact_ran || tie_ran) {
    // The exact selection's first pass counted NaN keys of its rows; a wait
    // of the sort that ran out, or a tie list that does not hold exactly the
    // R_gt keys above tau, is recorded in the error bits.
    char* rep = static_cast<char*>(hbuf) + sizeof(int) * rows * 4;
    PK_CHECK(cudaMemcpy2DAsync(rep, REPORT_BYTES, st, sizeof(RowState), REPORT_BYTES, rows, cudaMemcpyDeviceToHost,
                               stream));
    PK_CHECK(cudaStreamSynchronize(stream));
    for (int64_t r = 0; r < rows; ++r) {
      unsigned long long q = 0;
      unsigned errf = 0;
      std::memcpy(&q, rep + REPORT_BYTES * r + offsetof(RowState, sel_nan), 8);
      std::memcpy(&errf, rep + REPORT_BYTES * r + offsetof(RowState, error), 4);
      if (q && exact_ran) {
        c.status = PROFK_ERR_NAN;
        goto done;
      }
      if (errf) {
        c.status = (errf & 8u) ? PROFK_ERR_DEVICE_TIMEOUT : PROFK_ERR_CUDA;
        goto done;
      }
    }
  }

done:
  ws_free(c);
  if (timing)
    t_stage_ms[5] = std::chrono::duration<float, std::milli>(std::chrono::steady_clock::now() - wall0).count();
  if (stats) {
    for (int64_t r = 0; r < rows; ++r) {
      st_host[r].aux_bytes = c.ws_bytes;
      st_host[r].filter_ms = filter_ms;
      st_host[r].cuda_error = static_cast<int32_t>(c.err);
      st_host[r].launches = static_cast<int32_t>(launch_count() - launches0 + (resume ? resume->launches : 0));
      stats[r] = st_host[r];
    }
  }
  return c.status;
}

}  // namespace

bool pdl_enabled() { return g_opt[PROFK_OPT_PDL].load(std::memory_order_relaxed) != 0; }

}  // namespace profk

using namespace profk;

// An asynchronous call (profk_topk_async / profk_topk_batched_async): its
// first attempt (and the speculative attempts after it) is enqueued and the
// check's report is waited for later, in profk_wait.  A call that the check
// does not clear continues synchronously from that report at that point (the
// same seed gives the same attempts, so the outputs and statistics are those
// of the synchronous call); a call whose report never came is run again.
struct profk_call {
  const float* x = nullptr;
  int64_t rows = 0, n = 0, ld = 0, k = 0;
  double eps = 0.0;
  uint64_t seed = 0;
  float* out_vals = nullptr;
  int64_t* out_idx = nullptr;
  cudaStream_t stream = nullptr;
  bool complete = false;  // already run synchronously at submission
  int status = PROFK_OK;
  std::vector<profk_stats> stats;
  Params P{};
  size_t ws_bytes = 0;
  void* ws = nullptr;
  char* host = nullptr;  // pinned: the report, then the flag
  size_t host_bytes = 0;
  unsigned long long* flag = nullptr;
  unsigned long long seq = 0;
  cudaEvent_t copied = nullptr;  // the report copy of more than REPORT_ROWS_MAPPED rows
  int64_t launches = 0;
  bool tie_exit = true;  // PROFK_OPT_TIE_EXIT at submission
  int extra = 0;         // attempts enqueued after the first (PROFK_OPT_SPECULATIVE)
};

namespace {

// Process-wide sequence numbers of asynchronous reports (never reused, so a
// recycled pinned block cannot show a stale match).
std::atomic<unsigned long long> g_async_seq{0};

// Pinned report blocks, recycled per host thread.
struct PinnedBlock {
  char* p;
  size_t bytes;
};
thread_local std::vector<PinnedBlock> t_free_blocks;

cudaError_t take_block(size_t bytes, char** out, size_t* got) {
  for (size_t i = 0; i < t_free_blocks.size(); ++i) {
    if (t_free_blocks[i].bytes >= bytes) {
      *out = t_free_blocks[i].p;
      *got = t_free_blocks[i].bytes;
      t_free_blocks.erase(t_free_blocks.begin() + static_cast<std::ptrdiff_t>(i));
      return cudaSuccess;
    }
  }
  const size_t cap = std::max<size_t>(bytes, 4096);
  void* p = nullptr;
  const cudaError_t e = cudaHostAlloc(&p, cap, cudaHostAllocDefault);
  if (e != cudaSuccess) return e;
  *out = static_cast<char*>(p);
  *got = cap;
  return cudaSuccess;
}

void give_block(char* p, size_t bytes) {
  if (p) t_free_blocks.push_back({p, bytes});
}

int submit_async(const float* x, int64_t rows, int64_t n, int64_t ld, int64_t k, double eps, uint64_t seed,
                 float* out_vals, int64_t* out_idx, cudaStream_t stream, profk_call** out) {
  if (!out) return PROFK_ERR_INVALID;
  *out = nullptr;
  if (!x || !out_vals || !out_idx) return PROFK_ERR_INVALID;
  if (rows < 1 || n < 1 || k < 1 || k > n || ld < n || !(eps > 0.0 && eps < 1.0)) return PROFK_ERR_INVALID;
  if (rows > (1 << 20)) return PROFK_ERR_INVALID;
  if (n >= MAX_ROW) return PROFK_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) & 3) != 0) return PROFK_ERR_UNSUPPORTED;  // not a float pointer
  profk_call* call = new profk_call;
  call->x = x;
  call->rows = rows;
  call->n = n;
  call->ld = ld;
  call->k = k;
  call->eps = eps;
  call->seed = seed;
  call->out_vals = out_vals;
  call->out_idx = out_idx;
  call->stream = stream;
  call->stats.resize(static_cast<size_t>(rows));
  *out = call;

  const int mode = static_cast<int>(g_opt[PROFK_OPT_PARAM_MODE].load());
  const bool plain = g_opt[PROFK_OPT_FORCE_S].load() == 0 && g_opt[PROFK_OPT_FORCE_T].load() == 0 &&
                     g_opt[PROFK_OPT_FORCE_M].load() == 0 && g_opt[PROFK_OPT_TIMING].load() == 0 &&
                     g_opt[PROFK_OPT_MAX_ATTEMPTS].load() > 0 && t_user_ws == nullptr && n <= max_segment();
  const Params P = cached_params(n, k, eps / static_cast<double>(rows), mode);
  if (!plain || !uses_filter(P, n, k, rows)) {
    // Options, routes and caller workspaces outside the asynchronous form:
    // the call runs now; profk_wait returns its result.
    call->status = run_topk(x, rows, n, ld, k, eps, seed, out_vals, out_idx, stream, call->stats.data());
    call->complete = true;
    return PROFK_OK;
  }
  call->P = P;
  const int64_t launches0 = launch_count();
  const Layout L = make_layout(rows, n, k, P.S, P.M, true);
  Call c;
  c.stream = stream;
  cudaError_t e = ws_alloc(c, L.total, false);
  if (e == cudaSuccess) {
    call->ws = c.ws;
    call->ws_bytes = L.total;
    e = take_block(REPORT_BYTES * rows + 512, &call->host, &call->host_bytes);
  }
  call->tie_exit = g_opt[PROFK_OPT_TIE_EXIT].load() != 0;
  call->extra = speculative_attempts(P, rows, static_cast<int>(g_opt[PROFK_OPT_MAX_ATTEMPTS].load()));
  for (int a = 0; e == cudaSuccess && a <= call->extra; ++a)
    e = enqueue_attempt(L, call->ws, P, a, static_cast<int>(rows), nullptr, rows, x, ld, n, k, seed,
                        g_opt[PROFK_OPT_FILTER_CTAS_PER_SM].load(), out_vals, out_idx, stream, nullptr,
                        call->tie_exit && rows_aligned(x, rows, ld), call->tie_exit);
  if (e == cudaSuccess) {
    call->flag = reinterpret_cast<unsigned long long*>(
        align_up(reinterpret_cast<uintptr_t>(call->host + REPORT_BYTES * rows)));
    call->seq = ++g_async_seq;
    clear_flag(call->flag);
    e = enqueue_report(at<RowState>(call->ws, L.off_state), rows, call->host, call->flag, call->seq, stream);
  }
  if (e == cudaSuccess && rows > REPORT_ROWS_MAPPED) {
    e = cudaEventCreateWithFlags(&call->copied, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(call->copied, stream);
  }
  call->launches = launch_count() - launches0;
  if (e != cudaSuccess) {
    // Nothing usable was enqueued: the call completes with the error.
    if (call->ws) cudaFreeAsync(call->ws, stream);
    call->ws = nullptr;
    give_block(call->host, call->host_bytes);
    call->host = nullptr;
    for (auto& s : call->stats) s.cuda_error = static_cast<int32_t>(e);
    call->status = PROFK_ERR_CUDA;
    call->complete = true;
  }
  return PROFK_OK;
}

int finish_async(profk_call* call, profk_stats* stats) {
  int status = call->status;
  if (!call->complete) {
    cudaError_t e = call->rows <= REPORT_ROWS_MAPPED ? wait_report(call->flag, call->seq, call->stream)
                                                     : cudaEventSynchronize(call->copied);
    bool clear = e == cudaSuccess;
    const unsigned long long k = static_cast<unsigned long long>(call->k);
    for (int64_t r = 0; clear && r < call->rows; ++r) {
      const char* h = call->host + REPORT_BYTES * r;
      unsigned long long Rg = 0, Rt = 0, nanc = 0, R1 = 0, Rt1 = 0;
      unsigned distinct = 0, tau_key = 0, errf = 0, settled = 0, tau1 = 0;
      std::memcpy(&settled, h + offsetof(RowState, settled), 4);
      std::memcpy(&R1, h + offsetof(RowState, R_first), 8);
      std::memcpy(&Rt1, h + offsetof(RowState, R_gt_first), 8);
      std::memcpy(&tau1, h + offsetof(RowState, tau_first), 4);
      std::memcpy(&Rg, h + offsetof(RowState, R_ge), 8);
      std::memcpy(&Rt, h + offsetof(RowState, R_gt), 8);
      std::memcpy(&nanc, h + offsetof(RowState, nan), 8);
      std::memcpy(&distinct, h + offsetof(RowState, distinct), 4);
      std::memcpy(&tau_key, h + offsetof(RowState, tau_key), 4);
      std::memcpy(&errf, h + offsetof(RowState, error), 4);
      // With attempts after the first, a passing row's report is that of
      // the attempt that settled it, and attempt 0's counts are its copy.
      clear = nanc == 0 && errf == 0 && static_cast<int64_t>(distinct) >= call->P.S && k <= Rg &&
              Rg <= static_cast<unsigned long long>(call->P.M) && (call->extra == 0 || settled != 0);
      if (clear) {
        profk_stats& s = call->stats[static_cast<size_t>(r)];
        fill_stats_params(&s, call->P);
        const bool own = call->extra == 0;
        s.R_first = static_cast<int64_t>(own ? Rg : R1);
        s.R_gt_first = static_cast<int64_t>(own ? Rt : Rt1);
        s.tau_first = key_to_float(own ? tau_key : tau1);
        s.R_final = static_cast<int64_t>(Rg);
        s.R_gt_final = static_cast<int64_t>(Rt);
        s.tau_final = key_to_float(tau_key);
        s.attempts = own ? 1 : static_cast<int32_t>(settled);
        s.path = PROFK_PATH_FILTER;
        s.aux_bytes = call->ws_bytes;
        s.launches = static_cast<int32_t>(call->launches);
      }
    }
    if (call->copied) cudaEventDestroy(call->copied);
    if (clear) {
      cudaFreeAsync(call->ws, call->stream);
      status = PROFK_OK;
    } else if (e == cudaSuccess) {
      // Not cleared (a redraw, the tie exit, the fallback, NaN, a device
      // error): the synchronous loop continues from this first attempt, in
      // its workspace (which it frees), with the same result and statistics
      // as profk_topk.
      Resume rs;
      rs.ws = call->ws;
      rs.ws_bytes = call->ws_bytes;
      rs.report = call->host;
      rs.P = call->P;
      rs.launches = call->launches;
      rs.tie_exit = call->tie_exit;
      rs.extra = call->extra;
      status = run_topk(call->x, call->rows, call->n, call->ld, call->k, call->eps, call->seed, call->out_vals,
                        call->out_idx, call->stream, call->stats.data(), &rs);
    } else {
      // The report never came: the whole call again, synchronously.
      cudaFreeAsync(call->ws, call->stream);
      status = run_topk(call->x, call->rows, call->n, call->ld, call->k, call->eps, call->seed, call->out_vals,
                        call->out_idx, call->stream, call->stats.data());
    }
    call->ws = nullptr;
    give_block(call->host, call->host_bytes);
    call->host = nullptr;
  }
  if (stats)
    for (int64_t r = 0; r < call->rows; ++r) stats[r] = call->stats[static_cast<size_t>(r)];
  delete call;
  return status;
}

}  // namespace

extern "C" {

int profk_topk(const float* x, int64_t n, int64_t k, double eps, uint64_t seed, float* out_vals, int64_t* out_idx,
               cudaStream_t stream, profk_stats* stats) {
  return run_topk(x, 1, n, n, k, eps, seed, out_vals, out_idx, stream, stats);
}

int profk_topk_async(const float* x, int64_t n, int64_t k, double eps, uint64_t seed, float* out_vals,
                     int64_t* out_idx, cudaStream_t stream, profk_call** call) {
  return submit_async(x, 1, n, n, k, eps, seed, out_vals, out_idx, stream, call);
}

int profk_topk_batched_async(const float* x, int64_t rows, int64_t n, int64_t ld, int64_t k, double eps,
                             uint64_t seed, float* out_vals, int64_t* out_idx, cudaStream_t stream,
                             profk_call** call) {
  return submit_async(x, rows, n, ld, k, eps, seed, out_vals, out_idx, stream, call);
}

int profk_wait(profk_call* call, profk_stats* stats) {
  if (!call) return PROFK_ERR_INVALID;
  return finish_async(call, stats);
}

int profk_topk_batched(const float* x, int64_t rows, int64_t n, int64_t ld, int64_t k, double eps, uint64_t seed,
                       float* out_vals, int64_t* out_idx, cudaStream_t stream, profk_stats* stats) {
  return run_topk(x, rows, n, ld, k, eps, seed, out_vals, out_idx, stream, stats);
}

int profk_params(int64_t n, int64_t k, double eps, int mode, int64_t* S, int64_t* t, int64_t* M) {
  if (n < 1 || k < 1 || k > n || !(eps > 0.0 && eps < 1.0) || mode < 0 || mode > 3 || !S || !t || !M)
    return PROFK_ERR_INVALID;
  const Params p = cached_params(n, k, eps, mode);
  *S = p.S;
  *t = p.t;
  *M = p.M;
  return PROFK_OK;
}

int profk_set_workspace(void* dev_ptr, size_t bytes) {
  if (dev_ptr && (reinterpret_cast<uintptr_t>(dev_ptr) & 255u)) return PROFK_ERR_INVALID;
  t_user_ws = bytes ? dev_ptr : nullptr;
  t_user_ws_bytes = dev_ptr ? bytes : 0;
  return PROFK_OK;
}

namespace profk {
namespace {
size_t layout_bytes(int64_t rows, int64_t n, int64_t k, double eps) {
  const Params P = cached_params(n, k, eps / static_cast<double>(rows), static_cast<int>(g_opt[0].load()));
  const bool sampling = uses_filter(P, n, k, rows);
  return make_layout(rows, n, k, P.S, P.M, sampling).total;
}
}  // namespace
}  // namespace profk

size_t profk_workspace_size(int64_t rows, int64_t n, int64_t k, double eps) {
  if (rows < 1 || n < 1 || k < 1 || k > n || !(eps > 0.0 && eps < 1.0) || n >= MAX_ROW) return 0;
  if (n <= max_segment()) return layout_bytes(rows, n, k, eps);
  // A long row: the larger of its segment calls plus the merge's candidate lists.
  const SegmentPlan sp = plan_segments(n, max_segment());
  if (sp.P > MAX_SEGMENTS || sp.tail_len < 1) return 0;
  const int64_t k_main = std::min(k, sp.seg_len);
  const bool has_tail = sp.main_rows < sp.P;
  const int64_t k_tail = has_tail ? std::min(k, sp.tail_len) : 0;
  const int64_t cand = sp.main_rows * k_main + k_tail;
  const double eps_seg = eps / static_cast<double>(rows) / static_cast<double>(sp.P);
  size_t need = layout_bytes(sp.main_rows, sp.seg_len, k_main, eps_seg * static_cast<double>(sp.main_rows));
  if (has_tail) need = std::max(need, layout_bytes(1, sp.tail_len, k_tail, eps_seg));
  return align_up(need) + align_up(sizeof(float) * cand) + align_up(sizeof(int64_t) * cand);
}

int profk_set_option(int option, int64_t value) {
  if (option < 0 || option >= PROFK_OPT__COUNT) return PROFK_ERR_INVALID;
  if (option == PROFK_OPT_PARAM_MODE && (value < 0 || value > 3)) return PROFK_ERR_INVALID;
  if (option == PROFK_OPT_SAMPLER && (value < PROFK_SAMPLER_AUTO || value > PROFK_SAMPLER_LISTS))
    return PROFK_ERR_INVALID;
  if (option == PROFK_OPT_WAIT_TEST && (value < PROFK_WAIT_TEST_OFF || value > PROFK_WAIT_TEST_SORT))
    return PROFK_ERR_INVALID;
  if (option == PROFK_OPT_SPECULATIVE && value > 8) return PROFK_ERR_INVALID;
  if (option == PROFK_OPT_PREFIX_TEST && value > 33) return PROFK_ERR_INVALID;
  if (option == PROFK_OPT_MAX_SEGMENT && value != 0 && (value < (1 << 16) || value > (int64_t(1) << 32) || (value & 3)))
    return PROFK_ERR_INVALID;
  if (value < 0) return PROFK_ERR_INVALID;
  g_opt[option].store(value);
  return PROFK_OK;
}

int64_t profk_get_option(int option) {
  if (option < 0 || option >= PROFK_OPT__COUNT) return PROFK_ERR_INVALID;
  return g_opt[option].load();
}

const char* profk_strerror(int code) {
  switch (code) {
    case PROFK_OK: return "ok";
    case PROFK_ERR_INVALID: return "invalid argument";
    case PROFK_ERR_CUDA: return "CUDA error";
    case PROFK_ERR_NAN: return "input contains NaN";
    case PROFK_ERR_UNSUPPORTED: return "unsupported input (a row longer than the library takes, or x not 4-byte aligned)";
    case PROFK_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case PROFK_ERR_SCRATCH: return "problem needs more workspace than the fixed scratch or the caller's workspace";
    default: return "unknown status";
  }
}

int profk_last_stage_ms(float* out, int count) {
  if (!out || count < 1) return PROFK_ERR_INVALID;
  const int m = count < 6 ? count : 6;
  for (int q = 0; q < m; ++q) out[q] = t_stage_ms[q];
  return m;
}

int profk_sample(const float* x, int64_t n, int64_t S, uint64_t seed, int64_t row, int32_t attempt,
                 int64_t* out_sidx, float* out_vals, cudaStream_t stream) {
  if (!x || !out_sidx || !out_vals || n < 1 || S < 1 || S > n || n > (1ll << 32) || row < 0 || attempt < 0)
    return PROFK_ERR_INVALID;
  Call c;
  c.stream = stream;
  const Layout L = make_layout(1, n, 1, S, 1, true);
  void* hbuf = nullptr;
  PK_CHECK(ws_alloc(c, L.total));
  {
    RowState* st = at<RowState>(c.ws, L.off_state);
    PK_CHECK(cudaMemsetAsync(st, 0, sizeof(RowState), stream));
    SampleArgs sa{x, n, static_cast<uint64_t>(n), S, seed, attempt, 1, nullptr, st, at<uint32_t>(c.ws, L.off_sidx),
                  at<uint32_t>(c.ws, L.off_skeys), false, 1ull, row};
    // The main path's kernel for one row (it also finds a tau, of rank 1
    // here, which is not used), else the step-by-step one.
    const Sampler form = choose_sampler(S, 1, 1);
    if (form == Sampler::Grid) {
      PK_CHECK(cudaMemsetAsync(at<char>(c.ws, L.off_sctl), 0, sample_tau_ctl_bytes(), stream));
      PK_CHECK(launch_sample_tau(sa, at<char>(c.ws, L.off_sctl), 1, stream));
    } else if (form == Sampler::Lists) {
      PK_CHECK(launch_sample_lists(sa, at<char>(c.ws, L.off_sctl), 1, stream));
    } else {
      launch_sample_rows(sa, row, stream);
    }
    PK_CHECK(cudaGetLastError());
    PK_CHECK(pinned(REPORT_BYTES, &hbuf));
    PK_CHECK(cudaMemcpyAsync(hbuf, st, REPORT_BYTES, cudaMemcpyDeviceToHost, stream));
    PK_CHECK(cudaStreamSynchronize(stream));
    unsigned errf = 0;
    std::memcpy(&errf, static_cast<char*>(hbuf) + offsetof(RowState, error), 4);
    if (errf) {
      c.status = (errf & 8u) ? PROFK_ERR_DEVICE_TIMEOUT : PROFK_ERR_CUDA;
      goto done;
    }
    const unsigned b = static_cast<unsigned>(std::min<int64_t>((S + 255) / 256, 1024));
    launch_kernel(k_sample_out, b, 256, 0, stream, at<uint32_t>(c.ws, L.off_sidx), S, x, out_sidx, out_vals);
    PK_CHECK(cudaGetLastError());
  }
done:
  ws_free(c);
  return c.status;
}

int profk_threshold(const float* vals, int64_t S, int64_t t, float* out_tau, cudaStream_t stream) {
  if (!vals || !out_tau || S < 1 || t < 1 || t > S || S > (1ll << 31)) return PROFK_ERR_INVALID;
  Call c;
  c.stream = stream;
  const size_t bytes = align_up(sizeof(RowState)) + align_up(sizeof(uint32_t) * S);
  PK_CHECK(ws_alloc(c, bytes));
  {
    RowState* st = at<RowState>(c.ws, 0);
    uint32_t* keys = at<uint32_t>(c.ws, align_up(sizeof(RowState)));
    PK_CHECK(cudaMemsetAsync(st, 0, sizeof(RowState), stream));
    const unsigned b = static_cast<unsigned>(std::min<int64_t>((S + 255) / 256, 1024));
    launch_kernel(k_vals_to_keys, b, 256, 0, stream, vals, S, keys);
    SelectArgs ta{KeySource::SampleKeys, keys, S, S, 1, nullptr, st};
    launch_select(ta, static_cast<uint64_t>(t), true, 0, stream);
    launch_store_tau(1, nullptr, st, stream);
    launch_kernel(k_tau_out, 1, 1, 0, stream, st, out_tau);
    PK_CHECK(cudaGetLastError());
  }
done:
  ws_free(c);
  return c.status;
}

int profk_filter(const float* x, int64_t n, float tau, int64_t M, uint64_t* out_keys, uint64_t* out_counts,
                 cudaStream_t stream) {
  if (!x || !out_counts || n < 1 || M < 0 || (M > 0 && !out_keys) || n > (1ll << 32)) return PROFK_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(x) & 3) != 0) return PROFK_ERR_UNSUPPORTED;
  Call c;
  c.stream = stream;
  PK_CHECK(ws_alloc(c, align_up(sizeof(RowState))));
  {
    RowState* st = at<RowState>(c.ws, 0);
    PK_CHECK(cudaMemsetAsync(st, 0, sizeof(RowState), stream));
    launch_kernel(k_set_tau, 1, 1, 0, stream, st, tau);
    const int64_t cps = g_opt[PROFK_OPT_FILTER_CTAS_PER_SM].load();
    FilterArgs fa{x, n, n, M, 1, nullptr, st, reinterpret_cast<unsigned long long*>(out_keys), filter_grid(cps)};
    launch_filter(fa, stream);
    PK_CHECK(cudaMemcpyAsync(out_counts, &st->R_ge, 3 * sizeof(unsigned long long), cudaMemcpyDeviceToDevice, stream));
    PK_CHECK(cudaGetLastError());
  }
done:
  ws_free(c);
  return c.status;
}

int profk_refine(const uint64_t* keys, int64_t R, int64_t k, const float* x, int64_t n, float* out_vals,
                 int64_t* out_idx, cudaStream_t stream) {
  if (!keys || !x || !out_vals || !out_idx || k < 1 || R < k || n < 1) return PROFK_ERR_INVALID;
  Call c;
  c.stream = stream;
  const int64_t ks = sort_stride(k);
  PK_CHECK(ws_alloc(c, align_up(sizeof(RowState)) + align_up(sizeof(unsigned long long) * ks)));
  {
    RowState* st = at<RowState>(c.ws, 0);
    unsigned long long* sel = at<unsigned long long>(c.ws, align_up(sizeof(RowState)));
    PK_CHECK(cudaMemsetAsync(st, 0, sizeof(RowState), stream));
    launch_kernel(k_set_count, 1, 1, 0, stream, st, static_cast<unsigned long long>(R));
    if (k <= refine_one_max_k() && R <= refine_one_max_m()) {
      RefineOneArgs oa{reinterpret_cast<const unsigned long long*>(keys), R, 1, nullptr, st, k, x, 0, n,
                       out_vals, out_idx};
      launch_refine_one(oa, stream);
    } else {
      SelectArgs ra{KeySource::Buffer, keys, R, R, 1, nullptr, st};
      launch_select(ra, static_cast<uint64_t>(k), false, 0, stream);
      launch_compact(ra, reinterpret_cast<uint64_t*>(sel), ks, k, stream);
      launch_sort_emit(reinterpret_cast<uint64_t*>(sel), ks, k, 1, nullptr, x, 0, n, out_vals, out_idx, stream);
    }
    PK_CHECK(cudaGetLastError());
  }
done:
  ws_free(c);
  return c.status;
}

int profk_exact(const float* x, int64_t n, int64_t k, float* out_vals, int64_t* out_idx, cudaStream_t stream) {
  if (!x || !out_vals || !out_idx || n < 1 || k < 1 || k > n) return PROFK_ERR_INVALID;
  if (n > (1ll << 32)) return PROFK_ERR_UNSUPPORTED;
  Call c;
  c.stream = stream;
  Layout L = make_layout(1, n, k, 0, 0, false);
  void* hbuf = nullptr;
  PK_CHECK(ws_alloc(c, L.total));
  {
    RowState* st = at<RowState>(c.ws, L.off_state);
    PK_CHECK(cudaMemsetAsync(st, 0, sizeof(RowState), stream));
    launch_exact(L, c.ws, x, n, 1, nullptr, out_vals, out_idx, stream);
    PK_CHECK(cudaGetLastError());
    PK_CHECK(pinned(REPORT_BYTES, &hbuf));
    PK_CHECK(cudaMemcpyAsync(hbuf, st, REPORT_BYTES, cudaMemcpyDeviceToHost, stream));
    PK_CHECK(cudaStreamSynchronize(stream));
    unsigned long long q = 0;
    std::memcpy(&q, static_cast<char*>(hbuf) + offsetof(RowState, sel_nan), 8);
    if (q) c.status = PROFK_ERR_NAN;
  }
done:
  ws_free(c);
  return c.status;
}

}  // extern "C"
