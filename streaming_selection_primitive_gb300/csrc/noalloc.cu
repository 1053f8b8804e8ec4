// profk_topk_noalloc: the single-row Prof-K call of profk_topk, run entirely
// inside a fixed scratch array that the library reserves when it is loaded,
// so that the call itself allocates no device (or pinned host) memory.
//
// Who needs this: callers that must not allocate on the call path, such as a
// latency-bounded serving loop (an allocation may synchronize or stall), a
// plugin embedded in a host program that owns all device memory through its
// own allocator, or a process whose memory pool has already reserved nearly
// all of the GPU.  They still pass the input and the outputs.
//
// The scratch is one file-scope device array of PROFK_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  All
// calls share it, and it keeps whatever the previous call left there, so each
// call clears what must start at zero (the row's counters).  Two calls whose GPU work overlaps (different streams, or different
// host threads, on the same device) race on the array and give wrong results:
// order them on one stream or serialize them.
//
// Set-up: the first call on each device (with that device current) asks the
// runtime for the array's device address (cudaGetSymbolAddress) and caches it;
// later calls on that device reuse the cached address.  Make that first call
// before capturing any stream.
#include <cstddef>
#include <cstring>
#include <mutex>

#include "../../include/profk.h"
#include "kernels.h"
#include "params.h"

static __device__ __align__(256) unsigned char profk_noalloc_scratch[PROFK_NOALLOC_SCRATCH_BYTES];

namespace profk {
namespace {

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {};

// Device address of the scratch array on the current device (set-up step).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, profk_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Single-row layout inside the scratch array.
struct ScratchLayout {
  int64_t kstride = 0;
  size_t off_sidx = 0, off_skeys = 0, off_buf = 0, off_sel = 0, total = 0;
};

ScratchLayout plan(int64_t S, int64_t M, int64_t k, bool sampling) {
  ScratchLayout L;
  L.kstride = sort_stride(k);
  size_t off = up256(sizeof(RowState));
  if (sampling) {
    L.off_sidx = off;
    off = up256(off + sizeof(uint32_t) * S);
    L.off_skeys = off;
    off = up256(off + sizeof(uint32_t) * S);
    L.off_buf = off;
    off = up256(off + sizeof(unsigned long long) * M);
  }
  L.off_sel = off;
  off = up256(off + sizeof(unsigned long long) * L.kstride);
  L.total = off;
  return L;
}

template <class T>
T* in(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

}  // namespace
}  // namespace profk

using namespace profk;

extern "C" int profk_topk_noalloc(const float* x, int64_t n, int64_t k, double eps, uint64_t seed, float* out_vals,
                                  int64_t* out_idx, cudaStream_t stream, profk_stats* stats) {
  if (!x || !out_vals || !out_idx) return PROFK_ERR_INVALID;
  if (n < 1 || k < 1 || k > n || !(eps > 0.0 && eps < 1.0)) return PROFK_ERR_INVALID;
  if (n > (1ll << 32)) return PROFK_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) & 3) != 0) return PROFK_ERR_UNSUPPORTED;  // not a float pointer

  const int mode = static_cast<int>(profk_get_option(PROFK_OPT_PARAM_MODE));
  const int64_t max_attempts = profk_get_option(PROFK_OPT_MAX_ATTEMPTS);
  const bool tie_exit = profk_get_option(PROFK_OPT_TIE_EXIT) != 0;
  const Params P = compute_params(n, k, eps, mode);
  const bool sampling = uses_filter(P, n, k);
  const ScratchLayout L = plan(P.S, P.M, k, sampling);
  if (L.total > PROFK_NOALLOC_SCRATCH_BYTES) return PROFK_ERR_SCRATCH;

  profk_stats s;
  std::memset(&s, 0, sizeof(s));
  s.S = P.S;
  s.t = P.t;
  s.M = P.M;
  s.R_first = s.R_gt_first = s.R_final = s.R_gt_final = -1;
  s.filter_ms = -1.f;
  s.path = sampling ? PROFK_PATH_FALLBACK : PROFK_PATH_EXACT;
  const int64_t launches0 = launch_count();
  int status = PROFK_OK;
  cudaError_t err = cudaSuccess;
  void* base = nullptr;
  RowState* st = nullptr;
  alignas(16) unsigned char rep[offsetof(RowState, hist)];
  bool ended = false;  // a terminal path (refinement, tie exit, exact selection) was enqueued
  int sms = 1;

  // The row state's head (counts, error bits) back on the host, the stream synchronized.
  auto read_report = [&]() -> bool {
    err = cudaMemcpyAsync(rep, st, sizeof(rep), cudaMemcpyDeviceToHost, stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) status = PROFK_ERR_CUDA;
    return err == cudaSuccess;
  };
  auto word = [&](size_t off) {
    unsigned v = 0;
    std::memcpy(&v, rep + off, 4);
    return v;
  };
  auto dword = [&](size_t off) {
    unsigned long long v = 0;
    std::memcpy(&v, rep + off, 8);
    return v;
  };
  // A device-side check that failed (a bounded wait that ran out: bit 8) ends the call.
  auto error_status = [](unsigned errf) { return (errf & 8u) ? PROFK_ERR_DEVICE_TIMEOUT : PROFK_ERR_CUDA; };

  err = scratch_address(&base);
  if (err == cudaSuccess) {
    int dev = 0;
    err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  if (err != cudaSuccess) status = PROFK_ERR_CUDA;
  st = in<RowState>(base, 0);

  // Steps 1-4 per attempt; redraws with attempt + 1, up to max_attempts.
  for (int64_t a = 0; status == PROFK_OK && sampling && !ended && a < max_attempts;) {
    err = cudaMemsetAsync(st, 0, sizeof(RowState), stream);
    if (err != cudaSuccess) {
      status = PROFK_ERR_CUDA;
      break;
    }
    SampleArgs sa{x, n, static_cast<uint64_t>(n), P.S, seed, static_cast<int>(a), 1, nullptr, st,
                  in<uint32_t>(base, L.off_sidx), in<uint32_t>(base, L.off_skeys)};
    launch_sample(sa, stream);
    SelectArgs ta{KeySource::SampleKeys, in<uint32_t>(base, L.off_skeys), P.S, P.S, 1, nullptr, st};
    launch_select(ta, static_cast<uint64_t>(P.t), true, 0, stream);
    launch_store_tau(1, nullptr, st, stream);
    FilterArgs fa{x, n, n, P.M, 1, nullptr, st, in<unsigned long long>(base, L.off_buf), filter_default_grid(sms)};
    launch_filter(fa, stream);
    err = cudaGetLastError();
    if (err != cudaSuccess) {
      status = PROFK_ERR_CUDA;
      break;
    }
    if (!read_report()) break;
    const unsigned long long Rg = dword(offsetof(RowState, R_ge)), Rt = dword(offsetof(RowState, R_gt));
    const unsigned errf = word(offsetof(RowState, error));
    if (dword(offsetof(RowState, nan)) > 0) {
      status = PROFK_ERR_NAN;
      break;
    }
    if (errf) {
      status = error_status(errf);
      break;
    }
    if (static_cast<int64_t>(word(offsetof(RowState, distinct))) != P.S) {  // always S (a consistency check)
      status = PROFK_ERR_CUDA;
      break;
    }
    s.attempts = static_cast<int32_t>(a + 1);
    const float tau = key_to_float(word(offsetof(RowState, tau_key)));
    if (a == 0) {
      s.R_first = static_cast<int64_t>(Rg);
      s.R_gt_first = static_cast<int64_t>(Rt);
      s.tau_first = tau;
    }
    s.R_final = static_cast<int64_t>(Rg);
    s.R_gt_final = static_cast<int64_t>(Rt);
    s.tau_final = tau;
    uint64_t* sel = in<uint64_t>(base, L.off_sel);
    if (static_cast<uint64_t>(k) <= Rg && Rg <= static_cast<uint64_t>(P.M)) {
      // Refinement: exact top-k of the R buffered keys.
      s.path = PROFK_PATH_FILTER;
      SelectArgs ra{KeySource::Buffer, in<unsigned long long>(base, L.off_buf), P.M, P.M, 1, nullptr, st};
      launch_select(ra, static_cast<uint64_t>(k), false, 0, stream);
      launch_compact(ra, sel, L.kstride, k, stream);
      launch_sort_emit(sel, L.kstride, k, 1, nullptr, x, n, n, out_vals, out_idx, stream);
      ended = true;
    } else if (tie_exit && Rg > static_cast<uint64_t>(P.M) && Rt < static_cast<uint64_t>(k)) {
      // Tie exit: tau is the k-th largest value; x > tau and the lowest-index copies of tau.
      s.path = PROFK_PATH_TIE;
      launch_tie_init(1, nullptr, st, k, stream);
      SelectArgs ia{KeySource::Input, x, n, n, 1, nullptr, st};
      launch_select(ia, 0, false, 3, stream);
      launch_compact(ia, sel, L.kstride, k, stream);
      launch_sort_emit(sel, L.kstride, k, 1, nullptr, x, n, n, out_vals, out_idx, stream);
      ended = true;
    } else {
      ++a;
    }
  }
  if (status == PROFK_OK && !ended) {
    // The exact selection over the row: the exact route, or the fallback after
    // every attempt failed the check.
    err = cudaMemsetAsync(st, 0, sizeof(RowState), stream);
    if (err != cudaSuccess) status = PROFK_ERR_CUDA;
    if (status == PROFK_OK) {
      uint64_t* sel = in<uint64_t>(base, L.off_sel);
      SelectArgs ea{KeySource::Input, x, n, n, 1, nullptr, st};
      launch_select(ea, static_cast<uint64_t>(k), false, 0, stream);
      launch_compact(ea, sel, L.kstride, k, stream);
      launch_sort_emit(sel, L.kstride, k, 1, nullptr, x, n, n, out_vals, out_idx, stream);
      ended = true;
    }
  }
  if (status == PROFK_OK && ended) {
    // The terminal path's own device checks: a NaN found by the exact
    // selection's first pass, or any error bit (a selection that found no
    // digit, a bounded wait that ran out) fails the call as profk_topk does.
    err = cudaGetLastError();
    if (err != cudaSuccess) {
      status = PROFK_ERR_CUDA;
    } else if (read_report()) {
      const unsigned errf = word(offsetof(RowState, error));
      if (s.path >= PROFK_PATH_FALLBACK && dword(offsetof(RowState, sel_nan)) > 0)
        status = PROFK_ERR_NAN;
      else if (errf)
        status = error_status(errf);
    }
  }
  if (stats) {
    s.aux_bytes = 0;  // nothing was allocated; the call used L.total bytes of the fixed scratch
    s.cuda_error = static_cast<int32_t>(err);
    s.launches = static_cast<int32_t>(launch_count() - launches0);
    *stats = s;
  }
  return status;
}
