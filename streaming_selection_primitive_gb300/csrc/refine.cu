// Prof-K step 4 for k <= 8192 ("Prof-K: Probabilistic One-Pass Filtering for
// Efficient Top-k Selection", Section 3, stage 4): the exact top-k of the
// filter's candidate buffer, sorted, written as (value, index).
//
// One persistent kernel, one 1024-thread CTA per SM and contiguous chunk of
// the candidates; all CTAs of the launch are resident together (chunks x rows
// <= the SM count), so that they can meet at grid barriers (bounded waits on
// a per-row arrival counter).  MSD passes of 11-bit digits over the 64-bit
// keys narrow the bucket that holds the k-th largest key, starting at the
// highest bit where the candidates may differ (the filter records which
// value bits of its passers differ from tau's: above them every key is the
// same, so a pass there would find one bucket).  Each CTA histograms its
// chunk's keys inside the current bucket, the histograms meet in global
// atomics, and after the barrier every CTA reads the same totals and takes
// the same decision.  As soon as the keys above the bucket plus the bucket
// fit the gather budget (at least 2k, at most 8192 keys), every CTA appends
// its keys at or above the bucket's bound to a gather list.  Once every CTA
// has gathered, every CTA reads the list, and each key's output position is
// the number of listed keys above it, counted by one warp per key over all
// warps of the launch; the first k are written.  The launch is sized by M,
// before R is known: the passes and the gather run on only as many CTAs as
// chunks of RG_KEYS_PER_CTA keys need, so that their barriers wait for fewer
// arrivals; the other CTAs leave at once when those can count the list
// alone, and otherwise wait for the gather and join the counting, whose cost
// grows with the square of the list.  Values are
// decoded from the keys (they hold them exactly), except zero, whose sign
// the key does not keep: it is read from x.
//
// Two shortcuts take no barrier: a row of at most 2048 candidates (few
// enough to place by counting) is placed at once by every CTA from the
// buffer itself, and rows that would get two CTAs or fewer (many rows share
// the SMs) get one CTA each, in their own instantiation (SOLO), whose
// histograms and gather list stay in shared memory.
//
// The kernel is enqueued before the host has checked k <= R <= M; a row that
// fails the check is marked skip and its outputs are not touched.  The check's
// outcome is recorded in the row state (settle_row), so that the kernels of
// an attempt enqueued after this one leave a settled row alone.
#include "blocksort.cuh"
#include "kernels.h"

namespace profk {

// Per-row control block, zeroed at the start of every attempt.
struct RefineCtl {
  unsigned hist[7][HIST_BINS];  // pass histograms, summed over the chunks
  unsigned bar;                 // grid-barrier arrivals
  unsigned cursor;              // gather-list length
  unsigned abort;               // set by a CTA whose wait gave up
  unsigned broken;              // set by a CTA that found a key outside the shared prefix
  unsigned gdone;               // CTAs whose passes and gather are done
  unsigned pad[59];
};
static_assert(sizeof(RefineCtl) % 16 == 0, "RefineCtl is zeroed with 16-byte stores");

namespace {

constexpr int RG_THREADS = 1024;
constexpr int RG_KPT = 4;                         // keys per thread held across the passes
constexpr int RG_PIECE = RG_THREADS * RG_KPT;     // 4096
constexpr int RG_OUT = 8192;                      // gather capacity (64 KB of shared memory)
constexpr int RG_MAX_K = 8192;
constexpr int64_t RG_MAX_M = int64_t(1) << 19;
#ifndef PROFK_REFINE_KEYS_PER_CTA
#define PROFK_REFINE_KEYS_PER_CTA 256
#endif
constexpr int64_t RG_KEYS_PER_CTA = PROFK_REFINE_KEYS_PER_CTA;  // fewest keys a pass chunk gets (0: one per CTA)
constexpr int64_t RG_PLACE_CMP = 256;  // comparisons a thread may spend counting the list on fewer CTAs
// Every CTA of the row arrives (a release: the CTA's writes, ordered before
// it by the block barrier, become visible with it), then waits until all
// have (target arrivals; acquire loads of the arrival count).  A wait that
// ends without them (bounded, see wait_count) sets *err, which every thread
// reads afterwards.
__device__ __forceinline__ void grid_sync(RefineCtl& c, unsigned target, int* err, int limit) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&c.bar) : "memory");
    if (!wait_count(&c.bar, target, &c.abort, limit)) *err = 1;
  }
  __syncthreads();
}

// Block-wide exclusive scan of one u64 per thread (thread order).
__device__ __forceinline__ unsigned long long excl_scan(unsigned long long v, unsigned long long* sw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sw[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = sw[lane];
    unsigned long long wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(FULL_MASK, wi, o);
      if (lane >= o) wi += t;
    }
    sw[lane] = wi - w;
  }
  __syncthreads();
  const unsigned long long r = sw[warp] + incl - v;
  __syncthreads();
  return r;
}

template <int E>
__device__ __forceinline__ void sort_padded(unsigned long long* s, int cnt) {
  for (int i = cnt + static_cast<int>(threadIdx.x); i < RG_THREADS * E; i += RG_THREADS) s[i] = 0ull;
  __syncthreads();
  block_sort_desc<E>(s);
}

// SOLO: one CTA for the row (many rows share the SMs): the histograms and
// the gather list stay in its shared memory, with no global atomics and no
// barrier; its own instantiation, so that the grid form's code is that of a
// kernel without it.
template <bool SOLO>
__global__ void __launch_bounds__(RG_THREADS, 1) k_refine_grid(RefineGridArgs a, RefineCtl* ctl,
                                                              unsigned long long* gather) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ unsigned long long s_out[];  // RG_OUT keys: the gather list
  __shared__ unsigned h[HIST_BINS];
  __shared__ unsigned long long sw[32];
  __shared__ int s_digit, s_err;
  __shared__ unsigned s_cursor;  // the gather list's length in s_out (one CTA per row)
  __shared__ unsigned long long s_above, s_count;
  const int row = launch_row(a.rows);
  RowState& S = a.st[row];
  RefineCtl& c = ctl[row];
  const int tid = threadIdx.x, lane = tid & 31;
  const unsigned long long R = S.R_ge;
  const unsigned long long k = static_cast<unsigned long long>(a.k);
  // A row that fails the check, or whose earlier steps reported an error,
  // is left alone (its outputs are not touched); so is a row that an
  // earlier attempt settled.  One thread decides for the block; the first
  // CTA's also records the check's outcome (settle_row).
  if (tid == 0) {
    if (settled_before(S, a.attempt)) {
      s_digit = 2;
    } else {
      s_digit = !(k <= R && R <= static_cast<unsigned long long>(a.M)) || __ldcg(&S.error) != 0u;
      if (blockIdx.x == 0) settle_row(S, a.attempt, k, static_cast<unsigned long long>(a.M), a.tie_exit);
    }
  }
  __syncthreads();
  if (s_digit) {
    if (s_digit == 1 && blockIdx.x == 0 && tid == 0) S.skip = 1;
    return;  // every CTA of the row leaves: no barrier is met
  }
  const int limit = wait_limit(a.wait);
  if (tid == 0) {
    s_err = 0;
    s_cursor = 0;
    if (blockIdx.x == 0) S.skip = 0;
  }
  const int64_t len = static_cast<int64_t>(R);
  const int64_t GA = gridDim.x;  // CTAs of the row: all of them place the gathered keys
  int64_t G = GA;                // chunks of the passes (fewer below, once R is known)
  int64_t PG = GA;               // CTAs that count the gathered list (the G alone below, if they can)
  const unsigned long long* keys = a.buf + static_cast<int64_t>(row) * a.M;
  // A key's output slot e < k: (value, index).
  auto emit = [&](int64_t e, unsigned long long key) {
    const uint32_t idx = cand_index(key);
    const uint32_t vk = static_cast<uint32_t>(key >> 32);
    const int64_t o = static_cast<int64_t>(row) * a.k + e;
    // The index is checked against the row length, so that a selection
    // that went wrong never reads outside x: such an entry is (NaN, -1).
    if (static_cast<int64_t>(idx) < a.n) {
      a.out_idx[o] = static_cast<int64_t>(idx);
      a.out_vals[o] = vk == ord_key(0.0f) ? a.x[static_cast<int64_t>(row) * a.ld + idx] : key_to_float(vk);
    } else {
      a.out_idx[o] = -1;
      a.out_vals[o] = __int_as_float(0x7fc00000);
    }
  };
  // Output positions: every CTA reads the list of cnt keys into shared
  // memory (unless it is there already), and each key's position is the
  // number of listed keys above it (keys are distinct), counted by one warp
  // per key, the keys spread over all warps of the launch; the first k are
  // written.
  auto place = [&](const unsigned long long* list, int cnt) {
    if (list)
      for (int i = tid; i < cnt; i += RG_THREADS) s_out[i] = __ldcg(list + i);
    __syncthreads();
    const int warp = tid >> 5;
    for (int e = blockIdx.x * (RG_THREADS / 32) + warp; e < cnt; e += PG * (RG_THREADS / 32)) {
      const unsigned long long key = s_out[e];
      unsigned above = 0;
      for (int j = lane; j < cnt; j += 32) above += s_out[j] > key;
      for (int o = 16; o >= 1; o >>= 1) above += __shfl_xor_sync(FULL_MASK, above, o);
      if (lane == 0 && above < k) emit(above, key);
    }
  };
  // Few candidates (at most 2048, at most 256 comparisons a thread to place
  // them all): no passes and no barrier; the list is the buffer's first R
  // slots (2^22, k = 32: 27.8 -> 22.8 us a call; at R ~ 4K the passes were
  // as fast).  (The test setting of the waits keeps the passes.)
  if (R <= 2048ull && R * R <= 256ull * static_cast<unsigned long long>(GA) * RG_THREADS && a.wait.skew == 0) {
    place(keys, static_cast<int>(R));
    return;
  }
  // One CTA: a pass costs little, so the gather waits for a smaller bucket.
  const unsigned long long lo_budget = SOLO ? 256 : 2048;
  unsigned long long budget = k * 2 < lo_budget ? lo_budget : (k * 2 > RG_OUT ? RG_OUT : k * 2);
  // The launch was sized by M before R was known: with fewer candidates,
  // the passes and the gather take chunks of at least RG_KEYS_PER_CTA keys
  // on the first G CTAs, so that their barriers wait only for those.  When
  // those G can also count the gathered list alone (2k keys at most
  // RG_PLACE_CMP comparisons a thread; the budget is then capped there), the
  // other CTAs leave at once, which frees their SMs for the kernels that
  // follow.  Otherwise they wait until the G have gathered (the row's gdone
  // count) and help count.
  if constexpr (!SOLO) {
    if (RG_KEYS_PER_CTA > 0) {
      const int64_t need = (len + RG_KEYS_PER_CTA - 1) / RG_KEYS_PER_CTA;
      if (need < G) G = need < 1 ? 1 : need;
    }
    const unsigned long long cap =
        static_cast<unsigned long long>(sqrtf(static_cast<float>(G * RG_THREADS * RG_PLACE_CMP)));
    if (G < GA && 2 * k <= cap) {
      if (budget > cap) budget = cap;
      PG = G;
      if (blockIdx.x >= G) return;
    }
    if (blockIdx.x >= G) {
      if (tid == 0 && !wait_count(&c.gdone, static_cast<unsigned>(G), &c.abort, limit)) s_err = 1;
      __syncthreads();
      if (s_err) {
        if (tid == 0) atomicOr(&S.error, ERR_WAIT);
        return;
      }
      const unsigned cur = __ldcg(&c.cursor);
      place(gather + static_cast<int64_t>(row) * RG_OUT, static_cast<int>(cur < RG_OUT ? cur : RG_OUT));
      return;
    }
  }
  const int64_t C = (((len + G - 1) / G) + 31) & ~int64_t(31);
  const int64_t lo = blockIdx.x * C < len ? blockIdx.x * C : len;
  const int64_t hi = lo + C < len ? lo + C : len;
  const bool held = hi - lo <= RG_PIECE;  // the chunk stays in registers across the passes
  unsigned long long kk[RG_KPT];
  if (held) {
#pragma unroll
    for (int r = 0; r < RG_KPT; ++r) {
      const int64_t i = lo + r * RG_THREADS + tid;
      kk[r] = i < hi ? __ldcg(keys + i) : 0ull;
    }
  }
  // The digits start at the highest bit where the candidates may differ.
  // Every value the filter stored agrees with tau above the highest set bit
  // of the row's vdiff word, so the keys share those bits (all 32 value bits
  // when the word is 0: every value equals tau) and the first digit starts
  // just below them.  The first pass checks every key against that prefix;
  // if one breaks it (a buffer the filter did not fill), every CTA learns so
  // at the pass's barrier and the passes start again from bit 63.
  const uint32_t vd = __ldcg(&S.vdiff) & a.vdiff_keep;
  int hib = vd != 0u ? 63 - __clz(vd) : 31;  // the next digit's highest bit
  unsigned long long prefix =
      hib == 63 ? 0ull : (static_cast<unsigned long long>(__ldcg(&S.tau_key)) << 32) >> (hib + 1);
  unsigned long long want = k, thresh = 0, total = k;
  bool checking = hib < 63;
  unsigned target = 0;
#pragma unroll 1
  for (int p = 0; p < 7 && hib >= 0; ++p) {
    // Digits of 11 bits down from hib (the last one narrower).
    const int width = hib < 11 ? hib + 1 : 11;
    const int hs = hib + 1, shift = hs - width, nb = 1 << width;
    for (int b = tid; b < nb; b += RG_THREADS) h[b] = 0;
    __syncthreads();
    bool broken = false;
    for (int64_t base = lo; base < hi; base += RG_PIECE) {
#pragma unroll
      for (int r = 0; r < RG_KPT; ++r) {
        const int64_t i = base + r * RG_THREADS + tid;
        const unsigned long long key = held ? kk[r] : (i < hi ? __ldcg(keys + i) : 0ull);
        const bool m = i < hi && (hs == 64 || (key >> hs) == prefix);
        broken |= checking && i < hi && !m;
        hist_add(h, static_cast<uint32_t>(key >> shift) & (nb - 1), m);
      }
    }
    const bool brk = __syncthreads_or(broken) != 0;
    if constexpr (!SOLO) {
      if (brk && tid == 0) atomicOr(&c.broken, 1u);
      for (int b = tid; b < nb; b += RG_THREADS)
        if (h[b]) atomicAdd(&c.hist[p][b], h[b]);
      grid_sync(c, (target += static_cast<unsigned>(G)) + (p == 0 ? a.wait.skew : 0u), &s_err, limit);
      if (s_err) break;  // block-uniform (read after a block barrier)
    }
    if (checking) {
      checking = false;
      if (SOLO ? brk : __ldcg(&c.broken) != 0u) {  // block-uniform: every CTA reads the same word
        hib = 63;
        prefix = 0;
        __syncthreads();
        continue;
      }
    }
    // Every CTA finds the same digit: the bins counted down from the top,
    // thread t owning max(nb / 1024, 1) of them.
    if (tid == 0) {
      s_digit = 0;
      s_above = 0;
      s_count = 0;
    }
    const int per = nb > RG_THREADS ? nb / RG_THREADS : 1;
    const int top = nb - 1 - tid * per;
    unsigned hv[2] = {0u, 0u};
    unsigned long long local = 0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (q < per && top - q >= 0) {
        hv[q] = SOLO ? h[top - q] : __ldcg(&c.hist[p][top - q]);
        local += hv[q];
      }
    }
    const unsigned long long excl = excl_scan(local, sw);
    if (excl < want && want <= excl + local) {
      unsigned long long acc = excl;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (q < per && top - q >= 0 && want <= acc + hv[q]) {
          s_digit = top - q;
          s_above = acc;
          s_count = hv[q];
          break;
        }
        acc += hv[q];
      }
    }
    __syncthreads();
    prefix = (prefix << width) | static_cast<unsigned long long>(s_digit);
    want -= s_above;
    hib = shift - 1;
    const unsigned long long above_all = k - want;  // keys above the bucket, all in the top-k
    if (s_count == want || shift == 0) {  // the whole bucket is in the top-k: keys >= its bound are exactly k
      thresh = prefix << shift;
      total = k;
      break;
    }
    if (above_all + s_count <= budget) {  // gather the whole bucket and finish in shared memory
      thresh = prefix << shift;
      total = above_all + s_count;
      break;
    }
    __syncthreads();
  }
  // After a wait that gave up, the CTA reports it and leaves without writing
  // anything else.
  if (s_err) {
    if (tid == 0) atomicOr(&S.error, ERR_WAIT);
    return;
  }
  // Gather every key >= thresh (exactly `total` of them, at most RG_OUT):
  // into the row's list in global memory, or into s_out for one CTA.
  unsigned long long* gr = SOLO ? s_out : gather + static_cast<int64_t>(row) * RG_OUT;
  unsigned* cursor = SOLO ? &s_cursor : &c.cursor;
  for (int64_t base = lo; base < hi; base += RG_PIECE) {
#pragma unroll
    for (int r = 0; r < RG_KPT; ++r) {
      const int64_t i = base + r * RG_THREADS + tid;
      const unsigned long long key = held ? kk[r] : (i < hi ? __ldcg(keys + i) : 0ull);
      const bool sel = i < hi && key >= thresh;
      const unsigned m = __ballot_sync(FULL_MASK, sel);
      if (m) {
        unsigned pos0 = 0;
        if (lane == 0) pos0 = atomicAdd(cursor, static_cast<unsigned>(__popc(m)));
        pos0 = __shfl_sync(FULL_MASK, pos0, 0);
        if (sel) {
          const unsigned pos = pos0 + __popc(m & ((1u << lane) - 1u));
          if (pos < RG_OUT) gr[pos] = key;
        }
      }
    }
  }
  if constexpr (SOLO) {
    const int cnt = static_cast<int>(total < RG_OUT ? total : RG_OUT);
    if (cnt <= RG_THREADS) {
      place(nullptr, cnt);  // its barrier orders the list
      return;
    }
    // More keys than counting suits one CTA: a bitonic sort of the list
    // (padded with zero keys, which sort last), then the first k.
    __syncthreads();
    if (cnt <= 2 * RG_THREADS)
      sort_padded<2>(s_out, cnt);
    else if (cnt <= 4 * RG_THREADS)
      sort_padded<4>(s_out, cnt);
    else
      sort_padded<8>(s_out, cnt);
    __syncthreads();
    for (int e = tid; e < static_cast<int>(k); e += RG_THREADS) emit(e, s_out[e]);
    return;
  }
  // Every CTA of the row waits for the G gathers (its own included).
  __syncthreads();
  if (tid == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&c.gdone) : "memory");
    if (!wait_count(&c.gdone, static_cast<unsigned>(G), &c.abort, limit)) s_err = 1;
  }
  __syncthreads();
  if (s_err) {
    if (tid == 0) atomicOr(&S.error, ERR_WAIT);
    return;
  }
  const unsigned cur = __ldcg(&c.cursor);  // = total; read as the waiting CTAs read it
  place(gr, static_cast<int>(cur < RG_OUT ? cur : RG_OUT));
}

}  // namespace

size_t refine_grid_scratch_bytes(int64_t rows) {
  return ((sizeof(RefineCtl) * rows + 255) & ~size_t(255)) + sizeof(unsigned long long) * RG_OUT * rows;
}

void* refine_grid_ctl(void* scratch) { return scratch; }

size_t refine_grid_ctl_bytes() { return sizeof(RefineCtl); }

int64_t refine_grid_max_k() { return RG_MAX_K; }

int64_t refine_grid_max_m() { return RG_MAX_M; }

cudaError_t launch_refine_grid(const RefineGridArgs& a, void* scratch, int64_t total_rows, cudaStream_t stream) {
  RefineCtl* ctl = static_cast<RefineCtl*>(scratch);
  unsigned long long* gather = reinterpret_cast<unsigned long long*>(
      static_cast<char*>(scratch) + ((sizeof(RefineCtl) * total_rows + 255) & ~size_t(255)));
  // Chunks per row: all CTAs (chunks x rows) resident at once, one per SM,
  // and no chunk shorter than 256 keys.
  int64_t G = sms() / (a.nrows > 0 ? a.nrows : 1);
  const int64_t by_len = (a.M + 255) / 256;
  if (G > by_len) G = by_len;
  // Two CTAs a row gain less than their two grid barriers cost: one CTA,
  // with no barrier (k_refine_grid<true>; 64 rows of 2^24, k = 32: the
  // refinement 22.6 -> 18.6 us).
  if (G <= 2) G = 1;
  // (The test setting of the waits keeps the barriers.)
  auto k = G == 1 && a.wait.skew == 0 ? k_refine_grid<true> : k_refine_grid<false>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(sizeof(unsigned long long) * RG_OUT));
  launch_kernel(k, dim3(static_cast<unsigned>(G), static_cast<unsigned>(a.nrows)), RG_THREADS,
                sizeof(unsigned long long) * RG_OUT, stream, a, ctl, gather);
  return cudaGetLastError();
}

}  // namespace profk
