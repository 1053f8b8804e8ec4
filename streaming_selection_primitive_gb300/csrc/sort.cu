// Descending sort and emission of a row's candidate keys when there are too
// many for one CTA (Prof-K step 4 on the filter buffer, and the last step of
// the exact and tie paths; "Prof-K: Probabilistic One-Pass Filtering for
// Efficient Top-k Selection", Section 3, stage 4).
//
// One persistent kernel per sort.  The keys of a row are cut into G
// contiguous chunks, one 1024-thread CTA per chunk; all CTAs of the launch are
// resident together (G x rows <= the SM count, one CTA per SM), so that they
// can meet at grid barriers (bounded waits on a per-row arrival counter).
//  1. Histograms of the eight byte positions of the keys, summed over the
//     chunks; every CTA then derives the same plan from them: a position
//     where every key has the same byte is skipped, and each byte value's
//     global start is the exclusive scan of its position's histogram.
//  2. Stable least-significant-digit radix passes (8-bit digits, on ~key, so
//     that ascending ~key is descending key) over the VALUE bytes only (the
//     upper 32 bits).  In a pass a CTA counts its chunk's digits and
//     publishes the counts at once, ranks its keys stably in shared memory
//     (a warp splits its keys by digit with nine ballots; per-warp counts are
//     scanned across warps), finds the counts of all earlier chunks by a
//     decoupled look-back over their published flags (32 chunks per step,
//     stopping at the nearest chunk whose inclusive prefix is known), and
//     writes the chunk out in digit order, so that the keys of one digit
//     leave as a contiguous run.  A chunk of more than 8192 keys is ranked
//     and written 8192 keys at a time.
//  3. The keys are now in value order, equal values in arbitrary order.  If
//     no run of equal values is longer than 256, each run is put in index
//     order: a warp places every key of a run at the run's start plus the
//     number of the run's larger keys; the first k positions are written as
//     (value, index).
//     Otherwise (heavy ties) the full sort runs: passes over all eight
//     positions, the last of which writes the output.  When the histograms
//     already prove a run longer than 256 (fewer than len / 256 distinct
//     values are possible), steps 2-3 are skipped and the full sort runs at
//     once.
//  B. For rows of at least 8192 keys, a bucket stage runs between steps 1
//     and 2 instead of the passes: the keys are counted into at most 2^14
//     buckets in key order, each digit of the highest varying byte split by
//     the bits below it into as many as its step-1 count calls for (about
//     len / 7500 keys a bucket), scattered once into bucket order, and then
//     sorted: when no bucket holds more than 256 keys, each bucket by one warp
//     in registers; otherwise range by
//     range: a range is a run of whole buckets of at most 8191 keys, sorted
//     completely (value and index) by one CTA in shared memory (runs of 256
//     keys sorted in registers by each warp, then merged pairwise), so ties
//     need no further work; ranges that start at or beyond position k are not
//     sorted.  Three grid barriers in all.  When some bucket holds more than
//     4096 keys (a few values repeated very often), every CTA sees it in the
//     same histogram and the row takes steps 2-3 instead.
// Output values are decoded from the key (it holds them exactly), except
// zero, whose sign the key does not keep: it is read from x.  Every wait is
// bounded; a wait that runs out sets an error bit in the row state.
#include <type_traits>

#include "blocksort.cuh"
#include "kernels.h"

namespace profk {

// Per-row sort control, in the scratch; zero before each sort.
struct SortCtl {
  unsigned long long start[8][256];  // digit counts of every position, over all chunks
  unsigned bar;                      // grid-barrier arrivals
  unsigned long_run;                 // 1: some run of equal values is longer than 32
  unsigned long long kmax;           // the largest key
  unsigned long long nkmax;          // the largest ~key (the smallest key, complemented)
  unsigned abort;                    // set by a CTA whose wait gave up
  unsigned pad[25];
};
static_assert(sizeof(SortCtl) % 16 == 0, "SortCtl is zeroed with 16-byte stores");

namespace {

constexpr int RS_THREADS = 1024;
constexpr int RS_KMAX = 8;                                       // keys per thread in one piece
constexpr int RS_SUB = RS_THREADS * RS_KMAX;                     // 8192 keys ranked at a time
constexpr size_t RS_SMEM = sizeof(unsigned long long) * RS_SUB;  // staging of a piece (64 KB)
constexpr int RUN_MAX = 256;   // runs up to this long are ordered by a warp
constexpr int HI_POS = 5;      // step 1 counts byte positions HI_POS..7 (the value's top three bytes)
constexpr int BK_BITS = 14;
constexpr int BK = 1 << BK_BITS;           // buckets of the bucket stage
constexpr unsigned BK_CAP = 4096;          // largest bucket the stage takes
constexpr int64_t BK_MIN_LEN = RS_SUB;     // rows of fewer keys take the passes
constexpr int64_t RANGE_MAX = RS_SUB;      // keys one CTA sorts in shared memory at once
// Dynamic shared memory: the staging area (a piece, a range) and, for the
// bucket stage, the buckets' starts and the merge buffer of a range.
constexpr size_t RS_SMEM_LAUNCH = 2 * RS_SMEM + sizeof(unsigned) * BK;
// Look-back flag: status (2 bits) | pass sequence number (4 bits) | count (58 bits).
constexpr unsigned long long FLAG_AGG = 1ull << 62;   // the chunk's own digit count
constexpr unsigned long long FLAG_INCL = 2ull << 62;  // count of this and every earlier chunk
constexpr int FLAG_SEQ_SHIFT = 58;
constexpr unsigned long long FLAG_COUNT = (1ull << FLAG_SEQ_SHIFT) - 1;

__device__ __forceinline__ unsigned digit_of(unsigned long long key, int pos) {
  return static_cast<unsigned>((~key) >> (8 * pos)) & 255u;
}

__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ bool flag_ready(unsigned long long f, int seq) {
  return (f >> 62) != 0 && ((f >> FLAG_SEQ_SHIFT) & 15ull) == static_cast<unsigned long long>(seq);
}

// Lanes of the warp whose digit equals this lane's (9-bit digits; 256 marks
// a lane without a key): one ballot per bit.
__device__ __forceinline__ unsigned same_digit_lanes(unsigned d) {
  unsigned peers = FULL_MASK;
#pragma unroll
  for (int b = 0; b < 9; ++b) {
    const bool bit = (d >> b) & 1u;
    const unsigned m = __ballot_sync(FULL_MASK, bit);
    peers &= bit ? m : ~m;
  }
  return peers;
}

// Keys a row sorts, or -1 when the row is left alone.
__device__ __forceinline__ int64_t row_count(const RadixSortArgs& a, int row) {
  if (a.mode == SortCount::FromState) {
    // The refinement of the filter buffer: rows that fail the check, or whose
    // earlier steps reported an error, are left alone.
    const unsigned long long R = a.st[row].R_ge;
    const bool ok = static_cast<unsigned long long>(a.k) <= R && R <= static_cast<unsigned long long>(a.key_stride) &&
                    __ldcg(&a.st[row].error) == 0u;
    return ok ? static_cast<int64_t>(R) : -1;
  }
  if (a.mode == SortCount::KUnlessSkip && a.st[row].skip) return -1;
  return a.k;
}

// Writes output position pos of a row from its key.  The index is checked
// against the row length, so that a sort that went wrong never reads outside
// x: such an entry is (NaN, -1).
__device__ __forceinline__ void emit_key(const RadixSortArgs& a, int row, int64_t pos, unsigned long long kk) {
  const uint32_t idx = cand_index(kk);
  const uint32_t vk = static_cast<uint32_t>(kk >> 32);
  const int64_t o = static_cast<int64_t>(row) * a.k + pos;
  if (static_cast<int64_t>(idx) < a.n) {
    a.out_idx[o] = static_cast<int64_t>(idx);
    a.out_vals[o] = vk == ord_key(0.0f) ? a.x[static_cast<int64_t>(row) * a.ld + idx] : key_to_float(vk);
  } else {
    a.out_idx[o] = -1;
    a.out_vals[o] = __int_as_float(0x7fc00000);
  }
}

struct Smem {
  unsigned long long start[8][256];  // global start of each digit of each position
  unsigned long long cur[256];       // where the chunk's next key of each digit goes
  long long base[256];
  unsigned hist[256], tot[256], texcl[256], wsum[8];
  int trivial[8];
  unsigned distinct[8];  // byte values present at each position
  unsigned nruns;  // runs of 2 .. RUN_MAX keys starting in this chunk
  int err;
  int limit;          // bound on one wait
  long long row_len;  // keys of the row, or -1: the row is skipped
  unsigned long long blo[256];  // bucket stage, per digit of the top position: the lowest bits below it,
  unsigned boff[256];           // the digit's first bucket,
  unsigned char bbits[256];     // log2 of its buckets
  unsigned char bsh[256];       // and the shift of (low bits - blo) that gives the bucket
  unsigned long long kmax, nkmax;
  unsigned nbuckets;
  unsigned bwsum[32];         // bucket stage: per-warp sums of the starts' scan
  unsigned bmax[32];          // and per-warp largest buckets
  long long rlo, rhi;         // the range a CTA sorts next
};

// Every CTA of the row arrives (a release: the CTA's writes, ordered before
// it by the block barrier, become visible with it), then waits until all
// have (target arrivals; acquire loads of the arrival count).
// A wait that ends without them (bounded, see wait_count) sets sm.err, which
// every thread reads afterwards.
__device__ __forceinline__ void grid_sync(SortCtl& c, unsigned target, Smem& sm) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&c.bar) : "memory");
    if (!wait_count(&c.bar, target, &c.abort, sm.limit)) sm.err = 1;
  }
  __syncthreads();
}

// A piece of cnt keys at `base`: warp w holds positions [w span, (w + 1)
// span), span = 32 kp; round r, lane l holds w span + 32 r + l, so (warp,
// round, lane) order is input order.
__device__ __forceinline__ bool in_piece(int r, int kp, int cnt) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  return r < kp && warp * 32 * kp + r * 32 + lane < cnt;
}

__device__ __forceinline__ void load_piece(const unsigned long long* in, int64_t base, int cnt, int kp,
                                           unsigned long long (&key)[RS_KMAX]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int r = 0; r < RS_KMAX; ++r)
    key[r] = in_piece(r, kp, cnt) ? __ldcg(in + base + warp * 32 * kp + r * 32 + lane) : 0ull;
}

// One stable pass over byte position `pos` of the chunk [lo, hi) (chunk
// number `chunk`, sequence number `seq` for the flags): in -> out, or to the
// output when `emit`.
__device__ __forceinline__ void radix_pass(const RadixSortArgs& a, int row, int64_t chunk, int64_t lo, int64_t hi,
                                           int pos, int seq, bool emit, const unsigned long long* in,
                                           unsigned long long* out, unsigned long long* fr, Smem& sm,
                                           unsigned long long* s_keys, SortCtl& c) {
  unsigned short(*cntw)[256] = reinterpret_cast<unsigned short(*)[256]>(s_keys);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const unsigned long long tag = static_cast<unsigned long long>(seq) << FLAG_SEQ_SHIFT;
  if (threadIdx.x < 256) {
    sm.hist[threadIdx.x] = 0;
    sm.cur[threadIdx.x] = sm.start[pos][threadIdx.x];
  }
  __syncthreads();
  if (lo >= hi) return;  // an empty chunk: the last ones, on which no chunk waits
  const int nsub = static_cast<int>((hi - lo + RS_SUB - 1) / RS_SUB);

  // Count the chunk's digits and publish the counts (chunk 0's are already
  // inclusive).  The first piece stays in registers for the ranking.
  unsigned long long key[RS_KMAX];
  int cnt = static_cast<int>(hi - lo < RS_SUB ? hi - lo : RS_SUB);
  int kp = (cnt + RS_THREADS - 1) / RS_THREADS;
  load_piece(in, lo, cnt, kp, key);
#pragma unroll
  for (int r = 0; r < RS_KMAX; ++r)
    if (r < kp) hist_add(sm.hist, digit_of(key[r], pos), in_piece(r, kp, cnt));
  for (int s = 1; s < nsub; ++s) {
    const int64_t b = lo + static_cast<int64_t>(s) * RS_SUB;
    const int sc = static_cast<int>(hi - b < RS_SUB ? hi - b : RS_SUB);
    for (int i = threadIdx.x; i < ((sc + 31) & ~31); i += RS_THREADS) {
      const bool v = i < sc;
      hist_add(sm.hist, v ? digit_of(__ldcg(in + b + i), pos) : 0u, v);
    }
  }
  __syncthreads();
  if (threadIdx.x < 256)
    st_relaxed(fr + chunk * 256 + threadIdx.x, (chunk == 0 ? FLAG_INCL : FLAG_AGG) | tag | sm.hist[threadIdx.x]);

  for (int s = 0; s < nsub; ++s) {
    const int64_t base = lo + static_cast<int64_t>(s) * RS_SUB;
    if (s > 0) {
      cnt = static_cast<int>(hi - base < RS_SUB ? hi - base : RS_SUB);
      kp = (cnt + RS_THREADS - 1) / RS_THREADS;
      load_piece(in, base, cnt, kp, key);
    }
    // Rank among the warp's keys of the same digit, in position order.
    for (int d = lane; d < 256; d += 32) cntw[warp][d] = 0;
    __syncwarp();
    unsigned info[RS_KMAX];  // digit (9 bits) | rank among the warp's keys of that digit << 9
#pragma unroll
    for (int r = 0; r < RS_KMAX; ++r) {
      info[r] = 256u;
      if (r < kp) {
        const bool valid = in_piece(r, kp, cnt);
        const unsigned d = valid ? digit_of(key[r], pos) : 256u;
        const unsigned peers = same_digit_lanes(d);
        const unsigned prior = valid ? cntw[warp][d] : 0u;
        __syncwarp();
        if (valid && (peers & lt) == 0) cntw[warp][d] = static_cast<unsigned short>(prior + __popc(peers));
        __syncwarp();
        info[r] = d | ((prior + __popc(peers & lt)) << 9);
      }
    }
    __syncthreads();
    // Per digit, the exclusive scan of the 32 warp counts: four threads per
    // digit, eight warps each, combined by shuffles among the four.
    {
      const int d = threadIdx.x >> 2, q = threadIdx.x & 3;
      unsigned v[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[i] = cntw[8 * q + i][d];
        sum += v[i];
      }
      unsigned incl = sum;
      unsigned t = __shfl_up_sync(FULL_MASK, incl, 1, 4);
      if (q >= 1) incl += t;
      t = __shfl_up_sync(FULL_MASK, incl, 2, 4);
      if (q >= 2) incl += t;
      const unsigned total = __shfl_sync(FULL_MASK, incl, 3, 4);
      unsigned run = incl - sum;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cntw[8 * q + i][d] = static_cast<unsigned short>(run);
        run += v[i];
      }
      if (q == 0) sm.tot[d] = total;
    }
    __syncthreads();
    // Piece-local start of each digit (exclusive scan of tot over digits).
    if (threadIdx.x < 256) {
      const unsigned v = sm.tot[threadIdx.x];
      unsigned incl = v;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) sm.wsum[warp] = incl;
      sm.texcl[threadIdx.x] = incl - v;
    }
    __syncthreads();
    if (threadIdx.x < 256) {
      unsigned add = 0;
      for (int w = 0; w < warp; ++w) add += sm.wsum[w];
      sm.texcl[threadIdx.x] += add;
    }
    __syncthreads();
    // Piece-local positions; then the piece in digit order in shared memory
    // (the counts are dead once every thread holds its positions).
#pragma unroll
    for (int r = 0; r < RS_KMAX; ++r) {
      const unsigned d = info[r] & 511u;
      info[r] = d < 256 ? sm.texcl[d] + cntw[warp][d] + (info[r] >> 9) : ~0u;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RS_KMAX; ++r)
      if (info[r] != ~0u) s_keys[info[r]] = key[r];

    if (s == 0 && chunk > 0) {
      // Look-back: four threads per digit, each reading the flags of 8
      // earlier chunks (32 per step for the four), nearest first; the loads
      // are issued together and a flag not yet published is polled.
      // Positions before the first chunk read as an empty inclusive prefix.
      const int d = threadIdx.x >> 2, q = threadIdx.x & 3;
      const unsigned gmask = 0xFu << (lane & ~3);
      unsigned long long excl = 0;
      bool timed_out = false;
      for (int64_t j = chunk - 1; j >= 0; j -= 32) {
        unsigned long long f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int64_t tt = j - 8 * q - i;
          f[i] = tt >= 0 ? ld_relaxed(fr + tt * 256 + d) : (FLAG_INCL | tag);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          for (int poll = 0; !flag_ready(f[i], seq); ++poll) {
            if (wait_should_stop(poll, sm.limit, &c.abort)) {
              timed_out = true;
              f[i] = FLAG_INCL | tag;  // give up here: adds nothing, ends the walk
              break;
            }
            f[i] = ld_relaxed(fr + (j - 8 * q - i) * 256 + d);
          }
        }
        unsigned long long part = 0;
        bool found = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (!found) {
            part += f[i] & FLAG_COUNT;
            found = (f[i] >> 62) == 2;
          }
        }
        // The nearest thread (lowest q) that met an inclusive prefix ends
        // the walk; its part and the nearer ones are added.
        const unsigned fb = (__ballot_sync(gmask, found) >> (lane & ~3)) & 0xFu;
        const int stop = fb ? __ffs(fb) - 1 : 4;
        unsigned long long mine = q <= stop ? part : 0ull;
        mine += __shfl_xor_sync(gmask, mine, 1, 4);
        mine += __shfl_xor_sync(gmask, mine, 2, 4);
        excl += mine;
        if (fb) break;
      }
      // A group whose walk gave up publishes nothing: later chunks then walk
      // past this chunk's own count, and this CTA leaves below.
      const bool gave_up = ((__ballot_sync(gmask, timed_out) >> (lane & ~3)) & 0xFu) != 0u;
      if (gave_up) sm.err = 1;
      if (q == 0 && !gave_up) {
        st_relaxed(fr + chunk * 256 + d, FLAG_INCL | tag | ((excl + sm.hist[d]) & FLAG_COUNT));
        sm.cur[d] += excl;
      }
    }
    __syncthreads();
    if (sm.err) return;  // block-uniform: read after the block barrier
    if (threadIdx.x < 256)
      sm.base[threadIdx.x] = static_cast<long long>(sm.cur[threadIdx.x]) - static_cast<long long>(sm.texcl[threadIdx.x]);
    __syncthreads();

    // Position i of the digit-ordered piece goes to base[digit] + i.
    for (int i = threadIdx.x; i < cnt; i += RS_THREADS) {
      const unsigned long long kk = s_keys[i];
      const int64_t p = sm.base[digit_of(kk, pos)] + i;
      if (!emit) {
        out[p] = kk;
      } else if (p < a.k) {
        emit_key(a, row, p, kk);
      }
    }
    __syncthreads();  // the next piece reuses shared memory
    if (threadIdx.x < 256) sm.cur[threadIdx.x] += sm.tot[threadIdx.x];
  }
}

// The plan of byte positions [plo, phi), the same in every CTA: the row's
// digit counts of each position (c.start, complete) into the start of each
// digit (an exclusive scan), whether the position is the same in every key
// (trivial), and how many digits occur (distinct).
__device__ __forceinline__ void plan_positions(SortCtl& c, Smem& sm, int64_t len, int plo, int phi) {
  for (int i = plo * 256 + threadIdx.x; i < phi * 256; i += RS_THREADS) {
    const unsigned long long v = __ldcg(&c.start[0][0] + i);
    (&sm.start[0][0])[i] = v;
    if (static_cast<int64_t>(v) == len) sm.trivial[i >> 8] = 1;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pos = plo + warp;
  if (pos < phi) {  // exclusive scan of position `pos`, 8 digits per lane
    unsigned long long v[8], s = 0;
    unsigned present = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = sm.start[pos][lane * 8 + j];
      s += v[j];
      present += v[j] != 0;
    }
    for (int o = 16; o >= 1; o >>= 1) present += __shfl_xor_sync(FULL_MASK, present, o);
    if (lane == 0) sm.distinct[pos] = present;
    unsigned long long incl = s;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += t;
    }
    unsigned long long run = incl - s;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sm.start[pos][lane * 8 + j] = run;
      run += v[j];
    }
  }
  __syncthreads();
}

// First position of the bucket starts st[0..BK) (nondecreasing) at or after
// pos: the start of the first bucket beginning there, or len.
__device__ __forceinline__ int64_t bucket_at(const unsigned* st, int64_t pos, int64_t len) {
  int lo = 0, hi = BK;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(st[mid]) >= pos)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo < BK ? static_cast<int64_t>(st[lo]) : len;
}

// The bucket stage (B in the header).  Returns true when it sorted and
// emitted the row, false (in every CTA alike, after one grid barrier) when a
// bucket is too large; the row's keys are then untouched.
__device__ bool bucket_stage(const RadixSortArgs& a, int row, int64_t len, int64_t lo, int64_t hi, SortCtl& c,
                             unsigned& target, unsigned* bkr, unsigned long long* tmp_row, Smem& sm,
                             unsigned long long* s_keys) {
  const unsigned long long* keys = a.keys + row * a.key_stride;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned G = gridDim.x;
  // Buckets in key order, sized from the data: the bytes above ps, the
  // highest position with more than one digit, are the same in every key;
  // each digit d of position ps gets 2^b(d) buckets, equal parts of the range
  // of the bits below it that its keys can take, with b(d) the least for
  // which its c(d) keys average at most
  // ceil(len / 7500) per bucket (2^b(d) < 2 c(d) / that + 1, so fewer than
  // 15,256 in all).
  int ps = -1;
  for (int p = 7; p >= 0 && ps < 0; --p)
    if (!sm.trivial[p]) ps = p;
  if (ps < 0) ps = 0;  // a single key
  const int pb = 8 * ps;
  const unsigned long long lowmask = (1ull << pb) - 1ull;  // pb <= 56
  if (warp == 0) {
    const int64_t target = (len + 7499) / 7500;  // >= len / 7500, so the buckets number < 15,000 + 256
    // The first and last digits hold keys only from the largest (smallest)
    // key on: their buckets split that part of the digit, not all of it.
    const unsigned long long nkmin = ~sm.kmax, nkmaxv = sm.nkmax;
    const unsigned dfirst = static_cast<unsigned>(nkmin >> pb) & 255u, dlast = static_cast<unsigned>(nkmaxv >> pb) & 255u;
    unsigned nb[8], tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int d = lane * 8 + j;
      const int64_t c = static_cast<int64_t>((d < 255 ? sm.start[ps][d + 1] : static_cast<unsigned long long>(len)) -
                                             sm.start[ps][d]);
      const unsigned long long blo = d == static_cast<int>(dfirst) ? (nkmin & lowmask) : 0ull;
      const unsigned long long bhi = d == static_cast<int>(dlast) ? (nkmaxv & lowmask) : lowmask;
      const unsigned long long span = bhi >= blo ? bhi - blo : 0ull;
      const int wbits = span ? 64 - __clzll(span) : 0;  // (low - blo) < 2^wbits
      int b = 0;
      while (b < BK_BITS && b < wbits && (static_cast<int64_t>(1) << b) * target < c) ++b;
      sm.bbits[d] = static_cast<unsigned char>(b);
      sm.bsh[d] = static_cast<unsigned char>(wbits - b);
      sm.blo[d] = blo;
      nb[j] = 1u << b;
      tot += nb[j];
    }
    unsigned incl = tot;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += t;
    }
    unsigned run = incl - tot;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sm.boff[lane * 8 + j] = run;
      run += nb[j];
    }
    if (lane == 31) sm.nbuckets = incl;
  }
  __syncthreads();
  if (sm.nbuckets > static_cast<unsigned>(BK)) return false;  // (not reached, see above)
  auto bucket_of = [&](unsigned long long kk) {
    const unsigned long long nk = ~kk;
    const unsigned d = static_cast<unsigned>(nk >> pb) & 255u;
    return sm.boff[d] + (sm.bbits[d] ? static_cast<unsigned>(((nk & lowmask) - sm.blo[d]) >> sm.bsh[d]) : 0u);
  };
  unsigned* h = reinterpret_cast<unsigned*>(s_keys);            // the chunk's counts, then its cursors
  unsigned* st = reinterpret_cast<unsigned*>(s_keys + RS_SUB);  // every bucket's start in the row
  // The chunk's keys: in shared memory when step 1 kept them there.
  const unsigned long long* cst = s_keys + 2 * RS_SUB;
  const bool staged = hi - lo <= RS_SUB;
  auto key_at = [&](int64_t i) { return staged ? cst[i - lo] : __ldcg(keys + i); };
  // The chunk in pieces of RS_SUB keys, RS_KMAX per thread loaded together
  // (their L2 round trips overlap), then handled.
  auto each_piece = [&](auto&& fn) {
    for (int64_t b0 = lo; b0 < hi; b0 += RS_SUB) {
      unsigned long long kv[RS_KMAX];
#pragma unroll
      for (int r = 0; r < RS_KMAX; ++r) {
        const int64_t i = b0 + r * RS_THREADS + threadIdx.x;
        kv[r] = i < hi ? key_at(i) : 0ull;
      }
      fn(kv, b0);
    }
  };
  for (int i = threadIdx.x; i < BK; i += RS_THREADS) h[i] = 0;
  __syncthreads();
  each_piece([&](const unsigned long long(&kv)[RS_KMAX], int64_t b0) {
#pragma unroll
    for (int r = 0; r < RS_KMAX; ++r)
      if (b0 + r * RS_THREADS + threadIdx.x < hi) atomicAdd(&h[bucket_of(kv[r])], 1u);
  });
  __syncthreads();
  for (int i = threadIdx.x; i < BK; i += RS_THREADS)
    if (h[i]) atomicAdd(&bkr[i], h[i]);
  grid_sync(c, target += G, sm);
  if (sm.err) return true;  // the wait gave up: the caller reports it and leaves

  // Starts: the exclusive scan of the row's counts.  The counts come into
  // shared memory with coalesced loads; each thread then scans 16 consecutive
  // ones (four 16-byte reads).
  constexpr int PER = BK / RS_THREADS;
  {
    unsigned cv[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) cv[j] = __ldcg(bkr + j * RS_THREADS + threadIdx.x);
#pragma unroll
    for (int j = 0; j < PER; ++j) st[j * RS_THREADS + threadIdx.x] = cv[j];
  }
  __syncthreads();
  unsigned v[PER], sum = 0, mx = 0;
  {
    const uint4* s4 = reinterpret_cast<const uint4*>(st + threadIdx.x * PER);
#pragma unroll
    for (int q = 0; q < PER / 4; ++q) {
      const uint4 u = s4[q];
      v[4 * q] = u.x;
      v[4 * q + 1] = u.y;
      v[4 * q + 2] = u.z;
      v[4 * q + 3] = u.w;
    }
  }
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    sum += v[j];
    mx = v[j] > mx ? v[j] : mx;
  }
  unsigned incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += t;
    mx = max(mx, __shfl_xor_sync(FULL_MASK, mx, o));
  }
  if (lane == 31) sm.bwsum[warp] = incl;
  if (lane == 0) sm.bmax[warp] = mx;
  __syncthreads();
  unsigned run = incl - sum;
  for (int w = 0; w < warp; ++w) run += sm.bwsum[w];
  {
    uint4* s4 = reinterpret_cast<uint4*>(st + threadIdx.x * PER);
#pragma unroll
    for (int q = 0; q < PER / 4; ++q) {
      uint4 u;
      u.x = run;
      run += v[4 * q];
      u.y = run;
      run += v[4 * q + 1];
      u.z = run;
      run += v[4 * q + 2];
      u.w = run;
      run += v[4 * q + 3];
      s4[q] = u;
    }
  }
  unsigned maxb = 0;
  for (int w = 0; w < RS_THREADS / 32; ++w) maxb = sm.bmax[w] > maxb ? sm.bmax[w] : maxb;
  __syncthreads();
  if (maxb > BK_CAP) return false;

  // Scatter: the chunk reserves its slots of each bucket at once (the
  // reservations of a thread are issued together); its keys then take
  // consecutive slots (in any order: each bucket is sorted whole).
  unsigned* gcur = bkr + BK;
  {
    unsigned res[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = j * RS_THREADS + threadIdx.x;
      res[j] = h[i] ? atomicAdd(&gcur[i], h[i]) : 0u;
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = j * RS_THREADS + threadIdx.x;
      if (h[i]) h[i] = st[i] + res[j];
    }
  }
  __syncthreads();
  each_piece([&](const unsigned long long(&kv)[RS_KMAX], int64_t b0) {
    unsigned slot[RS_KMAX];
#pragma unroll
    for (int r = 0; r < RS_KMAX; ++r)
      if (b0 + r * RS_THREADS + threadIdx.x < hi) slot[r] = atomicAdd(&h[bucket_of(kv[r])], 1u);
#pragma unroll
    for (int r = 0; r < RS_KMAX; ++r)
      if (b0 + r * RS_THREADS + threadIdx.x < hi) tmp_row[slot[r]] = kv[r];
  });
  grid_sync(c, target += G, sm);
  if (sm.err) return true;

  if (maxb <= 256) {
    // Small buckets: each is sorted by one warp in registers (the smallest
    // network of 32, 64, 128 or 256 keys that holds it), bucket b by the
    // grid's warp b mod (32 G); buckets that start at or beyond k are skipped.
    const unsigned nbk = sm.nbuckets;
    for (unsigned b = blockIdx.x * (RS_THREADS / 32) + warp; b < nbk; b += G * (RS_THREADS / 32)) {
      const int64_t bs = st[b], be = b + 1 < nbk ? static_cast<int64_t>(st[b + 1]) : len;
      if (bs >= be || bs >= a.k) continue;
      const int sz = static_cast<int>(be - bs);
      auto sort_emit = [&](auto tagE) {
        constexpr int E = decltype(tagE)::value;
        unsigned long long kv[E];  // key lane * E + r of the bucket in kv[r]
#pragma unroll
        for (int r = 0; r < E; ++r) kv[r] = lane * E + r < sz ? __ldcg(tmp_row + bs + lane * E + r) : 0ull;
        warp_sort_desc<E>(kv);
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const int q = lane * E + r;
          if (q < sz && bs + q < a.k) emit_key(a, row, bs + q, kv[r]);
        }
      };
      if (sz <= 32)
        sort_emit(std::integral_constant<int, 1>{});
      else if (sz <= 64)
        sort_emit(std::integral_constant<int, 2>{});
      else if (sz <= 128)
        sort_emit(std::integral_constant<int, 4>{});
      else
        sort_emit(std::integral_constant<int, 8>{});
    }
    return true;
  }

  // Ranges: positions [r T, (r + 1) T) widened to whole buckets (fewer than
  // T + maxb <= RANGE_MAX keys), taken by the CTAs in turn.
  const int64_t room = RANGE_MAX - 1 - static_cast<int64_t>(maxb);
  const int64_t m = (len + static_cast<int64_t>(G) * room - 1) / (static_cast<int64_t>(G) * room);
  const int64_t T = (len + static_cast<int64_t>(G) * m - 1) / (static_cast<int64_t>(G) * m);
  const int64_t nr = (len + T - 1) / T;
  for (int64_t r = blockIdx.x; r < nr; r += G) {
    if (threadIdx.x == 0) {
      const int64_t plo = r * T, phi = plo + T < len ? plo + T : len;
      sm.rlo = bucket_at(st, plo, len);
      sm.rhi = bucket_at(st, phi, len);
    }
    __syncthreads();
    const int64_t rs = sm.rlo, re = sm.rhi;
    __syncthreads();
    if (rs >= re || rs >= a.k) continue;
    const int L = static_cast<int>(re - rs);
    const int P = (L + 255) & ~255;  // zero keys pad the last run and sort last
    unsigned long long* mbuf = s_keys + 2 * RS_SUB;
    {
      unsigned long long kv[RS_KMAX];  // P <= RS_SUB: at most RS_KMAX per thread, loaded together
#pragma unroll
      for (int r = 0; r < RS_KMAX; ++r) {
        const int i = r * RS_THREADS + threadIdx.x;
        kv[r] = i < L ? __ldcg(tmp_row + rs + i) : 0ull;
      }
#pragma unroll
      for (int r = 0; r < RS_KMAX; ++r) {
        const int i = r * RS_THREADS + threadIdx.x;
        if (i < P) s_keys[mswz(i)] = kv[r];
      }
    }
    __syncthreads();
    const unsigned long long* srt = block_merge_sort_desc(s_keys, mbuf, P);
    for (int i = threadIdx.x; i < L; i += RS_THREADS)
      if (rs + i < a.k) emit_key(a, row, rs + i, srt[mswz(i)]);
    __syncthreads();
  }
  return true;
}

__global__ void __launch_bounds__(RS_THREADS, 1) k_rs_sort(RadixSortArgs a, SortCtl* ctl, unsigned long long* tmp,
                                                          unsigned long long* flags, int64_t flag_stride,
                                                          unsigned* bk) {
  // No early trigger: the next kernels of the stream launch when this one has
  // finished.  Triggered at the start, they took SMs as this kernel's CTAs
  // left them, and with calls in flight back to back that cost about 80 us
  // per call at k = 2^17 .. 2^19 (measured); the kernel after a sort is the
  // small report, so nothing is lost by waiting.
  pdl_wait();
  // 64 KB: a piece, its per-warp counts, or histograms; then 64 KB of bucket
  // starts and a 64 KB merge buffer (the bucket stage).
  extern __shared__ unsigned long long s_keys[];
  __shared__ Smem sm;
  const int row = launch_row(a.rows);
  if (threadIdx.x == 0) {
    // One thread decides for the block.  The refinement of the filter buffer
    // leaves alone a row that an earlier attempt settled, and its first CTA
    // records the check's outcome (settle_row).
    if (a.mode == SortCount::FromState && settled_before(a.st[row], a.attempt)) {
      sm.row_len = -1;
    } else {
      sm.row_len = row_count(a, row);
      if (a.mode == SortCount::FromState && blockIdx.x == 0)
        settle_row(a.st[row], a.attempt, static_cast<unsigned long long>(a.k),
                   static_cast<unsigned long long>(a.key_stride), a.tie_exit);
    }
    sm.err = 0;
    sm.limit = wait_limit(a.wait);
  }
  __syncthreads();
  const int64_t len = sm.row_len;
  if (len < 0) return;  // every CTA of the row leaves: no barrier is met
  SortCtl& c = ctl[row];
  unsigned long long* fr = flags + row * flag_stride;
  const int64_t G = gridDim.x, chunk = blockIdx.x;
  const int64_t C = (((len + G - 1) / G) + 31) & ~int64_t(31);
  const int64_t lo = chunk * C < len ? chunk * C : len;
  const int64_t hi = lo + C < len ? lo + C : len;
  unsigned target = 0;
// After a wait that gave up, the CTA reports it and leaves without writing
// anything else (sm.err is block-uniform where this is used).
#define RS_LEAVE_IF_GAVE_UP()                                           \
  if (sm.err) {                                                         \
    if (threadIdx.x == 0 && a.st) atomicOr(&a.st[row].error, ERR_WAIT); \
    return;                                                             \
  }

  unsigned* bkr = bk + static_cast<int64_t>(row) * 2 * BK;  // bucket counts, then cursors

  // 1. Histograms of the value positions HI_POS..7 (and this chunk's flags
  // and share of the bucket counters zeroed).  The other positions are
  // counted later, only when the bucket stage cannot take the row (all keys
  // share the top HI_POS bytes' values, or a bucket is too large): their
  // digits are mostly the index bits, whose 256 bins are all populated in
  // every chunk, and their global atomics cost more than the rest of step 1.
  {
    unsigned(*h)[256] = reinterpret_cast<unsigned(*)[256]>(s_keys);
    for (int i = threadIdx.x; i < 8 * 256; i += RS_THREADS) (&h[0][0])[i] = 0;
    if (threadIdx.x < 256) fr[chunk * 256 + threadIdx.x] = 0;
    for (int64_t i = chunk * RS_THREADS + threadIdx.x; i < 2 * BK; i += G * RS_THREADS) bkr[i] = 0;
    if (threadIdx.x == 0) sm.kmax = sm.nkmax = 0;
    __syncthreads();
    unsigned long long kmx = 0, nkmx = 0;
    // Pieces of RS_SUB keys, RS_KMAX loads per thread issued together; a
    // chunk of at most RS_SUB keys is also kept in shared memory (the merge
    // buffer's place) for the bucket stage.
    unsigned long long* cst = s_keys + 2 * RS_SUB;
    for (int64_t b0 = lo; b0 < hi; b0 += RS_SUB) {
      const int cnt = static_cast<int>(hi - b0 < RS_SUB ? hi - b0 : RS_SUB);
      unsigned long long kv[RS_KMAX];
#pragma unroll
      for (int r = 0; r < RS_KMAX; ++r) {
        const int j = r * RS_THREADS + threadIdx.x;
        kv[r] = j < cnt ? __ldcg(a.keys + row * a.key_stride + b0 + j) : 0ull;
      }
#pragma unroll
      for (int r = 0; r < RS_KMAX; ++r) {
        const int j = r * RS_THREADS + threadIdx.x;
        if (r * RS_THREADS >= cnt) break;  // uniform across the block
        const bool valid = j < cnt;
#pragma unroll
        for (int p = HI_POS; p < 8; ++p) hist_add(h[p], digit_of(kv[r], p), valid);
        if (valid) {
          kmx = kv[r] > kmx ? kv[r] : kmx;
          nkmx = ~kv[r] > nkmx ? ~kv[r] : nkmx;
          if (hi - lo <= RS_SUB) cst[j] = kv[r];
        }
      }
    }
    // The chunk's largest key and largest ~key, then the row's (one atomic each).
    for (int o = 16; o >= 1; o >>= 1) {
      const unsigned long long t1 = __shfl_xor_sync(FULL_MASK, kmx, o), t2 = __shfl_xor_sync(FULL_MASK, nkmx, o);
      kmx = t1 > kmx ? t1 : kmx;
      nkmx = t2 > nkmx ? t2 : nkmx;
    }
    if ((threadIdx.x & 31) == 0 && kmx) {
      atomicMax(&sm.kmax, kmx);
      atomicMax(&sm.nkmax, nkmx);
    }
    __syncthreads();
    if (threadIdx.x == 0 && sm.kmax) {
      atomicMax(&c.kmax, sm.kmax);
      atomicMax(&c.nkmax, sm.nkmax);
    }
    for (int i = HI_POS * 256 + threadIdx.x; i < 8 * 256; i += RS_THREADS)
      if ((&h[0][0])[i]) atomicAdd(&c.start[0][0] + i, static_cast<unsigned long long>((&h[0][0])[i]));
  }
  grid_sync(c, (target += G) + a.wait.skew, sm);
  RS_LEAVE_IF_GAVE_UP();
  // The plan, the same in every CTA.
  if (threadIdx.x < 8) sm.trivial[threadIdx.x] = 0;  // unknown positions count as varying
  if (threadIdx.x == 0) {
    sm.kmax = __ldcg(&c.kmax);
    sm.nkmax = __ldcg(&c.nkmax);
  }
  __syncthreads();
  plan_positions(c, sm, len, HI_POS, 8);
  // Positions 0 .. HI_POS-1 counted (a pass over the chunk, its atomics and
  // one more barrier) and planned: for the bucket stage when the keys share
  // the values of the top positions, and for the passes.
  bool low_planned = false;
  auto plan_low = [&]() {
    unsigned(*h)[256] = reinterpret_cast<unsigned(*)[256]>(s_keys);
    for (int i = threadIdx.x; i < HI_POS * 256; i += RS_THREADS) (&h[0][0])[i] = 0;
    __syncthreads();
    const unsigned long long* cst = s_keys + 2 * RS_SUB;  // the chunk, when step 1 kept it
    const bool staged = hi - lo <= RS_SUB;
    for (int64_t b0 = lo; b0 < hi; b0 += RS_THREADS) {
      const int64_t i = b0 + threadIdx.x;
      const bool valid = i < hi;
      const unsigned long long kk = valid ? (staged ? cst[i - lo] : __ldcg(a.keys + row * a.key_stride + i)) : 0ull;
#pragma unroll
      for (int q = 0; q < HI_POS; ++q) hist_add(h[q], digit_of(kk, q), valid);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < HI_POS * 256; i += RS_THREADS)
      if ((&h[0][0])[i]) atomicAdd(&c.start[0][0] + i, static_cast<unsigned long long>((&h[0][0])[i]));
    grid_sync(c, target += G, sm);
    if (!sm.err) plan_positions(c, sm, len, 0, HI_POS);
    low_planned = true;
  };
  bool top_varies = false;
  for (int q = HI_POS; q < 8; ++q) top_varies |= !sm.trivial[q];
  if (!top_varies) {
    plan_low();
    RS_LEAVE_IF_GAVE_UP();
  }

  if (len >= BK_MIN_LEN && len < (int64_t(1) << 31) &&
      bucket_stage(a, row, len, lo, hi, c, target, bkr, tmp + row * a.key_stride, sm, s_keys)) {
    __syncthreads();
    RS_LEAVE_IF_GAVE_UP();
    return;
  }
  if (!low_planned) {
    plan_low();
    RS_LEAVE_IF_GAVE_UP();
  }

  // When the value bytes allow fewer than len / RUN_MAX distinct values,
  // some value repeats more than RUN_MAX times: the full sort is certain to
  // be needed and the value passes would be wasted.
  unsigned long long distinct_max = 1;
  for (int p = 4; p < 8; ++p) distinct_max *= sm.distinct[p];
  // (Step 3 keeps the chunk, RUN_MAX keys on each side of it and the list of
  // its runs, at most C / 2, in the staging area: 8 (C + 2 RUN_MAX) + 2 C
  // bytes; longer chunks take the full sort too.)
  bool full = len > RUN_MAX * static_cast<int64_t>(distinct_max) ||
              10 * C + 16 * RUN_MAX > static_cast<int64_t>(RS_SMEM);
  int seq = 0, cur = 0;
  if (!full) {
    // 2. Value positions.
    for (int p = 4; p < 8; ++p) {
      if (sm.trivial[p]) continue;
      radix_pass(a, row, chunk, lo, hi, p, seq, false, (cur ? tmp : a.keys) + row * a.key_stride,
                 (cur ? a.keys : tmp) + row * a.key_stride, fr, sm, s_keys, c);
      RS_LEAVE_IF_GAVE_UP();
      ++seq;
      cur ^= 1;
      grid_sync(c, target += G, sm);
      RS_LEAVE_IF_GAVE_UP();
    }
    // 3. Runs of equal values: a run longer than RUN_MAX has equal values
    // RUN_MAX positions apart.
    const unsigned long long* srt = (cur ? tmp : a.keys) + row * a.key_stride;
    for (int64_t i = lo + threadIdx.x; i < hi; i += RS_THREADS)
      if (i + RUN_MAX < len && (__ldcg(srt + i) >> 32) == (__ldcg(srt + i + RUN_MAX) >> 32)) c.long_run = 1u;
    grid_sync(c, target += G, sm);
    RS_LEAVE_IF_GAVE_UP();
    full = __ldcg(&c.long_run) != 0;
    if (!full) {
      // The chunk and RUN_MAX keys on each side go to shared memory.  A key
      // alone with its value is in place, and the first key of a pair places
      // both; a longer run is listed by its first key, and a warp finds its
      // end and places each of its keys at the run's start plus the number of
      // the run's larger keys (keys are distinct).
      const int64_t wlo = lo > RUN_MAX ? lo - RUN_MAX : 0;
      const int64_t whi = hi + RUN_MAX < len ? hi + RUN_MAX : len;
      for (int64_t j = wlo + threadIdx.x; j < whi; j += RS_THREADS) s_keys[j - wlo] = __ldcg(srt + j);
      unsigned* runs = reinterpret_cast<unsigned*>(s_keys + (whi - wlo));  // run starts, relative to lo
      if (threadIdx.x == 0) sm.nruns = 0;
      __syncthreads();
      auto val = [&](int64_t j) { return static_cast<uint32_t>(s_keys[j - wlo] >> 32); };
      for (int64_t i = lo + threadIdx.x; i < hi; i += RS_THREADS) {
        const unsigned long long kk = s_keys[i - wlo];
        const uint32_t v = static_cast<uint32_t>(kk >> 32);
        if (i > 0 && val(i - 1) == v) continue;  // not the first of its run
        if (i + 1 == len || val(i + 1) != v) {
          if (i < a.k) emit_key(a, row, i, kk);
        } else if (i + 2 == len || val(i + 2) != v) {  // a pair: the larger key first
          const unsigned long long k2 = s_keys[i + 1 - wlo];
          if (i < a.k) emit_key(a, row, i, kk > k2 ? kk : k2);
          if (i + 1 < a.k) emit_key(a, row, i + 1, kk > k2 ? k2 : kk);
        } else {
          runs[atomicAdd(&sm.nruns, 1u)] = static_cast<unsigned>(i - lo);
        }
      }
      __syncthreads();
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
      for (unsigned t = warp; t < sm.nruns; t += RS_THREADS / 32) {
        const int64_t st = lo + runs[t];
        const uint32_t v = val(st);
        int64_t L = 0;  // run length (at most RUN_MAX, so within the staged keys)
        for (int64_t b = st;; b += 32) {
          const int64_t j = b + lane;
          const unsigned same = __ballot_sync(FULL_MASK, j < whi && val(j) == v);
          if (same != FULL_MASK) {
            L = b - st + __ffs(~same) - 1;
            break;
          }
        }
        for (int64_t q = lane; q < L; q += 32) {
          const unsigned long long kk = s_keys[st + q - wlo];
          int64_t p = st;
          for (int64_t j = 0; j < L; ++j) p += s_keys[st + j - wlo] > kk;
          if (p < a.k) emit_key(a, row, p, kk);
        }
      }
    }
  }
  if (full) {
    // Heavy ties: the full sort (from whatever order the keys are in).
    int lastp = -1;
    for (int p = 0; p < 8; ++p)
      if (!sm.trivial[p]) lastp = p;
    for (int p = 0; p < 8; ++p) {
      if (sm.trivial[p]) continue;
      radix_pass(a, row, chunk, lo, hi, p, seq, p == lastp, (cur ? tmp : a.keys) + row * a.key_stride,
                 (cur ? a.keys : tmp) + row * a.key_stride, fr, sm, s_keys, c);
      RS_LEAVE_IF_GAVE_UP();
      ++seq;
      cur ^= 1;
      if (p != lastp) {
        grid_sync(c, target += G, sm);
        RS_LEAVE_IF_GAVE_UP();
      }
    }
  }
#undef RS_LEAVE_IF_GAVE_UP
}

struct Scratch {
  unsigned long long* tmp;
  unsigned long long* flags;
  int64_t flag_stride;
  SortCtl* ctl;
  unsigned* bk;  // per row: the bucket stage's counts and cursors (2 BK)
};

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// Chunks per row: no chunk shorter than 32 keys, and all CTAs of the launch
// (chunks x rows) resident at once, one per SM.
int64_t chunks_per_row(int64_t key_stride, int64_t nrows) {
  int64_t g = sms() / (nrows > 0 ? nrows : 1);
  const int64_t by_len = (key_stride + 31) / 32;
  if (g > by_len) g = by_len;
  return g < 1 ? 1 : g;
}

Scratch carve(void* scratch, int64_t key_stride, int64_t rows) {
  Scratch s;
  char* p = static_cast<char*>(scratch);
  s.tmp = reinterpret_cast<unsigned long long*>(p);
  p += align256(sizeof(unsigned long long) * key_stride * rows);
  s.flag_stride = chunks_per_row(key_stride, 1) * 256;
  s.flags = reinterpret_cast<unsigned long long*>(p);
  p += align256(sizeof(unsigned long long) * s.flag_stride * rows);
  s.ctl = reinterpret_cast<SortCtl*>(p);
  p += align256(sizeof(SortCtl) * rows);
  s.bk = reinterpret_cast<unsigned*>(p);
  return s;
}

}  // namespace

size_t radix_sort_scratch_bytes(int64_t key_stride, int64_t rows) {
  return align256(sizeof(unsigned long long) * key_stride * rows) +
         align256(sizeof(unsigned long long) * chunks_per_row(key_stride, 1) * 256 * rows) +
         align256(sizeof(SortCtl) * rows) + align256(sizeof(unsigned) * 2 * BK * rows);
}

void* radix_sort_ctl(void* scratch, int64_t key_stride, int64_t rows) { return carve(scratch, key_stride, rows).ctl; }

size_t radix_sort_ctl_bytes() { return sizeof(SortCtl); }

cudaError_t launch_radix_sort(const RadixSortArgs& a, cudaStream_t stream) {
  const Scratch s = carve(a.scratch, a.key_stride, a.total_rows);
  if (!a.ctl_zeroed) {
    const cudaError_t e = cudaMemsetAsync(s.ctl, 0, sizeof(SortCtl) * a.total_rows, stream);
    if (e != cudaSuccess) return e;
  }
  const unsigned G = static_cast<unsigned>(chunks_per_row(a.key_stride, a.nrows));
  cudaFuncSetAttribute(k_rs_sort, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(RS_SMEM_LAUNCH));
  launch_kernel(k_rs_sort, dim3(G, static_cast<unsigned>(a.nrows)), RS_THREADS, RS_SMEM_LAUNCH, stream, a, s.ctl,
                s.tmp, s.flags, s.flag_stride, s.bk);
  return cudaGetLastError();
}

}  // namespace profk
