// Rows longer than a candidate key's 32-bit index can address.
//
// The paper runs Prof-K on single rows of up to 4.3e9 elements (corrected
// version, Section 5, Table 4).  A candidate here is the 64-bit key
// (ord(v) << 32) | ~i, whose index field holds 32 bits, so a longer row is
// split into P contiguous segments of at most 2^32 elements; the exact top-k
// of every segment is selected by the batched path (each segment with the
// budget eps / P, so one attempt of the whole row fails with probability at
// most eps by the union bound), and this kernel merges the P sorted candidate
// lists into the row's top k.
//
// Why the merge is exact: an element whose rank in the whole row is r < k is
// preceded by r elements, each of which is in the top k of its own segment, so
// all of them are among the candidates and its rank among the candidates is r.
// An element of rank >= k is preceded among the candidates by at least k
// elements (either all of those preceding it are candidates, or a preceding
// non-candidate f is, and then the k candidates of f's segment all precede it).
// Hence a candidate lands at position r < k exactly when r is its rank in the
// row, and positions 0..k-1 are each written once.
#include "kernels.h"

namespace profk {
namespace {

// Number of entries of the list keys[0..len) (descending order keys; equal keys
// ascending by index) that precede a candidate with order key q: those with a
// larger key, and also those with an equal key when `ties_first` (the list's
// segment lies before the candidate's, so its equal values have lower indices).
__device__ __forceinline__ int64_t count_before(const float* vals, int64_t len, uint32_t q, bool ties_first) {
  int64_t lo = 0, hi = len;  // first position whose entry does not precede
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    const uint32_t m = ord_key(vals[mid]);
    const bool before = ties_first ? m >= q : m > q;
    if (before)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(256) k_merge_segments(MergeSegmentsArgs a) {
  pdl_wait();
  const int64_t total = a.list_len * (a.lists - 1) + a.last_len;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < total;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int s = static_cast<int>(c / a.list_len);
    const int64_t p = c - static_cast<int64_t>(s) * a.list_len;
    const float v = a.vals[c];
    const int64_t li = a.idx[c];
    if (li < 0) continue;  // a segment's emission rejected an index (never for a valid selection)
    const uint32_t q = ord_key(v);
    int64_t rank = p;
    for (int o = 0; o < a.lists && rank < a.k; ++o) {
      if (o == s) continue;
      const int64_t len = o == a.lists - 1 ? a.last_len : a.list_len;
      rank += count_before(a.vals + static_cast<int64_t>(o) * a.list_len, len, q, o < s);
    }
    if (rank < a.k) {
      a.out_vals[rank] = v;
      a.out_idx[rank] = static_cast<int64_t>(s) * a.seg_len + li;
    }
  }
}

}  // namespace

void launch_merge_segments(const MergeSegmentsArgs& a, cudaStream_t stream) {
  const int64_t total = a.list_len * (a.lists - 1) + a.last_len;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  launch_kernel(k_merge_segments, static_cast<unsigned>(blocks), 256, 0, stream, a);
}

}  // namespace profk
