// Validity bits of 64 tokens for one token of the other side, and what a
// 64-token chunk's summary decides about them without reading the tokens:
// pure functions of plain integers.  The kernels use them on the general
// masking path; the CPU tests compile this header for the host and check
// every decision against the token-by-token rule.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define ATTN_MASK_HD __host__ __device__ __forceinline__
#else
#define ATTN_MASK_HD inline
#endif

namespace attn_mask {

// Bit c set for lo <= c < hi, c in [0, 64).  Masks are applied with selects on
// these bits so the element loops stay branch-free.
ATTN_MASK_HD uint64_t range_bits64(int lo, int hi) {
  lo = lo < 0 ? 0 : lo;
  hi = hi > 64 ? 64 : hi;
  if (hi <= lo) return 0ull;
  const uint64_t upper = (hi >= 64) ? ~0ull : ((1ull << hi) - 1ull);
  const uint64_t lower = (lo <= 0) ? 0ull : ((1ull << lo) - 1ull);
  return upper & ~lower;
}

// A chunk's tokens are valid for a token with nonzero segment id `id` whose
// band admits the positions [px, py] when they carry the same id and sit at a
// position inside the band.  From the chunk's summary (smallest and largest
// nonzero id, smallest and largest position over its nonzero-id tokens; uniform:
// all 64 tokens exist and carry one nonzero id; consec: uniform, and token k
// sits at min_pos + k), write the 64 validity bits to *bits and return true
// when the summary decides them; return false otherwise (the caller then
// compares token by token).
ATTN_MASK_HD bool chunk_decide(int min_id, int max_id, int min_pos, int max_pos, int uniform,
                               int consec, int id, int px, int py, uint64_t* bits) {
  if (max_id == 0 || id < min_id || id > max_id || max_pos < px || min_pos > py) {
    *bits = 0ull;  // no token carries the id, or none sits inside the band
    return true;
  }
  if (!uniform) return false;
  // every token carries the id (min_id <= id <= max_id == min_id)
  if (min_pos >= px && max_pos <= py) {
    *bits = ~0ull;
    return true;
  }
  if (!consec) return false;
  // token k at position min_pos + k: the band keeps k in [px - min_pos, py - min_pos]
  const int lo = px <= min_pos ? 0 : px - min_pos;
  const int hi = py >= max_pos ? 64 : py - min_pos + 1;
  *bits = range_bits64(lo, hi);
  return true;
}

}  // namespace attn_mask
