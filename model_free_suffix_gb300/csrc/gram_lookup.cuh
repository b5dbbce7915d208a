// gram_lookup.cuh -- one warp's lookup of an m-gram in the snapshot's n-gram
// table (the table is described in sgd_internal.h).
#pragma once

#include "sgd_internal.h"

namespace sgd {

// [lo, hi): the suffix-array interval of the m-gram g (g.x its first token in
// text order, then g.y, g.z, g.w; 2 <= m <= 4), by one warp; slot7: the
// entry's [7] (for m = 2, 3 with gram drafts the gram's draft block, else
// -2); empty and -2 when the gram begins no suffix.  Lanes 0..7 read one
// 128-byte bucket (lanes 2e and 2e + 1 hold entry e) and two ballots find
// the entry; a bucket with an empty entry ends the search.
__device__ inline void gt_lookup(const int32_t *GT, uint64_t gtm, const int4 &P, int m, int lane,
                                 long long &lo, long long &hi, int &slot7) {
  const int4 g = make_int4(P.x, m >= 2 ? P.y : KEY_END, m >= 3 ? P.z : KEY_END, m >= 4 ? P.w : KEY_END);
  uint64_t b = gram_hash(m, g.x, g.y, g.z, g.w) & gtm;
  lo = hi = 0;
  slot7 = -2;
  for (uint64_t step = 0; step <= gtm; ++step, b = (b + 1) & gtm) {
    int4 v = make_int4(0, 0, 0, 0);
    if (lane < 2 * GT_BUCKET)
      v = __ldg(reinterpret_cast<const int4 *>(GT + (size_t)b * GT_BUCKET * GT_ENTRY) + lane);
    const bool even = (lane & 1) == 0 && lane < 2 * GT_BUCKET;
    const bool odd = (lane & 1) == 1 && lane < 2 * GT_BUCKET;
    const unsigned e0 = __ballot_sync(FULL, even && v.x == m && v.y == g.x && v.z == g.y && v.w == g.z);
    const unsigned e1 = __ballot_sync(FULL, odd && v.x == g.w);
    const unsigned match = e0 & (e1 >> 1);  // bit 2e: entry e holds the gram
    if (match) {
      const int src = __ffs(match);          // lane 2e + 1: (t3, lo, hi, [7])
      lo = __shfl_sync(FULL, v.y, src);
      hi = __shfl_sync(FULL, v.z, src);
      slot7 = __shfl_sync(FULL, v.w, src);
      return;
    }
    if (__ballot_sync(FULL, even && v.x == 0)) return;
  }
}

}  // namespace sgd
