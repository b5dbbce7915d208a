// update_row.cuh -- the row update of a step: the accepted sampled ids
// appended to a request's token row.
#pragma once

#include "sgd_internal.h"

namespace sgd {

// Appends the leading run of ids in [0, V) of sp[0, T) to row at n (ids past
// S dropped) and returns the new length.  The first 64 ids are read once
// (`sp` may be page-locked host memory read in place).  With tail != null the
// appended ids also go to tail[0 .. min(appended, dtail)), newest first
// (tail[i] = the token at new length - 1 - i).  Whole warp.
__device__ inline int update_row_warp(int32_t *row, int n, const int32_t *sp, int T, int S, int V,
                                      int lane, uint32_t &fl, int *tail = nullptr, int dtail = 0) {
  int c = T;
  bool bad = false;
  int keep0 = 0, keep1 = 0;  // sp[lane], sp[32 + lane]
  for (int base = 0; base < T; base += 32) {
    const int i = base + lane;
    const int v = i < T ? sp[i] : 0;
    if (base == 0) keep0 = v;
    else if (base == 32) keep1 = v;
    const bool term = i < T && (v < 0 || v >= V);
    const unsigned m = __ballot_sync(FULL, term);
    if (m) {
      const int f = __ffs(m) - 1;
      const int vf = __shfl_sync(FULL, v, f);
      c = base + f;
      bad = vf >= V;
      break;
    }
  }
  const int ca = (int)min((long long)c, (long long)S - n);  // ids that fit
  for (int i = lane; i < ca; i += 32) {
    const int v = i < 32 ? keep0 : (i < 64 ? keep1 : sp[i]);
    row[n + i] = v;
    if (tail != nullptr && ca - 1 - i < dtail) tail[ca - 1 - i] = v;
  }
  if (bad) fl |= SGD_ERR_SAMPLED_TOKEN;
  return n + max(ca, 0);
}

}  // namespace sgd
