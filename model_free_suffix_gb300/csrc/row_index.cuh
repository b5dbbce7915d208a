// row_index.cuh -- per-row bigram position index: the row's own match without
// a scan of the row.
//
// Every end j of the row's self match with L(j) >= 2 holds the row's last two
// tokens at j-1, j.  So when the positions of that bigram in the row are known
// in full, the self match is their backward extension against the tail, and
// the row (4 n bytes per step) need not be read.  This is the per-request
// structure the suffix-decoding RFC keeps on the device so that a step costs
// work in what changed, not in the row's length (RFC "Suffix decoding on GPU
// (suffix_gpu)", Summary).  The index is kept exact:
//   - the update inserts every appended position p >= 1 under (t[p-1], t[p]);
//   - an entry lists up to RI_K positions and counts all of them: a bigram
//     seen more often is "overflowed" and its rows are scanned as before;
//   - per row, `covered` = the row length the entries account for; a row whose
//     length at a launch differs from it (changed by the caller without
//     sgd_reset_rows) is marked invalid (-1) and scanned until it is reset;
//   - sgd_reset_rows starts a row's entries over (a new 8-bit generation: every
//     entry of an older one reads as empty) and inserts the row's positions.
//
// Table: per row H entries (a power of two >= 2 S, so at most half full) of
// RI_ENTRY ints (64 bytes).  Ints 0-1 of an entry are one 64-bit word: bits
// 0-7 the count (saturating at 255), 8-15 the generation, 16-39 t0, 40-63 t1
// (ids below 2^24); ints 4 .. 4 + RI_K hold positions, in no order.  Linear
// probing, at most RI_PROBES entries; nothing is ever deleted.
#pragma once

#include "sgd_internal.h"

namespace sgd {

constexpr int RI_K = 12;
constexpr int RI_ENTRY = 16;
constexpr int RI_PROBES = 64;
constexpr int RI_MAX_TOKEN = (1 << 24) - 1;

__host__ __device__ inline long long ri_entries(int S) {
  long long h = 1;
  while (h < 2LL * S) h <<= 1;
  return h;
}

__device__ __forceinline__ unsigned long long ri_key(int t1, int t0, int gen) {
  return ((unsigned long long)(unsigned)t1 << 40) | ((unsigned long long)(unsigned)t0 << 16) |
         ((unsigned long long)(unsigned)gen << 8);
}

__device__ __forceinline__ long long ri_slot(int t1, int t0, long long H) {
  unsigned long long h = ((unsigned long long)(unsigned)t1 << 24) ^ (unsigned)t0;
  h *= 0x9E3779B97F4A7C15ull;
  h ^= h >> 29;
  h *= 0xBF58476D1CE4E5B9ull;
  h ^= h >> 32;
  return (long long)(h & (unsigned long long)(H - 1));
}

// Inserts position p under (t1, t0) into a row's table.  Returns false when
// no entry could be found within RI_PROBES (the table is then unusable for the
// row).  Safe with other threads inserting into the same table.
__device__ inline bool ri_insert(int32_t *tab, long long H, int gen, int t1, int t0, int p) {
  const unsigned long long key = ri_key(t1, t0, gen);
  long long s = ri_slot(t1, t0, H);
  for (int probe = 0; probe < RI_PROBES; ++probe, s = (s + 1) & (H - 1)) {
    unsigned long long *w = reinterpret_cast<unsigned long long *>(tab + s * RI_ENTRY);
    unsigned long long cur = atomicAdd(w, 0ull);
    for (int tries = 0; tries < 4096; ++tries) {
      const bool empty = (int)((cur >> 8) & 255u) != gen;
      if (!empty && (cur & ~255ull) != key) break;  // another bigram: next entry
      const unsigned c = empty ? 0u : (unsigned)(cur & 255u);
      if (c == 255u) return true;                    // saturated: overflowed for good
      const unsigned long long nw = key | (unsigned long long)(c + 1);
      const unsigned long long old = atomicCAS(w, cur, nw);
      if (old == cur) {
        if ((int)c < RI_K) tab[s * RI_ENTRY + 4 + c] = p;
        return true;
      }
      cur = old;
    }
    if ((int)((cur >> 8) & 255u) == gen && (cur & ~255ull) == key) return false;  // (contention bound)
  }
  return false;
}

// Looks (t1, t0) up in a row's table, one 64-byte entry per probe (lanes 0-15
// read its ints).  Returns the bigram's count (0 when absent; > RI_K when its
// list is incomplete) and, when count <= RI_K, writes the positions to
// pos[0 .. count); -1 when the probe bound ran out.  Whole warp.
__device__ inline int ri_lookup(const int32_t *tab, long long H, int gen, int t1, int t0, int lane,
                                int *pos) {
  const unsigned long long key = ri_key(t1, t0, gen);
  long long s = ri_slot(t1, t0, H);
  for (int probe = 0; probe < RI_PROBES; ++probe, s = (s + 1) & (H - 1)) {
    const int v = lane < RI_ENTRY ? __ldcg(tab + s * RI_ENTRY + lane) : 0;
    const unsigned lo = (unsigned)__shfl_sync(FULL, v, 0), hi = (unsigned)__shfl_sync(FULL, v, 1);
    const unsigned long long w = ((unsigned long long)hi << 32) | lo;
    if ((int)((w >> 8) & 255u) != gen) return 0;
    if ((w & ~255ull) == key) {
      const int c = (int)(w & 255u);
      if (c <= RI_K && lane >= 4 && lane < 4 + c) pos[lane - 4] = v;
      __syncwarp();
      return c;
    }
  }
  return -1;
}

// After a row's update from n_old to n tokens (n_old the row length the
// launch read): when the row's entries cover n_old, inserts positions
// [max(1, n_old), n) and records n as covered; otherwise the row is (or
// stays) invalid until it is reset.  Whole warp; row is the row's tokens.
__device__ inline void ri_after_update(const RowIndexArgs &ri, int b, const int32_t *row, int n_old,
                                       int n, bool valid, int lane) {
  int32_t *meta = ri.meta + 2 * (size_t)b;
  if (!valid) {
    if (lane == 0 && meta[0] != -1) meta[0] = -1;
    return;
  }
  int32_t *tab = ri.tab + (size_t)b * ri.H * RI_ENTRY;
  const int gen = meta[1];
  bool ok = true;
  for (int p = max(1, n_old) + lane; p < n; p += 32)
    ok &= ri_insert(tab, ri.H, gen, row[p - 1], row[p], p);
  ok = __all_sync(FULL, ok);
  if (lane == 0) meta[0] = ok ? n : -1;
}

}  // namespace sgd
