// delta_sig.cuh -- per-window gram signatures of the corpus ring, the filter
// that lets a row read only the parts of the delta that can hold its match.
//
// Each ring window of WIN positions has an 8192-bit signature: bit
// sig_bucket(m, ...) is set for every m-gram (m = 2, 3, 4) that ENDS at a
// position of the window and consists of ids only (no sentinel).  A row whose
// last m tokens do not hash to a set bit has no end of match length >= m in
// that window, so the window need not be read; a set bit only means "maybe"
// (the window is then read and checked exactly).  Signatures are kept with
// the ring: after each ingest call has written its docs, every window the
// call touched is recomputed from the ring's contents, except that the window
// holding the call's first position only gains the new grams' bits (rows of
// the same fused step may be reading it).  So a gram present in the ring
// always has its bit set; a bit may outlive its gram (a harmless extra read).
//
// Layout: sig[word * W + w] holds bits 32 word .. 32 word + 31 of window w
// (W = C / WIN windows), so the words one bucket takes in consecutive windows
// are consecutive.
#pragma once

#include "sgd_internal.h"

namespace sgd {

constexpr int SIG_LOG = 13;
constexpr int SIG_WORDS = (1 << SIG_LOG) / 32;  // 256 words = 8192 bits per window
constexpr int SIG_BATCH = 16;                   // windows one CTA builds in shared memory at a time

__host__ __device__ __forceinline__ unsigned sig_mix(unsigned h, int v) {
  h ^= (unsigned)v * 0x85EBCA77u;
  h = (h << 13) | (h >> 19);
  return h * 5u + 0xE6546B64u;
}

// Bucket of the m-gram whose last token is a0 (a1 the one before it, ...).
__host__ __device__ __forceinline__ unsigned sig_bucket(int m, int a0, int a1, int a2, int a3) {
  unsigned h = 0x9E3779B1u * (unsigned)m;
  h = sig_mix(h, a0);
  h = sig_mix(h, a1);
  if (m >= 3) h = sig_mix(h, a2);
  if (m >= 4) h = sig_mix(h, a3);
  h ^= h >> 16;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  return h & ((1u << SIG_LOG) - 1u);
}

struct SigBuild {
  int32_t *ring;
  long long C;
  int Z;          // sentinel (ids are < Z)
  uint32_t *sig;  // SIG_WORDS * W words
  long long W;    // C / WIN
};

struct SigBatchSmem {
  uint32_t words[SIG_BATCH * SIG_WORDS];
  int32_t tok[SIG_BATCH * WIN + 4];  // the batch's tokens, after the 3 before its first
};

// Bits of the grams ending at position p, given x0 = x[p] .. x3 = x[p-3].
template <typename F>
__device__ __forceinline__ void sig_grams(int x0, int x1, int x2, int x3, int Z, F &&set) {
  if (x0 >= Z || x1 >= Z) return;
  set(sig_bucket(2, x0, x1, 0, 0));
  if (x2 >= Z) return;
  set(sig_bucket(3, x0, x1, x2, 0));
  if (x3 >= Z) return;
  set(sig_bucket(4, x0, x1, x2, x3));
}

// The signatures after a write of positions [first, first + count) (mod C;
// count > 0), as part `part` of `nparts` CTAs.  The first window gains bits
// only (unless the write starts at its first position or covers the whole
// ring); every other window the write touched is rebuilt from the ring, in
// contiguous shares per CTA.  The writes to the ring are visible to the
// calling CTAs (an earlier kernel, or a __syncthreads after them).
__device__ inline void sig_update_cta(const SigBuild &g, long long first, long long count,
                                      SigBatchSmem &s, int part = 0, int nparts = 1) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const long long C = g.C, W = g.W;
  auto tok_at = [&](long long p) {
    p %= C;
    if (p < 0) p += C;
    return g.ring[p];
  };
  const bool whole = count >= C;
  const long long fw = whole ? 0 : first / WIN;  // windows numbered from fw, without wrap
  const long long nw = whole ? W : (first % WIN + count + WIN - 1) / WIN;
  const long long rb = !whole && first % WIN != 0 ? 1 : 0;  // windows rebuilt start at fw + rb
  if (rb == 1 && part == 0) {
    // the first window: add the new positions' grams
    const long long end = min(first + count, (fw + 1) * WIN);
    for (long long p = first + tid; p < end; p += nthr)
      sig_grams(tok_at(p), tok_at(p - 1), tok_at(p - 2), tok_at(p - 3), g.Z, [&](unsigned b) {
        atomicOr(&g.sig[(size_t)(b >> 5) * W + fw], 1u << (b & 31));
      });
  }
  const long long share = (nw - rb + nparts - 1) / nparts;
  const long long wa = rb + part * share, wb = min(nw, wa + share);
  for (long long w0 = wa; w0 < wb; w0 += SIG_BATCH) {
    const int nb = (int)min((long long)SIG_BATCH, wb - w0);
    const long long p0 = (fw + w0) * WIN;  // first position of the batch (unwrapped)
    for (int i = tid; i < nb * SIG_WORDS; i += nthr) s.words[i] = 0u;
    for (int i = tid; i < nb * WIN + 3; i += nthr) s.tok[i] = tok_at(p0 - 3 + i);
    __syncthreads();
    for (int i = tid; i < nb * WIN; i += nthr) {
      const int j = i / WIN;
      const int32_t *t = s.tok + i + 3;
      sig_grams(t[0], t[-1], t[-2], t[-3], g.Z, [&](unsigned b) {
        atomicOr(&s.words[j * SIG_WORDS + (b >> 5)], 1u << (b & 31));
      });
    }
    __syncthreads();
    for (int i = tid; i < nb * SIG_WORDS; i += nthr) {
      const int wd = i / nb, j = i - wd * nb;  // consecutive threads: consecutive windows
      const long long w = (fw + w0 + j) % W;
      g.sig[(size_t)wd * W + w] = s.words[j * SIG_WORDS + wd];
    }
    __syncthreads();
  }
}

}  // namespace sgd
