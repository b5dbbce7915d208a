// ingest_cta.cuh -- appending finished responses to the corpus ring from a
// single CTA, for calls of up to SMALL_DOCS docs.  Used by the ingest kernel
// of corpus.cu and by the fused step kernel of propose.cu (there the CTA runs
// beside the row CTAs and first waits for each doc's row to be updated).
//
// Sources (page title, section):
//   "SuffixGPU" (suffix-gpu 0.1.1, PyPI): Quickstart (harvest_finished);
//     How it works, step 4 (new documents append; oldest documents are
//     evicted when the ring is full).
//   "Suffix Decoding" (vLLM docs): Model Runner V2 (a token budget, oldest
//     first out).
#pragma once

#include <climits>

#include "delta_sig.cuh"
#include "sgd_internal.h"

namespace sgd {
namespace {

constexpr int PLAN_WINDOW = 1024;  // oldest FIFO lengths staged for evictions
constexpr int SMALL_DOCS = 64;     // calls up to this size run in one CTA (of > 64 threads)
constexpr int SMALL_BATCH = 4;     // loads each thread has in flight per sweep
constexpr unsigned STEP_SPIN_LIMIT = 1u << 17;  // ~0.1 s of polling; a normal wait is microseconds

// Sequential placement, in call order: evict the oldest docs while the new
// doc would not fit (or the FIFO is full), then append at the write offset.
// A doc pushed by this call and evicted by a later doc of the same call is
// not copied.  One thread walks the docs; the lengths of the oldest FIFO
// docs are staged in shared memory first (`win` of them), so the walk
// rarely waits on global memory.
struct PlanWalk {
  RingState r;
  int r0_ndocs;  // docs live before the call
  int win;       // staged oldest lengths
  int evicted, pushed, ev_call;
  uint32_t fl;
  long long placed;  // ring tokens the call's placements took (from the old write offset on)
};

__device__ inline void place_doc(PlanWalk &w, int i, int L, long long C, const int *s_dl,
                                 int64_t *doc_start, int32_t *doc_len, int max_docs, int64_t *dest,
                                 int32_t *order) {
  RingState &r = w.r;
  dest[i] = -1;
  if (L <= 0) return;
  const long long s = (long long)L + 1;
  if (s > C) {
    w.fl |= SGD_ERR_DOC_TOO_LONG;
    return;
  }
  while (r.ndocs > 0 && (r.live + s > C || r.ndocs == max_docs)) {
    const int len = w.evicted < w.win ? s_dl[w.evicted] : doc_len[r.head];
    r.live -= (long long)len + 1;
    r.head = (r.head + 1) % max_docs;
    r.ndocs--;
    if (w.evicted >= w.r0_ndocs) dest[order[w.ev_call++]] = -1;  // pushed by this call
    ++w.evicted;
  }
  const int slot = (r.head + r.ndocs) % max_docs;
  doc_start[slot] = r.wp;
  doc_len[slot] = L;
  dest[i] = r.wp;
  order[w.pushed++] = i;
  r.wp = (r.wp + s) % C;
  r.live += s;
  r.ndocs++;
  r.pushed++;
  w.placed += s;
}

// Warp 0: inclusive prefix sums of c[0 .. SMALL_DOCS) (two per lane) into
// s_cum[1 .. SMALL_DOCS].
__device__ __forceinline__ void small_cum(const int *c, int *s_cum) {
  const int lane = threadIdx.x & 31;
  const int c0 = c[2 * lane], c1 = c[2 * lane + 1];
  int x = c0 + c1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(FULL, x, off);
    if (lane >= off) x += y;
  }
  s_cum[2 * lane + 1] = x - c1;
  s_cum[2 * lane + 2] = x;
  if (lane == 0) s_cum[0] = 0;
}

// The doc d < m holding flattened token g: the last d with s_cum[d] <= g
// (s_cum is non-decreasing, so empty docs are stepped over).
__device__ __forceinline__ int small_doc(const int *s_cum, int m, int g) {
  int d = 0;
#pragma unroll
  for (int step = SMALL_DOCS / 2; step; step >>= 1)
    if (d + step < m && s_cum[d + step] <= g) d += step;
  return d;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct SmallIngestSmem {
  int64_t dest[SMALL_DOCS];
  int row[SMALL_DOCS], st[SMALL_DOCS], ln[SMALL_DOCS], first[SMALL_DOCS], order[SMALL_DOCS];
  int cum[SMALL_DOCS + 1];
  int cnt[SMALL_DOCS];  // per doc: the tokens to scan / to copy
  int dl[PLAN_WINDOW];
  RingState rs;
  int stop;  // a wait gave up: no doc of the call is placed
  long long placed;
  SigBatchSmem sig;
};

struct SmallIngest {
  const int32_t *tok;   // [B, S]
  const int32_t *ntok;  // [B] or null
  int B, S, V;
  const int32_t *rows, *starts, *lengths;
  int m;  // 1..SMALL_DOCS
  int32_t *ring;
  long long C;
  RingState *rs;
  int64_t *doc_start;
  int32_t *doc_len;
  int max_docs;
  uint32_t *err;
  const uint32_t *ready;  // per row: == expect once the row's update is written; or null
  uint32_t expect;
  // Fused step whose rows also read the delta from the ring (dcap > 0): the
  // ring state is changed only once every row CTA has read it (sync[0], the
  // step epoch, == expect), and if the new docs' tokens could land on the
  // rows' visible delta, only once every row CTA is done (sync[3] == expect).
  const uint32_t *sync;
  const CorpusDesc *desc;
  long long dcap;
  uint32_t *sig;  // the ring's window signatures (null: none kept)
};

// Bounded wait for *f == expect; false if it gave up.
__device__ inline bool wait_flag(const uint32_t *f, uint32_t expect) {
  unsigned spins = 0;
  while (ld_acquire_u32(f) != expect) {
    if (++spins > STEP_SPIN_LIMIT) return false;
    if (spins > 16) __nanosleep(64);
  }
  return true;
}

// The whole call in one CTA (a block of more than SMALL_DOCS threads, a
// multiple of 32).  Each
// phase issues all of its loads at once over the docs' tokens laid end to
// end: (1) the arguments and the ring state; [the bounded wait for the
// rows' updates;] (2) the num_tokens bounds, the oldest FIFO lengths and
// every token (first id outside [0, V) per doc); thread 0 then places the
// docs from shared memory; (3) the copy into the ring.
__device__ inline void ingest_small_cta(const SmallIngest &g, SmallIngestSmem &s) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int m = g.m;
  if (tid < SMALL_DOCS) {
    int ln = 0;
    bool ok = false;
    if (tid < m) {
      const int row = g.rows[tid], st = g.starts[tid];
      ln = g.lengths[tid];
      // inside the row buffer; the bound by num_tokens is checked once it arrives
      ok = row >= 0 && row < g.B && st >= 0 && ln >= 0 && (long long)st + ln <= g.S;
      s.row[tid] = row;
      s.st[tid] = st;
      s.ln[tid] = ok ? ln : -1;
      s.first[tid] = ln;
    }
    s.cnt[tid] = ok ? ln : 0;
  } else if (tid == SMALL_DOCS) {
    s.rs = *g.rs;
    s.stop = 0;
  }
  __syncthreads();
  if (tid < 32) small_cum(s.cnt, s.cum);
  __syncthreads();
  const bool delta = g.ready != nullptr && g.sync != nullptr && g.dcap > 0;
  if (g.ready != nullptr) {
    if (tid < m && s.ln[tid] >= 0) {
      // give the doc up rather than read a row mid-update
      if (!wait_flag(g.ready + s.row[tid], g.expect)) s.ln[tid] = -2;
      __threadfence();
    }
    if (delta && tid == SMALL_DOCS && !wait_flag(g.sync, g.expect)) s.stop = 1;  // every row CTA counted in
    __syncthreads();
  }
  const RingState r0 = s.rs;
  const int win = min(r0.ndocs, PLAN_WINDOW);
  for (int j = tid; j < win; j += nthr) s.dl[j] = g.doc_len[(r0.head + j) % g.max_docs];
  long long ntv = LLONG_MAX;
  if (tid < m && g.ntok != nullptr && s.ln[tid] >= 0) ntv = g.ntok[s.row[tid]];
  const int total = s.cum[SMALL_DOCS];
  for (int g0 = 0; g0 < total; g0 += nthr * SMALL_BATCH) {
    int v[SMALL_BATCH], dd[SMALL_BATCH], uu[SMALL_BATCH];
#pragma unroll
    for (int b = 0; b < SMALL_BATCH; ++b) {
      const int gi = g0 + b * nthr + tid;
      dd[b] = -1;
      if (gi < total) {
        const int d = small_doc(s.cum, m, gi);
        dd[b] = d;
        uu[b] = gi - s.cum[d];
        v[b] = g.tok[(size_t)s.row[d] * g.S + s.st[d] + uu[b]];
      }
    }
#pragma unroll
    for (int b = 0; b < SMALL_BATCH; ++b)
      if (dd[b] >= 0 && (v[b] < 0 || v[b] >= g.V)) atomicMin(&s.first[dd[b]], uu[b]);
  }
  __syncthreads();
  if (tid < m) {
    const int ln = s.stop ? -2 : s.ln[tid];
    if (ln == -2) {
      s.first[tid] = -1;
      atomicOr(g.err, SGD_ERR_INGEST_WAIT);
    } else if (ln < 0 || (long long)s.st[tid] + ln > ntv) {
      s.first[tid] = -1;
      atomicOr(g.err, SGD_ERR_DOC_ARGS);
    } else if (s.first[tid] < ln) {
      atomicOr(g.err, SGD_ERR_DOC_TOKEN);
    }
  }
  __syncthreads();
  if (tid == 0) {
    if (delta && !s.stop) {
      // the call writes at most T tokens from the write offset on; the rows'
      // visible delta ends at the write offset and starts len tokens before it,
      // so the writes reach it only if T > C - len -- and the rebuilt
      // signatures of the windows they touch reach its windows only if
      // T > C - len - 2 WIN
      long long T = 0;
      for (int i = 0; i < m; ++i)
        if (s.first[i] > 0) T += s.first[i] + 1;
      const DeltaView v = delta_view(r0, g.desc->lin_pushed, g.desc->lin_wp, g.C, g.doc_start);
      if (min(v.len, g.dcap) > 0 && T + 2 * WIN > g.C - v.len && !wait_flag(g.sync + 3, g.expect)) {
        for (int i = 0; i < m; ++i) s.first[i] = -1;
        atomicOr(g.err, SGD_ERR_INGEST_WAIT);
      }
    }
    PlanWalk w{r0, r0.ndocs, win, 0, 0, 0, 0u, 0};
    for (int i = 0; i < m; ++i)
      place_doc(w, i, s.first[i], g.C, s.dl, g.doc_start, g.doc_len, g.max_docs, s.dest, s.order);
    *g.rs = w.r;
    s.placed = w.placed;
    if (w.fl) atomicOr(g.err, w.fl);
  }
  __syncthreads();
  if (tid < SMALL_DOCS) s.cnt[tid] = tid < m && s.dest[tid] >= 0 ? s.first[tid] + 1 : 0;
  __syncthreads();
  if (tid < 32) small_cum(s.cnt, s.cum);
  __syncthreads();
  const int total2 = s.cum[SMALL_DOCS];
  for (int g0 = 0; g0 < total2; g0 += nthr * SMALL_BATCH) {
    int v[SMALL_BATCH];
    long long pos[SMALL_BATCH];
#pragma unroll
    for (int b = 0; b < SMALL_BATCH; ++b) {
      const int gi = g0 + b * nthr + tid;
      pos[b] = -1;
      if (gi < total2) {
        const int d = small_doc(s.cum, m, gi);
        const int u = gi - s.cum[d];
        v[b] = u < s.first[d] ? g.tok[(size_t)s.row[d] * g.S + s.st[d] + u] : g.V;
        long long p = s.dest[d] + u;
        if (p >= g.C) p -= g.C;
        pos[b] = p;
      }
    }
#pragma unroll
    for (int b = 0; b < SMALL_BATCH; ++b)
      if (pos[b] >= 0) g.ring[pos[b]] = v[b];
  }
  if (g.sig != nullptr && s.placed > 0) {
    __syncthreads();  // the docs are in the ring
    sig_update_cta(SigBuild{g.ring, g.C, g.V, g.sig, g.C / WIN}, r0.wp, s.placed, s.sig);
  }
}

}  // namespace
}  // namespace sgd
