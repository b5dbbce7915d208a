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
constexpr int SMALL_BATCH = 8;     // loads each thread has in flight per sweep
constexpr int STAGE_TOKENS = 8192; // validated doc tokens kept on chip for the copy
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
  int vcum[SMALL_DOCS + 1];  // the scan's prefix sums (where a doc's staged tokens start)
  int cnt[SMALL_DOCS];  // per doc: the tokens to scan / to copy
  int pcum[SMALL_DOCS + 1], kcum[SMALL_DOCS + 1];  // placement: ring tokens, docs before each
  int ev[SMALL_DOCS];   // placement: oldest docs evicted before each doc is placed
  int ntv[SMALL_DOCS];  // the num_tokens bound of each doc's row
  int dl[PLAN_WINDOW];
  int esum[PLAN_WINDOW + 1];  // ring tokens of the oldest docs, prefix sums
  RingState rs;
  int stop;    // a wait gave up: no doc of the call is placed
  int serial;  // the parallel placement does not apply: one thread walks the docs
  long long placed;
  union {
    SigBatchSmem sig;             // (after the copy)
    int32_t tok[STAGE_TOKENS];    // the first STAGE_TOKENS doc tokens, as scanned
  } u;
};

// (a static shared-memory array in the standalone ingest kernel)
static_assert(sizeof(SmallIngestSmem) <= 48 * 1024, "SmallIngestSmem exceeds static shared memory");

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
// multiple of 32): (1) the arguments and the ring state; (2) per doc, by the
// warps in turn, [the bounded wait for its row's update,] its tokens read
// once (the first id outside [0, V) ends it) and staged on chip, and its
// row's num_tokens bound; the oldest FIFO lengths; (3) the placement (in
// parallel from prefix sums; one thread when evictions reach past the staged
// FIFO lengths); (4) the copy into the ring from the staged tokens.
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
  if (delta && tid == SMALL_DOCS && !wait_flag(g.sync, g.expect)) s.stop = 1;  // every row CTA counted in
  const RingState r0 = s.rs;
  const int win = min(r0.ndocs, PLAN_WINDOW);
  for (int j = tid; j < win; j += nthr) s.dl[j] = g.doc_len[(r0.head + j) % g.max_docs];
  if (tid <= SMALL_DOCS) s.vcum[tid] = s.cum[tid];
  // Each warp takes docs w, w + warps, ...: waits (bounded) for the doc's row
  // to be updated, then reads the doc's tokens once -- the first id outside
  // [0, V) ends it -- staging them on chip for the copy.  Docs of rows that
  // were updated early are read while later rows are still being drafted.
  const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
  for (int d = warp; d < m; d += nwarps) {
    if (s.ln[d] < 0) continue;  // bad arguments
    if (g.ready != nullptr) {
      // give the doc up rather than read a row mid-update
      bool ok = true;
      if (lane == 0) ok = wait_flag(g.ready + s.row[d], g.expect);
      ok = __shfl_sync(FULL, ok, 0);
      __threadfence();
      if (!ok) {
        if (lane == 0) s.ln[d] = -2;
        continue;
      }
    }
    const int ln = s.ln[d];
    const int32_t *src = g.tok + (size_t)s.row[d] * g.S + s.st[d];
    int bad = ln;  // first id outside [0, V)
    for (int u0 = 0; u0 < ln; u0 += 32 * SMALL_BATCH) {
      int v[SMALL_BATCH];
#pragma unroll
      for (int b = 0; b < SMALL_BATCH; ++b) {
        const int u = u0 + 32 * b + lane;
        v[b] = u < ln ? src[u] : 0;
      }
#pragma unroll
      for (int b = 0; b < SMALL_BATCH; ++b) {
        const int u = u0 + 32 * b + lane;
        if (u < ln) {
          if (v[b] < 0 || v[b] >= g.V) bad = min(bad, u);
          const int sg = s.cum[d] + u;  // (s.vcum is copied from s.cum meanwhile)
          if (sg < STAGE_TOKENS) s.u.tok[sg] = v[b];
        }
      }
    }
    bad = __reduce_min_sync(FULL, (unsigned)bad);
    if (lane == 0) {
      s.first[d] = bad;
      s.ntv[d] = g.ntok != nullptr ? g.ntok[s.row[d]] : INT_MAX;
    }
  }
  __syncthreads();
  if (tid < m) {
    const int ln = s.stop ? -2 : s.ln[tid];
    if (ln == -2) {
      s.first[tid] = -1;
      atomicOr(g.err, SGD_ERR_INGEST_WAIT);
    } else if (ln < 0 || (long long)s.st[tid] + ln > s.ntv[tid]) {
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
  }
  __syncthreads();
  // Placement.  Docs go to the write offset in call order, each after
  // evicting the oldest docs while it would not fit (or the FIFO is full).
  // Doc i's place follows from the ring sizes of the docs before it (pcum),
  // and the evictions before it from the prefix sums of the oldest docs'
  // sizes (esum): the fewest oldest docs whose removal makes room, a count
  // that can only grow with i.  This holds while those docs are among the
  // staged oldest ones and no doc of this call has to go; otherwise thread 0
  // walks the docs one by one.
  if (tid < SMALL_DOCS) {
    const int L = tid < m ? s.first[tid] : -1;
    const bool too_long = L > 0 && (long long)L + 1 > g.C;
    if (too_long) atomicOr(g.err, SGD_ERR_DOC_TOO_LONG);
    s.cnt[tid] = L > 0 && !too_long ? L + 1 : 0;
  } else if (tid == SMALL_DOCS) {
    s.serial = 0;
  }
  __syncthreads();
  if (tid < 32) {
    small_cum(s.cnt, s.pcum);
    // the oldest docs' ring sizes, prefix sums over the staged window
    int run = 0;
    if (tid == 0) s.esum[0] = 0;
    for (int j0 = 0; j0 < win; j0 += 32) {
      const int j = j0 + tid;
      int x = j < win ? s.dl[j] + 1 : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(FULL, x, off);
        if (tid >= off) x += y;
      }
      if (j < win) s.esum[j + 1] = run + x;
      run += __shfl_sync(FULL, x, 31);
    }
  } else if (tid >= 32 && tid < 64) {
    // docs placed before each: the same scan over 0/1
    int c[2];
    const int l = tid - 32;
    c[0] = s.cnt[2 * l] > 0;
    c[1] = s.cnt[2 * l + 1] > 0;
    int x = c[0] + c[1];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(FULL, x, off);
      if (l >= off) x += y;
    }
    s.kcum[2 * l + 1] = x - c[1];
    s.kcum[2 * l + 2] = x;
    if (l == 0) s.kcum[0] = 0;
  }
  __syncthreads();
  if (tid < m && s.cnt[tid] > 0) {
    // the fewest oldest docs e with live - esum[e] + pcum[tid + 1] <= C and
    // ndocs - e + kcum[tid + 1] <= max_docs
    const long long need = r0.live + s.pcum[tid + 1] - g.C;
    int lo = 0, hi = win + 1;  // esum[e] >= need for the smallest e in [lo, hi)
    if (need > 0) {
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s.esum[mid] >= need) hi = mid;
        else lo = mid + 1;
      }
    }
    const int e = max(lo, r0.ndocs + s.kcum[tid + 1] - g.max_docs);
    if (e > win || e > r0.ndocs) s.serial = 1;
    s.ev[tid] = e;
  }
  __syncthreads();
  if (s.serial) {
    if (tid == 0) {
      PlanWalk w{r0, r0.ndocs, win, 0, 0, 0, 0u, 0};
      for (int i = 0; i < m; ++i)
        place_doc(w, i, s.first[i], g.C, s.dl, g.doc_start, g.doc_len, g.max_docs, s.dest, s.order);
      *g.rs = w.r;
      s.placed = w.placed;
    }
  } else {
    if (tid < m) {
      if (s.cnt[tid] > 0) {
        const long long d = (r0.wp + s.pcum[tid]) % g.C;
        const int slot = (int)(((long long)r0.head + r0.ndocs + s.kcum[tid]) % g.max_docs);
        g.doc_start[slot] = d;
        g.doc_len[slot] = s.first[tid];
        s.dest[tid] = d;
        s.order[s.kcum[tid]] = tid;
      } else {
        s.dest[tid] = -1;
      }
    }
    if (tid == 0) {
      const int K = s.kcum[m], P = s.pcum[m];
      int e = 0;  // evictions by the last doc placed
      for (int i = m - 1; i >= 0; --i)
        if (s.cnt[i] > 0) { e = s.ev[i]; break; }
      RingState r = r0;
      r.live = r0.live - s.esum[e] + P;
      r.head = (int)(((long long)r0.head + e) % g.max_docs);
      r.ndocs = r0.ndocs - e + K;
      r.wp = (r0.wp + P) % g.C;
      r.pushed = r0.pushed + K;
      *g.rs = r;
      s.placed = P;
    }
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
        const int sg = s.vcum[d] + u;  // where the scan staged it
        v[b] = u < s.first[d] ? (sg < STAGE_TOKENS ? s.u.tok[sg] : g.tok[(size_t)s.row[d] * g.S + s.st[d] + u])
                              : g.V;
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
    sig_update_cta(SigBuild{g.ring, g.C, g.V, g.sig, g.C / WIN}, r0.wp, s.placed, s.u.sig);
  }
}

}  // namespace
}  // namespace sgd
