// backoff.cu -- multi-length backoff: every row drafts from several candidate
// match lengths per path and the best-scored candidate wins.
//
// Sources (page title, section):
//   "SuffixGPU" (suffix-gpu 0.1.1, PyPI): Highlights ("Multi-length backoff
//     matching": the longest suffix plus shorter, better-supported lengths);
//     How it works, step 1 (for support threshold t, the largest length
//     occurring at least t times: the t-th largest match_back value), step 2
//     (the corpus side: the suffix-array interval of the tail plus a
//     brute-force scan of the not-yet-indexed delta, serving every length),
//     step 3 (each candidate expanded by majority vote and scored; the best
//     wins per path and the two winners compete by the same score).
//
// One CTA of 512 threads per row.  Match lengths are exact: every end of the
// row is measured against the tail, and so is every end of the corpus that
// can match >= 2 tokens -- the hits of the suffix-array interval of the last
// two tokens, and every delta position in a ring window whose gram signature
// holds the last two tokens (no other window can hold such an end).  A
// histogram of the lengths gives the candidate lengths (thresholds 1..nb);
// one more pass per path collects, for each candidate, its R most recent ends
// (the row's and the delta's by a backward scan, the snapshot's by a radix
// selection on the end position over the interval's hits).  Each warp then
// votes one candidate, and thread 0 picks the winner with exact integer
// comparisons.
//
// With the snapshot's n-gram table and gram drafts, and no delta ends, the
// interval walked is that of the shortest of the last 2-, 3- and 4-gram
// without a draft block.  An end matching m or more tokens ends the last
// m-gram, so the ends reaching length m are the valid hits of its interval;
// a block holds their number and the vote of the R most recent of them
// (built with the snapshot), which is exactly the corpus candidate of length
// m.  So the lengths below the walked gram's are counted from the blocks, and
// their candidates come from them, without reading their (largest) intervals.
#include <climits>

#include "delta_sig.cuh"
#include "gram_lookup.cuh"
#include "update_row.cuh"

namespace sgd {

namespace {

constexpr int BO_THREADS = 512;
constexpr int BO_WARPS = BO_THREADS / 32;
constexpr int BO_CANDS = 2 * MAX_BACKOFF;  // row candidates, then corpus candidates
constexpr int BO_LCACHE = 16384;           // interval hits whose length is kept on chip
constexpr int BO_TOPC = 5;                 // length classes of the first radix digit
constexpr int BO_RLCAP = 16384;            // row ends whose match length is kept on chip (dynamic)
static_assert(BO_LCACHE % (4 * BO_THREADS) == 0, "hit_ends: four hits on one side of the cache end");

struct BoShared {
  int tail[MAX_D];
  int hs[MAX_D + 1];  // row ends by match length
  int hc[MAX_D + 1];  // corpus ends (snapshot and delta) by match length
  int hd[MAX_D + 1];  // delta ends by match length
  int len[BO_CANDS];  // candidate lengths (row: [0, ns), corpus: [MAX_BACKOFF, MAX_BACKOFF + nc))
  int tot[BO_CANDS];  // ends reaching each length
  int dtot[BO_CANDS]; // delta ends reaching each length
  int cnt[BO_CANDS];  // ends collected
  int occ[BO_CANDS][MAX_R];  // row: position; corpus: snapshot end e >= 0, delta end u as -(u + 1)
  unsigned wb[MAX_BACKOFF][BO_WARPS];  // per-warp ballots of one chunk
  int hist[MAX_BACKOFF][256];          // radix selection
  long long pref[MAX_BACKOFF];
  int need[MAX_BACKOFF];
  int mode[MAX_BACKOFF];               // snapshot ends: 0 none, 1 every qualifying end, 2 the need most recent
  union {
    unsigned char lc[BO_LCACHE];       // interval hit lengths (0: no continuation), until the votes
    struct {
      int key[MAX_R];                  // a warp's vote: open-addressing count table
      int cnt[MAX_R];
    } ht[BO_WARPS];
  } u;
  union {
    struct {
      int tok[BO_CANDS][MAX_K];        // each candidate's voted tokens
      int cnt[BO_CANDS][MAX_K];        // and their vote counts
    } d;
    int top[BO_TOPC][256];             // until the votes: valid interval hits by length
                                       // class (2, 3, 4, 5, >= 6) and top digit of the end
  } v;
  int dlen[BO_CANDS];
  long long dsum[BO_CANDS];
  int wl[BO_THREADS];                   // delta windows that can hold an end (one batch)
  long long lo, hi, ds;
  long long glo[3], ghi[3];             // the last 2-, 3-, 4-gram's interval (n-gram table)
  int gblk[3];                          // the last 2-, 3-gram's draft block, or -2
  int n, dv, ns, nc, win;
};

// Ordered compaction over the CTA: the values of the threads whose pred holds,
// in thread order, into out; returns their number.  wbuf: BO_WARPS words.
__device__ __forceinline__ int block_compact(bool pred, int val, int *out, unsigned *wbuf, int warp,
                                             int lane) {
  const unsigned bal = __ballot_sync(FULL, pred);
  if (lane == 0) wbuf[warp] = bal;
  __syncthreads();
  int base = 0, total = 0;
  for (int w = 0; w < BO_WARPS; ++w) {
    const int c = __popc(wbuf[w]);
    if (w < warp) base += c;
    total += c;
  }
  if (pred) out[base + __popc(bal & ((1u << lane) - 1u))] = val;
  __syncthreads();
  return total;
}

struct BoRow {
  const int32_t *row;  // the row's tokens
  int n, dl;           // tokens; min(D, n)
  const int32_t *X;    // snapshot text (null: none)
  const int32_t *SA;
  const int4 *K;
  long long N;
  const int32_t *ring;  // the delta: Y[i] = ring[(ds + i) mod C], i < dv
  long long C, ds;
  int dv, Z;
  const int *tail;
};

__device__ __forceinline__ int y_at(const BoRow &r, long long i) {
  return __ldg(r.ring + (r.ds + i) % r.C);
}

// The largest L in [l0, lim] with at(j - i) == tail[i] for every i in
// [l0, L) (at(j - i) is read only for i < lim): eight tokens per round trip,
// their loads issued together.
template <class At>
__device__ __forceinline__ int match_back(const At &at, long long j, int l0, int lim, const int *tail) {
  int L = l0;
  while (L < lim) {
    const int cn = min(8, lim - L);
    int v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = q < cn ? at(j - L - q) : 0;
    int f = cn;  // first mismatch in the chunk
#pragma unroll
    for (int q = 7; q >= 0; --q)
      if (q < cn && v[q] != tail[L + q]) f = q;
    L += f;
    if (f < cn) break;
  }
  return L;
}

// Row end j (j <= n-2): the longest l <= min(D, j+1) with t[j-i] == t[n-1-i], i < l.
// (The row is read with ordinary loads: this kernel appends the step's ids.)
__device__ __forceinline__ int self_len(const BoRow &r, int j) {
  const int lim = min(r.dl, j + 1);
  if (lim <= 0 || r.row[j] != r.tail[0]) return 0;  // (most ends: one load)
  return match_back([&](long long p) { return r.row[p]; }, j, 1, lim, r.tail);
}

// The lengths of hits p0 + j * BO_THREADS (j < 4; l[j] = -1 past hi) of the
// interval of the last m-gram (2 <= m <= 4; end e = SA[p] + m - 1), their
// loads issued together: the continuation X[e+1] (from the key for m <= 3:
// its token m, KEY_END past the text), then the token before the gram for the
// valid hits; the rare longer matches are extended one token at a time.
__device__ __forceinline__ void hit_lens(const BoRow &r, int m, long long p0, long long hi, int l[4],
                                         long long e[4]) {
  int cn[4], ii[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const long long p = p0 + (long long)j * BO_THREADS;
    cn[j] = KEY_END;
    ii[j] = 0;
    if (p < hi) {
      if (m <= 3) {
        const int4 kk = __ldg(r.K + p);
        cn[j] = m == 2 ? kk.z : kk.w;
      }
      ii[j] = __ldg(r.SA + p);
    }
  }
  int xb[4];
  bool more[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool in = p0 + (long long)j * BO_THREADS < hi;
    if (m == 4 && in) cn[j] = (long long)ii[j] + 4 < r.N ? __ldg(r.X + ii[j] + 4) : KEY_END;
    more[j] = in && r.dl > m && ii[j] >= 1;
    xb[j] = more[j] ? __ldg(r.X + ii[j] - 1) : 0;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool valid = cn[j] != KEY_END && cn[j] != r.Z;
    more[j] = more[j] && valid;
    e[j] = (long long)ii[j] + m - 1;
    l[j] = p0 + (long long)j * BO_THREADS < hi ? (valid ? m : 0) : -1;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (more[j] && xb[j] == r.tail[m])
      l[j] = match_back([&](long long p) { return __ldg(r.X + p); }, e[j], m + 1,
                        (int)min((long long)r.dl, e[j] + 1), r.tail);
}

// Delta end u (u <= dv-2): 0 without a continuation, else its match length
// within the delta (its first token follows the snapshot's final sentinel).
__device__ __forceinline__ int delta_len(const BoRow &r, long long u) {
  if (y_at(r, u + 1) == r.Z) return 0;
  return match_back([&](long long p) { return y_at(r, p); }, u, 0, (int)min((long long)r.dl, u + 1),
                    r.tail);
}

// First suffix-array index whose key's first two tokens are >= (upper: >) P,
// by one warp: 32 probes inside the bracket per round, monotone predicate.
__device__ long long pair_bound(const int4 *K, long long N, int p0, int p1, bool upper, int lane) {
  long long lo = 0, hi = N;  // the answer lies in [lo, hi]
  while (hi > lo) {
    const long long span = hi - lo;
    const bool dense = span <= 32;
    const long long q = dense ? lo + lane : lo + (long long)(lane + 1) * span / 33;
    bool ok = !dense || q < hi;
    bool pred = true;
    if (ok) {
      const int4 k = __ldg(K + q);
      const int c = k.x != p0 ? (k.x < p0 ? -1 : 1) : (k.y != p1 ? (k.y < p1 ? -1 : 1) : 0);
      pred = upper ? c > 0 : c >= 0;
    }
    const unsigned below = __ballot_sync(FULL, ok && !pred);  // a prefix of the lanes
    const int f = __popc(below);
    if (dense) return lo + f;
    const long long qlo = __shfl_sync(FULL, q, f > 0 ? f - 1 : 0);
    const long long qhi = __shfl_sync(FULL, q, f < 32 ? f : 31);
    if (f > 0) lo = qlo + 1;
    if (f < 32) hi = qhi;
  }
  return lo;
}

// min(k, floor(factor * M) + offset, S - n - 1) [, D - M]; Model Runner V2
// drafts: k and the context only.
__device__ __forceinline__ int bo_cap(const ProposeArgs &a, int M, int n) {
  long long c = a.fixed ? (long long)a.k : min((long long)a.k, a.fN * M / a.fD + a.offset);
  long long room = (long long)a.S - n - 1;
  if (room < 0) room = 0;
  c = min(c, room);
  if (a.depth_sum_cap && !a.fixed) c = min(c, (long long)a.D - M);
  return c < 0 ? 0 : (int)c;
}

// The distinct lengths covering thresholds 1..nb from a length histogram.
__device__ int pick_lengths(const int *h, int top, int minlen, int nb, int *len, int *tot) {
  int c = 0, cum = 0;
  for (int m = top; m >= minlen && cum < nb; --m) {
    if (h[m] == 0) continue;
    cum += h[m];
    len[c] = m;
    tot[c] = cum;
    ++c;
  }
  return c;
}

// Continuation token of end o at depth d (-1: none).  src 1: the row; src 2:
// the corpus (o >= 0 a snapshot end, o < 0 the delta end -(o + 1)).
__device__ __forceinline__ int bo_cont(const BoRow &r, int src, int o, int d) {
  if (src == 1) {
    const int q = o + 1 + d;
    return q <= r.n - 1 ? r.row[q] : -1;
  }
  if (o >= 0) {
    const long long q = (long long)o + 1 + d;
    if (q >= r.N) return -1;
    const int v = __ldg(r.X + q);
    return v == r.Z ? -1 : v;
  }
  const long long q = (long long)(-(o + 1)) + 1 + d;
  if (q >= r.dv) return -1;
  const int v = y_at(r, q);
  return v == r.Z ? -1 : v;
}

// Frequency-greedy expansion of candidate ci by one warp: at each depth the
// most frequent continuation among the surviving ends (ties: the smallest
// id), kept while its share of the c0 ends reaches min_token_prob (Model
// Runner V2 drafts: while any end continues), up to the candidate's cap.
__device__ void bo_vote(const ProposeArgs &a, const BoRow &r, BoShared &s, int ci, int src, int warp,
                        int lane) {
  const int c0 = s.cnt[ci], M = s.len[ci];
  const int cap = bo_cap(a, M, r.n);
  int *hkey = s.u.ht[warp].key;
  int *hcnt = s.u.ht[warp].cnt;
  bool alive[MAX_R / 32];
  int v[MAX_R / 32];
#pragma unroll
  for (int u = 0; u < MAX_R / 32; ++u) alive[u] = lane + 32 * u < c0;
  int len = 0;
  long long sum = 0;
  int ahead[MAX_R / 32][4];  // continuation tokens of depths d0 .. d0+3, read together
  for (int d = 0; d < cap; ++d) {
    if ((d & 3) == 0) {
#pragma unroll
      for (int u = 0; u < MAX_R / 32; ++u) {
        const int o = alive[u] ? s.occ[ci][lane + 32 * u] : 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          ahead[u][q] = alive[u] && d + q < cap ? bo_cont(r, src, o, d + q) : -1;
      }
    }
    bool any = false;
#pragma unroll
    for (int u = 0; u < MAX_R / 32; ++u) {
      v[u] = -1;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if ((d & 3) == q && alive[u]) v[u] = ahead[u][q];
      any |= v[u] >= 0;
    }
    if (!__any_sync(FULL, any)) break;
    // The first continuing end's token: when more than half of the continuing
    // ends share it, it is the most frequent (and no other ties it).
    int np = 0, ref = -1;
#pragma unroll
    for (int u = 0; u < MAX_R / 32; ++u) {
      const unsigned m = __ballot_sync(FULL, v[u] >= 0);
      np += __popc(m);
      const int t = __shfl_sync(FULL, v[u], m ? __ffs(m) - 1 : 0);
      if (ref < 0 && m) ref = t;
    }
    int nref = 0;
#pragma unroll
    for (int u = 0; u < MAX_R / 32; ++u) nref += __popc(__ballot_sync(FULL, v[u] == ref));
    int bc, bt;
    if (2 * nref > np) {
      bc = nref;
      bt = ref;
    } else {
      // count each continuation token in a table of MAX_R slots (>= the
      // distinct tokens, at most c0 <= MAX_R, so an insert always finds its slot)
#pragma unroll
      for (int u = 0; u < MAX_R / 32; ++u) {
        hkey[lane + 32 * u] = -1;
        hcnt[lane + 32 * u] = 0;
      }
      __syncwarp();
      int hs[MAX_R / 32];
#pragma unroll
      for (int u = 0; u < MAX_R / 32; ++u) {
        hs[u] = -1;
        if (v[u] < 0) continue;
        static_assert(MAX_R == 128, "the slot hash takes 7 bits");
        unsigned h = ((unsigned)v[u] * 2654435761u) >> 25;
        for (;;) {
          const int prev = atomicCAS(&hkey[h], -1, v[u]);
          if (prev == -1 || prev == v[u]) break;
          h = (h + 1) & (MAX_R - 1);
        }
        atomicAdd(&hcnt[h], 1);
        hs[u] = (int)h;
      }
      __syncwarp();
      int best = 0, cu[MAX_R / 32];
#pragma unroll
      for (int u = 0; u < MAX_R / 32; ++u) {
        cu[u] = hs[u] >= 0 ? hcnt[hs[u]] : 0;
        best = max(best, cu[u]);
      }
      bc = (int)__reduce_max_sync(FULL, (unsigned)best);
      unsigned mine = UINT_MAX;
#pragma unroll
      for (int u = 0; u < MAX_R / 32; ++u)
        if (v[u] >= 0 && cu[u] == bc) mine = min(mine, (unsigned)v[u]);
      bt = (int)__reduce_min_sync(FULL, mine);
      __syncwarp();  // every lane done reading the table before the next depth clears it
    }
    if (!a.fixed && (long long)bc * a.pD < a.pN * (long long)c0) break;
    if (lane == 0) {
      s.v.d.tok[ci][d] = bt;
      s.v.d.cnt[ci][d] = bc;
    }
    sum += bc;
    ++len;
#pragma unroll
    for (int u = 0; u < MAX_R / 32; ++u) alive[u] = v[u] == bt;
  }
  if (lane == 0) {
    s.dlen[ci] = len;
    s.dsum[ci] = sum;
  }
}

// Ends and lengths of interval hits p0 + q * BO_THREADS (q < 4; l = -1 past
// hi): the suffix-array entries read together and the lengths from the
// on-chip cache, or beyond it both evaluated again as in the first pass (the
// four hits of a call lie on one side of the cache's end: p0 - lo is
// tid + a multiple of 4 * BO_THREADS, and the cache size is a multiple of it).
__device__ __forceinline__ void hit_ends(const BoRow &r, const BoShared &s, int m, long long lo,
                                         long long p0, long long hi, long long e[4], int l[4]) {
  if (p0 - lo >= BO_LCACHE) {
    hit_lens(r, m, p0, hi, l, e);
    return;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const long long p = p0 + (long long)q * BO_THREADS;
    e[q] = p < hi ? (long long)__ldg(r.SA + p) + m - 1 : -1;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const long long p = p0 + (long long)q * BO_THREADS;
    l[q] = p >= hi ? -1 : (int)s.u.lc[p - lo];
  }
}

// One chunk of a backward scan: thread tid holds end `val` with length l
// (ends in descending recency by tid).  Each candidate c < ncand of list
// `off` (length s.len[off + c]) appends the chunk's ends reaching its length,
// in order, up to R.  Returns, in every thread, whether every list now holds
// min(R, target[c]) ends.
__device__ bool bo_collect(BoShared &s, int off, int ncand, const int *target, int l, int val, int R,
                           int tid, int warp, int lane) {
  for (int c = 0; c < ncand; ++c) {
    const unsigned bal = __ballot_sync(FULL, l >= s.len[off + c]);
    if (lane == 0) s.wb[c][warp] = bal;
  }
  __syncthreads();
  for (int c = 0; c < ncand; ++c) {
    if (l < s.len[off + c]) continue;
    int rank = __popc(s.wb[c][warp] & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) rank += __popc(s.wb[c][w]);
    const int slot = s.cnt[off + c] + rank;
    if (slot < R) s.occ[off + c][slot] = val;
  }
  __syncthreads();
  bool full = true;
  if (tid < ncand) {  // thread c: candidate c's count
    int t = 0;
    for (int w = 0; w < BO_WARPS; ++w) t += __popc(s.wb[tid][w]);
    const int cn = min(R, s.cnt[off + tid] + t);
    s.cnt[off + tid] = cn;
    full = cn >= min(R, target[tid]);
  }
  return __syncthreads_and(full) != 0;
}

__global__ void __launch_bounds__(BO_THREADS, 2) backoff_kernel(const ProposeArgs a) {
  __shared__ BoShared s;
  // the match lengths of row ends j < rlc (byte j), from the length pass, for
  // the backward scan that collects the row's candidates
  extern __shared__ unsigned char s_rl[];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = a.S, D = a.D, R = a.R, k = a.k, nb = a.nb;
  const int rlc = min(S, BO_RLCAP);
  int32_t *row = a.tok + (size_t)b * S;
  const CorpusDesc *cd = a.desc;
  if (warp == 0) {
    // the step's update (with sampled ids): the accepted ids appended to the
    // row; the tail (the last D tokens, newest first) is the appended ids
    // followed by the row's old last tokens, read before the update
    int n = a.ntok[b];
    uint32_t fl = 0;
    if (n < 0) { n = 0; fl |= SGD_ERR_NUM_TOKENS; }
    if (n > S) { n = S; fl |= SGD_ERR_NUM_TOKENS; }
    const int n_old = n, dl0 = min(D, n_old);
    int ot[MAX_D / 32];
#pragma unroll
    for (int u = 0; u < MAX_D / 32; ++u) {
      const int i = lane + 32 * u;
      ot[u] = i < dl0 ? row[n_old - 1 - i] : 0;
    }
    if (a.do_update) n = update_row_warp(row, n, a.sampled + (size_t)b * a.T, a.T, S, a.V, lane, fl, s.tail, D);
    const int ca = n - n_old, dl1 = min(D, n);
#pragma unroll
    for (int u = 0; u < MAX_D / 32; ++u) {
      const int i = lane + 32 * u;
      if (i < dl0 && i + ca < dl1) s.tail[i + ca] = ot[u];
    }
    if (lane == 0) {
      if (a.do_update) a.ntok[b] = n;
      if (fl) atomicOr(a.err, fl);
      s.n = n;
      s.ds = 0;
      s.dv = 0;
      if (a.dcap > 0 && cd != nullptr) {  // the docs placed since the snapshot was linearised
        const DeltaView v = delta_view(*a.rs, cd->lin_pushed, cd->lin_wp, a.C, a.doc_start);
        s.ds = v.start;
        s.dv = (int)min(v.len, a.dcap);
      }
      s.lo = 0;
      s.hi = 0;
      s.win = -1;
    }
  }
  for (int i = tid; i <= MAX_D; i += BO_THREADS) {
    s.hs[i] = 0;
    s.hc[i] = 0;
    s.hd[i] = 0;
  }
  for (int i = tid; i < BO_TOPC * 256; i += BO_THREADS) s.v.top[i >> 8][i & 255] = 0;
  __syncthreads();
  const int n = s.n;
  int32_t *dr = a.drafts + (size_t)b * k;
  float *pr = a.probs ? a.probs + (size_t)b * k : nullptr;
  if (!((a.active == nullptr || a.active[b] != 0) && n > 0)) {
    for (int d = tid; d < k; d += BO_THREADS) {
      dr[d] = -1;
      if (pr) pr[d] = 0.f;
    }
    if (tid == 0) {
      a.num_valid[b] = 0;
      if (a.score) a.score[b] = 0.f;
      if (a.match_info) { a.match_info[2 * b] = 0; a.match_info[2 * b + 1] = 0; }
    }
    return;
  }
  const int dl = min(D, n);
  BoRow r;
  r.row = row;
  r.n = n;
  r.dl = dl;
  r.X = cd != nullptr ? cd->text : nullptr;
  r.SA = cd != nullptr ? cd->sa : nullptr;
  r.K = cd != nullptr ? cd->keys : nullptr;
  r.N = cd != nullptr ? cd->n : 0;
  r.ring = a.ring;
  r.C = a.C;
  r.ds = s.ds;
  r.dv = s.dv;
  r.Z = a.V;
  r.tail = s.tail;
  const bool snap = r.N >= 2 && n >= 2 && D >= 2;
  const bool delta = r.dv >= 2 && n >= 2 && D >= 2;
  __syncthreads();

  // ---- match lengths: the row's ends, the interval of the last two tokens, the delta ----
  const bool grams = snap && !delta && cd->gt != nullptr;
  if (grams && warp < 3) {  // the last 2-, 3-, 4-gram (warp 0, 1, 2)
    const int m = 2 + warp;
    long long glo = 0, ghi = 0;
    int blk = -2;
    bool endless = dl >= m;  // (no suffix holds KEY_END: a pattern with it has no hit)
    for (int i = 0; i < m && endless; ++i) endless = s.tail[i] != KEY_END;
    if (endless) {
      const int4 P = make_int4(s.tail[m - 1], s.tail[m - 2], m >= 3 ? s.tail[m - 3] : 0,
                               m >= 4 ? s.tail[m - 4] : 0);
      gt_lookup(cd->gt, cd->gt_mask, P, m, lane, glo, ghi, blk);
    }
    if (lane == 0) {
      s.glo[warp] = glo;
      s.ghi[warp] = ghi;
      if (warp < 2) s.gblk[warp] = cd->gd != nullptr ? blk : -2;
    }
  } else if (snap && !grams && warp < 2) {
    const long long q = pair_bound(r.K, r.N, s.tail[1], s.tail[0], warp == 1, lane);
    if (lane == 0) (warp == 0 ? s.lo : s.hi) = q;
  }
  for (int j0 = tid; j0 <= n - 2; j0 += 4 * BO_THREADS) {  // four ends' first tokens at once
    int x[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + q * BO_THREADS;
      x[q] = j <= n - 2 ? row[j] : -1;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + q * BO_THREADS;
      int l = 0;
      if (x[q] == s.tail[0]) {
        l = self_len(r, j);
        atomicAdd(&s.hs[l], 1);
      }
      if (j <= n - 2 && j < rlc) s_rl[j] = (unsigned char)l;
    }
  }
  // The delta in 128-token windows of the ring (window w holds Y indices
  // [w * WIN - off, w * WIN - off + WIN)); an end matching >= 2 tokens ends
  // the row's last pair, whose bucket is then set in its window's gram
  // signature, so the windows without it are skipped (exactly).
  const int d_off = (int)(r.ds % WIN);
  const int d_nw = delta ? (d_off + r.dv - 1) / WIN + 1 : 0;
  const int d_nrw = (int)(r.C / WIN);
  const unsigned d_b2 = delta ? sig_bucket(2, s.tail[0], s.tail[1], 0, 0) : 0u;
  auto d_cand = [&](int w) {  // window w may hold an end matching >= 2 tokens
    const int rw = (int)((r.ds / WIN + w) % d_nrw);
    return ((__ldg(a.sig + (size_t)(d_b2 >> 5) * d_nrw + rw) >> (d_b2 & 31)) & 1u) != 0;
  };
  for (int wb = 0; wb < d_nw; wb += BO_THREADS) {
    const int w = wb + tid;
    const int nl = block_compact(w < d_nw && d_cand(w), w, s.wl, s.wb[0], warp, lane);
    for (int i = warp; i < nl; i += BO_WARPS) {  // a warp per listed window, 4 tokens per lane
      const int wi = s.wl[i];
      const long long rw = (r.ds / WIN + wi) % d_nrw;
      const int4 v = __ldg(reinterpret_cast<const int4 *>(r.ring + rw * WIN) + lane);
      const int tok[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const long long u = (long long)wi * WIN - d_off + 4 * lane + c;
        if (u < 0 || u > r.dv - 2 || tok[c] != s.tail[0]) continue;
        const int l = delta_len(r, u);
        if (l >= 2) {
          atomicAdd(&s.hc[l], 1);
          atomicAdd(&s.hd[l], 1);
        }
      }
    }
    __syncthreads();
  }
  __syncthreads();
  // the walked gram: the shortest without a draft block (lengths below it
  // come from the blocks)
  int wm = 2;
  if (grams && s.gblk[0] >= 0) wm = s.gblk[1] >= 0 ? 4 : 3;
  const long long lo = grams ? (wm <= dl ? s.glo[wm - 2] : 0) : s.lo;
  const long long hi = grams ? (wm <= dl ? s.ghi[wm - 2] : 0) : s.hi;
  // the radix selection's first digit (end bits sh_top and up) is counted here
  // too, per length class, so that its first pass needs no walk of the interval
  const int sh_top = snap ? ((64 - __clzll(r.N - 1) + 7) / 8 - 1) * 8 : 0;
  for (long long p0 = lo + tid; p0 < hi; p0 += 4LL * BO_THREADS) {
    int l[4];
    long long e[4];
    hit_lens(r, wm, p0, hi, l, e);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long p = p0 + (long long)j * BO_THREADS;
      if (l[j] < 0) continue;
      if (p - lo < BO_LCACHE) s.u.lc[p - lo] = (unsigned char)l[j];
      if (l[j] > 0) {
        atomicAdd(&s.hc[l[j]], 1);
        atomicAdd(&s.v.top[min(l[j], 6) - 2][(e[j] >> sh_top) & 255], 1);
      }
    }
  }
  __syncthreads();

  const int k4 = (k + 3) & ~3;
  auto gblock = [&](int m) { return cd->gd + (size_t)s.gblk[m - 2] * gd_ints(k); };
  if (wm > 2 && tid == 0) {
    // ends of exactly m < wm tokens: the valid ends of the m-gram less those
    // of the (m + 1)-gram (counted by the walk for m + 1 = wm)
    int walked = 0;
    for (int L = wm; L <= dl; ++L) walked += s.hc[L];
    const int q2 = __ldg(gblock(2) + 2);
    if (wm == 3) {
      s.hc[2] = q2 - walked;
    } else {
      const int q3 = __ldg(gblock(3) + 2);
      s.hc[2] = q2 - q3;
      s.hc[3] = q3 - walked;
    }
  }
  __syncthreads();

  // ---- candidate lengths: thresholds 1..nb of each path ----
  if (tid == 0) s.ns = pick_lengths(s.hs, dl, 1, nb, s.len, s.tot);
  if (tid == 32) s.nc = pick_lengths(s.hc, dl, 2, nb, s.len + MAX_BACKOFF, s.tot + MAX_BACKOFF);
  if (tid < BO_CANDS) s.cnt[tid] = 0;
  __syncthreads();
  const int ns = s.ns, nc = s.nc;
  if (tid < nc) {  // the delta's ends reaching each corpus length
    int t = 0;
    for (int m = s.len[MAX_BACKOFF + tid]; m <= dl; ++m) t += s.hd[m];
    s.dtot[MAX_BACKOFF + tid] = t;
  }
  __syncthreads();

  // ---- the row's candidates: their R most recent ends, by a backward scan ----
  if (ns > 0)
    for (int base = n - 2; base >= 0; base -= BO_THREADS) {
      const int j = base - tid;
      const int l = j < 0 ? 0 : (j < rlc ? (int)s_rl[j] : self_len(r, j));
      if (bo_collect(s, 0, ns, s.tot, l, j, R, tid, warp, lane)) break;
    }
  // ---- the corpus's: the delta's ends first (the most recent), then the snapshot's ----
  if (nc > 0 && delta) {
    bool stop = true;  // (no delta end reaches any corpus length)
    for (int c = 0; c < nc; ++c) stop &= s.dtot[MAX_BACKOFF + c] == 0;
    // listed windows newest first, four per chunk: thread tid takes position
    // WIN - 1 - tid % WIN of the chunk's window tid / WIN (recency falls with tid)
    for (int wb = 0; wb < d_nw && !stop; wb += BO_THREADS) {
      const int w = d_nw - 1 - wb - tid;
      const int nl = block_compact(w >= 0 && d_cand(w), w, s.wl, s.wb[0], warp, lane);
      for (int c0 = 0; c0 < nl; c0 += BO_THREADS / WIN) {
        const int li = c0 + tid / WIN;
        long long u = -1;
        if (li < nl) u = (long long)s.wl[li] * WIN - d_off + (WIN - 1 - tid % WIN);
        const bool ok = u >= 0 && u <= r.dv - 2;
        stop = bo_collect(s, MAX_BACKOFF, nc, s.dtot + MAX_BACKOFF, ok ? delta_len(r, u) : 0,
                          (int)(-(u + 1)), R, tid, warp, lane);
        if (stop) break;
      }
      __syncthreads();  // (the list is rewritten by the next batch)
    }
  }
  if (nc > 0 && snap && hi > lo) {
    if (tid < nc) {
      const int c = MAX_BACKOFF + tid;
      const int room = R - s.cnt[c], xq = s.tot[c] - s.dtot[c];
      // (a length below the walked gram's: its candidate is the gram's block)
      s.mode[tid] = room <= 0 || xq <= 0 || s.len[c] < wm ? 0 : (xq <= room ? 1 : 2);
      s.need[tid] = min(room, xq);
      s.pref[tid] = 0;
    }
    __syncthreads();
    bool radix = false;
    for (int c = 0; c < nc; ++c) radix |= s.mode[c] == 2;
    bool classed = true;  // every selecting candidate's length within the counted classes
    for (int c = 0; c < nc; ++c) classed &= s.mode[c] != 2 || s.len[MAX_BACKOFF + c] <= 6;
    if (radix) {  // the need most recent qualifying ends: MSB-first radix selection on e
      for (int sh = sh_top; sh >= 0; sh -= 8) {
        if (sh == sh_top && classed) {  // the first digit from the length pass's counts
          for (int i = tid; i < nc * 256; i += BO_THREADS) {
            const int c = i >> 8, d = i & 255;
            int t = 0;
            if (s.mode[c] == 2)
              for (int k = s.len[MAX_BACKOFF + c] - 2; k < BO_TOPC; ++k) t += s.v.top[k][d];
            s.hist[c][d] = t;
          }
          __syncthreads();
        } else {
          for (int i = tid; i < nc * 256; i += BO_THREADS) s.hist[i >> 8][i & 255] = 0;
          __syncthreads();
          for (long long p0 = lo + tid; p0 < hi; p0 += 4LL * BO_THREADS) {
            long long e[4];
            int l[4];
            hit_ends(r, s, wm, lo, p0, hi, e, l);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              for (int c = 0; c < nc; ++c)
                if (s.mode[c] == 2 && l[q] >= s.len[MAX_BACKOFF + c] &&
                    (e[q] >> (sh + 8)) == (s.pref[c] >> (sh + 8)))
                  atomicAdd(&s.hist[c][(e[q] >> sh) & 255], 1);
          }
          __syncthreads();
        }
        if (warp < nc && s.mode[warp] == 2) {
          // warp c picks candidate c's digit: lane L sums bins 255 - 8L .. 248 - 8L,
          // a scan over the lanes finds the lane where the count from the top
          // reaches `need`, and that lane walks its eight bins
          const int c = warp;
          int hb[8], loc = 0;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            hb[q] = s.hist[c][255 - 8 * lane - q];
            loc += hb[q];
          }
          int incl = loc;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += y;
          }
          const int need = s.need[c];
          const int excl = incl - loc;
          if (excl < need && incl >= need) {  // exactly one lane
            int cum = excl;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              if (cum + hb[q] >= need) {
                s.pref[c] |= (long long)(255 - 8 * lane - q) << sh;
                s.need[c] = need - cum;
                break;
              }
              cum += hb[q];
            }
          }
        }
        __syncthreads();
      }
    }
    for (long long p0 = lo + tid; p0 < hi; p0 += 4LL * BO_THREADS) {
      long long e[4];
      int l[4];
      hit_ends(r, s, wm, lo, p0, hi, e, l);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        for (int c = 0; c < nc; ++c) {
          const int m = s.mode[c];
          if (m == 0 || l[q] < s.len[MAX_BACKOFF + c] || (m == 2 && e[q] < s.pref[c])) continue;
          const int slot = atomicAdd(&s.cnt[MAX_BACKOFF + c], 1);
          if (slot < R) s.occ[MAX_BACKOFF + c][slot] = (int)e[q];
        }
    }
    __syncthreads();
    if (tid < nc) s.cnt[MAX_BACKOFF + tid] = min(R, s.cnt[MAX_BACKOFF + tid]);  // (exactly room or fewer)
    __syncthreads();
  }
  if (wm > 2 && tid < nc && s.len[MAX_BACKOFF + tid] < wm)  // a block's candidate: its c0 = min(Q, R)
    s.cnt[MAX_BACKOFF + tid] = __ldg(gblock(s.len[MAX_BACKOFF + tid]));
  __syncthreads();

  // ---- every candidate voted (one warp each), the best score wins ----
  for (int q = warp; q < ns + nc; q += BO_WARPS) {
    const int ci = q < ns ? q : MAX_BACKOFF + (q - ns);
    if (q >= ns && s.len[ci] < wm) {
      // the gram's block: its vote to depth k, cut at this candidate's cap
      // (the vote at a depth never depends on where it will stop)
      const int32_t *gb = gblock(s.len[ci]);
      const int len = min(__ldg(gb + 1), bo_cap(a, s.len[ci], n));
      unsigned part = 0;
      for (int d = lane; d < len; d += 32) {
        const int cnt = __ldg(gb + 4 + k4 + d);
        s.v.d.tok[ci][d] = __ldg(gb + 4 + d);
        s.v.d.cnt[ci][d] = cnt;
        part += (unsigned)cnt;
      }
      const unsigned sum = __reduce_add_sync(FULL, part);
      if (lane == 0) {
        s.dlen[ci] = len;
        s.dsum[ci] = sum;
      }
      continue;
    }
    bo_vote(a, r, s, ci, q < ns ? 1 : 2, warp, lane);
  }
  __syncthreads();
  if (tid == 0) {
    int w = -1;
    for (int q = 0; q < ns + nc; ++q) {  // the row's first, longest first
      const int ci = q < ns ? q : MAX_BACKOFF + (q - ns);
      if (w < 0) {
        w = ci;
        continue;
      }
      const long long lhs = s.dsum[ci] * s.cnt[w], rhs = s.dsum[w] * s.cnt[ci];
      if (lhs > rhs || (lhs == rhs && s.len[ci] > s.len[w])) w = ci;
    }
    s.win = w;
  }
  __syncthreads();
  const int w = s.win;
  const int len = w >= 0 ? s.dlen[w] : 0;
  const int fill = a.fixed ? s.tail[0] : -1;
  for (int d = tid; d < k; d += BO_THREADS) {
    dr[d] = d < len ? s.v.d.tok[w][d] : fill;
    if (pr) pr[d] = d < len ? (float)((double)s.v.d.cnt[w][d] / (double)s.cnt[w]) : 0.f;
  }
  if (tid == 0) {
    a.num_valid[b] = a.fixed ? k : len;
    if (a.score) a.score[b] = w >= 0 ? (float)((double)s.dsum[w] / (double)s.cnt[w]) : 0.f;
    if (a.match_info) {
      a.match_info[2 * b] = w >= 0 ? s.len[w] : 0;
      a.match_info[2 * b + 1] = w < 0 ? 0 : (w < MAX_BACKOFF ? 1 : 2);
    }
  }
}

}  // namespace

cudaError_t backoff_set_smem_limit() {
  // (and the largest shared memory carveout: two CTAs per SM, one launch for
  // every row of a batch of up to two per SM)
  cudaError_t e = cudaFuncSetAttribute((const void *)backoff_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, BO_RLCAP);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute((const void *)backoff_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t launch_backoff(const ProposeArgs &a, cudaStream_t st) {
  if (a.B <= 0) return cudaSuccess;
  const size_t dyn = (size_t)((min(a.S, BO_RLCAP) + 15) & ~15);
  backoff_kernel<<<a.B, BO_THREADS, dyn, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sgd
