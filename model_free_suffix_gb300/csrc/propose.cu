// propose.cu -- the per-step drafting kernel (update + self match + corpus
// probe + frequency-greedy expansion), one CTA per request row.
//
// Sources (page title, section):
//   "SuffixGPU" (suffix-gpu 0.1.1, PyPI): How it works, steps 1-3; Highlights.
//   "Suffix Decoding" (vLLM docs): Model Runner V2 (longest suffix up to
//     max_tree_depth; corpus probe on the last 2 / last 4 tokens extended to
//     the longest match; the longer match wins).
//   "vLLM Suffix Decoding 投机解码实战": section 4 (max_spec_factor,
//     min_token_prob), section 5 (max_model_len - num_tokens - 1).
//
// CTA layout: `nself` warps scan the row for the self match (warp-per-segment,
// int4 loads, ballot early-outs) while, when a corpus exists, 4 more warps
// run the suffix-array probes (32-ary searches).  The whole CTA then scans
// the probe interval with batched loads, and warp 0 runs the depth-wise
// vote.  All decisions are integer; the only floating-point values are the
// reported probabilities and score.
#include <climits>

#include "sgd_internal.h"

namespace sgd {

namespace {

constexpr int LCAP = 16384;  // interval entries whose match length is cached on chip

__device__ __forceinline__ int4 load_win(const int32_t *row, int widx, int lane, int S) {
  const int p = widx * WIN + 4 * lane;
  if (widx < 0 || p >= S) return make_int4(0, 0, 0, 0);
  return *reinterpret_cast<const int4 *>(row + p);
}

// value of component `vc`/`vp` held by lane `src` of the current window, or
// of the window below it when src < 0 (src >= -32)
__device__ __forceinline__ int pick(int vc, int vp, int src) {
  const int a = __shfl_sync(FULL, vc, src & 31);
  const int b = __shfl_sync(FULL, vp, src & 31);
  return src >= 0 ? a : b;
}

// Tokens at positions (4*lane + c) - i, c = 0..3, relative to the window
// start, for 1 <= i <= 127.
__device__ __forceinline__ void shifted(const int4 &c, const int4 &p, int lane, int i, int &v0,
                                        int &v1, int &v2, int &v3) {
  const int q = i >> 2;
  const int sA = lane - q, sB = lane - q - 1;
  switch (i & 3) {
    case 0:
      v0 = pick(c.x, p.x, sA); v1 = pick(c.y, p.y, sA); v2 = pick(c.z, p.z, sA); v3 = pick(c.w, p.w, sA);
      break;
    case 1:
      v0 = pick(c.w, p.w, sB); v1 = pick(c.x, p.x, sA); v2 = pick(c.y, p.y, sA); v3 = pick(c.z, p.z, sA);
      break;
    case 2:
      v0 = pick(c.z, p.z, sB); v1 = pick(c.w, p.w, sB); v2 = pick(c.x, p.x, sA); v3 = pick(c.y, p.y, sA);
      break;
    default:
      v0 = pick(c.y, p.y, sB); v1 = pick(c.z, p.z, sB); v2 = pick(c.w, p.w, sB); v3 = pick(c.x, p.x, sA);
      break;
  }
}

// One 128-token window of the self match.  L(j) for the 4 ends j this lane
// holds: the length of the common run of t[j-i] and tail[i] = t[n-1-i],
// bounded by D and by j + 1; ends j >= J = n - 1 do not count.  Keeps the
// warp's running maximum Mw and its most recent ends (descending) in `list`.
__device__ __forceinline__ void self_window(int wi, const int4 &cur, const int4 &prv, int lane,
                                            int J, int D, const int *s_tail, int t0, int R,
                                            int *list, int &Mw, int &cnt) {
  const int base = wi * WIN + 4 * lane;
  bool a0 = cur.x == t0 && base + 0 < J;
  bool a1 = cur.y == t0 && base + 1 < J;
  bool a2 = cur.z == t0 && base + 2 < J;
  bool a3 = cur.w == t0 && base + 3 < J;
  if (!__any_sync(FULL, a0 | a1 | a2 | a3)) return;
  int L0 = a0, L1 = a1, L2 = a2, L3 = a3;
  for (int i = 1; i < D; ++i) {
    const int ti = s_tail[i];
    int v0, v1, v2, v3;
    shifted(cur, prv, lane, i, v0, v1, v2, v3);
    a0 = a0 && base + 0 >= i && v0 == ti;
    a1 = a1 && base + 1 >= i && v1 == ti;
    a2 = a2 && base + 2 >= i && v2 == ti;
    a3 = a3 && base + 3 >= i && v3 == ti;
    L0 += a0; L1 += a1; L2 += a2; L3 += a3;
    if (!__any_sync(FULL, a0 | a1 | a2 | a3)) break;
  }
  const int lm = max(max(L0, L1), max(L2, L3));
  const int wm = (int)__reduce_max_sync(FULL, (unsigned)lm);
  if (wm > Mw) { Mw = wm; cnt = 0; }
  if (wm == Mw && cnt < R) {
    const int f0 = L0 == wm, f1 = L1 == wm, f2 = L2 == wm, f3 = L3 == wm;
    const int q = f0 + f1 + f2 + f3;
    int x = q;  // inclusive suffix sum over lanes >= lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_down_sync(FULL, x, off);
      if (lane + off < 32) x += y;
    }
    const int total = __shfl_sync(FULL, x, 0);
    int slot = cnt + (x - q);
    if (f3) { if (slot < R) list[slot] = base + 3; ++slot; }
    if (f2) { if (slot < R) list[slot] = base + 2; ++slot; }
    if (f1) { if (slot < R) list[slot] = base + 1; ++slot; }
    if (f0) { if (slot < R) list[slot] = base + 0; ++slot; }
    cnt = min(R, cnt + total);
  }
}

// Warp w scans windows [wlo, whi] from the top down (most recent first).
__device__ void self_scan(const int32_t *row, int n, int S, int D, int R, const int *s_tail, int *list,
                          int w, int nself, int lane, int &Mw, int &cnt) {
  Mw = 0;
  cnt = 0;
  const int J = n - 1;
  if (J <= 0) return;
  const int nwin = (J + WIN - 1) / WIN;
  const int per = (nwin + nself - 1) / nself;
  const int wlo = w * per;
  const int whi = min(nwin, wlo + per) - 1;
  if (whi < wlo) return;
  const int t0 = s_tail[0];
  const int4 z = make_int4(0, 0, 0, 0);
  int4 b0 = load_win(row, whi, lane, S);
  int4 b1 = load_win(row, whi - 1, lane, S);
  int4 b2 = whi - 2 >= wlo - 1 ? load_win(row, whi - 2, lane, S) : z;
  int4 b3 = whi - 3 >= wlo - 1 ? load_win(row, whi - 3, lane, S) : z;
  int4 b4 = whi - 4 >= wlo - 1 ? load_win(row, whi - 4, lane, S) : z;
  for (int wi = whi; wi >= wlo; --wi) {
    const int nx = wi - 5;
    const int4 nb = nx >= wlo - 1 ? load_win(row, nx, lane, S) : z;
    self_window(wi, b0, b1, lane, J, D, s_tail, t0, R, list, Mw, cnt);
    b0 = b1; b1 = b2; b2 = b3; b3 = b4; b4 = nb;
  }
}

// Three-way compare of the suffix starting at SA[q] with pattern P[0..m):
// token by token as signed int32; running off the text sorts first.
__device__ __forceinline__ int cmp_suffix(const int32_t *SA, const int32_t *X, long long N, long long q,
                                          const int *P, int m) {
  const long long i = __ldg(SA + q);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    if (u >= m) break;
    if (i + u >= N) return -1;
    const int x = __ldg(X + i + u);
    if (x != P[u]) return x < P[u] ? -1 : 1;
  }
  return 0;
}

// First q in [0, N) whose suffix compares >= P (upper = false) or > P
// (upper = true) on its first m tokens; N if none.  A warp probes 32 evenly
// spaced positions per step, narrowing the range 33-fold.
__device__ long long kary_search(const int32_t *SA, const int32_t *X, long long N, const int *P, int m,
                                 bool upper, int lane) {
  long long lo = 0, hi = N;
  while (lo < hi) {
    const long long len = hi - lo;
    const bool small = len <= 32;
    const long long q = small ? lo + lane : lo + (len * (lane + 1)) / 33;
    bool pr = false;
    if (!small || lane < len) {
      const int c = cmp_suffix(SA, X, N, q, P, m);
      pr = upper ? (c > 0) : (c >= 0);
    }
    const unsigned bal = __ballot_sync(FULL, pr);
    if (small) return bal ? lo + (__ffs(bal) - 1) : hi;
    if (bal == 0) {
      lo = __shfl_sync(FULL, q, 31) + 1;
    } else {
      const int f = __ffs(bal) - 1;
      const long long qf = __shfl_sync(FULL, q, f);
      const long long qp = __shfl_sync(FULL, q, f > 0 ? f - 1 : 0);
      hi = qf;
      if (f > 0) lo = qp + 1;
    }
  }
  return lo;
}

// Backward extension of a corpus end e already known to match l0 tokens.
__device__ __forceinline__ int extend(const int32_t *X, long long e, int l0, const int *s_tail, int n,
                                      int D) {
  const long long lim = min((long long)min(D, n), e + 1);
  int L = l0;
  while (L < lim && __ldg(X + e - L) == s_tail[L]) ++L;
  return L;
}

// Corpus end behind SA entry p for a pattern of length lvl, if it has a
// continuation (X[e+1] != Z); returns its match length, or 0.
__device__ __forceinline__ int corpus_entry(const int32_t *SA, const int32_t *X, long long N, int Z,
                                            long long p, int lvl, const int *s_tail, int n, int D,
                                            long long &e) {
  e = (long long)__ldg(SA + p) + lvl - 1;
  if (e + 1 >= N) return 0;
  if (__ldg(X + e + 1) == Z) return 0;
  return extend(X, e, lvl, s_tail, n, D);
}

// Match length of every end in the SA interval [lo, hi) of a pattern of
// length lvl, by the whole CTA.  Each thread takes 4 entries per round and
// issues their loads together (SA entries, then the continuation token and
// the first token before the pattern), so a long interval costs a few
// dependent round trips per round rather than one chain per entry.  The
// length of entry lo + i (0 for an end without continuation) is kept in
// s_L[i] for i < lcap; s_lhist[L] counts the valid ends of each length.
__device__ void scan_interval(const int32_t *SA, const int32_t *X, long long N, int Z, long long lo,
                              long long hi, int lvl, const int *s_tail, int n, int D,
                              unsigned char *s_L, int lcap, int *s_lhist, int tid, int nthr) {
  const long long dn = min(D, n);
  for (long long base = lo + tid; base < hi; base += 4LL * nthr) {
    long long e[4];
    int x1[4], x0[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long p = base + (long long)u * nthr;
      e[u] = p < hi ? (long long)__ldg(SA + p) + lvl - 1 : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = e[u] >= 0 && e[u] + 1 < N;
      x1[u] = ok ? __ldg(X + e[u] + 1) : Z;
      x0[u] = ok && lvl < min(dn, e[u] + 1) ? __ldg(X + e[u] - lvl) : 0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long p = base + (long long)u * nthr;
      if (p >= hi) continue;
      int L = 0;
      if (x1[u] != Z) {
        const long long lim = min(dn, e[u] + 1);
        L = lvl;
        if (L < lim && x0[u] == s_tail[L]) {
          ++L;
          while (L < lim && __ldg(X + e[u] - L) == s_tail[L]) ++L;
        }
        atomicAdd(&s_lhist[L], 1);
      }
      if (p - lo < lcap) s_L[p - lo] = (unsigned char)L;
    }
  }
}

// Match length of SA entry p during selection: from the cache when scanned
// into it, else recomputed.
__device__ __forceinline__ int entry_len(const int32_t *SA, const int32_t *X, long long N, int Z,
                                         long long p, long long lo, int lvl, const int *s_tail, int n,
                                         int D, const unsigned char *s_L, int lcap, long long &e) {
  if (p - lo < lcap) {
    e = (long long)__ldg(SA + p) + lvl - 1;
    return s_L[p - lo];
  }
  return corpus_entry(SA, X, N, Z, p, lvl, s_tail, n, D, e);
}

// Descending bitonic sort of s[0..P2) (P2 a power of two), whole CTA.
__device__ void bitonic_desc(int *s, int P2, int tid, int nthr) {
  for (int k2 = 2; k2 <= P2; k2 <<= 1) {
    for (int j = k2 >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P2; i += nthr) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const int x = s[i], y = s[ixj];
          const bool first_half = (i & k2) == 0;
          if (first_half ? (x < y) : (x > y)) { s[i] = y; s[ixj] = x; }
        }
      }
      __syncthreads();
    }
  }
}

__device__ int update_row_warp(int32_t *row, int n, const int32_t *sp, int T, int S, int V, int lane,
                               uint32_t &fl) {
  int c = T;
  bool bad = false;
  for (int base = 0; base < T; base += 32) {
    const int i = base + lane;
    const int v = i < T ? sp[i] : 0;
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
  for (int i = lane; i < c; i += 32)
    if ((long long)n + i < S) row[n + i] = sp[i];
  if (bad) fl |= SGD_ERR_SAMPLED_TOKEN;
  return (int)min((long long)S, (long long)n + c);
}

__global__ void __launch_bounds__(128) update_kernel(int32_t *tok, int32_t *ntok, const int32_t *sampled,
                                                     int B, int T, int S, int V, uint32_t *err) {
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  int n = ntok[b];
  uint32_t fl = 0;
  if (n < 0) { n = 0; fl |= SGD_ERR_NUM_TOKENS; }
  if (n > S) { n = S; fl |= SGD_ERR_NUM_TOKENS; }
  n = update_row_warp(tok + (size_t)b * S, n, sampled + (size_t)b * T, T, S, V, lane, fl);
  if (lane == 0) {
    ntok[b] = n;
    if (fl) atomicOr(err, fl);
  }
}

__device__ __forceinline__ void propose_body(const ProposeArgs &a) {
  extern __shared__ __align__(16) int dsm[];
  __shared__ int s_wM[MAX_SELF_WARPS], s_wcnt[MAX_SELF_WARPS];
  __shared__ int s_hist[256];
  __shared__ long long s_bound[NPROBE];
  __shared__ int s_lhist[MAX_D + 1];
  __shared__ int s_n, s_Ms, s_cs, s_c0, s_q, s_sel, s_need, s_corpus_ok;

  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nthr = blockDim.x;
  const int S = a.S, R = a.R, k = a.k, D = a.D;
  int32_t *row = a.tok + (size_t)b * S;
  int *s_tail = dsm;                   // MAX_D
  int *s_wlist = s_tail + MAX_D;       // nself * R
  int *s_occ = s_wlist + a.nself * R;  // R
  int *s_run = s_occ + R;              // R
  int *s_big = s_run + R;              // max(cand_cap, R * k)
  unsigned char *s_L = reinterpret_cast<unsigned char *>(s_big + max(a.cand_cap, R * k));  // LCAP

  // ---- the row's length, and the update when fused ----
  if (warp == 0) {
    int n = a.ntok[b];
    uint32_t fl = 0;
    if (n < 0) { n = 0; fl |= SGD_ERR_NUM_TOKENS; }
    if (n > S) { n = S; fl |= SGD_ERR_NUM_TOKENS; }
    if (a.do_update) n = update_row_warp(row, n, a.sampled + (size_t)b * a.T, a.T, S, a.V, lane, fl);
    if (lane == 0) {
      if (a.do_update) a.ntok[b] = n;
      if (fl) atomicOr(a.err, fl);
      s_n = n;
    }
  }
  __syncthreads();
  const int n = s_n;
  int32_t *dr = a.drafts + (size_t)b * k;
  float *pr = a.probs ? a.probs + (size_t)b * k : nullptr;
  if (!((a.active == nullptr || a.active[b] != 0) && n > 0)) {
    for (int d = tid; d < k; d += nthr) {
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

  // ---- tail[i] = t[n-1-i] ----
  const int dl = min(D, n);
  for (int i = tid; i < dl; i += nthr) s_tail[i] = row[n - 1 - i];
  if (tid == 0) {
    s_corpus_ok = a.desc != nullptr && D >= 2 && n >= 2 && a.desc->n >= 2;
  }
  __syncthreads();

  const int Z = a.V;
  const int32_t *X = nullptr, *SA = nullptr;
  long long N = 0;
  if (s_corpus_ok) {
    X = a.desc->text;
    SA = a.desc->sa;
    N = a.desc->n;
  }

  // ---- self match (nself warps) || suffix-array probes (4 warps) ----
  if (warp < a.nself) {
    int Mw, cnt;
    self_scan(row, n, S, D, R, s_tail, s_wlist + warp * R, warp, a.nself, lane, Mw, cnt);
    if (lane == 0) { s_wM[warp] = Mw; s_wcnt[warp] = cnt; }
  } else if (s_corpus_ok) {
    const int pw = warp - a.nself;
    const bool use4 = D >= 4 && n >= 4;
    const int m = pw < 2 ? 4 : 2;
    if (pw >= 2 || use4) {
      int P[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) P[u] = u < m ? s_tail[m - 1 - u] : 0;
      const long long r = kary_search(SA, X, N, P, m, (pw & 1) != 0, lane);
      if (lane == 0) s_bound[pw] = r;
    } else if (lane == 0) {
      s_bound[pw] = 0;
    }
  }
  __syncthreads();

  // ---- merge the self scans: max length, most recent ends first ----
  if (warp == 0) {
    int Ms = 0;
    for (int w = 0; w < a.nself; ++w) Ms = max(Ms, s_wM[w]);
    int c = 0;
    if (Ms > 0) {
      for (int w = a.nself - 1; w >= 0 && c < R; --w) {
        if (s_wM[w] != Ms) continue;
        const int mm = min(s_wcnt[w], R - c);
        for (int i = lane; i < mm; i += 32) s_occ[c + i] = s_wlist[w * R + i];
        c += mm;
      }
    }
    if (lane == 0) { s_Ms = Ms; s_cs = c; }
  }
  __syncthreads();
  const int Ms = s_Ms;

  // ---- corpus: longest match among the probe hits, where it can still win ----
  // Ends with a match >= 4 are exactly the P4 hits; if none of them has a
  // continuation, valid matches of 2 or 3 are exactly the valid P2 hits.  A
  // level is scanned only if its longest possible match exceeds Ms, which
  // leaves the chosen source and its occurrences unchanged.
  int Mc = 0, lvl = 4;
  long long lo = 0, hi = 0;
  if (s_corpus_ok) {
    const int dn = min(D, n);
    const bool use4 = D >= 4 && n >= 4;
    bool have4 = false;
    for (int pass = 0; pass < 2; ++pass) {
      const int L_hi = pass == 0 ? dn : min(3, dn);
      if (pass == 0 && !use4) continue;
      if (pass == 1 && have4) break;
      if (Ms >= L_hi) break;
      const int lv = pass == 0 ? 4 : 2;
      const long long l0 = pass == 0 ? s_bound[0] : s_bound[2];
      const long long h0 = pass == 0 ? s_bound[1] : s_bound[3];
      if (h0 <= l0) continue;
      __syncthreads();  // the previous pass's histogram has been read
      for (int i = tid; i <= MAX_D; i += nthr) s_lhist[i] = 0;
      __syncthreads();
      scan_interval(SA, X, N, Z, l0, h0, lv, s_tail, n, D, s_L, LCAP, s_lhist, tid, nthr);
      __syncthreads();
      int best = 0;
      for (int L = dn; L >= 1; --L)
        if (s_lhist[L] > 0) { best = L; break; }
      if (best > 0) {
        if (pass == 0) have4 = true;
        if (best >= 2) { Mc = best; lvl = lv; lo = l0; hi = h0; }
      }
    }
  }
  int src, M;
  if (Mc > Ms) { src = 2; M = Mc; }
  else { src = Ms > 0 ? 1 : 0; M = Ms; }

  if (src == 2) {
    // the R largest ends with length Mc (cached lengths; no second random pass)
    int *cand = s_big;
    const int Q = s_lhist[Mc];
    if (Q <= a.cand_cap) {
      if (tid == 0) s_q = 0;
      __syncthreads();
      for (long long p = lo + tid; p < hi; p += nthr) {
        long long e;
        if (entry_len(SA, X, N, Z, p, lo, lvl, s_tail, n, D, s_L, LCAP, e) == Mc)
          cand[atomicAdd(&s_q, 1)] = (int)e;
      }
    } else {
      // more candidates than fit on chip: radix-select the R-th largest end
      // byte by byte, then collect the R ends at or above it
      unsigned prefix = 0, mask = 0;
      int need = R;
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += nthr) s_hist[i] = 0;
        __syncthreads();
        for (long long p = lo + tid; p < hi; p += nthr) {
          long long e;
          if (entry_len(SA, X, N, Z, p, lo, lvl, s_tail, n, D, s_L, LCAP, e) == Mc &&
              ((unsigned)e & mask) == prefix)
            atomicAdd(&s_hist[((unsigned)e >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid == 0) {
          int acc = 0;
          for (int v = 255; v >= 0; --v) {
            if (acc + s_hist[v] >= need) { s_sel = v; s_need = need - acc; break; }
            acc += s_hist[v];
          }
        }
        __syncthreads();
        prefix |= (unsigned)s_sel << shift;
        mask |= 255u << shift;
        need = s_need;
      }
      if (tid == 0) s_q = 0;
      __syncthreads();
      for (long long p = lo + tid; p < hi; p += nthr) {
        long long e;
        if (entry_len(SA, X, N, Z, p, lo, lvl, s_tail, n, D, s_L, LCAP, e) == Mc &&
            (unsigned)e >= prefix) {
          const int slot = atomicAdd(&s_q, 1);
          if (slot < a.cand_cap) cand[slot] = (int)e;
        }
      }
    }
    __syncthreads();
    const int Qc = min(s_q, a.cand_cap);
    int P2 = 1;
    while (P2 < Qc) P2 <<= 1;
    for (int i = Qc + tid; i < P2; i += nthr) cand[i] = -1;
    __syncthreads();
    bitonic_desc(cand, P2, tid, nthr);
    const int c0 = min(Qc, R);
    for (int i = tid; i < c0; i += nthr) s_occ[i] = cand[i];
    if (tid == 0) s_c0 = c0;
  } else if (tid == 0) {
    s_c0 = s_cs;
  }
  __syncthreads();

  // ---- length cap and the continuation matrix ----
  const int c0 = s_c0;
  long long capl = 0;
  if (M > 0 && c0 > 0) {
    capl = min((long long)k, a.fN * M / a.fD + a.offset);
    long long room = (long long)S - n - 1;
    if (room < 0) room = 0;
    capl = min(capl, room);
    if (a.depth_sum_cap) capl = min(capl, (long long)D - M);
    if (capl < 0) capl = 0;
  }
  const int cap = (int)capl;
  int *cont = s_big;
  if (cap > 0) {
    const int tot = c0 * cap;
    for (int idx = tid; idx < tot; idx += nthr) {
      const int o = idx / cap, d = idx - o * cap;
      const long long pos = (long long)s_occ[o] + 1 + d;
      int v;
      if (src == 1) v = pos <= n - 1 ? row[pos] : 0;
      else v = pos < N ? __ldg(X + pos) : Z;
      cont[idx] = v;
    }
    __syncthreads();
    for (int o = tid; o < c0; o += nthr) {
      int r;
      if (src == 1) {
        r = min(cap, n - 1 - s_occ[o]);
      } else {
        r = 0;
        while (r < cap && cont[o * cap + r] != Z) ++r;
      }
      s_run[o] = r;
    }
    __syncthreads();
  }
  if (warp != 0) return;

  // ---- depth-wise majority vote (one warp, up to 4 occurrences per lane) ----
  int len = 0;
  long long sum = 0;
  if (cap > 0) {
    bool alive[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) alive[s] = lane + 32 * s < c0;
    for (int d = 0; d < cap; ++d) {
      int val[4];
      bool part[4];
      int npart = 0;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int o = lane + 32 * s;
        part[s] = alive[s] && d < s_run[o];
        val[s] = part[s] ? cont[o * cap + d] : 0;
        npart += __popc(__ballot_sync(FULL, part[s]));
      }
      if (npart == 0) break;
      bool pend[4] = {part[0], part[1], part[2], part[3]};
      int remaining = npart, best_cnt = 0, best_tok = 0;
      while (remaining > 0) {
        const unsigned m0 = __ballot_sync(FULL, pend[0]);
        const unsigned m1 = __ballot_sync(FULL, pend[1]);
        const unsigned m2 = __ballot_sync(FULL, pend[2]);
        const unsigned m3 = __ballot_sync(FULL, pend[3]);
        const int ss = m0 ? 0 : (m1 ? 1 : (m2 ? 2 : 3));
        const unsigned mm = m0 ? m0 : (m1 ? m1 : (m2 ? m2 : m3));
        const int ll = __ffs(mm) - 1;
        const int x0 = __shfl_sync(FULL, val[0], ll);
        const int x1 = __shfl_sync(FULL, val[1], ll);
        const int x2 = __shfl_sync(FULL, val[2], ll);
        const int x3 = __shfl_sync(FULL, val[3], ll);
        const int v = ss == 0 ? x0 : (ss == 1 ? x1 : (ss == 2 ? x2 : x3));
        int cnt = 0;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const bool e = pend[s] && val[s] == v;
          cnt += __popc(__ballot_sync(FULL, e));
          pend[s] = pend[s] && !e;
        }
        if (cnt > best_cnt || (cnt == best_cnt && v < best_tok)) { best_cnt = cnt; best_tok = v; }
        remaining -= cnt;
        if (best_cnt > remaining) break;
      }
      if ((long long)best_cnt * a.pD < a.pN * (long long)c0) break;
      if (lane == 0) {
        dr[d] = best_tok;
        if (pr) pr[d] = (float)((double)best_cnt / (double)c0);
      }
      sum += best_cnt;
      ++len;
#pragma unroll
      for (int s = 0; s < 4; ++s) alive[s] = part[s] && val[s] == best_tok;
    }
  }
  for (int d = len + lane; d < k; d += 32) {
    dr[d] = -1;
    if (pr) pr[d] = 0.f;
  }
  if (lane == 0) {
    a.num_valid[b] = len;
    if (a.score) a.score[b] = c0 > 0 ? (float)((double)sum / (double)c0) : 0.f;
    if (a.match_info) { a.match_info[2 * b] = M; a.match_info[2 * b + 1] = src; }
  }
}

// Two instantiations: up to 12 warps with room for two CTAs per SM, and up
// to 20 warps with one.
template <int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) propose_kernel(const ProposeArgs a) {
  propose_body(a);
}

}  // namespace

size_t propose_smem_bytes(int nself, int R, int k, int cand_cap) {
  const size_t big = (size_t)max(cand_cap, R * k);
  return sizeof(int) * ((size_t)MAX_D + (size_t)nself * R + 2 * (size_t)R + big) + LCAP;
}

cudaError_t launch_propose(const ProposeArgs &a, cudaStream_t st) {
  if (a.B <= 0) return cudaSuccess;
  const int warps = a.nself + (a.desc ? NPROBE : 0);
  const size_t smem = propose_smem_bytes(a.nself, a.R, a.k, a.cand_cap);
  if (warps <= 12)
    propose_kernel<384, 2><<<a.B, 32 * warps, smem, st>>>(a);
  else
    propose_kernel<640, 1><<<a.B, 32 * warps, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_update(int32_t *tok, int32_t *ntok, const int32_t *sampled, int B, int T, int S,
                          int V, uint32_t *err, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  update_kernel<<<(B + 3) / 4, 128, 0, st>>>(tok, ntok, sampled, B, T, S, V, err);
  return cudaGetLastError();
}

cudaError_t propose_set_smem_limit(size_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(propose_kernel<384, 2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(propose_kernel<640, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

}  // namespace sgd
