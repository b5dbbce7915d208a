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
// int4 loads, ballot early-outs) while, when a corpus exists, 3 more warps
// find the suffix-array intervals of the last 4, 3 and 2 tokens by a 32-ary
// descent of the suffix-key array.  The whole CTA then evaluates the hits of
// the longest useful interval, and warp 0 runs the depth-wise vote.  All
// decisions are integer; the only floating-point values are the reported
// probabilities and score.
//
// Corpus levels.  An end e matches >= 4 tokens iff the suffix starting at
// e-3 begins with the last 4 tokens (the P4 interval), and likewise for 3 and
// 2.  If no P4 hit has a continuation, every valid end matching >= 3 tokens
// matches exactly 3, so the valid P3 hits (read from the key array alone)
// are the answer; if there are none, the valid P2 hits are.  A level is
// evaluated only when its longest possible match exceeds the row's own
// match, which leaves the chosen source and its occurrences unchanged.
#include <climits>

#include "gram_lookup.cuh"
#include "ingest_cta.cuh"
#include "row_index.cuh"
#include "update_row.cuh"

namespace sgd {

namespace {

constexpr int LCAP = 40960;    // P4 hits whose match length is cached on chip
// A small P4 interval is evaluated from one round trip of context: for each
// hit, its k continuation tokens and the tokens before the pattern, fetched
// with cp.async into the L-cache area (lengths, then ends, then contexts).
constexpr int P4C_MAX = 512;                                   // hits
constexpr int P4C_CTX = (LCAP - P4C_MAX - 4 * P4C_MAX) / 4;    // context ints
constexpr int NPROBE3 = 3;     // probe warps: P4, P3, P2
constexpr int TOP_KEYS = 32;   // staged keys of the top level of the descent
constexpr int MID_KEYS = 1024; // staged keys of the level below it
constexpr long long BIG_INTERVAL = 4096;  // probe hits worth waiting for the self match

// barrier of the three probe warps only
__device__ __forceinline__ void probe_sync() { asm volatile("bar.sync 1, 96;" ::: "memory"); }
// the self warps (warps 0 .. nself-1) of a CTA
__device__ __forceinline__ void self_sync(int nself) {
  asm volatile("bar.sync 2, %0;" ::"r"(32 * nself) : "memory");
}

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

// The windows of warp w: [wlo, whi], scanned from the top down (most recent
// first).  They stream through a per-warp ring of SR 512-byte slots in shared
// memory, filled with cp.async: each lane copies (and later reads) only its
// own 16 bytes of every window, so the ring needs no synchronisation beyond
// the lane's own cp.async groups.  Window s of the sequence (whi - s; the
// window below wlo is fetched too, as the last window's predecessor) uses
// slot s % SR; SPF windows are in flight while one is scanned.
constexpr int SPF = 8;            // windows in flight per self warp
constexpr int SR = SPF + 2;       // ring slots: the window scanned, its predecessor, SPF ahead

struct SelfScan {
  int wlo, whi;
  int4 *ring;  // this warp's SR slots; lane l owns ring[slot * 32 + l]
};

// Copy window widx (zeros outside [0, S)) into ring slot `slot`, one group.
__device__ __forceinline__ void self_fetch(const int32_t *row, int widx, int lane, int S, int4 *ring,
                                           int slot) {
  const int p = widx * WIN + 4 * lane;
  const bool in = widx >= 0 && p < S;
  const unsigned sa = (unsigned)__cvta_generic_to_shared(ring + slot * 32 + lane);
  const int32_t *src = in ? row + p : row;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n\tcp.async.commit_group;" ::"r"(sa),
               "l"(src), "r"(in ? 16 : 0)
               : "memory");
}

// Returns whether the warp has windows (and so committed SPF + 1 groups).
__device__ __forceinline__ bool self_prefetch(const int32_t *row, int n, int S, int w, int nself,
                                              int lane, int4 *ring, SelfScan &sc) {
  const int J = n - 1;
  sc.wlo = 0;
  sc.whi = -1;
  sc.ring = ring;
  if (J <= 0) return false;
  const int nwin = (J + WIN - 1) / WIN;
  const int per = (nwin + nself - 1) / nself;
  sc.wlo = w * per;
  sc.whi = min(nwin, sc.wlo + per) - 1;
  if (sc.whi < sc.wlo) return false;
  // windows 0 .. SPF of the sequence (the last of them may lie below wlo - 1:
  // those slots are never read)
#pragma unroll
  for (int q = 0; q <= SPF; ++q) self_fetch(row, sc.whi - q, lane, S, ring, q);
  return true;
}

// The match length of an end whose last two tokens already match the tail
// (x[jr] = tail[0], x[jr-1] = tail[1]), read from a window pair [pw | cw] in
// the ring: jr is the end's index in the pair (in [WIN, 2 WIN)), and indices
// below lo (before the start of the text) hold no token.  Lane i compares
// x[jr-1-i] with tail[1+i], 32 depths per round, up to depth dlim (the
// comparisons reach back at most 127 positions, never past pw).
// tail1 = tail[1 + lane].
__device__ __forceinline__ int pair_extend(int jr, int lo, const int *cw, const int *pw, int dlim,
                                           const int *s_tail, int tail1, int lane) {
  int L = 1;
  for (int r = 0; r < 4; ++r) {
    const int i = 32 * r + lane;
    const int p = jr - 1 - i;
    bool ok = false;
    if (i + 1 < dlim && p >= lo) {
      const int v = p >= WIN ? cw[p - WIN] : pw[p];
      ok = v == (r == 0 ? tail1 : s_tail[1 + i]);
    }
    const unsigned mis = __ballot_sync(FULL, !ok);
    if (mis) return L + __ffs(mis) - 1;
    L += 32;
  }
  return L;
}

constexpr int LANE_DEPTH = 8;  // depth one lane extends an end to on its own

// The match depth of a window's ends, from the window's tokens alone: lane l's
// component c is the end at pair index jr = WIN + 4 l + c (x[jr] = cur.c; the
// three tokens before lane l's first are the previous lane's last three, or
// the window below's for lane 0: p1, p2, p3 = x[jr0 - 1 .. jr0 - 3] for
// jr0 = WIN + 4 l).  L_c = 0 when the end is not wanted (ok_c false) or
// matches fewer than k (2 <= k <= 4) of the tail's tokens; else its match
// length when that is below 4 or below dlim; else -4 (at least 4, to be
// extended).  Pair indices below lo hold no token.
__device__ __forceinline__ void window_depths(const int4 &cur, int p1, int p2, int p3, int t0, int t1,
                                              int t2, int t3, int dlim, int k, int lo, int lane,
                                              bool ok0, bool ok1, bool ok2, bool ok3, int &L0,
                                              int &L1, int &L2, int &L3) {
  const int jr0 = WIN + 4 * lane;
  auto depth = [&](bool ok, int x0, int x1, int x2, int x3, int jr) {
    if (!ok || x0 != t0 || x1 != t1) return 0;
    int d = 2;
    if (dlim > 2 && x2 == t2) {
      d = 3;
      if (dlim > 3 && x3 == t3) d = 4;
    }
    d = min(d, jr - lo + 1);  // (only tokens at pair index >= lo exist)
    if (d < k) return 0;
    return d == 4 && dlim > 4 && jr - lo + 1 > 4 ? -4 : d;
  };
  L3 = depth(ok3, cur.w, cur.z, cur.y, cur.x, jr0 + 3);
  L2 = depth(ok2, cur.z, cur.y, cur.x, p1, jr0 + 2);
  L1 = depth(ok1, cur.y, cur.x, p1, p2, jr0 + 1);
  L0 = depth(ok0, cur.x, p1, p2, p3, jr0);
}

// A window's ends (lengths from window_depths) into the warp's longest length
// Mw and its list of the R most recent ends of that length, positions
// descending (higher lanes first, then higher components).  An end of at
// least 4 is extended here: with more than two of them each lane extends its
// own token by token up to LANE_DEPTH, and those that may go deeper (all of
// them when there are at most two) are extended by the whole warp, one at a
// time.  Lane l's end c is stored as position pos0 + c.
__device__ __forceinline__ void window_ends(int L0, int L1, int L2, int L3, int pos0, int lo,
                                            const int *cw, const int *pw, int dlim, const int *s_tail,
                                            int tail1, int lane, int R, int *list, int &Mw, int &cnt) {
  unsigned m0 = __ballot_sync(FULL, L0 < 0), m1 = __ballot_sync(FULL, L1 < 0);
  unsigned m2 = __ballot_sync(FULL, L2 < 0), m3 = __ballot_sync(FULL, L3 < 0);
  if (m0 | m1 | m2 | m3) {
    if (__popc(m0) + __popc(m1) + __popc(m2) + __popc(m3) > 2) {
      const int jr = WIN + 4 * lane, lim = min(dlim, LANE_DEPTH);
      auto ext = [&](int j) {  // the end at pair index j matches at least 4 tokens
        int L = 4;
        while (L < lim && j - L >= lo) {
          const int p = j - L;
          if ((p >= WIN ? cw[p - WIN] : pw[p]) != s_tail[L]) break;
          ++L;
        }
        return L;
      };
      if (L0 < 0) L0 = ext(jr);
      if (L1 < 0) L1 = ext(jr + 1);
      if (L2 < 0) L2 = ext(jr + 2);
      if (L3 < 0) L3 = ext(jr + 3);
      const bool deep = lim < dlim;  // (one stopped by lo at exactly lim is redone: same length)
      m0 = __ballot_sync(FULL, (m0 >> lane & 1u) && deep && L0 == lim);
      m1 = __ballot_sync(FULL, (m1 >> lane & 1u) && deep && L1 == lim);
      m2 = __ballot_sync(FULL, (m2 >> lane & 1u) && deep && L2 == lim);
      m3 = __ballot_sync(FULL, (m3 >> lane & 1u) && deep && L3 == lim);
    }
    for (;;) {  // warp-wide, in descending position 4 * lane + c
      int best = -1;
      if (m0) best = 4 * (31 - __clz(m0));
      if (m1) best = max(best, 4 * (31 - __clz(m1)) + 1);
      if (m2) best = max(best, 4 * (31 - __clz(m2)) + 2);
      if (m3) best = max(best, 4 * (31 - __clz(m3)) + 3);
      if (best < 0) break;
      const unsigned keep = ~(1u << (best >> 2));
      const int bc = best & 3;
      m0 = bc == 0 ? m0 & keep : m0;
      m1 = bc == 1 ? m1 & keep : m1;
      m2 = bc == 2 ? m2 & keep : m2;
      m3 = bc == 3 ? m3 & keep : m3;
      const int L = pair_extend(WIN + best, lo, cw, pw, dlim, s_tail, tail1, lane);
      if (lane == (best >> 2)) {
        if (bc == 0) L0 = L;
        else if (bc == 1) L1 = L;
        else if (bc == 2) L2 = L;
        else L3 = L;
      }
    }
  }
  const int Lw = (int)__reduce_max_sync(FULL, (unsigned)max(max(L0, L1), max(L2, L3)));
  if (Lw == 0 || Lw < Mw) return;
  if (Lw > Mw) { Mw = Lw; cnt = 0; }
  if (cnt >= R) return;
  const bool e0 = L0 == Mw, e1 = L1 == Mw, e2 = L2 == Mw, e3 = L3 == Mw;
  const unsigned E0 = __ballot_sync(FULL, e0), E1 = __ballot_sync(FULL, e1);
  const unsigned E2 = __ballot_sync(FULL, e2), E3 = __ballot_sync(FULL, e3);
  const unsigned above = lane == 31 ? 0u : (FULL << (lane + 1));  // the more recent lanes
  int slot = cnt + __popc(E0 & above) + __popc(E1 & above) + __popc(E2 & above) + __popc(E3 & above);
  if (e3) { if (slot < R) list[slot] = pos0 + 3; ++slot; }
  if (e2) { if (slot < R) list[slot] = pos0 + 2; ++slot; }
  if (e1) { if (slot < R) list[slot] = pos0 + 1; ++slot; }
  if (e0) { if (slot < R) list[slot] = pos0; }
  cnt = min(R, cnt + __popc(E0) + __popc(E1) + __popc(E2) + __popc(E3));
}

// The warp's windows, most recent first.  Ends with L >= 1 are exactly the
// positions holding tail[0] = t0; those with L >= 2 also hold tail[1] just
// before.  Each lane holds four consecutive tokens of a window (its own 16
// bytes of the ring slot), so a window without t0 costs one load, four
// compares and a vote.  Otherwise the R most recent t0 positions are kept
// (list1: the answer when no end matches two tokens) and every (t1, t0)
// position's depth is taken from the lanes' registers up to 4 tokens;
// deeper ends are extended (window_ends) into (Mw, list).
__device__ void self_process(const int32_t *row, int n, int S, int D, int R, const int *s_tail,
                             int *list, int *list1, int lane, SelfScan &sc, int &Mw, int &cnt,
                             int &cnt1) {
  Mw = 0;
  cnt = 0;
  cnt1 = 0;
  if (sc.whi < sc.wlo) return;
  const int J = n - 1;
  const int t0 = s_tail[0];
  const bool two = D >= 2 && n >= 2;
  const int t1 = two ? s_tail[1] : 0;
  const int t2 = D >= 3 && n >= 3 ? s_tail[2] : 0, t3 = D >= 4 && n >= 4 ? s_tail[3] : 0;
  const int tail1 = lane + 1 < min(D, n) ? s_tail[1 + lane] : 0;
  for (int wi = sc.whi, q = 0; wi >= sc.wlo; --wi, ++q) {
    // keep SPF windows in flight; then windows q and q + 1 must have landed
    self_fetch(row, wi - SPF - 1, lane, S, sc.ring, (q + SPF + 1) % SR);
    asm volatile("cp.async.wait_group %0;" ::"n"(SPF) : "memory");
    const int4 cur = sc.ring[(q % SR) * 32 + lane];
    const int base = wi * WIN, p0 = base + 4 * lane;
    const bool a0 = cur.x == t0 && p0 < J, a1 = cur.y == t0 && p0 + 1 < J;
    const bool a2 = cur.z == t0 && p0 + 2 < J, a3 = cur.w == t0 && p0 + 3 < J;
    if (__any_sync(FULL, a0 | a1 | a2 | a3)) {
      // t0 positions, most recent first: higher lanes, then higher components
      if (cnt1 < R) {
        const int mine = (int)a0 + (int)a1 + (int)a2 + (int)a3;
        int x = mine;  // over lanes >= this one
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_down_sync(FULL, x, off);
          if (lane + off < 32) x += y;
        }
        const int total = __shfl_sync(FULL, x, 0);
        int slot = cnt1 + x - mine;
        if (a3) { if (slot < R) list1[slot] = p0 + 3; ++slot; }
        if (a2) { if (slot < R) list1[slot] = p0 + 2; ++slot; }
        if (a1) { if (slot < R) list1[slot] = p0 + 1; ++slot; }
        if (a0) { if (slot < R) list1[slot] = p0; }
        cnt1 = min(R, cnt1 + total);
      }
      // (t1, t0) positions.  The three tokens before a lane's first are the
      // previous lane's last three, or the window below's for lane 0.  Depths
      // 2..4 come from these registers; only ends matching at least four
      // tokens are extended (window_ends: by their own lane, deeper ones by the
      // whole warp), so a bigram occurring hundreds of times in the row costs
      // no serial extension per occurrence.
      const int4 prv = sc.ring[((q + 1) % SR) * 32 + lane];
      int py = __shfl_up_sync(FULL, cur.y, 1), pz = __shfl_up_sync(FULL, cur.z, 1);
      int pv = __shfl_up_sync(FULL, cur.w, 1);
      const int by = __shfl_sync(FULL, prv.y, 31), bz = __shfl_sync(FULL, prv.z, 31);
      const int bw = __shfl_sync(FULL, prv.w, 31);
      if (lane == 0) { py = by; pz = bz; pv = bw; }
      const bool c0 = a0 && two && pv == t1, c1 = a1 && two && cur.x == t1;
      const bool c2 = a2 && two && cur.y == t1, c3 = a3 && two && cur.z == t1;
      if (__any_sync(FULL, c0 | c1 | c2 | c3)) {
        __syncwarp();  // every lane's copies visible to the warp (the extension reads across lanes)
        const int *cw = reinterpret_cast<const int *>(sc.ring + (q % SR) * 32);
        const int *pw = reinterpret_cast<const int *>(sc.ring + ((q + 1) % SR) * 32);
        // (the row's text starts at position 0: pair index WIN - base)
        const int lo = WIN - base;
        int L0, L1, L2, L3;
        window_depths(cur, pv, pz, py, t0, t1, t2, t3, D, 2, lo, lane, c0, c1, c2, c3, L0, L1, L2, L3);
        window_ends(L0, L1, L2, L3, base + 4 * lane, lo, cw, pw, D, s_tail, tail1, lane, R, list, Mw,
                    cnt);
        __syncwarp();  // cross-lane reads of the slot done before it is refilled
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // nothing of the ring left in flight
}

// The self result from the self warps' lists (warps hold ascending ranges):
// the longest length over the warps and its R most recent ends; when no end
// matches two tokens, the R most recent positions of the last token (L = 1).
// One warp.
__device__ __forceinline__ void merge_self_lists(int nself, int R, const int *s_wM, const int *s_wcnt,
                                                 const int *s_wcnt1, const int *s_wlist,
                                                 const int *s_wlist1, int *s_occ, int lane, int &Ms,
                                                 int &c) {
  Ms = 0;
  for (int w = 0; w < nself; ++w) Ms = max(Ms, s_wM[w]);
  c = 0;
  if (Ms > 0) {
    for (int w = nself - 1; w >= 0 && c < R; --w) {
      if (s_wM[w] != Ms) continue;
      const int mm = min(s_wcnt[w], R - c);
      for (int i = lane; i < mm; i += 32) s_occ[c + i] = s_wlist[w * R + i];
      c += mm;
    }
  } else {  // no end matches two tokens: the ends are the t0 positions (L = 1)
    for (int w = nself - 1; w >= 0 && c < R; --w) {
      const int mm = min(s_wcnt1[w], R - c);
      for (int i = lane; i < mm; i += 32) s_occ[c + i] = s_wlist1[w * R + i];
      c += mm;
    }
    if (c > 0) Ms = 1;
  }
}

// ---------------------------------------------------------------------------
// The row's self match from its bigram index, run by the self warps after the
// barrier that follows the lookup (icnt, pos: the bigram's count and listed
// positions, all below n_old).  The ends with L >= 2 are the positions
// j <= n - 2 holding the tail's last bigram (t1, t0): the listed ones and the
// appended positions [max(1, n_old), n - 2] that hold it.  Each is extended
// backwards against the tail (every (end, depth) comparison loaded in one
// batch), and the R most recent ends of the longest length are kept.
// Returns 1 when the match was found this way (s_Ms, s_cs, s_occ written and
// published through s_ms_ready); 2 when no end matches two tokens (the match
// is at most 1; published as 1 with no ends -- the caller scans the row if
// the corpus does not decide the row); 0 when the row must be scanned (the
// list is incomplete, or the ends do not fit in `cap`).  Every self warp
// returns the same value.
__device__ int index_self(const int32_t *row, int n, int n_old, int D, int R, int nself, int warp,
                          int lane, int t1, int t0, int icnt, const int *pos, const int *s_tail,
                          int *cand, int *candL, int cap, int *s_nc, int *s_occ, int *s_Ms,
                          int *s_cs, int *s_ms_ready) {
  if (icnt < 0 || icnt > RI_K) return 0;
  if (warp == 0) {
    const bool keep = lane < icnt && pos[lane] <= n - 2;
    const unsigned mk = __ballot_sync(FULL, keep);
    const unsigned lt = (1u << lane) - 1u;
    if (keep && __popc(mk & lt) < cap) cand[__popc(mk & lt)] = pos[lane];
    int c = __popc(mk);
    for (int base = max(1, n_old); base <= n - 2; base += 32) {
      const int p = base + lane;
      const bool hit = p <= n - 2 && row[p - 1] == t1 && row[p] == t0;
      const unsigned mh = __ballot_sync(FULL, hit);
      const int slot = c + __popc(mh & lt);
      if (hit && slot < cap) cand[slot] = p;
      c += __popc(mh);
    }
    for (int i = lane; i < min(c, cap); i += 32) candL[i] = min(D, cand[i] + 1);
    if (lane == 0) *s_nc = c;
  }
  self_sync(nself);
  const int nc = *s_nc;
  if (nc > cap) return 0;
  if (nc == 0) {
    if (warp == 0 && lane == 0) {
      *s_Ms = 1;
      *s_cs = 0;
      __threadfence_block();
      *(volatile int *)s_ms_ready = 1;
    }
    return 2;
  }
  // every (end, depth >= 2) pair: the first depth that differs bounds the end
  const int W = D - 2, tot = nc * W, st = 32 * nself;
  for (int f0 = 32 * warp + lane; f0 < tot; f0 += 4 * st) {
    int v[4], cidx[4], dep[4];
    bool in[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int f = f0 + u * st;
      cidx[u] = f < tot ? f / W : 0;
      dep[u] = f < tot ? 2 + f % W : D;
      // (depths past the text start are excluded by candL's initial bound)
      in[u] = f < tot && dep[u] <= cand[cidx[u]];
      v[u] = in[u] ? row[cand[cidx[u]] - dep[u]] : 0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (in[u] && v[u] != s_tail[dep[u]]) atomicMin(&candL[cidx[u]], dep[u]);
  }
  self_sync(nself);
  if (warp == 0) {
    int M = 0;
    for (int i = lane; i < nc; i += 32) M = max(M, candL[i]);
    M = (int)__reduce_max_sync(FULL, (unsigned)M);
    int cnt = 0;
    for (int i = lane; i < nc; i += 32) {
      if (candL[i] != M) continue;
      ++cnt;
      int rank = 0;  // the more recent ends of length M
      for (int q = 0; q < nc; ++q) rank += candL[q] == M && cand[q] > cand[i];
      if (rank < R) s_occ[rank] = cand[i];
    }
    cnt = (int)__reduce_add_sync(FULL, (unsigned)cnt);
    if (lane == 0) {
      *s_Ms = M;
      *s_cs = min(cnt, R);
      __threadfence_block();
      *(volatile int *)s_ms_ready = 1;
    }
  }
  return 1;
}

// ---------------------------------------------------------------------------
// corpus: the delta
//
// The delta is the text Y[0, dv) of the docs placed after the snapshot was
// linearised, read in place from the ring: Y[u] = ring[(ds + u) mod C].  An
// end u counts when it has a continuation (u + 1 < dv and Y[u+1] is not the
// sentinel) and matches at least the last two tokens (a corpus match needs
// two); u >= 1 and positions before ds hold no token.  The self warps share
// its windows of WIN aligned ring positions (C is a multiple of WIN) in
// contiguous ranges, each keeping its longest length and the R most recent
// ends of that length.  Every end is accounted for, as a brute-force scan
// would, but a window is read only when its gram signature (delta_sig.cuh)
// says it may hold an end that can still matter: one matching at least
// `need` tokens, where need is the warp's longest length (one more once R
// ends of it are kept) and at least the CTA's longest so far.  A window that
// is read is checked token by token, as the row's own windows are.

// The delta's windows are numbered r = 0 .. nw-1 from the one holding Y[0]:
// window r starts at Y index r WIN - off (off = ds mod WIN) and is ring
// window (ds / WIN + r) mod (C / WIN).  All Y indices fit in 32 bits.
constexpr int DNB = 4;  // windows read per batch: each with the one below (8 slots) + slot 8

// The delta's windows are scanned newest first, in two stages.  Rounds: in
// round t warp w takes the block of DNB windows that is (t nself + nself-1-w)
// blocks below the newest, so that all warps work on the most recent windows
// at once; after each round the warps' ends join one list for the CTA (most
// recent first).  Rounds go on while they keep finding many ends and the
// CTA's list holds fewer than R ends of its longest length: rows with a short
// but frequent match find their R most recent ends this way in few steps.
// Ranges: the windows below the rounds, split into contiguous ranges (warp
// nself - 1 the newest).  Everything the rounds covered is more recent than
// every range.
struct DeltaScan {
  int nw;   // windows
  int off;  // Y index 0 lies at this offset of window 0
  int w0;   // ring window of window 0
  int nrw;  // ring windows (C / WIN)
  __device__ __forceinline__ int rwin(int r) const {  // ring window of delta window r (r >= -1)
    const int x = (w0 + r) % nrw;
    return x < 0 ? x + nrw : x;
  }
};

// The row's last 2, 3 and 4 tokens as signature buckets.
struct DeltaGrams {
  unsigned b2, b3, b4;
};

// A block's signature words requested ahead of its round (lane i < DNB: the
// words of window hi - i for the row's 2-, 3- and 4-gram buckets).
struct SigAhead {
  uint32_t w2, w3, w4;
};

__device__ __forceinline__ SigAhead sig_ahead(const uint32_t *sig, const DeltaScan &sc,
                                              const DeltaGrams &g, int hi, int dlim, int lane) {
  SigAhead p{0u, 0u, 0u};
  const int r = hi - lane;
  if (lane < DNB && r >= 0) {
    const size_t rw = (size_t)sc.rwin(r);
    p.w2 = sig[(size_t)(g.b2 >> 5) * sc.nrw + rw];
    if (dlim >= 3) p.w3 = sig[(size_t)(g.b3 >> 5) * sc.nrw + rw];
    if (dlim >= 4) p.w4 = sig[(size_t)(g.b4 >> 5) * sc.nrw + rw];
  }
  return p;
}

__device__ __forceinline__ void delta_windows(long long C, long long ds, int dv, DeltaScan &sc) {
  sc.off = (int)(ds % WIN);
  sc.nw = (sc.off + dv - 1) / WIN + 1;
  sc.nrw = (int)(C / WIN);
  sc.w0 = (int)(ds / WIN);
}

// Copy 16 bytes per lane of ring window rw into ring slot `slot` (no commit).
__device__ __forceinline__ void ring_copy(const int32_t *ring, int rw, int lane, int4 *sring, int slot) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(sring + slot * 32 + lane);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa),
               "l"(ring + (size_t)rw * WIN + 4 * lane)
               : "memory");
}

// The windows [rlo, rhi] of a warp's block or range into (Mw, cnt, list).
// s_state[w]: warp w's (longest length << 16 | ends kept) in the same stage,
// published as one word so that a warp can tell when more recent windows --
// the CTA's list (cN ends of length cB) and the blocks or ranges of the warps
// above -- already hold R ends of the CTA's longest length (its own ends of
// that length then cannot vote).  A stale word only under-counts, which costs
// reads, never results.
__device__ void delta_process(const int32_t *ring, const uint32_t *sig, int dv, int Z, int D, int n,
                              int R, const int *s_tail, int lane, int4 *sring, const DeltaScan &sc,
                              int rlo, int rhi, int *list, int *s_best, int *s_state, int cB, int cN,
                              int warp, int nself, const DeltaGrams &grams, const SigAhead *ahead,
                              int &Mw, int &cnt) {
  Mw = 0;
  cnt = 0;
  const int t0 = s_tail[0], t1 = s_tail[1];
  const int dlim = min(D, n);
  const int tail1 = lane + 1 < dlim ? s_tail[1 + lane] : 0;
  const int t2 = dlim >= 3 ? s_tail[2] : 0, t3 = dlim >= 4 ? s_tail[3] : 0;
  const unsigned b2 = grams.b2, b3 = grams.b3, b4 = grams.b4;
  const int nrw = sc.nrw;
  auto rwin = [&](int r) { return sc.rwin(r); };
  // the shortest end that can still change the result (> dlim: none)
  auto need = [&]() {
    const int B = max(*(const volatile int *)s_best, 2);
    int above = cB == B ? cN : 0;
    for (int i = warp + 1; i < nself; ++i) {
      const int st = ((const volatile int *)s_state)[i];
      if ((st >> 16) == B) above += st & 0xffff;
    }
    int nd = max(cnt < R ? Mw : Mw + 1, B);
    if (above >= R && nd <= B) nd = B + 1;
    return nd;
  };
  // windows r - 31 .. r whose signature has the bucket of the `o`-gram (o <= 4): bit i
  // (ahead: the words of the block [rlo, rhi], at most DNB windows, already read)
  auto candidates = [&](int r, int o, int ilo) {
    const unsigned bk = o == 2 ? b2 : (o == 3 ? b3 : b4);
    const int rr = r - lane;
    bool hit = false;
    if (lane >= ilo && rr >= rlo) {
      const uint32_t w = ahead != nullptr ? (o == 2 ? ahead->w2 : (o == 3 ? ahead->w3 : ahead->w4))
                                          : sig[(size_t)(bk >> 5) * nrw + rwin(rr)];
      hit = (w >> (bk & 31)) & 1u;
    }
    return __ballot_sync(FULL, hit);
  };
  bool done = false;
  for (int r = rhi; r >= rlo && !done; r -= 32) {
    int nd = need();
    if (nd > dlim) break;  // no end can matter any more
    int o = min(nd, 4);
    unsigned mask = candidates(r, o, 0);
    while (mask) {
      // the next DNB windows of the mask (descending), each with the one below
      // and the first tokens of the one above
      int wl[DNB];
      int nb = 0;
#pragma unroll
      for (int j = 0; j < DNB; ++j) {
        wl[j] = -1;
        if (mask) {
          const int i = __ffs(mask) - 1;
          mask &= mask - 1;
          wl[j] = r - i;
          nb = j + 1;
          ring_copy(ring, rwin(r - i), lane, sring, 2 * j);
          ring_copy(ring, rwin(r - i - 1), lane, sring, 2 * j + 1);
        }
      }
      if (lane < nb) {  // lane j: the first four tokens of the window above wl[j]
        int wa = wl[0];
#pragma unroll
        for (int j = 1; j < DNB; ++j) wa = lane == j ? wl[j] : wa;
        const unsigned sa = (unsigned)__cvta_generic_to_shared(sring + 8 * 32 + lane);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa),
                     "l"(ring + (size_t)rwin(wa + 1) * WIN)
                     : "memory");
      }
      asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
      __syncwarp();  // every lane's copies visible to the warp
      nd = need();
#pragma unroll
      for (int j = 0; j < DNB; ++j) {
        if (j >= nb || nd > dlim) break;
        const int rj = wl[j];
        const int4 cur = sring[(2 * j) * 32 + lane];
        const int *cw = reinterpret_cast<const int *>(sring + (2 * j) * 32);
        const int *pw = reinterpret_cast<const int *>(sring + (2 * j + 1) * 32);
        const int top = reinterpret_cast<const int *>(sring + 8 * 32 + j)[0];  // the token after the window
        // the depth of the ends matching at least k tokens (k = 2, 3 or 4 by
        // the shortest end that can still matter); the three tokens before
        // each lane's first are the previous lane's last three, or the window
        // below's
        const int4 bl = reinterpret_cast<const int4 *>(pw)[31];
        int py = __shfl_up_sync(FULL, cur.y, 1), pz = __shfl_up_sync(FULL, cur.z, 1);
        int pv = __shfl_up_sync(FULL, cur.w, 1);
        if (lane == 0) { py = bl.y; pz = bl.z; pv = bl.w; }
        // ends: a continuation (the token after lane 31's last is the window
        // above's first), Y index >= 1
        const int dn = __shfl_down_sync(FULL, cur.x, 1);
        const int after3 = lane == 31 ? top : dn;
        const int yb = rj * WIN - sc.off;  // Y index of the window's first token
        const int u0 = yb + 4 * lane;
        // pair index of Y[0] (clamped: below the pair nothing is excluded)
        const int lo = max(-1, min(2 * WIN, WIN - yb));
        int L0, L1, L2, L3;
        window_depths(cur, pv, pz, py, t0, t1, t2, t3, dlim, min(nd, 4), lo, lane,
                      cur.y != Z && u0 >= 1 && u0 + 1 < dv, cur.z != Z && u0 + 1 >= 1 && u0 + 2 < dv,
                      cur.w != Z && u0 + 2 >= 1 && u0 + 3 < dv,
                      after3 != Z && u0 + 3 >= 1 && u0 + 4 < dv, L0, L1, L2, L3);
        if (__any_sync(FULL, (L0 | L1 | L2 | L3) != 0)) {
          const int M0 = Mw, c0 = cnt;
          window_ends(L0, L1, L2, L3, u0, lo, cw, pw, dlim, s_tail, tail1, lane, R, list, Mw, cnt);
          if (Mw > M0 && lane == 0) atomicMax(s_best, Mw);
          if (Mw != M0 || cnt != c0) nd = need();
        }
      }
      if (lane == 0) *(volatile int *)&s_state[warp] = Mw << 16 | cnt;
      __syncwarp();  // cross-lane reads of the slots done before they are refilled
      // fewer windows can matter once longer ends are needed: narrow the rest
      nd = need();
      if (nd > dlim) {
        done = true;
        break;
      }
      if (min(nd, 4) != o && mask) {
        o = min(nd, 4);
        const int ilo = 32 - __clz(~mask & (mask - 1u));  // (bits below the lowest set one are done)
        mask &= candidates(r, o, ilo);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// corpus: key-array descent

// First m tokens of a suffix key against the pattern P (signed order).
__device__ __forceinline__ int key_cmp(const int4 &k, const int4 &P, int m) {
  if (k.x != P.x) return k.x < P.x ? -1 : 1;
  if (m < 2) return 0;
  if (k.y != P.y) return k.y < P.y ? -1 : 1;
  if (m < 3) return 0;
  if (k.z != P.z) return k.z < P.z ? -1 : 1;
  if (m < 4) return 0;
  if (k.w != P.w) return k.w < P.w ? -1 : 1;
  return 0;
}

// Smallest level l whose samples (positions multiple of 32^l) number <= 32.
__device__ __forceinline__ int top_level(long long N) {
  int l = 0;
  while (((N + (1LL << (5 * l)) - 1) >> (5 * l)) > 32) ++l;
  return l;
}

struct Corpus {
  const int32_t *X;
  const int32_t *SA;
  const int4 *K;
  const int32_t *Rec;  // per-position records, or null
  RecShape rs;
  const int32_t *GT;   // n-gram table, or null
  uint64_t gtm;        // its buckets - 1
  const int32_t *GD;   // gram drafts, or null
  long long N;
  int Lmax;
  const int4 *s_top;  // K[j * 32^Lmax]
  const int4 *s_mid;  // K[j * 32^(Lmax-1)]
};

__device__ __forceinline__ int4 key_at(const Corpus &c, int l, long long q) {
  if (c.s_top != nullptr && l == c.Lmax) return c.s_top[q >> (5 * l)];
  if (c.s_mid != nullptr && l == c.Lmax - 1) return c.s_mid[q >> (5 * l)];
  return __ldg(c.K + q);
}

__device__ __forceinline__ void narrow(long long &a, long long &b, long long q, bool v, bool pr) {
  const unsigned bp = __ballot_sync(FULL, pr);
  const unsigned bv = __ballot_sync(FULL, v);
  if (bp) {
    const int f = __ffs(bp) - 1;
    const long long qf = __shfl_sync(FULL, q, f);
    const long long qp = __shfl_sync(FULL, q, f > 0 ? f - 1 : 0);
    b = qf;
    if (f > 0) a = qp;
  } else if (bv) {
    a = __shfl_sync(FULL, q, 31 - __clz((int)bv));
  }
}

// [lo, hi): the suffixes whose first m tokens equal P, by one warp.  Both
// bounds descend together: at level l the answer lies in (a, b], and the at
// most 32 positions strictly inside that are multiples of 32^l are probed;
// the first probe at or above P (lower) / above P (upper) narrows it.  At
// level 0 every position of the bracket has been probed.
__device__ void probe_bounds(const Corpus &c, const int4 &P, int m, int lane, long long &lo,
                             long long &hi) {
  long long aL = -1, bL = c.N, aU = -1, bU = c.N;
  for (int l = c.Lmax; l >= 0; --l) {
    const long long st = 1LL << (5 * l);
    const long long qL = (aL < 0 ? 0 : aL + st) + (long long)lane * st;
    const long long qU = (aU < 0 ? 0 : aU + st) + (long long)lane * st;
    const bool vL = qL < bL, vU = qU < bU;
    bool pL = false, pU = false;
    if (vL) pL = key_cmp(key_at(c, l, qL), P, m) >= 0;
    if (vU) pU = key_cmp(key_at(c, l, qU), P, m) > 0;
    narrow(aL, bL, qL, vL, pL);
    narrow(aU, bU, qU, vU, pU);
  }
  lo = bL;
  hi = bU;
}

// [lo, hi) for the m-gram P from the snapshot's n-gram table, by one warp.
__device__ __forceinline__ void gram_bounds(const Corpus &c, const int4 &P, int m, int lane, long long &lo,
                                            long long &hi, int &slot7) {
  gt_lookup(c.GT, c.gtm, P, m, lane, lo, hi, slot7);
}

// The interval of the last m tokens (t[i] = the i-th token from the end),
// written to bound[0..1] by lane 0; empty when the row is shorter, m > D or
// the pattern holds KEY_END (corpus tokens are in [0, V], so it cannot occur).
// *blk: the gram's draft block (m = 2, 3 with gram drafts), else -2.
__device__ void pattern_bounds(const Corpus &c, const int *t, int m, int D, int n, int lane,
                               long long *bound, int *blk) {
  long long plo = 0, phi = 0;
  int slot7 = -2;
  if (D >= m && n >= m) {
    const int4 P = make_int4(t[m - 1], m >= 2 ? t[m - 2] : 0, m >= 3 ? t[m - 3] : 0,
                             m >= 4 ? t[m - 4] : 0);
    const bool endless = P.x != KEY_END && (m < 2 || P.y != KEY_END) &&
                         (m < 3 || P.z != KEY_END) && (m < 4 || P.w != KEY_END);
    if (endless) {
      if (c.GT != nullptr) gram_bounds(c, P, m, lane, plo, phi, slot7);
      else probe_bounds(c, P, m, lane, plo, phi);
    }
  }
  if (lane == 0) {
    bound[0] = plo;
    bound[1] = phi;
    *blk = c.GD != nullptr && m <= 3 ? slot7 : -2;
  }
}

// ---------------------------------------------------------------------------
// corpus: the P4 level (random access into the text)

// Backward extension of a corpus end e already known to match l0 tokens.
// Tokens are compared 8 at a time, their loads issued together.
__device__ __forceinline__ int extend_from(const int32_t *X, long long e, int L, long long lim,
                                           const int *s_tail) {
  while (L < lim) {
    const int cn = (int)min(8LL, lim - L);
    int v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = j < cn ? __ldg(X + e - L - j) : 0;
    int j = cn;  // first mismatch in the chunk
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t < j && v[t] != s_tail[L + t]) j = t;
    L += j;
    if (j < cn) break;
  }
  return L;
}

__device__ __forceinline__ int extend(const int32_t *X, long long e, int l0, const int *s_tail, int n,
                                      int D) {
  const long long lim = min((long long)min(D, n), e + 1);
  return extend_from(X, e, l0, lim, s_tail);
}

// Match length of the end behind P4 hit p, 0 without a continuation.
__device__ __forceinline__ int p4_entry(const Corpus &c, int Z, long long p, const int *s_tail, int n,
                                        int D, long long &e) {
  e = (long long)__ldg(c.SA + p) + 3;
  if (e + 1 >= c.N) return 0;
  if (__ldg(c.X + e + 1) == Z) return 0;
  return extend(c.X, e, 4, s_tail, n, D);
}

// Match lengths of the P4 hits [lo, hi), by the whole CTA.  Each thread
// takes 4 hits per round and issues their loads together (SA entries, then
// the continuation token and the token before the pattern).  The length of
// hit lo + i (0 without a continuation) is kept in s_L[i] for i < LCAP;
// s_lhist[L] counts the valid ends of each length.
__device__ void scan_p4(const Corpus &c, int Z, long long lo, long long hi, const int *s_tail, int n,
                        int D, unsigned char *s_L, int *s_lhist, int tid, int nthr) {
  const long long dn = min(D, n);
  for (long long base = lo + tid; base < hi; base += 4LL * nthr) {
    long long e[4];
    int x1[4], x0[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long p = base + (long long)u * nthr;
      e[u] = p < hi ? (long long)__ldg(c.SA + p) + 3 : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = e[u] >= 0 && e[u] + 1 < c.N;
      x1[u] = ok ? __ldg(c.X + e[u] + 1) : Z;
      x0[u] = ok && 4 < min(dn, e[u] + 1) ? __ldg(c.X + e[u] - 4) : 0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long p = base + (long long)u * nthr;
      if (p >= hi) continue;
      int L = 0;
      if (x1[u] != Z) {
        const long long lim = min(dn, e[u] + 1);
        L = 4;
        if (L < lim && x0[u] == s_tail[L]) L = extend_from(c.X, e[u], L + 1, lim, s_tail);
        atomicAdd(&s_lhist[L], 1);
      }
      if (p - lo < LCAP) s_L[p - lo] = (unsigned char)L;
    }
  }
}

// Whether the P4 interval [lo, hi) is small enough for scan_p4_ctx.
__device__ __forceinline__ bool p4_ctx_fits(long long cnt, int W) {
  return cnt <= P4C_MAX && cnt * W <= P4C_CTX;
}

// Match lengths of a small P4 interval: the ends (SA entries) in one round
// trip, then every hit's context in a second one, all on chip afterwards.
// Context of hit i, W = kc + dl - 4 ints at s_ctx[i * W]: X[e+1 .. e+kc]
// (Z past the end of the text), then X[e-4-j] for j < dl - 4.  Lengths go to
// s_L[i] (0 without a continuation), ends to s_e[i], counts to s_lhist.
__device__ void scan_p4_ctx(const Corpus &c, int Z, long long lo, long long hi, const int *s_tail,
                            int n, int D, int kc, unsigned char *s_L, int *s_e, int *s_ctx,
                            int *s_lhist, int tid, int nthr) {
  const int cnt = (int)(hi - lo);
  const int dl = min(D, n);
  if (c.Rec != nullptr) {
    // the snapshot's records hold all of it: one round trip of 16-byte copies
    const int ri = c.rs.ri, q4 = ri >> 2;
    for (int f = tid; f < cnt * q4; f += nthr) {
      const int i = f / q4, j = f - i * q4;
      cp_async16(&s_ctx[i * ri + 4 * j], c.Rec + (size_t)(lo + i) * ri + 4 * j);
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
    probe_sync();
    for (int i = tid; i < cnt; i += nthr) {
      const int *x = s_ctx + (size_t)i * ri;
      const long long e = (long long)x[0] + 3;
      s_e[i] = (int)e;
      int L = 0;
      if (x[1] != Z) {
        // back tokens against tail[4..], four per 16-byte load of each
        const int lim = (int)min((long long)dl, e + 1);
        const int4 *xb = reinterpret_cast<const int4 *>(x + 4);
        const int4 *tb = reinterpret_cast<const int4 *>(s_tail + 4);
        L = 4;
        for (int q = 0; 4 + 4 * q < lim; ++q) {
          const int4 u = xb[q], v = tb[q];
          int f = 4;
          if (u.w != v.w) f = 3;
          if (u.z != v.z) f = 2;
          if (u.y != v.y) f = 1;
          if (u.x != v.x) f = 0;
          L = min(4 + 4 * q + f, lim);
          if (f < 4) break;
        }
        atomicAdd(&s_lhist[L], 1);
      }
      s_L[i] = (unsigned char)L;
    }
    return;
  }
  const int W = kc + dl - 4;
  for (int i = tid; i < cnt; i += nthr) s_e[i] = __ldg(c.SA + lo + i) + 3;
  probe_sync();
  for (int f = tid; f < cnt * W; f += nthr) {
    const int i = f / W, j = f - i * W;
    const long long e = s_e[i];
    const long long pos = j < kc ? e + 1 + j : e - 4 - (j - kc);
    if (pos >= 0 && pos < c.N) cp_async4(&s_ctx[f], c.X + pos);
    else s_ctx[f] = Z;  // past the end (continuation) or before the start (never compared)
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
  probe_sync();
  for (int i = tid; i < cnt; i += nthr) {
    const int *x = s_ctx + (size_t)i * W;
    const long long e = s_e[i];
    int L = 0;
    if (x[0] != Z) {
      const long long lim = min((long long)dl, e + 1);
      L = 4;
      while (L < lim && x[kc + L - 4] == s_tail[L]) ++L;
      atomicAdd(&s_lhist[L], 1);
    }
    s_L[i] = (unsigned char)L;
  }
}

// ---------------------------------------------------------------------------
// corpus: the P3 / P2 levels (key array only)

// A P3 (lvl 3) or P2 (lvl 2) hit is valid when the suffix has a token after
// the pattern that is not a sentinel (nor the end of the text); its end is
// SA[p] + lvl - 1.
// The token after the pattern of a P3 / P2 hit, from the key array.
__device__ __forceinline__ int short_token(const Corpus &c, long long p, int lvl) {
  const int *k = reinterpret_cast<const int *>(c.K + p);
  return __ldg(k + (lvl == 2 ? 2 : 3));
}

// Hits p0 + u * stride (u < SB) of the chosen level: q[u] whether the hit is
// an end of length Mc, e[u] its end.  All loads of the batch are issued
// before any is used (one round trip per batch).
constexpr int SB = 8;
__device__ __forceinline__ void select_batch(const Corpus &c, int Z, long long p0, int stride,
                                             long long lo, long long hi, int lvl, int Mc,
                                             const int *s_tail, int n, int D,
                                             const unsigned char *s_L, int *e, bool *q) {
  if (lvl != 4) {
    int t[SB];
#pragma unroll
    for (int u = 0; u < SB; ++u) {
      const long long p = p0 + (long long)u * stride;
      const bool in = p < hi;
      t[u] = in ? short_token(c, p, lvl) : Z;
      e[u] = in ? __ldg(c.SA + p) + lvl - 1 : 0;
    }
#pragma unroll
    for (int u = 0; u < SB; ++u) q[u] = t[u] != Z && t[u] != KEY_END;
    return;
  }
#pragma unroll
  for (int u = 0; u < SB; ++u) {
    const long long p = p0 + (long long)u * stride;
    q[u] = p < hi && p - lo < LCAP && s_L[p - lo] == Mc;
    e[u] = q[u] ? __ldg(c.SA + p) + 3 : 0;
  }
#pragma unroll
  for (int u = 0; u < SB; ++u) {
    const long long p = p0 + (long long)u * stride;
    if (p < hi && p - lo >= LCAP) {  // beyond the length cache: evaluate again
      long long ee;
      q[u] = p4_entry(c, Z, p, s_tail, n, D, ee) == Mc;
      e[u] = (int)ee;
    }
  }
}

// ---------------------------------------------------------------------------
// Radix selection step, one warp: walking the 256 bins from the top, the bin
// where the running count first reaches `need`, and what is still needed
// inside it.  The caller guarantees the bins hold at least `need`.
__device__ void pick_bin(const int *hist, int need, int lane, int *s_sel, int *s_need) {
  int h[8];
  int tot = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = hist[255 - (lane * 8 + j)];
    tot += h[j];
  }
  int x = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(FULL, x, off);
    if (lane >= off) x += y;
  }
  const unsigned m = __ballot_sync(FULL, x >= need);
  if (lane == __ffs(m) - 1) {
    int acc = x - tot;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (acc + h[j] >= need) {
        *s_sel = 255 - (lane * 8 + j);
        *s_need = need - acc;
        break;
      }
      acc += h[j];
    }
  }
}


// draft length bound: min(k, floor(factor * M) + offset, S - n - 1) [, D - M]
// Tokens the vote may emit: k, the factor cap and the context (Model Runner
// V2 drafts: k and the context only).
__device__ __forceinline__ int draft_cap(const ProposeArgs &a, int M, int n) {
  long long c = a.fixed ? (long long)a.k : min((long long)a.k, a.fN * M / a.fD + a.offset);
  long long room = (long long)a.S - n - 1;
  if (room < 0) room = 0;
  c = min(c, room);
  if (a.depth_sum_cap && !a.fixed) c = min(c, (long long)a.D - M);
  return c < 0 ? 0 : (int)c;
}

__global__ void __launch_bounds__(128) update_kernel(int32_t *tok, int32_t *ntok, const int32_t *sampled,
                                                     int B, int T, int S, int V, uint32_t *err,
                                                     const RowIndexArgs ri) {
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const int n_in = ntok[b];
  const int covered = ri.tab ? ri.meta[2 * (size_t)b] : -1;
  int n = n_in;
  uint32_t fl = 0;
  if (n < 0) { n = 0; fl |= SGD_ERR_NUM_TOKENS; }
  if (n > S) { n = S; fl |= SGD_ERR_NUM_TOKENS; }
  const int n_old = n;
  int32_t *row = tok + (size_t)b * S;
  n = update_row_warp(row, n, sampled + (size_t)b * T, T, S, V, lane, fl);
  if (lane == 0) {
    ntok[b] = n;
    if (fl) atomicOr(err, fl);
  }
  if (ri.tab) {
    __syncwarp();  // the appended ids visible to every lane
    ri_after_update(ri, b, row, n_old, n, covered == n_in && covered == n_old, lane);
  }
}

// sgd_reset_rows, first launch: each listed row is claimed by its last listing
// (the largest index i), so that a row listed twice is rebuilt once.
__global__ void __launch_bounds__(256) ri_claim_kernel(const int32_t *rows, int m, int max_batch,
                                                       unsigned long long *claim,
                                                       unsigned long long epoch) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= m) return;
  const int r = rows[i];
  if (r < 0 || r >= max_batch) return;
  atomicMax(claim + r, (epoch << 24) | (unsigned long long)i);
}

// Second launch, one CTA per listing: the claimed row takes the next
// generation (every older entry reads as empty; after generation 255 the
// table is cleared and generation 1 is used again) and every position p >= 1
// of its current contents is inserted.  Ids outside [0, 2^24) or a full table
// leave the row invalid (scanned) until its next reset.
__global__ void __launch_bounds__(1024) ri_reset_kernel(const RowIndexArgs ri, const int32_t *tok,
                                                        const int32_t *ntok, int S,
                                                        const int32_t *rows, int max_batch,
                                                        const unsigned long long *claim,
                                                        unsigned long long epoch) {
  __shared__ int s_gen, s_wrap, s_ok;
  const int i = blockIdx.x;
  const int r = rows[i];
  if (r < 0 || r >= max_batch) return;
  if (claim[r] != ((epoch << 24) | (unsigned long long)i)) return;  // listed again later
  int n = ntok[r];
  n = n < 0 ? 0 : (n > S ? S : n);
  int32_t *meta = ri.meta + 2 * (size_t)r;
  int32_t *tab = ri.tab + (size_t)r * ri.H * RI_ENTRY;
  if (threadIdx.x == 0) {
    const int g = meta[1];
    s_wrap = g >= 255;
    s_gen = g >= 255 || g < 1 ? 1 : g + 1;
    s_ok = 1;
    meta[0] = -1;
    meta[1] = s_gen;
  }
  __syncthreads();
  if (s_wrap) {
    for (long long e = threadIdx.x; e < ri.H; e += blockDim.x)
      *reinterpret_cast<unsigned long long *>(tab + e * RI_ENTRY) = 0ull;
    __syncthreads();
  }
  const int gen = s_gen;
  const int32_t *row = tok + (size_t)r * S;
  bool ok = true;
  for (int p = 1 + threadIdx.x; p < n; p += blockDim.x) {
    const int t1 = row[p - 1], t0 = row[p];
    if (t1 < 0 || t1 > RI_MAX_TOKEN || t0 < 0 || t0 > RI_MAX_TOKEN) ok = false;
    else ok &= ri_insert(tab, ri.H, gen, t1, t0, p);
  }
  if (!ok) s_ok = 0;
  __syncthreads();
  if (threadIdx.x == 0) meta[0] = s_ok ? n : -1;
}

// ---------------------------------------------------------------------------
// Fused step: every CTA of the launch reads the step epoch E, then counts
// itself in; the last one to arrive resets the count and advances E (all
// CTAs have read it by then), so each launch has its own epoch.
__device__ __forceinline__ void step_arrive(uint32_t *sync, uint32_t e0) {
  __threadfence();
  if (atomicAdd(&sync[1], 1u) == gridDim.x - 1) {
    sync[1] = 0;
    atomicExch(&sync[0], e0 + 1);
  }
}

// Fused step with a delta: each row CTA counts itself out once it no longer
// reads the ring; the last one publishes the epoch in sync[3] (the ingest CTA
// waits for it before appending over the rows' visible delta).
__device__ __forceinline__ void step_done(uint32_t *sync, uint32_t e0) {
  __threadfence();
  if (atomicAdd(&sync[2], 1u) == gridDim.x - 2) {  // the row CTAs are all but CTA 0
    sync[2] = 0;
    __threadfence();
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(sync + 3), "r"(e0 + 1) : "memory");
  }
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t *p) {
  return *reinterpret_cast<const volatile uint32_t *>(p);
}

__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// CTA 0 of a fused step: the ingest of the step's finished docs.
__device__ __forceinline__ void step_ingest(const ProposeArgs &a, long long dcap) {
  extern __shared__ __align__(16) int dsm[];
  __shared__ uint32_t s_e0;
  if (threadIdx.x == 0 && a.step_ready != nullptr) {
    const uint32_t e0 = ld_volatile_u32(&a.step_sync[0]);
    s_e0 = e0;
    step_arrive(a.step_sync, e0);
  }
  __syncthreads();
  const SmallIngest g{a.tok, a.ntok, a.B, a.S, a.V, a.ing_rows, a.ing_starts, a.ing_lengths,
                      a.ing_m, a.ring, a.C, a.rs, a.doc_start, a.doc_len, a.max_docs, a.err,
                      a.step_ready, s_e0 + 1 + a.ing_skew, a.step_sync, a.desc, dcap, a.sig};
  ingest_small_cta(g, *reinterpret_cast<SmallIngestSmem *>(dsm));
}

// Depth-wise majority vote of one candidate (one warp, up to 4 occurrences
// per lane): cont[o * capp + d] is occurrence o's continuation at depth d,
// run[o] how many of them exist; the emitted tokens and their probabilities
// go to dr / pr (nothing past them is written), their number to len and the
// sum of their counts to sum (score = sum / c0).  Scratch: s_hist (256 ints),
// s_vv (c0 ints), s_hash (256 x 12 bytes).
//
// With a reference survivor chosen at depth d, let diff(o) be the first
// depth >= d where survivor o disagrees with the reference or runs out.
// Then at depth x the survivors are {diff >= x}, the participants are those
// not running out at x, and the reference's token is continued by
// c(x) = #{diff > x}.  While the reference takes part and c(x) is a strict
// majority of the participants, the reference's token wins with count
// c(x): two histograms of diff give every c(x) at once, so a whole run of
// depths is decided in one warp scan.  Where the majority fails, all
// participants' tokens are counted (most frequent wins, ties to the
// smallest id) and a new reference is taken among the winners.
// Probabilities are quotients c / c0 of integers with c <= 64 * c0 and
// c0 <= 128: both are exact floats, and a correctly rounded single
// division gives the same float as rounding the double quotient (checked
// over that whole range by the test suite), so no double arithmetic.
__device__ void vote_warp(const ProposeArgs &a, const int *cont, int capp, const int *s_run, int c0,
                          int cap, int *s_hist, int *s_vv, unsigned char *s_hash, int32_t *dr,
                          float *pr, int &len, long long &sum) {
  const int lane = threadIdx.x & 31;
  unsigned char *s_L = s_hash;
  len = 0;
  sum = 0;
  if (cap > 0) {
    bool alive[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) alive[s] = lane + 32 * s < c0;
    const unsigned lt = (1u << lane) - 1u;
    int *H = s_hist, *HR = s_hist + 128;  // diff histogram; run-outs among them
    int d = 0;
    while (d < cap) {
      unsigned am[4];
      int nalive = 0;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        am[s] = __ballot_sync(FULL, alive[s]);
        nalive += __popc(am[s]);
      }
      if (nalive == 0) break;
      const int ss = am[0] ? 0 : (am[1] ? 1 : (am[2] ? 2 : 3));
      const unsigned mm = am[0] ? am[0] : (am[1] ? am[1] : (am[2] ? am[2] : am[3]));
      const int ref = (__ffs(mm) - 1) + 32 * ss;
      const int run_ref = min(s_run[ref], cap);
      for (int i = lane; i <= cap; i += 32) { H[i] = 0; HR[i] = 0; }
      __syncwarp();
      int diff[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        diff[s] = cap;
        if (!alive[s]) continue;
        const int o = lane + 32 * s;
        const int r = min(s_run[o], cap);
        // first depth in [d, r) where o disagrees with the reference, else r;
        // four depths per 16-byte load of each row
        const int4 *ro = reinterpret_cast<const int4 *>(cont + o * capp);
        const int4 *rr = reinterpret_cast<const int4 *>(cont + ref * capp);
        int dd = r;
        for (int q = d >> 2; (q << 2) < r; ++q) {
          const int4 x = ro[q], y = rr[q];
          const int b = q << 2;
          int f = -1;
          if (b + 3 >= d && b + 3 < r && x.w != y.w) f = b + 3;
          if (b + 2 >= d && b + 2 < r && x.z != y.z) f = b + 2;
          if (b + 1 >= d && b + 1 < r && x.y != y.y) f = b + 1;
          if (b >= d && b < r && x.x != y.x) f = b;
          if (f >= 0) { dd = f; break; }
        }
        diff[s] = dd;
        atomicAdd(&H[dd], 1);
        if (dd == r && r < cap) atomicAdd(&HR[dd], 1);
      }
      __syncwarp();
      // c(x) = nalive - #{diff <= x}, for x = d + lane and x = d + 32 + lane
      const int x1 = d + lane, x2 = d + 32 + lane;
      const int h1 = x1 <= cap ? H[x1] : 0, h2 = x2 <= cap ? H[x2] : 0;
      int p1 = h1, p2 = h2;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y1 = __shfl_up_sync(FULL, p1, off), y2 = __shfl_up_sync(FULL, p2, off);
        if (lane >= off) { p1 += y1; p2 += y2; }
      }
      p2 += __shfl_sync(FULL, p1, 31);
      const int c1 = nalive - p1, c2 = nalive - p2;
      const int part1 = c1 + h1 - (x1 <= cap ? HR[x1] : 0);
      const int part2 = c2 + h2 - (x2 <= cap ? HR[x2] : 0);
      const bool maj1 = x1 < run_ref && 2 * c1 > part1, maj2 = x2 < run_ref && 2 * c2 > part2;
      const bool ok1 = maj1 && (long long)c1 * a.pD >= a.pN * (long long)c0;
      const bool ok2 = maj2 && (long long)c2 * a.pD >= a.pN * (long long)c0;
      const unsigned bad1 = __ballot_sync(FULL, x1 < cap && !ok1);
      const unsigned bad2 = __ballot_sync(FULL, x2 < cap && !ok2);
      const int F = bad1 ? d + __ffs(bad1) - 1 : (bad2 ? d + 32 + __ffs(bad2) - 1 : cap);
      // emit depths [d, F): the reference's tokens
      unsigned part_sum = 0;  // (at most 64 depths of at most 128 each)
      if (x1 < F) {
        dr[x1] = cont[ref * capp + x1];
        if (pr) pr[x1] = (float)c1 / (float)c0;
        part_sum += (unsigned)c1;
      }
      if (x2 < F) {
        dr[x2] = cont[ref * capp + x2];
        if (pr) pr[x2] = (float)c2 / (float)c0;
        part_sum += (unsigned)c2;
      }
      sum += (long long)__reduce_add_sync(FULL, part_sum);
      len += F - d;
      if (F >= cap) break;
      // depth F: stop if the reference's majority only missed the threshold
      const bool majF = __shfl_sync(FULL, F - d < 32 ? maj1 : maj2, (F - d) & 31);
      if (majF) break;
      d = F;
      // full count among the participants at depth d
      bool part[4];
      unsigned pm[4];
      int npart = 0;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        alive[s] = alive[s] && diff[s] >= d;
        part[s] = alive[s] && d < s_run[lane + 32 * s];
        pm[s] = __ballot_sync(FULL, part[s]);
        npart += __popc(pm[s]);
      }
      if (npart == 0) break;
      int val[4];
      int base = 0;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        val[s] = part[s] ? cont[(lane + 32 * s) * capp + d] : 0;
        if (part[s]) s_vv[base + __popc(pm[s] & lt)] = val[s];
        base += __popc(pm[s]);
      }
      __syncwarp();
      unsigned mycnt = 0, myv = 0xffffffffu;
      int cnt;
      if (npart <= 32) {
        const unsigned vm = npart == 32 ? FULL : ((1u << npart) - 1u);
        const int v = lane < npart ? s_vv[lane] : 0;
        if (lane < npart) mycnt = __popc(__match_any_sync(vm, v));
        const unsigned maxc = __reduce_max_sync(FULL, mycnt);
        if (lane < npart && mycnt == maxc) myv = (unsigned)v ^ 0x80000000u;
        cnt = (int)maxc;
      } else {
        // more than 32 participants: count every value in a 256-entry open
        // addressing table in shared memory (the probe's idle length cache);
        // a key is (1 << 32) | value, so 0 marks a free entry for any value
        unsigned long long *hk = reinterpret_cast<unsigned long long *>(s_L);
        unsigned *hc = reinterpret_cast<unsigned *>(s_L + 256 * sizeof(unsigned long long));
        for (int i = lane; i < 256; i += 32) { hk[i] = 0ull; hc[i] = 0u; }
        __syncwarp();
        int hs[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          hs[s] = 0;
          if (!part[s]) continue;
          const unsigned long long key = (1ull << 32) | (unsigned)val[s];
          unsigned h = ((unsigned)val[s] * 0x9E3779B1u) >> 24;
          for (int t = 0; t < 256; ++t, h = (h + 1) & 255u) {  // <= 128 keys: ends early
            const unsigned long long old = atomicCAS(&hk[h], 0ull, key);
            if (old == 0ull || old == key) {
              atomicAdd(&hc[h], 1u);
              hs[s] = (int)h;
              break;
            }
          }
        }
        __syncwarp();
        unsigned c4[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          c4[s] = part[s] ? hc[hs[s]] : 0u;
          mycnt = max(mycnt, c4[s]);
        }
        const unsigned maxc = __reduce_max_sync(FULL, mycnt);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          if (part[s] && c4[s] == maxc) myv = min(myv, (unsigned)val[s] ^ 0x80000000u);
        cnt = (int)maxc;
      }
      const int tau = (int)(__reduce_min_sync(FULL, myv) ^ 0x80000000u);
      __syncwarp();
      if ((long long)cnt * a.pD < a.pN * (long long)c0) break;
      if (lane == 0) {
        dr[d] = tau;
        if (pr) pr[d] = (float)cnt / (float)c0;
      }
      sum += cnt;
      ++len;
#pragma unroll
      for (int s = 0; s < 4; ++s) alive[s] = part[s] && val[s] == tau;
      ++d;
    }
  }
}

// MODE 0: the whole step in one kernel.  MODE 1 (long rows, first launch):
// the update and the self scan only; the row's self result is written to
// a.self_res.  MODE 2 (second launch): one warp reads that result back in
// place of the scan, the probe warps and the vote run as in MODE 0.
// ---------------------------------------------------------------------------
// Gram drafts (built with each snapshot).  For a row whose corpus match is a
// 2- or 3-gram G (no hit of its last four tokens has a continuation, resp. no
// hit of its last three), the corpus candidate is the R most recent valid ends
// of G in the snapshot and their vote, which depend on G alone: the row only
// truncates the vote at its cap (the vote at depth d depends only on the
// occurrences still agreeing at d, never on where it will stop).  So each
// snapshot holds, for every 2-/3-gram whose interval has GD_MIN_HITS or more
// hits (where a row's own evaluation would select among them), a
// block: [0] c0, [1] the tokens the vote emits up to depth k, [2] Q (its
// valid ends), [4, 4 + k) the tokens, [4 + k4, 4 + k4 + k) the count agreeing
// at each depth (k4 = k rounded up to 4); its index sits in the gram's
// table entry ([7]; -2: no block, the row evaluates the interval itself).

constexpr int GD_MIN_HITS = 8;  // smaller intervals are evaluated by the row (one short pass)

// Pass 1: every 2-/3-gram entry with >= GD_MIN_HITS hits takes a block (while
// there are blocks); the others get -2.
__global__ void __launch_bounds__(256) gd_assign_kernel(int32_t *gt, unsigned long long entries,
                                                        int32_t *count, int cap, int32_t *owner) {
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  for (unsigned long long e = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; e < entries;
       e += stride) {
    int32_t *en = gt + e * GT_ENTRY;
    const int m = en[0];
    if (m != 2 && m != 3) continue;
    int idx = -2;
    if (en[6] - en[5] >= GD_MIN_HITS) {
      const int c = atomicAdd(count, 1);
      if (c < cap) {
        idx = c;
        owner[c] = (int32_t)e;
      }
    }
    en[7] = idx;
  }
}

constexpr int GD_THREADS = 128;
constexpr int GD_CAND = 1024;  // candidate ends kept on chip
constexpr int GD_LOADS = 4;    // interval hits each thread has in flight

// The R largest of s_cand[0, *cnt) (distinct values) kept in s_cand[0, R),
// *cnt = R; returns the smallest kept.  A radix select from the top byte.
__device__ unsigned gd_keep_top(int *s_cand, int *cnt, int R, int *s_hist, int *s_sel, int *s_need,
                                int *s_tmp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = *cnt;
  unsigned thr = 0, mk = 0;
  int need = R;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += GD_THREADS) s_hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < c; i += GD_THREADS) {
      const unsigned e = (unsigned)s_cand[i];
      if ((e & mk) == thr) atomicAdd(&s_hist[(e >> shift) & 255u], 1);
    }
    __syncthreads();
    if (warp == 0) pick_bin(s_hist, need, lane, s_sel, s_need);
    __syncthreads();
    thr |= (unsigned)*s_sel << shift;
    mk |= 255u << shift;
    need = *s_need;
    __syncthreads();
  }
  // compact the kept ones to the front (through s_tmp, R entries)
  if (tid == 0) *s_sel = 0;
  __syncthreads();
  for (int i = tid; i < c; i += GD_THREADS)
    if ((unsigned)s_cand[i] >= thr) s_tmp[atomicAdd(s_sel, 1)] = s_cand[i];
  __syncthreads();
  for (int i = tid; i < R; i += GD_THREADS) s_cand[i] = s_tmp[i];
  if (tid == 0) *cnt = R;
  __syncthreads();
  return thr;
}

// Pass 2: one CTA per block.  The gram's valid ends in one pass over its
// interval, keeping the R most recent: ends above the current R-th largest
// join a candidate buffer, which is cut back to its R largest when it fills
// (end positions are distinct).  Then their continuations up to k tokens and
// the vote (vote_warp, the drafting vote, to depth k).
__global__ void __launch_bounds__(GD_THREADS) gd_build_kernel(const int32_t *gt, const int32_t *owner,
                                                             const int4 *K, const int32_t *SA,
                                                             const int32_t *X, long long N, int Z,
                                                             int k, int R, long long pN, long long pD,
                                                             int32_t *gd) {
  // dynamic: GD_CAND candidates, then R continuation rows of roundup4(k) ints
  extern __shared__ __align__(16) int gd_dsm[];
  int *s_cand = gd_dsm;
  int *s_cont = gd_dsm + GD_CAND;
  __shared__ int s_run[MAX_R], s_vv[MAX_R], s_tmp[MAX_R];
  __shared__ int s_hist[256];
  __shared__ __align__(16) unsigned char s_hash[256 * 12];
  __shared__ int s_tok[MAX_K];
  __shared__ float s_prob[MAX_K];
  __shared__ int s_q, s_cnt, s_sel, s_need;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bi = blockIdx.x;
  const int k4 = (k + 3) & ~3;
  const int32_t *en = gt + (size_t)owner[bi] * GT_ENTRY;
  const int m = en[0];
  const long long lo = en[5], hi = en[6];
  if (tid == 0) {
    s_q = 0;
    s_cnt = 0;
  }
  __syncthreads();
  unsigned thr = 0;  // ends below it cannot be among the R largest
  for (long long p0 = lo; p0 < hi; p0 += (long long)GD_THREADS * GD_LOADS) {
    int e[GD_LOADS];
    bool v[GD_LOADS];
#pragma unroll
    for (int u = 0; u < GD_LOADS; ++u) {
      const long long p = p0 + u * GD_THREADS + tid;
      v[u] = false;
      e[u] = 0;
      if (p < hi) {
        const int4 kk = __ldg(K + p);
        const int t = m == 2 ? kk.z : kk.w;  // the token after the gram
        v[u] = t != Z && t != KEY_END;
        e[u] = __ldg(SA + p) + m - 1;
      }
    }
    int nv = 0;
#pragma unroll
    for (int u = 0; u < GD_LOADS; ++u) {
      nv += v[u];
      if (v[u] && (unsigned)e[u] >= thr) s_cand[atomicAdd(&s_cnt, 1)] = e[u];
    }
    if (nv) atomicAdd(&s_q, nv);
    __syncthreads();
    if (s_cnt > GD_CAND - GD_THREADS * GD_LOADS) thr = gd_keep_top(s_cand, &s_cnt, R, s_hist, &s_sel, &s_need, s_tmp);
  }
  __syncthreads();
  if (s_cnt > R) gd_keep_top(s_cand, &s_cnt, R, s_hist, &s_sel, &s_need, s_tmp);
  const int Q = s_q, c0 = s_cnt;  // c0 = min(Q, R)
  // continuations: X[e + 1 ..], up to k tokens, stopping at the sentinel
  for (int idx = tid; idx < c0 * k; idx += GD_THREADS) {
    const int o = idx / k, d = idx - o * k;
    const long long pos = (long long)s_cand[o] + 1 + d;
    s_cont[o * k4 + d] = pos < N ? __ldg(X + pos) : Z;
  }
  __syncthreads();
  for (int o = tid; o < c0; o += GD_THREADS) {
    int r = 0;
    while (r < k && s_cont[o * k4 + r] != Z) ++r;
    s_run[o] = r;
  }
  __syncthreads();
  if (warp == 0) {
    ProposeArgs va{};
    va.pN = pN;
    va.pD = pD;
    int len = 0;
    long long sum = 0;
    if (c0 > 0) vote_warp(va, s_cont, k4, s_run, c0, k, s_hist, s_vv, s_hash, s_tok, s_prob, len, sum);
    __syncwarp();
    int32_t *blk = gd + (size_t)bi * gd_ints(k);
    for (int d = lane; d < k; d += 32) {
      blk[4 + d] = d < len ? s_tok[d] : -1;
      blk[4 + k4 + d] = d < len ? __float2int_rn(s_prob[d] * (float)c0) : 0;
    }
    if (lane == 0) {
      blk[0] = c0;
      blk[1] = len;
      blk[2] = Q;
      blk[3] = 0;
    }
  }
}

template <int MODE, bool EXT>
__device__ __forceinline__ void propose_body(const ProposeArgs &a, const int b) {
  constexpr bool SELF_ONLY = MODE == 1, FROM_RES = MODE == 2;
  extern __shared__ __align__(16) int dsm[];
  __shared__ int s_wM[MAX_SELF_WARPS], s_wcnt[MAX_SELF_WARPS], s_wcnt1[MAX_SELF_WARPS];
  __shared__ int s_hist[256];
  __shared__ int s_lhist[MAX_D + 1];
  __shared__ int s_vv[MAX_R];
  __shared__ long long s_bound[2 * NPROBE3];
  __shared__ int s_n, s_Ms, s_cs, s_q, s_sel, s_need, s_have_corpus;
  __shared__ int s_self_done, s_ms_ready, s_pms, s_Mc, s_c0c, s_cpf;
  __shared__ int s_ckey;  // short level whose continuation comes from keys and records, or 0
  // the delta: ring start, visible tokens, longest match and its ends (their
  // list is in s_wlist1 once merged); the fused step's epoch
  __shared__ long long s_ds;
  __shared__ int s_dv, s_Md, s_cd;
  __shared__ int s_best_delta;  // longest delta match so far (over the self warps)
  __shared__ int s_dstate[MAX_SELF_WARPS];  // per self warp: its delta (length << 16 | ends)
  __shared__ int s_dcB, s_dcN, s_dmore;     // the CTA's delta list: length, ends; another round
  __shared__ uint32_t s_ep;
  __shared__ int s_scan;  // suffix-array hits the probe warps scanned (row statistics)
  // the last four tokens known from the sampled ids (probe warps, phase 0)
  __shared__ int s_l4[4], s_pre, s_pre_n;
  // gram drafts: each probe level's block (-2: none); the block the corpus
  // candidate comes from, or -1
  __shared__ int s_bidx[NPROBE3], s_blk;
  // the row's bigram index: its entries cover the row (maintenance), the self
  // match may come from it, the row length before the update, the looked-up
  // count and positions, self match deferred
  __shared__ int s_iok, s_iuse, s_nold, s_icnt, s_idefer, s_igen, s_inc;
  __shared__ int s_imode;  // how the row's own match was found (row statistics)
  __shared__ int s_ipos[RI_K];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nthr = blockDim.x;
  const int S = a.S, R = a.R, k = a.k, D = a.D, Z = a.V;
  int32_t *row = a.tok + (size_t)b * S;
  // the row index is used by the one-launch kernel without a delta or
  // score-ranked selection (the host enables it only there)
  // (MODE 3: the one-launch kernel of a context with row indexes)
  constexpr bool IDX = MODE == 3 && !EXT;
  const int big = SELF_ONLY ? 0 : max(a.cand_cap, R * ((k + 3) & ~3));
  int *s_tail = dsm;                   // MAX_D
  int *s_wlist = s_tail + MAX_D;       // nself * R: per warp, ends matching >= 2 tokens
  int *s_wlist1 = s_wlist + a.nself * R;  // nself * R: per warp, the t0 positions
  int *s_occ = s_wlist1 + a.nself * R; // R
  int *s_run = s_occ + R;              // R
  int *s_occc = s_run + R;             // R (corpus ends)
  // s_big and everything after it start on 16-byte boundaries (int4 access)
  const int boff = (MAX_D + 2 * a.nself * R + 3 * R + 3) & ~3;
  int *s_big = dsm + boff;             // max(cand_cap, R * roundup4(k))
  const int koff = (boff + big + 3) & ~3;
  // the top two levels of the key array, staged only for a descent (a
  // context without n-gram tables)
  int4 *s_keys = reinterpret_cast<int4 *>(dsm + koff);
  int4 *s_top = a.stage_keys ? s_keys : nullptr;                       // TOP_KEYS
  int4 *s_mid = a.stage_keys ? s_keys + TOP_KEYS : nullptr;            // MID_KEYS
  unsigned char *s_L =
      reinterpret_cast<unsigned char *>(s_keys + (a.stage_keys ? TOP_KEYS + MID_KEYS : 0));  // LCAP
  // nself * SR windows; the self-only launch has no corpus areas before them
  int4 *s_ring = SELF_ONLY ? s_keys : reinterpret_cast<int4 *>(s_L + LCAP);

  // ---- phase 0: warp 0 updates the row; the others fetch the snapshot
  // descriptor and stage the top two levels of its key array ----
  Corpus cp{nullptr, nullptr, nullptr, nullptr, a.rsh, nullptr, 0, nullptr, 0, 0, s_top, s_mid};
  if (!SELF_ONLY && a.desc != nullptr) {
    cp.X = a.desc->text;
    cp.SA = a.desc->sa;
    cp.K = a.desc->keys;
    cp.Rec = a.desc->rec;
    cp.GT = a.desc->gt;
    cp.gtm = a.desc->gt_mask;
    // gram drafts: used by the one-launch kernel without a delta or
    // score-ranked selection (the corpus candidate is then the gram's alone)
    cp.GD = (MODE == 0 || MODE == 3) && !EXT ? a.desc->gd : nullptr;
    cp.N = a.desc->n;
    cp.Lmax = cp.N >= 2 ? top_level(cp.N) : 0;
  }
  if (warp == 0) {
    const bool signal = a.ing_m > 0 && a.step_ready != nullptr;
    const uint32_t e0 = signal && lane == 0 ? ld_volatile_u32(&a.step_sync[0]) : 0u;
    // Where the delta lies.  In a fused step this is read before the CTA counts
    // itself in below: the ingest CTA changes the ring state only after every
    // row CTA has, so all rows see the ring as it was before the step's docs.
    if (EXT && !FROM_RES && a.dcap > 0 && a.desc != nullptr && lane == 0) {
      const DeltaView v = delta_view(*a.rs, a.desc->lin_pushed, a.desc->lin_wp, a.C, a.doc_start);
      s_ds = v.start;
      s_dv = (int)min(v.len, a.dcap);
    } else if (!FROM_RES && lane == 0) {
      s_ds = 0;
      s_dv = 0;
    }
    const int n_in = a.ntok[b];
    const int covered = IDX && a.ri.tab ? a.ri.meta[2 * (size_t)b] : -1;
    const int igen = IDX && a.ri.tab ? a.ri.meta[2 * (size_t)b + 1] : 0;
    int n = n_in;
    uint32_t fl = 0;
    if (n < 0) { n = 0; fl |= SGD_ERR_NUM_TOKENS; }
    if (n > S) { n = S; fl |= SGD_ERR_NUM_TOKENS; }
    const int n_old = n;
    // The row's last D tokens before the update, read with the sampled ids: the
    // tail after the update is the appended ids (newest first) followed by
    // them, so it never has to be read back from the row.
    const int dl0 = min(D, n_old);
    int ot[MAX_D / 32];
#pragma unroll
    for (int u = 0; u < MAX_D / 32; ++u) {
      const int i = lane + 32 * u;
      ot[u] = i < dl0 ? row[n_old - 1 - i] : 0;
    }
    if (a.do_update)
      n = update_row_warp(row, n, a.sampled + (size_t)b * a.T, a.T, S, a.V, lane, fl, s_tail, D);
    if (lane == 0 && a.do_update) a.ntok[b] = n;
    {
      const int ca = n - n_old, dl1 = min(D, n);
#pragma unroll
      for (int u = 0; u < MAX_D / 32; ++u) {
        const int i = lane + 32 * u;
        if (i < dl0 && i + ca < dl1) s_tail[i + ca] = ot[u];
      }
    }
    if (IDX && lane == 0) {
      const bool iok = a.ri.tab != nullptr && covered == n_in && covered == n_old;
      // the last two tokens after the update: appended ids, else the old ones
      s_iok = iok;
      s_iuse = iok && n >= 2 && D >= 2;
      s_nold = n_old;
      s_icnt = -1;
      s_idefer = 0;
      s_igen = igen;
      s_imode = 0;
    }
    if (FROM_RES) {  // the first launch's result: Ms, cs, the last four tokens; the delta's
      const int32_t *res = a.self_res + (size_t)b * self_res_ints(R);
      const int v = lane < 6 ? __ldg(res + lane) : (EXT && lane < 10 ? __ldg(res + R + lane) : 0);
      const int Ms = __shfl_sync(FULL, v, 0), cs = __shfl_sync(FULL, v, 1);
      const int Md = __shfl_sync(FULL, v, 6), cd = __shfl_sync(FULL, v, 7);
      const int ds = __shfl_sync(FULL, v, 8), dv = __shfl_sync(FULL, v, 9);
      if (lane == 0) {
        s_Ms = Ms;
        s_cs = cs;
        s_Md = Md;
        s_cd = cd;
        s_ds = ds;
        s_dv = dv;
      }
    }
    if (signal) {  // publish the updated row to the ingest CTA
      __threadfence();
      __syncwarp();
      if (lane == 0) {
        st_release_u32(&a.step_ready[b], e0 + 1);
        step_arrive(a.step_sync, e0);
      }
    }
    if (lane == 0) {
      if (fl) atomicOr(a.err, fl);
      s_n = n;
      s_have_corpus = a.desc != nullptr && cp.N >= 2;
      s_self_done = 0;
      s_ms_ready = 0;
      if (!FROM_RES) {
        s_Ms = 0;
        s_cs = 0;
      }
      s_Mc = 0;
      s_c0c = 0;
      s_cpf = 0;
      s_ckey = 0;
      s_ep = e0;
      s_scan = 0;
      s_blk = -1;
      s_best_delta = 0;
      for (int w = 0; w < MAX_SELF_WARPS; ++w) s_dstate[w] = 0;
      s_dcB = 0;
      s_dcN = 0;
      if (!FROM_RES) {
        s_Md = 0;
        s_cd = 0;
      }
    }
  } else if (!SELF_ONLY && !FROM_RES && a.do_update && cp.GT != nullptr && cp.N >= 2 && D >= 2 &&
             warp >= a.nself) {
    // When the update appends >= 4 ids, the last four tokens are those ids:
    // the probe warps look their n-grams up now, beside warp 0's update,
    // instead of after the tail is assembled.  Probe warp 0 reads the row's
    // length and the sampled ids itself (the same leading run of ids in
    // [0, V) the update accepts).
    const int pw = warp - a.nself;
    if (pw == 0) {
      int n0 = a.ntok[b];
      n0 = n0 < 0 ? 0 : (n0 > S ? S : n0);
      const int32_t *sp = a.sampled + (size_t)b * a.T;
      int c = a.T, kp0 = 0, kp1 = 0;
      for (int base = 0; base < a.T; base += 32) {
        const int i = base + lane;
        const int v = i < a.T ? sp[i] : 0;  // (plain loads: `sampled` may be host memory)
        if (base == 0) kp0 = v;
        else if (base == 32) kp1 = v;
        const unsigned m = __ballot_sync(FULL, i < a.T && (v < 0 || v >= a.V));
        if (m) {
          c = base + __ffs(m) - 1;
          break;
        }
      }
      const int ca = min(c, S - n0);
      const bool pre = ca >= 4 && ca <= 64;
      if (pre) {
        int l4 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = ca - 1 - i;  // tail[i] is appended id j
          const int v0 = __shfl_sync(FULL, kp0, j & 31), v1 = __shfl_sync(FULL, kp1, j & 31);
          if (lane == i) l4 = j < 32 ? v0 : v1;
        }
        if (lane < 4) s_l4[lane] = l4;
      }
      if (lane == 0) {
        s_pre = pre;
        s_pre_n = n0 + max(ca, 0);
      }
    }
    probe_sync();
    if (s_pre) pattern_bounds(cp, s_l4, 4 - pw, D, s_pre_n, lane, &s_bound[2 * pw], &s_bidx[pw]);
  } else if (!SELF_ONLY && a.stage_keys && a.desc != nullptr && cp.N >= 2 && cp.GT == nullptr) {
    const int sh = 5 * cp.Lmax;
    const long long ntop = (cp.N + (1LL << sh) - 1) >> sh;
    const long long nmid = cp.Lmax > 0 ? (cp.N + (1LL << (sh - 5)) - 1) >> (sh - 5) : 0;
    for (long long j = tid - 32; j < ntop + nmid; j += nthr - 32) {
      if (j < ntop) cp_async16(&s_top[j], cp.K + (j << sh));
      else cp_async16(&s_mid[j - ntop], cp.K + ((j - ntop) << (sh - 5)));
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  __syncthreads();
  const int n = s_n;
  int32_t *dr = a.drafts + (size_t)b * k;
  float *pr = a.probs ? a.probs + (size_t)b * k : nullptr;
  // fused step with a delta: the ingest CTA may wait for every row CTA to be
  // done with the ring before appending to it
  const bool done_signal = EXT && MODE == 0 && a.dcap > 0 && a.ing_m > 0 && a.step_ready != nullptr;
  if (!((a.active == nullptr || a.active[b] != 0) && n > 0)) {
    if (done_signal && tid == 0) step_done(a.step_sync, s_ep);
    // (the update applies to inactive rows too: their index follows it)
    if (IDX && a.ri.tab && warp == 0) ri_after_update(a.ri, b, row, s_nold, n, s_iok, lane);
    if constexpr (!SELF_ONLY) {  // (the self-only launch leaves the outputs to the second)
      for (int d = tid; d < k; d += nthr) {
        dr[d] = -1;
        if (pr) pr[d] = 0.f;
      }
      if (tid == 0) {
        a.num_valid[b] = 0;
        if (a.score) a.score[b] = 0.f;
        if (a.match_info) { a.match_info[2 * b] = 0; a.match_info[2 * b + 1] = 0; }
        if (a.row_stats) *reinterpret_cast<int4 *>(a.row_stats + 4 * (size_t)b) = make_int4(0, 0, 0, 0);
      }
    }
    return;
  }
  const bool corpus_ok = s_have_corpus && D >= 2 && n >= 2;

  // ---- phase 1: (tail[i] = t[n-1-i] is in shared memory already) the self
  // warps prefetch their first windows; with an n-gram table the probe warps
  // find their intervals ----
  const int dl = min(D, n);
  const bool early_bounds = corpus_ok && cp.GT != nullptr;
  const bool pre_bounds = !SELF_ONLY && !FROM_RES && a.do_update && cp.GT != nullptr && cp.N >= 2 &&
                          D >= 2 && s_pre;
  if (early_bounds && warp >= a.nself && !pre_bounds)
    pattern_bounds(cp, s_tail, 4 - (warp - a.nself), D, n, lane, &s_bound[2 * (warp - a.nself)],
                   &s_bidx[warp - a.nself]);
  SelfScan sc;
  // With a usable row index, warp 0 looks the row's last bigram up while the
  // tail is read, and the self warps fetch no window before they know whether
  // the row must be scanned at all.
  const bool use_idx = IDX && s_iuse;
  if (use_idx && warp == 0) {
    const int c = ri_lookup(a.ri.tab + (size_t)b * a.ri.H * RI_ENTRY, a.ri.H, s_igen, s_tail[1], s_tail[0],
                            lane, s_ipos);
    if (lane == 0) s_icnt = c;
  }
  // staged keys landed (no-op without any); a self warp's window groups,
  // committed after them, stay in flight
  if (!FROM_RES && warp < a.nself && !use_idx &&
      self_prefetch(row, n, S, warp, a.nself, lane, s_ring + warp * (SR * 32), sc))
    asm volatile("cp.async.wait_group %0;" ::"n"(SPF + 1) : "memory");
  else
    asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // ---- phase 2: self match (nself warps) || corpus chain (3 probe warps) ----
  // The corpus side does not need the row's own match: while the self warps
  // scan, the probe warps find the intervals, evaluate the winning corpus
  // level and collect its R most recent ends, requesting their continuation
  // tokens.  The last self warp to finish merges the self result and
  // publishes it through a shared flag; the probe warps read it at their
  // decision points to skip levels that cannot win, which only saves work.
  if (FROM_RES && warp == 0) {
    // the self result of the first launch: the most recent ends of length Ms;
    // the delta's most recent ends of length Md
    const int32_t *res = a.self_res + (size_t)b * self_res_ints(R);
    const int c = s_cs, cd = s_cd;
    for (int i = lane; i < c; i += 32) s_occ[i] = __ldg(res + 6 + i);
    for (int i = lane; i < cd; i += 32) s_wlist1[i] = __ldg(res + R + 10 + i);
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      *(volatile int *)&s_ms_ready = 1;
    }
  } else if (!FROM_RES && warp < a.nself) {
    // 0: scan the row; 1: the row index gave the match; 2: no end matches two
    // tokens (decided after the corpus, see below)
    int imode = 0;
    if (use_idx) {
      imode = index_self(row, n, s_nold, D, R, a.nself, warp, lane, s_tail[1], s_tail[0], s_icnt, s_ipos, s_tail,
                         s_wlist, s_wlist1, a.nself * R, &s_inc, s_occ, &s_Ms, &s_cs, &s_ms_ready);
      if (imode == 2 && warp == 0 && lane == 0) s_idefer = 1;
      if (warp == 0 && lane == 0) s_imode = imode;
      if (imode == 0) self_prefetch(row, n, S, warp, a.nself, lane, s_ring + warp * (SR * 32), sc);
    }
    if (imode == 0) {
      int Mw, cnt, cnt1;
      self_process(row, n, S, D, R, s_tail, s_wlist + warp * R, s_wlist1 + warp * R, lane, sc, Mw, cnt,
                   cnt1);
      if (lane == 0) { s_wM[warp] = Mw; s_wcnt[warp] = cnt; s_wcnt1[warp] = cnt1; }
      // The self result: the longest length over the warps and its most recent
      // ends (warps hold ascending ranges); published to the probe warps.
      auto merge_self = [&]() {
        __threadfence_block();
        int Ms, c;
        merge_self_lists(a.nself, R, s_wM, s_wcnt, s_wcnt1, s_wlist, s_wlist1, s_occ, lane, Ms, c);
        if (lane == 0) {
          s_Ms = Ms;
          s_cs = c;
          __threadfence_block();
          *(volatile int *)&s_ms_ready = 1;
        }
        if (SELF_ONLY) {  // the row's self result for the second launch
          __syncwarp();
          int32_t *res = a.self_res + (size_t)b * self_res_ints(R);
          for (int i = lane; i < c; i += 32) res[6 + i] = s_occ[i];
          if (lane < 4) res[2 + lane] = lane < dl ? s_tail[lane] : 0;
          if (lane == 0) {
            res[0] = Ms;
            res[1] = c;
          }
        }
      };
      if (EXT && s_dv > 0 && D >= 2 && n >= 2) {
        // The delta, after the row.  Its first windows are requested before the
        // self merge (each warp's ring is free again); the per-warp lists are
        // reused once warp 0 has merged the row's.
        int4 *sring = s_ring + warp * (SR * 32);
        DeltaScan dsc;
        delta_windows(a.C, s_ds, s_dv, dsc);
        const int G = DNB * a.nself;  // windows per round
        const int dlim = min(D, n);
        const int t2 = dlim >= 3 ? s_tail[2] : 0, t3 = dlim >= 4 ? s_tail[3] : 0;
        const DeltaGrams grams{sig_bucket(2, s_tail[0], s_tail[1], 0, 0),
                               dlim >= 3 ? sig_bucket(3, s_tail[0], s_tail[1], t2, 0) : 0u,
                               dlim >= 4 ? sig_bucket(4, s_tail[0], s_tail[1], t2, t3) : 0u};
        // the signature words of each round's block are read one round ahead
        // (round 0's while the row's result is merged)
        SigAhead ahead = sig_ahead(a.sig, dsc, grams, dsc.nw - 1 - DNB * (a.nself - 1 - warp), dlim, lane);
        self_sync(a.nself);
        if (warp == 0) merge_self();
        self_sync(a.nself);
        // (the row's per-warp lists are free now: s_wlist holds each warp's
        // ends of a block or range, s_wlist1[0, R) the CTA's list)
        int *wl = s_wlist + warp * R;
        int covered = 0;
        for (int t = 0;; ++t) {
          const int hi = dsc.nw - 1 - t * G - DNB * (a.nself - 1 - warp);
          const SigAhead cur = ahead;
          ahead = sig_ahead(a.sig, dsc, grams, hi - G, dlim, lane);  // the next round's
          int M = 0, c = 0;
          delta_process(a.ring, a.sig, s_dv, Z, D, n, R, s_tail, lane, sring, dsc, max(0, hi - DNB + 1),
                        hi, wl, &s_best_delta, s_dstate, s_dcB, s_dcN, warp, a.nself, grams, &cur, M, c);
          if (lane == 0) s_dstate[warp] = M << 16 | c;
          self_sync(a.nself);
          covered = min(dsc.nw, covered + G);
          if (warp == 0) {  // the round's ends join the CTA's list (blocks newest first)
            const int st = lane < a.nself ? s_dstate[lane] : 0;
            const int Bn = max(s_dcB, (int)__reduce_max_sync(FULL, (unsigned)(st >> 16)));
            int N = Bn > s_dcB ? 0 : s_dcN;
            const int N0 = N;
            if (Bn >= 2)
              for (int w = a.nself - 1; w >= 0 && N < R; --w) {
                const int sw = s_dstate[w];
                if ((sw >> 16) != Bn) continue;
                const int mm = min(sw & 0xffff, R - N);
                for (int i = lane; i < mm; i += 32) s_wlist1[N + i] = s_wlist[w * R + i];
                N += mm;
              }
            __syncwarp();
            if (lane < a.nself) s_dstate[lane] = 0;
            if (lane == 0) {
              s_dcB = Bn;
              s_dcN = N;
              // another round if windows remain, the list is not full and this
              // round was dense
              s_dmore = covered < dsc.nw && N < R && 4 * (N - N0) >= R;
            }
          }
          self_sync(a.nself);
          if (!s_dmore) break;
        }
        // the ranges below the rounds
        const int rest = dsc.nw - covered;
        const int per = (rest + a.nself - 1) / a.nself;
        int dM = 0, dcnt = 0;
        delta_process(a.ring, a.sig, s_dv, Z, D, n, R, s_tail, lane, sring, dsc, warp * per,
                      min(rest, (warp + 1) * per) - 1, wl, &s_best_delta, s_dstate, s_dcB, s_dcN, warp,
                      a.nself, grams, nullptr, dM, dcnt);
        if (lane == 0) s_dstate[warp] = dM << 16 | dcnt;
        self_sync(a.nself);
        if (warp == 0) {
          // longest delta match; its ends, most recent first: the CTA's list
          // (when of that length), then the ranges from the newest warp down
          const int st = lane < a.nself ? s_dstate[lane] : 0;
          const int Md = max(s_dcB, (int)__reduce_max_sync(FULL, (unsigned)(st >> 16)));
          int c = Md >= 2 && s_dcB == Md ? s_dcN : 0;
          if (Md >= 2)
            for (int w = a.nself - 1; w >= 0 && c < R; --w) {
              const int sw = s_dstate[w];
              if ((sw >> 16) != Md) continue;
              const int mm = min(sw & 0xffff, R - c);
              for (int i = lane; i < mm; i += 32) s_wlist1[c + i] = s_wlist[w * R + i];
              c += mm;
            }
          if (lane == 0) {
            s_Md = Md >= 2 ? Md : 0;
            s_cd = Md >= 2 ? c : 0;
          }
          if (SELF_ONLY) {
            __syncwarp();
            int32_t *res = a.self_res + (size_t)b * self_res_ints(R);
            for (int i = lane; i < c; i += 32) res[R + 10 + i] = s_wlist1[i];
            if (lane == 0) {
              res[R + 6] = Md >= 2 ? Md : 0;
              res[R + 7] = Md >= 2 ? c : 0;
              res[R + 8] = (int)s_ds;
              res[R + 9] = s_dv;
            }
          }
        }
      } else {
        __threadfence_block();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&s_self_done, 1) == a.nself - 1;
        last = __shfl_sync(FULL, last, 0);
        if (last) merge_self();  // the last self warp to finish
        if (EXT && SELF_ONLY && warp == 0 && lane == 0) {  // no delta for this row
          int32_t *res = a.self_res + (size_t)b * self_res_ints(R);
          res[R + 6] = 0;
          res[R + 7] = 0;
          res[R + 8] = (int)s_ds;
          res[R + 9] = 0;
        }
      }
    }
  } else if (corpus_ok) {
    const int pw = warp - a.nself;  // 0: last 4 tokens, 1: last 3, 2: last 2
    const int ptid = tid - 32 * a.nself, pthr = 32 * NPROBE3;
    if (!early_bounds) pattern_bounds(cp, s_tail, 4 - pw, D, n, lane, &s_bound[2 * pw], &s_bidx[pw]);
    probe_sync();
    // The row's own match length, -1 while the self warps still scan.  Before
    // a large piece of work the probe warps wait for it (bounded; on time-out
    // they go on without pruning, which only costs time).
    // (Score-ranked selection: a shorter corpus match may still win, so the
    // corpus candidate is always found in full.)
    auto self_len = [&](bool wait) {
      if (EXT && a.by_score) return -1;
      if (ptid == 0) {
        unsigned spins = 0;
        while (wait && *(volatile int *)&s_ms_ready == 0 && ++spins < (1u << 22)) __nanosleep(64);
        const int ready = *(volatile int *)&s_ms_ready;
        __threadfence_block();
        s_pms = ready ? *(volatile int *)&s_Ms : -1;
      }
      probe_sync();
      return s_pms;
    };
    int pms = self_len(false);
    int Mc = 0, lvl = 0, Q = 0;
    int blk = -1;  // the gram draft block the candidate comes from
    bool p4ctx = false;   // the P4 interval was evaluated on chip (scan_p4_ctx)
    bool oncand = false;  // a short level's ends are all in s_big already
    // A short level's candidates also keep their suffix-array positions (in the
    // idle length-cache area), so that their continuation is read from the key
    // array (just read, so cached) and the records instead of the text.
    int *s_candp = reinterpret_cast<int *>(s_L);
    int *s_occp = s_candp + a.cand_cap;
    const bool keep_p = (size_t)(a.cand_cap + R) * sizeof(int) <= (size_t)LCAP;
    int *s_e4 = reinterpret_cast<int *>(s_L + P4C_MAX);  // small-P4 ends, then contexts
    int *s_ctx = s_e4 + P4C_MAX;
    long long lo = 0, hi = 0;
    if (pms < dl) {
      bool decided = false;
      if (D >= 4 && n >= 4 && s_bound[1] > s_bound[0]) {
        if (pms < 0 && s_bound[1] - s_bound[0] > BIG_INTERVAL) pms = self_len(true);
      }
      if (D >= 4 && n >= 4 && s_bound[1] > s_bound[0] && pms < dl) {
        for (int i = ptid; i <= MAX_D; i += pthr) s_lhist[i] = 0;
        probe_sync();
        if (ptid == 0) s_scan += (int)min(s_bound[1] - s_bound[0], (long long)INT_MAX);
        p4ctx = p4_ctx_fits(s_bound[1] - s_bound[0], cp.Rec ? cp.rs.ri : k + dl - 4);
        if (p4ctx)
          scan_p4_ctx(cp, Z, s_bound[0], s_bound[1], s_tail, n, D, k, s_L, s_e4, s_ctx, s_lhist,
                      ptid, pthr);
        else
          scan_p4(cp, Z, s_bound[0], s_bound[1], s_tail, n, D, s_L, s_lhist, ptid, pthr);
        probe_sync();
        int lbest = 0;
        for (int L = 4 + lane; L <= dl; L += 32)
          if (s_lhist[L] > 0) lbest = L;
        lbest = (int)__reduce_max_sync(FULL, (unsigned)lbest);
        if (lbest > 0) {
          Mc = lbest;
          lvl = 4;
          lo = s_bound[0];
          hi = s_bound[1];
          Q = s_lhist[lbest];
          decided = true;
        }
      }
      for (int lv = 3; lv >= 2 && !decided; --lv) {
        if (D < lv || n < lv) continue;
        if (pms >= lv) break;  // neither this level nor the next can win
        const long long l0 = s_bound[2 * (4 - lv)], h0 = s_bound[2 * (4 - lv) + 1];
        if (h0 <= l0) continue;
        const int bi = s_bidx[4 - lv];
        if (bi >= 0) {
          // the gram's draft block: its valid ends are counted there (every
          // end matching lv tokens matches exactly lv when the longer level
          // has none that continues), and its candidate is decided
          const int qb = __ldg(cp.GD + (size_t)bi * gd_ints(k) + 2);
          if (qb > 0) {
            Mc = lv;
            lvl = lv;
            lo = l0;
            hi = h0;
            Q = qb;
            blk = bi;
            decided = true;
          }
          continue;
        }
        if (pms < 0 && h0 - l0 > BIG_INTERVAL) {
          pms = self_len(true);
          if (pms >= lv) break;
        }
        probe_sync();  // s_q from an earlier level has been read
        if (ptid == 0) {
          s_q = 0;
          s_scan = (int)min((long long)s_scan + (h0 - l0), (long long)INT_MAX);
        }
        probe_sync();
        // one pass: count the valid hits and keep their ends on chip (while
        // they fit); a warp takes its slots with one shared atomic per batch
        const unsigned lt = (1u << lane) - 1u;
        for (long long p0 = l0 + 32 * pw; p0 < h0; p0 += (long long)SB * pthr) {
          int t[SB], eb[SB];
#pragma unroll
          for (int u = 0; u < SB; ++u) {
            const long long q = p0 + lane + (long long)u * pthr;
            t[u] = q < h0 ? short_token(cp, q, lv) : Z;
            eb[u] = q < h0 ? __ldg(cp.SA + q) + lv - 1 : 0;
          }
#pragma unroll
          for (int u = 0; u < SB; ++u) {
            const bool v = t[u] != Z && t[u] != KEY_END;
            const unsigned m = __ballot_sync(FULL, v);
            int base = 0;
            if (lane == 0 && m) base = atomicAdd(&s_q, __popc(m));
            base = __shfl_sync(FULL, base, 0);
            const int slot = base + __popc(m & lt);
            if (v && slot < a.cand_cap) {
              s_big[slot] = eb[u];
              if (keep_p) s_candp[slot] = (int)(p0 + lane + (long long)u * pthr);
            }
          }
        }
        probe_sync();
        if (s_q > 0) {
          Mc = lv;
          lvl = lv;
          lo = l0;
          hi = h0;
          Q = s_q;
          oncand = Q <= a.cand_cap;
          decided = true;
        }
      }
    }
    if (Mc > 0 && blk < 0 && pms < 0 && Q > R) pms = self_len(true);
    if (blk >= 0 && Mc > pms) {
      // a gram draft: nothing to select, gather or vote
      if (ptid == 0) {
        s_Mc = Mc;
        s_c0c = min(Q, R);
        s_cpf = 0;
        s_ckey = 0;
        s_blk = blk;
      }
    } else if (Mc > 0 && Mc > pms && lvl == 4 && p4ctx) {
      // A small P4 interval: ends, lengths and continuations are on chip.
      // The R largest ends of length Mc (a radix select over the ends when
      // there are more), their continuations copied for the vote.
      const int capc = draft_cap(a, Mc, n), capp = (capc + 3) & ~3;  // row stride 16-B aligned
      const int cnt = (int)(hi - lo);
      const int W = cp.Rec ? cp.rs.ri : k + dl - 4;      // context stride
      const int co = cp.Rec ? cp.rs.co : 0;              // where the continuation starts
      probe_sync();
      if (ptid == 0) s_q = 0;
      unsigned thr = 0;
      if (Q > R) {
        unsigned mk = 0;
        int need = R;
        for (int shift = 24; shift >= 0; shift -= 8) {
          for (int i = ptid; i < 256; i += pthr) s_hist[i] = 0;
          probe_sync();
          for (int i = ptid; i < cnt; i += pthr) {
            const unsigned e = (unsigned)s_e4[i];
            if (s_L[i] == Mc && (e & mk) == thr) atomicAdd(&s_hist[(e >> shift) & 255u], 1);
          }
          probe_sync();
          if (pw == 0) pick_bin(s_hist, need, lane, &s_sel, &s_need);
          probe_sync();
          thr |= (unsigned)s_sel << shift;
          mk |= 255u << shift;
          need = s_need;
        }
      }
      probe_sync();
      for (int i = ptid; i < cnt; i += pthr) {
        const unsigned e = (unsigned)s_e4[i];
        if (s_L[i] == Mc && e >= thr) {
          const int slot = atomicAdd(&s_q, 1);
          s_occc[slot] = (int)e;
          const int *x = s_ctx + (size_t)i * W + co;
          for (int d = 0; d < capc; ++d) s_big[slot * capp + d] = x[d];
        }
      }
      if (ptid == 0) { s_Mc = Mc; s_c0c = min(Q, R); s_cpf = 1; }
    } else if (Mc > 0 && Mc > pms) {
      // The R largest ends among the Q of length Mc.  O_0 is a set (the vote
      // does not depend on its order), so nothing is sorted.  With at most R
      // of them, all are kept and their continuations requested right away.
      const int capc = draft_cap(a, Mc, n), capp = (capc + 3) & ~3;
      const bool pf = Q <= R && !oncand;
      int *cand = s_big;
      probe_sync();
      if (!oncand) {
        if (ptid == 0) s_q = 0;
        unsigned prefix = 0;
        if (Q > a.cand_cap) {
          // more than fit on chip: radix-select the R-th largest end over the
          // interval, byte by byte; the R ends at or above it are collected below
          unsigned mask = 0;
          int need = R;
          for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = ptid; i < 256; i += pthr) s_hist[i] = 0;
            probe_sync();
            for (long long p0 = lo + ptid; p0 < hi; p0 += (long long)SB * pthr) {
              int e[SB];
              bool q[SB];
              select_batch(cp, Z, p0, pthr, lo, hi, lvl, Mc, s_tail, n, D, s_L, e, q);
  #pragma unroll
              for (int u = 0; u < SB; ++u)
                if (q[u] && ((unsigned)e[u] & mask) == prefix)
                  atomicAdd(&s_hist[((unsigned)e[u] >> shift) & 255u], 1);
            }
            probe_sync();
            if (pw == 0) pick_bin(s_hist, need, lane, &s_sel, &s_need);
            probe_sync();
            prefix |= (unsigned)s_sel << shift;
            mask |= 255u << shift;
            need = s_need;
          }
        }
        probe_sync();
        const unsigned lt = (1u << lane) - 1u;
        for (long long p0 = lo + 32 * pw; p0 < hi; p0 += (long long)SB * pthr) {
          int eb[SB];
          bool qb[SB];
          select_batch(cp, Z, p0 + lane, pthr, lo, hi, lvl, Mc, s_tail, n, D, s_L, eb, qb);
  #pragma unroll
          for (int u = 0; u < SB; ++u) {
            const bool v = qb[u] && (unsigned)eb[u] >= prefix;
            const unsigned m = __ballot_sync(FULL, v);
            int base = 0;
            if (lane == 0 && m) base = atomicAdd(&s_q, __popc(m));
            base = __shfl_sync(FULL, base, 0);
            if (!v) continue;
            const int e = eb[u];
            const int slot = base + __popc(m & lt);
            if (pf) {
              s_occc[slot] = e;
              for (int d = 0; d < capc; ++d) {
                const long long pos = (long long)e + 1 + d;
                if (pos < cp.N) cp_async4(&s_big[slot * capp + d], cp.X + pos);
                else s_big[slot * capp + d] = Z;
              }
            } else if (slot < a.cand_cap) {
              cand[slot] = e;
            }
          }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      }
      probe_sync();
      const int Qc = min(s_q, a.cand_cap);
      int c0c;
      if (Qc > R) {
        // radix-select the R largest among the on-chip candidates
        unsigned pf2 = 0, mk = 0;
        int need = R;
        for (int shift = 24; shift >= 0; shift -= 8) {
          for (int i = ptid; i < 256; i += pthr) s_hist[i] = 0;
          probe_sync();
          for (int i = ptid; i < Qc; i += pthr)
            if (((unsigned)cand[i] & mk) == pf2) atomicAdd(&s_hist[((unsigned)cand[i] >> shift) & 255u], 1);
          probe_sync();
          if (pw == 0) pick_bin(s_hist, need, lane, &s_sel, &s_need);
          probe_sync();
          pf2 |= (unsigned)s_sel << shift;
          mk |= 255u << shift;
          need = s_need;
        }
        if (ptid == 0) s_q = 0;
        probe_sync();
        for (int i = ptid; i < Qc; i += pthr)
          if ((unsigned)cand[i] >= pf2) {
            const int slot = atomicAdd(&s_q, 1);
            s_occc[slot] = cand[i];
            if (oncand && keep_p) s_occp[slot] = s_candp[i];
          }
        c0c = R;
      } else {
        if (!pf)
          for (int i = ptid; i < Qc; i += pthr) {
            s_occc[i] = cand[i];
            if (oncand && keep_p) s_occp[i] = s_candp[i];
          }
        c0c = Qc;
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
      if (ptid == 0) {
        s_Mc = Mc;
        s_c0c = c0c;
        s_cpf = pf;
        s_ckey = oncand && keep_p ? lvl : 0;
      }
    } else if (ptid == 0) {
      s_Mc = 0;
    }
  }
  if (SELF_ONLY) return;
  __syncthreads();

  if (IDX && s_idefer && (corpus_ok ? s_Mc : 0) < 2) {
    // No earlier end holds the row's last bigram, so its match is at most 1,
    // and the corpus has no match of 2 or more: the row's own result decides
    // after all, from a scan of the row.
    if (warp < a.nself) {
      SelfScan sd;
      self_prefetch(row, n, S, warp, a.nself, lane, s_ring + warp * (SR * 32), sd);
      int Mw, cnt, cnt1;
      self_process(row, n, S, D, R, s_tail, s_wlist + warp * R, s_wlist1 + warp * R, lane, sd, Mw, cnt,
                   cnt1);
      if (lane == 0) { s_wM[warp] = Mw; s_wcnt[warp] = cnt; s_wcnt1[warp] = cnt1; }
      self_sync(a.nself);
      if (warp == 0) {
        int Ms, c;
        merge_self_lists(a.nself, R, s_wM, s_wcnt, s_wcnt1, s_wlist, s_wlist1, s_occ, lane, Ms, c);
        if (lane == 0) {
          s_Ms = Ms;
          s_cs = c;
          s_imode = 0;
        }
      }
    }
    __syncthreads();
  }

  // ---- the longer match wins (equal lengths: the row itself) ----
  // The corpus is the snapshot followed by the delta: its longest match is
  // the longer of the two, and at equal lengths the delta's ends are the more
  // recent, so they come first and the snapshot's fill the rest of the R.
  const int Ms = s_Ms, Mcs = corpus_ok ? s_Mc : 0, Md = EXT ? s_Md : 0;
  const int Mc = max(Mcs, Md);
  // score-ranked selection with both candidates: the corpus's is prepared as
  // below, the row's beside it, and the vote decides
  const bool both = EXT && a.by_score && Ms > 0 && Mc > 0;
  int src, M;
  if (Mc > Ms || both) { src = 2; M = Mc; }
  else { src = Ms > 0 ? 1 : 0; M = Ms; }
  const int nd = EXT && src == 2 && Md == Mc ? s_cd : 0;        // delta ends voting
  const int ns = src == 2 && Mcs == Mc ? min(s_c0c, R - nd) : 0;  // snapshot ends voting
  const int cap = M > 0 ? draft_cap(a, M, n) : 0;
  const int c0 = src == 2 ? nd + ns : s_cs;
  // the corpus candidate is a gram draft: its tokens and counts are read, cut at the cap
  const int dblk = src == 2 && nd == 0 ? s_blk : -1;
  const int *occ = src == 2 ? s_occc : s_occ;
  if (nd > 0) {
    // occurrences: the delta's ends, then the ns most recent of the snapshot's
    // (ranked by position; they are distinct) -- into s_wlist, free by now
    const int c0c = Mcs == Mc ? s_c0c : 0;
    for (int i = tid; i < nd; i += nthr) s_wlist[i] = s_wlist1[i];
    for (int i = tid; i < c0c; i += nthr) {
      const int e = s_occc[i];
      int rank = 0;
      if (ns < c0c)
        for (int j = 0; j < c0c; ++j) rank += s_occc[j] > e;
      else
        rank = i;
      if (rank < ns) s_wlist[nd + rank] = e;
    }
    __syncthreads();
    occ = s_wlist;
  }
  int *cont = s_big;                  // cont[o * capp + d]: rows 16-byte aligned
  const int capp = (cap + 3) & ~3;
  if (cap > 0 && c0 > 0 && dblk < 0) {
    // (prefetched by the probe warps when only the snapshot's ends vote)
    const int tot = (src == 2 && s_cpf && nd == 0) ? 0 : c0 * cap;
    const int ck = src == 2 && nd == 0 ? s_ckey : 0;
    const int *occp = reinterpret_cast<const int *>(s_L) + a.cand_cap;
    auto item = [&](int idx) {
      const int o = idx / cap, d = idx - o * cap;
      const long long pos = (long long)occ[o] + 1 + d;
      int v;
      if (src == 1) {
        v = pos <= n - 1 ? row[pos] : 0;
      } else if (o < nd) {  // a delta end: Y[pos], the sentinel past the visible part
        long long q = s_ds + pos;
        if (q >= a.C) q -= a.C;
        v = pos < s_dv ? a.ring[q] : Z;
      } else if (ck != 0 && ck + d <= 3) {  // inside the hit's suffix key (KEY_END: past the text)
        const int *kq = reinterpret_cast<const int *>(cp.K + occp[o]);
        v = __ldg(kq + ck + d);
        if (v == KEY_END) v = Z;
      } else if (ck != 0 && cp.Rec != nullptr && ck + d <= 6) {  // the record's first 16 bytes
        v = __ldg(cp.Rec + (size_t)occp[o] * cp.rs.ri + (ck + d - 3));
      } else {
        v = pos < cp.N ? __ldg(cp.X + pos) : Z;
      }
      return v;
    };
    // four loads in flight per thread: the continuations are independent reads
    constexpr int GB = 4;
    for (int i0 = tid; i0 < tot; i0 += GB * nthr) {
      int v[GB];
#pragma unroll
      for (int u = 0; u < GB; ++u) v[u] = i0 + u * nthr < tot ? item(i0 + u * nthr) : 0;
#pragma unroll
      for (int u = 0; u < GB; ++u) {
        const int idx = i0 + u * nthr;
        if (idx < tot) {
          const int o = idx / cap;
          cont[o * capp + (idx - o * cap)] = v[u];
        }
      }
    }
    __syncthreads();
    for (int o = tid; o < c0; o += nthr) {
      int r;
      if (src == 1) {
        r = min(cap, n - 1 - occ[o]);
      } else {
        r = 0;
        while (r < cap && cont[o * capp + r] != Z) ++r;
      }
      s_run[o] = r;
    }
    __syncthreads();
  }
  // the row's candidate beside it (score-ranked selection): its continuations
  // in the probe's scratch (done with by now), after the vote's hash area
  int *cont_s = reinterpret_cast<int *>(s_L) + 768;
  const int cap_s = both ? draft_cap(a, Ms, n) : 0, capp_s = (cap_s + 3) & ~3, cs = s_cs;
  int *run_s = cont_s + cs * capp_s;
  if constexpr (EXT) if (both && cap_s > 0) {
    for (int idx = tid; idx < cs * cap_s; idx += nthr) {
      const int o = idx / cap_s, d = idx - o * cap_s;
      const int pos = s_occ[o] + 1 + d;
      cont_s[o * capp_s + d] = pos <= n - 1 ? row[pos] : 0;
    }
    for (int o = tid; o < cs; o += nthr) run_s[o] = min(cap_s, n - 1 - s_occ[o]);
    __syncthreads();
  }
  if (done_signal && tid == 0) step_done(a.step_sync, s_ep);  // the row's ring reads are over
  // the row index follows this step's update (for the next step), off the
  // vote's path: warp 1 when there is one
  const int iwarp = nthr > 32 ? 1 : 0;
  if (IDX && a.ri.tab && warp == iwarp && iwarp != 0) ri_after_update(a.ri, b, row, s_nold, n, s_iok, lane);
  if (warp != 0) return;

  // ---- depth-wise majority vote (one warp) ----
  int len = 0;
  long long sum = 0;
  if (dblk >= 0) {
    const int k4 = (k + 3) & ~3;
    const int32_t *gb = cp.GD + (size_t)dblk * gd_ints(k);
    len = min(__ldg(gb + 1), cap);
    int part = 0;
    for (int d = lane; d < len; d += 32) {
      const int cnt = __ldg(gb + 4 + k4 + d);
      dr[d] = __ldg(gb + 4 + d);
      if (pr) pr[d] = (float)cnt / (float)c0;
      part += cnt;
    }
    sum = (long long)__reduce_add_sync(FULL, (unsigned)part);
  } else {
    vote_warp(a, cont, capp, s_run, c0, cap, s_hist, s_vv, s_L, dr, pr, len, sum);
  }
  int cw = c0;  // the winner's occurrences
  if (both) {
    // the row's draft, staged; it wins unless the corpus's score (sum / c0) is
    // higher, or equal with the longer match
    int *stage = run_s + cs;
    float *pstage = reinterpret_cast<float *>(stage + k);
    int len_s = 0;
    long long sum_s = 0;
    __syncwarp();
    if (cap_s > 0)
      vote_warp(a, cont_s, capp_s, run_s, cs, cap_s, s_hist, s_vv, s_L, stage, pstage, len_s, sum_s);
    __syncwarp();
    const long long lhs = sum * cs, rhs = sum_s * c0;
    if (!(lhs > rhs || (lhs == rhs && Mc > Ms))) {
      for (int d = lane; d < len_s; d += 32) {
        dr[d] = stage[d];
        if (pr) pr[d] = pstage[d];
      }
      len = len_s;
      sum = sum_s;
      cw = cs;
      M = Ms;
      src = 1;
    }
  }

  // the slots the vote left empty: -1, or (Model Runner V2 drafts) the row's last token
  const int fill = a.fixed ? s_tail[0] : -1;
  for (int d = len + lane; d < k; d += 32) {
    dr[d] = fill;
    if (pr) pr[d] = 0.f;
  }
  if (IDX && a.ri.tab && iwarp == 0) ri_after_update(a.ri, b, row, s_nold, n, s_iok, lane);
  if (lane == 0) {
    a.num_valid[b] = a.fixed ? k : len;
    if (a.score) a.score[b] = cw > 0 ? (float)sum / (float)cw : 0.f;
    if (a.match_info) { a.match_info[2 * b] = M; a.match_info[2 * b + 1] = src; }
    if (a.row_stats)
      *reinterpret_cast<int4 *>(a.row_stats + 4 * (size_t)b) =
          make_int4(s_scan, cw, src == 1 && both ? cap_s : cap,
                    src | (IDX ? s_imode << 8 : 0) | (src == 2 && dblk >= 0 ? 1 << 12 : 0));
  }
}

// Instantiations.  One kernel per step: up to 12 warps with room for two CTAs
// per SM, and up to 20 warps with one.  Long rows, two launches: the update
// and self scan (self warps only, small footprint, many CTAs per SM), then
// the corpus chain and vote (one warp + the probe warps).
// EXT: the kernel also handles the delta and score-ranked selection; the
// instantiations without them are what a context with neither runs (the
// extra code costs registers and latency even when unused).  MODE 3 is the
// one-launch kernel of a context with row indexes (their lookup, the
// candidates' extension and the deferred scan are compiled only there).
template <int MAXT, int MINB, int MODE, bool EXT>
__global__ void __launch_bounds__(MAXT, MINB) propose_kernel(const ProposeArgs a) {
  // (one call site of the body: its code is inlined once)
  const int b = MODE != 1 && a.ing_m > 0 ? (int)blockIdx.x - 1 : (int)blockIdx.x;
  if (b < 0) step_ingest(a, EXT ? a.dcap : 0);
  else propose_body<MODE, EXT>(a, b);
}

template <int MAXT, int MINB, int MODE>
void launch_kernel(bool ext, int grid, int threads, size_t smem, cudaStream_t st, const ProposeArgs &a) {
  if (ext)
    propose_kernel<MAXT, MINB, MODE, true><<<grid, threads, smem, st>>>(a);
  else
    propose_kernel<MAXT, MINB, MODE, false><<<grid, threads, smem, st>>>(a);
}

}  // namespace

size_t propose_smem_bytes(int mode, int nself, int R, int k, int cand_cap, int stage_keys) {
  const size_t big = mode == 1 ? 0 : (size_t)max(cand_cap, R * ((k + 3) & ~3));
  const size_t boff = ((size_t)MAX_D + 2 * (size_t)nself * R + 3 * (size_t)R + 3) & ~(size_t)3;
  const size_t ints = (boff + big + 3) & ~(size_t)3;
  const size_t ring = (size_t)nself * SR * 32 * sizeof(int4);
  size_t bytes = sizeof(int) * ints;
  if (mode == 1) return bytes + ring;
  bytes += sizeof(int4) * (stage_keys ? TOP_KEYS + MID_KEYS : 0) + LCAP + (mode == 0 ? ring : 0);
  return bytes > sizeof(SmallIngestSmem) ? bytes : sizeof(SmallIngestSmem);
}

int propose_step_max_docs() { return SMALL_DOCS; }

cudaError_t launch_propose(const ProposeArgs &a, cudaStream_t st) {
  if (a.B <= 0) return cudaSuccess;
  const int probe = a.desc ? NPROBE3 : 0;
  const bool ext = a.dcap > 0 || a.by_score;
  if (!a.split) {
    const int warps = a.nself + probe;
    const size_t smem = propose_smem_bytes(0, a.nself, a.R, a.k, a.cand_cap, a.stage_keys);
    const int grid = a.B + (a.ing_m > 0 ? 1 : 0);
    if (a.ri.tab != nullptr) {  // row indexes (never with the delta or score-ranked selection)
      if (warps <= 12)
        propose_kernel<384, 2, 3, false><<<grid, 32 * warps, smem, st>>>(a);
      else
        propose_kernel<640, 1, 3, false><<<grid, 32 * warps, smem, st>>>(a);
    } else if (warps <= 12) {
      launch_kernel<384, 2, 0>(ext, grid, 32 * warps, smem, st, a);
    } else {
      launch_kernel<640, 1, 0>(ext, grid, 32 * warps, smem, st, a);
    }
    return cudaGetLastError();
  }
  // first launch: update + self scan of every row, and of the delta (no
  // snapshot probe, no ingest; the descriptor only tells where the delta starts)
  ProposeArgs a1 = a;
  if (a.dcap == 0) a1.desc = nullptr;
  a1.ing_m = 0;
  const size_t smem1 = propose_smem_bytes(1, a.nself, a.R, a.k, a.cand_cap, a.stage_keys);
  if (a.nself <= 8)
    launch_kernel<256, 3, 1>(ext, a.B, 32 * a.nself, smem1, st, a1);
  else
    launch_kernel<512, 1, 1>(ext, a.B, 32 * a.nself, smem1, st, a1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // second launch: corpus chain and vote; the rows are updated already, so the
  // ingest CTA needs no signal from them
  ProposeArgs a2 = a;
  a2.do_update = 0;
  a2.nself = 1;
  a2.step_ready = nullptr;
  a2.step_sync = nullptr;
  const size_t smem2 = propose_smem_bytes(2, 1, a.R, a.k, a.cand_cap, a.stage_keys);
  const int grid2 = a.B + (a.ing_m > 0 ? 1 : 0);
  launch_kernel<128, 3, 2>(ext, grid2, 32 * (1 + probe), smem2, st, a2);
  return cudaGetLastError();
}

cudaError_t launch_update(int32_t *tok, int32_t *ntok, const int32_t *sampled, int B, int T, int S,
                          int V, uint32_t *err, const RowIndexArgs &ri, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  update_kernel<<<(B + 3) / 4, 128, 0, st>>>(tok, ntok, sampled, B, T, S, V, err, ri);
  return cudaGetLastError();
}

cudaError_t launch_row_index_reset(const RowIndexArgs &ri, const int32_t *tok, const int32_t *ntok,
                                   int S, const int32_t *rows, int m, int max_batch,
                                   unsigned long long *claim, unsigned long long epoch,
                                   cudaStream_t st) {
  if (m <= 0 || ri.tab == nullptr) return cudaSuccess;
  ri_claim_kernel<<<(m + 255) / 256, 256, 0, st>>>(rows, m, max_batch, claim, epoch);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ri_reset_kernel<<<m, 1024, 0, st>>>(ri, tok, ntok, S, rows, max_batch, claim, epoch);
  return cudaGetLastError();
}

cudaError_t launch_gram_drafts(int32_t *gt, uint64_t gt_mask, const int4 *keys, const int32_t *sa,
                               const int32_t *text, int64_t n, int Z, int k, int R, long long pN,
                               long long pD, int32_t *gd, int cap, int32_t *count, int32_t *owner,
                               int32_t *h_count, cudaStream_t st) {
  if (gt == nullptr || gd == nullptr || n <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(count, 0, 4, st);
  if (e != cudaSuccess) return e;
  const unsigned long long entries = (gt_mask + 1) * GT_BUCKET;
  gd_assign_kernel<<<152 * 8, 256, 0, st>>>(gt, entries, count, cap, owner);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // one short CTA per block, so that a drafting launch finds SMs between them
  // (the caller is the build's host thread: it may wait for the count)
  int32_t blocks = 0;
  e = cudaMemcpyAsync(h_count, count, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  blocks = *h_count < cap ? *h_count : cap;
  const size_t dyn = (size_t)(GD_CAND + R * ((k + 3) & ~3)) * 4;
  if (blocks > 0)
    gd_build_kernel<<<blocks, GD_THREADS, dyn, st>>>(gt, owner, keys, sa, text, n, Z, k, R, pN, pD, gd);
  return cudaGetLastError();
}

cudaError_t propose_set_smem_limit(size_t bytes) {
  // every instantiation may be launched with up to `bytes` of dynamic shared memory
  const void *fns[] = {
      (const void *)propose_kernel<384, 2, 0, false>, (const void *)propose_kernel<640, 1, 0, false>,
      (const void *)propose_kernel<384, 2, 3, false>, (const void *)propose_kernel<640, 1, 3, false>,
      (const void *)propose_kernel<256, 3, 1, false>, (const void *)propose_kernel<512, 1, 1, false>,
      (const void *)propose_kernel<128, 3, 2, false>, (const void *)propose_kernel<384, 2, 0, true>,
      (const void *)propose_kernel<640, 1, 0, true>,  (const void *)propose_kernel<256, 3, 1, true>,
      (const void *)propose_kernel<512, 1, 1, true>,  (const void *)propose_kernel<128, 3, 2, true>};
  for (const void *f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace sgd
