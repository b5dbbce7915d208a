/*
 * sgd_oracle.c -- CPU oracle for GPU-resident suffix decoding.
 *
 * TEST INFRASTRUCTURE ONLY (see sgd_oracle.h).  Plain, single-threaded,
 * written for readability: every step follows the definition on the pages,
 * with no blocking, fusion or reordering.  Source abbreviations are listed in
 * sgd_oracle.h.
 *
 * Readings taken where the pages are silent or disagree (each also listed in
 * the design notes of the repository):
 *   - an occurrence must have a continuation: self ends j <= n-2, corpus ends
 *     e with X[e+1] != Z;
 *   - only the longest match length votes, unless num_backoff > 1: then the
 *     t-th largest match lengths (t = 1..num_backoff) of each path are
 *     candidates too, each with its own ends, and the best score wins;
 *   - up to R occurrences are kept, the most recent (largest position) first;
 *   - vote ties go to the smallest token id;
 *   - chain probability P_d = |O_{d+1}| / |O_0|; a token is emitted iff
 *     P_d >= min_token_prob, decided on integers by cross-multiplication;
 *   - cap = min(k, floor(factor * M) + offset, S - n - 1);
 *   - self wins equal match lengths; the corpus needs a match of at least 2;
 *   - suffixes compare as signed int32, a proper prefix first.
 */
#include "sgd_oracle.h"

#include <stdlib.h>
#include <string.h>

static int32_t min32(int32_t a, int32_t b) { return a < b ? a : b; }
static int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

/* ------------------------------------------------------------------------ */
/* Update: [PYPI] Quickstart -- sampled_token_ids [B, T] is "-1 padded", and
 * propose_with_update appends the last verifier output to the resident buffer
 * before drafting; [RFC] Design -- the same device bookkeeping as ngram_gpu.
 * Only the leading run of valid ids is the accepted prefix.  An id >= V ends
 * the prefix and is reported.  Ids that would land at or past S are dropped
 * and n saturates at S. */
uint32_t orc_update_row(int32_t *row, int32_t *n_io, const int32_t *sampled,
                        int32_t T, int32_t S, int32_t V) {
  uint32_t flags = 0;
  int64_t n = *n_io;
  if (n < 0) { n = 0; flags |= ORC_ERR_NUM_TOKENS; }
  if (n > S) { n = S; flags |= ORC_ERR_NUM_TOKENS; }
  int32_t c = 0;
  while (c < T && sampled[c] >= 0 && sampled[c] < V) c++;
  if (c < T && sampled[c] >= V) flags |= ORC_ERR_SAMPLED_TOKEN;
  for (int32_t i = 0; i < c; i++)
    if (n + i < S) row[n + i] = sampled[i];
  *n_io = (int32_t)min64(S, n + c);
  return flags;
}

uint32_t orc_update_state(int32_t *token_ids, int32_t *num_tokens,
                          const int32_t *sampled, int32_t B, int32_t T,
                          int32_t S, int32_t V) {
  uint32_t flags = 0;
  for (int32_t b = 0; b < B; b++)
    flags |= orc_update_row(token_ids + (int64_t)b * S, &num_tokens[b],
                            sampled + (int64_t)b * T, T, S, V);
  return flags;
}

/* ------------------------------------------------------------------------ */
/* Self match: [DOCS] Model Runner V2 -- each request is matched against its
 * own prompt and output using the longest matching suffix, up to
 * max_tree_depth tokens; [PYPI] How it works, step 1 -- one backward pass
 * over the request's own context.
 *   L(j) = largest l <= min(D, j+1) with t[j-i] == t[n-1-i] for all i < l,
 *   for every candidate end j in [0, n-2];
 *   M = max_j L(j);  O = the (up to R) largest j with L(j) == M. */
int32_t orc_self_match(const int32_t *t, int32_t n, int32_t D, int32_t R,
                       int32_t *occ, int32_t *count) {
  *count = 0;
  if (n < 2 || D < 1) return 0;
  int32_t *L = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n - 1));
  int32_t M = 0;
  for (int32_t j = 0; j <= n - 2; j++) {
    int32_t lim = min32(D, j + 1);
    int32_t l = 0;
    while (l < lim && t[j - l] == t[n - 1 - l]) l++;
    L[j] = l;
    if (l > M) M = l;
  }
  if (M > 0) {
    for (int32_t j = n - 2; j >= 0 && *count < R; j--)
      if (L[j] == M) occ[(*count)++] = j;
  }
  free(L);
  return M;
}

/* ------------------------------------------------------------------------ */
/* Corpus match: [DOCS] Model Runner V2 -- finished responses are kept in a
 * corpus; every request looks up candidate positions by its last 2 and last 4
 * tokens and extends them to the longest suffix match, so corpus matching
 * needs a depth of at least 2.  Written here as the definition that probe
 * procedure computes, by a direct scan of every end position:
 *   valid end e in [0, N-2] with X[e+1] != Z (it has a continuation);
 *   Lc(e) = largest l <= min(D, n, e+1) with X[e-i] == t[n-1-i] for i < l;
 *   M = max over valid e if that is >= 2, else 0;
 *   O = the (up to R) largest valid e with Lc(e) == M (larger = more recent,
 *   since the text is ordered oldest to newest). */
static int32_t corpus_L(const int32_t *X, int64_t e, const int32_t *t,
                        int32_t n, int32_t D) {
  int64_t lim = min64(min64(D, n), e + 1);
  int32_t l = 0;
  while (l < lim && X[e - l] == t[n - 1 - l]) l++;
  return l;
}

int32_t orc_corpus_match(const int32_t *X, int64_t N, int32_t Z,
                         const int32_t *t, int32_t n, int32_t D, int32_t R,
                         int32_t *occ, int32_t *count) {
  *count = 0;
  if (D < 2 || N < 2 || n < 2 || X == NULL) return 0;
  int32_t M = 0;
  for (int64_t e = 0; e <= N - 2; e++) {
    if (X[e + 1] == Z) continue;
    int32_t l = corpus_L(X, e, t, n, D);
    if (l > M) M = l;
  }
  if (M < 2) return 0;
  for (int64_t e = N - 2; e >= 0 && *count < R; e--) {
    if (X[e + 1] == Z) continue;
    if (corpus_L(X, e, t, n, D) == M) occ[(*count)++] = (int32_t)e;
  }
  return M;
}

/* ------------------------------------------------------------------------ */
/* One row, [PYPI] How it works, step 3 and Highlights ("Score-ranked
 * expansion"); [DOCS] Model Runner V2 ("The longer match wins"); [BLOG]
 * section 4 (max_spec_factor * prefix_match_length; tokens whose estimated
 * probability is below min_token_prob are not proposed) and section 5 (the
 * draft never passes max_model_len - num_tokens - 1).
 *
 * Continuation of occurrence o at depth d (⊥ = none):
 *   self:   t[o+1+d]  if o+1+d <= n-1;
 *   corpus: X[o+1+d]  if o+1+d < N and X[o+1+d] != Z.
 * Depth-wise majority vote: tau_d = the most frequent continuation among the
 * surviving occurrences (ties: smallest id); survivors = those that continue
 * with tau_d; P_d = |survivors| / |O_0|; stop before emitting when
 * P_d < min_token_prob; score = sum of the emitted P_d. */
static int32_t cont_of(int32_t source, const int32_t *t, int32_t n,
                       const int32_t *X, int64_t N, int32_t Z, int32_t o,
                       int32_t d, int32_t *tok) {
  int64_t q = (int64_t)o + 1 + d;
  if (source == 1) {
    if (q > n - 1) return 0;
    *tok = t[q];
    return 1;
  }
  if (q >= N || X[q] == Z) return 0;
  *tok = X[q];
  return 1;
}

/* Frequency-greedy expansion of one candidate (source 1: the row's own ends,
 * 2: the corpus ends; M its match length, occ its c0 ends): the draft into
 * drafts / probs (left as they are past the emitted tokens), the number of
 * tokens emitted and the sum of their vote counts (score = sum / c0). */
static void expand(const orc_params *p, int32_t source, const int32_t *t, int32_t n,
                   const int32_t *X, int64_t N, int32_t Z, const int32_t *occ, int32_t c0,
                   int32_t M, int32_t *drafts, float *probs, int32_t *len_out,
                   int64_t *sum_out) {
  *len_out = 0;
  *sum_out = 0;
  if (M == 0 || c0 == 0) return;
  /* length cap (Model Runner V2: no factor, only k and the context) */
  int64_t cap = p->k;
  if (!p->fixed_length) cap = min64(cap, (p->fN * (int64_t)M) / p->fD + p->offset);
  int64_t room = (int64_t)p->S - n - 1;
  if (room < 0) room = 0;
  cap = min64(cap, room);
  if (p->depth_sum_cap && !p->fixed_length) cap = min64(cap, (int64_t)p->D - M);
  if (cap < 0) cap = 0;

  uint8_t *alive = (uint8_t *)malloc((size_t)c0);
  int32_t *val = (int32_t *)malloc(sizeof(int32_t) * (size_t)c0);
  uint8_t *has = (uint8_t *)malloc((size_t)c0);
  for (int32_t o = 0; o < c0; o++) alive[o] = 1;
  int64_t sum = 0;
  int32_t len = 0;
  for (int32_t d = 0; d < cap; d++) {
    int32_t any = 0;
    for (int32_t o = 0; o < c0; o++) {
      has[o] = alive[o] && cont_of(source, t, n, X, N, Z, occ[o], d, &val[o]);
      any |= has[o];
    }
    if (!any) break;
    int32_t best_cnt = 0, best_tok = 0;
    for (int32_t o = 0; o < c0; o++) {
      if (!has[o]) continue;
      int32_t cnt = 0;
      for (int32_t q = 0; q < c0; q++)
        if (has[q] && val[q] == val[o]) cnt++;
      if (cnt > best_cnt || (cnt == best_cnt && val[o] < best_tok)) {
        best_cnt = cnt;
        best_tok = val[o];
      }
    }
    if (!p->fixed_length && (int64_t)best_cnt * p->pD < p->pN * (int64_t)c0) break;
    drafts[d] = best_tok;
    if (probs) probs[d] = (float)((double)best_cnt / (double)c0);
    sum += best_cnt;
    len++;
    for (int32_t o = 0; o < c0; o++) alive[o] = has[o] && val[o] == best_tok;
  }
  free(alive); free(val); free(has);
  *len_out = len;
  *sum_out = sum;
}

/* ------------------------------------------------------------------------ */
/* Multi-length backoff: [PYPI] Highlights ("Multi-length backoff matching":
 * the longest suffix plus shorter, better-supported lengths) and How it
 * works, steps 1-3 (for support threshold t the largest length occurring at
 * least t times, i.e. the t-th largest match_back value; every candidate is
 * expanded and scored, the best wins per path and the two winners compete by
 * the same score).  The thresholds t = 1..nb name at most nb distinct
 * lengths: each is found by a plain scan for the largest value below the
 * previous one, until nb ends are covered. */
int32_t orc_backoff_lengths(const int32_t *L, int64_t nends, int32_t minlen,
                            int32_t nb, int32_t *len, int64_t *support) {
  int32_t cnt = 0, prev = INT32_MAX;
  int64_t covered = 0; /* ends with L >= the last length found: thresholds 1..covered */
  while (covered < nb) {
    int32_t best = 0;
    for (int64_t e = 0; e < nends; e++)
      if (L[e] >= minlen && L[e] < prev && L[e] > best) best = L[e];
    if (best == 0) break;
    int64_t sup = 0;
    for (int64_t e = 0; e < nends; e++)
      if (L[e] >= best) sup++;
    len[cnt] = best;
    support[cnt] = sup;
    cnt++;
    covered = sup;
    prev = best;
  }
  return cnt;
}

/* Backoff selection for one row (p->num_backoff > 1).  The self lengths L(j)
 * and corpus lengths Lc(e) are those of orc_self_match / orc_corpus_match
 * (an end without a continuation has none).  A candidate (path, length l)
 * votes with the R most recent ends of L >= l, capped as a match of length l.
 * Best: the higher score sum / c0 (exact), then the longer length, then the
 * row itself.  Writes the winner's draft, probabilities and (M, source, c0,
 * len, sum); M = 0 when neither path has a candidate. */
static void propose_backoff(const orc_params *p, const int32_t *t, int32_t n,
                            const int32_t *X, int64_t N, int32_t Z, int32_t *drafts,
                            float *probs, int32_t *M_out, int32_t *source_out,
                            int32_t *c0_out, int32_t *len_out, int64_t *sum_out) {
  const int32_t nb = p->num_backoff;
  const int32_t k = p->k;
  int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
  int32_t *d2 = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
  float *p2 = (float *)malloc(sizeof(float) * (size_t)k);
  int32_t *occ = (int32_t *)malloc(sizeof(int32_t) * (size_t)p->R);
  int32_t *lens = (int32_t *)malloc(sizeof(int32_t) * (size_t)nb);
  int64_t *sup = (int64_t *)malloc(sizeof(int64_t) * (size_t)nb);
  for (int32_t d = 0; d < k; d++) fill[d] = drafts[d];
  *M_out = 0; *source_out = 0; *c0_out = 0; *len_out = 0; *sum_out = 0;
  for (int32_t source = 1; source <= 2; source++) {
    int64_t nends = 0;
    int32_t *L = NULL;
    if (source == 1 && n >= 2 && p->D >= 1) {
      nends = n - 1;
      L = (int32_t *)malloc(sizeof(int32_t) * (size_t)nends);
      for (int32_t j = 0; j <= n - 2; j++) {
        int32_t lim = min32(p->D, j + 1), l = 0;
        while (l < lim && t[j - l] == t[n - 1 - l]) l++;
        L[j] = l;
      }
    } else if (source == 2 && X != NULL && N >= 2 && n >= 2 && p->D >= 2) {
      nends = N - 1;
      L = (int32_t *)malloc(sizeof(int32_t) * (size_t)nends);
      for (int64_t e = 0; e <= N - 2; e++)
        L[e] = X[e + 1] == Z ? 0 : corpus_L(X, e, t, n, p->D);
    }
    if (L == NULL) continue;
    const int32_t nl = orc_backoff_lengths(L, nends, source == 1 ? 1 : 2, nb, lens, sup);
    for (int32_t i = 0; i < nl; i++) {
      int32_t c0 = 0;
      for (int64_t e = nends - 1; e >= 0 && c0 < p->R; e--)
        if (L[e] >= lens[i]) occ[c0++] = (int32_t)e;
      for (int32_t d = 0; d < k; d++) { d2[d] = fill[d]; p2[d] = 0.0f; }
      int32_t len;
      int64_t sum;
      expand(p, source, t, n, X, N, Z, occ, c0, lens[i], d2, p2, &len, &sum);
      int better = *M_out == 0;
      if (!better) {
        const int64_t lhs = sum * *c0_out, rhs = *sum_out * c0;
        better = lhs > rhs || (lhs == rhs && lens[i] > *M_out);
      }
      if (better) {
        *M_out = lens[i]; *source_out = source; *c0_out = c0; *len_out = len; *sum_out = sum;
        for (int32_t d = 0; d < k; d++) { drafts[d] = d2[d]; if (probs) probs[d] = p2[d]; }
      }
    }
    free(L);
  }
  free(fill); free(d2); free(p2); free(occ); free(lens); free(sup);
}

void orc_propose_row(const orc_params *p, const int32_t *t, int32_t n_in,
                     const int32_t *X, int64_t N, int32_t active,
                     int32_t *drafts, int32_t *num_valid, float *score,
                     float *probs, int32_t *match_info, uint32_t *flags) {
  for (int32_t d = 0; d < p->k; d++) {
    drafts[d] = -1;
    if (probs) probs[d] = 0.0f;
  }
  *num_valid = 0;
  if (score) *score = 0.0f;
  if (match_info) { match_info[0] = 0; match_info[1] = 0; }

  int32_t n = n_in;
  if (n < 0) { n = 0; *flags |= ORC_ERR_NUM_TOKENS; }
  if (n > p->S) { n = p->S; *flags |= ORC_ERR_NUM_TOKENS; }
  if (!active || n == 0) return;

  const int32_t Z = p->V;
  int32_t *occ_s = (int32_t *)malloc(sizeof(int32_t) * (size_t)p->R);
  int32_t *occ_c = (int32_t *)malloc(sizeof(int32_t) * (size_t)p->R);
  int32_t cs = 0, cc = 0;
  int32_t Ms = orc_self_match(t, n, p->D, p->R, occ_s, &cs);
  int32_t Mc = (X != NULL && N > 0)
                   ? orc_corpus_match(X, N, Z, t, n, p->D, p->R, occ_c, &cc)
                   : 0;

  /* Model Runner V2 drafts: the slots the vote leaves empty hold the row's
   * last token, all k of them when there is no match ([DOCS] Model Runner V2) */
  if (p->fixed_length)
    for (int32_t d = 0; d < p->k; d++) drafts[d] = t[n - 1];

  int32_t source, M, c0, len = 0;
  int64_t sum = 0;
  if (p->num_backoff > 1) {
    propose_backoff(p, t, n, X, N, Z, drafts, probs, &M, &source, &c0, &len, &sum);
  } else if (p->select_by_score && Ms > 0 && Mc > 0) {
    /* [PYPI] How it works, step 3: both candidates are expanded and the
     * better score (sum / c0, compared exactly) wins; equal scores go to the
     * longer match, then to the row itself */
    int32_t *d2 = (int32_t *)malloc(sizeof(int32_t) * (size_t)p->k);
    float *p2 = (float *)malloc(sizeof(float) * (size_t)p->k);
    for (int32_t d = 0; d < p->k; d++) { d2[d] = drafts[d]; p2[d] = probs ? probs[d] : 0.0f; }
    int32_t len_c;
    int64_t sum_c;
    expand(p, 1, t, n, X, N, Z, occ_s, cs, Ms, drafts, probs, &len, &sum);
    expand(p, 2, t, n, X, N, Z, occ_c, cc, Mc, d2, p2, &len_c, &sum_c);
    const int64_t lhs = sum_c * cs, rhs = sum * cc;  /* score_c vs score_s */
    if (lhs > rhs || (lhs == rhs && Mc > Ms)) {
      source = 2; M = Mc; c0 = cc; len = len_c; sum = sum_c;
      for (int32_t d = 0; d < p->k; d++) { drafts[d] = d2[d]; if (probs) probs[d] = p2[d]; }
    } else {
      source = 1; M = Ms; c0 = cs;
    }
    free(d2); free(p2);
  } else {
    /* the longer match wins; equal lengths stay with the request itself */
    const int32_t *occ;
    if (Mc > Ms) { source = 2; M = Mc; occ = occ_c; c0 = cc; }
    else { source = Ms > 0 ? 1 : 0; M = Ms; occ = occ_s; c0 = cs; }
    expand(p, source, t, n, X, N, Z, occ, c0, M, drafts, probs, &len, &sum);
  }
  if (match_info) { match_info[0] = M; match_info[1] = source; }
  *num_valid = p->fixed_length ? p->k : len;
  if (score && M > 0 && c0 > 0) *score = (float)((double)sum / (double)c0);
  free(occ_s); free(occ_c);
}

uint32_t orc_propose(const orc_params *p, const int32_t *token_ids,
                     const int32_t *num_tokens, const uint8_t *active, int32_t B,
                     const int32_t *X, int64_t N, int32_t *drafts,
                     int32_t *num_valid, float *score, float *probs,
                     int32_t *match_info) {
  uint32_t flags = 0;
  for (int32_t b = 0; b < B; b++)
    orc_propose_row(p, token_ids + (int64_t)b * p->S, num_tokens[b], X, N,
                    active ? active[b] : 1, drafts + (int64_t)b * p->k,
                    &num_valid[b], score ? &score[b] : NULL,
                    probs ? probs + (int64_t)b * p->k : NULL,
                    match_info ? match_info + 2 * (int64_t)b : NULL, &flags);
  return flags;
}

/* ------------------------------------------------------------------------ */
/* Suffix array: [PYPI] References (Manber & Myers) and How it works, step 4.
 * The order itself is the definition: suffixes compared token by token as
 * signed int32, a proper prefix before its extensions.  Sorted here by a
 * plain bottom-up merge sort of the start positions. */
static int suffix_less(const int32_t *X, int64_t N, int64_t a, int64_t b) {
  while (a < N && b < N) {
    if (X[a] != X[b]) return X[a] < X[b];
    a++;
    b++;
  }
  return a == N && b != N; /* the one that ended first is smaller */
}

void orc_suffix_array(const int32_t *X, int64_t N, int32_t *SA) {
  if (N <= 0) return;
  int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
  for (int64_t i = 0; i < N; i++) SA[i] = (int32_t)i;
  for (int64_t w = 1; w < N; w *= 2) {
    for (int64_t lo = 0; lo < N; lo += 2 * w) {
      int64_t mid = min64(lo + w, N), hi = min64(lo + 2 * w, N);
      int64_t i = lo, j = mid, o = lo;
      while (i < mid && j < hi)
        tmp[o++] = suffix_less(X, N, SA[j], SA[i]) ? SA[j++] : SA[i++];
      while (i < mid) tmp[o++] = SA[i++];
      while (j < hi) tmp[o++] = SA[j++];
    }
    memcpy(SA, tmp, sizeof(int32_t) * (size_t)N);
  }
  free(tmp);
}

int64_t orc_check_suffix_array(const int32_t *X, int64_t N, const int32_t *SA) {
  uint8_t *seen = (uint8_t *)calloc((size_t)(N > 0 ? N : 1), 1);
  int64_t bad = 0;
  for (int64_t i = 0; i < N && !bad; i++) {
    if (SA[i] < 0 || SA[i] >= N || seen[SA[i]]) bad = i + 1;
    else seen[SA[i]] = 1;
  }
  for (int64_t i = 0; i + 1 < N && !bad; i++)
    if (!suffix_less(X, N, SA[i], SA[i + 1])) bad = i + 1;
  free(seen);
  return bad;
}

/* ------------------------------------------------------------------------ */
/* Corpus of finished responses: [PYPI] How it works, step 4 (oldest
 * documents are evicted when the ring is full); [DOCS] Model Runner V2
 * (a token budget, oldest first out).  Modelled as a plain FIFO of documents;
 * each doc occupies len + 1 tokens (its sentinel).  The FIFO also holds at
 * most max_docs documents. */
struct orc_ring {
  int64_t C;
  int32_t max_docs, V;
  int32_t **doc;   /* FIFO storage, index (head + i) % max_docs */
  int32_t *len;
  int32_t head, ndocs;
  int64_t live;
  int64_t pushed;  /* docs ever placed; the doc at FIFO index i has sequence
                      number pushed - ndocs + i */
};

orc_ring *orc_ring_create(int64_t capacity, int32_t max_docs, int32_t V) {
  orc_ring *r = (orc_ring *)calloc(1, sizeof(orc_ring));
  r->C = capacity;
  r->max_docs = max_docs;
  r->V = V;
  r->doc = (int32_t **)calloc((size_t)max_docs, sizeof(int32_t *));
  r->len = (int32_t *)calloc((size_t)max_docs, sizeof(int32_t));
  return r;
}

void orc_ring_destroy(orc_ring *r) {
  if (!r) return;
  for (int32_t i = 0; i < r->max_docs; i++) free(r->doc[i]);
  free(r->doc);
  free(r->len);
  free(r);
}

static void ring_evict_oldest(orc_ring *r) {
  r->live -= (int64_t)r->len[r->head] + 1;
  free(r->doc[r->head]);
  r->doc[r->head] = NULL;
  r->head = (r->head + 1) % r->max_docs;
  r->ndocs--;
}

uint32_t orc_ring_ingest(orc_ring *r, const int32_t *token_ids,
                         const int32_t *num_tokens, int32_t B, int32_t S,
                         const int32_t *rows, const int32_t *starts,
                         const int32_t *lengths, int32_t m) {
  uint32_t flags = 0;
  for (int32_t i = 0; i < m; i++) {
    int32_t row = rows[i], st = starts[i], ln = lengths[i];
    if (row < 0 || row >= B || st < 0 || ln < 0 || (int64_t)st + ln > S ||
        (num_tokens && (int64_t)st + ln > num_tokens[row])) {
      flags |= ORC_ERR_DOC_ARGS;
      continue;
    }
    const int32_t *src = token_ids + (int64_t)row * S + st;
    int32_t eff = 0;
    while (eff < ln && src[eff] >= 0 && src[eff] < r->V) eff++;
    if (eff < ln) flags |= ORC_ERR_DOC_TOKEN;
    if (eff == 0) continue;
    if ((int64_t)eff + 1 > r->C) {
      flags |= ORC_ERR_DOC_TOO_LONG;
      continue;
    }
    while (r->live + eff + 1 > r->C || r->ndocs == r->max_docs)
      ring_evict_oldest(r);
    int32_t slot = (r->head + r->ndocs) % r->max_docs;
    r->doc[slot] = (int32_t *)malloc(sizeof(int32_t) * (size_t)eff);
    memcpy(r->doc[slot], src, sizeof(int32_t) * (size_t)eff);
    r->len[slot] = eff;
    r->ndocs++;
    r->live += (int64_t)eff + 1;
    r->pushed++;
  }
  return flags;
}

int64_t orc_ring_live(const orc_ring *r) { return r->live; }
int32_t orc_ring_ndocs(const orc_ring *r) { return r->ndocs; }
int64_t orc_ring_pushed(const orc_ring *r) { return r->pushed; }

int64_t orc_ring_snapshot(const orc_ring *r, int32_t *X) {
  int64_t pos = 0;
  for (int32_t i = 0; i < r->ndocs; i++) {
    int32_t slot = (r->head + i) % r->max_docs;
    memcpy(X + pos, r->doc[slot], sizeof(int32_t) * (size_t)r->len[slot]);
    pos += r->len[slot];
    X[pos++] = r->V;
  }
  return pos;
}

/* ------------------------------------------------------------------------ */
/* Delta: [PYPI] How it works, step 2 (global matching also scans, by brute
 * force, the buffer of documents not yet in the suffix array) and step 4 (new
 * documents append to that buffer until a rebuild indexes them).  The docs
 * not yet indexed by a snapshot are those placed after it was taken: the live
 * docs whose sequence number is >= `since` (the ring's pushed count when the
 * snapshot was linearised), oldest first, each followed by Z.  The buffer
 * holds at most `cap` tokens: what does not fit waits for the next rebuild,
 * and a doc cut by the capacity is visible up to the cut.  The corpus a row
 * is matched against is then the snapshot followed by this text. */
int64_t orc_ring_delta(const orc_ring *r, int64_t since, int64_t cap, int32_t *Y) {
  int64_t pos = 0;
  for (int32_t i = 0; i < r->ndocs && pos < cap; i++) {
    if (r->pushed - r->ndocs + i < since) continue;
    int32_t slot = (r->head + i) % r->max_docs;
    for (int32_t j = 0; j <= r->len[slot] && pos < cap; j++)
      Y[pos++] = j < r->len[slot] ? r->doc[slot][j] : r->V;
  }
  return pos;
}
