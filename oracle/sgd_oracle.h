/*
 * sgd_oracle.h -- CPU oracle for GPU-resident suffix decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C
 * restatement of what the drafter computes, written from the public pages'
 * description and used only by the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark.  The product path (the CUDA library)
 * never includes, links or calls anything here, and nothing here includes the
 * product's headers.
 *
 * Sources (page title, section):
 *   [RFC] "Suffix decoding on GPU (suffix_gpu)", vLLM issue: Summary, Design.
 *   [PYPI] "SuffixGPU" (suffix-gpu 0.1.1 on PyPI): Highlights, Quickstart,
 *          How it works (steps 1-4), References.
 *   [DOCS] "Suffix Decoding" (vLLM docs): Model Runner V2.
 *   [BLOG] "vLLM Suffix Decoding 投机解码实战": section 4 (config table),
 *          section 5 (proposer flow, max_model_len bound).
 *
 * Parity status: every function is pinned by tests (hand-worked examples,
 * brute force over every suffix length and occurrence, closed forms, the
 * suffix order invariant).  Agreement with the third-party CPU suffix tree
 * and with the prior Triton kernels is unpinned: neither is available.
 *
 * Error-flag bits returned by the functions below (the CUDA library reports
 * the same conditions with the same bit values, defined on its own side):
 */
#ifndef SGD_ORACLE_H
#define SGD_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_ERR_SAMPLED_TOKEN 0x1u  /* a sampled id >= V ended the accepted prefix      */
#define ORC_ERR_NUM_TOKENS    0x2u  /* num_tokens outside [0, S]; clamped               */
#define ORC_ERR_DOC_ARGS      0x4u  /* ingest: bad row/start/length; doc skipped        */
#define ORC_ERR_DOC_TOKEN     0x8u  /* ingest: token outside [0, V); doc truncated there */
#define ORC_ERR_DOC_TOO_LONG  0x10u /* ingest: doc + sentinel exceeds the ring; skipped  */

typedef struct {
  int32_t S;            /* row capacity; acts as max_model_len                    */
  int32_t V;            /* vocabulary size; the corpus sentinel Z equals V        */
  int32_t k;            /* max draft tokens                                        */
  int32_t D;            /* max_tree_depth                                          */
  int32_t R;            /* max_occurrences                                         */
  int64_t fN, fD;       /* max_spec_factor = fN / fD                               */
  int64_t offset;       /* max_spec_offset                                         */
  int64_t pN, pD;       /* min_token_prob = pN / pD                                */
  int32_t depth_sum_cap;/* 1: also bound the draft by D - M                        */
  int32_t fixed_length; /* 1: Model Runner V2 drafts ([DOCS] Model Runner V2): k
                           tokens always, slots without a voted continuation hold
                           the row's last token; factor, offset, min_token_prob
                           and depth_sum_cap unused                              */
  int32_t select_by_score; /* 1: the row's and the corpus's candidates are both
                           expanded and the better score wins ([PYPI] How it
                           works, step 3); 0: the longer match wins ([DOCS])    */
  int32_t num_backoff;  /* candidate lengths per path ([PYPI] How it works, steps
                           1-3: for t = 1..num_backoff the t-th largest match
                           length); > 1 ranks every candidate by score.  0 or 1:
                           the longest match only                               */
} orc_params;

/* Append the accepted prefix of one row's sampled ids ([PYPI] Quickstart,
 * propose_with_update; [RFC] Design, token bookkeeping). */
uint32_t orc_update_row(int32_t *row, int32_t *n, const int32_t *sampled,
                        int32_t T, int32_t S, int32_t V);

/* Longest suffix self-match; returns M, fills up to R positions, most recent
 * first ([DOCS] Model Runner V2, first bullet; [PYPI] How it works, step 1). */
int32_t orc_self_match(const int32_t *t, int32_t n, int32_t D, int32_t R,
                       int32_t *occ, int32_t *count);

/* Longest match of the row's tail inside the corpus text X (sentinel Z);
 * returns M (0 if below 2), fills up to R end positions, most recent first
 * ([DOCS] Model Runner V2, second bullet; [PYPI] How it works, step 2). */
int32_t orc_corpus_match(const int32_t *X, int64_t N, int32_t Z,
                         const int32_t *t, int32_t n, int32_t D, int32_t R,
                         int32_t *occ, int32_t *count);

/* Multi-length backoff ([PYPI] Highlights, "Multi-length backoff matching";
 * How it works, step 1): the distinct values among the nb largest entries of
 * the multiset {L(e)} over the path's ends (self: L >= 1, ends j <= n-2;
 * corpus: L >= 2, ends with a continuation), longest first.  Returns their
 * count; len[i] and support[i] (the number of ends with L >= len[i]). */
int32_t orc_backoff_lengths(const int32_t *L, int64_t nends, int32_t minlen,
                            int32_t nb, int32_t *len, int64_t *support);

/* One row: match, select, cap, frequency-greedy expansion. */
void orc_propose_row(const orc_params *p, const int32_t *t, int32_t n,
                     const int32_t *X, int64_t N, int32_t active,
                     int32_t *drafts, int32_t *num_valid, float *score,
                     float *probs, int32_t *match_info, uint32_t *flags);

/* Batch forms over row-major [B, S] buffers. */
uint32_t orc_update_state(int32_t *token_ids, int32_t *num_tokens,
                          const int32_t *sampled, int32_t B, int32_t T,
                          int32_t S, int32_t V);
uint32_t orc_propose(const orc_params *p, const int32_t *token_ids,
                     const int32_t *num_tokens, const uint8_t *active, int32_t B,
                     const int32_t *X, int64_t N, int32_t *drafts,
                     int32_t *num_valid, float *score, float *probs,
                     int32_t *match_info);

/* Suffix array by a plain comparison sort ([PYPI] References: suffix arrays). */
void orc_suffix_array(const int32_t *X, int64_t N, int32_t *SA);
/* 0 if SA is a permutation of [0, N) in strictly increasing suffix order,
 * else 1 + the first failing index. */
int64_t orc_check_suffix_array(const int32_t *X, int64_t N, const int32_t *SA);

/* FIFO corpus of finished responses ([PYPI] How it works, step 4;
 * [DOCS] Model Runner V2: oldest first out). */
typedef struct orc_ring orc_ring;
orc_ring *orc_ring_create(int64_t capacity, int32_t max_docs, int32_t V);
void orc_ring_destroy(orc_ring *r);
uint32_t orc_ring_ingest(orc_ring *r, const int32_t *token_ids,
                         const int32_t *num_tokens, int32_t B, int32_t S,
                         const int32_t *rows, const int32_t *starts,
                         const int32_t *lengths, int32_t m);
int64_t orc_ring_live(const orc_ring *r);
int32_t orc_ring_ndocs(const orc_ring *r);
/* Writes the live docs, oldest first, each followed by Z; returns the length. */
int64_t orc_ring_snapshot(const orc_ring *r, int32_t *X);
/* Docs placed so far (each placed doc, evicted or not, counts once). */
int64_t orc_ring_pushed(const orc_ring *r);
/* The docs not yet indexed by a snapshot taken when orc_ring_pushed() was
 * `since` ([PYPI] How it works, steps 2 and 4): the live docs with sequence
 * number >= since, oldest first, each followed by Z, cut after `cap` tokens.
 * Y holds at least min(cap, orc_ring_live(r)) ints; returns the length. */
int64_t orc_ring_delta(const orc_ring *r, int64_t since, int64_t cap, int32_t *Y);

#ifdef __cplusplus
}
#endif
#endif
