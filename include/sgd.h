/*
 * sgd.h -- C ABI of the GPU-resident suffix-decoding drafter (libsgd).
 *
 * One library context per GPU.  All drafting work runs in hand-written CUDA
 * kernels for sm_103a on streams the caller passes; no call on the drafting
 * path synchronises with the host, allocates memory or changes a device
 * address, so sgd_update_state / sgd_propose / sgd_propose_with_update /
 * sgd_ingest / sgd_step can be captured in a CUDA graph.
 *
 * Sources (page title, section):
 *   [RFC]  "Suffix decoding on GPU (suffix_gpu)", vLLM issue: Summary, Design.
 *   [PYPI] "SuffixGPU" (suffix-gpu 0.1.1 on PyPI): Highlights, Quickstart,
 *          How it works (steps 1-4), References.
 *   [DOCS] "Suffix Decoding" (vLLM docs): Model Runner V2.
 *   [BLOG] "vLLM Suffix Decoding 投机解码实战": section 4 (knob defaults),
 *          section 5 (proposer flow).
 *
 * Conventions for every entry point below:
 *   - Return value: an SGD_* status.  Negative values are errors detected on
 *     the host before anything was enqueued (nothing ran), or a CUDA error.
 *   - Pointers marked DEVICE are caller-owned device memory of the context's
 *     GPU; the library never frees or keeps them past the call's stream work.
 *     Token buffers must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Problems found on the device (bad token ids, out-of-range lengths) are
 *     never traps: they set bits in a sticky device word (SGD_ERR_*), read by
 *     sgd_get_error, and the offending id or document is treated as a stop.
 *   - A context is not thread-safe: call it from one host thread at a time.
 */
#ifndef SGD_H
#define SGD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define SGD_OK          0   /* done (sgd_poll: nothing new to swap in)          */
#define SGD_OK_SWAPPED  1   /* sgd_poll: a finished suffix array is now current */
#define SGD_PENDING     2   /* sgd_poll: a build is still running               */
#define SGD_EINVAL     -1   /* bad argument (sizes, alignment, NULL)            */
#define SGD_ECUDA      -2   /* a CUDA runtime call failed                       */
#define SGD_ENOMEM     -3   /* device or host allocation failed in sgd_create   */
#define SGD_ETIMEDOUT  -4   /* sgd_poll(wait=1) ran out of time                 */
#define SGD_EBUSY      -5   /* a build is in flight or not yet swapped in       */
#define SGD_EBUILD     -6   /* the finished build reported failure; old index kept */
#define SGD_ENOCORPUS  -7   /* the context was created without a corpus         */
#define SGD_ETOOLARGE  -8   /* longer than the fixed scratch of sgd_suffix_array_noalloc */
#define SGD_EIO        -9   /* sgd_save / sgd_load: the file could not be written or read */

/* ---- sticky device error bits (sgd_get_error) --------------------------- */
#define SGD_ERR_SAMPLED_TOKEN 0x1u  /* a sampled id >= V ended the accepted prefix    */
#define SGD_ERR_NUM_TOKENS    0x2u  /* num_tokens outside [0, S]; clamped             */
#define SGD_ERR_DOC_ARGS      0x4u  /* ingest: bad row/start/length; doc skipped      */
#define SGD_ERR_DOC_TOKEN     0x8u  /* ingest: token outside [0, V); doc truncated    */
#define SGD_ERR_DOC_TOO_LONG  0x10u /* ingest: doc + sentinel exceeds the ring; skipped */
#define SGD_ERR_LOOKBACK      0x20u /* suffix sort: a radix look-back gave up waiting */
#define SGD_ERR_INGEST_WAIT   0x40u /* sgd_step: a doc's row update never showed; doc skipped */

typedef struct sgd_ctx sgd_ctx; /* opaque, library-owned */

/* Knobs.  Defaults (sgd_config_default) follow [BLOG] section 4 and
 * [DOCS] Model Runner V2: max_tree_depth 24, max_spec_factor 1.0,
 * min_token_prob 0.1, offset 0, corpus of 2^20 tokens; k = 16 and
 * max_occurrences = 64.  Floating knobs are kept as rationals so that every
 * stop decision is an integer cross-multiplication. */
typedef struct {
  int32_t  max_batch;          /* rows B the context may be called with            */
  int32_t  seq_capacity;       /* S: row stride of token_ids and max context; S % 4 == 0 */
  int32_t  vocab_size;         /* V: ids are in [0, V); the corpus sentinel is V   */
  int32_t  k;                  /* draft width (1..64)                              */
  int32_t  max_tree_depth;     /* D: longest match considered (1..128)             */
  int32_t  max_occurrences;    /* R: occurrences voting per row (1..128)           */
  int32_t  max_sampled;        /* largest T passed to the update (1..1024)         */
  uint32_t spec_factor_num;    /* max_spec_factor = num / den (den > 0)            */
  uint32_t spec_factor_den;
  int32_t  spec_offset;        /* max_spec_offset                                   */
  uint32_t min_prob_num;       /* min_token_prob = num / den (den > 0, num <= den)  */
  uint32_t min_prob_den;
  int32_t  depth_sum_cap;      /* 1: also bound the draft by D - M (CPU-tree style) */
  int64_t  corpus_capacity;    /* ring tokens incl. sentinels (0: no corpus); <= 2^30 */
  int32_t  max_docs;           /* documents the ring can hold at once              */
  int32_t  max_ingest_docs;    /* documents per sgd_ingest call                    */
  int32_t  corpus_cand_cap;    /* power of two >= R: on-chip candidate buffer of the
                                  corpus occurrence selection (larger match sets take
                                  an exact multi-pass path)                        */
  int32_t  self_warps;         /* warps scanning each row (0: chosen from B and S) */
  int32_t  corpus_records;     /* 1 (default): each snapshot also holds, per suffix-array
                                  position, the suffix's position, the D-4 tokens before
                                  it and the k tokens after its first four, so that a
                                  small 4-token interval is evaluated from one read;
                                  4*roundup4(1+max(D-4,0)+k) bytes per corpus token per
                                  snapshot, used only while both snapshots' records fit
                                  in SGD_RECORD_BUDGET bytes.  0: off.  Drafts are the
                                  same either way. */
  int32_t  corpus_gram_index;  /* 1 (default): each snapshot also holds a hash table from
                                  every distinct 2-, 3- and 4-gram that begins a suffix
                                  to its suffix-array interval, so that the probe finds
                                  an interval in one read instead of a descent;
                                  128 * next_pow2(corpus_capacity) bytes per snapshot,
                                  used only while both snapshots' tables fit in
                                  SGD_RECORD_BUDGET bytes.  0: off (descent of the key
                                  array).  Drafts are the same either way. */
  int32_t  propose_mode;       /* 0 (default) or 1: each propose is one kernel launch
                                  (a CTA per row scans its row while probing the
                                  corpus).  2: two launches, the update and self match
                                  in small CTAs (more per SM), then the corpus chain and
                                  vote.  Drafts are the same either way; on the long-
                                  context workload mode 1 is currently the faster. */
  int64_t  delta_capacity;     /* 0 (default): a doc becomes matchable once a suffix array
                                  built after its ingest is swapped in.  > 0: the docs
                                  placed since the current snapshot was linearised (the
                                  delta, [PYPI] How it works, steps 2 and 4) are matched
                                  too: up to delta_capacity of their tokens (sentinels
                                  included), oldest first; a doc cut by the capacity is
                                  visible up to the cut and the rest waits for the next
                                  swap.  The corpus a row matches is then the snapshot
                                  followed by that text; delta ends count as more recent
                                  than snapshot ends.  Every delta position is accounted
                                  for, as by a brute-force scan, but each row reads only
                                  the 128-token ring windows whose 2/3/4-gram signature
                                  (kept with the ring: 8 bytes per ring token) can hold
                                  an end that matters.  Requires corpus_capacity to be a
                                  multiple of 128; <= corpus_capacity. */
  int32_t  draft_mode;         /* 0 (default): the draft stops where the vote's chain
                                  probability falls below min_token_prob or at
                                  floor(max_spec_factor * M) + max_spec_offset tokens;
                                  -1 padded.  1: Model Runner V2 drafts ([DOCS] Model
                                  Runner V2): always k tokens -- the vote runs while an
                                  occurrence continues (within k and the context), the
                                  slots it leaves hold the row's last token (probability
                                  0), num_valid = k; max_spec_factor, max_spec_offset,
                                  min_token_prob and depth_sum_cap are not used.  Rows
                                  that are inactive or empty stay -1 / 0 either way. */
  int32_t  select_by_score;    /* 0 (default): the longer match wins, the row's own at
                                  equal length ([DOCS] Model Runner V2).  1: the row's and
                                  the corpus's longest-match candidates are both voted
                                  and the better score (expected accepted tokens, the sum
                                  of the emitted probabilities) wins; equal scores go to
                                  the longer match, then to the row ([PYPI] How it works,
                                  step 3).  The corpus candidate is then always found in
                                  full (no pruning by the row's match). */
  int32_t  num_backoff;        /* 1 (default): one candidate length per path, the longest
                                  match.  2..8: multi-length backoff ([PYPI] Highlights,
                                  How it works, steps 1-3): for each support threshold
                                  t = 1..num_backoff the t-th largest match length of the
                                  path (the row: lengths >= 1; the corpus, snapshot and
                                  delta together: >= 2) is a candidate, voted with the R
                                  most recent ends reaching that length and capped as a
                                  match of that length; every candidate of both paths is
                                  ranked by score as with select_by_score = 1 (equal
                                  scores: the longer length, then the row), whatever
                                  select_by_score says.  The match lengths are exact
                                  (every row end, every corpus end matching the last two
                                  tokens, every delta position): this mode runs its own
                                  kernel (the update included, one launch like the
                                  default; a step's ingest is a second launch), which
                                  scans the row and the suffix-array interval of the
                                  shortest of the row's last 2-, 3-, 4-gram that has no
                                  gram draft block (gram_drafts; without them, or with
                                  delta ends, that of the last two tokens). */
  int32_t  row_index;          /* 0 (default): each step scans every row's valid tokens
                                  for its own match.  1: each row also keeps a bigram
                                  position index on the device (the per-request
                                  structure of the [RFC] Summary), kept current by every
                                  update, so that a step reads only the earlier
                                  positions of the row's last two tokens, extended
                                  backwards, instead of the whole row; a row whose
                                  last bigram occurs more than 12 times, or not at all
                                  when the corpus has no match of 2 or more, is still
                                  scanned.  Drafts are the same either way.  The
                                  caller must call sgd_reset_rows for every row it
                                  writes other than through this library's updates
                                  (a new request in a row, rows written before the
                                  first step); a row whose length changed unseen is
                                  scanned until it is reset.  Requires propose_mode 0,
                                  delta_capacity 0, select_by_score 0, num_backoff 1
                                  and vocab_size <= 2^24; 64 * next_pow2(2 S) bytes
                                  per row (max_batch rows). */
  int32_t  gram_drafts;        /* 1 (default, with corpus_gram_index): each snapshot also
                                  holds, for every 2- and 3-token gram whose suffix-array
                                  interval has 8 or more hits, the R most recent of its
                                  ends that continue and their vote to depth k, so that a
                                  row whose corpus match is such a gram reads its draft
                                  (cut at the row's cap) instead of evaluating the
                                  interval and voting; up to corpus_capacity / 4 grams,
                                  (16 + 8 roundup4(k)) bytes each, per snapshot, used only
                                  while both snapshots' blocks fit in SGD_RECORD_BUDGET.
                                  0: off.  Drafts are the same either way. */
} sgd_config;

#define SGD_RECORD_BUDGET (8ull << 30)

/* Fills *cfg with the defaults above (max_batch 256, S 4096, V 151936). */
int sgd_config_default(sgd_config *cfg);

/* Sets max_spec_factor and min_token_prob from floats, as x rounded to a
 * multiple of 1e-6 (exact for 0.1, 1.0, 2.0, ...).  SGD_EINVAL if negative
 * or min_token_prob > 1. */
int sgd_config_set_float(sgd_config *cfg, double max_spec_factor, double min_token_prob);

/* Creates a context on `device` and allocates everything it will ever use:
 * ring, document FIFO, two suffix-array snapshots, the device descriptor of
 * the current snapshot, scratch and streams-independent events.
 * SGD_EINVAL for knobs out of range, SGD_ENOMEM / SGD_ECUDA on failure
 * (nothing is leaked). */
int sgd_create(const sgd_config *cfg, int device, sgd_ctx **out);

/* Waits for an in-flight build, then frees everything the context owns. */
int sgd_destroy(sgd_ctx *ctx);

/* Appends each row's accepted sampled ids ([PYPI] Quickstart: sampled ids
 * [B, T] are -1 padded; [RFC] Design: the ngram_gpu token bookkeeping).
 *   token_ids  DEVICE int32 [B, S] row-major, updated in place.
 *   num_tokens DEVICE int32 [B], updated in place.
 *   sampled    DEVICE int32 [B, T].
 * Row b takes the leading run of ids in [0, V) of sampled[b, :]; an id >= V
 * ends the run and sets SGD_ERR_SAMPLED_TOKEN.  Ids landing at or past S are
 * dropped; num_tokens saturates at S (values outside [0, S] are clamped and
 * set SGD_ERR_NUM_TOKENS).  B <= max_batch, 1 <= T <= max_sampled. */
int sgd_update_state(sgd_ctx *ctx, int32_t *token_ids, int32_t *num_tokens,
                     const int32_t *sampled, int32_t B, int32_t T, void *stream);

/* Drafts up to k tokens per row ([PYPI] How it works, steps 1-3; [DOCS]
 * Model Runner V2; [BLOG] sections 4-5):
 *   1. longest suffix self-match of the row's tail in its own context (length
 *      <= D; ends j <= n-2), keeping the R most recent ends of that length;
 *   2. corpus lookup through the current suffix array: the last 4 (else last
 *      2) tokens are searched and every hit is extended backwards to the
 *      longest match (length >= 2, <= D; only ends with a continuation), the
 *      R most recent ends kept;
 *   3. the longer match wins (equal lengths: the row itself);
 *   4. cap = min(k, floor(factor * M) + offset, S - n - 1) [, D - M];
 *   5. depth by depth the surviving occurrences vote on their next token
 *      (ties: smallest id); the winner is emitted while |survivors| / c0 >=
 *      min_token_prob (integer cross-multiplication).
 *   token_ids  DEVICE int32 [B, S];  num_tokens DEVICE int32 [B] (clamped to [0, S]).
 *   active     DEVICE uint8 [B] or NULL (all rows); a 0 row drafts nothing.
 *   drafts     DEVICE int32 [B, k]: draft ids, then -1.
 *   num_valid  DEVICE int32 [B].
 *   score      DEVICE float [B] or NULL: sum of the emitted chain probabilities,
 *              float(integer sum / c0) rounded from double.
 *   probs      DEVICE float [B, k] or NULL: chain probability per emitted slot, 0 after.
 *   match_info DEVICE int32 [B, 2] or NULL: {M, source} with source 0 = no
 *              match, 1 = the row itself, 2 = corpus.
 * One kernel launch on `stream`; reads the snapshot current at launch time. */
int sgd_propose(sgd_ctx *ctx, const int32_t *token_ids, const int32_t *num_tokens,
                const uint8_t *active, int32_t B, int32_t *drafts, int32_t *num_valid,
                float *score, float *probs, int32_t *match_info, void *stream);

/* sgd_update_state followed by sgd_propose, fused into one kernel launch
 * ([PYPI] Quickstart: propose_with_update).  The update applies to every row;
 * `active` masks only the drafting. */
int sgd_propose_with_update(sgd_ctx *ctx, int32_t *token_ids, int32_t *num_tokens,
                            const int32_t *sampled, int32_t T, const uint8_t *active,
                            int32_t B, int32_t *drafts, int32_t *num_valid, float *score,
                            float *probs, int32_t *match_info, void *stream);

/* One decoding step: sgd_propose_with_update, then sgd_ingest of n_docs docs
 * read from the rows after their update ([PYPI] Quickstart: the serving loop
 * calls propose_with_update and harvest_finished every step).  Results equal
 * those of the two calls made in that order on `stream` (num_tokens, after
 * the update, bounds the docs).  With 1 <= n_docs <= 64 everything runs in
 * ONE kernel launch: one extra CTA appends the docs while the row CTAs
 * draft, after waiting (bounded, ~0.1 s) for each doc's row to be updated; a
 * wait that runs out skips that doc and sets SGD_ERR_INGEST_WAIT.  Larger
 * n_docs run as the two calls.  Steps of one context must not overlap (one
 * stream at a time).  SGD_ENOCORPUS if n_docs > 0 without a corpus. */
int sgd_step(sgd_ctx *ctx, int32_t *token_ids, int32_t *num_tokens, const int32_t *sampled,
             int32_t T, const uint8_t *active, int32_t B, int32_t *drafts, int32_t *num_valid,
             float *score, float *probs, int32_t *match_info, const int32_t *rows,
             const int32_t *starts, const int32_t *lengths, int32_t n_docs, void *stream);

/* sgd_step with the step's inputs and outputs in HOST memory: copies h_sampled
 * [B, T] (and, with n_docs > 0, h_rows / h_starts / h_lengths [n_docs]) into
 * library-owned device staging buffers, runs sgd_step on the DEVICE token_ids /
 * num_tokens (the rows stay resident), and copies drafts [B, k] and num_valid
 * [B] (and score [B], probs [B, k], match_info [B, 2] where the pointer is not
 * NULL) back to host memory, all queued on `stream` in that order.  Returns
 * once queued: the host outputs are valid after the stream is synchronised,
 * and the host inputs must not change before then.  When every given host
 * buffer is page-locked and mapped (cudaHostAlloc / pinned memory on a
 * unified-address system) no staging copy is made: the kernel reads the inputs
 * and writes the outputs in host memory in place.  Otherwise (e.g. pageable
 * memory) the copies go through the device staging buffers.  All rows are active.  Errors as sgd_step; T <= max_sampled, B <= max_batch,
 * n_docs <= max_ingest_docs. */
int sgd_step_host(sgd_ctx *ctx, int32_t *token_ids, int32_t *num_tokens, const int32_t *h_sampled,
                  int32_t T, int32_t B, const int32_t *h_rows, const int32_t *h_starts,
                  const int32_t *h_lengths, int32_t n_docs, int32_t *h_drafts,
                  int32_t *h_num_valid, float *h_score, float *h_probs, int32_t *h_match_info,
                  void *stream);

/* Appends finished responses to the corpus ring ([PYPI] Quickstart:
 * harvest_finished; How it works, step 4: oldest documents are evicted when
 * the ring is full; [DOCS] Model Runner V2: oldest first out).
 *   token_ids  DEVICE int32 [B, S];  num_tokens DEVICE int32 [B] or NULL.
 *   rows, starts, lengths  DEVICE int32 [n_docs]: doc i is
 *              token_ids[rows[i], starts[i] : starts[i] + lengths[i]].
 * Docs are appended in order, each followed by the sentinel V; before each,
 * the oldest docs are evicted while the ring would exceed corpus_capacity or
 * hold max_docs docs.  Bad (row, start, length) -> skipped, SGD_ERR_DOC_ARGS;
 * an id outside [0, V) truncates the doc there (SGD_ERR_DOC_TOKEN); a doc
 * longer than the ring is skipped (SGD_ERR_DOC_TOO_LONG).  New docs become
 * visible to drafting only after the next build is swapped in.
 * n_docs <= max_ingest_docs.  SGD_ENOCORPUS without a corpus. */
int sgd_ingest(sgd_ctx *ctx, const int32_t *token_ids, const int32_t *num_tokens,
               int32_t B, const int32_t *rows, const int32_t *starts,
               const int32_t *lengths, int32_t n_docs, void *stream);

/* Starts a background suffix-array build ([PYPI] How it works, step 4 and
 * Highlights: rebuilt on a side CUDA stream, double-buffered, swapped in
 * place).  The live ring is copied (oldest doc first) into the spare
 * snapshot buffer on `stream` -- so it reflects every ingest enqueued there
 * before -- and the suffix array is then built by prefix doubling on
 * `side_stream`, driven by a library-owned host thread.  Returns at once.
 * `stream` must also be ordered after every propose that may still read the
 * spare buffer (a propose enqueued before the previous swap).
 * SGD_EBUSY while an earlier build is running or not yet swapped in. */
int sgd_build_sa(sgd_ctx *ctx, void *stream, void *side_stream);

/* Swaps in a finished build ([PYPI] Quickstart: poll).  If the build is done
 * and succeeded, a 32-byte descriptor write is enqueued on `stream`, so every
 * later propose on `stream` (including replays of graphs captured earlier)
 * reads the new snapshot; returns SGD_OK_SWAPPED.  SGD_PENDING while running
 * (wait = 0); with wait = 1 blocks up to timeout_us (< 0: forever), then
 * SGD_ETIMEDOUT.  SGD_OK if no build was started.  SGD_EBUILD if the build
 * failed (the previous snapshot stays current).  *generation (may be NULL)
 * receives the number of swaps so far. */
int sgd_poll(sgd_ctx *ctx, int wait, int64_t timeout_us, void *stream, uint64_t *generation);

/* Suffix array of a caller text, with the context's scratch, blocking the
 * host until done ([PYPI] References: Manber & Myers prefix doubling).
 *   text DEVICE int32 [n], any int32 values; sa DEVICE int32 [n] output.
 * Order: token by token as signed int32, a proper prefix first.
 * n <= corpus_capacity.  SGD_EBUSY while a background build runs;
 * SGD_EBUILD if the sort reported a failure. */
int sgd_suffix_array(sgd_ctx *ctx, const int32_t *text, int64_t n, int32_t *sa, void *stream);

/* Suffix array of a caller text without allocating anything: no device,
 * pinned-host or library allocation happens in the call.  This is for
 * callers that cannot call cudaMalloc where they need the array -- a server
 * whose own caching allocator owns the device memory, code running under
 * another framework's memory budget, or code that must not risk an
 * out-of-memory error or the device-wide synchronisation of cudaMalloc /
 * cudaFree mid-work.  (The pages describe no such entry point; it has no
 * counterpart there.)
 *   text DEVICE int32 [n] (any values), sa DEVICE int32 [n] output, both
 *   caller-owned; same order as sgd_suffix_array; no context is needed.
 * The working memory is one fixed device array of the library, sized for
 * SGD_NOALLOC_MAX_TOKENS tokens (about 2.5 MB, held on every GPU that loads the
 * library until the process exits); longer texts return SGD_ETOOLARGE.  The
 * first call on a device (with that device current) looks the array up on
 * that device; make that first call before any stream capture.  `stream`
 * must belong to the current device (SGD_EINVAL otherwise).  All calls in a
 * process share the array and find the previous call's contents in it: two
 * calls whose GPU work overlapped would race on it.  The call prevents that
 * itself: callers on different host threads are serialised, and each call
 * waits for its own GPU work (blocking the host) before it returns.
 * SGD_EBUILD if the sort reported a failure. */
#define SGD_NOALLOC_MAX_TOKENS 65536
int sgd_suffix_array_noalloc(const int32_t *text, int64_t n, int32_t *sa, void *stream);

/* Reads (and with clear = 1 resets) the sticky device error word; this
 * synchronises the device and is not meant for the drafting path. */
int sgd_get_error(sgd_ctx *ctx, uint32_t *flags, int clear);

/* Copies the current snapshot (text and suffix array) into caller DEVICE
 * buffers of `capacity` elements and returns its length and generation.
 * Synchronises the device.  SGD_EINVAL if capacity is too small. */
int sgd_export_snapshot(sgd_ctx *ctx, int32_t *text, int32_t *sa, int64_t capacity,
                        int64_t *n, uint64_t *generation);

/* Live ring tokens (incl. sentinels) and documents.  Synchronises the device. */
int sgd_corpus_stats(sgd_ctx *ctx, int64_t *live_tokens, int32_t *ndocs);

/* The cross-request corpus to a file and back ([PYPI] Roadmap: global tree
 * save & load), so that it survives a restart: the ring (live docs, their
 * FIFO, docs ever placed), the current snapshot's text and where its delta
 * starts.  Derived structures (suffix array, keys, records, n-gram table,
 * delta signatures) are rebuilt by sgd_load, so a file is
 * 4 C + 12 max_docs + 4 n bytes plus an 88-byte header, in the host's byte
 * order.  After sgd_load the context drafts exactly as the saved one did and
 * its generation has advanced by one.
 *   sgd_save: waits for `stream` (the drafting stream), then writes `path`.
 *   sgd_load: needs a context of the same vocab_size, corpus_capacity and
 *   max_docs; reads and checks the whole file (layout, sizes, ids in [0, V],
 *   the documents back to back ending at the write offset) before changing
 *   anything, then rebuilds the snapshot's index on `stream` and waits for it.
 * Both: SGD_EBUSY while a build is in flight or not yet swapped in,
 * SGD_ENOCORPUS without a corpus, SGD_EIO if the file cannot be written or
 * read (short file), SGD_EINVAL for a file that is not such a save or does
 * not fit the context (nothing is changed then). */
int sgd_save(sgd_ctx *ctx, const char *path, void *stream);
int sgd_load(sgd_ctx *ctx, const char *path, void *stream);

/* Figures of the last finished suffix-array build. */
typedef struct {
  int64_t n;              /* tokens sorted                                        */
  int32_t rounds;         /* prefix-doubling rounds, the initial sort included     */
  int32_t passes;         /* radix passes run                                      */
  int64_t sorted_elems;   /* sum over rounds of the suffixes still unresolved      */
  int64_t pass_elems;     /* sum over passes of the elements moved                 */
  int64_t model_bytes;    /* algorithmic bytes of the build (see the design notes) */
  double  ms;             /* device time of the whole build (events, side stream)  */
  double  pass_ms;        /* device time inside the radix-pass kernels             */
  int32_t status;         /* SGD_OK or SGD_EBUILD                                  */
} sgd_build_info;
int sgd_build_stats(sgd_ctx *ctx, sgd_build_info *info);

/* Host-side fault injection for tests (no GPU fault is ever provoked):
 *   SGD_INJECT_NONE        clear;
 *   SGD_INJECT_BUILD_FAIL  the next build reports failure;
 *   SGD_INJECT_BUILD_HANG  the next build never reports completion (its
 *                          kernels still run; sgd_poll stays pending);
 *   SGD_INJECT_STEP_WAIT   the ingest CTA of the next fused sgd_step waits for
 *                          a row signal that no CTA sends: its bounded wait
 *                          (~0.1 s) runs out, the docs are skipped and
 *                          SGD_ERR_INGEST_WAIT is set; drafting is unaffected. */
#define SGD_INJECT_NONE       0
#define SGD_INJECT_BUILD_FAIL 1
#define SGD_INJECT_BUILD_HANG 2
#define SGD_INJECT_STEP_WAIT  3
int sgd_debug_inject(sgd_ctx *ctx, int what);

/* Kernel launches the context made since creation (every library kernel). */
int sgd_launch_count(sgd_ctx *ctx, uint64_t *count);

/* Per-row statistics of the drafting launches made after this call, for
 * measuring the bytes a step touched (SuffixGPU (PyPI), How it works, steps
 * 2-3: the suffix-array hits scanned and the continuations gathered).
 *   row_stats: caller-owned DEVICE int32 [max_batch, 4], 16-byte aligned, or
 *   null to stop.  Each launch of the default drafting kernel (num_backoff =
 *   1) writes, for every row b < B: [4b] the suffix-array hits the corpus
 *   probe scanned (every level evaluated), [4b+1] the occurrences that voted
 *   (c0), [4b+2] the draft cap, [4b+3] the source (0 none, 1 row, 2 corpus)
 *   plus 256 times how the row's own match was found: 0 by a scan of the
 *   row, 1 from its bigram index (row_index), 2 not needed (row_index: the
 *   row's last bigram occurs nowhere earlier and the corpus matched >= 2),
 *   plus 4096 when the corpus draft came from a gram draft (gram_drafts).
 * The pointer is read when a call is made, so a CUDA graph captured after
 * this call keeps writing to it.  SGD_EINVAL for an unaligned buffer. */
int sgd_set_row_stats(sgd_ctx *ctx, int32_t *row_stats);

/* Starts the bigram position indexes of rows[0, m) over from the rows'
 * current contents (row_index = 1; no-op otherwise).  Call it after writing a
 * row other than through sgd_update_state / sgd_propose_with_update /
 * sgd_step: a new request placed in a row, and every row before its first
 * step.  Until then such a row is scanned, and a row rewritten with the same
 * length as before would be matched against stale positions.
 *   token_ids DEVICE int32 [>= max row + 1, S], num_tokens DEVICE int32 (the
 *   rows' lengths), rows DEVICE int32 [m], row indices (a row listed twice is
 *   reset once; indices outside [0, max_batch) are skipped); async on stream.
 * Cost: one pass over each listed row (an atomic insert per position).
 * SGD_EINVAL for m < 0 or m > 2^20. */
int sgd_reset_rows(sgd_ctx *ctx, const int32_t *token_ids, const int32_t *num_tokens,
                   const int32_t *rows, int32_t m, void *stream);

/* Memory the context allocated at sgd_create (it allocates nothing later):
 * device bytes (ring, both snapshots with their indexes, sort scratch,
 * staging) and page-locked host bytes.  Either pointer may be null. */
int sgd_memory(sgd_ctx *ctx, int64_t *device_bytes, int64_t *pinned_bytes);

const char *sgd_strerror(int status);
int sgd_version(void); /* major * 10000 + minor * 100 + patch */

#ifdef __cplusplus
}
#endif
#endif /* SGD_H */
