// sgd_internal.h -- shared declarations of the libsgd CUDA sources.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sgd.h"

namespace sgd {

constexpr unsigned FULL = 0xffffffffu;
constexpr int WIN = 128;        // tokens per warp window: 32 lanes x int4
constexpr int MAX_D = 128;      // the halo of one window covers D - 1 <= 127
constexpr int MAX_R = 128;      // up to 4 occurrences per lane in the vote warp
constexpr int MAX_K = 64;
constexpr int MAX_SELF_WARPS = 16;
constexpr int MAX_BACKOFF = 8;      // candidate lengths per path
constexpr int MAX_PROPOSE_THREADS = 640;

// Descriptor of the suffix-array snapshot drafting reads.  It lives in device
// memory at a fixed address, so graphs captured before a swap see the new
// snapshot after it.
struct CorpusDesc {
  const int32_t *text;  // X[0..n): live docs oldest first, each followed by Z
  const int32_t *sa;    // suffix array of X
  const int4 *keys;     // keys[p] = X[sa[p] .. sa[p]+3], KEY_END past the text
  int64_t n;
  uint64_t gen;
  const int32_t *rec;   // per-position records (RecShape), or null
  const int32_t *gt;    // n-gram table (below), or null
  uint64_t gt_mask;     // buckets - 1
  int64_t lin_pushed;   // the ring's docs placed when X was linearised
  int64_t lin_wp;       // the ring's write offset then (where the next doc went)
  const int32_t *gd;    // gram drafts (blocks of 4 + 2 roundup4(k) ints), or null
};

// n-gram table: for every distinct m-gram (m = 2, 3, 4) that begins a suffix
// of the snapshot, its suffix-array interval [lo, hi).  Open addressing over
// buckets of GT_BUCKET entries of GT_ENTRY ints: [0] m (0: empty), [1..4] the
// tokens (KEY_END past m), [5] lo, [6] hi, [7] for m = 2, 3 with gram drafts:
// the gram's draft block, or -2.  A bucket is 128 bytes.
constexpr int GT_BUCKET = 4;
constexpr int GT_ENTRY = 8;
__host__ __device__ inline uint64_t gram_hash(int m, int t0, int t1, int t2, int t3) {
  uint64_t h = 0x9E3779B97F4A7C15ull * (uint64_t)(m + 1);
  const uint32_t t[4] = {(uint32_t)t0, (uint32_t)t1, (uint32_t)t2, (uint32_t)t3};
  for (int i = 0; i < 4; ++i) {
    h ^= t[i];
    h *= 0xff51afd7ed558ccdull;
    h ^= h >> 32;
  }
  return h;
}

// Record of suffix-array position p (i = sa[p]), ri ints, every region on a
// 16-byte boundary: [0] i, [1..3] X[i+4], X[i+5], X[i+6] (Z past the end);
// [4, 4+bk) the bk tokens before the suffix, X[i-1-j] (KEY_END before the
// text); [co, co+kc) the kc tokens after its first four, X[i+4+j] (Z past
// the end); zero padding.
struct RecShape {
  int ri, bk, kc, co;
};
inline RecShape rec_shape(int D, int k) {
  RecShape r;
  r.bk = D > 4 ? D - 4 : 0;
  r.kc = k;
  r.co = 4 + ((r.bk + 3) & ~3);
  r.ri = r.co + ((r.kc + 3) & ~3);
  return r;
}
constexpr int KEY_END = (int)0x80000000;  // below every id: the text ran out

// Ring bookkeeping, device resident.  The doc FIFO lives in two arrays of
// max_docs entries indexed (head + i) % max_docs.
struct RingState {
  int64_t wp;      // next write offset in [0, C)
  int64_t live;    // tokens of live docs, sentinels included
  int32_t head;    // FIFO index of the oldest doc
  int32_t ndocs;
  int64_t snap_n;  // length of the last linearised snapshot
  int64_t pushed;  // docs ever placed; the doc at FIFO index i is number pushed - ndocs + i
  int64_t snap_pushed, snap_wp;  // pushed and wp when the last snapshot was linearised
};

// The docs placed after a snapshot was linearised (not in its index yet: the
// delta), as one circular run of the ring, [start, start + len) mod C, len
// tokens with the sentinels.  Docs are placed at the write offset in order,
// so while older docs are still live the first delta doc starts where the
// write offset was at linearisation; once every live doc is a delta doc, the
// run is the whole live ring.
struct DeltaView {
  long long start, len;
};

__host__ __device__ inline DeltaView delta_view(const RingState &r, long long since, long long lin_wp,
                                                long long C, const int64_t *doc_start) {
  const long long first = since - (r.pushed - r.ndocs);  // FIFO index of the oldest delta doc
  DeltaView v{0, 0};
  if (first >= r.ndocs) return v;
  if (first <= 0) {
    v.start = doc_start[r.head];
    v.len = r.live;
  } else {
    v.start = lin_wp;
    v.len = r.wp - lin_wp;
    if (v.len < 0) v.len += C;
  }
  return v;
}

// Per-row bigram position index (row_index.cuh), or tab == null.
struct RowIndexArgs {
  int32_t *tab;    // [max_batch][H][16] entries
  int32_t *meta;   // [max_batch][2]: row length the entries cover (-1: invalid), generation
  long long H;     // entries per row
};

struct ProposeArgs {
  int32_t *tok;            // [B, S]
  int32_t *ntok;           // [B]
  const int32_t *sampled;  // [B, T] or null
  int T;
  int do_update;
  const uint8_t *active;   // [B] or null
  int B, S, V, k, D, R;
  long long fN, fD, offset, pN, pD;
  int depth_sum_cap;
  const CorpusDesc *desc;  // null when the context has no corpus
  int32_t *drafts;         // [B, k]
  int32_t *num_valid;      // [B]
  float *score;            // [B] or null
  float *probs;            // [B, k] or null
  int32_t *match_info;     // [B, 2] or null
  uint32_t *err;
  int nself;               // self-scan warps per row
  int cand_cap;            // corpus candidate buffer (power of two >= R)
  RecShape rsh;            // layout of the snapshot's records (desc->rec)
  // fused step: ing_m > 0 adds CTA 0, which appends ing_m docs to the ring
  // once their rows are updated (the row CTAs are 1..B)
  int ing_m;
  const int32_t *ing_rows, *ing_starts, *ing_lengths;
  int32_t *ring;
  long long C;
  RingState *rs;
  int64_t *doc_start;
  int32_t *doc_len;
  int max_docs;
  uint32_t *step_ready;  // [max_batch] per row: the step epoch once updated
  // [0] step epoch, [1] CTAs arrived in this launch, [2] row CTAs finished,
  // [3] the epoch whose row CTAs have all finished
  uint32_t *step_sync;
  uint32_t ing_skew;     // added to the awaited epoch (0; 1 only under test injection)
  // split launch (long rows): the self kernel writes per row, at self_res + b *
  // self_res_ints(R): Ms, cs, the last four tokens, the cs most recent ends;
  // then Md, cd, the delta's start and visible length, the cd most recent
  // delta ends.  The corpus kernel reads them back instead of scanning.
  int32_t *self_res;
  int split;             // 0: one fused kernel; 1: self kernel + corpus kernel
  // Delta (docs placed after the snapshot was linearised): searched up to
  // dcap tokens, oldest first; 0: not searched.  Needs ring, C (a multiple of
  // WIN), rs, doc_start and sig, the ring's window signatures.
  long long dcap;
  uint32_t *sig;
  // Model Runner V2 drafts: k tokens always, the vote not stopped by
  // min_token_prob (pN = 0) nor capped by the factor, empty slots hold the
  // row's last token
  int fixed;
  // score-ranked selection: the row's and the corpus's candidates are both
  // voted and the better score wins (ties: the longer match, then the row)
  int by_score;
  // multi-length backoff: candidate lengths per path (> 1: backoff.cu)
  int nb;
  // [B, 4] or null: per row, the suffix-array hits the corpus probe scanned,
  // the occurrences that voted (c0), the draft cap and the source (0/1/2)
  int32_t *row_stats;
  // the rows' bigram position indexes: the self match from them when complete
  // (one fused kernel per step, no delta, no score-ranked selection)
  RowIndexArgs ri;
  // 1: the snapshots have no n-gram tables, so the probe descends the key
  // array and its top two levels are staged in shared memory
  int stage_keys;
};

__host__ __device__ constexpr int self_res_ints(int R) { return 2 * R + 10; }

// propose.cu
// mode as the kernel's; stage_keys: the top key-array levels are staged (no n-gram tables)
size_t propose_smem_bytes(int mode, int nself, int R, int k, int cand_cap, int stage_keys);
int propose_step_max_docs();  // largest doc count a fused step ingests in-kernel
cudaError_t launch_propose(const ProposeArgs &a, cudaStream_t st);
cudaError_t launch_update(int32_t *tok, int32_t *ntok, const int32_t *sampled, int B,
                          int T, int S, int V, uint32_t *err, const RowIndexArgs &ri,
                          cudaStream_t st);
// Starts the indexes of rows[0, m) over from their current contents (distinct
// rows; a row listed twice is reset once).  claim: [max_batch] u64 words,
// epoch: a number the context never passed before.
cudaError_t launch_row_index_reset(const RowIndexArgs &ri, const int32_t *tok, const int32_t *ntok,
                                   int S, const int32_t *rows, int m, int max_batch,
                                   unsigned long long *claim, unsigned long long epoch,
                                   cudaStream_t st);
cudaError_t propose_set_smem_limit(size_t bytes);

// backoff.cu: multi-length backoff drafting of rows [0, B), one CTA per row
// (no update: the caller launches it first)
cudaError_t launch_backoff(const ProposeArgs &a, cudaStream_t st);
cudaError_t backoff_set_smem_limit();  // the backoff kernel's dynamic shared memory (its row-length cache)

// corpus.cu
struct IngestScratch {
  int32_t *eff;     // [max_ingest_docs] effective doc length (-1: skip)
  int64_t *dest;    // [max_ingest_docs] ring offset or -1
  int32_t *order;   // [max_ingest_docs] docs pushed by this call, push order
  int64_t *span;    // [2] the call's first ring position and the tokens its placements took
};
cudaError_t launch_ingest(const int32_t *tok, const int32_t *ntok, int B, int S, int V,
                          const int32_t *rows, const int32_t *starts, const int32_t *lengths,
                          int m, int32_t *ring, int64_t C, RingState *rs, int64_t *doc_start,
                          int32_t *doc_len, int max_docs, const IngestScratch &sc,
                          uint32_t *sig, uint32_t *err, cudaStream_t st, int *launches);
cudaError_t launch_sig_all(int32_t *ring, int64_t C, int V, uint32_t *sig, cudaStream_t st);
cudaError_t launch_linearize(const int32_t *ring, int64_t C, RingState *rs,
                             const int64_t *doc_start, int max_docs, int32_t *out,
                             cudaStream_t st, int *launches);
cudaError_t launch_records(const int32_t *text, const int32_t *sa, int64_t n, RecShape shape, int Z,
                           int32_t *rec, cudaStream_t st);
cudaError_t launch_gram_table(const int4 *keys, int64_t n, int32_t *gt, uint64_t mask,
                              cudaStream_t st);
cudaError_t launch_swap(CorpusDesc *desc, const int32_t *text, const int32_t *sa, const int4 *keys,
                        const int32_t *rec, const int32_t *gt, uint64_t gt_mask, const int32_t *gd,
                        int64_t n, uint64_t gen, const RingState *rs, cudaStream_t st);
// gram drafts of a snapshot (propose.cu): blocks for its 2-/3-grams' votes
// (cap blocks of 4 + 2 roundup4(k) ints), their indexes in the n-gram table.
// Waits once for the stream (the number of blocks, read into pinned h_count).
cudaError_t launch_gram_drafts(int32_t *gt, uint64_t gt_mask, const int4 *keys, const int32_t *sa,
                               const int32_t *text, int64_t n, int Z, int k, int R, long long pN,
                               long long pD, int32_t *gd, int cap, int32_t *count, int32_t *owner,
                               int32_t *h_count, cudaStream_t st);
__host__ __device__ inline int gd_ints(int k) { return 4 + 2 * ((k + 3) & ~3); }
// keys[p] = text[sa[p] .. sa[p]+3] (KEY_END past n), on `st`
cudaError_t launch_suffix_keys(const int32_t *text, const int32_t *sa, int64_t n, int4 *keys,
                               cudaStream_t st);

// sa_build.cu
struct SaScratch {
  int64_t cap;                  // elements the scratch can sort
  uint64_t *keyA, *keyB;
  int32_t *valA, *valB;
  int32_t *rank;                // head-position ranks
  int32_t *act, *act2;          // SA positions of unresolved suffixes
  unsigned long long *status;   // radix look-back words, [tiles][256]
  unsigned long long *pstatus;  // post-pass look-back words, [tiles]
  uint32_t *hist;               // [8][256] digit histograms
  uint32_t *counter;            // active count, tickets
  int32_t *h_pinned;            // host words for counts read back by the driver
  uint32_t *h_hist;             // host [8][256]
  int64_t status_words;
  unsigned char *owned;         // device block owned by this scratch (alloc), else null
};
struct SaStats {
  int rounds = 0, passes = 0;
  long long sorted_elems = 0, pass_elems = 0, model_bytes = 0;
  double pass_ms = 0;
};
size_t sa_scratch_bytes(int64_t cap);
cudaError_t sa_scratch_alloc(SaScratch *s, int64_t cap);
void sa_scratch_free(SaScratch *s);
// Lays the device buffers of a scratch for `cap` elements out in
// [base, base + bytes) (256-byte aligned pieces, no allocation); returns the
// bytes needed, and leaves *s empty if they exceed `bytes`.  Host words
// (h_pinned, h_hist) are left to the caller.
size_t sa_scratch_carve(SaScratch *s, unsigned char *base, size_t bytes, int64_t cap);
// Builds the suffix array of text[0..n) into sa; host-driven rounds on `st`
// (blocks the calling thread).  Returns 0 on success, else SGD_ERR_* bits
// (through *dev_flags as well) or -1 on a CUDA error.
int sa_build(const SaScratch &s, const int32_t *text, int64_t n, int32_t *sa,
             uint32_t *err, cudaStream_t st, SaStats *stats, bool time_passes,
             int *launches);

}  // namespace sgd
