// api.cu -- host side of libsgd: the context, argument checks, launches on
// the caller's streams and the background suffix-array build.
//
// The build of a new suffix array is driven by one host thread per context
// (its prefix-doubling rounds read small counts back to size the next round),
// while drafting keeps running on the caller's stream; sgd_poll swaps the
// finished snapshot in with a 32-byte device write ("SuffixGPU", PyPI: How it
// works, step 4 -- rebuilt on a side stream, double-buffered, swapped in
// place so captured CUDA graphs keep working).
#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "delta_sig.cuh"
#include "row_index.cuh"
#include "sgd_internal.h"

using namespace sgd;

namespace {

enum BuildState { B_IDLE = 0, B_RUNNING = 1, B_DONE = 2, B_HUNG = 3 };

}  // namespace

struct sgd_ctx {
  sgd_config cfg;
  int device = 0;
  int nself = 1;
  size_t smem = 0;
  bool corpus = false;
  // device state
  uint32_t *d_err = nullptr;        // sticky error bits of drafting and ingest
  uint32_t *d_build_err = nullptr;  // error bits of the build in progress
  uint32_t *d_step_ready = nullptr; // [max_batch] fused step: per-row update epoch
  uint32_t *d_step_sync = nullptr;  // fused step: epoch, arrivals
  int32_t *d_hin = nullptr;         // sgd_step_host inputs: sampled, rows, starts, lengths
  int32_t *d_hout = nullptr;        // sgd_step_host outputs: drafts, num_valid, score, probs, match_info
  int32_t *d_self_res = nullptr;    // two-launch propose: per-row self results
  int32_t *d_row_stats = nullptr;   // caller's [max_batch, 4] statistics buffer, or null
  int64_t dev_bytes = 0;            // device memory the context allocated
  int64_t pinned_bytes = 0;         // page-locked host memory the context allocated
  RowIndexArgs ri{};                // per-row bigram position indexes (row_index = 1)
  unsigned long long *d_ri_claim = nullptr;  // sgd_reset_rows: the listing that resets a row
  unsigned long long ri_epoch = 0;
  // sgd_step_host: the last set of host buffers checked for in-place access
  const void *zc_key[9] = {};
  void *zc_dev[9] = {};
  bool zc_ok = false;
  int split = 0;
  int stage_keys = 0;               // the probe descends the key array (no n-gram tables)
  int32_t *d_ring = nullptr;
  RingState *d_rs = nullptr;
  int64_t *d_doc_start = nullptr;
  int32_t *d_doc_len = nullptr;
  int32_t *d_text[2] = {nullptr, nullptr};
  int32_t *d_sa[2] = {nullptr, nullptr};
  int4 *d_keys[2] = {nullptr, nullptr};
  int32_t *d_rec[2] = {nullptr, nullptr};  // per-position records, or null (off / over budget)
  RecShape rsh{};
  int32_t *d_gt[2] = {nullptr, nullptr};   // n-gram tables, or null (off / over budget)
  int32_t *d_gd[2] = {nullptr, nullptr};   // gram drafts, or null (off / over budget)
  int32_t *d_gd_count = nullptr, *d_gd_owner = nullptr;  // their build's counter, block owners
  int gd_cap = 0;                          // blocks per snapshot
  int32_t *h_gd_count = nullptr;           // pinned: the blocks a build assigned
  uint64_t gt_mask = 0;
  CorpusDesc *d_desc = nullptr;
  IngestScratch ing{};
  uint32_t *d_sig = nullptr;        // ring window signatures (with a delta)
  SaScratch sa{};
  int64_t *h_n = nullptr;      // pinned
  uint32_t *h_err = nullptr;   // pinned
  cudaEvent_t ev_lin = nullptr, ev_b0 = nullptr, ev_b1 = nullptr;
  // snapshots
  int front = 0;
  int64_t front_n = 0;
  uint64_t gen = 0;
  // build worker
  std::thread worker;
  std::mutex mu;
  std::condition_variable cv;
  bool quit = false;
  bool job_ready = false;
  int job_back = 1;
  cudaStream_t job_side = nullptr;
  int bstate = B_IDLE;
  int bstatus = SGD_OK;
  int64_t built_n = 0;
  int inject = SGD_INJECT_NONE;
  int job_inject = SGD_INJECT_NONE;
  sgd_build_info last{};
  std::atomic<uint64_t> launches{0};
};

namespace {

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int check_cuda(cudaError_t e) { return e == cudaSuccess ? SGD_OK : SGD_ECUDA; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

int validate(const sgd_config &c) {
  if (c.max_batch < 1 || c.seq_capacity < 4 || c.seq_capacity % 4 != 0) return SGD_EINVAL;
  if (c.vocab_size < 1 || c.vocab_size == 0x7fffffff) return SGD_EINVAL;
  if (c.k < 1 || c.k > MAX_K) return SGD_EINVAL;
  if (c.max_tree_depth < 1 || c.max_tree_depth > MAX_D) return SGD_EINVAL;
  if (c.max_occurrences < 1 || c.max_occurrences > MAX_R) return SGD_EINVAL;
  if (c.max_sampled < 1 || c.max_sampled > 1024) return SGD_EINVAL;
  if (c.spec_factor_den == 0 || c.min_prob_den == 0 || c.min_prob_num > c.min_prob_den)
    return SGD_EINVAL;
  if (c.spec_offset < 0) return SGD_EINVAL;
  if (c.corpus_capacity < 0 || c.corpus_capacity > (1LL << 30)) return SGD_EINVAL;
  if (c.corpus_capacity > 0 && (c.max_docs < 1 || c.max_ingest_docs < 1)) return SGD_EINVAL;
  if (!is_pow2(c.corpus_cand_cap) || c.corpus_cand_cap < c.max_occurrences ||
      c.corpus_cand_cap > 16384)
    return SGD_EINVAL;
  if (c.self_warps < 0 || c.self_warps > MAX_SELF_WARPS) return SGD_EINVAL;
  if (c.corpus_records != 0 && c.corpus_records != 1) return SGD_EINVAL;
  if (c.corpus_gram_index != 0 && c.corpus_gram_index != 1) return SGD_EINVAL;
  if (c.propose_mode < 0 || c.propose_mode > 2) return SGD_EINVAL;
  if (c.delta_capacity < 0 || c.delta_capacity > c.corpus_capacity) return SGD_EINVAL;
  if (c.delta_capacity > 0 && c.corpus_capacity % WIN != 0) return SGD_EINVAL;
  if (c.draft_mode != 0 && c.draft_mode != 1) return SGD_EINVAL;
  if (c.select_by_score != 0 && c.select_by_score != 1) return SGD_EINVAL;
  if (c.num_backoff < 1 || c.num_backoff > MAX_BACKOFF) return SGD_EINVAL;
  if (c.row_index != 0 && c.row_index != 1) return SGD_EINVAL;
  if (c.gram_drafts != 0 && c.gram_drafts != 1) return SGD_EINVAL;
  if (c.row_index && (c.propose_mode == 2 || c.delta_capacity > 0 || c.select_by_score ||
                      c.num_backoff > 1 || c.vocab_size > RI_MAX_TOKEN + 1))
    return SGD_EINVAL;
  return SGD_OK;
}

int choose_self_warps(const sgd_config &c) {
  if (c.self_warps > 0) return c.self_warps;
  int w = c.seq_capacity / 512;
  if (w < 1) w = 1;
  const int cap = c.max_batch <= 76 ? 16 : 8;
  if (w > cap) w = cap;
  return w;
}

void free_ctx(sgd_ctx *x) {
  cudaFree(x->d_err);
  cudaFree(x->ri.tab);
  for (int i = 0; i < 2; ++i) cudaFree(x->d_gd[i]);
  cudaFree(x->d_gd_count);
  cudaFree(x->d_gd_owner);
  cudaFree(x->ri.meta);
  cudaFree(x->d_ri_claim);
  cudaFree(x->d_step_ready);
  cudaFree(x->d_hin);
  cudaFree(x->d_self_res);
  cudaFree(x->d_hout);
  cudaFree(x->d_rec[0]);
  cudaFree(x->d_rec[1]);
  cudaFree(x->d_gt[0]);
  cudaFree(x->d_gt[1]);
  cudaFree(x->d_step_sync);
  cudaFree(x->d_build_err);
  cudaFree(x->d_ring);
  cudaFree(x->d_rs);
  cudaFree(x->d_doc_start);
  cudaFree(x->d_doc_len);
  for (int i = 0; i < 2; ++i) {
    cudaFree(x->d_text[i]);
    cudaFree(x->d_sa[i]);
    cudaFree(x->d_keys[i]);
  }
  cudaFree(x->d_desc);
  cudaFree(x->ing.eff);
  cudaFree(x->ing.dest);
  cudaFree(x->ing.order);
  cudaFree(x->ing.span);
  cudaFree(x->d_sig);
  if (x->sa.keyA) sa_scratch_free(&x->sa);
  if (x->h_n) cudaFreeHost(x->h_n);
  if (x->h_err) cudaFreeHost(x->h_err);
  if (x->h_gd_count) cudaFreeHost(x->h_gd_count);
  if (x->ev_lin) cudaEventDestroy(x->ev_lin);
  if (x->ev_b0) cudaEventDestroy(x->ev_b0);
  if (x->ev_b1) cudaEventDestroy(x->ev_b1);
}

// One background build: wait for the snapshot copy, sort, report.
void worker_main(sgd_ctx *x) {
  cudaSetDevice(x->device);
  std::unique_lock<std::mutex> lk(x->mu);
  for (;;) {
    x->cv.wait(lk, [&] { return x->quit || x->job_ready; });
    if (x->quit) return;
    x->job_ready = false;
    const int back = x->job_back;
    cudaStream_t side = x->job_side;
    const int inj = x->job_inject;
    lk.unlock();

    int status = SGD_OK;
    int64_t n = 0;
    SaStats st;
    int launches = 0;
    float ms = 0.f;
    cudaError_t e = cudaStreamWaitEvent(side, x->ev_lin, 0);
    if (e == cudaSuccess) e = cudaMemsetAsync(x->d_build_err, 0, 4, side);
    if (e == cudaSuccess) e = cudaEventRecord(x->ev_b0, side);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(x->h_n, &x->d_rs->snap_n, 8, cudaMemcpyDeviceToHost, side);
    if (e == cudaSuccess) e = cudaStreamSynchronize(side);
    if (e == cudaSuccess) {
      n = *x->h_n;
      const int r = sa_build(x->sa, x->d_text[back], n, x->d_sa[back], x->d_build_err, side, &st,
                             true, &launches);
      if (r != 0) status = SGD_EBUILD;
      if (r == 0 && launch_suffix_keys(x->d_text[back], x->d_sa[back], n, x->d_keys[back], side) !=
                        cudaSuccess)
        status = SGD_EBUILD;
      ++launches;
      if (r == 0 && x->d_gt[back] != nullptr) {
        if (launch_gram_table(x->d_keys[back], n, x->d_gt[back], x->gt_mask, side) != cudaSuccess)
          status = SGD_EBUILD;
        launches += 2;
        if (x->d_gd[back] != nullptr) {
          // (the drafting vote's stop rule: no probability floor for fixed-length drafts)
          const long long pN = x->cfg.draft_mode == 1 ? 0 : x->cfg.min_prob_num;
          const long long pD = x->cfg.draft_mode == 1 ? 1 : x->cfg.min_prob_den;
          if (launch_gram_drafts(x->d_gt[back], x->gt_mask, x->d_keys[back], x->d_sa[back],
                                 x->d_text[back], n, x->cfg.vocab_size, x->cfg.k,
                                 x->cfg.max_occurrences, pN, pD, x->d_gd[back], x->gd_cap,
                                 x->d_gd_count, x->d_gd_owner, x->h_gd_count, side) != cudaSuccess)
            status = SGD_EBUILD;
          launches += 2;
        }
      }
      if (r == 0 && x->d_rec[back] != nullptr) {
        if (launch_records(x->d_text[back], x->d_sa[back], n, x->rsh, x->cfg.vocab_size,
                           x->d_rec[back], side) != cudaSuccess)
          status = SGD_EBUILD;
        ++launches;
      }
      e = cudaEventRecord(x->ev_b1, side);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(x->h_err, x->d_build_err, 4, cudaMemcpyDeviceToHost, side);
      if (e == cudaSuccess) e = cudaStreamSynchronize(side);
      if (e == cudaSuccess) cudaEventElapsedTime(&ms, x->ev_b0, x->ev_b1);
      if (e == cudaSuccess && *x->h_err != 0) status = SGD_EBUILD;
    }
    if (e != cudaSuccess) status = SGD_EBUILD;
    if (inj == SGD_INJECT_BUILD_FAIL) status = SGD_EBUILD;
    x->launches += (uint64_t)launches + 1;

    lk.lock();
    x->built_n = n;
    x->bstatus = status;
    x->last.n = n;
    x->last.rounds = st.rounds;
    x->last.passes = st.passes;
    x->last.sorted_elems = st.sorted_elems;
    x->last.pass_elems = st.pass_elems;
    x->last.model_bytes = st.model_bytes;
    x->last.ms = ms;
    x->last.pass_ms = st.pass_ms;
    x->last.status = status;
    x->bstate = inj == SGD_INJECT_BUILD_HANG ? B_HUNG : B_DONE;
    x->cv.notify_all();
  }
}

}  // namespace

extern "C" {

int sgd_version(void) { return 100; }

const char *sgd_strerror(int s) {
  switch (s) {
    case SGD_OK: return "ok";
    case SGD_OK_SWAPPED: return "ok: new suffix array swapped in";
    case SGD_PENDING: return "build pending";
    case SGD_EINVAL: return "invalid argument";
    case SGD_ECUDA: return "CUDA error";
    case SGD_ENOMEM: return "out of memory";
    case SGD_ETIMEDOUT: return "timed out";
    case SGD_EBUSY: return "a suffix-array build is in flight";
    case SGD_EBUILD: return "suffix-array build failed";
    case SGD_ENOCORPUS: return "context has no corpus";
    case SGD_ETOOLARGE: return "text longer than the fixed no-allocation scratch";
    default: return "unknown status";
  }
}

int sgd_config_default(sgd_config *c) {
  if (!c) return SGD_EINVAL;
  std::memset(c, 0, sizeof(*c));
  c->max_batch = 256;
  c->seq_capacity = 4096;
  c->vocab_size = 151936;
  c->k = 16;
  c->max_tree_depth = 24;
  c->max_occurrences = 64;
  c->max_sampled = 64;
  c->spec_factor_num = 1;
  c->spec_factor_den = 1;
  c->spec_offset = 0;
  c->min_prob_num = 1;
  c->min_prob_den = 10;
  c->depth_sum_cap = 0;
  c->corpus_capacity = 1LL << 20;
  c->max_docs = 65536;
  c->max_ingest_docs = 4096;
  c->corpus_cand_cap = 2048;
  c->corpus_records = 1;
  c->corpus_gram_index = 1;
  c->propose_mode = 0;
  c->delta_capacity = 0;
  c->draft_mode = 0;
  c->select_by_score = 0;
  c->num_backoff = 1;
  c->self_warps = 0;
  c->row_index = 0;
  c->gram_drafts = 1;
  return SGD_OK;
}

static void to_rational(double x, uint32_t *num, uint32_t *den) {
  long long n = (long long)(x * 1e6 + 0.5);
  long long d = 1000000;
  long long a = n, b = d;
  while (b) {
    const long long t = a % b;
    a = b;
    b = t;
  }
  if (a == 0) a = 1;
  *num = (uint32_t)(n / a);
  *den = (uint32_t)(d / a);
}

int sgd_config_set_float(sgd_config *c, double factor, double min_prob) {
  if (!c || !(factor >= 0) || !(min_prob >= 0) || min_prob > 1 || factor > 4000) return SGD_EINVAL;
  to_rational(factor, &c->spec_factor_num, &c->spec_factor_den);
  to_rational(min_prob, &c->min_prob_num, &c->min_prob_den);
  return SGD_OK;
}

int sgd_create(const sgd_config *cfg, int device, sgd_ctx **out) {
  if (!cfg || !out) return SGD_EINVAL;
  *out = nullptr;
  int v = validate(*cfg);
  if (v != SGD_OK) return v;
  if (cudaSetDevice(device) != cudaSuccess) return SGD_ECUDA;
  sgd_ctx *x = new (std::nothrow) sgd_ctx;
  if (!x) return SGD_ENOMEM;
  x->cfg = *cfg;
  x->device = device;
  x->nself = choose_self_warps(*cfg);
  x->corpus = cfg->corpus_capacity > 0;
  x->split = cfg->propose_mode == 2;
  {
    // with n-gram tables the probe never descends the key array, so its top
    // levels are not staged in shared memory
    bool gt_on = false;
    if (x->corpus) {
      unsigned long long nb = 1;
      while (nb < (unsigned long long)cfg->corpus_capacity) nb <<= 1;
      gt_on = cfg->corpus_gram_index && 2ull * nb * GT_BUCKET * GT_ENTRY * 4ull <= SGD_RECORD_BUDGET;
    }
    x->stage_keys = x->corpus && !gt_on;
    const int R = cfg->max_occurrences, k = cfg->k, cc = cfg->corpus_cand_cap, sk = x->stage_keys;
    x->smem = x->split ? std::max(propose_smem_bytes(1, x->nself, R, k, cc, sk),
                                  propose_smem_bytes(2, 1, R, k, cc, sk))
                       : propose_smem_bytes(0, x->nself, R, k, cc, sk);
  }
  cudaError_t e = cudaSuccess;
  auto al = [&](void **p, size_t bytes) {
    if (e == cudaSuccess) e = cudaMalloc(p, bytes);
    if (e == cudaSuccess) x->dev_bytes += (int64_t)bytes;
  };
  al((void **)&x->d_err, 4);
  al((void **)&x->d_build_err, 4);
  if (x->split)
    al((void **)&x->d_self_res, (size_t)cfg->max_batch * self_res_ints(cfg->max_occurrences) * 4);
  {
    const size_t Bm = (size_t)cfg->max_batch, kk = (size_t)cfg->k;
    al((void **)&x->d_hin, 4 * (Bm * (size_t)cfg->max_sampled + 3 * (size_t)cfg->max_ingest_docs));
    al((void **)&x->d_hout, 4 * (Bm * kk + Bm + Bm + Bm * kk + 2 * Bm));
  }
  if (e == cudaSuccess) e = cudaMemset(x->d_err, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(x->d_build_err, 0, 4);
  if (cfg->row_index) {
    // every entry empty (generation 0); every row invalid until it is reset
    const size_t Bm = (size_t)cfg->max_batch;
    x->ri.H = ri_entries(cfg->seq_capacity);
    al((void **)&x->ri.tab, Bm * (size_t)x->ri.H * RI_ENTRY * 4);
    al((void **)&x->ri.meta, Bm * 2 * 4);
    al((void **)&x->d_ri_claim, Bm * 8);
    if (e == cudaSuccess) e = cudaMemset(x->ri.tab, 0, Bm * (size_t)x->ri.H * RI_ENTRY * 4);
    if (e == cudaSuccess) e = cudaMemset(x->d_ri_claim, 0, Bm * 8);
    if (e == cudaSuccess) {
      std::vector<int32_t> m0(2 * Bm);
      for (size_t i = 0; i < Bm; ++i) { m0[2 * i] = -1; m0[2 * i + 1] = 0; }
      e = cudaMemcpy(x->ri.meta, m0.data(), m0.size() * 4, cudaMemcpyHostToDevice);
    }
  }
  if (x->corpus) {
    const int64_t C = cfg->corpus_capacity;
    al((void **)&x->d_ring, (size_t)C * 4);
    al((void **)&x->d_rs, sizeof(RingState));
    al((void **)&x->d_doc_start, (size_t)cfg->max_docs * 8);
    al((void **)&x->d_doc_len, (size_t)cfg->max_docs * 4);
    for (int i = 0; i < 2; ++i) {
      al((void **)&x->d_text[i], (size_t)C * 4);
      al((void **)&x->d_sa[i], (size_t)C * 4);
      al((void **)&x->d_keys[i], (size_t)C * 16);
    }
    al((void **)&x->d_desc, sizeof(CorpusDesc));
    x->rsh = rec_shape(cfg->max_tree_depth, cfg->k);
    if (cfg->corpus_records &&
        2ull * (unsigned long long)C * (unsigned long long)x->rsh.ri * 4ull <= SGD_RECORD_BUDGET) {
      al((void **)&x->d_rec[0], (size_t)C * x->rsh.ri * 4);
      al((void **)&x->d_rec[1], (size_t)C * x->rsh.ri * 4);
    }
    {
      // buckets: next power of two >= C, so 3 C grams fill at most 3/4 of the entries
      unsigned long long nb = 1;
      while (nb < (unsigned long long)C) nb <<= 1;
      const unsigned long long bytes = nb * GT_BUCKET * GT_ENTRY * 4ull;
      if (cfg->corpus_gram_index && 2ull * bytes <= SGD_RECORD_BUDGET) {
        x->gt_mask = nb - 1;
        al((void **)&x->d_gt[0], (size_t)bytes);
        al((void **)&x->d_gt[1], (size_t)bytes);
        if (e == cudaSuccess) e = cudaMemset(x->d_gt[0], 0, (size_t)bytes);
        // gram drafts: a block for up to C / 4 grams per snapshot
        const long long cap = std::max(1024LL, (long long)(C / 4));
        const unsigned long long gbytes = (unsigned long long)cap * gd_ints(cfg->k) * 4ull;
        if (cfg->gram_drafts && 2ull * gbytes <= SGD_RECORD_BUDGET && cap < (1LL << 31)) {
          x->gd_cap = (int)cap;
          al((void **)&x->d_gd[0], (size_t)gbytes);
          al((void **)&x->d_gd[1], (size_t)gbytes);
          al((void **)&x->d_gd_count, 4);
          al((void **)&x->d_gd_owner, (size_t)cap * 4);
        }
      }
    }
    al((void **)&x->d_step_ready, (size_t)cfg->max_batch * 4);
    al((void **)&x->d_step_sync, 16);
    if (e == cudaSuccess) e = cudaMemset(x->d_step_ready, 0, (size_t)cfg->max_batch * 4);
    if (e == cudaSuccess) e = cudaMemset(x->d_step_sync, 0, 16);
    al((void **)&x->ing.eff, (size_t)cfg->max_ingest_docs * 4);
    al((void **)&x->ing.dest, (size_t)cfg->max_ingest_docs * 8);
    al((void **)&x->ing.order, (size_t)cfg->max_ingest_docs * 4);
    al((void **)&x->ing.span, 16);
    if (cfg->delta_capacity > 0) {
      // (C / WIN windows of SIG_WORDS words: 8 bytes per ring token)
      al((void **)&x->d_sig, (size_t)(C / WIN) * SIG_WORDS * 4);
      if (e == cudaSuccess) e = cudaMemset(x->d_sig, 0, (size_t)(C / WIN) * SIG_WORDS * 4);
    }
    if (e == cudaSuccess) e = sa_scratch_alloc(&x->sa, C);
    if (e == cudaSuccess) {
      x->dev_bytes += (int64_t)sa_scratch_bytes(C);
      x->pinned_bytes += 64 + 8 * 256 * 4 + 8 + 4 + 4;  // the sort's read-back words, h_n, h_err, h_gd_count
    }
    if (e == cudaSuccess) e = cudaMemset(x->d_rs, 0, sizeof(RingState));
    if (e == cudaSuccess) e = cudaMemset(x->d_doc_start, 0, (size_t)cfg->max_docs * 8);
    if (e == cudaSuccess) e = cudaMemset(x->d_doc_len, 0, (size_t)cfg->max_docs * 4);
    if (e == cudaSuccess) {
      CorpusDesc d0{x->d_text[0], x->d_sa[0], x->d_keys[0], 0, 0, x->d_rec[0], x->d_gt[0], x->gt_mask,
                    0, 0, x->d_gd[0]};
      e = cudaMemcpy(x->d_desc, &d0, sizeof(d0), cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = cudaMallocHost((void **)&x->h_n, 8);
    if (e == cudaSuccess) e = cudaMallocHost((void **)&x->h_err, 4);
    if (e == cudaSuccess) e = cudaMallocHost((void **)&x->h_gd_count, 4);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&x->ev_lin, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreate(&x->ev_b0);
    if (e == cudaSuccess) e = cudaEventCreate(&x->ev_b1);
  }
  if (e == cudaSuccess && x->smem > 48 * 1024) e = propose_set_smem_limit(x->smem);
  if (e == cudaSuccess && cfg->num_backoff > 1) e = backoff_set_smem_limit();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    const bool oom = e == cudaErrorMemoryAllocation;
    free_ctx(x);
    delete x;
    cudaGetLastError();
    return oom ? SGD_ENOMEM : SGD_ECUDA;
  }
  if (x->corpus) {
    try {
      x->worker = std::thread(worker_main, x);
    } catch (...) {
      free_ctx(x);
      delete x;
      return SGD_ENOMEM;
    }
  }
  *out = x;
  return SGD_OK;
}

int sgd_destroy(sgd_ctx *x) {
  if (!x) return SGD_EINVAL;
  cudaSetDevice(x->device);
  if (x->worker.joinable()) {
    {
      std::unique_lock<std::mutex> lk(x->mu);
      x->cv.wait(lk, [&] { return x->bstate != B_RUNNING && !x->job_ready; });
      x->quit = true;
      x->cv.notify_all();
    }
    x->worker.join();
  }
  cudaDeviceSynchronize();
  free_ctx(x);
  delete x;
  return SGD_OK;
}

static ProposeArgs base_args(sgd_ctx *x) {
  ProposeArgs a{};
  const sgd_config &c = x->cfg;
  a.S = c.seq_capacity;
  a.V = c.vocab_size;
  a.k = c.k;
  a.D = c.max_tree_depth;
  a.R = c.max_occurrences;
  a.fN = c.spec_factor_num;
  a.fD = c.spec_factor_den;
  a.offset = c.spec_offset;
  a.pN = c.min_prob_num;
  a.pD = c.min_prob_den;
  a.depth_sum_cap = c.depth_sum_cap;
  a.desc = x->corpus ? x->d_desc : nullptr;
  a.err = x->d_err;
  a.nself = x->nself;
  a.cand_cap = c.corpus_cand_cap;
  a.rsh = x->rsh;
  a.split = x->split;
  a.self_res = x->d_self_res;
  a.by_score = c.select_by_score;
  a.nb = c.num_backoff;
  a.row_stats = x->d_row_stats;
  a.ri = x->ri;
  a.stage_keys = x->stage_keys;
  if (c.draft_mode == 1) {  // no probability floor: the vote runs while an occurrence continues
    a.fixed = 1;
    a.pN = 0;
    a.pD = 1;
  }
  if (x->corpus && c.delta_capacity > 0) {  // the delta is read from the ring in place
    a.dcap = c.delta_capacity;
    a.ring = x->d_ring;
    a.C = c.corpus_capacity;
    a.rs = x->d_rs;
    a.doc_start = x->d_doc_start;
    a.sig = x->d_sig;
  }
  return a;
}

int sgd_update_state(sgd_ctx *x, int32_t *token_ids, int32_t *num_tokens, const int32_t *sampled,
                     int32_t B, int32_t T, void *stream) {
  if (!x || B < 0 || B > x->cfg.max_batch || T < 1 || T > x->cfg.max_sampled) return SGD_EINVAL;
  if (B == 0) return SGD_OK;
  if (!token_ids || !num_tokens || !sampled) return SGD_EINVAL;
  if (!aligned16(token_ids)) return SGD_EINVAL;
  x->launches++;
  return check_cuda(launch_update(token_ids, num_tokens, sampled, B, T, x->cfg.seq_capacity,
                                  x->cfg.vocab_size, x->d_err, x->ri, (cudaStream_t)stream));
}

static int propose_impl(sgd_ctx *x, int32_t *token_ids, int32_t *num_tokens, const int32_t *sampled,
                        int32_t T, const uint8_t *active, int32_t B, int32_t *drafts,
                        int32_t *num_valid, float *score, float *probs, int32_t *match_info,
                        void *stream) {
  if (!x || B < 0 || B > x->cfg.max_batch) return SGD_EINVAL;
  if (sampled && (T < 1 || T > x->cfg.max_sampled)) return SGD_EINVAL;
  if (B == 0) return SGD_OK;
  if (!token_ids || !num_tokens || !drafts || !num_valid) return SGD_EINVAL;
  if (!aligned16(token_ids)) return SGD_EINVAL;
  ProposeArgs a = base_args(x);
  a.tok = token_ids;
  a.ntok = num_tokens;
  a.sampled = sampled;
  a.T = sampled ? T : 0;
  a.do_update = sampled != nullptr;
  a.active = active;
  a.B = B;
  a.drafts = drafts;
  a.num_valid = num_valid;
  a.score = score;
  a.probs = probs;
  a.match_info = match_info;
  if (a.nb > 1) {  // multi-length backoff: one kernel, the update included
    x->launches++;
    return check_cuda(launch_backoff(a, (cudaStream_t)stream));
  }
  x->launches++;
  return check_cuda(launch_propose(a, (cudaStream_t)stream));
}

int sgd_propose(sgd_ctx *x, const int32_t *token_ids, const int32_t *num_tokens,
                const uint8_t *active, int32_t B, int32_t *drafts, int32_t *num_valid, float *score,
                float *probs, int32_t *match_info, void *stream) {
  return propose_impl(x, const_cast<int32_t *>(token_ids), const_cast<int32_t *>(num_tokens),
                      nullptr, 0, active, B, drafts, num_valid, score, probs, match_info, stream);
}

int sgd_propose_with_update(sgd_ctx *x, int32_t *token_ids, int32_t *num_tokens,
                            const int32_t *sampled, int32_t T, const uint8_t *active, int32_t B,
                            int32_t *drafts, int32_t *num_valid, float *score, float *probs,
                            int32_t *match_info, void *stream) {
  if (!sampled && B != 0) return SGD_EINVAL;
  return propose_impl(x, token_ids, num_tokens, sampled, T, active, B, drafts, num_valid, score,
                      probs, match_info, stream);
}

int sgd_step(sgd_ctx *x, int32_t *token_ids, int32_t *num_tokens, const int32_t *sampled, int32_t T,
             const uint8_t *active, int32_t B, int32_t *drafts, int32_t *num_valid, float *score,
             float *probs, int32_t *match_info, const int32_t *rows, const int32_t *starts,
             const int32_t *lengths, int32_t n_docs, void *stream) {
  if (!x) return SGD_EINVAL;
  if (n_docs < 0 || n_docs > x->cfg.max_ingest_docs) return SGD_EINVAL;
  if (n_docs > 0 && !x->corpus) return SGD_ENOCORPUS;
  if (n_docs > 0 && (!rows || !starts || !lengths)) return SGD_EINVAL;
  // (two launches for the long-row mode with a delta: its second kernel must
  // not append to the ring while its rows read delta continuations)
  if (n_docs == 0 || n_docs > propose_step_max_docs() || B == 0 ||
      (x->split && x->cfg.delta_capacity > 0) || x->cfg.num_backoff > 1) {
    int r = sgd_propose_with_update(x, token_ids, num_tokens, sampled, T, active, B, drafts,
                                    num_valid, score, probs, match_info, stream);
    if (r != SGD_OK || n_docs == 0) return r;
    return sgd_ingest(x, token_ids, num_tokens, B, rows, starts, lengths, n_docs, stream);
  }
  if (B < 0 || B > x->cfg.max_batch || !sampled || T < 1 || T > x->cfg.max_sampled)
    return SGD_EINVAL;
  if (!token_ids || !num_tokens || !drafts || !num_valid) return SGD_EINVAL;
  if (!aligned16(token_ids)) return SGD_EINVAL;
  ProposeArgs a = base_args(x);
  a.tok = token_ids;
  a.ntok = num_tokens;
  a.sampled = sampled;
  a.T = T;
  a.do_update = 1;
  a.active = active;
  a.B = B;
  a.drafts = drafts;
  a.num_valid = num_valid;
  a.score = score;
  a.probs = probs;
  a.match_info = match_info;
  a.ing_m = n_docs;
  a.ing_rows = rows;
  a.ing_starts = starts;
  a.ing_lengths = lengths;
  a.ring = x->d_ring;
  a.C = x->cfg.corpus_capacity;
  a.rs = x->d_rs;
  a.doc_start = x->d_doc_start;
  a.doc_len = x->d_doc_len;
  a.max_docs = x->cfg.max_docs;
  a.step_ready = x->d_step_ready;
  a.step_sync = x->d_step_sync;
  {
    std::unique_lock<std::mutex> lk(x->mu);
    if (x->inject == SGD_INJECT_STEP_WAIT) {
      a.ing_skew = 1;
      x->inject = SGD_INJECT_NONE;
    }
  }
  x->launches++;
  return check_cuda(launch_propose(a, (cudaStream_t)stream));
}

int sgd_step_host(sgd_ctx *x, int32_t *token_ids, int32_t *num_tokens, const int32_t *h_sampled,
                  int32_t T, int32_t B, const int32_t *h_rows, const int32_t *h_starts,
                  const int32_t *h_lengths, int32_t n_docs, int32_t *h_drafts, int32_t *h_num_valid,
                  float *h_score, float *h_probs, int32_t *h_match_info, void *stream) {
  if (!x) return SGD_EINVAL;
  if (B < 0 || B > x->cfg.max_batch || T < 1 || T > x->cfg.max_sampled) return SGD_EINVAL;
  if (n_docs < 0 || n_docs > x->cfg.max_ingest_docs) return SGD_EINVAL;
  if (B == 0) return SGD_OK;
  if (!h_sampled || !h_drafts || !h_num_valid) return SGD_EINVAL;
  if (n_docs > 0 && (!h_rows || !h_starts || !h_lengths)) return SGD_EINVAL;
  const size_t k = (size_t)x->cfg.k, BT = (size_t)B * T, m = (size_t)n_docs, Bk = (size_t)B * k;
  // In place: when every host buffer is page-locked and mapped into the GPU's
  // address space (cudaHostAlloc, pinned torch tensors), the kernel reads the
  // step's inputs and writes its outputs in host memory directly, over the
  // GPU's coherent link to it; no staging copies.  Checked once per set of
  // buffers.
  {
    const void *key[9] = {h_sampled, h_rows, h_starts, h_lengths, h_drafts, h_num_valid, h_score,
                          h_probs, h_match_info};
    bool same = true;
    for (int i = 0; i < 9; ++i) same = same && key[i] == x->zc_key[i];
    if (!same) {
      bool ok = true;
      for (int i = 0; i < 9; ++i) {
        x->zc_key[i] = key[i];
        x->zc_dev[i] = nullptr;
        if (key[i] == nullptr) continue;
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, key[i]) != cudaSuccess || at.type != cudaMemoryTypeHost ||
            at.devicePointer == nullptr) {
          cudaGetLastError();
          ok = false;
          continue;
        }
        x->zc_dev[i] = at.devicePointer;
      }
      x->zc_ok = ok;
    }
    if (x->zc_ok) {
      void **d = x->zc_dev;
      return sgd_step(x, token_ids, num_tokens, (const int32_t *)d[0], T, nullptr, B, (int32_t *)d[4],
                      (int32_t *)d[5], (float *)d[6], (float *)d[7], (int32_t *)d[8],
                      (const int32_t *)d[1], (const int32_t *)d[2], (const int32_t *)d[3], n_docs, stream);
    }
  }
  // device staging laid out like a host block [sampled | rows | starts | lengths]
  // and [drafts | num_valid | score | probs | match_info], so that host buffers
  // that sit back to back move in one copy each way
  int32_t *d_samp = x->d_hin;
  int32_t *d_rows = d_samp + BT, *d_starts = d_rows + m, *d_lens = d_starts + m;
  int32_t *d_drafts = x->d_hout;
  int32_t *d_nv = d_drafts + Bk;
  float *d_score = reinterpret_cast<float *>(d_nv + B);
  float *d_probs = d_score + B;
  int32_t *d_mi = reinterpret_cast<int32_t *>(d_probs + Bk);
  cudaStream_t st = (cudaStream_t)stream;
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  cudaError_t e;
  if (m == 0) {
    e = cudaMemcpyAsync(d_samp, h_sampled, BT * 4, h2d, st);
  } else if (h_rows == h_sampled + BT && h_starts == h_rows + m && h_lengths == h_starts + m) {
    e = cudaMemcpyAsync(d_samp, h_sampled, (BT + 3 * m) * 4, h2d, st);
  } else {
    e = cudaMemcpyAsync(d_samp, h_sampled, BT * 4, h2d, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_rows, h_rows, m * 4, h2d, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_starts, h_starts, m * 4, h2d, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_lens, h_lengths, m * 4, h2d, st);
  }
  if (e != cudaSuccess) return check_cuda(e);
  const int r = sgd_step(x, token_ids, num_tokens, d_samp, T, nullptr, B, d_drafts, d_nv,
                         h_score ? d_score : nullptr, h_probs ? d_probs : nullptr,
                         h_match_info ? d_mi : nullptr, d_rows, d_starts, d_lens, n_docs, stream);
  if (r != SGD_OK) return r;
  // outputs: the longest requested run that is contiguous on the host goes in one copy
  size_t run = Bk + B;
  const bool nv_next = h_num_valid == h_drafts + Bk;
  if (nv_next && h_score && (void *)h_score == (void *)(h_num_valid + B)) {
    run += B;
    if (h_probs && h_probs == h_score + B) {
      run += Bk;
      if (h_match_info && (void *)h_match_info == (void *)(h_probs + Bk)) run += 2 * (size_t)B;
    }
  }
  if (nv_next) {
    e = cudaMemcpyAsync(h_drafts, d_drafts, run * 4, d2h, st);
  } else {
    e = cudaMemcpyAsync(h_drafts, d_drafts, Bk * 4, d2h, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h_num_valid, d_nv, (size_t)B * 4, d2h, st);
    run = Bk + B;
  }
  if (e == cudaSuccess && h_score && run <= Bk + B)
    e = cudaMemcpyAsync(h_score, d_score, (size_t)B * 4, d2h, st);
  if (e == cudaSuccess && h_probs && run <= Bk + 2 * (size_t)B)
    e = cudaMemcpyAsync(h_probs, d_probs, Bk * 4, d2h, st);
  if (e == cudaSuccess && h_match_info && run <= 2 * Bk + 2 * (size_t)B)
    e = cudaMemcpyAsync(h_match_info, d_mi, (size_t)B * 8, d2h, st);
  return check_cuda(e);
}

int sgd_ingest(sgd_ctx *x, const int32_t *token_ids, const int32_t *num_tokens, int32_t B,
               const int32_t *rows, const int32_t *starts, const int32_t *lengths, int32_t n_docs,
               void *stream) {
  if (!x) return SGD_EINVAL;
  if (!x->corpus) return SGD_ENOCORPUS;
  if (n_docs < 0 || n_docs > x->cfg.max_ingest_docs || B < 0) return SGD_EINVAL;
  if (n_docs == 0) return SGD_OK;
  if (!token_ids || !rows || !starts || !lengths) return SGD_EINVAL;
  int launches = 0;
  const cudaError_t e =
      launch_ingest(token_ids, num_tokens, B, x->cfg.seq_capacity, x->cfg.vocab_size, rows, starts,
                    lengths, n_docs, x->d_ring, x->cfg.corpus_capacity, x->d_rs, x->d_doc_start,
                    x->d_doc_len, x->cfg.max_docs, x->ing, x->d_sig, x->d_err, (cudaStream_t)stream,
                    &launches);
  x->launches += launches;
  return check_cuda(e);
}

int sgd_build_sa(sgd_ctx *x, void *stream, void *side_stream) {
  if (!x) return SGD_EINVAL;
  if (!x->corpus) return SGD_ENOCORPUS;
  std::unique_lock<std::mutex> lk(x->mu);
  if (x->bstate != B_IDLE || x->job_ready) return SGD_EBUSY;
  const int back = 1 - x->front;
  int launches = 0;
  cudaError_t e = launch_linearize(x->d_ring, x->cfg.corpus_capacity, x->d_rs, x->d_doc_start,
                                   x->cfg.max_docs, x->d_text[back], (cudaStream_t)stream, &launches);
  x->launches += launches;
  if (e == cudaSuccess) e = cudaEventRecord(x->ev_lin, (cudaStream_t)stream);
  if (e != cudaSuccess) return SGD_ECUDA;
  x->job_back = back;
  x->job_side = (cudaStream_t)side_stream;
  x->job_inject = x->inject == SGD_INJECT_STEP_WAIT ? SGD_INJECT_NONE : x->inject;
  if (x->inject != SGD_INJECT_STEP_WAIT) x->inject = SGD_INJECT_NONE;
  x->job_ready = true;
  x->bstate = B_RUNNING;
  x->cv.notify_all();
  return SGD_OK;
}

int sgd_poll(sgd_ctx *x, int wait, int64_t timeout_us, void *stream, uint64_t *generation) {
  if (!x) return SGD_EINVAL;
  if (!x->corpus) return SGD_ENOCORPUS;
  std::unique_lock<std::mutex> lk(x->mu);
  if (x->bstate == B_IDLE) {
    if (generation) *generation = x->gen;
    return SGD_OK;
  }
  if (x->bstate != B_DONE) {
    if (!wait) {
      if (generation) *generation = x->gen;
      return SGD_PENDING;
    }
    auto ready = [&] { return x->bstate == B_DONE; };
    if (timeout_us < 0) {
      x->cv.wait(lk, ready);
    } else if (!x->cv.wait_for(lk, std::chrono::microseconds(timeout_us), ready)) {
      if (generation) *generation = x->gen;
      return SGD_ETIMEDOUT;
    }
  }
  x->bstate = B_IDLE;
  if (x->bstatus != SGD_OK) {
    if (generation) *generation = x->gen;
    return SGD_EBUILD;
  }
  const int back = 1 - x->front;
  const cudaError_t e = launch_swap(x->d_desc, x->d_text[back], x->d_sa[back], x->d_keys[back],
                                    x->d_rec[back], x->d_gt[back], x->gt_mask, x->d_gd[back],
                                    x->built_n, x->gen + 1, x->d_rs, (cudaStream_t)stream);
  if (e != cudaSuccess) return SGD_ECUDA;
  x->launches++;
  x->front = back;
  x->front_n = x->built_n;
  x->gen++;
  if (generation) *generation = x->gen;
  return SGD_OK_SWAPPED;
}

int sgd_suffix_array(sgd_ctx *x, const int32_t *text, int64_t n, int32_t *sa, void *stream) {
  if (!x) return SGD_EINVAL;
  if (!x->corpus) return SGD_ENOCORPUS;
  if (n < 0 || n > x->cfg.corpus_capacity || (n > 0 && (!text || !sa))) return SGD_EINVAL;
  std::unique_lock<std::mutex> lk(x->mu);
  if (x->bstate != B_IDLE || x->job_ready) return SGD_EBUSY;
  cudaStream_t st = (cudaStream_t)stream;
  SaStats stats;
  int launches = 0;
  if (cudaMemsetAsync(x->d_build_err, 0, 4, st) != cudaSuccess) return SGD_ECUDA;
  if (cudaEventRecord(x->ev_b0, st) != cudaSuccess) return SGD_ECUDA;
  const int r = sa_build(x->sa, text, n, sa, x->d_build_err, st, &stats, true, &launches);
  x->launches += launches;
  if (r < 0) return SGD_ECUDA;
  float ms = 0.f;
  if (cudaEventRecord(x->ev_b1, st) != cudaSuccess) return SGD_ECUDA;
  if (cudaMemcpyAsync(x->h_err, x->d_build_err, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SGD_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SGD_ECUDA;
  cudaEventElapsedTime(&ms, x->ev_b0, x->ev_b1);
  const int status = (r != 0 || *x->h_err != 0) ? SGD_EBUILD : SGD_OK;
  x->last.n = n;
  x->last.rounds = stats.rounds;
  x->last.passes = stats.passes;
  x->last.sorted_elems = stats.sorted_elems;
  x->last.pass_elems = stats.pass_elems;
  x->last.model_bytes = stats.model_bytes;
  x->last.ms = ms;
  x->last.pass_ms = stats.pass_ms;
  x->last.status = status;
  return status;
}

int sgd_get_error(sgd_ctx *x, uint32_t *flags, int clear) {
  if (!x || !flags) return SGD_EINVAL;
  if (cudaSetDevice(x->device) != cudaSuccess) return SGD_ECUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return SGD_ECUDA;
  uint32_t a = 0, b = 0;
  if (cudaMemcpy(&a, x->d_err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return SGD_ECUDA;
  if (cudaMemcpy(&b, x->d_build_err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return SGD_ECUDA;
  *flags = a | b;
  if (clear) {
    if (cudaMemset(x->d_err, 0, 4) != cudaSuccess) return SGD_ECUDA;
    std::unique_lock<std::mutex> lk(x->mu);
    if (x->bstate == B_IDLE && cudaMemset(x->d_build_err, 0, 4) != cudaSuccess) return SGD_ECUDA;
  }
  return SGD_OK;
}

int sgd_export_snapshot(sgd_ctx *x, int32_t *text, int32_t *sa, int64_t capacity, int64_t *n,
                        uint64_t *generation) {
  if (!x || !n) return SGD_EINVAL;
  if (!x->corpus) return SGD_ENOCORPUS;
  if (cudaDeviceSynchronize() != cudaSuccess) return SGD_ECUDA;
  *n = x->front_n;
  if (generation) *generation = x->gen;
  if (x->front_n > capacity) return SGD_EINVAL;
  if (x->front_n > 0) {
    if (!text || !sa) return SGD_EINVAL;
    if (cudaMemcpy(text, x->d_text[x->front], (size_t)x->front_n * 4, cudaMemcpyDeviceToDevice) !=
            cudaSuccess ||
        cudaMemcpy(sa, x->d_sa[x->front], (size_t)x->front_n * 4, cudaMemcpyDeviceToDevice) !=
            cudaSuccess)
      return SGD_ECUDA;
  }
  return SGD_OK;
}

// ---------------------------------------------------------------------------
// Save / load of the cross-request corpus ("SuffixGPU" (PyPI), Roadmap: global
// tree save & load).  File: a header, then the ring [C] int32, the document
// FIFO's starts [max_docs] int64 and lengths [max_docs] int32, and the current
// snapshot's text [n] int32, all in the host's byte order.  Loading validates
// everything it reads before anything on the device changes.

namespace {

struct CorpusFileHeader {
  char magic[8];       // "SGDCORP1"
  uint32_t version;    // 1
  int32_t vocab_size;  // V
  int64_t capacity;    // C
  int32_t max_docs;
  int32_t reserved;
  int64_t wp, live, pushed;  // ring state
  int32_t head, ndocs;
  int64_t snap_n;      // tokens of the snapshot text
  int64_t lin_pushed;  // the ring's docs placed and write offset when it was linearised
  int64_t lin_wp;
};

constexpr char kMagic[8] = {'S', 'G', 'D', 'C', 'O', 'R', 'P', '1'};

struct FileCloser {
  FILE *f;
  ~FileCloser() {
    if (f) fclose(f);
  }
};

}  // namespace

int sgd_save(sgd_ctx *x, const char *path, void *stream) {
  if (!x || !path) return SGD_EINVAL;
  if (!x->corpus) return SGD_ENOCORPUS;
  {
    std::unique_lock<std::mutex> lk(x->mu);
    if (x->bstate != B_IDLE || x->job_ready) return SGD_EBUSY;
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SGD_ECUDA;
  const int64_t C = x->cfg.corpus_capacity;
  const int md = x->cfg.max_docs;
  RingState r;
  CorpusDesc d;
  if (cudaMemcpy(&r, x->d_rs, sizeof(r), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(&d, x->d_desc, sizeof(d), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SGD_ECUDA;
  const int64_t n = x->front_n;
  std::vector<int32_t> ring((size_t)C), dl((size_t)md), text((size_t)n);
  std::vector<int64_t> ds((size_t)md);
  if (cudaMemcpy(ring.data(), x->d_ring, (size_t)C * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(ds.data(), x->d_doc_start, (size_t)md * 8, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(dl.data(), x->d_doc_len, (size_t)md * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      (n > 0 && cudaMemcpy(text.data(), x->d_text[x->front], (size_t)n * 4,
                           cudaMemcpyDeviceToHost) != cudaSuccess))
    return SGD_ECUDA;
  CorpusFileHeader h{};
  memcpy(h.magic, kMagic, 8);
  h.version = 1;
  h.vocab_size = x->cfg.vocab_size;
  h.capacity = C;
  h.max_docs = md;
  h.wp = r.wp;
  h.live = r.live;
  h.pushed = r.pushed;
  h.head = r.head;
  h.ndocs = r.ndocs;
  h.snap_n = n;
  h.lin_pushed = d.lin_pushed;
  h.lin_wp = d.lin_wp;
  FileCloser fc{fopen(path, "wb")};
  if (!fc.f) return SGD_EIO;
  bool ok = fwrite(&h, sizeof(h), 1, fc.f) == 1 && fwrite(ring.data(), 4, ring.size(), fc.f) == ring.size() &&
            fwrite(ds.data(), 8, ds.size(), fc.f) == ds.size() &&
            fwrite(dl.data(), 4, dl.size(), fc.f) == dl.size() &&
            fwrite(text.data(), 4, text.size(), fc.f) == text.size();
  ok = fclose(fc.f) == 0 && ok;
  fc.f = nullptr;
  return ok ? SGD_OK : SGD_EIO;
}

int sgd_load(sgd_ctx *x, const char *path, void *stream) {
  if (!x || !path) return SGD_EINVAL;
  if (!x->corpus) return SGD_ENOCORPUS;
  {
    std::unique_lock<std::mutex> lk(x->mu);
    if (x->bstate != B_IDLE || x->job_ready) return SGD_EBUSY;
  }
  const int64_t C = x->cfg.corpus_capacity;
  const int md = x->cfg.max_docs, V = x->cfg.vocab_size;
  FileCloser fc{fopen(path, "rb")};
  if (!fc.f) return SGD_EIO;
  CorpusFileHeader h;
  if (fread(&h, sizeof(h), 1, fc.f) != 1) return SGD_EIO;
  // the file must be this layout, for a context of the same shape, and
  // describe a ring this library could have produced
  if (memcmp(h.magic, kMagic, 8) != 0 || h.version != 1) return SGD_EINVAL;
  if (h.vocab_size != V || h.capacity != C || h.max_docs != md) return SGD_EINVAL;
  if (h.wp < 0 || h.wp >= C || h.live < 0 || h.live > C || h.ndocs < 0 || h.ndocs > md ||
      h.head < 0 || h.head >= md || h.pushed < h.ndocs || h.snap_n < 0 || h.snap_n > C ||
      h.lin_pushed < 0 || h.lin_pushed > h.pushed || h.lin_wp < 0 || h.lin_wp >= C)
    return SGD_EINVAL;
  std::vector<int32_t> ring((size_t)C), dl((size_t)md), text((size_t)h.snap_n);
  std::vector<int64_t> ds((size_t)md);
  if (fread(ring.data(), 4, ring.size(), fc.f) != ring.size() ||
      fread(ds.data(), 8, ds.size(), fc.f) != ds.size() ||
      fread(dl.data(), 4, dl.size(), fc.f) != dl.size() ||
      fread(text.data(), 4, text.size(), fc.f) != text.size())
    return SGD_EIO;
  for (int32_t v : ring)
    if (v < 0 || v > V) return SGD_EINVAL;
  for (int32_t v : text)
    if (v < 0 || v > V) return SGD_EINVAL;
  // the live docs: back to back from the oldest, each followed by the sentinel,
  // ending at the write offset
  int64_t pos = h.ndocs > 0 ? ds[(size_t)h.head] : h.wp, tot = 0;
  for (int32_t i = 0; i < h.ndocs; ++i) {
    const size_t slot = (size_t)((h.head + i) % md);
    if (ds[slot] != pos || dl[slot] < 1 || (int64_t)dl[slot] + 1 > C) return SGD_EINVAL;
    tot += dl[slot] + 1;
    pos = (pos + dl[slot] + 1) % C;
  }
  if (tot != h.live || pos != h.wp) return SGD_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  RingState r{};
  r.wp = h.wp;
  r.live = h.live;
  r.head = h.head;
  r.ndocs = h.ndocs;
  r.pushed = h.pushed;
  r.snap_n = h.snap_n;  // the snapshot to rebuild, and where its delta starts
  r.snap_pushed = h.lin_pushed;
  r.snap_wp = h.lin_wp;
  const int back = 1 - x->front;
  if (cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemcpy(x->d_ring, ring.data(), (size_t)C * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(x->d_doc_start, ds.data(), (size_t)md * 8, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(x->d_doc_len, dl.data(), (size_t)md * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(x->d_rs, &r, sizeof(r), cudaMemcpyHostToDevice) != cudaSuccess ||
      (h.snap_n > 0 && cudaMemcpy(x->d_text[back], text.data(), (size_t)h.snap_n * 4,
                                  cudaMemcpyHostToDevice) != cudaSuccess))
    return SGD_ECUDA;
  if (launch_sig_all(x->d_ring, C, V, x->d_sig, st) != cudaSuccess) return SGD_ECUDA;
  if (h.snap_n == 0) {  // no snapshot: an empty one, the delta from the saved point
    if (launch_swap(x->d_desc, x->d_text[back], x->d_sa[back], x->d_keys[back], x->d_rec[back],
                    x->d_gt[back], x->gt_mask, x->d_gd[back], 0, x->gen + 1, x->d_rs, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return SGD_ECUDA;
    std::unique_lock<std::mutex> lk(x->mu);
    x->front = back;
    x->front_n = 0;
    x->gen++;
    return SGD_OK;
  }
  // the snapshot's index is rebuilt by the worker (as after sgd_build_sa) and swapped in
  if (cudaEventRecord(x->ev_lin, st) != cudaSuccess) return SGD_ECUDA;
  {
    std::unique_lock<std::mutex> lk(x->mu);
    x->job_back = back;
    x->job_side = st;
    x->job_inject = SGD_INJECT_NONE;
    x->job_ready = true;
    x->bstate = B_RUNNING;
    x->cv.notify_all();
  }
  uint64_t gen = 0;
  const int pr = sgd_poll(x, 1, -1, stream, &gen);
  if (pr != SGD_OK_SWAPPED) return pr < 0 ? pr : SGD_ECUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? SGD_OK : SGD_ECUDA;
}

int sgd_corpus_stats(sgd_ctx *x, int64_t *live_tokens, int32_t *ndocs) {
  if (!x) return SGD_EINVAL;
  if (!x->corpus) return SGD_ENOCORPUS;
  if (cudaDeviceSynchronize() != cudaSuccess) return SGD_ECUDA;
  RingState r;
  if (cudaMemcpy(&r, x->d_rs, sizeof(r), cudaMemcpyDeviceToHost) != cudaSuccess) return SGD_ECUDA;
  if (live_tokens) *live_tokens = r.live;
  if (ndocs) *ndocs = r.ndocs;
  return SGD_OK;
}

int sgd_build_stats(sgd_ctx *x, sgd_build_info *info) {
  if (!x || !info) return SGD_EINVAL;
  std::unique_lock<std::mutex> lk(x->mu);
  *info = x->last;
  return SGD_OK;
}

int sgd_debug_inject(sgd_ctx *x, int what) {
  if (!x) return SGD_EINVAL;
  if (what < SGD_INJECT_NONE || what > SGD_INJECT_STEP_WAIT) return SGD_EINVAL;
  std::unique_lock<std::mutex> lk(x->mu);
  x->inject = what;
  if (what == SGD_INJECT_NONE && x->bstate == B_HUNG) {
    x->bstate = B_DONE;
    x->cv.notify_all();
  }
  return SGD_OK;
}

int sgd_reset_rows(sgd_ctx *x, const int32_t *token_ids, const int32_t *num_tokens,
                   const int32_t *rows, int32_t m, void *stream) {
  if (!x || m < 0 || m > (1 << 20)) return SGD_EINVAL;
  if (m == 0 || x->ri.tab == nullptr) return SGD_OK;
  if (!token_ids || !num_tokens || !rows) return SGD_EINVAL;
  x->launches += 2;
  return check_cuda(launch_row_index_reset(x->ri, token_ids, num_tokens, x->cfg.seq_capacity, rows,
                                           m, x->cfg.max_batch, x->d_ri_claim, ++x->ri_epoch,
                                           (cudaStream_t)stream));
}

int sgd_set_row_stats(sgd_ctx *x, int32_t *row_stats) {
  if (!x) return SGD_EINVAL;
  if (row_stats && !aligned16(row_stats)) return SGD_EINVAL;
  x->d_row_stats = row_stats;
  return SGD_OK;
}

int sgd_memory(sgd_ctx *x, int64_t *device_bytes, int64_t *pinned_bytes) {
  if (!x) return SGD_EINVAL;
  if (device_bytes) *device_bytes = x->dev_bytes;
  if (pinned_bytes) *pinned_bytes = x->pinned_bytes;
  return SGD_OK;
}

int sgd_launch_count(sgd_ctx *x, uint64_t *count) {
  if (!x || !count) return SGD_EINVAL;
  *count = x->launches.load();
  return SGD_OK;
}

}  // extern "C"
