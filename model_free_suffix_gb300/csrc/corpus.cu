// corpus.cu -- the ring of finished responses: ingest (scatter_append),
// linearisation of the live docs into a snapshot, and the descriptor swap.
//
// Sources (page title, section):
//   "SuffixGPU" (suffix-gpu 0.1.1, PyPI): Quickstart (harvest_finished, poll);
//     How it works, step 4 (new documents append; oldest documents are
//     evicted when the ring is full; the suffix array is swapped in place).
//   "Suffix Decoding" (vLLM docs): Model Runner V2 (a token budget, oldest
//     first out).
//
// Layout: ring[C] int32 holds the live docs back to back (circularly), each
// followed by the sentinel Z = V.  Because docs are appended at the write
// offset and evicted from the oldest end, the live tokens always form one
// circular run starting at the oldest doc: doc_start[head] + live == wp (mod C).
#include "ingest_cta.cuh"

namespace sgd {

namespace {

// Per doc: check (row, start, length) and find the first id outside [0, V).
__global__ void __launch_bounds__(256) ingest_measure(const int32_t *tok, const int32_t *ntok, int B,
                                                      int S, int V, const int32_t *rows,
                                                      const int32_t *starts, const int32_t *lengths,
                                                      int m, int32_t *eff, uint32_t *err) {
  const int i = blockIdx.x;
  if (i >= m) return;
  __shared__ int s_first;
  const int row = rows[i], st = starts[i], ln = lengths[i];
  const bool ok = row >= 0 && row < B && st >= 0 && ln >= 0 && (long long)st + ln <= S &&
                  (ntok == nullptr || (long long)st + ln <= (long long)ntok[row]);
  if (!ok) {
    if (threadIdx.x == 0) {
      eff[i] = -1;
      atomicOr(err, SGD_ERR_DOC_ARGS);
    }
    return;
  }
  if (threadIdx.x == 0) s_first = ln;
  __syncthreads();
  const int32_t *src = tok + (size_t)row * S + st;
  for (int u = threadIdx.x; u < ln; u += blockDim.x) {
    const int v = src[u];
    if (v < 0 || v >= V) atomicMin(&s_first, u);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    eff[i] = s_first;
    if (s_first < ln) atomicOr(err, SGD_ERR_DOC_TOKEN);
  }
}

constexpr int PLAN_THREADS = 1024;
constexpr int PLAN_CHUNK = 4096;   // docs whose lengths are staged per round

__global__ void __launch_bounds__(PLAN_THREADS) ingest_plan(const int32_t *eff, int m, long long C,
                                                            RingState *rs, int64_t *doc_start,
                                                            int32_t *doc_len, int max_docs,
                                                            int64_t *dest, int32_t *order,
                                                            int64_t *span, uint32_t *err) {
  __shared__ int s_eff[PLAN_CHUNK];
  __shared__ int s_dl[PLAN_WINDOW];
  __shared__ RingState s_rs;
  const int tid = threadIdx.x;
  if (tid == 0) s_rs = *rs;
  __syncthreads();
  PlanWalk w{s_rs, s_rs.ndocs, min(s_rs.ndocs, PLAN_WINDOW), 0, 0, 0, 0u, 0};
  for (int j = tid; j < w.win; j += blockDim.x) s_dl[j] = doc_len[(w.r.head + j) % max_docs];
  for (int c0 = 0; c0 < m; c0 += PLAN_CHUNK) {
    const int cn = min(PLAN_CHUNK, m - c0);
    for (int j = tid; j < cn; j += blockDim.x) s_eff[j] = eff[c0 + j];
    __syncthreads();
    if (tid == 0)
      for (int j = 0; j < cn; ++j)
        place_doc(w, c0 + j, s_eff[j], C, s_dl, doc_start, doc_len, max_docs, dest, order);
    __syncthreads();
  }
  if (tid == 0) {
    *rs = w.r;
    span[0] = s_rs.wp;
    span[1] = w.placed;
    if (w.fl) atomicOr(err, w.fl);
  }
}

// The window signatures after a large call (its span: first position, tokens).
__global__ void __launch_bounds__(256) sig_kernel(SigBuild g, const int64_t *span) {
  __shared__ SigBatchSmem s;
  if (span[1] <= 0) return;
  sig_update_cta(g, span[0], span[1], s, blockIdx.x, gridDim.x);
}

// Every window's signature, from the ring (a restored ring).
__global__ void __launch_bounds__(256) sig_all_kernel(SigBuild g) {
  __shared__ SigBatchSmem s;
  sig_update_cta(g, 0, g.C, s, blockIdx.x, gridDim.x);
}

// A call of up to SMALL_DOCS docs as one CTA.
__global__ void __launch_bounds__(PLAN_THREADS) ingest_small(SmallIngest g) {
  __shared__ SmallIngestSmem s;
  ingest_small_cta(g, s);
}

__global__ void __launch_bounds__(256) ingest_copy(const int32_t *tok, int S, const int32_t *rows,
                                                   const int32_t *starts, const int32_t *eff,
                                                   const int64_t *dest, int m, int32_t *ring,
                                                   long long C, int Z) {
  const int i = blockIdx.x;
  if (i >= m) return;
  const long long d0 = dest[i];
  if (d0 < 0) return;
  const int L = eff[i];
  const int32_t *src = tok + (size_t)rows[i] * S + starts[i];
  for (int u = threadIdx.x; u <= L; u += blockDim.x) {
    long long pos = d0 + u;
    if (pos >= C) pos -= C;
    ring[pos] = u < L ? src[u] : Z;
  }
}

__global__ void __launch_bounds__(256) linearize_kernel(const int32_t *ring, long long C,
                                                        RingState *rs, const int64_t *doc_start,
                                                        int32_t *out) {
  const long long live = rs->live;
  const long long start = rs->ndocs > 0 ? doc_start[rs->head] : 0;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < live; i += stride) {
    long long p = start + i;
    if (p >= C) p -= C;
    out[i] = ring[p];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    rs->snap_n = live;
    rs->snap_pushed = rs->pushed;  // docs placed after this point form the delta
    rs->snap_wp = rs->wp;
  }
}

// The new snapshot becomes current; its delta starts where its linearisation
// stopped (the last linearisation is the one this snapshot was built from:
// no other starts while a build is outstanding).
__global__ void swap_kernel(CorpusDesc *desc, const int32_t *text, const int32_t *sa,
                            const int4 *keys, const int32_t *rec, const int32_t *gt,
                            uint64_t gt_mask, const int32_t *gd, long long n, uint64_t gen,
                            const RingState *rs) {
  desc->gd = gd;
  desc->lin_pushed = rs->snap_pushed;
  desc->lin_wp = rs->snap_wp;
  desc->text = text;
  desc->sa = sa;
  desc->keys = keys;
  desc->rec = rec;
  desc->gt = gt;
  desc->gt_mask = gt_mask;
  desc->n = n;
  desc->gen = gen;
}

// The first m tokens of a key (the rest KEY_END), and whether they exist.
__device__ __forceinline__ bool gram_of(const int4 &k, int m, int4 &g) {
  g = make_int4(k.x, m >= 2 ? k.y : KEY_END, m >= 3 ? k.z : KEY_END, m >= 4 ? k.w : KEY_END);
  return k.x != KEY_END && (m < 2 || k.y != KEY_END) && (m < 3 || k.z != KEY_END) &&
         (m < 4 || k.w != KEY_END);
}

__device__ __forceinline__ bool same_gram(const int4 &a, const int4 &b, int m) {
  return a.x == b.x && (m < 2 || a.y == b.y) && (m < 3 || a.z == b.z) && (m < 4 || a.w == b.w);
}

// n-gram table, pass 1: the first suffix of every run of equal m-grams
// inserts the gram with lo = its position (each gram once, so claims by
// compare-and-swap on the m word are the only contention).
__global__ void __launch_bounds__(256) gram_insert_kernel(const int4 *K, long long n, int32_t *gt,
                                                          uint64_t mask) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x; p < n; p += stride) {
    const int4 k = K[p];
    const int4 kp = p > 0 ? K[p - 1] : make_int4(KEY_END, KEY_END, KEY_END, KEY_END);
    for (int m = 2; m <= 4; ++m) {
      int4 g;
      if (!gram_of(k, m, g)) break;  // shorter than m tokens, so also than m + 1
      if (p > 0 && same_gram(kp, k, m)) continue;
      uint64_t b = gram_hash(m, g.x, g.y, g.z, g.w) & mask;
      for (uint64_t step = 0; step <= mask; ++step, b = (b + 1) & mask) {
        int32_t *e = gt + (size_t)b * GT_BUCKET * GT_ENTRY;
        int j = 0;
        for (; j < GT_BUCKET; ++j, e += GT_ENTRY)
          if (atomicCAS(e, 0, m) == 0) break;
        if (j == GT_BUCKET) continue;
        e[1] = g.x; e[2] = g.y; e[3] = g.z; e[4] = g.w;
        e[5] = (int32_t)p;
        break;
      }
    }
  }
}

// pass 2: the last suffix of every run finds its gram and writes hi.
__global__ void __launch_bounds__(256) gram_hi_kernel(const int4 *K, long long n, int32_t *gt,
                                                      uint64_t mask) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x; p < n; p += stride) {
    const int4 k = K[p];
    const int4 kn = p + 1 < n ? K[p + 1] : make_int4(KEY_END, KEY_END, KEY_END, KEY_END);
    for (int m = 2; m <= 4; ++m) {
      int4 g;
      if (!gram_of(k, m, g)) break;
      if (p + 1 < n && same_gram(kn, k, m)) continue;
      uint64_t b = gram_hash(m, g.x, g.y, g.z, g.w) & mask;
      for (uint64_t step = 0; step <= mask; ++step, b = (b + 1) & mask) {
        int32_t *e = gt + (size_t)b * GT_BUCKET * GT_ENTRY;
        bool done = false;
        for (int j = 0; j < GT_BUCKET && !done; ++j, e += GT_ENTRY)
          if (e[0] == m && e[1] == g.x && e[2] == g.y && e[3] == g.z && e[4] == g.w) {
            e[6] = (int32_t)(p + 1);
            done = true;
          }
        if (done) break;
      }
    }
  }
}

// The record of every suffix-array position, one warp per record: lane f
// writes int f (RecShape: position, tokens before, tokens after the first
// four).  The text around a suffix is contiguous, so a warp's reads fall in
// a few sectors.
__global__ void __launch_bounds__(256) records_kernel(const int32_t *text, const int32_t *sa,
                                                      long long n, RecShape sh, int Z, int32_t *rec) {
  const int lane = threadIdx.x & 31;
  const long long nw = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long p = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < n; p += nw) {
    const long long i = sa[p];
    int32_t *r = rec + (size_t)p * sh.ri;
    for (int f = lane; f < sh.ri; f += 32) {
      int v = 0;
      if (f == 0) {
        v = (int)i;
      } else if (f <= 3) {
        v = i + 3 + f < n ? text[i + 3 + f] : Z;
      } else if (f >= 4 && f < 4 + sh.bk) {
        const long long q = i - 1 - (f - 4);
        v = q >= 0 ? text[q] : KEY_END;
      } else if (f >= sh.co && f < sh.co + sh.kc) {
        const long long q = i + 4 + (f - sh.co);
        v = q < n ? text[q] : Z;
      }
      r[f] = v;
    }
  }
}

// The first four tokens of every suffix, in suffix-array order.  Corpus
// tokens are in [0, V], so KEY_END (INT_MIN) marks the end of the text and
// sorts below every token, as the end of the text does in the suffix order.
__global__ void __launch_bounds__(256) suffix_keys_kernel(const int32_t *text, const int32_t *sa,
                                                          long long n, int4 *keys) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x; p < n; p += stride) {
    const long long i = sa[p];
    int4 k;
    k.x = i < n ? text[i] : KEY_END;
    k.y = i + 1 < n ? text[i + 1] : KEY_END;
    k.z = i + 2 < n ? text[i + 2] : KEY_END;
    k.w = i + 3 < n ? text[i + 3] : KEY_END;
    keys[p] = k;
  }
}

}  // namespace

cudaError_t launch_ingest(const int32_t *tok, const int32_t *ntok, int B, int S, int V,
                          const int32_t *rows, const int32_t *starts, const int32_t *lengths, int m,
                          int32_t *ring, int64_t C, RingState *rs, int64_t *doc_start,
                          int32_t *doc_len, int max_docs, const IngestScratch &sc, uint32_t *sig,
                          uint32_t *err, cudaStream_t st, int *launches) {
  if (m <= 0) return cudaSuccess;
  if (m <= SMALL_DOCS) {
    const SmallIngest g{tok, ntok, B, S, V, rows, starts, lengths, m, ring, C, rs,
                        doc_start, doc_len, max_docs, err, nullptr, 0u, nullptr, nullptr, 0, sig};
    ingest_small<<<1, PLAN_THREADS, 0, st>>>(g);
    *launches += 1;
    return cudaGetLastError();
  }
  ingest_measure<<<m, 256, 0, st>>>(tok, ntok, B, S, V, rows, starts, lengths, m, sc.eff, err);
  ingest_plan<<<1, PLAN_THREADS, 0, st>>>(sc.eff, m, C, rs, doc_start, doc_len, max_docs, sc.dest,
                                          sc.order, sc.span, err);
  ingest_copy<<<m, 256, 0, st>>>(tok, S, rows, starts, sc.eff, sc.dest, m, ring, C, V);
  *launches += 3;
  if (sig != nullptr) {
    sig_kernel<<<2 * 152, 256, 0, st>>>(SigBuild{ring, C, V, sig, C / WIN}, sc.span);
    *launches += 1;
  }
  return cudaGetLastError();
}

cudaError_t launch_sig_all(int32_t *ring, int64_t C, int V, uint32_t *sig, cudaStream_t st) {
  if (sig == nullptr || C <= 0) return cudaSuccess;
  sig_all_kernel<<<2 * 152, 256, 0, st>>>(SigBuild{ring, C, V, sig, C / WIN});
  return cudaGetLastError();
}

cudaError_t launch_linearize(const int32_t *ring, int64_t C, RingState *rs, const int64_t *doc_start,
                             int max_docs, int32_t *out, cudaStream_t st, int *launches) {
  (void)max_docs;
  long long blocks = (C + 1023) / 1024;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  linearize_kernel<<<(int)blocks, 256, 0, st>>>(ring, C, rs, doc_start, out);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_swap(CorpusDesc *desc, const int32_t *text, const int32_t *sa, const int4 *keys,
                        const int32_t *rec, const int32_t *gt, uint64_t gt_mask, const int32_t *gd,
                        int64_t n, uint64_t gen, const RingState *rs, cudaStream_t st) {
  swap_kernel<<<1, 1, 0, st>>>(desc, text, sa, keys, rec, gt, gt_mask, gd, n, gen, rs);
  return cudaGetLastError();
}

cudaError_t launch_gram_table(const int4 *keys, int64_t n, int32_t *gt, uint64_t mask,
                              cudaStream_t st) {
  if (gt == nullptr) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(gt, 0, (size_t)(mask + 1) * GT_BUCKET * GT_ENTRY * 4, st);
  if (e != cudaSuccess || n <= 0) return e;
  long long blocks = (n + 1023) / 1024;
  if (blocks > 152 * 16) blocks = 152 * 16;
  gram_insert_kernel<<<(int)blocks, 256, 0, st>>>(keys, n, gt, mask);
  gram_hi_kernel<<<(int)blocks, 256, 0, st>>>(keys, n, gt, mask);
  return cudaGetLastError();
}

cudaError_t launch_records(const int32_t *text, const int32_t *sa, int64_t n, RecShape shape, int Z,
                           int32_t *rec, cudaStream_t st) {
  if (n <= 0 || rec == nullptr) return cudaSuccess;
  long long blocks = (n + 7) / 8;
  if (blocks > 152 * 16) blocks = 152 * 16;
  records_kernel<<<(int)blocks, 256, 0, st>>>(text, sa, n, shape, Z, rec);
  return cudaGetLastError();
}

cudaError_t launch_suffix_keys(const int32_t *text, const int32_t *sa, int64_t n, int4 *keys,
                               cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  long long blocks = (n + 1023) / 1024;
  if (blocks > 152 * 16) blocks = 152 * 16;
  suffix_keys_kernel<<<(int)blocks, 256, 0, st>>>(text, sa, n, keys);
  return cudaGetLastError();
}

}  // namespace sgd
