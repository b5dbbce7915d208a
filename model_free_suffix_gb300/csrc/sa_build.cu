// sa_build.cu -- suffix array of the corpus snapshot by prefix doubling.
//
// Sources (page title, section):
//   "SuffixGPU" (suffix-gpu 0.1.1, PyPI): References (Manber & Myers, "Suffix
//     Arrays: A New Method for On-Line String Searches": prefix doubling);
//     How it works, step 4 (built on a side CUDA stream).
//
// Order: suffixes compare token by token as signed int32, a proper prefix
// first.  Construction (Manber & Myers): sort by the first h0 tokens (h0
// tokens packed into one 64-bit key: as many as fit at the text's token
// range, at most 4), give every suffix the SA position of the first member of
// its group ("head rank"), then for h = h0, 2h0, 4h0, ... re-sort only the
// suffixes whose group has more than one member by the pair (rank[i],
// rank[i + h]) (rank -1 past the end), until every group is a singleton.
//
// Per round: one kernel builds the keys of the unresolved suffixes and all
// digit histograms; the host reads the round's size and histograms back
// (the one synchronisation of a round) and runs one onesweep LSD radix pass
// per digit place that is not constant; one more kernel writes the sorted
// suffixes back, finds the new groups (a max-scan of group heads) and lists
// the suffixes still unresolved (a sum-scan), both in a single pass.
//
// The passes and the post-processing are single-pass chained scans: a tile
// publishes its aggregate, then looks back over earlier tiles' published
// values.  Tiles take tickets in launch order, so an earlier tile is already
// running; every wait is bounded (after SPIN_LIMIT polls SGD_ERR_LOOKBACK is
// set, the build reports failure and the previous snapshot stays current).
#include <algorithm>
#include <climits>
#include <vector>

#include "sgd_internal.h"

namespace sgd {

namespace {

constexpr int OS_THREADS = 256;
constexpr int OS_ITEMS = 8;
constexpr int OS_TILE = OS_THREADS * OS_ITEMS;  // 2048 items per tile
constexpr int RADIX = 256;
constexpr unsigned SPIN_LIMIT = 1u << 18;  // polls (backing off to 256 ns): ~0.2 s; a normal wait is microseconds
constexpr int MAX_PASSES = 250;            // ticket counters per build
constexpr int LB = 4;                      // look-back words a thread reads per round trip (wider reads more that go unused)

// counter layout (uint32 words): [0] active count written by the post pass,
// [1] [2] smallest and largest token (order-preserving unsigned codes), [3]
// post ticket, [4..] radix-pass tickets
constexpr int CNT_ACTIVE = 0, CNT_MIN = 1, CNT_MAX = 2, CNT_POST = 3, CNT_PASS = 4;
static_assert(CNT_PASS + 250 <= 256, "ticket block is 1 KB");

__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Histograms of the digit places [0, ndig) of the keys this CTA produced,
// accumulated in shared memory and added to the global ones.
__device__ __forceinline__ void hist_flush(uint32_t *s, int ndig, uint32_t *hist) {
  __syncthreads();
  for (int i = threadIdx.x; i < ndig * RADIX; i += blockDim.x)
    if (s[i]) atomicAdd(&hist[i], s[i]);
}

__host__ __device__ inline int bits_of(unsigned long long x) {
  int b = 0;
  while (x) { ++b; x >>= 1; }
  return b;
}

// Round 0 sorts by the first h0 tokens of every suffix at once: token t is
// coded as t - min + 1 in b bits (0 past the end of the text, which sorts a
// proper prefix first), h0 codes packed into one 64-bit key.  Sorting by h0
// tokens before doubling skips the most expensive early rounds.
__host__ __device__ inline void pack_params(uint32_t lo, uint32_t hi, int &h0, int &b) {
  b = bits_of((unsigned long long)(hi - lo) + 1);
  h0 = 64 / b;
  if (h0 > 4) h0 = 4;
  if (h0 < 1) h0 = 1;
}

// smallest and largest token, as order-preserving unsigned codes
__global__ void __launch_bounds__(256) k_minmax(const int32_t *text, long long n, uint32_t *counter) {
  __shared__ uint32_t s_lo[8], s_hi[8];
  uint32_t lo = 0xffffffffu, hi = 0u;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint32_t u = (uint32_t)text[i] ^ 0x80000000u;
    lo = min(lo, u);
    hi = max(hi, u);
  }
  lo = __reduce_min_sync(FULL, lo);
  hi = __reduce_max_sync(FULL, hi);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) { s_lo[warp] = lo; s_hi[warp] = hi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) { lo = min(lo, s_lo[w]); hi = max(hi, s_hi[w]); }
    atomicMin(&counter[CNT_MIN], lo);
    atomicMax(&counter[CNT_MAX], hi);
  }
}

// round 0 keys (h0 packed tokens) and the histograms of their digit places
__global__ void __launch_bounds__(256) k_init_keys(const int32_t *text, long long n,
                                                   const uint32_t *counter, uint64_t *key,
                                                   int32_t *val, uint32_t *hist) {
  __shared__ uint32_t s[8 * RADIX];
  const uint32_t lo = counter[CNT_MIN], hi = counter[CNT_MAX];
  int h0, b;
  pack_params(lo, hi, h0, b);
  const int nd = (h0 * b + 7) / 8;
  for (int i = threadIdx.x; i < nd * RADIX; i += blockDim.x) s[i] = 0;
  __syncthreads();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    uint64_t k = 0;
    for (int t = 0; t < h0; ++t) {
      const long long j = i + t;
      const uint64_t c = j < n ? (uint64_t)(((uint32_t)text[j] ^ 0x80000000u) - lo) + 1 : 0;
      k = (k << b) | c;
    }
    key[i] = k;
    val[i] = (int32_t)i;
    for (int d = 0; d < nd; ++d) atomicAdd(&s[d * RADIX + ((k >> (8 * d)) & 255u)], 1u);
  }
  hist_flush(s, nd, hist);
}

// doubling round: (head rank of i, 1 + head rank of i + h, or 0 past the end)
// for the na unresolved suffixes (na read on the device), with histograms
__global__ void __launch_bounds__(256) k_round_keys(const int32_t *act, const uint32_t *count,
                                                    const int32_t *SA, const int32_t *rank, long long h,
                                                    long long n, int ndig, uint64_t *key, int32_t *val,
                                                    uint32_t *hist) {
  __shared__ uint32_t s[8 * RADIX];
  for (int i = threadIdx.x; i < ndig * RADIX; i += blockDim.x) s[i] = 0;
  __syncthreads();
  const long long na = count[CNT_ACTIVE];
  const long long stride = (long long)gridDim.x * blockDim.x;
  const uint64_t base = (uint64_t)n + 1;
  for (long long a = (long long)blockIdx.x * blockDim.x + threadIdx.x; a < na; a += stride) {
    const int32_t i = SA[act[a]];
    const uint64_t r1 = (uint64_t)rank[i];
    const uint64_t r2 = (long long)i + h < n ? (uint64_t)rank[i + h] + 1 : 0;
    const uint64_t k = r1 * base + r2;
    key[a] = k;
    val[a] = i;
    for (int d = 0; d < ndig; ++d) atomicAdd(&s[d * RADIX + ((k >> (8 * d)) & 255u)], 1u);
  }
  hist_flush(s, ndig, hist);
}

// One LSD pass over the digit at `shift`.  A tile ranks its items stably
// (items in (warp, item, lane) order are the input order), publishes its
// per-digit counts, looks back for the counts of earlier tiles, then stages
// its items in shared memory in digit order so that consecutive threads
// write consecutive outputs.  Look-back words: epoch (bits 63..34, the
// build's pass number), flag (33..32: 1 aggregate, 2 inclusive), count.
__global__ void __launch_bounds__(OS_THREADS, 4) k_onesweep(const uint64_t *kin, const int32_t *vin,
                                                         uint64_t *kout, int32_t *vout, long long n,
                                                         int shift, const uint32_t *hist_d,
                                                         unsigned long long *status, uint32_t *ticket,
                                                         unsigned long long epoch, uint32_t *err) {
  constexpr int NW = OS_THREADS / 32;
  __shared__ uint32_t s_whist[NW][RADIX];
  __shared__ uint32_t s_base[RADIX];    // global start of each digit
  __shared__ uint32_t s_tstart[RADIX];  // start of each digit inside this tile
  __shared__ uint32_t s_excl[RADIX];    // items of each digit in earlier tiles
  __shared__ uint32_t s_wsum[NW];
  __shared__ uint64_t s_k[OS_TILE];
  __shared__ int32_t s_v[OS_TILE];
  __shared__ int s_tile;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_tile = (int)atomicAdd(ticket, 1u);
  for (int i = tid; i < NW * RADIX; i += OS_THREADS) (&s_whist[0][0])[i] = 0;
  {
    const uint32_t c = hist_d[tid];
    uint32_t x = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    uint32_t pre = 0;
    for (int w = 0; w < warp; ++w) pre += s_wsum[w];
    s_base[tid] = pre + x - c;
  }
  __syncthreads();
  const long long tile = s_tile;
  const long long tbase = tile * OS_TILE + (long long)warp * (OS_ITEMS * 32);
  uint64_t key[OS_ITEMS];
  int32_t val[OS_ITEMS];
  uint32_t rk[OS_ITEMS];
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int it = 0; it < OS_ITEMS; ++it) {
    const long long idx = tbase + it * 32 + lane;
    const bool valid = idx < n;
    key[it] = valid ? kin[idx] : 0;
    val[it] = valid ? vin[idx] : 0;
  }
#pragma unroll
  for (int it = 0; it < OS_ITEMS; ++it) {
    const long long idx = tbase + it * 32 + lane;
    const bool valid = idx < n;
    const unsigned vm = __ballot_sync(FULL, valid);
    const uint32_t dg = (uint32_t)(key[it] >> shift) & 255u;
    unsigned peers = 0;
    uint32_t before = 0;
    if (valid) {
      peers = __match_any_sync(vm, dg);
      before = s_whist[warp][dg];
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) s_whist[warp][dg] = before + __popc(peers);
    __syncwarp();
    rk[it] = before + __popc(peers & lt);
  }
  __syncthreads();
  // per digit d: warp-exclusive offsets, the tile count, its start in the tile
  const int d = tid;
  uint32_t cnt = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const uint32_t c = s_whist[w][d];
    s_whist[w][d] = cnt;
    cnt += c;
  }
  {
    uint32_t x = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, x, off);
      if (lane >= off) x += y;
    }
    __syncthreads();  // s_wsum reuse
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    uint32_t pre = 0;
    for (int w = 0; w < warp; ++w) pre += s_wsum[w];
    s_tstart[d] = pre + x - cnt;
  }
  // decoupled look-back for digit d
  unsigned long long *my = status + (size_t)tile * RADIX + d;
  const unsigned long long tag = epoch << 34;
  uint32_t excl = 0;
  if (tile == 0) {
    st_relaxed64(my, tag | (2ull << 32) | cnt);
  } else {
    st_relaxed64(my, tag | (1ull << 32) | cnt);
    // LB predecessors per round trip; consume them nearest first and stop at
    // the first inclusive word (done) or the first one not yet published
    long long t = tile - 1;
    unsigned spins = 0;
    bool failed = false;
    for (;;) {
      unsigned long long w[LB];
#pragma unroll
      for (int j = 0; j < LB; ++j)
        w[j] = t - j >= 0 ? ld_relaxed64(status + (size_t)(t - j) * RADIX + d) : 0ull;
      int used = 0;
      bool done = false;
#pragma unroll
      for (int j = 0; j < LB; ++j) {
        if (done || used != j || (w[j] >> 34) != epoch) continue;
        excl += (uint32_t)w[j];
        used = j + 1;
        done = ((w[j] >> 32) & 3ull) == 2ull;
      }
      if (done) break;
      t -= used;
      if (used == 0) {
        if (++spins > SPIN_LIMIT) { failed = true; break; }
        if (spins > 2) __nanosleep(spins < 8 ? 64 : 256);  // back off: polls cost issue slots
      }
    }
    if (failed) atomicOr(err, SGD_ERR_LOOKBACK);
    st_relaxed64(my, tag | (2ull << 32) | (uint32_t)(excl + cnt));
  }
  s_excl[d] = excl;
  __syncthreads();
  // stage the tile in digit order
#pragma unroll
  for (int it = 0; it < OS_ITEMS; ++it) {
    const long long idx = tbase + it * 32 + lane;
    if (idx < n) {
      const uint32_t dg = (uint32_t)(key[it] >> shift) & 255u;
      const uint32_t lp = s_tstart[dg] + s_whist[warp][dg] + rk[it];
      s_k[lp] = key[it];
      s_v[lp] = val[it];
    }
  }
  __syncthreads();
  const long long tn = min((long long)OS_TILE, n - tile * OS_TILE);
  for (int i = tid; i < tn; i += OS_THREADS) {
    const uint64_t k = s_k[i];
    const uint32_t dg = (uint32_t)(k >> shift) & 255u;
    const uint64_t dst = (uint64_t)s_base[dg] + s_excl[dg] + (i - s_tstart[dg]);
    if (dst < (uint64_t)n) {  // always true unless a look-back gave up (the build then fails)
      kout[dst] = k;
      vout[dst] = s_v[i];
    }
  }
}

// After a round's sort (na sorted keys/values; act maps them to SA slots, or
// is the identity in round 0): write each suffix to its slot, give it the SA
// position of the first member of its new group (a running max of the
// positions of group heads), and list the suffixes whose group still has
// another member (a running count of them gives their place in act2).  Both
// scans run in one pass; look-back words pack flag (bits 63..62), the max
// head position + 1 (61..31) and the count (30..0).
__global__ void __launch_bounds__(OS_THREADS) k_post(const int32_t *act, long long na,
                                                     const uint64_t *key, const int32_t *val,
                                                     int32_t *SA, int32_t *rank, int32_t *act2,
                                                     unsigned long long *pstatus, uint32_t *counter,
                                                     uint32_t *err) {
  constexpr int NW = OS_THREADS / 32;
  __shared__ uint32_t s_wmax[NW], s_wsum[NW];
  __shared__ uint32_t s_emax, s_esum;
  __shared__ int s_tile;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_tile = (int)atomicAdd(&counter[CNT_POST], 1u);
  __syncthreads();
  const long long tile = s_tile;
  const long long base = tile * OS_TILE + (long long)tid * OS_ITEMS;
  uint32_t hp[OS_ITEMS];  // head position + 1, or 0
  uint32_t keep = 0;      // bit i: item i stays unresolved
  uint32_t tmax = 0, tsum = 0;
#pragma unroll
  for (int i = 0; i < OS_ITEMS; ++i) {
    const long long a = base + i;
    hp[i] = 0;
    if (a < na) {
      const uint64_t k = key[a];
      const bool head = a == 0 || key[a - 1] != k;
      const bool last = a == na - 1 || key[a + 1] != k;
      const int32_t p = act ? act[a] : (int32_t)a;
      if (head) hp[i] = (uint32_t)p + 1;
      if (!(head && last)) { keep |= 1u << i; ++tsum; }
      tmax = max(tmax, hp[i]);
    }
  }
  // block-exclusive (max, sum) over threads
  uint32_t xm = tmax, xs = tsum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t ym = __shfl_up_sync(FULL, xm, off), ys = __shfl_up_sync(FULL, xs, off);
    if (lane >= off) { xm = max(xm, ym); xs += ys; }
  }
  if (lane == 31) { s_wmax[warp] = xm; s_wsum[warp] = xs; }
  __syncthreads();
  uint32_t pm = 0, ps = 0, Tm = 0, Ts = 0;
  for (int w = 0; w < NW; ++w) {
    if (w < warp) { pm = max(pm, s_wmax[w]); ps += s_wsum[w]; }
    Tm = max(Tm, s_wmax[w]);
    Ts += s_wsum[w];
  }
  uint32_t em = max(pm, __shfl_up_sync(FULL, xm, 1)), es = ps + __shfl_up_sync(FULL, xs, 1);
  if (lane == 0) { em = pm; es = ps; }
  // tile look-back (warp 0): lane i reads the word of tile t - i, 32 tiles
  // per round trip, consumed nearest first up to the first inclusive word or
  // the first word not yet published
  if (warp == 0) {
    unsigned long long *my = pstatus + tile;
    uint32_t bm = 0, bs = 0;
    auto pack = [](unsigned long long flag, uint32_t m, uint32_t s) {
      return (flag << 62) | ((unsigned long long)m << 31) | (unsigned long long)s;
    };
    if (tile == 0) {
      if (lane == 0) st_relaxed64(my, pack(2, Tm, Ts));
    } else {
      if (lane == 0) st_relaxed64(my, pack(1, Tm, Ts));
      long long t = tile - 1;
      unsigned spins = 0;
      bool failed = false;
      for (;;) {
        const unsigned long long w = t - lane >= 0 ? ld_relaxed64(pstatus + (t - lane)) : 0ull;
        const unsigned fl = (unsigned)(w >> 62);
        const unsigned inc = __ballot_sync(FULL, fl == 2), unp = __ballot_sync(FULL, fl == 0);
        const int first_inc = inc ? __ffs(inc) - 1 : 32, first_unp = unp ? __ffs(unp) - 1 : 32;
        const bool done = first_inc < first_unp;
        const int used = done ? first_inc + 1 : first_unp;  // lanes [0, used) are consumed
        const bool take = lane < used;
        const uint32_t m = take ? (uint32_t)((w >> 31) & 0x7fffffffull) : 0u;
        const uint32_t c = take ? (uint32_t)(w & 0x7fffffffull) : 0u;
        bm = max(bm, __reduce_max_sync(FULL, m));
        bs += __reduce_add_sync(FULL, c);
        if (done) break;
        t -= used;
        if (used == 0) {
          if (++spins > SPIN_LIMIT) { failed = true; break; }
          if (spins > 2) __nanosleep(spins < 8 ? 64 : 256);  // back off: polls cost issue slots
        }
      }
      if (lane == 0) {
        if (failed) atomicOr(err, SGD_ERR_LOOKBACK);
        st_relaxed64(my, pack(2, max(bm, Tm), bs + Ts));
      }
    }
    if (lane == 0) {
      s_emax = bm;
      s_esum = bs;
      if ((tile + 1) * (long long)OS_TILE >= na) counter[CNT_ACTIVE] = bs + Ts;  // the last tile
    }
  }
  __syncthreads();
  uint32_t rm = max(s_emax, em), rs = s_esum + es;
#pragma unroll
  for (int i = 0; i < OS_ITEMS; ++i) {
    const long long a = base + i;
    if (a >= na) break;
    rm = max(rm, hp[i]);
    const int32_t p = act ? act[a] : (int32_t)a;
    const int32_t v = val[a];
    SA[p] = v;
    rank[v] = (int32_t)rm - 1;
    if (keep & (1u << i)) act2[rs++] = p;
  }
}

int grid_for(long long n, int per_block) {
  long long g = (n + per_block - 1) / per_block;
  if (g > 152 * 16) g = 152 * 16;
  if (g < 1) g = 1;
  return (int)g;
}


}  // namespace

size_t sa_scratch_bytes(int64_t cap) {
  const long long c = cap > 0 ? cap : 1;
  const long long tiles = (c + OS_TILE - 1) / OS_TILE;
  return (size_t)c * (8 + 8 + 4 * 5) + (size_t)tiles * RADIX * 8 + (size_t)tiles * 8 +
         8 * RADIX * 4 + 1024 + 16 * 256;
}

size_t sa_scratch_carve(SaScratch *s, unsigned char *base, size_t bytes, int64_t cap) {
  *s = SaScratch{};
  const long long c = cap > 0 ? cap : 1;
  const long long tiles = (c + OS_TILE - 1) / OS_TILE;
  size_t off = 0;
  auto take = [&](size_t n) {
    unsigned char *p = base + off;
    off += (n + 255) & ~(size_t)255;
    return p;
  };
  s->cap = cap;
  s->status_words = tiles * RADIX;
  s->keyA = (uint64_t *)take(c * 8);
  s->keyB = (uint64_t *)take(c * 8);
  s->valA = (int32_t *)take(c * 4);
  s->valB = (int32_t *)take(c * 4);
  s->rank = (int32_t *)take(c * 4);
  s->act = (int32_t *)take(c * 4);
  s->act2 = (int32_t *)take(c * 4);
  s->status = (unsigned long long *)take(s->status_words * 8);
  s->pstatus = (unsigned long long *)take(tiles * 8);
  s->hist = (uint32_t *)take(8 * RADIX * 4);
  s->counter = (uint32_t *)take(1024);
  if (off > bytes) *s = SaScratch{};
  return off;
}

cudaError_t sa_scratch_alloc(SaScratch *s, int64_t cap) {
  *s = SaScratch{};
  const size_t bytes = sa_scratch_bytes(cap);
  unsigned char *base = nullptr;
  cudaError_t e = cudaMalloc((void **)&base, bytes);
  if (e != cudaSuccess) return e;
  sa_scratch_carve(s, base, bytes, cap);
  s->owned = base;
  e = cudaMallocHost((void **)&s->h_pinned, 64);
  if (e == cudaSuccess) e = cudaMallocHost((void **)&s->h_hist, 8 * RADIX * 4);
  // four radix-pass CTAs per SM (64 registers, 36 KB of shared memory each):
  // the largest shared-memory carveout
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute((const void *)k_onesweep, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) sa_scratch_free(s);
  return e;
}

void sa_scratch_free(SaScratch *s) {
  if (s->owned) cudaFree(s->owned);
  if (s->h_pinned) cudaFreeHost(s->h_pinned);
  if (s->h_hist) cudaFreeHost(s->h_hist);
  *s = SaScratch{};
}

int sa_build(const SaScratch &s, const int32_t *text, int64_t n, int32_t *sa, uint32_t *err,
             cudaStream_t st, SaStats *stats, bool time_passes, int *launches) {
  SaStats local;
  if (!stats) stats = &local;
  *stats = SaStats{};
  if (n <= 0) return 0;
  if (n > s.cap || s.keyA == nullptr) return -1;
  if (n == 1) return cudaMemsetAsync(sa, 0, 4, st) == cudaSuccess ? 0 : -1;
  const long long tiles_max = (n + OS_TILE - 1) / OS_TILE;
  std::vector<cudaEvent_t> evs;
  unsigned long long epoch = 0;
  int pass_idx = 0;
  uint64_t *kin = s.keyA, *kout = s.keyB;
  int32_t *vin = s.valA, *vout = s.valB;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (!ok(cudaMemsetAsync(s.status, 0, (size_t)tiles_max * RADIX * 8, st))) return -1;
  if (!ok(cudaMemsetAsync(s.counter, 0, 1024, st))) return -1;
  if (!ok(cudaMemsetAsync(s.counter + CNT_MIN, 0xff, 4, st))) return -1;

  // LSD passes over the non-constant digit places of (kin, vin)[0..na)
  auto passes = [&](long long na, int ndig) -> bool {
    const long long tiles = (na + OS_TILE - 1) / OS_TILE;
    kin = s.keyA; vin = s.valA; kout = s.keyB; vout = s.valB;
    for (int d = 0; d < ndig; ++d) {
      bool trivial = false;
      for (int v = 0; v < RADIX; ++v)
        if ((long long)s.h_hist[d * RADIX + v] == na) trivial = true;
      if (trivial) continue;
      if (pass_idx >= MAX_PASSES) return false;
      cudaEvent_t e0 = nullptr, e1 = nullptr;
      if (time_passes) {
        cudaEventCreate(&e0);
        cudaEventCreate(&e1);
        cudaEventRecord(e0, st);
      }
      k_onesweep<<<(unsigned)tiles, OS_THREADS, 0, st>>>(kin, vin, kout, vout, na, 8 * d,
                                                         s.hist + d * RADIX, s.status,
                                                         s.counter + CNT_PASS + pass_idx, ++epoch, err);
      ++pass_idx;
      ++*launches;
      if (time_passes) {
        cudaEventRecord(e1, st);
        evs.push_back(e0);
        evs.push_back(e1);
      }
      if (!ok(cudaGetLastError())) return false;
      stats->passes++;
      stats->pass_elems += na;
      std::swap(kin, kout);
      std::swap(vin, vout);
    }
    return true;
  };
  auto read_back = [&](int ndig) -> bool {
    if (!ok(cudaMemcpyAsync(s.h_pinned, s.counter + CNT_ACTIVE, 12, cudaMemcpyDeviceToHost, st)))
      return false;
    if (!ok(cudaMemcpyAsync(s.h_hist, s.hist, (size_t)ndig * RADIX * 4, cudaMemcpyDeviceToHost, st)))
      return false;
    return ok(cudaStreamSynchronize(st));
  };

  // round 0: sort by the first h0 tokens
  if (!ok(cudaMemsetAsync(s.hist, 0, 8 * RADIX * 4, st))) return -1;
  k_minmax<<<grid_for(n, 256 * 8), 256, 0, st>>>(text, n, s.counter);
  k_init_keys<<<grid_for(n, 256 * 4), 256, 0, st>>>(text, n, s.counter, s.keyA, s.valA, s.hist);
  *launches += 2;
  if (!read_back(8)) return -1;
  int h0 = 1, b0 = 32;
  pack_params((uint32_t)s.h_pinned[1], (uint32_t)s.h_pinned[2], h0, b0);
  if (!passes(n, (h0 * b0 + 7) / 8)) return -1;
  long long na = n;
  const int32_t *act = nullptr;
  int32_t *act_next = s.act;
  long long h = h0;
  const int ndig = (bits_of((unsigned long long)(n - 1) * (unsigned long long)(n + 1) +
                            (unsigned long long)n) + 7) / 8;
  for (;;) {
    stats->rounds++;
    stats->sorted_elems += na;
    const long long tiles = (na + OS_TILE - 1) / OS_TILE;
    if (!ok(cudaMemsetAsync(s.pstatus, 0, (size_t)tiles * 8, st))) return -1;
    if (!ok(cudaMemsetAsync(s.counter + CNT_POST, 0, 4, st))) return -1;
    k_post<<<(unsigned)tiles, OS_THREADS, 0, st>>>(act, na, kin, vin, sa, s.rank, act_next, s.pstatus,
                                                   s.counter, err);
    ++*launches;
    if (h >= n) break;  // cannot happen for a valid order; guards the loop
    // next round's keys over the unresolved suffixes (their number is read on
    // the device), then its size and histograms in one read-back
    if (!ok(cudaMemsetAsync(s.hist, 0, 8 * RADIX * 4, st))) return -1;
    k_round_keys<<<grid_for(na, 256 * 4), 256, 0, st>>>(act_next, s.counter, sa, s.rank, h, n, ndig,
                                                        s.keyA, s.valA, s.hist);
    ++*launches;
    if (!read_back(ndig)) return -1;
    const long long next = s.h_pinned[0];
    stats->model_bytes += na * (16 + 12);
    if (next == 0) break;
    act = act_next;
    act_next = (act_next == s.act) ? s.act2 : s.act;
    na = next;
    const int passes_before = stats->passes;
    if (!passes(na, ndig)) return -1;
    stats->model_bytes += na * 24LL * (stats->passes - passes_before);
    h *= 2;
  }
  stats->model_bytes += 8LL * n;
  if (!ok(cudaStreamSynchronize(st))) return -1;
  for (size_t i = 0; i + 1 < evs.size(); i += 2) {
    float ms = 0;
    cudaEventElapsedTime(&ms, evs[i], evs[i + 1]);
    stats->pass_ms += ms;
    cudaEventDestroy(evs[i]);
    cudaEventDestroy(evs[i + 1]);
  }
  return 0;
}

}  // namespace sgd
