// sa_build.cu -- suffix array of the corpus snapshot by prefix doubling.
//
// Sources (page title, section):
//   "SuffixGPU" (suffix-gpu 0.1.1, PyPI): References (Manber & Myers, "Suffix
//     Arrays: A New Method for On-Line String Searches": prefix doubling);
//     How it works, step 4 (built on a side CUDA stream).
//
// Order: suffixes compare token by token as signed int32, a proper prefix
// first.  Construction (Manber & Myers): sort by the first token, give every
// suffix the SA position of the first member of its group ("head rank"),
// then for h = 1, 2, 4, ... re-sort only the suffixes whose group has more
// than one member by the pair (rank[i], rank[i + h]) (rank -1 past the end),
// until every group is a singleton.  Each sort is an LSD radix sort over
// 8-bit digits with one onesweep pass per digit: one kernel per pass that
// ranks each tile's items, publishes the tile's per-digit counts and looks
// back over earlier tiles' published counts (decoupled look-back, with a
// bounded wait) to place its items.  Digit places whose 256 buckets hold
// everything in one bucket are skipped.
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
constexpr uint32_t FLAG_AGG = 1u << 30;
constexpr uint32_t FLAG_INC = 2u << 30;
constexpr uint32_t VALUE_MASK = (1u << 30) - 1;
constexpr unsigned SPIN_LIMIT = 1u << 18;  // ~0.1 s of polling; a normal wait is microseconds

constexpr int SC_THREADS = 256;
constexpr int SC_ITEMS = 8;
constexpr int SC_TILE = SC_THREADS * SC_ITEMS;

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed(uint32_t *p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// round 0 keys: the token itself, order-preserving for signed int32
__global__ void k_init0(const int32_t *text, long long n, uint64_t *key, int32_t *val) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    key[i] = (uint64_t)((uint32_t)text[i] ^ 0x80000000u);
    val[i] = (int32_t)i;
  }
}

// doubling-round keys: (head rank of i, 1 + head rank of i + h, or 0 past the end)
__global__ void k_keys(const int32_t *act, long long na, const int32_t *SA, const int32_t *rank,
                       long long h, long long n, uint64_t *key, int32_t *val) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const uint64_t base = (uint64_t)n + 1;
  for (long long a = (long long)blockIdx.x * blockDim.x + threadIdx.x; a < na; a += stride) {
    const int32_t i = SA[act[a]];
    const uint64_t r1 = (uint64_t)rank[i];
    const uint64_t r2 = (long long)i + h < n ? (uint64_t)rank[i + h] + 1 : 0;
    key[a] = r1 * base + r2;
    val[a] = i;
  }
}

// all digit-place histograms in one read of the keys
__global__ void __launch_bounds__(256) k_hist(const uint64_t *key, long long n, int ndig,
                                              uint32_t *hist) {
  __shared__ uint32_t s[8 * RADIX];
  for (int i = threadIdx.x; i < ndig * RADIX; i += blockDim.x) s[i] = 0;
  __syncthreads();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t k = key[i];
    for (int d = 0; d < ndig; ++d) atomicAdd(&s[d * RADIX + ((k >> (8 * d)) & 255u)], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ndig * RADIX; i += blockDim.x)
    if (s[i]) atomicAdd(&hist[i], s[i]);
}

// One LSD pass over the digit at `shift`.  Tiles take tickets in launch
// order; tile t waits only for tiles < t, which hold earlier tickets and so
// are already running, and every tile publishes its own counts before it
// waits.  A wait longer than SPIN_LIMIT polls sets SGD_ERR_LOOKBACK (the
// build is then reported failed) instead of hanging.
__global__ void __launch_bounds__(OS_THREADS) k_onesweep(const uint64_t *kin, const int32_t *vin,
                                                         uint64_t *kout, int32_t *vout, long long n,
                                                         int shift, const uint32_t *hist_d,
                                                         uint32_t *status, uint32_t *ticket,
                                                         uint32_t *err) {
  constexpr int NW = OS_THREADS / 32;
  __shared__ uint32_t s_whist[NW][RADIX];
  __shared__ uint32_t s_base[RADIX];
  __shared__ uint32_t s_excl[RADIX];
  __shared__ uint32_t s_wsum[NW];
  __shared__ int s_tile;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_tile = (int)atomicAdd(ticket, 1u);
  for (int i = tid; i < NW * RADIX; i += OS_THREADS) (&s_whist[0][0])[i] = 0;
  // global start of every digit: exclusive scan of this digit place's histogram
  {
    uint32_t c = hist_d[tid];
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
  // stable ranks inside the warp: items in (item, lane) order = input order
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
  // per digit: warp-exclusive offsets and the tile count
  const int d = tid;
  uint32_t cnt = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const uint32_t c = s_whist[w][d];
    s_whist[w][d] = cnt;
    cnt += c;
  }
  // decoupled look-back for digit d
  uint32_t *my = status + (size_t)tile * RADIX + d;
  uint32_t excl = 0;
  if (tile == 0) {
    st_relaxed(my, FLAG_INC | cnt);
  } else {
    st_relaxed(my, FLAG_AGG | cnt);
    long long t = tile - 1;
    unsigned spins = 0;
    bool failed = false;
    while (t >= 0) {
      const uint32_t s = ld_relaxed(status + (size_t)t * RADIX + d);
      const uint32_t fl = s & ~VALUE_MASK;
      if (fl == 0) {
        if (++spins > SPIN_LIMIT) { failed = true; break; }
        if (spins > 64) __nanosleep(32);
        continue;
      }
      excl += s & VALUE_MASK;
      if (fl == FLAG_INC) break;
      --t;
    }
    if (failed) atomicOr(err, SGD_ERR_LOOKBACK);
    st_relaxed(my, FLAG_INC | ((excl + cnt) & VALUE_MASK));
  }
  s_excl[d] = excl;
  __syncthreads();
#pragma unroll
  for (int it = 0; it < OS_ITEMS; ++it) {
    const long long idx = tbase + it * 32 + lane;
    if (idx < n) {
      const uint32_t dg = (uint32_t)(key[it] >> shift) & 255u;
      const uint32_t dst = s_base[dg] + s_excl[dg] + s_whist[warp][dg] + rk[it];
      if (dst < n) {  // always true unless a look-back gave up (the build then fails)
        kout[dst] = key[it];
        vout[dst] = val[it];
      }
    }
  }
}

// After a round's sort: write the suffixes back to their SA slots, mark the
// first member of every new group and give it its SA position.
__global__ void k_post(const int32_t *act, long long na, const uint64_t *key, const int32_t *val,
                       int32_t *SA, int32_t *headpos, int32_t *head) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long a = (long long)blockIdx.x * blockDim.x + threadIdx.x; a < na; a += stride) {
    const int32_t p = act ? act[a] : (int32_t)a;
    SA[p] = val[a];
    const int h = a == 0 || key[a] != key[a - 1];
    head[a] = h;
    headpos[a] = h ? p : -1;
  }
}

// rank[i] = head position of i's group; flag suffixes whose group has >= 2 members
__global__ void k_rank(long long na, const int32_t *val, const int32_t *newrank, const int32_t *head,
                       int32_t *rank, int32_t *keep) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long a = (long long)blockIdx.x * blockDim.x + threadIdx.x; a < na; a += stride) {
    rank[val[a]] = newrank[a];
    const bool single = head[a] && (a == na - 1 || head[a + 1]);
    keep[a] = single ? 0 : 1;
  }
}

__global__ void k_compact(long long na, const int32_t *act, const int32_t *head, const int32_t *pos,
                          int32_t *act2, int32_t *count) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long a = (long long)blockIdx.x * blockDim.x + threadIdx.x; a < na; a += stride) {
    const bool single = head[a] && (a == na - 1 || head[a + 1]);
    if (!single) act2[pos[a]] = act ? act[a] : (int32_t)a;
    if (a == na - 1) *count = pos[a] + (single ? 0 : 1);
  }
}

// ---------------------------------------------------------------------------
// device-wide scans (sum or max) in three steps: tile totals, a scan of the
// totals in one CTA, and the per-tile scan with its offset.
template <bool MAX>
__device__ __forceinline__ int sop(int a, int b) { return MAX ? max(a, b) : a + b; }
template <bool MAX>
__device__ __forceinline__ int sid() { return MAX ? INT_MIN : 0; }

// Block-wide scan of one value per thread: inclusive and exclusive prefixes
// and the block total.
template <bool MAX>
__device__ void block_scan(int v, int &incl, int &excl, int &total) {
  constexpr int NW = SC_THREADS / 32;
  __shared__ int s_w[NW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(FULL, x, off);
    if (lane >= off) x = sop<MAX>(x, y);
  }
  int wex = __shfl_up_sync(FULL, x, 1);
  if (lane == 0) wex = sid<MAX>();
  if (lane == 31) s_w[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NW ? s_w[lane] : sid<MAX>();
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(FULL, w, off);
      if (lane >= off) w = sop<MAX>(w, y);
    }
    if (lane < NW) s_w[lane] = w;
  }
  __syncthreads();
  const int pre = warp > 0 ? s_w[warp - 1] : sid<MAX>();
  incl = sop<MAX>(pre, x);
  excl = sop<MAX>(pre, wex);
  total = s_w[NW - 1];
  __syncthreads();
}

template <bool MAX>
__global__ void __launch_bounds__(SC_THREADS) k_scan_reduce(const int32_t *in, long long n,
                                                            int32_t *tile_sums) {
  const long long base = (long long)blockIdx.x * SC_TILE + (long long)threadIdx.x * SC_ITEMS;
  int acc = sid<MAX>();
#pragma unroll
  for (int i = 0; i < SC_ITEMS; ++i)
    if (base + i < n) acc = sop<MAX>(acc, in[base + i]);
  int incl, excl, total;
  block_scan<MAX>(acc, incl, excl, total);
  if (threadIdx.x == 0) tile_sums[blockIdx.x] = total;
}

// exclusive scan of the tile totals, in place, one CTA
template <bool MAX>
__global__ void __launch_bounds__(SC_THREADS) k_scan_tiles(int32_t *tile_sums, long long ntiles) {
  int carry = sid<MAX>();
  for (long long base = 0; base < ntiles; base += SC_THREADS) {
    const long long i = base + threadIdx.x;
    const int v = i < ntiles ? tile_sums[i] : sid<MAX>();
    int incl, excl, total;
    block_scan<MAX>(v, incl, excl, total);
    if (i < ntiles) tile_sums[i] = sop<MAX>(carry, excl);
    carry = sop<MAX>(carry, total);
  }
}

template <bool MAX, bool INCLUSIVE>
__global__ void __launch_bounds__(SC_THREADS) k_scan_apply(const int32_t *in, int32_t *out, long long n,
                                                           const int32_t *tile_sums) {
  const long long base = (long long)blockIdx.x * SC_TILE + (long long)threadIdx.x * SC_ITEMS;
  int v[SC_ITEMS];
  int acc = sid<MAX>();
#pragma unroll
  for (int i = 0; i < SC_ITEMS; ++i) {
    v[i] = base + i < n ? in[base + i] : sid<MAX>();
    acc = sop<MAX>(acc, v[i]);
  }
  int incl, excl, total;
  block_scan<MAX>(acc, incl, excl, total);
  int run = sop<MAX>(tile_sums[blockIdx.x], excl);
#pragma unroll
  for (int i = 0; i < SC_ITEMS; ++i) {
    if (base + i < n) {
      if (INCLUSIVE) {
        run = sop<MAX>(run, v[i]);
        out[base + i] = run;
      } else {
        out[base + i] = run;
        run = sop<MAX>(run, v[i]);
      }
    }
  }
}

int grid_for(long long n, int per_block) {
  long long g = (n + per_block - 1) / per_block;
  if (g > 152 * 16) g = 152 * 16;
  if (g < 1) g = 1;
  return (int)g;
}

template <bool MAX, bool INCLUSIVE>
cudaError_t device_scan(const int32_t *in, int32_t *out, long long n, int32_t *tile_sums,
                        cudaStream_t st, int *launches) {
  const long long tiles = (n + SC_TILE - 1) / SC_TILE;
  k_scan_reduce<MAX><<<(unsigned)tiles, SC_THREADS, 0, st>>>(in, n, tile_sums);
  k_scan_tiles<MAX><<<1, SC_THREADS, 0, st>>>(tile_sums, tiles);
  k_scan_apply<MAX, INCLUSIVE><<<(unsigned)tiles, SC_THREADS, 0, st>>>(in, out, n, tile_sums);
  *launches += 3;
  return cudaGetLastError();
}

int bits_of(unsigned long long x) {
  int b = 0;
  while (x) { ++b; x >>= 1; }
  return b;
}

}  // namespace

size_t sa_scratch_bytes(int64_t cap) {
  const long long c = cap > 0 ? cap : 1;
  const long long os_tiles = (c + OS_TILE - 1) / OS_TILE;
  const long long sc_tiles = (c + SC_TILE - 1) / SC_TILE;
  return (size_t)c * (8 + 8 + 4 + 4 + 4 + 4 + 4 + 4 + 4) + (size_t)sc_tiles * 4 + 8 * RADIX * 4 +
         (size_t)os_tiles * RADIX * 4 + 64;
}

cudaError_t sa_scratch_alloc(SaScratch *s, int64_t cap) {
  *s = SaScratch{};
  const long long c = cap > 0 ? cap : 1;
  s->cap = cap;
  const long long os_tiles = (c + OS_TILE - 1) / OS_TILE;
  const long long sc_tiles = (c + SC_TILE - 1) / SC_TILE;
  s->status_words = os_tiles * RADIX;
  cudaError_t e = cudaSuccess;
  auto al = [&](void **p, size_t bytes) {
    if (e == cudaSuccess) e = cudaMalloc(p, bytes);
  };
  al((void **)&s->keyA, c * 8);
  al((void **)&s->keyB, c * 8);
  al((void **)&s->valA, c * 4);
  al((void **)&s->valB, c * 4);
  al((void **)&s->rank, c * 4);
  al((void **)&s->act, c * 4);
  al((void **)&s->act2, c * 4);
  al((void **)&s->tmp, c * 4);
  al((void **)&s->head, c * 4);
  al((void **)&s->tile_sums, (sc_tiles + 1) * 4);
  al((void **)&s->hist, 8 * RADIX * 4);
  al((void **)&s->status, s->status_words * 4);
  al((void **)&s->counter, 64);
  if (e == cudaSuccess) e = cudaMallocHost((void **)&s->h_pinned, 64);
  if (e == cudaSuccess) e = cudaMallocHost((void **)&s->h_hist, 8 * RADIX * 4);
  if (e != cudaSuccess) sa_scratch_free(s);
  return e;
}

size_t sa_scratch_carve(SaScratch *s, unsigned char *base, size_t bytes, int64_t cap) {
  *s = SaScratch{};
  const long long c = cap > 0 ? cap : 1;
  const long long os_tiles = (c + OS_TILE - 1) / OS_TILE;
  const long long sc_tiles = (c + SC_TILE - 1) / SC_TILE;
  size_t off = 0;
  auto take = [&](size_t n) {
    unsigned char *p = base + off;
    off += (n + 255) & ~(size_t)255;
    return p;
  };
  s->cap = cap;
  s->status_words = os_tiles * RADIX;
  s->keyA = (uint64_t *)take(c * 8);
  s->keyB = (uint64_t *)take(c * 8);
  s->valA = (int32_t *)take(c * 4);
  s->valB = (int32_t *)take(c * 4);
  s->rank = (int32_t *)take(c * 4);
  s->act = (int32_t *)take(c * 4);
  s->act2 = (int32_t *)take(c * 4);
  s->tmp = (int32_t *)take(c * 4);
  s->head = (int32_t *)take(c * 4);
  s->tile_sums = (int32_t *)take((sc_tiles + 1) * 4);
  s->hist = (uint32_t *)take(8 * RADIX * 4);
  s->status = (uint32_t *)take(s->status_words * 4);
  s->counter = (uint32_t *)take(64);
  if (off > bytes) *s = SaScratch{};
  return off;
}

void sa_scratch_free(SaScratch *s) {
  cudaFree(s->keyA); cudaFree(s->keyB); cudaFree(s->valA); cudaFree(s->valB);
  cudaFree(s->rank); cudaFree(s->act); cudaFree(s->act2); cudaFree(s->tmp); cudaFree(s->head);
  cudaFree(s->tile_sums); cudaFree(s->hist); cudaFree(s->status); cudaFree(s->counter);
  if (s->h_pinned) cudaFreeHost(s->h_pinned);
  if (s->h_hist) cudaFreeHost(s->h_hist);
  *s = SaScratch{};
}

namespace {

struct Sorter {
  const SaScratch &s;
  cudaStream_t st;
  uint32_t *err;
  SaStats *stats;
  bool time_passes;
  int *launches;
  std::vector<cudaEvent_t> evs;

  // Sorts (keyA, valA)[0..n) by the low `bits` of the key.  Returns the
  // buffers holding the result through kres / vres.
  cudaError_t sort(long long n, int bits, uint64_t *&kres, int32_t *&vres) {
    uint64_t *kin = s.keyA, *kout = s.keyB;
    int32_t *vin = s.valA, *vout = s.valB;
    const int ndig = std::max(1, (bits + 7) / 8);
    cudaError_t e = cudaMemsetAsync(s.hist, 0, 8 * RADIX * 4, st);
    if (e != cudaSuccess) return e;
    k_hist<<<grid_for(n, 256 * 8), 256, 0, st>>>(kin, n, ndig, s.hist);
    ++*launches;
    e = cudaMemcpyAsync(s.h_hist, s.hist, (size_t)ndig * RADIX * 4, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    const long long tiles = (n + OS_TILE - 1) / OS_TILE;
    for (int d = 0; d < ndig; ++d) {
      bool trivial = false;
      for (int v = 0; v < RADIX; ++v)
        if ((long long)s.h_hist[d * RADIX + v] == n) trivial = true;
      if (trivial) continue;
      e = cudaMemsetAsync(s.status, 0, (size_t)tiles * RADIX * 4, st);
      if (e == cudaSuccess) e = cudaMemsetAsync(s.counter, 0, 4, st);
      if (e != cudaSuccess) return e;
      cudaEvent_t e0 = nullptr, e1 = nullptr;
      if (time_passes) {
        cudaEventCreate(&e0);
        cudaEventCreate(&e1);
        cudaEventRecord(e0, st);
      }
      k_onesweep<<<(unsigned)tiles, OS_THREADS, 0, st>>>(kin, vin, kout, vout, n, 8 * d,
                                                         s.hist + d * RADIX, s.status, s.counter, err);
      ++*launches;
      if (time_passes) {
        cudaEventRecord(e1, st);
        evs.push_back(e0);
        evs.push_back(e1);
      }
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      stats->passes++;
      stats->pass_elems += n;
      std::swap(kin, kout);
      std::swap(vin, vout);
    }
    kres = kin;
    vres = vin;
    return cudaSuccess;
  }
};

}  // namespace

int sa_build(const SaScratch &s, const int32_t *text, int64_t n, int32_t *sa, uint32_t *err,
             cudaStream_t st, SaStats *stats, bool time_passes, int *launches) {
  SaStats local;
  if (!stats) stats = &local;
  *stats = SaStats{};
  if (n <= 0) return 0;
  if (n > s.cap) return -1;
  if (n == 1) {
    if (cudaMemsetAsync(sa, 0, 4, st) != cudaSuccess) return -1;
    return 0;
  }
  Sorter so{s, st, err, stats, time_passes, launches, {}};
  cudaError_t e = cudaSuccess;
  const int G = grid_for(n, 256 * 4);
  // round 0: sort by the first token
  k_init0<<<G, 256, 0, st>>>(text, n, s.keyA, s.valA);
  ++*launches;
  uint64_t *kr;
  int32_t *vr;
  e = so.sort(n, 32, kr, vr);
  if (e != cudaSuccess) return -1;
  long long na = n;
  const int32_t *act = nullptr;
  int32_t *act_next = s.act;
  long long h = 1;
  const int round_bits = bits_of((unsigned long long)(n - 1) * (unsigned long long)(n + 1) +
                                 (unsigned long long)n);
  for (;;) {
    stats->rounds++;
    stats->sorted_elems += na;
    stats->model_bytes += na * (16 + 12);
    // write back, new heads, ranks, and the suffixes still unresolved
    int32_t *spare = (vr == s.valA) ? s.valB : s.valA;  // free int32 buffer of this round
    k_post<<<grid_for(na, 256 * 4), 256, 0, st>>>(act, na, kr, vr, sa, s.tmp, s.head);
    ++*launches;
    e = device_scan<true, true>(s.tmp, s.tmp, na, s.tile_sums, st, launches);
    if (e != cudaSuccess) return -1;
    k_rank<<<grid_for(na, 256 * 4), 256, 0, st>>>(na, vr, s.tmp, s.head, s.rank, spare);
    ++*launches;
    e = device_scan<false, false>(spare, spare, na, s.tile_sums, st, launches);
    if (e != cudaSuccess) return -1;
    k_compact<<<grid_for(na, 256 * 4), 256, 0, st>>>(na, act, s.head, spare, act_next,
                                                      (int32_t *)s.counter + 1);
    ++*launches;
    e = cudaMemcpyAsync(s.h_pinned, (int32_t *)s.counter + 1, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return -1;
    const long long next = s.h_pinned[0];
    if (next == 0) break;
    if (h >= n) break;  // cannot happen for a valid order; guards the loop
    // next round over the unresolved suffixes
    act = act_next;
    act_next = (act_next == s.act) ? s.act2 : s.act;
    na = next;
    k_keys<<<grid_for(na, 256 * 4), 256, 0, st>>>(act, na, sa, s.rank, h, n, s.keyA, s.valA);
    ++*launches;
    const int passes_before = stats->passes;
    e = so.sort(na, round_bits, kr, vr);
    if (e != cudaSuccess) return -1;
    stats->model_bytes += na * 24LL * (stats->passes - passes_before);
    h *= 2;
  }
  stats->model_bytes += 8LL * n;
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return -1;
  if (time_passes) {
    for (size_t i = 0; i + 1 < so.evs.size(); i += 2) {
      float ms = 0;
      cudaEventElapsedTime(&ms, so.evs[i], so.evs[i + 1]);
      stats->pass_ms += ms;
      cudaEventDestroy(so.evs[i]);
      cudaEventDestroy(so.evs[i + 1]);
    }
  }
  return 0;
}

}  // namespace sgd
