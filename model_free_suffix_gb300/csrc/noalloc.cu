// noalloc.cu -- suffix array of a caller text with no allocation at all.
//
// Some callers cannot call cudaMalloc at the moment they need a suffix array:
// a serving process whose own caching allocator has reserved the device
// memory up front and forbids further driver allocations, code that runs
// inside another framework's memory budget, or a caller that must not risk
// an out-of-memory failure (or the implicit device synchronisation of
// cudaMalloc / cudaFree) in the middle of its work.  For them this file
// keeps the sort's working memory in one fixed device array that exists as
// long as the library is loaded: the caller passes only the text and the
// output buffer, and the call performs no device or pinned-host allocation.
//
// The price: the array is sized for SGD_NOALLOC_MAX_TOKENS tokens and every
// GPU that loads the library holds it until the process exits; longer texts
// are rejected with SGD_ETOOLARGE.
#include <mutex>

#include "sgd_internal.h"

namespace sgd {
namespace {

constexpr long long kMax = SGD_NOALLOC_MAX_TOKENS;
constexpr long long kTiles = (kMax + 2047) / 2048 + 1;
// bytes of the pieces laid out by sa_scratch_carve for kMax elements, each
// rounded up to 256, plus the error word; checked against the carve per call
constexpr size_t kBytes = 2 * kMax * 8 + 5 * kMax * 4 + kTiles * 256 * 8 + kTiles * 8 +
                          8 * 256 * 4 + 1024 + 16 * 256;

// The fixed working memory.  From host code its name is only a stand-in:
// the device address is obtained with cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kBytes];

std::mutex g_mu;                 // calls share the array: one at a time
unsigned char *g_base[64] = {};  // resolved address per device
uint32_t g_h_hist[8 * 256];      // host words the sort reads back (pageable)
int32_t g_h_count[16];

}  // namespace
}  // namespace sgd

using namespace sgd;

extern "C" int sgd_suffix_array_noalloc(const int32_t *text, int64_t n, int32_t *sa, void *stream) {
  if (n < 0 || (n > 0 && (text == nullptr || sa == nullptr))) return SGD_EINVAL;
  if (n > kMax) return SGD_ETOOLARGE;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGD_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array's address is resolved for the current device; a stream of
  // another device would run the sort against that device's memory
  int sdev = -1;
  if (cudaStreamGetDevice(st, &sdev) != cudaSuccess) {
    cudaGetLastError();
    return SGD_EINVAL;
  }
  if (sdev != dev) return SGD_EINVAL;
  if (g_base[dev] == nullptr) {
    // first call on this device (with it current): resolve the array's address
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SGD_ECUDA;
    }
    g_base[dev] = static_cast<unsigned char *>(p);
  }
  if (n == 0) return SGD_OK;
  SaScratch s;
  const size_t used = sa_scratch_carve(&s, g_base[dev], kBytes, kMax);
  if (s.keyA == nullptr || used + 4 > kBytes) return SGD_ECUDA;
  s.h_pinned = g_h_count;
  s.h_hist = g_h_hist;
  uint32_t *err = reinterpret_cast<uint32_t *>(g_base[dev] + used);
  // the array keeps the previous call's contents: the error word must start
  // at zero (the sort clears its own histograms and look-back words per pass)
  if (cudaMemsetAsync(err, 0, 4, st) != cudaSuccess) return SGD_ECUDA;
  int launches = 0;
  const int r = sa_build(s, text, n, sa, err, st, nullptr, false, &launches);
  if (r < 0) return SGD_ECUDA;
  uint32_t h_err = 0;
  if (cudaMemcpyAsync(&h_err, err, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return SGD_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SGD_ECUDA;
  return (r != 0 || h_err != 0) ? SGD_EBUILD : SGD_OK;
}
