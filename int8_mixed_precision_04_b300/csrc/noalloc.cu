// bnb_int8_linear_noalloc: the decomposition linear for callers that cannot
// allocate device memory (declaration and contract in include/bnb_int8.h).
//
// The workspace of bnb_int8_linear is replaced by one file-scope device array,
// g_scratch, of BNB_NOALLOC_SCRATCH_BYTES.  The array is part of this
// library's device image: every GPU that loads the library holds it until the
// process exits, and nothing here calls cudaMalloc, cudaFree or any other
// allocating routine.
//
// In host code the name g_scratch is only a host-side stand-in for the
// array, not a device address.  The device address is looked up once per
// device, with that device current, by cudaGetSymbolAddress, and cached; the
// first call on a device does this set-up.  The cache is valid for the life
// of the device's primary context: a cudaDeviceReset invalidates it (the
// header tells callers not to use this entry point after one).
#include <atomic>

#include "common.cuh"

namespace bnb {
namespace {

static __device__ __align__(256) unsigned char g_scratch[BNB_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxCachedDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxCachedDevices];

// Device address of g_scratch on the current device (nullptr on failure).
void *scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < kMaxCachedDevices) {
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p) return p;
  }
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return nullptr;
  if (dev >= 0 && dev < kMaxCachedDevices) g_scratch_addr[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace
}  // namespace bnb

extern "C" bnb_status_t bnb_int8_linear_noalloc(const void *X, int64_t T, int64_t K,
                                                const int8_t *Wq, const float *Wscale,
                                                const void *W16, int64_t N, float tau, void *Y,
                                                void *stream) {
  if (!X || !Wq || !Wscale || !W16 || !Y) return BNB_ERR_INVALID_ARG;
  if (T <= 0 || N <= 0 || K <= 0) return BNB_ERR_INVALID_ARG;
  const size_t need = bnb_int8_linear_workspace_bytes(T, N, K);
  if (need == 0 || need > (size_t)BNB_NOALLOC_SCRATCH_BYTES) return BNB_ERR_UNSUPPORTED;
  void *scratch = bnb::scratch_on_current_device();
  if (!scratch) return BNB_ERR_CUDA;
  // bnb_int8_linear clears, on the device, every part of the workspace that
  // must start at zero (status word, counters, outlier mask) on each call.
  return bnb_int8_linear(X, T, K, Wq, Wscale, W16, N, tau, Y, scratch,
                         (size_t)BNB_NOALLOC_SCRATCH_BYTES, stream);
}
