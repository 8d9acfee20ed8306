// C-ABI host layer: argument validation, workspace carving, kernel dispatch.
// Declarations and the contract of every entry point are in include/bnb_int8.h.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace bnb {

static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
static inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

struct Layout {
  size_t status, counters, colmask, O, sx, sxd, xcodes, xo, w16o, total;
  int64_t kpad, opad;
};

static Layout layout_of(int64_t T, int64_t N, int64_t K) {
  Layout L;
  L.kpad = (K + 63) / 64 * 64;
  size_t off = 0;
  L.status = off;
  off += 256;
  L.counters = off;
  off += 256;
  L.colmask = off;
  off += align_up((size_t)((K + 255) / 256) * 8 * 4, 256);
  L.O = off;
  off += align_up((size_t)(K + 64) * 4, 256);
  L.sx = off;
  off += align_up((size_t)T * 4, 256);
  L.sxd = off;
  off += align_up((size_t)T * 4, 256);
  L.xcodes = off;
  off += align_up((size_t)T * (size_t)K * 2, 256);
  L.xo = off;
  off += align_up((size_t)T * (size_t)L.kpad * 2, 256);
  L.opad = ((K / 16 > 0 ? K / 16 : 1) + 63) / 64 * 64;  // holds any sparse outlier set
  L.w16o = off;
  off += align_up((size_t)N * (size_t)L.opad * 2, 256);
  L.total = off;
  return L;
}

static constexpr size_t kWsSlack = 256;  // the carved layout starts at the next 256-byte boundary

static Workspace carve(void *ws, int64_t T, int64_t N, int64_t K) {
  const Layout L = layout_of(T, N, K);
  char *base = reinterpret_cast<char *>(align_up((uintptr_t)ws, 256));
  Workspace w;
  w.status = reinterpret_cast<int32_t *>(base + L.status);
  w.counters = reinterpret_cast<uint32_t *>(base + L.counters);
  w.colmask = reinterpret_cast<uint32_t *>(base + L.colmask);
  w.O = reinterpret_cast<int32_t *>(base + L.O);
  w.sx = reinterpret_cast<float *>(base + L.sx);
  w.sxd = reinterpret_cast<float *>(base + L.sxd);
  w.xcodes = base + L.xcodes;
  w.xo = reinterpret_cast<__half *>(base + L.xo);
  w.kpad = L.kpad;
  w.w16o = reinterpret_cast<__half *>(base + L.w16o);
  w.opad = L.opad;
  return w;
}

// Exact fp16 value of a bit pattern (host side).
static double half_bits_value(uint32_t h) {
  const int e = (h >> 10) & 0x1f, m = h & 0x3ff;
  if (e == 0) return std::ldexp((double)m, -24);
  if (e == 31) return INFINITY;
  return std::ldexp((double)(1024 + m), e - 25);
}

// Exact bf16 value of a bit pattern (host side): the binary32 with the same
// leading 16 bits.
static double bf16_bits_value(uint32_t h) {
  uint32_t u = (h & 0xffffu) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Smallest non-negative fp16 (bf16) bit pattern whose value is >= tau
// (0x7c00 / 0x7f80, the infinity pattern, when no finite value reaches tau).
// For finite x:  |x| >= tau  <=>  (bits(x) & 0x7fff) >= threshold_bits(tau).
static uint32_t threshold_bits(float tau, bool bf16) {
  uint32_t lo = 0, hi = bf16 ? 0x7f80 : 0x7c00;  // answer in [lo, hi]
  while (lo < hi) {
    const uint32_t mid = (lo + hi) / 2;
    if ((bf16 ? bf16_bits_value(mid) : half_bits_value(mid)) >= (double)tau)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo;
}

static int device_sms(int dev) {
  static std::atomic<int> cache[64];
  if (dev < 0 || dev >= 64) return kB300Sms;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    v = kB300Sms;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// BNB_OK if the current device is compute capability 10.3.
static bnb_status_t check_device(int *dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BNB_ERR_CUDA;
  static std::atomic<int> ok_cache[64];
  if (dev >= 0 && dev < 64 && ok_cache[dev].load(std::memory_order_relaxed) == 1) {
    *dev_out = dev;
    return BNB_OK;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return BNB_ERR_CUDA;
  if (major != 10 || minor != 3) return BNB_ERR_UNSUPPORTED;
  if (dev >= 0 && dev < 64) ok_cache[dev].store(1, std::memory_order_relaxed);
  *dev_out = dev;
  return BNB_OK;
}

static bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

// 1: decode (T <= 16, K <= kDecodeMaxK, N within what the resident decode
// CTAs hold in one wave); 2: tcgen05 GEMM (every other shape, decode-sized T
// included); 3: legacy mma GEMM (only when a call's options ask for it).
static int choose_path(int64_t T, int64_t N, int64_t K, int dev, uint32_t opts = 0) {
  if (T <= 16 && !(opts & BNB_OPT_GEMM) && K <= kDecodeMaxK && N <= decode_max_n(dev, T, K)) return 1;
  return (opts & BNB_OPT_LEGACY_MMA) ? 3 : 2;
}

// The argument checks of bnb_int8_linear (nothing is enqueued).  W16 may be
// null only where the caller keeps the int8 weight alone (w16_optional).
static bnb_status_t linear_check(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                 const float *Wscale, const void *W16, int64_t N, float tau,
                                 const void *Y, const void *workspace, size_t workspace_bytes,
                                 bool w16_optional = false) {
  if (!X || !Wq || !Wscale || !Y || !workspace) return BNB_ERR_INVALID_ARG;
  if (!W16 && !w16_optional) return BNB_ERR_INVALID_ARG;
  if (T <= 0 || N <= 0 || K <= 0) return BNB_ERR_INVALID_ARG;
  if (std::isnan(tau) || tau < 0.0f) return BNB_ERR_INVALID_ARG;
  if (T > BNB_MAX_T || N > BNB_MAX_N || K > BNB_MAX_K) return BNB_ERR_UNSUPPORTED;
  if (workspace_bytes < bnb_int8_linear_workspace_bytes(T, N, K)) return BNB_ERR_INVALID_ARG;
  if (K % 16 != 0) return BNB_ERR_UNSUPPORTED;
  if (!aligned16(X) || !aligned16(Wq) || !aligned16(Wscale) || (W16 && !aligned16(W16)) ||
      !aligned16(Y) || !aligned16(workspace))
    return BNB_ERR_UNSUPPORTED;
  const size_t ybytes = (size_t)T * (size_t)N * 2;
  if (overlaps(Y, ybytes, X, (size_t)T * K * 2) ||
      (W16 && overlaps(Y, ybytes, W16, (size_t)N * K * 2)) ||
      overlaps(Y, ybytes, Wq, (size_t)N * K) || overlaps(Y, ybytes, workspace, workspace_bytes))
    return BNB_ERR_INVALID_ARG;
  return BNB_OK;
}

static bnb_status_t linear_impl(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                const float *Wscale, const void *W16, const void *bias,
                                int64_t N, float tau, bool bf16, void *Y, void *workspace,
                                size_t workspace_bytes,
                                void *stream_v, int8_t *dbg_xq, float *dbg_sx,
                                int32_t *dbg_O, int32_t *dbg_nO, int32_t *dbg_acc,
                                uint32_t opts = 0) {
  // (the entry points check W16 themselves: null means the int8 weight alone)
  bnb_status_t chk = linear_check(X, T, K, Wq, Wscale, W16, N, tau, Y, workspace, workspace_bytes,
                                  /*w16_optional=*/true);
  if (chk != BNB_OK) return chk;
  if ((dbg_xq && !aligned16(dbg_xq)) || (dbg_acc && !aligned16(dbg_acc)))
    return BNB_ERR_UNSUPPORTED;
  if (bias && !aligned16(bias)) return BNB_ERR_UNSUPPORTED;
  if (bias && overlaps(Y, (size_t)T * (size_t)N * 2, bias, (size_t)N * 2)) return BNB_ERR_INVALID_ARG;
  int dev = 0;
  bnb_status_t st = check_device(&dev);
  if (st != BNB_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  const Workspace ws = carve(workspace, T, N, K);
  const int path = choose_path(T, N, K, dev, opts);
  const uint32_t thr = threshold_bits(tau, bf16);
  cudaError_t e;
  if (path == 1) {
    // decode: no memset, the kernel clears the status word itself
    if (!(opts & BNB_OPT_ACT_ONLY)) {
      e = launch_decode(X, T, K, thr, Wq, Wscale, W16, bias, N, bf16, Y, ws, dbg_xq, dbg_acc,
                        opts, stream);
      if (e != cudaSuccess) return BNB_ERR_CUDA;
    }
  } else {
    if (!(opts & BNB_OPT_MAIN_ONLY)) {
      // status word, counters and the outlier column mask are contiguous and
      // zeroed by every call with one memset
      const size_t zero_bytes = 512 + (size_t)((K + 255) / 256) * 8 * 4;
      if (cudaMemsetAsync(ws.status, 0, zero_bytes, stream) != cudaSuccess) return BNB_ERR_CUDA;
      note_launch();
      // the tcgen05 GEMM reads fp16 integer codes, the mma GEMM int8 codes
      // (for the tcgen05 GEMM the same launch compacts W16 at a sparse outlier set)
      e = launch_act_pass(X, T, K, thr, ws, /*code_mode=*/path == 2 ? 1 : 0, /*with_xo=*/true,
                          W16, Wq, N, bf16, dbg_xq, device_sms(dev), stream,
                          /*pdl=*/!(opts & BNB_OPT_NO_PDL));
      if (e != cudaSuccess) return BNB_ERR_CUDA;
    }
    if (!(opts & BNB_OPT_ACT_ONLY)) {
      if (path == 2)
        e = launch_gemm_tc(T, K, Wq, Wscale, W16, bias, N, bf16, Y, ws, dbg_acc, device_sms(dev),
                           opts, stream);
      else
        e = launch_gemm_mma(T, K, Wq, Wscale, W16, bias, N, bf16, Y, ws, dbg_acc, stream);
      if (e != cudaSuccess) return BNB_ERR_CUDA;
    }
  }
  if (dbg_sx && cudaMemcpyAsync(dbg_sx, ws.sx, (size_t)T * 4, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return BNB_ERR_CUDA;
  if (dbg_O && cudaMemcpyAsync(dbg_O, ws.O, (size_t)K * 4, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return BNB_ERR_CUDA;
  if (dbg_nO && cudaMemcpyAsync(dbg_nO, ws.counters + 1, 4, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return BNB_ERR_CUDA;
  return BNB_OK;
}

}  // namespace bnb

using namespace bnb;

extern "C" {

size_t bnb_int8_linear_workspace_bytes(int64_t T, int64_t N, int64_t K) {
  if (T <= 0 || N <= 0 || K <= 0 || T > BNB_MAX_T || N > BNB_MAX_N || K > BNB_MAX_K) return 0;
  return layout_of(T, N, K).total + kWsSlack;
}

static bnb_status_t quantize_weight_impl(const void *W16, int64_t N, int64_t K, bool bf16,
                                         int8_t *Wq, float *Wscale, void *stream) {
  if (!W16 || !Wq || !Wscale) return BNB_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0) return BNB_ERR_INVALID_ARG;
  if (N > BNB_MAX_N || K > BNB_MAX_K) return BNB_ERR_UNSUPPORTED;
  if (K % 16 != 0 || !aligned16(W16) || !aligned16(Wq) || !aligned16(Wscale))
    return BNB_ERR_UNSUPPORTED;
  if (overlaps(Wq, (size_t)N * K, W16, (size_t)N * K * 2)) return BNB_ERR_INVALID_ARG;
  int dev = 0;
  bnb_status_t st = check_device(&dev);
  if (st != BNB_OK) return st;
  cudaError_t e =
      launch_quantize_weight(W16, N, K, bf16, Wq, Wscale, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BNB_OK : BNB_ERR_CUDA;
}

bnb_status_t bnb_int8_quantize_weight(const void *W16, int64_t N, int64_t K, int8_t *Wq,
                                      float *Wscale, void *stream) {
  return quantize_weight_impl(W16, N, K, false, Wq, Wscale, stream);
}

bnb_status_t bnb_int8_quantize_weight_ex(const void *W, int64_t N, int64_t K, int dtype,
                                         int8_t *Wq, float *Wscale, void *stream) {
  if (dtype != BNB_DTYPE_FP16 && dtype != BNB_DTYPE_BF16) return BNB_ERR_INVALID_ARG;
  return quantize_weight_impl(W, N, K, dtype == BNB_DTYPE_BF16, Wq, Wscale, stream);
}

static bool blockwise_size_ok(int64_t block) {
  return block >= 64 && block <= 2048 && (block & (block - 1)) == 0;
}

bnb_status_t bnb_int8_quantize_blockwise(const float *x, int64_t n, int64_t block, int8_t *codes,
                                         float *absmax, void *stream) {
  if (!x || !codes || !absmax || n <= 0) return BNB_ERR_INVALID_ARG;
  if (!blockwise_size_ok(block) || n > BNB_MAX_BLOCKWISE_N) return BNB_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(absmax)) return BNB_ERR_UNSUPPORTED;
  const size_t nb = (size_t)((n + block - 1) / block);
  if (overlaps(codes, (size_t)n, x, (size_t)n * 4) || overlaps(absmax, nb * 4, x, (size_t)n * 4) ||
      overlaps(absmax, nb * 4, codes, (size_t)n))
    return BNB_ERR_INVALID_ARG;
  int dev = 0;
  bnb_status_t st = check_device(&dev);
  if (st != BNB_OK) return st;
  const cudaError_t e = launch_quantize_blockwise(x, n, (int)block, codes, absmax, device_sms(dev),
                                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BNB_OK : BNB_ERR_CUDA;
}

bnb_status_t bnb_int8_dequantize_blockwise(const int8_t *codes, const float *absmax, int64_t n,
                                           int64_t block, float *y, void *stream) {
  if (!codes || !absmax || !y || n <= 0) return BNB_ERR_INVALID_ARG;
  if (!blockwise_size_ok(block) || n > BNB_MAX_BLOCKWISE_N) return BNB_ERR_UNSUPPORTED;
  if (!aligned16(codes) || !aligned16(absmax) || !aligned16(y)) return BNB_ERR_UNSUPPORTED;
  const size_t nb = (size_t)((n + block - 1) / block);
  if (overlaps(y, (size_t)n * 4, codes, (size_t)n) || overlaps(y, (size_t)n * 4, absmax, nb * 4))
    return BNB_ERR_INVALID_ARG;
  int dev = 0;
  bnb_status_t st = check_device(&dev);
  if (st != BNB_OK) return st;
  const cudaError_t e = launch_dequantize_blockwise(codes, absmax, n, (int)block, y,
                                                    device_sms(dev),
                                                    reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BNB_OK : BNB_ERR_CUDA;
}

bnb_status_t bnb_int8_linear(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                             const float *Wscale, const void *W16, int64_t N, float tau,
                             void *Y, void *workspace, size_t workspace_bytes, void *stream) {
  if (!W16) return BNB_ERR_INVALID_ARG;
  return linear_impl(X, T, K, Wq, Wscale, W16, nullptr, N, tau, false, Y, workspace, workspace_bytes,
                     stream, nullptr, nullptr, nullptr, nullptr, nullptr);
}

bnb_status_t bnb_int8_linear_bias(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                  const float *Wscale, const void *W16, const void *bias,
                                  int64_t N, float tau, void *Y, void *workspace,
                                  size_t workspace_bytes, void *stream) {
  if (!W16) return BNB_ERR_INVALID_ARG;
  return linear_impl(X, T, K, Wq, Wscale, W16, bias, N, tau, false, Y, workspace, workspace_bytes,
                     stream, nullptr, nullptr, nullptr, nullptr, nullptr);
}

bnb_status_t bnb_int8_linear_ex(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                const float *Wscale, const void *W16, const void *bias, int64_t N,
                                float tau, int dtype, void *Y, void *workspace,
                                size_t workspace_bytes, void *stream) {
  if (dtype != BNB_DTYPE_FP16 && dtype != BNB_DTYPE_BF16) return BNB_ERR_INVALID_ARG;
  return linear_impl(X, T, K, Wq, Wscale, W16, bias, N, tau, dtype == BNB_DTYPE_BF16, Y,
                     workspace, workspace_bytes, stream, nullptr, nullptr, nullptr, nullptr,
                     nullptr);
}

bnb_status_t bnb_int8_linear_wq_only(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                     const float *Wscale, const void *bias, int64_t N,
                                     float tau, void *Y, void *workspace,
                                     size_t workspace_bytes, void *stream) {
  return linear_impl(X, T, K, Wq, Wscale, nullptr, bias, N, tau, false, Y, workspace, workspace_bytes,
                     stream, nullptr, nullptr, nullptr, nullptr, nullptr);
}

static bnb_status_t from_host_impl(const void *X_host, int64_t T, int64_t K, const int8_t *Wq,
                                   const float *Wscale, const void *W16, const void *bias,
                                   int64_t N, float tau, bool bf16, void *Y_host, void *X_dev,
                                   void *Y_dev, void *workspace, size_t workspace_bytes,
                                   void *stream) {
  if (!X_host || !Y_host || !X_dev || !Y_dev) return BNB_ERR_INVALID_ARG;
  if (T <= 0 || K <= 0 || N <= 0) return BNB_ERR_INVALID_ARG;
  const size_t xbytes = (size_t)T * (size_t)K * 2, ybytes = (size_t)T * (size_t)N * 2;
  if (overlaps(X_dev, xbytes, Y_dev, ybytes)) return BNB_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the layer's own argument checks run before anything is enqueued
  bnb_status_t r = linear_check(X_dev, T, K, Wq, Wscale, W16, N, tau, Y_dev, workspace,
                                workspace_bytes, /*w16_optional=*/true);
  if (r != BNB_OK) return r;
  if (bias && !aligned16(bias)) return BNB_ERR_UNSUPPORTED;
  if (bias && overlaps(Y_dev, ybytes, bias, (size_t)N * 2)) return BNB_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(X_dev, X_host, xbytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return BNB_ERR_CUDA;
  r = linear_impl(X_dev, T, K, Wq, Wscale, W16, bias, N, tau, bf16, Y_dev, workspace,
                  workspace_bytes, stream, nullptr, nullptr, nullptr, nullptr, nullptr);
  if (r != BNB_OK) return r;
  if (cudaMemcpyAsync(Y_host, Y_dev, ybytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return BNB_ERR_CUDA;
  return BNB_OK;
}

bnb_status_t bnb_int8_linear_from_host(const void *X_host, int64_t T, int64_t K,
                                       const int8_t *Wq, const float *Wscale, const void *W16,
                                       const void *bias, int64_t N, float tau, void *Y_host,
                                       void *X_dev, void *Y_dev, void *workspace,
                                       size_t workspace_bytes, void *stream) {
  return from_host_impl(X_host, T, K, Wq, Wscale, W16, bias, N, tau, false, Y_host, X_dev, Y_dev,
                        workspace, workspace_bytes, stream);
}

bnb_status_t bnb_int8_linear_from_host_ex(const void *X_host, int64_t T, int64_t K,
                                          const int8_t *Wq, const float *Wscale, const void *W16,
                                          const void *bias, int64_t N, float tau, int dtype,
                                          void *Y_host, void *X_dev, void *Y_dev,
                                          void *workspace, size_t workspace_bytes,
                                          void *stream) {
  if (dtype != BNB_DTYPE_FP16 && dtype != BNB_DTYPE_BF16) return BNB_ERR_INVALID_ARG;
  return from_host_impl(X_host, T, K, Wq, Wscale, W16, bias, N, tau, dtype == BNB_DTYPE_BF16,
                        Y_host, X_dev, Y_dev, workspace, workspace_bytes, stream);
}

bnb_status_t bnb_int8_linear_debug(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                   const float *Wscale, const void *W16, int64_t N, float tau,
                                   void *Y, void *workspace, size_t workspace_bytes,
                                   void *stream, int8_t *Xq, float *Xscale,
                                   int32_t *outlier_idx, int32_t *n_outliers, int32_t *acc) {
  if (!W16) return BNB_ERR_INVALID_ARG;
  return linear_impl(X, T, K, Wq, Wscale, W16, nullptr, N, tau, false, Y, workspace, workspace_bytes,
                     stream, Xq, Xscale, outlier_idx, n_outliers, acc);
}

bnb_status_t bnb_int8_linear_debug_ex(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                      const float *Wscale, const void *W16, const void *bias,
                                      int64_t N, float tau, int dtype, void *Y, void *workspace,
                                      size_t workspace_bytes, void *stream, int8_t *Xq,
                                      float *Xscale, int32_t *outlier_idx, int32_t *n_outliers,
                                      int32_t *acc) {
  if (dtype != BNB_DTYPE_FP16 && dtype != BNB_DTYPE_BF16) return BNB_ERR_INVALID_ARG;
  return linear_impl(X, T, K, Wq, Wscale, W16, bias, N, tau, dtype == BNB_DTYPE_BF16, Y,
                     workspace, workspace_bytes, stream, Xq, Xscale, outlier_idx, n_outliers, acc);
}

bnb_status_t bnb_int8_linear_opts(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                  const float *Wscale, const void *W16, const void *bias,
                                  int64_t N, float tau, int dtype, void *Y, void *workspace,
                                  size_t workspace_bytes, void *stream, int8_t *Xq,
                                  float *Xscale, int32_t *outlier_idx, int32_t *n_outliers,
                                  int32_t *acc, uint32_t opts) {
  if (dtype != BNB_DTYPE_FP16 && dtype != BNB_DTYPE_BF16) return BNB_ERR_INVALID_ARG;
  constexpr uint32_t kKnown = BNB_OPT_MAIN_ONLY | BNB_OPT_ACT_ONLY | BNB_OPT_NO_PDL |
                              BNB_OPT_LEGACY_MMA | BNB_OPT_FORCE_TIMEOUT | BNB_OPT_SINGLE_CTA |
                              BNB_OPT_GEMM | BNB_OPT_CLUSTER(0xff);
  if (opts & ~kKnown) return BNB_ERR_INVALID_ARG;
  const uint32_t c = (opts >> 8) & 0xffu;
  if (c != 0 && c != 1 && c != 4 && c != 8 && c != 16) return BNB_ERR_INVALID_ARG;
  if ((opts & BNB_OPT_MAIN_ONLY) && (opts & BNB_OPT_ACT_ONLY)) return BNB_ERR_INVALID_ARG;
  return linear_impl(X, T, K, Wq, Wscale, W16, bias, N, tau, dtype == BNB_DTYPE_BF16, Y,
                     workspace, workspace_bytes, stream, Xq, Xscale, outlier_idx, n_outliers, acc,
                     opts);
}

bnb_status_t bnb_last_device_status(const void *workspace, void *stream, int32_t *out) {
  if (!workspace || !out) return BNB_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BNB_ERR_CUDA;
  int32_t *status = reinterpret_cast<int32_t *>(align_up((uintptr_t)workspace, 256));
  int32_t v = 0;
  if (cudaMemcpy(&v, status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return BNB_ERR_CUDA;
  if (cudaMemset(status, 0, 4) != cudaSuccess) return BNB_ERR_CUDA;
  *out = v;
  return BNB_OK;
}

const char *bnb_status_string(bnb_status_t s) {
  switch (s) {
    case BNB_OK: return "BNB_OK";
    case BNB_ERR_INVALID_ARG: return "BNB_ERR_INVALID_ARG";
    case BNB_ERR_UNSUPPORTED: return "BNB_ERR_UNSUPPORTED";
    case BNB_ERR_CUDA: return "BNB_ERR_CUDA";
    case BNB_ERR_TIMEOUT: return "BNB_ERR_TIMEOUT";
  }
  return "BNB_ERR_UNKNOWN";
}

uint64_t bnb_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int bnb_int8_linear_path(int64_t T, int64_t N, int64_t K) {
  if (T <= 0 || N <= 0 || K <= 0) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  return choose_path(T, N, K, dev);
}

int bnb_int8_decode_cluster(int64_t T, int64_t N, int64_t K) {
  if (T <= 0 || N <= 0 || K <= 0) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  return choose_path(T, N, K, dev) == 1 ? decode_cluster_size(dev, T, N, K) : 0;
}

}  // extern "C"
