// Shared device helpers for the int8 decomposition linear (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/bnb_int8.h"

namespace bnb {

// Device status word values (first int32 of the workspace).
constexpr int32_t kDevOk = 0;
constexpr int32_t kDevTimeout = BNB_ERR_TIMEOUT;

// Number of SMs of a B300 (2 dies x 74); grids are sized from the live
// device attribute, this is only a default for host-side heuristics.
constexpr int kB300Sms = 148;

// Workspace layout, carved identically by the host for every call.
struct Workspace {
  int32_t *status;     // [4]  device status word + spare
  uint32_t *counters;  // [4]  block-completion counter, |O| (counters[1])
  uint32_t *colmask;   // [ceil(K/32)] outlier column bitmask
  int32_t *O;          // [K + 64] outlier column list, ascending
  float *sx;           // [T] row scales
  void *xcodes;        // [T x K] codes: int8 (decode) or fp16 integers (GEMM)
  __half *xo;          // [T x kpad] compacted fp16 outlier block
  int64_t kpad;        // pitch of xo in elements (K rounded up to 64)
};

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

// |x| as fp16 bits, for exact threshold and absmax work on bit patterns:
// for finite fp16, |a| < |b|  <=>  (bits_a & 0x7fff) < (bits_b & 0x7fff).
__device__ __forceinline__ uint32_t abs_bits_lo(uint32_t w) { return w & 0x7fffu; }
__device__ __forceinline__ uint32_t abs_bits_hi(uint32_t w) { return (w >> 16) & 0x7fffu; }

// Exact fp16 bits -> float.
__device__ __forceinline__ float h2f_bits(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)h));
}

// Vector-wise int8 code of x against absmax a: rint(fl32(127 x) / a), ties to
// even; 0 when a == 0.  127*x is exact for fp16 x; the division is the IEEE
// round-to-nearest fp32 division.
__device__ __forceinline__ int code_of(float x, float a) {
  if (a == 0.0f) return 0;
  return __float2int_rn(__fdiv_rn(127.0f * x, a));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

}  // namespace bnb
