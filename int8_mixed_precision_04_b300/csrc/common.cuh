// Shared device helpers for the int8 decomposition linear (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "bnb_int8.h"

namespace bnb {

// Device status word values (first int32 of the workspace).
constexpr int32_t kDevOk = 0;
constexpr int32_t kDevTimeout = BNB_ERR_TIMEOUT;

// Number of SMs of a B300 (2 dies x 74); grids are sized from the live
// device attribute, this is only a default for host-side heuristics.
constexpr int kB300Sms = 148;

// Largest K of the decode path: 32 weight rows and 16 code rows of K + 64
// bytes plus the outlier list fit in 227 KB, and the activation pass gives
// each of 16 warps x 32 lanes one 8-column vector.
constexpr int64_t kDecodeMaxK = 4096;

// Largest T of the GEMM's 32-token tile (decode-sized calls the decode kernel
// does not hold); larger T take the 256-token tile.
constexpr int64_t kGemmSmallT = 32;

// The fp16 outlier block of the GEMM path is dense (X masked to the outlier
// columns over all K, multiplied as one dense fp16 GEMM against W16 tiles)
// when more than 1/16 of the columns are outliers; otherwise it is
// compacted, against W16's outlier columns compacted once per call.  A
// compacted column costs one scattered W16 sector per output channel, a
// dense one a fraction of a tensor-core stage: they break even near K/8.
__host__ __device__ __forceinline__ bool outlier_block_dense(int64_t nO, int64_t K) {
  return nO * 16 > K;
}

// Workspace layout, carved identically by the host for every call.
struct Workspace {
  int32_t *status;     // [4]  device status word + spare
  uint32_t *counters;  // [4]  block-completion counter, |O| (counters[1])
  uint32_t *colmask;   // [8 * ceil(K/256)] outlier column bitmask
  int32_t *O;          // [K + 64] outlier column list, ascending
  float *sx;           // [T] row scales
  float *sxd;          // [T] row scales / 127 (GEMM epilogue)
  void *xcodes;        // [T x K] codes: int8 (decode) or fp16 integers (GEMM)
  __half *xo;          // [T x kpad] 16-bit outlier block in X's format (compacted, or masked X when dense)
  int64_t kpad;        // pitch of xo in elements (K rounded up to 64)
  __half *w16o;        // [N x opad] W16 (or Wq as 16-bit integers) at the outlier columns, X's format
  int64_t opad;        // pitch of w16o in elements: floor(K / 16) rounded up to 64
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

// Vector-wise int8 code of x against absmax a > 0: the integer nearest to
// v = 127 x / a, ties to even (which is what rint(fl32(127 x) / a) gives,
// since a single fp32 rounding of that quotient never crosses or creates a
// half-integer).  Division-free and exact:
//   p = x * r with r ~ 127/a is within 127 * 2^-23 of v, so f = floor(p) and
//   the half-integer c = f + 0.5 bracket v's rounding decision;
//   fma(c, a, -127 x) rounds c*a - 127x once, so its SIGN is exact and equals
//   sign(c - v): negative -> round up, positive -> down, zero -> tie -> even.
// 127 x is exact in fp32 for fp16 x.  Requires |x| <= a, a > 0 finite.
__device__ __forceinline__ int code_exact(float x, float a, float r) {
  const float p = x * r;
  const float f = floorf(p);
  const float s = fmaf(f + 0.5f, a, -127.0f * x);
  int q = (int)f;
  if (s < 0.0f)
    q += 1;
  else if (s == 0.0f)
    q += q & 1;
  return q;
}

// 127 / a for the code rule above (0 when a == 0, in which case every code
// is 0 and code_exact is not used).
__device__ __forceinline__ float code_recip(float a) { return a > 0.0f ? 127.0f / a : 0.0f; }

// The same code as code_exact, from ALU operations only (no rounding or
// float-to-integer conversion instructions), returned as q mod 256 (the
// int8 code's byte):
//   M = 1.5 * 2^23 has unit spacing, so (p + M) - M is p rounded to an
//   integer and one comparison turns it into f = floor(p) (any f within a
//   few ulp of v's floor serves, since the fma below decides exactly);
//   f + M is exact for |f| < 2^22 with bit pattern bits(M) + f, whose low
//   byte is f mod 256 (bits(M) ends in a zero byte).
// Requires |x| <= a, a > 0 finite, or x = a = 0 (which gives 0).
__device__ __forceinline__ uint32_t code_byte(float x, float a, float r) {
  constexpr float kM = 12582912.0f;
  const float p = x * r;
  const float rn = (p + kM) - kM;
  const float f = rn > p ? rn - 1.0f : rn;
  const float s = fmaf(f + 0.5f, a, -127.0f * x);
  const uint32_t fb = __float_as_uint(f + kM);
  return fb + (s < 0.0f ? 1u : (s == 0.0f ? (fb & 1u) : 0u));
}

// The same code byte, from the product p = x * r first.  r = fl32(127 / a)
// and p = fl32(x r) put p within |v| (2^-23 + 2^-48) < 2^-16 of v = 127 x / a
// (|v| <= 127).  So when p lies more than 2^-15 from every half-integer, v
// rounds like p and is no tie: the code is rint(p), one magic-number add
// (ties to even) whose low byte is the code.  Otherwise (about one value in
// 2^14) code_byte decides exactly.  Requires what code_byte requires.
__device__ __forceinline__ uint32_t code_byte_fast(float x, float a, float r) {
  constexpr float kM = 12582912.0f;
  const float p = x * r;
  const float t = p + kM;          // M + rint(p), exact for |p| < 2^22
  const float e = p - (t - kM);    // p - rint(p), exact
  if (fabsf(e) < 0.5f - 0x1p-15f) return __float_as_uint(t);
  return code_byte(x, a, r);
}

__device__ __forceinline__ int code_of(float x, float a, float r) {
  return a > 0.0f ? code_exact(x, a, r) : 0;
}

// ---- the 16-bit element format of X, W16, the bias and Y ----
// kBf false: fp16; true: bf16 (1 sign, 8 exponent, 7 fraction bits).  For
// both, |a| < |b| <=> (bits_a & 0x7fff) < (bits_b & 0x7fff) on finite values,
// so thresholds and absmax work on bit patterns alike.
template <bool kBf>
__device__ __forceinline__ float e2f(uint32_t b) {  // low 16 bits -> float, exact
  if constexpr (kBf)
    return __uint_as_float(b << 16);
  else
    return h2f_bits(b);
}
template <bool kBf>
__device__ __forceinline__ uint16_t f2e(float v) {  // nearest-even
  if constexpr (kBf)
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  else
    return __half_as_ushort(__float2half_rn(v));
}
template <bool kBf>
__device__ __forceinline__ uint32_t f2e2(float lo, float hi) {  // a packed pair, nearest-even
  if constexpr (kBf) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
  } else {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
  }
}

// The code rule of one row (absmax a).  bf16 spans 2^-133 .. 2^128, where
// 127 x and 127 / a leave fp32's range, so for bf16 x and a are first scaled
// by one power of two 2^(1-e) (a = f 2^e, f in [0.5, 1)), applied as two
// normal factors so that every product is exact: the scaled a lies in
// [1, 2), and the code 127 x / a is unchanged.  A value whose scaled form
// underflows codes to 0 either way.
template <bool kBf>
struct RowCode {
  float a, r, s1, s2;
  RowCode() = default;
  __device__ __forceinline__ explicit RowCode(float absmax) {
    s1 = s2 = 1.0f;
    if (kBf && absmax > 0.0f) {
      const uint32_t b = __float_as_uint(absmax);
      const int E = (int)((b >> 23) & 0xffu);
      const int e = E ? E - 126 : 32 - (int)__clz(b & 0x7fffffu) - 149;
      const int k = 1 - e, k1 = k / 2, k2 = k - k1;  // each in [-64, 75]
      s1 = __uint_as_float((uint32_t)(k1 + 127) << 23);
      s2 = __uint_as_float((uint32_t)(k2 + 127) << 23);
    }
    a = kBf ? (absmax * s1) * s2 : absmax;
    r = code_recip(a);
  }
  // the code byte of x (|x| <= absmax), exact
  __device__ __forceinline__ uint32_t byte(float x) const {
    return code_byte_fast(kBf ? (x * s1) * s2 : x, a, r);
  }
  // The code bytes of one 16-byte vector (eight 16-bit values; value 2j is
  // the low half of w[j]), 0 where bit i of f is set, packed little-endian
  // into two words.  The same bytes as byte(): code_byte_fast's rounding for
  // all eight, and only for a vector with a value near a half-integer (about
  // one value in 2^14) code_byte_fast again, whose exact rule decides those.
  __device__ __forceinline__ void codes8(const uint32_t (&w)[4], uint32_t f, uint32_t &p0,
                                         uint32_t &p1) const {
    constexpr float kM = 12582912.0f;
    uint32_t b[8];
    bool near = false;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const float x0 = e2f<kBf>((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu));
      const float p = (kBf ? (x0 * s1) * s2 : x0) * r;
      const float t = p + kM;  // M + rint(p), exact for |p| < 2^22
      near |= !(fabsf(p - (t - kM)) < 0.5f - 0x1p-15f);
      b[i] = __float_as_uint(t);
    }
    if (near) {
#pragma unroll
      for (int i = 0; i < 8; i++)
        b[i] = byte(e2f<kBf>((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu)));
    }
#pragma unroll
    for (int i = 0; i < 8; i++) b[i] = ((f >> i) & 1u) ? 0u : b[i];
    p0 = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
    p1 = __byte_perm(__byte_perm(b[4], b[5], 0x0040), __byte_perm(b[6], b[7], 0x0040), 0x5410);
  }
};

// Four signed int8 codes (one 32-bit word) -> four fp16 integers (two half2
// words).  fp16 with exponent field 25 has unit spacing on [1024, 2048), so
// the bit pattern 0x6400 | u is exactly 1024 + u for a byte u; with
// u = code + 128 the value minus 1152 is the code, exactly.
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = w ^ 0x80808080u;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(u), "r"(0x64646464u));
  const uint32_t bias = 0x64806480u;  // (1152, 1152)
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(bias));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(bias));
}

// Programmatic dependent launch controls.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

}  // namespace bnb
