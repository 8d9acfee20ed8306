// The blockwise 8-bit codec of optimizer states.
//
// 8-bit optimizers keep their states quantized block-wise ("bitsandbytes:
// GPU-Accelerated Inference and Training at Lower Bit Depths", section
// "8-bit optimizers for full-model training"), each block carrying its own
// scaling factor so that one outlier only coarsens its own block (page
// "bitsandbytes", section "What it provides").  Blocks of B consecutive fp32
// values (B a power of two from 64 to 2048; the last block may be short);
// the scale is the block's absmax a; the code is rint(fl32(fl32(127 x) / a)),
// ties to even (0 when a = 0); the decoded value is fl32(fl32(q a) / 127).
// Every operation is one IEEE fp32 rounding (no contraction), so codes and
// decoded values are reproducible bit for bit.  For a >= 2^120, 127 x and
// q a would overflow fp32 (FLT_MAX / 127 is about 2^121): such a block is
// coded with x and a multiplied by 2^-8 and decoded at that scale, the value
// multiplied back by 2^8.  A power-of-two factor commutes with every IEEE
// rounding in the normal range, so this gives the plain formulas' results
// wherever those are finite (values pushed below the normal range have code
// 0 either way).
//
// Both kernels stream HBM: each thread moves 8 consecutive values (two
// 16-byte loads or stores of fp32, one 8-byte access of codes); the B/8
// threads of a block reduce its absmax with warp shuffles (and, for
// B >= 512, shared memory across the block's warps).
#include "common.cuh"
#include "kernels.h"

namespace bnb {

constexpr int kBwThreads = 256;                 // 2048 values per CTA and pass
constexpr int kBwPerThread = 8;
constexpr int64_t kBwChunk = (int64_t)kBwThreads * kBwPerThread;

// The code rint(fl32(num / a)), num = fl32(127 x), |num| <= 127 a.  With
// r = fl32(1 / a), p = fl32(num r) is within 2^-22 |v| < 2^-15 of v = num / a;
// when p is more than 2^-14 away from a half-integer, v and fl32(v) (which
// cannot cross a half-integer, only land on one) round like p, and rint(p)
// -- one magic-number add, ties to even -- is the code.  Otherwise (rarely)
// the IEEE division decides.
// The factor of a block with absmax a (see above).
__device__ __forceinline__ float bw_scale(float a) { return a >= 0x1p120f ? 0x1p-8f : 1.0f; }

__device__ __forceinline__ int8_t bw_code(float x, float a, float r) {
  if (!(a > 0.0f)) return 0;
  constexpr float kM = 12582912.0f;  // 1.5 * 2^23: unit spacing
  const float num = __fmul_rn(127.0f, x);
  const float p = __fmul_rn(num, r);
  const float t = __fadd_rn(p, kM);             // M + rint(p)
  const float e = __fsub_rn(p, __fsub_rn(t, kM));  // p - rint(p), exact
  if (fabsf(e) < 0.5f - 0x1p-14f) return (int8_t)(__float_as_uint(t) & 0xffu);
  return (int8_t)__float2int_rn(__fdiv_rn(num, a));
}

__global__ void __launch_bounds__(kBwThreads) quantize_blockwise_kernel(
    const float *__restrict__ x, int64_t n, int B, int8_t *__restrict__ codes,
    float *__restrict__ absmax) {
  __shared__ float wmax[kBwThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = B / kBwPerThread;  // threads per block (8 .. 256)
  const int64_t nchunks = (n + kBwChunk - 1) / kBwChunk;
  for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const int64_t e0 = c * kBwChunk + (int64_t)tid * kBwPerThread;
    float v[kBwPerThread];
    if (e0 + kBwPerThread <= n) {
      const float4 a = __ldg(reinterpret_cast<const float4 *>(x + e0));
      const float4 b = __ldg(reinterpret_cast<const float4 *>(x + e0) + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
      for (int i = 0; i < kBwPerThread; i++) v[i] = e0 + i < n ? __ldg(x + e0 + i) : 0.0f;
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kBwPerThread; i++) m = fmaxf(m, fabsf(v[i]));
    // the block's absmax: within the warp, then across its warps
    for (int o = (G < 32 ? G : 32) / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (G > 32) {
      if (lane == 0) wmax[warp] = m;
      __syncthreads();
      const int w0 = (warp / (G / 32)) * (G / 32);
      m = 0.0f;
      for (int w = w0; w < w0 + G / 32; w++) m = fmaxf(m, wmax[w]);
      __syncthreads();  // wmax is reused by the next chunk
    }
    if (e0 < n) {
      if ((tid % G) == 0) absmax[e0 / B] = m;
      const float s = bw_scale(m), ms = __fmul_rn(m, s);
      const float r = ms > 0.0f ? __frcp_rn(ms) : 0.0f;
      int8_t q[kBwPerThread];
#pragma unroll
      for (int i = 0; i < kBwPerThread; i++) q[i] = bw_code(__fmul_rn(v[i], s), ms, r);
      if (e0 + kBwPerThread <= n) {
        uint2 w;
        w.x = (uint32_t)(uint8_t)q[0] | ((uint32_t)(uint8_t)q[1] << 8) |
              ((uint32_t)(uint8_t)q[2] << 16) | ((uint32_t)(uint8_t)q[3] << 24);
        w.y = (uint32_t)(uint8_t)q[4] | ((uint32_t)(uint8_t)q[5] << 8) |
              ((uint32_t)(uint8_t)q[6] << 16) | ((uint32_t)(uint8_t)q[7] << 24);
        *reinterpret_cast<uint2 *>(codes + e0) = w;
      } else {
        for (int i = 0; i < kBwPerThread; i++)
          if (e0 + i < n) codes[e0 + i] = q[i];
      }
    }
  }
}

__global__ void __launch_bounds__(kBwThreads) dequantize_blockwise_kernel(
    const int8_t *__restrict__ codes, const float *__restrict__ absmax, int64_t n, int B,
    float *__restrict__ y) {
  const int64_t nchunks = (n + kBwChunk - 1) / kBwChunk;
  for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const int64_t e0 = c * kBwChunk + (int64_t)threadIdx.x * kBwPerThread;
    if (e0 >= n) continue;
    const float a0 = __ldg(absmax + e0 / B);  // the 8 values share one block (B >= 64)
    const float s = bw_scale(a0), a = __fmul_rn(a0, s), inv_s = a0 >= 0x1p120f ? 256.0f : 1.0f;
    int8_t q[kBwPerThread];
    if (e0 + kBwPerThread <= n) {
      const uint2 w = __ldg(reinterpret_cast<const uint2 *>(codes + e0));
#pragma unroll
      for (int i = 0; i < 4; i++) {
        q[i] = (int8_t)(w.x >> (8 * i));
        q[4 + i] = (int8_t)(w.y >> (8 * i));
      }
    } else {
#pragma unroll
      for (int i = 0; i < kBwPerThread; i++) q[i] = e0 + i < n ? codes[e0 + i] : 0;
    }
    float o[kBwPerThread];
#pragma unroll
    for (int i = 0; i < kBwPerThread; i++)
      o[i] = __fmul_rn(__fdiv_rn(__fmul_rn((float)q[i], a), 127.0f), inv_s);
    if (e0 + kBwPerThread <= n) {
      float4 *dst = reinterpret_cast<float4 *>(y + e0);
      dst[0] = make_float4(o[0], o[1], o[2], o[3]);
      dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    } else {
      for (int i = 0; i < kBwPerThread; i++)
        if (e0 + i < n) y[e0 + i] = o[i];
    }
  }
}

static int64_t bw_grid(int64_t n, int num_sms) {
  const int64_t chunks = (n + kBwChunk - 1) / kBwChunk;
  const int64_t cap = 8LL * num_sms;  // resident CTAs of 256 threads
  return chunks < cap ? chunks : cap;
}

cudaError_t launch_quantize_blockwise(const float *x, int64_t n, int B, int8_t *codes,
                                      float *absmax, int num_sms, cudaStream_t stream) {
  quantize_blockwise_kernel<<<(unsigned)bw_grid(n, num_sms), kBwThreads, 0, stream>>>(
      x, n, B, codes, absmax);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dequantize_blockwise(const int8_t *codes, const float *absmax, int64_t n,
                                        int B, float *y, int num_sms, cudaStream_t stream) {
  dequantize_blockwise_kernel<<<(unsigned)bw_grid(n, num_sms), kBwThreads, 0, stream>>>(
      codes, absmax, n, B, y);
  note_launch();
  return cudaGetLastError();
}

}  // namespace bnb
