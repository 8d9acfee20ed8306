// S4..S6 for decode-sized T (T <= 16): memory-bound int8 GEMV.
//
// acc = Xq Wq^T (exact int32) over all K, then
//   Y[t,n] = fp16( acc * (sx[t]/127) * (sw[n]/127) + sum_j XO[t,j] W16[n,O_j] ),
// "multiplied in int8 and only converted back to 16-bit at the end", the
// outlier dimensions in 16-bit ("Hugging Face Quantization with
// bitsandbytes", section 2).
//
// The T <= 16 codes sit in shared memory (rows >= T zero), each warp streams
// eight weight rows with 16-byte loads and multiplies them with the 16 x 32
// int8 warp MMA (tokens are the M = 16 side).  The outlier columns of W16 are
// gathered per output element in the epilogue.
#include "common.cuh"
#include "kernels.h"
#include "mma_frag.cuh"

namespace bnb {

constexpr int kGemvWarps = 4;
constexpr int kGemvUnroll = 4;

__host__ __device__ constexpr int64_t gemv_x_pitch(int64_t K) { return ((K + 127) / 128) * 128 + 64; }

__global__ void __launch_bounds__(kGemvWarps * 32) gemv_decode_kernel(
    int64_t T, int64_t K, const int8_t *__restrict__ Wq, const float *__restrict__ sw,
    const unsigned short *__restrict__ W16, int64_t N, __half *__restrict__ Y,
    const int8_t *__restrict__ xcodes, const float *__restrict__ sx,
    const int32_t *__restrict__ O, const uint32_t *__restrict__ counters,
    const __half *__restrict__ xo, int64_t kpad, int32_t *__restrict__ dbg_acc) {
  extern __shared__ __align__(16) int8_t xs[];
  const int64_t pitch = gemv_x_pitch(K);
  const int64_t chunks_per_row = pitch / 16;
  for (int64_t c = threadIdx.x; c < 16 * chunks_per_row; c += blockDim.x) {
    const int64_t r = c / chunks_per_row, col = (c % chunks_per_row) * 16;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < T && col < K) v = __ldg(reinterpret_cast<const uint4 *>(xcodes + r * K + col));
    *reinterpret_cast<uint4 *>(xs + r * pitch + col) = v;
  }
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n0 = ((int64_t)blockIdx.x * kGemvWarps + warp) * 8;
  if (n0 >= N) return;
  const uint32_t g = lane >> 2, q = lane & 3;
  const int64_t wrow = min(n0 + g, N - 1);
  const int8_t *wp = Wq + wrow * K + 16 * q;
  const int8_t *xa = xs + g * pitch + 16 * q;
  const int8_t *xb = xs + (g + 8) * pitch + 16 * q;
  int acc[4] = {0, 0, 0, 0};
  for (int64_t kb = 0; kb < K; kb += 64 * kGemvUnroll) {
    uint4 w[kGemvUnroll];
#pragma unroll
    for (int u = 0; u < kGemvUnroll; u++) {
      const int64_t off = kb + 64 * u;
      w[u] = (off + 16 * q < K) ? __ldg(reinterpret_cast<const uint4 *>(wp + off))
                                : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kGemvUnroll; u++) {
      const int64_t off = kb + 64 * u;
      if (off < K) {
        const uint4 a = *reinterpret_cast<const uint4 *>(xa + off);
        const uint4 b = *reinterpret_cast<const uint4 *>(xb + off);
        mma_s8_block(acc, a, b, w[u]);
      }
    }
  }
  // epilogue: element i is (t = g + 8*(i/2), n = n0 + 2q + (i%2))
  const int32_t nO = (int32_t)__ldg(counters + 1);
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  const int64_t na = min(n0 + 2 * q, N - 1), nb = min(n0 + 2 * q + 1, N - 1);
  for (int32_t j = 0; j < nO; j++) {
    const int32_t k = __ldg(O + j);
    const float wa = h2f_bits(__ldg(W16 + na * K + k));
    const float wb = h2f_bits(__ldg(W16 + nb * K + k));
    const float x0 = g < T ? __half2float(xo[(int64_t)g * kpad + j]) : 0.f;
    const float x1 = g + 8 < T ? __half2float(xo[(int64_t)(g + 8) * kpad + j]) : 0.f;
    o[0] = fmaf(x0, wa, o[0]);
    o[1] = fmaf(x0, wb, o[1]);
    o[2] = fmaf(x1, wa, o[2]);
    o[3] = fmaf(x1, wb, o[3]);
  }
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const int64_t t = g + 8 * (i / 2), n = n0 + 2 * q + (i % 2);
    if (t < T && n < N) {
      const float st = __fdiv_rn(sx[t], 127.0f), sn = __fdiv_rn(sw[n], 127.0f);
      const float y = fmaf((float)acc[i] * st, sn, o[i]);
      Y[t * N + n] = __float2half_rn(y);
      if (dbg_acc) dbg_acc[t * N + n] = acc[i];
    }
  }
}

cudaError_t launch_gemv_decode(int64_t T, int64_t K, const int8_t *Wq, const float *sw,
                               const void *W16, int64_t N, void *Y, const Workspace &ws,
                               int32_t *dbg_acc, cudaStream_t stream) {
  const size_t smem = (size_t)(16 * gemv_x_pitch(K));
  static bool attr_set = false;  // benign race: every writer sets the same value
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemv_decode_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t groups = (N + 7) / 8;
  const int64_t blocks = (groups + kGemvWarps - 1) / kGemvWarps;
  ProfScope ps(kKidGemv, stream);
  gemv_decode_kernel<<<(unsigned)blocks, kGemvWarps * 32, smem, stream>>>(
      T, K, Wq, sw, reinterpret_cast<const unsigned short *>(W16), N,
      reinterpret_cast<__half *>(Y), reinterpret_cast<const int8_t *>(ws.xcodes), ws.sx, ws.O,
      ws.counters, ws.xo, ws.kpad, dbg_acc);
  note_launch();
  return cudaGetLastError();
}

}  // namespace bnb
