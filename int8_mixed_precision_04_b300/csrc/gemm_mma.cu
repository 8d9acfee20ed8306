// S4..S6 with the warp-level tensor path (mma.sync), for any T.
//
// Two main loops over one 128 x 128 output tile:
//   1. int8 codes Xq x Wq^T with m16n8k32 s8 MMAs into exact int32;
//   2. after scaling the int32 result by (sx/127)(sw/127) in fp32, the fp16
//      outlier block XO x W16[:, O]^T with m16n8k16 f16 MMAs accumulating on
//      top of it in fp32 (the outlier dimensions "computed in 16-bit",
//      "Hugging Face Quantization with bitsandbytes", section 2);
// then Y is written once in fp16.  The outlier columns of W16 are gathered
// into shared memory per 32-column block.  With only the int8 weight kept
// (W16 null) the gathered columns are Wq's codes as fp16 integers, and
// sw / 127 scales the int8 and outlier sums together at the store.
//
// This is the legacy warp-level tensor path (compiled for sm_103a but not
// tcgen05); it also serves as the exact-int8 comparison route.
#include "common.cuh"
#include "kernels.h"
#include "mma_frag.cuh"

namespace bnb {

constexpr int kMmaBM = 128, kMmaBN = 128, kMmaBK = 64;  // BK in bytes
constexpr int kMmaThreads = 256;

template <bool kBf>  // X, W16, the bias and Y bf16 instead of fp16
__global__ void __launch_bounds__(kMmaThreads) gemm_mma_kernel(
    int64_t T, int64_t K, const int8_t *__restrict__ Wq, const float *__restrict__ sw,
    const unsigned short *__restrict__ W16, int64_t N, uint16_t *__restrict__ Y,
    const int8_t *__restrict__ xcodes, const float *__restrict__ sx,
    const int32_t *__restrict__ O, const uint32_t *__restrict__ counters,
    const __half *__restrict__ xo, int64_t kpad, const unsigned short *__restrict__ bias,
    int32_t *__restrict__ dbg_acc) {
  __shared__ __align__(128) int8_t As[2][kMmaBM * kMmaBK];
  __shared__ __align__(128) int8_t Bs[2][kMmaBN * kMmaBK];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp / 4, wn = warp % 4;  // warp tile 64 x 32
  const int g = lane >> 2, q = lane & 3;
  const int64_t m0 = (int64_t)blockIdx.y * kMmaBM, n0 = (int64_t)blockIdx.x * kMmaBN;

  auto load_int8 = [&](int stage, int64_t kb) {
#pragma unroll
    for (int i = 0; i < 2; i++) {
      const int c = tid + i * kMmaThreads;  // chunk id: row c/4, 16-byte column c%4
      const int r = c >> 2, cc = (c & 3) * 16;
      const bool va = (m0 + r < T) && (kb + cc < K);
      const bool vb = (n0 + r < N) && (kb + cc < K);
      cp_async16(&As[stage][c * 16], va ? (const void *)(xcodes + (m0 + r) * K + kb + cc) : xcodes, va);
      cp_async16(&Bs[stage][c * 16], vb ? (const void *)(Wq + (n0 + r) * K + kb + cc) : Wq, vb);
    }
    cp_async_commit();
  };

  int acc[4][4][4];
#pragma unroll
  for (int a = 0; a < 4; a++)
#pragma unroll
    for (int b = 0; b < 4; b++)
#pragma unroll
      for (int i = 0; i < 4; i++) acc[a][b][i] = 0;

  const int64_t nkb = (K + kMmaBK - 1) / kMmaBK;
  load_int8(0, 0);
  for (int64_t it = 0; it < nkb; it++) {
    const int st = it & 1;
    if (it + 1 < nkb) {
      load_int8(st ^ 1, (it + 1) * kMmaBK);
      cp_async_wait_1();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
    uint4 fa[4], fb[4], fw[4];
#pragma unroll
    for (int mt = 0; mt < 4; mt++) {
      const int r = wm * 64 + mt * 16 + g;
      fa[mt] = *reinterpret_cast<const uint4 *>(&As[st][r * kMmaBK + 16 * q]);
      fb[mt] = *reinterpret_cast<const uint4 *>(&As[st][(r + 8) * kMmaBK + 16 * q]);
    }
#pragma unroll
    for (int nt = 0; nt < 4; nt++) {
      const int r = wn * 32 + nt * 8 + g;
      fw[nt] = *reinterpret_cast<const uint4 *>(&Bs[st][r * kMmaBK + 16 * q]);
    }
#pragma unroll
    for (int mt = 0; mt < 4; mt++)
#pragma unroll
      for (int nt = 0; nt < 4; nt++) mma_s8_block(acc[mt][nt], fa[mt], fb[mt], fw[nt]);
    __syncthreads();
  }

  // scale: y = acc * (sx/127) * (sw/127); element i of tile (mt, nt) is at
  // t = m0 + wm*64 + mt*16 + g + 8*(i/2), n = n0 + wn*32 + nt*8 + 2q + (i%2)
  float y[4][4][4];
#pragma unroll
  for (int mt = 0; mt < 4; mt++)
#pragma unroll
    for (int nt = 0; nt < 4; nt++)
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int64_t t = m0 + wm * 64 + mt * 16 + g + 8 * (i / 2);
        const int64_t n = n0 + wn * 32 + nt * 8 + 2 * q + (i % 2);
        float v = 0.f;
        if (t < T && n < N) {
          if (dbg_acc) dbg_acc[t * N + n] = acc[mt][nt][i];
          // with only the int8 weight, sw / 127 is applied at the store,
          // to the int8 and outlier sums at once (and the bias after it)
          v = (float)acc[mt][nt][i] * __fdiv_rn(sx[t], 127.0f);
          if (W16) {
            v *= __fdiv_rn(sw[n], 127.0f);
            if (bias) v += e2f<kBf>(__ldg(bias + n));
          }
        }
        y[mt][nt][i] = v;
      }

  // outlier part: XO [T x nO] x W16[:, O]^T, 32 columns (64 bytes) per block
  const int32_t nO = (int32_t)__ldg(counters + 1);
  __half *Ah = reinterpret_cast<__half *>(As[0]);
  unsigned short *Bh = reinterpret_cast<unsigned short *>(Bs[0]);
  for (int32_t jb = 0; jb < nO; jb += 32) {
#pragma unroll
    for (int i = 0; i < 2; i++) {
      const int c = tid + i * kMmaThreads;
      const int r = c >> 2, cc = (c & 3) * 8;  // 8 halves per chunk
      const bool va = m0 + r < T;              // XO is zero-padded to 64 columns
      cp_async16(Ah + c * 8, va ? (const void *)(xo + (m0 + r) * kpad + jb + cc) : xo, va);
    }
    cp_async_commit();
    // gather: warp w fills rows 16w .. 16w+15, lane = column
    {
      const int32_t j = jb + lane;
      const int32_t k = j < nO ? __ldg(O + j) : 0;
#pragma unroll 4
      for (int rr = 0; rr < 16; rr++) {
        const int r = warp * 16 + rr;
        unsigned short v = 0;
        if (j < nO && n0 + r < N)
          v = W16 ? __ldg(W16 + (n0 + r) * K + k)
                  : f2e<kBf>((float)__ldg(Wq + (n0 + r) * K + k));  // exact
        Bh[r * 32 + lane] = v;
      }
    }
    cp_async_wait_all();
    __syncthreads();
    uint4 fa[4], fb[4], fw[4];
#pragma unroll
    for (int mt = 0; mt < 4; mt++) {
      const int r = wm * 64 + mt * 16 + g;
      fa[mt] = *reinterpret_cast<const uint4 *>(&As[0][r * kMmaBK + 16 * q]);
      fb[mt] = *reinterpret_cast<const uint4 *>(&As[0][(r + 8) * kMmaBK + 16 * q]);
    }
#pragma unroll
    for (int nt = 0; nt < 4; nt++) {
      const int r = wn * 32 + nt * 8 + g;
      fw[nt] = *reinterpret_cast<const uint4 *>(&Bs[0][r * kMmaBK + 16 * q]);
    }
#pragma unroll
    for (int mt = 0; mt < 4; mt++)
#pragma unroll
      for (int nt = 0; nt < 4; nt++) {
        if (kBf)
          mma_bf16_block(y[mt][nt], fa[mt], fb[mt], fw[nt]);
        else
          mma_f16_block(y[mt][nt], fa[mt], fb[mt], fw[nt]);
      }
    __syncthreads();
  }

  // store Y (fp16), two adjacent columns per lane
#pragma unroll
  for (int mt = 0; mt < 4; mt++)
#pragma unroll
    for (int nt = 0; nt < 4; nt++)
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const int64_t t = m0 + wm * 64 + mt * 16 + g + 8 * h;
        const int64_t n = n0 + wn * 32 + nt * 8 + 2 * q;
        if (t >= T) continue;
        if (!W16) {
#pragma unroll
          for (int u = 0; u < 2; u++)
            if (n + u < N) {
              float &yy = y[mt][nt][2 * h + u];
              yy *= __fdiv_rn(sw[n + u], 127.0f);
              if (bias) yy += e2f<kBf>(__ldg(bias + n + u));
            }
        }
        const uint16_t lo = f2e<kBf>(y[mt][nt][2 * h]);
        const uint16_t hi = f2e<kBf>(y[mt][nt][2 * h + 1]);
        if (n + 1 < N && ((t * N + n) & 1) == 0) {
          *reinterpret_cast<uint32_t *>(Y + t * N + n) = (uint32_t)lo | ((uint32_t)hi << 16);
        } else {
          if (n < N) Y[t * N + n] = lo;
          if (n + 1 < N) Y[t * N + n + 1] = hi;
        }
      }
}

cudaError_t launch_gemm_mma(int64_t T, int64_t K, const int8_t *Wq, const float *sw,
                            const void *W16, const void *bias, int64_t N, bool bf16, void *Y,
                            const Workspace &ws, int32_t *dbg_acc, cudaStream_t stream) {
  dim3 grid((unsigned)((N + kMmaBN - 1) / kMmaBN), (unsigned)((T + kMmaBM - 1) / kMmaBM));
  (bf16 ? gemm_mma_kernel<true> : gemm_mma_kernel<false>)<<<grid, kMmaThreads, 0, stream>>>(
      T, K, Wq, sw, reinterpret_cast<const unsigned short *>(W16), N,
      reinterpret_cast<uint16_t *>(Y), reinterpret_cast<const int8_t *>(ws.xcodes), ws.sx, ws.O,
      ws.counters, ws.xo, ws.kpad, reinterpret_cast<const unsigned short *>(bias), dbg_acc);
  note_launch();
  return cudaGetLastError();
}

}  // namespace bnb
