// S2 + S3: the activation pass of the decomposition.
//
// S2 (outlier_scan_kernel): column k is an outlier feature dimension when
//   |X[t,k]| >= tau for some row t ("Hugging Face Quantization with
//   bitsandbytes: 4-bit & 8-bit Models Explained", section 2: a few feature
//   dimensions carry the large values; section 3: the threshold).  The test
//   runs on fp16 bit patterns against the smallest fp16 value >= tau, which
//   is exact.  Per-block partial masks are OR-ed into a bitmask with one
//   atomic per 32 columns; the last block to finish compacts the mask into
//   the ascending index list O and |O| (no grid-wide wait is needed).
// S3 (quantize_rows_kernel): per row, sx[t] = max |X[t,k]| over non-outlier
//   k; codes rint(fl32(127 x)/sx) for non-outlier k, 0 for outliers; and the
//   fp16 outlier block: compacted, XO[t,j] = X[t,O[j]] zero-padded to a
//   multiple of 64, or, when outliers are dense (outlier_block_dense), X
//   masked to the outlier columns (zero elsewhere) over all K columns.
//
// Both kernels are HBM-bound: 16-byte coalesced loads, warp-shuffle and
// shared-memory reductions.
#include "common.cuh"
#include "kernels.h"

namespace bnb {

constexpr int kScanThreads = 256;  // 32 lanes x 8 columns = 256 columns per block row

__global__ void __launch_bounds__(kScanThreads) outlier_scan_kernel(
    const uint4 *__restrict__ X, int64_t T, int64_t K, uint32_t thr_bits,
    int64_t rows_per_block, uint32_t *__restrict__ colmask, uint32_t *__restrict__ counters,
    int32_t *__restrict__ O) {
  __shared__ uint32_t part[kScanThreads / 32][32];
  __shared__ uint32_t is_last;
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t vecs = K / 8;
  const int64_t v = (int64_t)blockIdx.x * 32 + lane;  // this lane's 8-column vector
  const int64_t t0 = (int64_t)blockIdx.y * rows_per_block;
  const int64_t t1 = min(T, t0 + rows_per_block);
  uint32_t flags = 0;
  if (v < vecs) {
    for (int64_t t = t0 + warp; t < t1; t += kScanThreads / 32) {
      uint4 q = __ldg(X + t * vecs + v);
      uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; i++) {
        flags |= (uint32_t)(abs_bits_lo(w[i]) >= thr_bits) << (2 * i);
        flags |= (uint32_t)(abs_bits_hi(w[i]) >= thr_bits) << (2 * i + 1);
      }
    }
  }
  part[warp][lane] = flags;
  __syncthreads();
  if (warp == 0) {
    uint32_t f = 0;
#pragma unroll
    for (int w = 0; w < kScanThreads / 32; w++) f |= part[w][lane];
    // lanes 4i..4i+3 hold the 32 flags of mask word (blockIdx.x*8 + i)
    uint32_t word = f << (8 * (lane & 3));
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    const int64_t wi = (int64_t)blockIdx.x * 8 + (lane >> 2);
    if ((lane & 3) == 0 && word != 0 && wi * 32 < K) atomicOr(colmask + wi, word);
  }
  // last-block compaction
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t total = gridDim.x * gridDim.y;
    is_last = (atomicAdd(counters, 1u) == total - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const int64_t words = (K + 31) / 32;
  const int64_t per = (words + kScanThreads - 1) / kScanThreads;
  const int64_t w0 = min(words, (int64_t)threadIdx.x * per), w1 = min(words, w0 + per);
  uint32_t cnt = 0;
  for (int64_t w = w0; w < w1; w++) cnt += __popc(__ldcg(colmask + w));
  // block exclusive scan of cnt
  __shared__ uint32_t scan[kScanThreads];
  scan[threadIdx.x] = cnt;
  __syncthreads();
  for (int off = 1; off < kScanThreads; off <<= 1) {
    uint32_t add = threadIdx.x >= (unsigned)off ? scan[threadIdx.x - off] : 0;
    __syncthreads();
    scan[threadIdx.x] += add;
    __syncthreads();
  }
  uint32_t pos = scan[threadIdx.x] - cnt;
  for (int64_t w = w0; w < w1; w++) {
    uint32_t m = __ldcg(colmask + w);
    while (m) {
      int b = __ffs(m) - 1;
      m &= m - 1;
      O[pos++] = (int32_t)(w * 32 + b);
    }
  }
  if (threadIdx.x == kScanThreads - 1) counters[1] = scan[kScanThreads - 1];
}

constexpr int kQuantThreads = 256;

// mode 0: int8 codes into `codes` (T x K int8)
// mode 1: fp16 integer codes into `codes` (T x K fp16)
template <int kMode>
__global__ void __launch_bounds__(kQuantThreads) quantize_rows_kernel(
    const uint4 *__restrict__ X, int64_t T, int64_t K, const uint32_t *__restrict__ colmask,
    const uint32_t *__restrict__ counters, const int32_t *__restrict__ O,
    float *__restrict__ sx, float *__restrict__ sxd, void *__restrict__ codes,
    __half *__restrict__ xo, int64_t kpad, int8_t *__restrict__ dbg_xq) {
  __shared__ uint32_t red[kQuantThreads / 32];
  const int64_t vecs = K / 8;
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t nO = (int32_t)__ldcg(counters + 1);
  const bool dense = kMode == 1 && outlier_block_dense(nO, K);  // the tcgen05 GEMM's form
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const uint4 *row = X + t * vecs;
    uint32_t m = 0;
    for (int64_t v = threadIdx.x; v < vecs; v += kQuantThreads) {
      const uint32_t fl = (__ldg(colmask + (v >> 2)) >> (8 * (v & 3))) & 0xffu;
      uint4 q = __ldg(row + v);
      uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; i++) {
        if (!((fl >> (2 * i)) & 1)) m = max(m, abs_bits_lo(w[i]));
        if (!((fl >> (2 * i + 1)) & 1)) m = max(m, abs_bits_hi(w[i]));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = 0;
#pragma unroll
    for (int w = 0; w < kQuantThreads / 32; w++) m = max(m, red[w]);
    __syncthreads();
    const float a = h2f_bits(m);
    const float r = code_recip(a);
    if (threadIdx.x == 0) {
      sx[t] = a;
      sxd[t] = __fdiv_rn(a, 127.0f);
    }
    for (int64_t v = threadIdx.x; v < vecs; v += kQuantThreads) {
      const uint32_t fl = (__ldg(colmask + (v >> 2)) >> (8 * (v & 3))) & 0xffu;
      uint4 q = __ldg(row + v);
      uint32_t w[4] = {q.x, q.y, q.z, q.w};
      int c[8];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        c[2 * i] = ((fl >> (2 * i)) & 1) ? 0 : code_of(h2f_bits(w[i] & 0xffffu), a, r);
        c[2 * i + 1] = ((fl >> (2 * i + 1)) & 1) ? 0 : code_of(h2f_bits(w[i] >> 16), a, r);
      }
      uint32_t p0 = 0, p1 = 0;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        p0 |= (uint32_t)(c[i] & 0xff) << (8 * i);
        p1 |= (uint32_t)(c[4 + i] & 0xff) << (8 * i);
      }
      if (kMode == 0) {
        reinterpret_cast<uint2 *>(codes)[t * vecs + v] = make_uint2(p0, p1);
      } else {
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
          __half2 hh = __halves2half2(__int2half_rn(c[2 * i]), __int2half_rn(c[2 * i + 1]));
          h[i] = *reinterpret_cast<uint32_t *>(&hh);
        }
        reinterpret_cast<uint4 *>(codes)[t * vecs + v] = make_uint4(h[0], h[1], h[2], h[3]);
      }
      if (dbg_xq) reinterpret_cast<uint2 *>(dbg_xq)[t * vecs + v] = make_uint2(p0, p1);
      if (xo && dense) {  // X masked to the outlier columns, zero elsewhere
        uint32_t m[4];
#pragma unroll
        for (int i = 0; i < 4; i++)
          m[i] = (((fl >> (2 * i)) & 1) ? (w[i] & 0xffffu) : 0u) |
                 (((fl >> (2 * i + 1)) & 1) ? (w[i] & 0xffff0000u) : 0u);
        *reinterpret_cast<uint4 *>(xo + t * kpad + 8 * v) = make_uint4(m[0], m[1], m[2], m[3]);
      }
    }
    if (xo && !dense) {  // compacted outlier block XO[t, j] = X[t, O[j]], zero to a multiple of 64
      const unsigned short *xr = reinterpret_cast<const unsigned short *>(row);
      const int32_t jend = (nO + 63) & ~63;
      for (int32_t j = threadIdx.x; j < jend; j += kQuantThreads) {
        unsigned short hb = j < nO ? __ldg(xr + O[j]) : (unsigned short)0;
        xo[t * kpad + j] = __ushort_as_half(hb);
      }
    }
  }
}

cudaError_t launch_act_pass(const void *X, int64_t T, int64_t K, uint32_t thr_bits,
                            const Workspace &ws, int code_mode, bool with_xo,
                            int8_t *dbg_xq, int num_sms, cudaStream_t stream) {
  // The caller has zeroed the status word, the counters and the column mask.
  cudaError_t e;
  // S2: 2-D grid, column slabs of 256 x row slabs, about 4 blocks per SM.
  const int64_t slabs = (K + 255) / 256;
  int64_t want_rows_blocks = (4LL * num_sms + slabs - 1) / slabs;
  if (want_rows_blocks < 1) want_rows_blocks = 1;
  int64_t rows_per_block = (T + want_rows_blocks - 1) / want_rows_blocks;
  if (rows_per_block < 8) rows_per_block = 8;
  const int64_t row_blocks = (T + rows_per_block - 1) / rows_per_block;
  dim3 grid((unsigned)slabs, (unsigned)row_blocks);
  {
    ProfScope ps(kKidOutlierScan, stream);
    outlier_scan_kernel<<<grid, kScanThreads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(X), T, K, thr_bits, rows_per_block, ws.colmask,
        ws.counters, ws.O);
  }
  note_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // S3: one block per row (grid-stride).
  const int64_t qblocks = T < 16LL * num_sms ? T : 16LL * num_sms;
  ProfScope ps(kKidQuantRows, stream);
  if (code_mode == 0)
    quantize_rows_kernel<0><<<(unsigned)qblocks, kQuantThreads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(X), T, K, ws.colmask, ws.counters, ws.O, ws.sx,
        ws.sxd, ws.xcodes, with_xo ? ws.xo : nullptr, ws.kpad, dbg_xq);
  else
    quantize_rows_kernel<1><<<(unsigned)qblocks, kQuantThreads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(X), T, K, ws.colmask, ws.counters, ws.O, ws.sx,
        ws.sxd, ws.xcodes, with_xo ? ws.xo : nullptr, ws.kpad, dbg_xq);
  note_launch();
  return cudaGetLastError();
}

// One warp per weight row: w16o[n, j] = W16[n, O[j]] for j < |O|, zero up to
// the next multiple of 64.  Each element is one scattered sector of W16; the
// copy is made once per call, so the GEMM's token tiles read it by TMA.
__global__ void __launch_bounds__(256) gather_outlier_weights_kernel(
    const unsigned short *__restrict__ W16, int64_t N, int64_t K, const int32_t *__restrict__ O,
    const uint32_t *__restrict__ counters, unsigned short *__restrict__ w16o, int64_t opad) {
  const int32_t nO = (int32_t)__ldcg(counters + 1);
  if (outlier_block_dense(nO, K)) return;  // the GEMM reads W16 itself
  const int32_t jend = (nO + 63) & ~63;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int lane = threadIdx.x & 31;
  for (int64_t n = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; n < N; n += warps)
    for (int32_t j = lane; j < jend; j += 32)
      w16o[n * opad + j] = j < nO ? __ldg(W16 + n * K + __ldcg(O + j)) : (unsigned short)0;
}

cudaError_t launch_gather_outlier_weights(const void *W16, int64_t N, int64_t K,
                                          const Workspace &ws, int num_sms, cudaStream_t stream) {
  int64_t blocks = (N + 7) / 8;
  if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
  ProfScope ps(kKidGatherW16, stream);
  gather_outlier_weights_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      reinterpret_cast<const unsigned short *>(W16), N, K, ws.O, ws.counters,
      reinterpret_cast<unsigned short *>(ws.w16o), ws.opad);
  note_launch();
  return cudaGetLastError();
}

}  // namespace bnb
