// S2 + S3: the activation pass of the decomposition, for the GEMM paths.
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
//   masked to the outlier columns (zero elsewhere) over all K columns.  For
//   the tcgen05 GEMM with a sparse outlier set, the same launch also compacts
//   W16's outlier columns once per call (w16o[n, j] = W16[n, O[j]]; with only
//   the int8 weight kept, Wq[n, O[j]] as an fp16 integer), so that the GEMM's
//   token tiles read them by TMA.
// X and W16 may be bf16 instead of fp16 (kBf): the bit-pattern tests are the
// same, the outlier block and gathered columns stay in X's format, and the
// codes are taken on x and sx scaled by one power of two (RowCode).
//
// All three are HBM-bound: 16-byte coalesced loads, every load of a thread
// issued before any is used (the row pass keeps its row in registers and
// reads it once), warp-shuffle and shared-memory reductions.
#include "common.cuh"
#include "kernels.h"

namespace bnb {

// The int8 codes of one 16-byte vector (8 fp16 or bf16 values, flags f:
// outlier columns get 0) under the row's code rule rc, as two words of four
// code bytes.  code_byte is exact and uses no conversion-pipe instruction;
// the GEMM's fp16 integer codes come from the bytes by s8x4_to_f16x4.
template <bool kBf>
__device__ __forceinline__ void codes8(const uint32_t (&w)[4], uint32_t f, const RowCode<kBf> &rc,
                                       uint32_t &p0, uint32_t &p1) {
  rc.codes8(w, f, p0, p1);
}

constexpr int kScanThreads = 256;  // 32 lanes x 8 columns = 256 columns per block row
constexpr int kScanUnroll = 8;     // rows of X in flight per warp

__global__ void __launch_bounds__(kScanThreads) outlier_scan_kernel(
    const uint4 *__restrict__ X, int64_t T, int64_t K, uint32_t thr_bits,
    int64_t rows_per_block, uint32_t *__restrict__ colmask, uint32_t *__restrict__ counters,
    int32_t *__restrict__ O) {
  __shared__ uint32_t part[kScanThreads / 32][32];
  __shared__ uint32_t is_last;
  // the row pass may launch now (it waits for this grid before reading it)
  pdl_trigger();
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t vecs = K / 8;
  const int64_t v = (int64_t)blockIdx.x * 32 + lane;  // this lane's 8-column vector
  const int64_t t0 = (int64_t)blockIdx.y * rows_per_block;
  const int64_t t1 = min(T, t0 + rows_per_block);
  uint32_t flags = 0;
  if (v < vecs) {
    for (int64_t t = t0 + warp; t < t1; t += (kScanThreads / 32) * kScanUnroll) {
      uint4 q[kScanUnroll];
#pragma unroll
      for (int u = 0; u < kScanUnroll; u++) {  // all loads in flight before any is used
        const int64_t tt = t + (kScanThreads / 32) * u;
        q[u] = tt < t1 ? __ldg(X + tt * vecs + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kScanUnroll; u++) {
        if (t + (kScanThreads / 32) * u >= t1) break;  // past the rows: no flags (tau = 0)
        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
          flags |= (uint32_t)(abs_bits_lo(w[i]) >= thr_bits) << (2 * i);
          flags |= (uint32_t)(abs_bits_hi(w[i]) >= thr_bits) << (2 * i + 1);
        }
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
  // last-block compaction (the lanes that published mask words order them
  // before the block's count)
  if (warp == 0) __threadfence();
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
  // block exclusive scan of cnt: warp scans, then the warp totals
  __shared__ uint32_t wsum[kScanThreads / 32];
  uint32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if ((int)lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kScanThreads / 32; w++) {
    if (w < (int)warp) before += wsum[w];
    total += wsum[w];
  }
  uint32_t pos = before + incl - cnt;
  for (int64_t w = w0; w < w1; w++) {
    uint32_t m = __ldcg(colmask + w);
    while (m) {
      int b = __ffs(m) - 1;
      m &= m - 1;
      O[pos++] = (int32_t)(w * 32 + b);
    }
  }
  if (threadIdx.x == 0) counters[1] = total;
}

constexpr int kQuantThreads = 256;
constexpr int kQuantRegVecs = 4;  // row vectors a thread keeps in registers (K <= 8192)

// The codes, row scale and outlier block of one row (a block per row).
// kMode 0: int8 codes into `codes` (T x K int8); kMode 1: fp16 integer codes
// (T x K fp16).  kReg: the row fits the block's registers (read once);
// otherwise it is read twice (maximum, then codes), the second time from L2.
template <int kMode, bool kReg, bool kBf>
__device__ __forceinline__ void quantize_row(const uint4 *__restrict__ row, int64_t t, int64_t vecs,
                                             const uint32_t *__restrict__ colmask, bool dense,
                                             float *__restrict__ sx, float *__restrict__ sxd,
                                             void *__restrict__ codes, __half *__restrict__ xo,
                                             int64_t kpad, int8_t *__restrict__ dbg_xq,
                                             uint32_t *red) {
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kV = kReg ? kQuantRegVecs : 1;
  uint4 q[kV];
  uint32_t fl[kV];
  uint32_t m = 0;
  if (kReg) {
#pragma unroll
    for (int i = 0; i < kV; i++) {  // all loads in flight before any is used
      const int64_t v = threadIdx.x + (int64_t)kQuantThreads * i;
      q[i] = v < vecs ? __ldg(row + v) : make_uint4(0, 0, 0, 0);
      fl[i] = v < vecs ? (__ldg(colmask + (v >> 2)) >> (8 * (v & 3))) & 0xffu : 0u;
    }
#pragma unroll
    for (int i = 0; i < kV; i++) {
      const uint32_t w[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        if (!((fl[i] >> (2 * j)) & 1)) m = max(m, abs_bits_lo(w[j]));
        if (!((fl[i] >> (2 * j + 1)) & 1)) m = max(m, abs_bits_hi(w[j]));
      }
    }
  } else {
    for (int64_t v = threadIdx.x; v < vecs; v += kQuantThreads) {
      const uint32_t f = (__ldg(colmask + (v >> 2)) >> (8 * (v & 3))) & 0xffu;
      const uint4 u = __ldg(row + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        if (!((f >> (2 * j)) & 1)) m = max(m, abs_bits_lo(w[j]));
        if (!((f >> (2 * j + 1)) & 1)) m = max(m, abs_bits_hi(w[j]));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = 0;
#pragma unroll
  for (int w = 0; w < kQuantThreads / 32; w++) m = max(m, red[w]);
  __syncthreads();  // red is reused by the next row
  const float a = e2f<kBf>(m);
  const RowCode<kBf> rc(a);
  if (threadIdx.x == 0) {
    sx[t] = a;
    sxd[t] = __fdiv_rn(a, 127.0f);
  }
  // the codes and the outlier block, vector by vector
  auto emit = [&](int64_t v, const uint4 &u, uint32_t f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t p0, p1;
    codes8<kBf>(w, f, rc, p0, p1);
    if (kMode == 0) {
      reinterpret_cast<uint2 *>(codes)[t * vecs + v] = make_uint2(p0, p1);
    } else {
      uint32_t h[4];
      s8x4_to_f16x4(p0, h[0], h[1]);
      s8x4_to_f16x4(p1, h[2], h[3]);
      reinterpret_cast<uint4 *>(codes)[t * vecs + v] = make_uint4(h[0], h[1], h[2], h[3]);
    }
    if (dbg_xq) reinterpret_cast<uint2 *>(dbg_xq)[t * vecs + v] = make_uint2(p0, p1);
    if (xo && dense) {  // X masked to the outlier columns, zero elsewhere
      uint32_t mk[4];
#pragma unroll
      for (int j = 0; j < 4; j++)
        mk[j] = (((f >> (2 * j)) & 1) ? (w[j] & 0xffffu) : 0u) |
                (((f >> (2 * j + 1)) & 1) ? (w[j] & 0xffff0000u) : 0u);
      *reinterpret_cast<uint4 *>(xo + t * kpad + 8 * v) = make_uint4(mk[0], mk[1], mk[2], mk[3]);
    }
  };
  if constexpr (kReg) {
#pragma unroll
    for (int i = 0; i < kV; i++) {
      const int64_t v = threadIdx.x + (int64_t)kQuantThreads * i;
      if (v < vecs) emit(v, q[i], fl[i]);
    }
  } else {
    for (int64_t v = threadIdx.x; v < vecs; v += kQuantThreads)
      emit(v, __ldg(row + v), (__ldg(colmask + (v >> 2)) >> (8 * (v & 3))) & 0xffu);
  }
}

struct QuantArgs {
  const uint4 *X;
  int64_t T, K;
  const uint32_t *colmask;
  const uint32_t *counters;
  const int32_t *O;
  float *sx, *sxd;
  void *codes;
  __half *xo;                  // null: no outlier block
  int64_t kpad;
  int8_t *dbg_xq;
  const unsigned short *W16;   // null: no W16 gather
  const int8_t *Wq;            // non-null (W16 null): gather the int8 weight's columns instead
  int64_t N;
  unsigned short *w16o;
  int64_t opad;
};

template <int kMode, bool kBf>
// (Three blocks per SM: the eight-at-a-time code rule fits 80 registers;
// unbounded it took 117, and at one value at a time the pass was slower.)
__global__ void __launch_bounds__(kQuantThreads, 3) quantize_rows_kernel(const QuantArgs p) {
  __shared__ uint32_t red[kQuantThreads / 32];
  // launched with programmatic dependent launch behind the column scan:
  // everything below reads what the scan wrote.  (No early trigger here: a
  // GEMM CTA needs a whole SM, and one launched early would hold SMs the
  // remaining row blocks need.)
  pdl_wait();
  const int64_t vecs = p.K / 8;
  const int32_t nO = (int32_t)__ldcg(p.counters + 1);
  const bool dense = kMode == 1 && outlier_block_dense(nO, p.K);  // the tcgen05 GEMM's form
  const bool reg = vecs <= (int64_t)kQuantThreads * kQuantRegVecs;
  for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x) {
    const uint4 *row = p.X + t * vecs;
    if (reg)
      quantize_row<kMode, true, kBf>(row, t, vecs, p.colmask, dense, p.sx, p.sxd, p.codes, p.xo,
                                p.kpad, p.dbg_xq, red);
    else
      quantize_row<kMode, false, kBf>(row, t, vecs, p.colmask, dense, p.sx, p.sxd, p.codes, p.xo,
                                 p.kpad, p.dbg_xq, red);
    if (p.xo && !dense) {  // compacted outlier block XO[t, j] = X[t, O[j]], zero to a multiple of 64
      const unsigned short *xr = reinterpret_cast<const unsigned short *>(row);
      const int32_t jend = (nO + 63) & ~63;
      for (int32_t j = threadIdx.x; j < jend; j += kQuantThreads) {
        unsigned short hb = j < nO ? __ldg(xr + __ldg(p.O + j)) : (unsigned short)0;
        p.xo[t * p.kpad + j] = __ushort_as_half(hb);
      }
    }
  }
  // W16 at a sparse outlier set, once per call: one warp per weight row,
  // w16o[n, j] = W16[n, O[j]] for j < |O|, zero up to the next multiple of
  // 64.  Each element is one scattered sector of W16, so every lane keeps
  // four loads in flight.  With only the int8 weight kept, its codes are
  // gathered instead, as fp16 integers (exact).
  if ((p.W16 || p.Wq) && !dense && nO > 0) {
    const int32_t jend = (nO + 63) & ~63;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kQuantThreads / 32);
    for (int64_t n = (int64_t)blockIdx.x * (kQuantThreads / 32) + threadIdx.x / 32; n < p.N;
         n += warps) {
      const unsigned short *wr = p.W16 ? p.W16 + n * p.K : nullptr;
      const int8_t *qr = p.Wq + n * p.K;
      for (int32_t j0 = 0; j0 < jend; j0 += 128) {
        unsigned short w[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
          const int32_t j = j0 + lane + 32 * u;
          w[u] = j >= nO ? (unsigned short)0
                 : wr    ? __ldg(wr + __ldg(p.O + j))
                         : f2e<kBf>((float)__ldg(qr + __ldg(p.O + j)));  // exact
        }
#pragma unroll
        for (int u = 0; u < 4; u++) {
          const int32_t j = j0 + lane + 32 * u;
          if (j < jend) p.w16o[n * p.opad + j] = w[u];
        }
      }
    }
  }
}

cudaError_t launch_act_pass(const void *X, int64_t T, int64_t K, uint32_t thr_bits,
                            const Workspace &ws, int code_mode, bool with_xo, const void *W16,
                            const int8_t *Wq, int64_t N, bool bf16, int8_t *dbg_xq,
                            int num_sms, cudaStream_t stream, bool pdl) {
  // The caller has zeroed the status word, the counters and the column mask.
  cudaError_t e;
  // S2: 2-D grid, column slabs of 256 x row slabs, about 8 blocks per SM,
  // each warp with kScanUnroll rows in flight: some 128 KB of loads in flight
  // per SM, to cover HBM latency (at 2 blocks per SM a 4096 x 8192 scan ran
  // at 0.4 of the copy bandwidth, latency-bound).
  const int64_t slabs = (K + 255) / 256;
  int64_t want_rows_blocks = (8LL * num_sms + slabs - 1) / slabs;
  if (want_rows_blocks < 1) want_rows_blocks = 1;
  int64_t rows_per_block = (T + want_rows_blocks - 1) / want_rows_blocks;
  // at least one full round of loads per warp (8 warps x kScanUnroll rows)
  if (rows_per_block < 8 * kScanUnroll) rows_per_block = 8 * kScanUnroll;
  const int64_t row_blocks = (T + rows_per_block - 1) / rows_per_block;
  dim3 grid((unsigned)slabs, (unsigned)row_blocks);
  outlier_scan_kernel<<<grid, kScanThreads, 0, stream>>>(
      reinterpret_cast<const uint4 *>(X), T, K, thr_bits, rows_per_block, ws.colmask,
      ws.counters, ws.O);
  note_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // S3: one block per row (grid-stride); with the W16 gather, enough blocks
  // for one weight row per warp up to 8 blocks per SM.
  QuantArgs a;
  a.X = reinterpret_cast<const uint4 *>(X);
  a.T = T;
  a.K = K;
  a.colmask = ws.colmask;
  a.counters = ws.counters;
  a.O = ws.O;
  a.sx = ws.sx;
  a.sxd = ws.sxd;
  a.codes = ws.xcodes;
  a.xo = with_xo ? ws.xo : nullptr;
  a.kpad = ws.kpad;
  a.dbg_xq = dbg_xq;
  a.W16 = code_mode == 1 ? reinterpret_cast<const unsigned short *>(W16) : nullptr;
  a.Wq = code_mode == 1 && W16 == nullptr ? Wq : nullptr;
  a.N = N;
  a.w16o = reinterpret_cast<unsigned short *>(ws.w16o);
  a.opad = ws.opad;
  int64_t qblocks = T < 16LL * num_sms ? T : 16LL * num_sms;
  if (a.W16 || a.Wq) {
    const int64_t gb = (N + 7) / 8 < 8LL * num_sms ? (N + 7) / 8 : 8LL * num_sms;
    if (gb > qblocks) qblocks = gb;
  }
  auto *kern = code_mode == 0 ? (bf16 ? quantize_rows_kernel<0, true> : quantize_rows_kernel<0, false>)
                              : (bf16 ? quantize_rows_kernel<1, true> : quantize_rows_kernel<1, false>);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)qblocks);
  cfg.blockDim = dim3(kQuantThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  note_launch();
  return e;
}

}  // namespace bnb
