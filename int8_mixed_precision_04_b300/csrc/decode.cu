// The whole layer for decode-sized T (T <= 16): two kernels chained with
// programmatic dependent launch (PDL), no memset.
//
//  dec_act    one thread-block cluster of 8 CTAs; every warp owns a 256-column
//             slab.  Phase 1 (slab-local): outlier columns (|x| >= tau in
//             some row: "Hugging Face Quantization with bitsandbytes",
//             sections 2 and 3) and, per row, the largest |x| over the slab's
//             NON-outlier columns.  The outlier test of a column needs only
//             that column, so phase 1 needs no communication.  Cluster
//             barrier; phase 2 reads every slab's partials over distributed
//             shared memory: row scales sx[t] and the offset of the slab's
//             outliers in the ascending list O.  Then the vector-wise int8
//             codes, O, and the fp16 outlier values XO[t, j] = X[t, O[j]].
//  dec_gemv   one CTA per slice of at most 32 output channels.  Before
//             waiting on dec_act it puts the whole int8 weight slice in
//             flight with bulk async copies into shared memory (the weight
//             does not depend on X), one copy per row and per consumer warp's
//             K-range, so each warp waits only for its own piece.  Each
//             consumer warp owns one K-range for all row groups: it widens
//             the int8 codes of X (shared memory) and of W to fp16 integers
//             in registers and runs 16x8x16 fp16 MMAs with fp32
//             accumulation, converted to int32 at least every 1024 columns
//             (127^2 * 1024 < 2^24, so every fp32 partial sum is an exact
//             integer).  The producer warp gathers the outlier columns of W16
//             for the slice while the MMAs run.  Epilogue: the int32 partials
//             are summed, scaled by (sx/127)(sw/127), the fp16 outlier
//             product is added ("converted back to 16-bit at the end", same
//             page, section 2) and Y is written once.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "mma_frag.cuh"
#include "sm100_ptx.cuh"

namespace bnb {

constexpr int kDecSlab = 256;       // columns per act-pass warp (32 lanes x 8)
constexpr int kActCluster = 8;      // CTAs of dec_act (one cluster)
constexpr int kDecWarps = 16;       // consumer warps of dec_gemv (one K-range each)
constexpr int kDecThreads = (kDecWarps + 1) * 32;  // + one producer warp
constexpr int kDecMaxRows = 32;     // output channels per CTA (4 groups of 8)
constexpr int kDecChunkK = 1024;    // fp32 accumulation is drained at least this often
constexpr int kDecOutSmall = 64;    // outlier columns the producer warp gathers itself

__host__ __device__ constexpr int64_t dec_pitch(int64_t K) { return K + 64; }  // bytes per row
// K columns of warp w: [w * range, min(K, (w + 1) * range)), range a multiple of 64
__host__ __device__ constexpr int64_t dec_range(int64_t K) {
  return ((K + kDecWarps - 1) / kDecWarps + 63) / 64 * 64;
}
// The weight region is reused for the cross-warp reduction after the main loop.
constexpr int64_t kDecRedBytes = (int64_t)kDecWarps * 32 * 16 * 4;
__host__ __device__ constexpr int64_t dec_wregion(int64_t K) {
  return kDecMaxRows * dec_pitch(K) > kDecRedBytes ? kDecMaxRows * dec_pitch(K) : kDecRedBytes;
}

size_t decode_smem_bytes(int64_t K) {
  return (size_t)(dec_wregion(K) + 16 * dec_pitch(K)) + (16 * 32 + 16) * sizeof(float) + 256;
}

// ---------------------------------------------------------------------------
// dec_act
// ---------------------------------------------------------------------------

__global__ void __cluster_dims__(kActCluster, 1, 1) __launch_bounds__(128)
    dec_act_kernel(const uint4 *__restrict__ X, int T, int64_t K, uint32_t thr, int nslab,
                   float *__restrict__ sx_out, int32_t *__restrict__ O,
                   uint32_t *__restrict__ nO_out, int8_t *__restrict__ codes,
                   unsigned short *__restrict__ xo, int64_t xo_pitch,
                   int8_t *__restrict__ dbg_xq, int32_t *__restrict__ status) {
  __shared__ uint32_t part[4][16];  // per warp (slab): row absmax bits of non-outlier columns
  __shared__ uint32_t cnt[4];       // per warp (slab): outlier columns
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  // Let the GEMV launch: its weight prefetch does not depend on this kernel,
  // and it waits for our completion before reading anything we write.
  pdl_trigger();
  // X may be the output of the previous kernel on the stream.
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpc = blockDim.x >> 5;  // warps (slabs) per CTA
  const int rank = (int)cluster.block_rank();
  const int64_t s = (int64_t)rank * wpc + warp;
  const int64_t vecs = K / 8;
  const int64_t v = s * 32 + lane;
  const bool live = s < nslab && v < vecs;
  if (rank == 0 && threadIdx.x == 0) *status = kDevOk;
  uint4 x[16];
  uint32_t flags = 0;
#pragma unroll
  for (int t = 0; t < 16; t++) {
    x[t] = (t < T && live) ? __ldg(X + t * vecs + v) : make_uint4(0, 0, 0, 0);
    if (t < T) {
      const uint32_t w[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
#pragma unroll
      for (int i = 0; i < 4; i++) {
        flags |= (uint32_t)(abs_bits_lo(w[i]) >= thr) << (2 * i);
        flags |= (uint32_t)(abs_bits_hi(w[i]) >= thr) << (2 * i + 1);
      }
    }
  }
  if (!live) flags = 0;
#pragma unroll
  for (int t = 0; t < 16; t++) {
    const uint32_t w[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      if (!((flags >> (2 * i)) & 1)) m = max(m, abs_bits_lo(w[i]));
      if (!((flags >> (2 * i + 1)) & 1)) m = max(m, abs_bits_hi(w[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) part[warp][t] = m;
  }
  const uint32_t pc = __popc(flags);
  uint32_t c = pc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if (lane == 0) cnt[warp] = c;
  cluster.sync();  // every slab's partials are in its CTA's shared memory

  // row scale of row `lane` (lanes 0..15) and this slab's outlier offset
  uint32_t m = 0, base = 0, total = 0;
  for (int r = 0; r < kActCluster; r++) {
    const uint32_t *rpart = cluster.map_shared_rank(&part[0][0], r);
    const uint32_t *rcnt = cluster.map_shared_rank(&cnt[0], r);
    for (int w = 0; w < wpc; w++) {
      if (lane < 16) m = max(m, rpart[w * 16 + lane]);
      const uint32_t cc = rcnt[w];
      total += cc;
      if ((int64_t)r * wpc + w < s) base += cc;
    }
  }
  cluster.sync();  // no CTA leaves while others may still read its shared memory
  const float a_lane = h2f_bits(m);
  if (s == 0) {
    if (lane < T) sx_out[lane] = a_lane;
    if (lane == 0) *nO_out = total;
  }
  // every lane takes part in the shuffles below; only live lanes store
  uint32_t incl = pc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t j0 = base + incl - pc;
  if (live) {
    uint32_t r = 0;
#pragma unroll
    for (int b = 0; b < 8; b++)
      if ((flags >> b) & 1) O[j0 + r++] = (int32_t)(8 * v + b);
  }
#pragma unroll
  for (int t = 0; t < 16; t++) {
    const float a = __shfl_sync(0xffffffffu, a_lane, t);
    if (t >= T || !live) continue;
    const float r = code_recip(a);
    const uint32_t w[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
    int cd[8];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      cd[2 * i] = ((flags >> (2 * i)) & 1) ? 0 : code_of(h2f_bits(w[i] & 0xffffu), a, r);
      cd[2 * i + 1] = ((flags >> (2 * i + 1)) & 1) ? 0 : code_of(h2f_bits(w[i] >> 16), a, r);
    }
    uint32_t p0 = 0, p1 = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      p0 |= (uint32_t)(cd[i] & 0xff) << (8 * i);
      p1 |= (uint32_t)(cd[4 + i] & 0xff) << (8 * i);
    }
    reinterpret_cast<uint2 *>(codes)[t * vecs + v] = make_uint2(p0, p1);
    if (dbg_xq) reinterpret_cast<uint2 *>(dbg_xq)[t * vecs + v] = make_uint2(p0, p1);
    if (flags) {
      uint32_t r2 = 0;
#pragma unroll
      for (int b = 0; b < 8; b++)
        if ((flags >> b) & 1) {
          const uint32_t hb = (w[b >> 1] >> (16 * (b & 1))) & 0xffffu;
          xo[(int64_t)t * xo_pitch + j0 + r2++] = (unsigned short)hb;
        }
    }
  }
}

// ---------------------------------------------------------------------------
// dec_gemv
// ---------------------------------------------------------------------------

struct DecGemvArgs {
  int T;
  int64_t K, N;
  int64_t rows_per_cta;
  const int8_t *Wq;
  const float *sw;
  const unsigned short *W16;
  __half *Y;
  const int8_t *codes;
  const float *sx;
  const int32_t *O;
  const uint32_t *nO;
  const unsigned short *xo;
  int64_t xo_pitch;
  int32_t *dbg_acc;
  int32_t *status;
};

// 16 int8 codes (one 16-byte vector) -> 16 fp16 integers in 8 words.
__device__ __forceinline__ void widen16(const uint4 &v, uint32_t (&h)[8]) {
  s8x4_to_f16x4(v.x, h[0], h[1]);
  s8x4_to_f16x4(v.y, h[2], h[3]);
  s8x4_to_f16x4(v.z, h[4], h[5]);
  s8x4_to_f16x4(v.w, h[6], h[7]);
}

// Fragment convention (see mma_frag.cuh): lane (g = lane/4, q = lane%4) holds
// columns [kb + 16q, kb + 16q + 16) of X rows g and g+8 and of weight row g
// of a group; word pair (2mm, 2mm+1) of each widened vector feeds MMA mm.
__global__ void __launch_bounds__(kDecThreads, 1) dec_gemv_kernel(const DecGemvArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int64_t K = p.K, pitch = dec_pitch(K), range = dec_range(K);
  uint8_t *ws = smem;                                  // [32][pitch] weight codes
  uint8_t *xs = smem + dec_wregion(K);                 // [16][pitch] activation codes
  uint32_t *red = reinterpret_cast<uint32_t *>(smem);  // [16 warps][32][16], after the main loop
  float *osm = reinterpret_cast<float *>(xs + 16 * pitch);  // [16 t][32 rows] small-outlier sums
  float *sxs = osm + 16 * 32;                                // [16] row scales
  uint64_t *bars = reinterpret_cast<uint64_t *>(sxs + 16);
  uint64_t *wbar = bars, *xbar = bars + kDecWarps, *obar = bars + kDecWarps + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = (int64_t)blockIdx.x * p.rows_per_cta;
  const int64_t rows = min(p.N, n0 + p.rows_per_cta) - n0;  // 1..32

  if (warp == kDecWarps) {
    // ---- producer warp: barriers, then the whole weight slice in flight ----
    if (lane == 0) {
      for (int i = 0; i < kDecWarps + 2; i++) mbar_init(bars + i, i == kDecWarps + 1 ? 32 : 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      for (int w = 0; w < kDecWarps; w++) {
        const int64_t k0 = w * range, len = max((int64_t)0, min(K, k0 + range) - k0);
        mbar_expect_tx(wbar + w, (uint32_t)(rows * len));
      }
    }
    __syncwarp();
    for (int64_t i = lane; i < (int64_t)kDecWarps * rows; i += 32) {
      const int64_t w = i / rows, r = i % rows;
      const int64_t k0 = w * range, len = min(K, k0 + range) - k0;
      if (len > 0)
        bulk_g2s(ws + r * pitch + k0, p.Wq + (n0 + r) * K + k0, (uint32_t)len, wbar + w);
    }
  } else {
    // zero what no copy writes: weight rows >= rows, code rows >= T, pads
    for (int64_t i = threadIdx.x; i < (kDecMaxRows + 16) * pitch / 16; i += kDecWarps * 32) {
      const int64_t r = (i * 16) / pitch, c = (i * 16) % pitch;
      const bool copied = c < K && (r < kDecMaxRows ? r < rows : r - kDecMaxRows < p.T);
      uint8_t *dst = r < kDecMaxRows ? ws + r * pitch + c : xs + (r - kDecMaxRows) * pitch + c;
      if (!copied) *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  // the next kernel on the stream may launch now; it waits for our completion
  pdl_trigger();

  if (warp == kDecWarps) {
    pdl_wait();  // codes, scales and outliers of this call are ready
    if (lane == 0) mbar_expect_tx(xbar, (uint32_t)(p.T * K));
    __syncwarp();
    if (lane < p.T) bulk_g2s(xs + lane * pitch, p.codes + lane * K, (uint32_t)K, xbar);
    // row scales and the first outlier columns for this slice: lane = row
    if (lane < 16) sxs[lane] = lane < p.T ? __ldcg(p.sx + lane) : 0.f;
    const int32_t nO = (int32_t)__ldcg(p.nO);
    const int32_t nsmall = min(nO, kDecOutSmall);
    float o[16];
#pragma unroll
    for (int t = 0; t < 16; t++) o[t] = 0.f;
    const int64_t n = n0 + min((int64_t)lane, rows - 1);
    for (int32_t j = 0; j < nsmall; j++) {
      const int32_t k = __ldcg(p.O + j);
      const float wv = h2f_bits(__ldg(p.W16 + n * K + k));
#pragma unroll
      for (int t = 0; t < 16; t++)
        if (t < p.T) o[t] = fmaf(h2f_bits(__ldcg(p.xo + (int64_t)t * p.xo_pitch + j)), wv, o[t]);
    }
#pragma unroll
    for (int t = 0; t < 16; t++) osm[t * 32 + lane] = o[t];
    mbar_arrive(obar);  // 32 arrivals: osm and sxs are written
    return;
  }

  // ---- consumer warps: K-range [k0, k1) for all four row groups ----
  pdl_wait();
  const int g = lane >> 2, q = lane & 3;
  const int64_t k0 = warp * range, k1 = min(K, k0 + range);
  int acc[4][4] = {};
  if (k1 > k0 && mbar_wait_bounded(xbar, 0, p.status) &&
      mbar_wait_bounded(wbar + warp, 0, p.status)) {
    float f[4][4] = {};
    int nb = 0;
    for (int64_t kb = k0; kb < k1; kb += 64) {
      const uint32_t lv = (kb + 16 * q < k1) ? 0xffffffffu : 0u;  // columns past K feed zeros
      uint32_t xa[8], xb[8];
      widen16(*reinterpret_cast<const uint4 *>(xs + g * pitch + kb + 16 * q), xa);
      widen16(*reinterpret_cast<const uint4 *>(xs + (g + 8) * pitch + kb + 16 * q), xb);
#pragma unroll
      for (int gi = 0; gi < 4; gi++) {
        uint32_t h[8];
        widen16(*reinterpret_cast<const uint4 *>(ws + (gi * 8 + g) * pitch + kb + 16 * q), h);
#pragma unroll
        for (int mm = 0; mm < 4; mm++)
          mma_f16_16x8x16(f[gi], xa[2 * mm] & lv, xb[2 * mm] & lv, xa[2 * mm + 1] & lv,
                          xb[2 * mm + 1] & lv, h[2 * mm] & lv, h[2 * mm + 1] & lv);
      }
      if (++nb == kDecChunkK / 64 || kb + 64 >= k1) {  // exact drain into int32
        nb = 0;
#pragma unroll
        for (int gi = 0; gi < 4; gi++)
#pragma unroll
          for (int j = 0; j < 4; j++) {
            acc[gi][j] += __float2int_rn(f[gi][j]);
            f[gi][j] = 0.f;
          }
      }
    }
  }
  // outlier columns beyond the first kDecOutSmall: split over the consumer warps
  const int32_t nO = (int32_t)__ldcg(p.nO);
  float o[4][4] = {};
  for (int32_t j = kDecOutSmall + warp; j < nO; j += kDecWarps) {
    const int32_t k = __ldcg(p.O + j);
    const float x0 = g < p.T ? h2f_bits(__ldcg(p.xo + (int64_t)g * p.xo_pitch + j)) : 0.f;
    const float x1 =
        g + 8 < p.T ? h2f_bits(__ldcg(p.xo + (int64_t)(g + 8) * p.xo_pitch + j)) : 0.f;
#pragma unroll
    for (int gi = 0; gi < 4; gi++) {
      const int64_t na = n0 + min((int64_t)gi * 8 + 2 * q, rows - 1);
      const int64_t nb = n0 + min((int64_t)gi * 8 + 2 * q + 1, rows - 1);
      const float wa = h2f_bits(__ldg(p.W16 + na * K + k));
      const float wb = h2f_bits(__ldg(p.W16 + nb * K + k));
      o[gi][0] = fmaf(x0, wa, o[gi][0]);
      o[gi][1] = fmaf(x0, wb, o[gi][1]);
      o[gi][2] = fmaf(x1, wa, o[gi][2]);
      o[gi][3] = fmaf(x1, wb, o[gi][3]);
    }
  }
  // cross-warp reduction: red[warp][lane][gi*4 + j], in the weight region once
  // every consumer warp is past its main loop
  asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32));
  uint32_t *mine = red + (warp * 32 + lane) * 16;
#pragma unroll
  for (int gi = 0; gi < 4; gi++)
#pragma unroll
    for (int j = 0; j < 4; j++) mine[gi * 4 + j] = (uint32_t)acc[gi][j];
  asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32));
  if (warp < 4) {
    const int gi = warp;
    int a[4] = {0, 0, 0, 0};
    for (int w = 0; w < kDecWarps; w++) {
      const uint32_t *src = red + (w * 32 + lane) * 16 + gi * 4;
#pragma unroll
      for (int j = 0; j < 4; j++) a[j] += (int)src[j];
    }
#pragma unroll
    for (int j = 0; j < 4; j++) acc[0][j] = a[j];
  }
  const bool big = nO > kDecOutSmall;  // the same in every warp
  if (big) {
    asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32));
#pragma unroll
    for (int gi = 0; gi < 4; gi++)
#pragma unroll
      for (int j = 0; j < 4; j++) mine[gi * 4 + j] = __float_as_uint(o[gi][j]);
    asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32));
  }
  if (warp < 4) {
    const int gi = warp;
    float ov[4] = {0.f, 0.f, 0.f, 0.f};
    if (big)
      for (int w = 0; w < kDecWarps; w++) {
        const uint32_t *src = red + (w * 32 + lane) * 16 + gi * 4;
#pragma unroll
        for (int j = 0; j < 4; j++) ov[j] += __uint_as_float(src[j]);
      }
    const bool ok_o = mbar_wait_bounded(obar, 0, p.status);
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int64_t t = g + 8 * (j / 2);
      const int64_t nl = (int64_t)gi * 8 + 2 * q + (j % 2);
      if (t < p.T && nl < rows && ok_o) {
        const int64_t n = n0 + nl;
        const float st = sxs[t] / 127.0f, sn = __ldg(p.sw + n) / 127.0f;
        const float y = fmaf((float)acc[0][j] * st, sn, ov[j] + osm[t * 32 + nl]);
        p.Y[t * p.N + n] = __float2half_rn(y);
        if (p.dbg_acc) p.dbg_acc[t * p.N + n] = acc[0][j];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_decode(const void *X, int64_t T, int64_t K, uint32_t thr, const int8_t *Wq,
                          const float *sw, const void *W16, int64_t N, void *Y,
                          const Workspace &ws, int8_t *dbg_xq, int32_t *dbg_acc, int num_sms,
                          cudaStream_t stream) {
  static bool attr_set = false;  // benign race: every writer sets the same value
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(dec_gemv_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)decode_smem_bytes(kDecodeMaxK));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int nslab = (int)((K + kDecSlab - 1) / kDecSlab);
  const int wpc = (nslab + kActCluster - 1) / kActCluster;  // <= 3 for K <= kDecodeMaxK
  cudaError_t e = cudaSuccess;
  const bool only_main = profile_only_main();
  if (!only_main) {
    ProfScope ps(kKidDecAct, stream);
    e = launch_pdl(dec_act_kernel, dim3(kActCluster), dim3(32 * wpc), 0, stream, true,
                   reinterpret_cast<const uint4 *>(X), (int)T, K, thr, nslab, ws.sx, ws.O,
                   ws.counters + 1, reinterpret_cast<int8_t *>(ws.xcodes),
                   reinterpret_cast<unsigned short *>(ws.xo), ws.kpad, dbg_xq, ws.status);
    note_launch();
  }
  if (e != cudaSuccess) return e;
  DecGemvArgs a;
  a.T = (int)T;
  a.K = K;
  a.N = N;
  int64_t ctas = min((int64_t)num_sms, (N + 7) / 8);
  a.rows_per_cta = (N + ctas - 1) / ctas;  // <= 32: the host only routes N <= 32 * SMs here
  ctas = (N + a.rows_per_cta - 1) / a.rows_per_cta;
  a.Wq = Wq;
  a.sw = sw;
  a.W16 = reinterpret_cast<const unsigned short *>(W16);
  a.Y = reinterpret_cast<__half *>(Y);
  a.codes = reinterpret_cast<const int8_t *>(ws.xcodes);
  a.sx = ws.sx;
  a.O = ws.O;
  a.nO = ws.counters + 1;
  a.xo = reinterpret_cast<const unsigned short *>(ws.xo);
  a.xo_pitch = ws.kpad;
  a.dbg_acc = dbg_acc;
  a.status = ws.status;
  {
    ProfScope ps(kKidGemv, stream);
    e = launch_pdl(dec_gemv_kernel, dim3((unsigned)ctas), dim3(kDecThreads),
                   decode_smem_bytes(K), stream, !only_main, a);
    note_launch();
  }
  return e;
}

}  // namespace bnb
