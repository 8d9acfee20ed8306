// The whole layer for decode-sized T (T <= 16) in one kernel per call.
//
// dec_fused: one CTA per slice of at most 32 output channels (one CTA per
// SM).  At launch all its threads put the CTA's whole int8 weight slice in
// flight with 16-byte async copies, before waiting on the previous kernel of
// the stream (the weight does not depend on X).  While the
// weight streams in, the 16 consumer warps run the activation pass over all
// of X themselves, so that no second kernel and no inter-kernel dependency
// sits on the path:
//   - warp w owns a slab of 256 columns; every lane one 8-column vector of
//     all T rows.  A column is an outlier feature dimension when |x| >= tau
//     in some row ("Hugging Face Quantization with bitsandbytes: 4-bit &
//     8-bit Models Explained", sections 2 and 3); the test needs only that
//     column, so it is lane-local.  The row maxima over non-outlier columns
//     are reduced per warp, then across warps through shared memory;
//   - vector-wise int8 codes rint(fl32(127 x) / sx) of the non-outlier
//     columns go to shared memory, and the ascending outlier column list is
//     compacted from per-warp counts.
// CTA 0 also writes sx, O and |O| to the workspace (and the codes when
// asked), for the debug entry point.
// Then each consumer warp owns one K-range for all four 8-row groups: it
// widens the int8 codes of X and W to fp16 integers in registers and runs
// 16x8x16 fp16 MMAs with fp32 accumulation, converted to int32 at least
// every 1024 columns (127^2 * 1024 < 2^24, so every fp32 partial sum is an
// exact integer).  The producer warp adds up the first outlier columns of W16
// times X for the slice while the MMAs run; the consumers split any further
// ones.  Epilogue: the int32 partials are summed, scaled by (sx/127)(sw/127),
// the 16-bit outlier product is added ("converted back to 16-bit at the end",
// same page, section 2) and Y is written once.
#include "common.cuh"
#include "kernels.h"
#include "mma_frag.cuh"
#include "sm100_ptx.cuh"

namespace bnb {

constexpr int kDecWarps = 16;                      // consumer warps (one K-range each)
constexpr int kDecThreads = (kDecWarps + 1) * 32;  // + one producer warp
constexpr int kDecMaxRows = 32;                    // output channels per CTA (4 groups of 8)
constexpr int kDecChunkK = 1024;                   // fp32 accumulation is drained this often
constexpr int kDecOutSmall = 64;                   // outlier columns the producer warp sums
static_assert(kDecodeMaxK <= kDecWarps * 256, "one 8-column vector per act-pass lane");

__host__ __device__ constexpr int64_t dec_pitch(int64_t K) { return K + 64; }  // bytes per row
// K columns of MMA warp w: [w * range, min(K, (w + 1) * range)), range a multiple of 64
__host__ __device__ constexpr int64_t dec_range(int64_t K) {
  return ((K + kDecWarps - 1) / kDecWarps + 63) / 64 * 64;
}
// The weight region is reused for the cross-warp reduction after the main loop.
constexpr int64_t kDecRedBytes = (int64_t)kDecWarps * 32 * 16 * 4;
__host__ __device__ constexpr int64_t dec_wregion(int64_t K) {
  return kDecMaxRows * dec_pitch(K) > kDecRedBytes ? kDecMaxRows * dec_pitch(K) : kDecRedBytes;
}
__host__ __device__ constexpr int64_t dec_ocap(int64_t K) { return (K + 7) / 8 * 8; }

// weight rows, code rows, outlier list (uint16), osm [16][32], sxs [16],
// part [16 warps][16 rows], cnt [16 warps], one mbarrier
size_t decode_smem_bytes(int64_t K) {
  return (size_t)(dec_wregion(K) + 16 * dec_pitch(K) + 2 * dec_ocap(K)) +
         (16 * 32 + 16 + kDecWarps * 16 + kDecWarps) * 4 + 8;
}

struct DecArgs {
  const uint4 *X;              // [T x K] fp16 as 16-byte vectors
  const unsigned short *X16;   // the same, as fp16 bit patterns
  int T;
  int64_t K, N;
  uint32_t thr;                // smallest fp16 magnitude bits >= tau
  int64_t rows_per_cta;
  const int8_t *Wq;
  const float *sw;
  const unsigned short *W16;
  __half *Y;
  float *sx_out;               // [T]  (CTA 0)
  int32_t *O_out;              // [K]  (CTA 0)
  uint32_t *nO_out;            // [1]  (CTA 0)
  int8_t *dbg_xq;              // [T x K] or null (CTA 0)
  int32_t *dbg_acc;            // [T x N] or null
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
__global__ void __launch_bounds__(kDecThreads, 1) dec_fused_kernel(const DecArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int64_t K = p.K, pitch = dec_pitch(K), range = dec_range(K);
  uint8_t *ws = smem;                                          // [32][pitch] weight codes
  uint8_t *xs = smem + dec_wregion(K);                         // [16][pitch] activation codes
  uint16_t *ocols = reinterpret_cast<uint16_t *>(xs + 16 * pitch);  // outlier columns
  float *osm = reinterpret_cast<float *>(ocols + dec_ocap(K));  // [16 t][32 rows]
  float *sxs = osm + 16 * 32;                                   // [16] row scales
  uint32_t *part = reinterpret_cast<uint32_t *>(sxs + 16);      // [16 warps][16 rows]
  uint32_t *cnt = part + kDecWarps * 16;                        // [16 warps]
  uint64_t *obar = reinterpret_cast<uint64_t *>(cnt + kDecWarps);
  uint32_t *red = reinterpret_cast<uint32_t *>(smem);  // [16 warps][32][16], after the main loop

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T;
  const int64_t n0 = (int64_t)blockIdx.x * p.rows_per_cta;
  const int64_t rows = min(p.N, n0 + p.rows_per_cta) - n0;  // 1..32

  if (threadIdx.x == 0) {
    mbar_init(obar, 32);
    mbar_init_fence();
  }
  // The whole weight slice in flight at once: every thread issues 16-byte
  // async copies of its share (consecutive threads, consecutive chunks of a
  // row).  Weight rows past `rows`, code rows past T and the pads past K are
  // never written: the MMAs mask columns past K, and accumulator rows >= T or
  // columns >= rows are never stored.
  {
    const int64_t cpr = K / 16;  // 16-byte chunks per row
    for (int64_t i = threadIdx.x; i < rows * cpr; i += kDecThreads) {
      const int64_t r = i / cpr, c = (i - r * cpr) * 16;
      cp_async16(ws + r * pitch + c, p.Wq + (n0 + r) * K + c, true);
    }
    cp_async_commit();
  }
  __syncthreads();
  // the next kernel on the stream may launch now; it waits for our completion
  pdl_trigger();
  // X may be the output of the previous kernel on the stream
  pdl_wait();

  // ---- activation pass, phase 1: outlier columns and partial row maxima ----
  const int64_t vecs = K / 8;
  const int64_t v = (int64_t)warp * 32 + lane;  // this lane's 8-column vector
  const bool live = warp < kDecWarps && v < vecs;
  uint4 x[16];
  uint32_t flags = 0;
  if (warp < kDecWarps) {
#pragma unroll
    for (int t = 0; t < 16; t++)  // all loads in flight before any is used
      x[t] = (t < T && live) ? __ldg(p.X + t * vecs + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int t = 0; t < 16; t++) {
      if (t < T) {  // padding rows must not flag columns (tau = 0 flags a zero)
        const uint32_t w[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
          flags |= (uint32_t)(abs_bits_lo(w[i]) >= p.thr) << (2 * i);
          flags |= (uint32_t)(abs_bits_hi(w[i]) >= p.thr) << (2 * i + 1);
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
      if (lane == 0) part[warp * 16 + t] = m;
    }
    uint32_t c = __popc(flags);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) cnt[warp] = c;
  }
  __syncthreads();

  // |O| and this warp's offset in the ascending outlier list
  uint32_t nO_u = 0, base = 0;
  for (int w = 0; w < kDecWarps; w++) {
    const uint32_t cc = cnt[w];
    nO_u += cc;
    if (w < warp) base += cc;
  }
  const int32_t nO = (int32_t)nO_u;

  // ---- activation pass, phase 2: row scales, outlier list, int8 codes ----
  if (warp < kDecWarps) {
    uint32_t m = 0;
    if (lane < 16)
      for (int w = 0; w < kDecWarps; w++) m = max(m, part[w * 16 + lane]);
    const float a_lane = h2f_bits(m);  // sx of row `lane` (0 for rows >= T)
    if (warp == 0 && lane < 16) sxs[lane] = a_lane;
    if (blockIdx.x == 0 && warp == 0) {
      if (lane < T) p.sx_out[lane] = a_lane;
      if (lane == 0) {
        *p.nO_out = nO_u;
        *p.status = kDevOk;
      }
    }
    const uint32_t pc = __popc(flags);
    uint32_t incl = pc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (live && flags) {
      uint32_t j = base + incl - pc;
#pragma unroll
      for (int b = 0; b < 8; b++)
        if ((flags >> b) & 1) {
          ocols[j] = (uint16_t)(8 * v + b);
          if (blockIdx.x == 0) p.O_out[j] = (int32_t)(8 * v + b);
          ++j;
        }
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
      *reinterpret_cast<uint2 *>(xs + t * pitch + 8 * v) = make_uint2(p0, p1);
      if (blockIdx.x == 0 && p.dbg_xq)
        reinterpret_cast<uint2 *>(p.dbg_xq)[t * vecs + v] = make_uint2(p0, p1);
    }
  }
  cp_async_wait_all();  // this thread's weight copies have landed
  __syncthreads();      // all weight rows, codes, outlier list and row scales are in shared memory

  if (warp == kDecWarps) {
    // ---- producer warp: the first outlier columns for this slice, lane = row ----
    const int32_t nsmall = min(nO, kDecOutSmall);
    float o[16];
#pragma unroll
    for (int t = 0; t < 16; t++) o[t] = 0.f;
    const int64_t n = n0 + min((int64_t)lane, rows - 1);
    for (int32_t j = 0; j < nsmall; j++) {
      const int64_t k = ocols[j];
      const float wv = h2f_bits(__ldg(p.W16 + n * K + k));
#pragma unroll
      for (int t = 0; t < 16; t++)
        if (t < T) o[t] = fmaf(h2f_bits(__ldg(p.X16 + t * K + k)), wv, o[t]);
    }
#pragma unroll
    for (int t = 0; t < 16; t++) osm[t * 32 + lane] = o[t];
    mbar_arrive(obar);  // 32 arrivals: osm is written
    return;
  }

  // ---- consumer warps: K-range [k0, k1) for all four row groups ----
  const int g = lane >> 2, q = lane & 3;
  const int64_t k0 = warp * range, k1 = min(K, k0 + range);
  int acc[4][4] = {};
  if (k1 > k0) {
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
  float o[4][4] = {};
  for (int32_t j = kDecOutSmall + warp; j < nO; j += kDecWarps) {
    const int64_t k = ocols[j];
    const float x0 = g < T ? h2f_bits(__ldg(p.X16 + (int64_t)g * K + k)) : 0.f;
    const float x1 = g + 8 < T ? h2f_bits(__ldg(p.X16 + (int64_t)(g + 8) * K + k)) : 0.f;
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
      if (t < T && nl < rows && ok_o) {
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

cudaError_t launch_decode(const void *X, int64_t T, int64_t K, uint32_t thr, const int8_t *Wq,
                          const float *sw, const void *W16, int64_t N, void *Y,
                          const Workspace &ws, int8_t *dbg_xq, int32_t *dbg_acc, int num_sms,
                          cudaStream_t stream) {
  static bool attr_set = false;  // benign race: every writer sets the same value
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(dec_fused_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)decode_smem_bytes(kDecodeMaxK));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  DecArgs a;
  a.X = reinterpret_cast<const uint4 *>(X);
  a.X16 = reinterpret_cast<const unsigned short *>(X);
  a.T = (int)T;
  a.K = K;
  a.N = N;
  a.thr = thr;
  int64_t ctas = min((int64_t)num_sms, (N + 7) / 8);
  a.rows_per_cta = (N + ctas - 1) / ctas;  // <= 32: the host only routes N <= 32 * SMs here
  ctas = (N + a.rows_per_cta - 1) / a.rows_per_cta;
  a.Wq = Wq;
  a.sw = sw;
  a.W16 = reinterpret_cast<const unsigned short *>(W16);
  a.Y = reinterpret_cast<__half *>(Y);
  a.sx_out = ws.sx;
  a.O_out = ws.O;
  a.nO_out = ws.counters + 1;
  a.dbg_xq = dbg_xq;
  a.dbg_acc = dbg_acc;
  a.status = ws.status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = decode_smem_bytes(K);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = profile_only_main() ? 0 : 1;  // profiling mode 2: no overlap with the previous call
  ProfScope ps(kKidDecFused, stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, dec_fused_kernel, a);
  note_launch();
  return e;
}

}  // namespace bnb
