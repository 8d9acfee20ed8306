// The whole layer for decode-sized T (T <= 16) in one kernel per call, for any
// N and K <= 8192, with K split across a thread-block cluster.
//
// What is computed (t a token, n an output channel):
//   O = { k : |X[t,k]| >= tau for some t }, sx[t] = max_{k not in O} |X[t,k]|,
//   Xq = vector-wise int8 codes of X outside O, acc = Xq Wq^T (exact int32),
//   Y[t,n] = fp16( acc (sx[t]/127)(sw[n]/127) + sum_{k in O} X[t,k] W16[n,k] )
// -- the LLM.int8() decomposition: outlier feature dimensions in 16-bit, the
// rest vector-wise in int8, converted back to 16-bit at the end ("Hugging Face
// Quantization with bitsandbytes: 4-bit & 8-bit Models Explained", section 2;
// threshold, section 3; "bitsandbytes: GPU-Accelerated Inference and Training
// at Lower Bit Depths", section "How LLM.int8() quantizes weights and
// activations").
//
// Layout of the work.  A cluster of C CTAs covers every column: CTA rank c owns
// the K-range [1024 c, 1024 c + 1024) for all of the cluster's output channels,
// so each CTA reads only its own slice of X and of each weight row:
//   1. Weight stream.  Right at the start, before the kernel waits for the
//      previous work on the stream (the weights are not written by it), warp g
//      puts the 8 rows x 1024 bytes of the cluster's 8-channel group g in
//      flight with 16-byte cp.async copies into a swizzled shared tile, counted
//      on that group's mbarrier.  Channels come in batches of G groups; with
//      more batches than fit, two weight buffers alternate and the next batch
//      streams while this one is multiplied.
//   2. Activation pass, local to the CTA: it loads X[0..T, its columns], flags
//      its columns that reach tau in any row and takes each row's maximum over
//      its other columns.  The only exchange before the MMAs follows: each CTA
//      stores its 16 row maxima and its outlier count into every CTA of the
//      cluster (st.async, counted on an mbarrier there).  Then sx is known, and
//      each CTA writes the int8 codes of its own columns, as fp16 integers, into
//      a shared tile.
//   3. MMAs.  Warp (ks, gl) keeps the codes of K-slice ks (256 columns, all 16
//      rows) in registers and, for the groups gl, gl + 4, ... of a batch, widens
//      the group's int8 weight slice to fp16 integers and runs 16x8x16 fp16 MMAs
//      (fp32 accumulation of integer products: every partial sum of 256
//      columns is below 127^2 * 256 < 2^24, so it is exact).  The four K-slices
//      of a group are added in shared memory, and the CTA's int32 partial of the
//      group goes to the group's owner CTA in the cluster (st.async).
//   4. Outlier product.  Two warps of their own add up X[t,k] W16[n,k] over the
//      CTA's own outlier columns for the batch's channels, in fp32, while the
//      MMAs run; the partial goes to the owner with the int32 one.
//   5. Epilogue.  The owner of a group adds the C partials of each output, scales
//      by (sx/127)(sw/127), adds the outlier product and the bias, and writes Y
//      once.
// With only the int8 weight kept (W16 null) the outlier weights are the codes,
// Wq sw / 127: Y = fp16((acc sx/127 + sum_{k in O} X Wq) sw/127 + b).
// Every wait is bounded; a wait that gives up records BNB_ERR_TIMEOUT in the
// workspace status word and the kernel runs on to its end (Y is then
// unspecified).  Before exiting, every thread waits for its own copies and
// passes one cluster barrier, so no CTA leaves while a peer may store into it.
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "mma_frag.cuh"
#include "sm100_ptx.cuh"

namespace bnb {

namespace {

constexpr int kGvMmaWarps = 16;                              // act pass, MMAs, epilogue
constexpr int kGvOutWarps = 2;                               // outlier product
constexpr int kGvConsumers = kGvMmaWarps * 32;               // 512
constexpr int kGvThreads = (kGvMmaWarps + kGvOutWarps) * 32;  // 576
constexpr int kGvKc = 1024;                                  // columns per CTA
constexpr int kGvKs = 4;                                     // 256-column K-slices
constexpr int kGvGl = kGvMmaWarps / kGvKs;                   // group lanes
constexpr int kGvVec = kGvKc / 8;                            // 8-column vectors per CTA
constexpr int kGvRg = kGvConsumers / kGvVec;                 // row groups of the act pass
constexpr int kGvRpt = 16 / kGvRg;                           // rows per act-pass thread
constexpr int kGvMaxC = 8;                                   // CTAs per cluster
constexpr int kGvMaxG = 16;                                  // 8-channel groups per batch
constexpr int kGvGroupBytes = 8 * kGvKc;                     // one group's weight slice
constexpr int kGvXcBytes = 16 * kGvKc * 2;                   // fp16 codes of 16 rows
constexpr int kGvRedBytes = kGvGl * 2 * kGvKs * 32 * 16;     // K-slice partials
constexpr int kGvPartBytes = 1024;  // one sender's partials of one group: int32 + fp32 [32][4]
static_assert(kGvRpt * kGvRg == 16 && kGvVec * kGvRg == kGvConsumers, "act-pass geometry");
static_assert(kGvOutWarps * 64 >= kGvMaxG * 8, "outlier warps cover a batch, 2 channels a lane");

struct GvArgs {
  const uint4 *X;             // [T x K] 16-bit, as 16-byte vectors
  const uint16_t *X16;        // the same, element bit patterns
  int T;
  int64_t K, N;
  uint32_t thr;               // smallest 16-bit magnitude pattern >= tau
  int C;                      // CTAs per cluster (K-ranges)
  int G;                      // 8-channel groups per batch
  int nbuf;                   // weight buffers (2 when a cluster runs more than one batch)
  int64_t batches;            // ceil(ceil(N / 8) / G)
  int64_t smem_w, smem_xc, smem_red, smem_opart, smem_recv;  // dynamic shared-memory offsets
  const int8_t *Wq;
  const float *sw;
  const uint16_t *W16;        // null: only the int8 weight
  const uint16_t *bias;       // [N] or null
  uint16_t *Y;
  float *sx_out;              // [T]  (CTA 0)
  int32_t *O_out;             // [K]  (cluster 0)
  uint32_t *nO_out;           // [1]  (CTA 0)
  int8_t *dbg_xq;             // [T x K] or null (cluster 0)
  int32_t *dbg_acc;           // [T x N] or null
  int32_t *status;
  int force_timeout;          // test option: CTA 0 waits on `never`, gives up, skips its stores of Y
};

struct GvSmall {
  uint64_t wbar[2][kGvMaxG];  // [buffer][group] the group's weight slice has landed
  uint64_t pbar;              // every CTA's row maxima and outlier count are in pubs
  uint64_t obar;              // the outlier warps have written this batch's outlier partials
  uint64_t rbar[2];           // [receive buffer] every partial of this CTA's groups has landed
  uint64_t fbar[2];           // [receive buffer] every owner has read this CTA's last partials
  uint64_t never;             // completed by nothing (forced-timeout test option)
  float sxs[16];
  uint32_t part[kGvMmaWarps][kGvRpt];  // partial row maxima (16-bit magnitude patterns)
  uint32_t pubs[kGvMaxC][17];          // [CTA][t] its row maxima, [CTA][16] its outlier count
  uint32_t wcnt[kGvVec / 32];          // outlier count of each vector warp of row group 0
  uint8_t fpart[kGvConsumers];         // [row group][vector] outlier flags
  uint16_t ocols[kGvKc];               // the CTA's outlier columns (local), ascending
  int epi_ok;                          // 0: this CTA leaves Y unwritten (forced timeout)
};

// The activation pass's vector -> shared code-tile chunk, and the weight
// tile's: 16-byte chunks are swizzled so that the MMA warps' fragment loads
// hit distinct banks (rows g and g + 1 of a quarter-warp read alternate
// halves of the bank space).
__device__ __forceinline__ uint32_t xc_off(int t, int chunk) {
  return (uint32_t)t * (kGvKc * 2) + (uint32_t)((chunk ^ (t & 1)) * 16);
}
__device__ __forceinline__ uint32_t w_off(int r, int chunk) {  // r: row within a group
  return (uint32_t)r * kGvKc + (uint32_t)((chunk ^ ((r & 1) << 2)) * 16);
}

// cp.async of 16 bytes, zero-filled when `valid` is false (then nothing is
// read); the source must be a valid address either way.
__device__ __forceinline__ void gv_cp16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
// The mbarrier receives one arrival once every cp.async this thread issued
// before has completed (its count must include this arrival).
__device__ __forceinline__ void gv_cp_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void gv_cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Arrival on the mbarrier at cluster address `rbar` of another CTA.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t rbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar)
               : "memory");
}

// Warp `w` puts group g of batch `gb` in flight into weight buffer `buf`:
// 8 rows x the CTA's 1024 columns, 16 bytes per copy, 16 copies per lane;
// rows past N and columns past K are zero-filled.
__device__ __forceinline__ void gv_issue_group(const GvArgs &p, uint8_t *smem, GvSmall &sm,
                                               int64_t kc0, int64_t kcn, int64_t gb, int buf,
                                               int g, int lane) {
  uint8_t *wt = smem + p.smem_w + ((int64_t)buf * p.G + g) * kGvGroupBytes;
  const uint32_t wbase = smem_addr(wt);
  const int64_t n0 = (gb * p.G + g) * 8;
#pragma unroll 4
  for (int i = 0; i < 16; i++) {
    const int idx = lane + 32 * i, r = idx >> 6, chunk = idx & 63;
    const int64_t n = n0 + r;
    const bool valid = n < p.N && chunk * 16 < kcn;
    const int8_t *src = valid ? p.Wq + n * p.K + kc0 + chunk * 16 : p.Wq;
    gv_cp16(wbase + w_off(r, chunk), src, valid);
  }
  gv_cp_arrive(&sm.wbar[buf][g]);
}

template <bool kWq, bool kBf>
__global__ void __launch_bounds__(kGvThreads, 1) gemv_kernel(const GvArgs p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ GvSmall sm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, C = p.C, G = p.G;
  const int64_t K = p.K, N = p.N;
  uint32_t crank;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
  const int64_t cl = blockIdx.x / C, ncl = gridDim.x / C;
  const int64_t kc0 = (int64_t)crank * kGvKc;
  const int64_t kcn = K - kc0 < kGvKc ? (K - kc0 > 0 ? K - kc0 : 0) : kGvKc;  // real columns
  // batches of this cluster: cl, cl + ncl, ...
  const int64_t nbl = p.batches > cl ? (p.batches - cl + ncl - 1) / ncl : 0;
  const int nrecv = nbl > 1 ? 2 : 1;
  const int own_groups = crank < (uint32_t)G ? (G - (int)crank + C - 1) / C : 0;
  uint8_t *xc = smem + p.smem_xc;
  uint8_t *red = smem + p.smem_red;
  float *opart = reinterpret_cast<float *>(smem + p.smem_opart);  // [G][16][8]
  uint8_t *recv = smem + p.smem_recv;  // [nrecv][own][C][int32 512 B, fp32 512 B]
  const int own_max = (G + C - 1) / C;

  if (tid == 0) {
    for (int b = 0; b < 2; b++)
      for (int g = 0; g < kGvMaxG; g++) mbar_init(&sm.wbar[b][g], 32);
    mbar_init(&sm.pbar, 1);
    mbar_init(&sm.obar, kGvOutWarps);
    for (int b = 0; b < 2; b++) {
      mbar_init(&sm.rbar[b], 1);
      mbar_init(&sm.fbar[b], C);
    }
    mbar_init(&sm.never, 1);
    sm.epi_ok = 1;
    mbar_init_fence();
  }
  __syncthreads();
  // The cluster's mbarriers are initialised once every CTA has arrived here;
  // each thread waits for that before its first remote operation.
  cluster_arrive_relaxed();
  // Weight stream of the first batches, ahead of everything else.
  if (warp < G) {
    for (int b = 0; b < p.nbuf && b < nbl; b++)
      gv_issue_group(p, smem, sm, kc0, kcn, cl + b * ncl, b, warp, lane);
  }
  pdl_trigger();  // the next kernel on the stream may launch; it waits for our completion
  pdl_wait();     // X may be the previous kernel's output
  if (blockIdx.x == 0 && tid == 0) *p.status = kDevOk;  // a wait that gives up overwrites it

  bool ok = true;  // this thread's waits all succeeded
  if (warp >= kGvMmaWarps) {
    // ======================= outlier warps =======================
    cluster_wait();
    named_bar_sync(2, kGvThreads);  // the activation pass is done
    int n_own = 0;
    for (int w = 0; w < kGvVec / 32; w++) n_own += (int)sm.wcnt[w];
    const int L = (warp - kGvMmaWarps) * 32 + lane;  // channels 2L, 2L + 1 of a batch
    for (int64_t bl = 0; bl < nbl; bl++) {
      if (n_own > 0) {
        const int64_t gb = cl + bl * ncl;
        const int64_t nb0 = gb * G * 8 + 2 * L;
        const bool on = 2 * L < 8 * G;
        const int g = L >> 2, ch = 2 * (L & 3);
        for (int h = 0; h < 2 && on; h++) {  // tokens 8h .. 8h + 7
          float o[8][2];
#pragma unroll
          for (int t = 0; t < 8; t++) o[t][0] = o[t][1] = 0.f;
          for (int j = 0; j < n_own; j++) {
            const int64_t k = kc0 + sm.ocols[j];
            float w[2];
#pragma unroll
            for (int e = 0; e < 2; e++) {
              const int64_t n = nb0 + e;
              if (n >= N)
                w[e] = 0.f;
              else if (kWq)
                w[e] = (float)p.Wq[n * K + k];
              else
                w[e] = e2f<kBf>(__ldg(p.W16 + n * K + k));
            }
#pragma unroll
            for (int t = 0; t < 8; t++) {
              const int tt = 8 * h + t;
              const float x = tt < T ? e2f<kBf>(__ldg(p.X16 + (int64_t)tt * K + k)) : 0.f;
              o[t][0] = fmaf(x, w[0], o[t][0]);
              o[t][1] = fmaf(x, w[1], o[t][1]);
            }
          }
#pragma unroll
          for (int t = 0; t < 8; t++)
            *reinterpret_cast<float2 *>(opart + (g * 16 + 8 * h + t) * 8 + ch) =
                make_float2(o[t][0], o[t][1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.obar);
      }
      named_bar_sync(2, kGvThreads);  // the batch is done: its outlier partials were read
    }
    gv_cp_wait_all();
    cluster_arrive_relaxed();
    cluster_wait();
    return;
  }

  // ======================= activation pass (512 threads) =======================
  const int v = tid % kGvVec, rg = tid / kGvVec;
  const bool live = v * 8 < kcn;
  uint4 x[kGvRpt];
#pragma unroll
  for (int j = 0; j < kGvRpt; j++) {
    const int t = rg + kGvRg * j;
    x[j] = (t < T && live) ? __ldg(p.X + ((int64_t)t * K + kc0) / 8 + v) : make_uint4(0, 0, 0, 0);
  }
  uint32_t flags = 0;
#pragma unroll
  for (int j = 0; j < kGvRpt; j++) {
    if (rg + kGvRg * j < T) {  // padding rows must not flag columns (tau = 0 flags a zero)
      const uint32_t w4[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
#pragma unroll
      for (int i = 0; i < 4; i++) {
        flags |= (uint32_t)(abs_bits_lo(w4[i]) >= p.thr) << (2 * i);
        flags |= (uint32_t)(abs_bits_hi(w4[i]) >= p.thr) << (2 * i + 1);
      }
    }
  }
  if (!live) flags = 0;
  sm.fpart[rg * kGvVec + v] = (uint8_t)flags;
  named_bar_sync(1, kGvConsumers);
  flags = 0;
  if (live)
#pragma unroll
    for (int r = 0; r < kGvRg; r++) flags |= sm.fpart[r * kGvVec + v];
#pragma unroll
  for (int j = 0; j < kGvRpt; j++) {
    const uint32_t w4[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      if (!((flags >> (2 * i)) & 1)) m = max(m, abs_bits_lo(w4[i]));
      if (!((flags >> (2 * i + 1)) & 1)) m = max(m, abs_bits_hi(w4[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) sm.part[warp][j] = m;
  }
  if (rg == 0) {  // row group 0 holds each of the CTA's columns once
    uint32_t c = __popc(flags);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) sm.wcnt[warp] = c;
  }
  named_bar_sync(1, kGvConsumers);
  cluster_wait();  // every CTA's mbarriers are initialised
  if (tid < 17) {
    // row t's maximum over this CTA's non-outlier columns (t < 16), or its
    // outlier count (16), stored into every CTA of the cluster
    uint32_t val = 0;
    if (tid < 16) {
      const int r = tid % kGvRg, j = tid / kGvRg;
#pragma unroll
      for (int w = 0; w < kGvVec / 32; w++) val = max(val, sm.part[r * (kGvVec / 32) + w][j]);
    } else {
#pragma unroll
      for (int w = 0; w < kGvVec / 32; w++) val += sm.wcnt[w];
    }
    const uint32_t dst = smem_addr(&sm.pubs[crank][tid]), bar = smem_addr(&sm.pbar);
    for (int c = 0; c < C; c++) st_async_b32(mapa(dst, c), val, mapa(bar, c));
    if (tid == 0) mbar_expect_tx(&sm.pbar, (uint32_t)C * 17u * 4u);
  }
  ok = mbar_wait_cluster_bounded(&sm.pbar, 0, p.status);
  uint32_t nO = 0, base = 0;
  for (int c = 0; c < C; c++) {
    const uint32_t n = sm.pubs[c][16];
    nO += n;
    if (c < (int)crank) base += n;
  }
  // codes of this thread's rows: fp16 integers in the shared tile (zeros in
  // outlier columns, past K and in rows >= T)
#pragma unroll
  for (int j = 0; j < kGvRpt; j++) {
    const int t = rg + kGvRg * j;
    uint32_t m = 0;
    for (int c = 0; c < C; c++) m = max(m, sm.pubs[c][t]);
    const RowCode<kBf> rc(e2f<kBf>(t < T ? m : 0u));
    const uint32_t w4[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
    uint32_t p0 = 0, p1 = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const uint32_t c0 = ((flags >> (2 * i)) & 1) ? 0u : rc.byte(e2f<kBf>(w4[i] & 0xffffu));
      const uint32_t c1 = ((flags >> (2 * i + 1)) & 1) ? 0u : rc.byte(e2f<kBf>(w4[i] >> 16));
      const uint32_t two = (c0 & 0xffu) | ((c1 & 0xffu) << 8);
      if (i < 2)
        p0 |= two << (16 * i);
      else
        p1 |= two << (16 * (i - 2));
    }
    if (t >= T || !live) p0 = p1 = 0;
    uint4 h;
    s8x4_to_f16x4(p0, h.x, h.y);
    s8x4_to_f16x4(p1, h.z, h.w);
    *reinterpret_cast<uint4 *>(xc + xc_off(t, v)) = h;
    if (p.dbg_xq && blockIdx.x < (unsigned)C && t < T && live)
      *reinterpret_cast<uint2 *>(p.dbg_xq + (int64_t)t * K + kc0 + 8 * v) = make_uint2(p0, p1);
  }
  if (rg == 0) {  // the CTA's outlier columns, ascending: by vector warp, lane, bit
    const uint32_t pc = __popc(flags);
    uint32_t incl = pc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    uint32_t pos = incl - pc;
    for (int w = 0; w < warp; w++) pos += sm.wcnt[w];
    for (int b = 0; b < 8; b++)
      if ((flags >> b) & 1) {
        sm.ocols[pos] = (uint16_t)(8 * v + b);
        if (blockIdx.x < (unsigned)C) p.O_out[base + pos] = (int32_t)(kc0 + 8 * v + b);
        ++pos;
      }
  }
  if (tid < 16) {
    uint32_t m = 0;
    for (int c = 0; c < C; c++) m = max(m, sm.pubs[c][tid]);
    sm.sxs[tid] = e2f<kBf>(tid < T ? m : 0u);
    if (blockIdx.x == 0 && tid < T) p.sx_out[tid] = sm.sxs[tid];
  }
  if (blockIdx.x == 0 && tid == 0) *p.nO_out = nO;
  // forced-timeout test option: one wait on a barrier that nothing completes
  if (p.force_timeout && blockIdx.x == 0 && tid == 0 &&
      !mbar_wait_bounded(&sm.never, 0, p.status, kForcedWaitNs))
    sm.epi_ok = 0;
  named_bar_sync(2, kGvThreads);  // codes, outlier list and scales are in place

  // ======================= MMA warps =======================
  const int ks = warp & (kGvKs - 1), gl = warp / kGvKs;
  const int g8 = lane >> 2, q = lane & 3;
  const bool slice_live = ks * 256 < kcn;
  int n_own = 0;
  for (int w = 0; w < kGvVec / 32; w++) n_own += (int)sm.wcnt[w];
  // codes of K-slice ks, rows g8 and g8 + 8, in registers for the whole call
  uint32_t xa[4][8], xb[4][8];
#pragma unroll
  for (int b = 0; b < 4; b++) {
    const int c0 = 32 * ks + 8 * b + 2 * q;
    const uint4 a0 = *reinterpret_cast<const uint4 *>(xc + xc_off(g8, c0));
    const uint4 a1 = *reinterpret_cast<const uint4 *>(xc + xc_off(g8, c0 + 1));
    const uint4 b0 = *reinterpret_cast<const uint4 *>(xc + xc_off(g8 + 8, c0));
    const uint4 b1 = *reinterpret_cast<const uint4 *>(xc + xc_off(g8 + 8, c0 + 1));
    xa[b][0] = a0.x; xa[b][1] = a0.y; xa[b][2] = a0.z; xa[b][3] = a0.w;
    xa[b][4] = a1.x; xa[b][5] = a1.y; xa[b][6] = a1.z; xa[b][7] = a1.w;
    xb[b][0] = b0.x; xb[b][1] = b0.y; xb[b][2] = b0.z; xb[b][3] = b0.w;
    xb[b][4] = b1.x; xb[b][5] = b1.y; xb[b][6] = b1.z; xb[b][7] = b1.w;
  }
  // senders whose outlier partials come with their int32 ones
  uint32_t fsend = 0, recv_bytes = 0;
  for (int c = 0; c < C; c++) {
    const bool f = sm.pubs[c][16] > 0;
    fsend |= (uint32_t)f << c;
    recv_bytes += f ? 1024u : 512u;
  }
  uint32_t itg = 0;  // groups this group lane has done, over all batches
  for (int64_t bl = 0; bl < nbl; bl++) {
    const int buf = (int)(bl % p.nbuf), rbuf = (int)(bl % nrecv);
    const int64_t gb = cl + bl * ncl;
    if (tid == 0 && own_groups > 0)
      mbar_expect_tx(&sm.rbar[rbuf], (uint32_t)own_groups * recv_bytes);
    const uint32_t wpar = (uint32_t)(bl / p.nbuf) & 1u;
    for (int g = gl; g < G; g += kGvGl, ++itg) {
      float f[4] = {0.f, 0.f, 0.f, 0.f};
      ok = mbar_wait_bounded(&sm.wbar[buf][g], wpar, p.status) && ok;
      if (slice_live) {
        const uint8_t *wt = smem + p.smem_w + ((int64_t)buf * G + g) * kGvGroupBytes;
#pragma unroll
        for (int b = 0; b < 4; b++) {
          const uint4 wv = *reinterpret_cast<const uint4 *>(wt + w_off(g8, 16 * ks + 4 * b + q));
          uint32_t h[8];
          s8x4_to_f16x4(wv.x, h[0], h[1]);
          s8x4_to_f16x4(wv.y, h[2], h[3]);
          s8x4_to_f16x4(wv.z, h[4], h[5]);
          s8x4_to_f16x4(wv.w, h[6], h[7]);
#pragma unroll
          for (int mm = 0; mm < 4; mm++)
            mma_f16_16x8x16(f, xa[b][2 * mm], xb[b][2 * mm], xa[b][2 * mm + 1],
                            xb[b][2 * mm + 1], h[2 * mm], h[2 * mm + 1]);
        }
      }
      // the four K-slices of the group meet in shared memory (two slots per
      // group lane, alternating, so one barrier per group suffices)
      int4 *slot = reinterpret_cast<int4 *>(red + ((gl * 2 + (itg & 1)) * kGvKs) * 512);
      slot[ks * 32 + lane] = make_int4(__float2int_rn(f[0]), __float2int_rn(f[1]),
                                       __float2int_rn(f[2]), __float2int_rn(f[3]));
      named_bar_sync(3 + gl, kGvKs * 32);
      if (ks == (int)(itg & (kGvKs - 1))) {
        int4 s = slot[lane];
#pragma unroll
        for (int k2 = 1; k2 < kGvKs; k2++) {
          const int4 u = slot[k2 * 32 + lane];
          s.x += u.x; s.y += u.y; s.z += u.z; s.w += u.w;
        }
        const int owner = g % C, og = g / C;
        if (nrecv == 2 && bl >= 2)  // the owner has read what this CTA sent two batches ago
          ok = mbar_wait_cluster_bounded(&sm.fbar[rbuf], (uint32_t)((bl - 2) / 2) & 1u, p.status) && ok;
        uint8_t *slotp = recv + (((int64_t)rbuf * own_max + og) * C + crank) * kGvPartBytes;
        const uint32_t dst = mapa(smem_addr(slotp + lane * 16), (uint32_t)owner);
        const uint32_t rb = mapa(smem_addr(&sm.rbar[rbuf]), (uint32_t)owner);
        st_async_v4(dst, (uint32_t)s.x, (uint32_t)s.y, (uint32_t)s.z, (uint32_t)s.w, rb);
        if (n_own > 0) {
          ok = mbar_wait_bounded(&sm.obar, (uint32_t)bl & 1u, p.status) && ok;
          const float *op = opart + g * 128;
          const float o0 = op[g8 * 8 + 2 * q], o1 = op[g8 * 8 + 2 * q + 1];
          const float o2 = op[(g8 + 8) * 8 + 2 * q], o3 = op[(g8 + 8) * 8 + 2 * q + 1];
          st_async_v4(dst + 512, __float_as_uint(o0), __float_as_uint(o1), __float_as_uint(o2),
                      __float_as_uint(o3), rb);
        }
      }
    }
    // the batch is done: its weight buffer and outlier partials may be reused
    named_bar_sync(2, kGvThreads);
    if (warp < G && bl + p.nbuf < nbl)
      gv_issue_group(p, smem, sm, kc0, kcn, gb + p.nbuf * ncl, buf, warp, lane);
    // ---- epilogue: this CTA's groups g = crank, crank + C, ... ----
    if (warp < own_groups) {
      const int og = warp, g = og * C + (int)crank;
      ok = mbar_wait_cluster_bounded(&sm.rbar[rbuf], (uint32_t)(bl / nrecv) & 1u, p.status) && ok;
      int4 acc = make_int4(0, 0, 0, 0);
      float o[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = 0; c < C; c++) {
        const uint8_t *sp = recv + (((int64_t)rbuf * own_max + og) * C + c) * kGvPartBytes;
        const int4 u = *reinterpret_cast<const int4 *>(sp + lane * 16);
        acc.x += u.x; acc.y += u.y; acc.z += u.z; acc.w += u.w;
        if ((fsend >> c) & 1) {
          const float4 fo = *reinterpret_cast<const float4 *>(sp + 512 + lane * 16);
          o[0] += fo.x; o[1] += fo.y; o[2] += fo.z; o[3] += fo.w;
        }
      }
      const int accs[4] = {acc.x, acc.y, acc.z, acc.w};
      const int64_t nbase = (gb * G + g) * 8 + 2 * q;
      float sn[2], bn[2];
#pragma unroll
      for (int e = 0; e < 2; e++) {
        const int64_t n = nbase + e;
        sn[e] = n < N ? __ldg(p.sw + n) / 127.0f : 0.f;
        bn[e] = (n < N && p.bias) ? e2f<kBf>(__ldg(p.bias + n)) : 0.f;
      }
      float yv[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int t = g8 + 8 * (i >> 1);
        const float st = sm.sxs[t] / 127.0f;
        yv[i] = kWq ? fmaf(fmaf((float)accs[i], st, o[i]), sn[i & 1], bn[i & 1])
                    : fmaf((float)accs[i] * st, sn[i & 1], o[i] + bn[i & 1]);
      }
      if (sm.epi_ok) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
          const int t = g8 + 8 * h;
          if (t >= T) continue;
          uint16_t *yr = p.Y + (int64_t)t * N;
          if (nbase + 1 < N && ((t * N) & 1) == 0) {
            *reinterpret_cast<uint32_t *>(yr + nbase) = f2e2<kBf>(yv[2 * h], yv[2 * h + 1]);
          } else {
            if (nbase < N) yr[nbase] = f2e<kBf>(yv[2 * h]);
            if (nbase + 1 < N) yr[nbase + 1] = f2e<kBf>(yv[2 * h + 1]);
          }
          if (p.dbg_acc) {
            if (nbase < N) p.dbg_acc[(int64_t)t * N + nbase] = accs[2 * h];
            if (nbase + 1 < N) p.dbg_acc[(int64_t)t * N + nbase + 1] = accs[2 * h + 1];
          }
        }
      }
    }
    if (nrecv == 2 && bl + 2 < nbl) {
      // this CTA's receive buffer rbuf is read: let every sender reuse it
      named_bar_sync(1, kGvConsumers);
      if (tid < C) mbar_arrive_remote(mapa(smem_addr(&sm.fbar[rbuf]), (uint32_t)tid));
    }
  }
  (void)ok;
  gv_cp_wait_all();
  cluster_arrive_relaxed();
  cluster_wait();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Shared memory of one CTA (the largest plan: one buffer of 16 groups, or two
// of 8) and the per-plan carve.
constexpr size_t kGvSmemMax = 212 * 1024;

struct GvPlan {
  int C, G, nbuf, nrecv;
  int64_t batches, ncl;
  size_t smem;
  int64_t off_w, off_xc, off_red, off_opart, off_recv;
};

using GvKern = void (*)(GvArgs);
const GvKern kGvKerns[4] = {gemv_kernel<false, false>, gemv_kernel<true, false>,
                            gemv_kernel<false, true>, gemv_kernel<true, true>};

// Clusters of C CTAs resident at once (one CTA per SM at this shared memory),
// queried once per device; the nominal B300 count when no device answers.
int gv_max_clusters(int dev, int C) {
  static std::atomic<int> cache[64][kGvMaxC + 1];
  if (dev >= 0 && dev < 64) {
    const int v = cache[dev][C].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int least = 1 << 30;
  for (GvKern f : kGvKerns) {
    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGvSmemMax) !=
        cudaSuccess) {
      least = 0;
      break;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(C * 16));
    cfg.blockDim = dim3(kGvThreads);
    cfg.dynamicSmemBytes = kGvSmemMax;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) n = 0;
    least = n < least ? n : least;  // every form must fit
  }
  (void)cudaGetLastError();  // a failed query is not a launch error
  if (least <= 0) least = kB300Sms / C;
  if (dev >= 0 && dev < 64) cache[dev][C].store(least, std::memory_order_relaxed);
  return least;
}

GvPlan gv_plan(int dev, int64_t N, int64_t K, int want_c) {
  GvPlan pl;
  const int cmin = (int)((K + kGvKc - 1) / kGvKc);
  pl.C = (want_c >= cmin && want_c <= kGvMaxC) ? want_c : cmin;
  const int64_t groups = (N + 7) / 8;
  const int64_t maxcl = gv_max_clusters(dev, pl.C);
  if (groups <= maxcl * kGvMaxG) {  // every channel in flight at once
    pl.G = (int)((groups + maxcl - 1) / maxcl);
    pl.nbuf = 1;
    pl.batches = (groups + pl.G - 1) / pl.G;
    pl.ncl = pl.batches;
  } else {  // batches of at most 8 groups, two weight buffers, balanced over the clusters
    const int64_t per = (groups + maxcl * 8 - 1) / (maxcl * 8);
    pl.G = (int)((groups + maxcl * per - 1) / (maxcl * per));
    pl.nbuf = 2;
    pl.batches = (groups + pl.G - 1) / pl.G;
    pl.ncl = maxcl < pl.batches ? maxcl : pl.batches;
  }
  pl.nrecv = pl.batches > pl.ncl ? 2 : 1;
  const int own_max = (pl.G + pl.C - 1) / pl.C;
  int64_t off = 0;
  pl.off_w = off;
  off += (int64_t)pl.nbuf * pl.G * kGvGroupBytes;
  pl.off_xc = off;
  off += kGvXcBytes;
  pl.off_red = off;
  off += kGvRedBytes;
  pl.off_opart = off;
  off += (int64_t)pl.G * 512;
  pl.off_recv = off;
  off += (int64_t)pl.nrecv * own_max * pl.C * kGvPartBytes;
  pl.smem = (size_t)off;
  return pl;
}

}  // namespace

cudaError_t launch_decode(const void *X, int64_t T, int64_t K, uint32_t thr, const int8_t *Wq,
                          const float *sw, const void *W16, const void *bias, int64_t N,
                          bool bf16, void *Y, const Workspace &ws, int8_t *dbg_xq,
                          int32_t *dbg_acc, uint32_t opts, cudaStream_t stream) {
  if (T < 1 || T > 16 || K > kDecodeMaxK) return cudaErrorInvalidValue;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const GvPlan pl = gv_plan(dev, N, K, (int)((opts >> 8) & 0xffu));
  if (pl.smem > kGvSmemMax) return cudaErrorInvalidValue;
  GvArgs a;
  a.X = reinterpret_cast<const uint4 *>(X);
  a.X16 = reinterpret_cast<const uint16_t *>(X);
  a.T = (int)T;
  a.K = K;
  a.N = N;
  a.thr = thr;
  a.C = pl.C;
  a.G = pl.G;
  a.nbuf = pl.nbuf;
  a.batches = pl.batches;
  a.smem_w = pl.off_w;
  a.smem_xc = pl.off_xc;
  a.smem_red = pl.off_red;
  a.smem_opart = pl.off_opart;
  a.smem_recv = pl.off_recv;
  a.Wq = Wq;
  a.sw = sw;
  a.W16 = reinterpret_cast<const uint16_t *>(W16);
  a.bias = reinterpret_cast<const uint16_t *>(bias);
  a.Y = reinterpret_cast<uint16_t *>(Y);
  a.sx_out = ws.sx;
  a.O_out = ws.O;
  a.nO_out = ws.counters + 1;
  a.dbg_xq = dbg_xq;
  a.dbg_acc = dbg_acc;
  a.status = ws.status;
  a.force_timeout = (opts & BNB_OPT_FORCE_TIMEOUT) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.ncl * pl.C));
  cfg.blockDim = dim3(kGvThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)pl.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (opts & BNB_OPT_NO_PDL) ? 1 : 2;
  const int form = (W16 == nullptr ? 1 : 0) | (bf16 ? 2 : 0);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kGvKerns[form], a);
  note_launch();
  return e;
}

}  // namespace bnb
