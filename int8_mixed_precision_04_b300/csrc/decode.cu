// The whole layer for decode-sized T (T <= 16) in one kernel launch per wave
// of channels (at most three): for T <= 5 (T <= 6 at K > 2048) dec_local
// (below the clustered kernel), where every CTA runs the whole activation
// pass itself, otherwise dec_fused.
//
// dec_fused: one CTA per slice of at most 40 output channels (one CTA per
// SM), in thread-block clusters of kC CTAs (16, 8 or 4 where T K <= 32768,
// else 8, 16 or 4: the first whose resident clusters hold every slice at
// once).  Right behind its X loads the
// producer warp puts the CTA's whole int8 weight slice in flight on the copy
// engine (one bulk copy per row).  While the weight streams in, the cluster
// runs the activation pass cooperatively, so that no second kernel and no
// inter-kernel dependency sits on the path, and no CTA repeats the others'
// work:
//   - CTA rank c owns 1/kC of the columns; each consumer thread one 8-column
//     vector of 16/kC rows.  A column is an outlier feature dimension when
//     |x| >= tau in some row ("Hugging Face Quantization with bitsandbytes:
//     4-bit & 8-bit Models Explained", sections 2 and 3): the row groups'
//     flags are OR-ed through shared memory.  Each CTA's row maxima over its
//     non-outlier columns and its outlier count go to every CTA of the
//     cluster;
//   - each CTA then sends its columns' vector-wise int8 codes
//     rint(fl32(127 x) / sx), its part of the outlier column mask and the X
//     values of the first outlier columns to every CTA of the cluster.
// Every exchange is a remote store into the receiving CTA's shared memory
// counted on an mbarrier there (no cluster-wide barrier: its release would
// wait for the weight copies in flight).  CTA 0 also writes sx, O and |O| to
// the workspace (and the codes when asked), for the debug entry point.
// Then each consumer warp owns one K-range for all of the slice's 8-channel
// groups: it widens the int8 codes of X and W to fp16 integers in registers
// and runs 16x8x16 fp16 MMAs with fp32 accumulation, converted to int32 at
// least every 1024 columns (127^2 * 1024 < 2^24, so every fp32 partial sum is
// an exact integer).  The producer warp lists the outlier columns and adds up
// the first ones of W16 times X for the slice while the MMAs run; the
// consumers split any further ones.  Epilogue (one output per consumer
// thread): the int32 partials are summed, scaled by (sx/127)(sw/127), the
// 16-bit outlier product is added ("converted back to 16-bit at the end",
// same page, section 2), then the bias if any, and Y is written once.
// With only the int8 weight kept (W16 null) the outlier weights are the
// slice's own codes, already in shared memory: Y = fp16((acc sx/127 +
// sum_{k in O} X Wq) sw/127 + b), and no W16 byte is read.
#include <atomic>
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"
#include "mma_frag.cuh"
#include "sm100_ptx.cuh"

namespace bnb {

constexpr int kDecWarps = 16;                      // consumer warps (one K-range each)
constexpr int kDecConsumers = kDecWarps * 32;      // consumer threads
constexpr int kDecThreads = kDecConsumers + 32;    // + one producer warp
constexpr int kDecGroups = 5;                      // 8-channel MMA groups of a slice, at most
constexpr int kDecMaxRows = kDecGroups * 8;        // output channels per CTA, at most
constexpr int kDecChunkK = 1024;                   // fp32 accumulation is drained this often
constexpr int kDecOutSmall = 8;                    // outlier columns of W16 fetched by TMA
constexpr int kDecRedStride = kDecGroups * 4 + 1;  // words per lane in the reduction (odd)
constexpr int kDecMaskWords = (int)(kDecodeMaxK / 32);

// Activation-pass geometry of a cluster of kC CTAs: a CTA covers at most
// kVpc 8-column vectors; consumer thread i takes vector i % kVpc of rows
// i / kVpc + kC * j (j < kRpt), so warp w holds vector block w % kWpg of row
// group w / kWpg.
template <int kC>
struct DecAct {
  static constexpr int kVpc = kDecConsumers / kC;  // 32, 64, 128 for kC 16, 8, 4
  static constexpr int kRpt = 16 / kC;             // rows per thread
  static constexpr int kWpg = kVpc / 32;           // warps per row group
  static_assert(kVpc % 32 == 0 && kRpt >= 1 && kRpt <= 4 && kWpg <= 4, "act-pass geometry");
  static_assert(kDecodeMaxK <= kC * kVpc * 8, "act-pass threads cover every column");
};

__host__ __device__ constexpr int64_t dec_pitch(int64_t K) { return K + 64; }  // bytes per row
// K columns of MMA warp w: [w * range, min(K, (w + 1) * range)), range a multiple of 64
__host__ __device__ constexpr int64_t dec_range(int64_t K) {
  return ((K + kDecWarps - 1) / kDecWarps + 63) / 64 * 64;
}
// The weight region is reused for the cross-warp reduction after the main loop.
constexpr int64_t kDecRedBytes = (int64_t)kDecWarps * 32 * kDecRedStride * 4;
__host__ __device__ constexpr int64_t dec_wregion(int64_t K, int64_t rows) {
  return rows * dec_pitch(K) > kDecRedBytes ? rows * dec_pitch(K) : kDecRedBytes;
}
__host__ __device__ constexpr int64_t dec_ocap(int64_t K) { return (K + 7) / 8 * 8; }

// dynamic: weight rows, code rows (xrows: 8 when T <= 8, else 16), outlier
// column list (uint16).  The MMAs also read the (unused) rows past `rows` of a
// partial 8-channel group: at most 7 rows, which land in the code rows.
size_t decode_smem_bytes(int64_t K, int64_t rows, int64_t xrows = 16) {
  return (size_t)(dec_wregion(K, rows) + xrows * dec_pitch(K) + 2 * dec_ocap(K));
}
constexpr int64_t dec_xrows(int64_t T) { return T <= 8 ? 8 : 16; }

// small static buffers of one CTA (partly written by the other CTAs of its cluster)
struct DecSmall {
  uint64_t wbar;            // the CTA's weight slice has landed
  uint64_t wobar;           // W16 at the first outlier columns is in wos
  uint64_t pbar;            // every CTA's row maxima and outlier count are in pubs
  uint64_t cbar;            // every CTA's codes and outlier-mask words are here
  uint64_t xbar;            // the first outlier columns and their X values are here
  uint64_t lbar;            // the producer warp has listed every outlier column
  uint64_t never;           // completed by nothing (forced-timeout test option)
  // [j][row][8]: W16[n0 + row, 8 (O[j] / 8) .. + 8), one TMA box per outlier column j
  alignas(128) uint16_t wos[kDecOutSmall][kDecMaxRows][8];
  float sxs[16];            // row scales sx
  uint32_t part[kDecWarps * 4];  // [warp][j] partial row maxima (fp16 bits)
  uint32_t pubs[16][17];    // [CTA][t] its row maxima (fp16 bits), [CTA][16] its outlier count
  uint32_t wcnt[4];         // outlier count of each vector block (row group 0's warps)
  uint32_t mask[kDecMaskWords];  // outlier columns, bit b of word w = column 32 w + b
  uint8_t fpart[kDecConsumers];  // [row group][vector] outlier flags
  uint32_t xo[16 * kDecOutSmall];  // [t][j] X at the first outlier columns (fp16 bits)
  uint32_t oc[kDecOutSmall];       // the first outlier columns
  uint16_t bias[kDecMaxRows];      // the slice's fp16 bias (written before wobar's arrival)
};

struct DecArgs {
  const uint4 *X;              // [T x K] fp16 as 16-byte vectors
  const unsigned short *X16;   // the same, as fp16 bit patterns
  int T;
  int64_t K, N;
  uint32_t thr;                // smallest fp16 magnitude bits >= tau
  int64_t n_base, n_end;       // this launch's output channels [n_base, n_end) of N
  int reset_status;            // the call's first launch: clears the status word
  int64_t rows_per_cta;        // <= kDecMaxRows
  int xrows;                   // code rows held: dec_xrows(T)
  int64_t wregion;             // bytes of the weight region, dec_wregion(K, rows_per_cta)
  const int8_t *Wq;
  const float *sw;
  const unsigned short *W16;
  const unsigned short *bias;  // [N] fp16 or null
  uint16_t *Y;                 // [T x N] fp16 or bf16 bits
  float *sx_out;               // [T]  (CTA 0)
  int32_t *O_out;              // [K]  (CTA 0)
  uint32_t *nO_out;            // [1]  (CTA 0)
  int8_t *dbg_xq;              // [T x K] or null (CTA 0)
  int32_t *dbg_acc;            // [T x N] or null
  int32_t *status;
  int force_timeout;           // test option: CTA 0's consumers give up after a wait on `never`
};

// Every thread of every CTA of the cluster passes this once before it exits,
// on every path: no CTA leaves while a peer may still store into it.
__device__ __forceinline__ void dec_cluster_exit() {
  cluster_arrive_relaxed();
  cluster_wait();
}

// 16 int8 codes (one 16-byte vector) -> 16 fp16 integers in 8 words.
__device__ __forceinline__ void widen16(const uint4 &v, uint32_t (&h)[8]) {
  s8x4_to_f16x4(v.x, h[0], h[1]);
  s8x4_to_f16x4(v.y, h[2], h[3]);
  s8x4_to_f16x4(v.z, h[4], h[5]);
  s8x4_to_f16x4(v.w, h[6], h[7]);
}

// One consumer warp's K-range [k0, k1) for the slice's first `ng` 8-channel
// groups, into exact int32 accumulators.  Fragment convention (see
// mma_frag.cuh): lane (g = lane/4, q = lane%4) holds columns
// [kb + 16q, kb + 16q + 16) of X rows g and g+8 and of weight row g of a
// group; word pair (2mm, 2mm+1) of each widened vector feeds MMA mm.
// kRagged: the range ends inside a 64-column block, whose columns past k1
// (never written in shared memory) are fed as zeros; otherwise no lane needs
// a mask.
// xhi: the code row the MMA's rows 8..15 read, row g + 8 when those rows
// are held (T > 8); with the 8-row code region it is row g again, whose
// products land in rows that no token reads.
template <bool kRagged>
__device__ __forceinline__ void dec_mma_range(const uint8_t *xs, const uint8_t *xhi,
                                              const uint8_t *ws, int64_t pitch, int g, int q,
                                              int64_t k0, int64_t k1, int ng,
                                              int (&acc)[kDecGroups][4]) {
  float f[kDecGroups][4] = {};
  int nb = 0;
  for (int64_t kb = k0; kb < k1; kb += 64) {
    const uint32_t lv = (!kRagged || kb + 16 * q < k1) ? 0xffffffffu : 0u;
    uint32_t xa[8], xb[8];
    widen16(*reinterpret_cast<const uint4 *>(xs + g * pitch + kb + 16 * q), xa);
    widen16(*reinterpret_cast<const uint4 *>(xhi + kb + 16 * q), xb);
#pragma unroll
    for (int gi = 0; gi < kDecGroups; gi++) {
      if (gi < ng) {
        uint32_t h[8];
        widen16(*reinterpret_cast<const uint4 *>(ws + (gi * 8 + g) * pitch + kb + 16 * q), h);
#pragma unroll
        for (int mm = 0; mm < 4; mm++)
          mma_f16_16x8x16(f[gi], xa[2 * mm] & lv, xb[2 * mm] & lv, xa[2 * mm + 1] & lv,
                          xb[2 * mm + 1] & lv, h[2 * mm] & lv, h[2 * mm + 1] & lv);
      }
    }
    if (++nb == kDecChunkK / 64 || kb + 64 >= k1) {  // exact drain into int32
      nb = 0;
#pragma unroll
      for (int gi = 0; gi < kDecGroups; gi++)
#pragma unroll
        for (int j = 0; j < 4; j++) {
          acc[gi][j] += __float2int_rn(f[gi][j]);
          f[gi][j] = 0.f;
        }
    }
  }
}

// kWq: only the int8 weight is kept (W16 null); kBf: X, W16, bias and Y are bf16
template <int kC, bool kWq, bool kBf>
__global__ void __launch_bounds__(kDecThreads, 1)
    dec_fused_kernel(const __grid_constant__ CUtensorMap tm_w16, const DecArgs p) {
  using G = DecAct<kC>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int64_t K = p.K, pitch = dec_pitch(K), range = dec_range(K);
  uint8_t *ws = smem;                                          // [rows][pitch] weight codes
  uint8_t *xs = smem + p.wregion;                              // [xrows][pitch] activation codes
  uint16_t *ocols = reinterpret_cast<uint16_t *>(xs + p.xrows * pitch);  // outlier columns
  __shared__ DecSmall sm;
  float *sxs = sm.sxs;
  uint32_t *red = reinterpret_cast<uint32_t *>(smem);  // [16 warps][32][21], after the main loop

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T;
  const int64_t n0 = p.n_base + (int64_t)blockIdx.x * p.rows_per_cta;
  const int64_t rows = min(p.n_end, n0 + p.rows_per_cta) - n0;  // <= 40; <= 0 for trailing CTAs

  if (warp == kDecWarps && lane == 0) {
    mbar_init(&sm.wbar, 1);
    mbar_init(&sm.wobar, 1);
    mbar_init(&sm.pbar, 1);
    mbar_init(&sm.cbar, 1);
    mbar_init(&sm.xbar, 1);
    mbar_init(&sm.lbar, 32);
    mbar_init(&sm.never, 1);
    mbar_init_fence();
  }
  __syncthreads();
  // The cluster's mbarriers are initialised once every CTA has arrived here;
  // each thread waits for that just before its first remote store.  No
  // thread publishes anything through this phase, so the arrival is relaxed
  // (a release arrival would also wait for the CTA's copies in flight).
  cluster_arrive_relaxed();
  // the next kernel on the stream may launch now; it waits for our completion
  pdl_trigger();
  // X may be the output of the previous kernel on the stream
  pdl_wait();
  // a wait that gives up overwrites it (a later launch of the same call keeps it)
  if (p.reset_status && blockIdx.x == 0 && threadIdx.x == 0) *p.status = kDevOk;

  uint32_t crank;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));

  const int64_t vecs = K / 8;
  // vectors per CTA (<= kVpc), a multiple of 4 so that each outlier-mask word
  // (four vectors) belongs to one CTA
  const int64_t vpc = ((vecs + kC - 1) / kC + 3) / 4 * 4;
  const int64_t words = (vecs + 3) / 4;  // outlier-mask words
  const int grp = (threadIdx.x & (kDecConsumers - 1)) / G::kVpc;  // row group (consumers)
  const int64_t vl = threadIdx.x % G::kVpc;
  const int64_t v = crank * vpc + vl;          // this thread's 8-column vector
  const bool live = warp < kDecWarps && vl < vpc && v < vecs;
  if (warp == kDecWarps) {
    // The whole weight slice in flight at once, on the copy engine: one bulk
    // copy per weight row, so that every warp is free for the activation
    // pass while the slice streams in.  It goes out right behind the X loads,
    // so that the few X bytes on the critical path do not queue behind the
    // weights.  Weight rows past `rows`, code rows past T and the pads past K
    // are never written: the MMAs mask columns past K, and accumulator rows
    // >= T or columns >= rows are never stored.
    named_bar_sync(2, kDecThreads);  // X loads issued
    // the slice's bias (rows <= 40: two per lane), loaded ahead of the weight
    // stream and stored once the copies are out; lane 0's arrival on wobar
    // below publishes it to the epilogue
    uint16_t bv[2] = {0, 0};
    if (p.bias)
#pragma unroll
      for (int i = 0; i < 2; i++)
        if (lane + 32 * i < rows) bv[i] = __ldg(p.bias + n0 + lane + 32 * i);
    if (lane == 0) mbar_expect_tx(&sm.wbar, (uint32_t)(rows > 0 ? rows * K : 0));
    __syncwarp();
    const uint64_t pol = l2_evict_first_policy();  // the slice is read once per call
    for (int64_t r = lane; r < rows; r += 32)
      bulk_g2s_once(ws + r * pitch, p.Wq + (n0 + r) * K, (uint32_t)K, &sm.wbar, pol);
#pragma unroll
    for (int i = 0; i < 2; i++)
      if (lane + 32 * i < kDecMaxRows) sm.bias[lane + 32 * i] = bv[i];
    __syncwarp();
    cluster_wait();
    // W16 at the first outlier columns for this slice, as soon as the columns
    // are known: one TMA box (8 columns x the slice's channels) per column.
    // The copy engine serves these right behind the weight slice; plain loads
    // issued now would wait behind the weight stream and the exchange traffic
    // for several microseconds.  Then the whole ascending outlier list from
    // the mask.  The consumers' waits are bounded, so wobar and lbar are
    // signalled even after a wait gave up.
    bool ok = mbar_wait_cluster_bounded(&sm.pbar, 0, p.status);
    int32_t nO = 0;
    if (ok)
#pragma unroll
      for (int c = 0; c < kC; c++) nO += (int32_t)sm.pubs[c][16];
    const int32_t nsmall = min(nO, kDecOutSmall);
    if (rows > 0) {
      // (without W16 the consumers read the outlier weights from the slice)
      const bool fetch = !kWq && ok && nsmall > 0 &&
                         mbar_wait_cluster_bounded(&sm.xbar, 0, p.status);
      if (lane == 0)
        mbar_expect_tx(&sm.wobar, fetch ? (uint32_t)(nsmall * 16 * p.rows_per_cta) : 0u);
      __syncwarp();
      if (fetch && lane < nsmall)
        tma_load_2d(&sm.wos[lane][0][0], &tm_w16, (int32_t)(sm.oc[lane] & ~7u), (int32_t)n0,
                    &sm.wobar);
    }
    ok = ok && mbar_wait_cluster_bounded(&sm.cbar, 0, p.status);
    if (ok) {
      const int64_t wpl = (words + 31) / 32;
      const int64_t w0 = min(words, lane * wpl), w1 = min(words, w0 + wpl);
      uint32_t cnt = 0;
      for (int64_t w = w0; w < w1; w++) cnt += __popc(sm.mask[w]);
      uint32_t incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t j = incl - cnt;
      for (int64_t w = w0; w < w1; w++)
        for (uint32_t m = sm.mask[w]; m; m &= m - 1) ocols[j++] = (uint16_t)(32 * w + __ffs(m) - 1);
      __syncwarp();
      if (blockIdx.x == 0) {
        for (int32_t i = lane; i < nO; i += 32) p.O_out[i] = ocols[i];
        if (lane == 0) *p.nO_out = (uint32_t)nO;
      }
    }
    mbar_arrive(&sm.lbar);  // 32 arrivals: the list is complete (or a wait gave up)
    if (rows > 0) {  // no copy outlives the CTA
      (void)mbar_wait_bounded(&sm.wbar, 0, p.status);
      (void)mbar_wait_bounded(&sm.wobar, 0, p.status);
    }
    dec_cluster_exit();
    return;
  }
  {
    // ---- activation pass 1: outlier columns and partial row maxima ----
    uint4 x[G::kRpt];
    uint32_t flags = 0;
#pragma unroll
    for (int j = 0; j < G::kRpt; j++) {  // all loads in flight before any is used
      const int t = grp + kC * j;
      x[j] = (t < T && live) ? __ldg(p.X + t * vecs + v) : make_uint4(0, 0, 0, 0);
    }
    named_bar_arrive(2, kDecThreads);
#pragma unroll
    for (int j = 0; j < G::kRpt; j++) {
      if (grp + kC * j < T) {  // padding rows must not flag columns (tau = 0 flags a zero)
        const uint32_t w[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
          flags |= (uint32_t)(abs_bits_lo(w[i]) >= p.thr) << (2 * i);
          flags |= (uint32_t)(abs_bits_hi(w[i]) >= p.thr) << (2 * i + 1);
        }
      }
    }
    if (!live) flags = 0;
    sm.fpart[grp * G::kVpc + vl] = (uint8_t)flags;
    named_bar_sync(1, kDecConsumers);
    // a column is an outlier if any of the call's rows flags it
    flags = 0;
    if (live)
#pragma unroll
      for (int r = 0; r < kC; r++) flags |= sm.fpart[r * G::kVpc + vl];
#pragma unroll
    for (int j = 0; j < G::kRpt; j++) {
      const uint32_t w[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        if (!((flags >> (2 * i)) & 1)) m = max(m, abs_bits_lo(w[i]));
        if (!((flags >> (2 * i + 1)) & 1)) m = max(m, abs_bits_hi(w[i]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) sm.part[warp * 4 + j] = m;
    }
    if (grp == 0) {  // row group 0 holds each column of this CTA once
      uint32_t c = __popc(flags);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      if (lane == 0) sm.wcnt[warp] = c;
    }
    named_bar_sync(1, kDecConsumers);
    cluster_wait();  // every CTA's mbarriers are initialised
    if (threadIdx.x < 17) {
      // this CTA's maximum of row t over its non-outlier columns (t < 16) or
      // its outlier count (16), stored into every CTA of the cluster
      uint32_t val = 0;
      if (threadIdx.x < 16) {
        const int t = threadIdx.x, rg = t % kC, j = t / kC;
#pragma unroll
        for (int w = 0; w < G::kWpg; w++) val = max(val, sm.part[(rg * G::kWpg + w) * 4 + j]);
      } else {
#pragma unroll
        for (int w = 0; w < G::kWpg; w++) val += sm.wcnt[w];
      }
      const uint32_t dst = smem_addr(&sm.pubs[crank][threadIdx.x]), bar = smem_addr(&sm.pbar);
#pragma unroll
      for (int c = 0; c < kC; c++) st_async_b32(mapa(dst, c), val, mapa(bar, c));
      if (threadIdx.x == 0) mbar_expect_tx(&sm.pbar, kC * 17 * 4);
    }
    if (mbar_wait_cluster_bounded(&sm.pbar, 0, p.status)) {
      // ---- activation pass 2: row scales, int8 codes, outlier mask (cluster-wide) ----
      uint32_t nO = 0, base = 0;
#pragma unroll
      for (int c = 0; c < kC; c++) {
        const uint32_t n = sm.pubs[c][16];
        nO += n;
        if (c < (int)crank) base += n;
      }
      // each row's code rule from sx (0 for rows >= T): one division per row
      RowCode<kBf> rcs[G::kRpt];
#pragma unroll
      for (int j = 0; j < G::kRpt; j++) {
        const int t = grp + kC * j;
        uint32_t m = 0;
#pragma unroll
        for (int c = 0; c < kC; c++) m = max(m, sm.pubs[c][t]);
        rcs[j] = RowCode<kBf>(e2f<kBf>(t < T ? m : 0u));
      }
      if (threadIdx.x < 16) {
        uint32_t m = 0;
#pragma unroll
        for (int c = 0; c < kC; c++) m = max(m, sm.pubs[c][threadIdx.x]);
        sxs[threadIdx.x] = e2f<kBf>((int)threadIdx.x < T ? m : 0u);
      }
      // bytes every CTA receives: the codes of all T rows and every mask word
      // (cbar); the first outlier columns and their X values (xbar)
      if (threadIdx.x == 0) {
        // every code but this CTA's own columns (stored locally), every mask word
        const int64_t own = min(vpc, max((int64_t)0, vecs - (int64_t)crank * vpc));
        mbar_expect_tx(&sm.cbar, (uint32_t)T * (uint32_t)(K - 8 * own) + 4u * (uint32_t)words);
        mbar_expect_tx(&sm.xbar, 4u * (1u + (uint32_t)T) * min(nO, (uint32_t)kDecOutSmall));
      }
      const uint32_t cbar = smem_addr(&sm.cbar), xbar = smem_addr(&sm.xbar);
      if (grp == 0) {  // mask word v/4 from the flags of vectors v .. v+3 (one CTA's)
        const uint32_t f1 = __shfl_down_sync(0xffffffffu, flags, 1);
        const uint32_t f2 = __shfl_down_sync(0xffffffffu, flags, 2);
        const uint32_t f3 = __shfl_down_sync(0xffffffffu, flags, 3);
        if ((vl & 3) == 0 && vl < vpc && v < vecs) {  // each word exactly once
          const uint32_t word = flags | (f1 << 8) | (f2 << 16) | (f3 << 24);
          const uint32_t dst = smem_addr(&sm.mask[v / 4]);
#pragma unroll
          for (int c = 0; c < kC; c++) st_async_b32(mapa(dst, c), word, mapa(cbar, c));
        }
      }
      // The first outlier columns and their X values: this CTA's outliers sit
      // at positions base.. of the ascending list, ordered by vector block,
      // lane and bit.  Every row group holds the same columns.
      if (__any_sync(0xffffffffu, flags != 0)) {
        const uint32_t pc = __popc(flags);
        uint32_t incl = pc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (live && flags) {
          uint32_t j = base + incl - pc;
          for (int w = 0; w < warp % G::kWpg; w++) j += sm.wcnt[w];
          for (int b = 0; b < 8 && j < (uint32_t)kDecOutSmall; b++)
            if ((flags >> b) & 1) {
              if (grp == 0) {
                const uint32_t dst = smem_addr(&sm.oc[j]);
                for (int c = 0; c < kC; c++)
                  st_async_b32(mapa(dst, c), (uint32_t)(8 * v + b), mapa(xbar, c));
              }
#pragma unroll
              for (int r = 0; r < G::kRpt; r++) {
                const int t = grp + kC * r;
                const uint32_t hb = ((&x[r].x)[b >> 1] >> (16 * (b & 1))) & 0xffffu;
                if (t < T) {
                  const uint32_t dst = smem_addr(&sm.xo[t * kDecOutSmall + j]);
                  for (int c = 0; c < kC; c++) st_async_b32(mapa(dst, c), hb, mapa(xbar, c));
                }
              }
              ++j;
            }
        }
      }
#pragma unroll
      for (int r = 0; r < G::kRpt; r++) {
        const int t = grp + kC * r;
        const uint32_t w[4] = {x[r].x, x[r].y, x[r].z, x[r].w};
        uint32_t p0, p1;
        rcs[r].codes8(w, flags, p0, p1);
        // even lanes store 16 codes (their vector and the next lane's) at once:
        // vpc is even, so an even thread's vector is even (16-byte aligned codes)
        // and its odd neighbour is live with it
        const uint32_t q0 = __shfl_down_sync(0xffffffffu, p0, 1);
        const uint32_t q1 = __shfl_down_sync(0xffffffffu, p1, 1);
        if (t >= T || !live || (lane & 1)) continue;
        // this CTA's copy by a plain store (the barrier before the MMAs
        // publishes it), the other CTAs' by remote stores
        *reinterpret_cast<uint4 *>(xs + t * pitch + 8 * v) = make_uint4(p0, p1, q0, q1);
        const uint32_t dst = smem_addr(xs + t * pitch + 8 * v);
#pragma unroll
        for (int c = 0; c < kC; c++)
          if (c != (int)crank) st_async_v4(mapa(dst, c), p0, p1, q0, q1, mapa(cbar, c));
      }
    }
  }
  // every CTA's codes, mask words, first outlier columns and their X values
  // are here (this also keeps the CTA alive until the last remote store into
  // it has landed)
  bool have = mbar_wait_cluster_bounded(&sm.pbar, 0, p.status);
  int32_t nO = 0;
  if (have)
#pragma unroll
    for (int c = 0; c < kC; c++) nO += (int32_t)sm.pubs[c][16];
  have = have && mbar_wait_cluster_bounded(&sm.cbar, 0, p.status) &&
         mbar_wait_cluster_bounded(&sm.xbar, 0, p.status);
  // forced-timeout test option: after every exchange has landed, one thread
  // of CTA 0 waits on a barrier nothing completes and gives up, so that CTA's
  // consumers take the timeout path below
  if (p.force_timeout && blockIdx.x == 0 && threadIdx.x == 0 &&
      !mbar_wait_bounded(&sm.never, 0, p.status, kForcedWaitNs))
    have = false;
  // the same outcome for every consumer thread: named barriers follow
  have = named_bar_and(1, kDecConsumers, have);

  if (blockIdx.x == 0) {  // the activation pass's results, for the debug entry point
    if (threadIdx.x < T) p.sx_out[threadIdx.x] = sxs[threadIdx.x];
    if (p.dbg_xq)
      for (int64_t i = threadIdx.x; i < (int64_t)T * vecs; i += kDecConsumers) {
        const int64_t t = i / vecs, vv = i - t * vecs;
        reinterpret_cast<uint2 *>(p.dbg_xq)[i] = *reinterpret_cast<const uint2 *>(xs + t * pitch + 8 * vv);
      }
  }
  if (!have || rows <= 0) {  // a wait gave up (status word), or no channels here
    dec_cluster_exit();
    return;
  }

  // ---- consumer warps: K-range [k0, k1) for every 8-channel group ----
  const int g = lane >> 2, q = lane & 3;
  const int ng = (int)((rows + 7) / 8);
  // Epilogue items: thread i takes accumulator word idx = i / 32 (and, for
  // i < 128, idx + 16: the fifth group) of lane i % 32 of every warp; the
  // channel scales are loaded while the MMAs run.
  const int el = threadIdx.x & 31, eg = el >> 2, eq = el & 3;
  const int nitems = threadIdx.x < 128 ? 2 : 1;
  int e_t[2], e_n[2];
  float e_sw[2];
#pragma unroll
  for (int it = 0; it < 2; it++) {
    const int idx = threadIdx.x / 32 + 16 * it, gi = idx >> 2, j = idx & 3;
    e_t[it] = eg + 8 * (j >> 1);
    e_n[it] = gi * 8 + 2 * eq + (j & 1);
    e_sw[it] = (it < nitems && e_n[it] < rows) ? __ldg(p.sw + n0 + e_n[it]) : 0.f;
  }
  const int64_t k0 = warp * range, k1 = min(K, k0 + range);
  int acc[kDecGroups][4] = {};
  if (k1 > k0 && mbar_wait_bounded(&sm.wbar, 0, p.status)) {
    const uint8_t *xhi = xs + (g + (p.xrows > 8 ? 8 : 0)) * pitch;
    if (((k1 - k0) & 63) == 0)
      dec_mma_range<false>(xs, xhi, ws, pitch, g, q, k0, k1, ng, acc);
    else
      dec_mma_range<true>(xs, xhi, ws, pitch, g, q, k0, k1, ng, acc);
  }
  // Only the int8 weight kept (W16 null): the outlier weights are the slice's
  // own codes, Wq sw / 127, with sw / 127 applied in the epilogue.  The first
  // outlier columns are read here, before the reduction reuses the weight
  // region (every thread waits for the slice: some warps had no K-range).
  constexpr bool wfree = kWq;
  float e_small[2] = {0.f, 0.f};
  if (wfree && mbar_wait_bounded(&sm.wbar, 0, p.status)) {
    const int nsm = nO < kDecOutSmall ? nO : kDecOutSmall;
#pragma unroll
    for (int it = 0; it < 2; it++)
      if (it < nitems && e_n[it] < rows)
        for (int j = 0; j < nsm; j++)
          e_small[it] = fmaf(e2f<kBf>(sm.xo[e_t[it] * kDecOutSmall + j]),
                             (float)(int8_t)ws[e_n[it] * pitch + sm.oc[j]], e_small[it]);
  }
  // outlier columns beyond the first kDecOutSmall: split over the consumer
  // warps, from the producer warp's list
  const bool big = nO > kDecOutSmall &&  // the same in every warp
                   mbar_wait_bounded(&sm.lbar, 0, p.status);
  float o[kDecGroups][4] = {};
  for (int32_t j = kDecOutSmall + warp; big && j < nO; j += kDecWarps) {
    const int64_t k = ocols[j];
    const float x0 = g < T ? e2f<kBf>(__ldg(p.X16 + (int64_t)g * K + k)) : 0.f;
    const float x1 = g + 8 < T ? e2f<kBf>(__ldg(p.X16 + (int64_t)(g + 8) * K + k)) : 0.f;
#pragma unroll
    for (int gi = 0; gi < kDecGroups; gi++) {
      if (gi < ng) {
        const int64_t ra = min((int64_t)gi * 8 + 2 * q, rows - 1);
        const int64_t rb = min((int64_t)gi * 8 + 2 * q + 1, rows - 1);
        const float wa = wfree ? (float)(int8_t)ws[ra * pitch + k]
                               : e2f<kBf>(__ldg(p.W16 + (n0 + ra) * K + k));
        const float wb = wfree ? (float)(int8_t)ws[rb * pitch + k]
                               : e2f<kBf>(__ldg(p.W16 + (n0 + rb) * K + k));
        o[gi][0] = fmaf(x0, wa, o[gi][0]);
        o[gi][1] = fmaf(x0, wb, o[gi][1]);
        o[gi][2] = fmaf(x1, wa, o[gi][2]);
        o[gi][3] = fmaf(x1, wb, o[gi][3]);
      }
    }
  }
  // cross-warp reduction: red[warp][lane][gi*4 + j] (stride 21 words, so that
  // the epilogue's column reads are free of bank conflicts), in the weight
  // region once every consumer warp is past its main loop
  named_bar_sync(1, kDecConsumers);
  uint32_t *mine = red + (warp * 32 + lane) * kDecRedStride;
#pragma unroll
  for (int gi = 0; gi < kDecGroups; gi++)
#pragma unroll
    for (int j = 0; j < 4; j++) mine[gi * 4 + j] = (uint32_t)acc[gi][j];
  named_bar_sync(1, kDecConsumers);
  int e_acc[2] = {0, 0};
#pragma unroll
  for (int it = 0; it < 2; it++)
    if (it < nitems) {
      const int idx = threadIdx.x / 32 + 16 * it;
#pragma unroll
      for (int w = 0; w < kDecWarps; w++) e_acc[it] += (int)red[(w * 32 + el) * kDecRedStride + idx];
    }
  float e_out[2] = {e_small[0], e_small[1]};
  if (big) {
    named_bar_sync(1, kDecConsumers);
#pragma unroll
    for (int gi = 0; gi < kDecGroups; gi++)
#pragma unroll
      for (int j = 0; j < 4; j++) mine[gi * 4 + j] = __float_as_uint(o[gi][j]);
    named_bar_sync(1, kDecConsumers);
#pragma unroll
    for (int it = 0; it < 2; it++)
      if (it < nitems) {
        const int idx = threadIdx.x / 32 + 16 * it;
#pragma unroll
        for (int w = 0; w < kDecWarps; w++)
          e_out[it] += __uint_as_float(red[(w * 32 + el) * kDecRedStride + idx]);
      }
  }
  // the first outlier columns: X from the exchange, W16 from the TMA boxes
  const int nsmall = nO < kDecOutSmall ? nO : kDecOutSmall;
  const bool ok_o = mbar_wait_bounded(&sm.wobar, 0, p.status);
#pragma unroll
  for (int it = 0; it < 2; it++)
    if (!wfree && it < nitems && e_n[it] < rows)
      for (int j = 0; j < nsmall; j++)
        e_out[it] = fmaf(e2f<kBf>(sm.xo[e_t[it] * kDecOutSmall + j]),
                         e2f<kBf>(sm.wos[j][e_n[it]][sm.oc[j] & 7u]), e_out[it]);
#pragma unroll
  for (int it = 0; it < 2; it++) {
    const int t = e_t[it], nl = e_n[it];
    if (it < nitems && t < T && nl < rows && ok_o) {
      const int64_t n = n0 + nl;
      const float st = sxs[t] / 127.0f, sn = e_sw[it] / 127.0f;
      const float b = e2f<kBf>(sm.bias[nl]);  // 0 without a bias
      const float y = wfree ? fmaf(fmaf((float)e_acc[it], st, e_out[it]), sn, b)
                            : fmaf((float)e_acc[it] * st, sn, e_out[it] + b);
      p.Y[t * p.N + n] = f2e<kBf>(y);
      if (p.dbg_acc) p.dbg_acc[t * p.N + n] = e_acc[it];
    }
  }
  dec_cluster_exit();
}

// ---------------------------------------------------------------------------
// dec_local: T <= 8 without a cluster.  Every CTA runs the whole activation
// pass itself (each consumer thread one 8-column vector of every row: a
// column's outlier flag and its codes need no other thread), so the codes are
// in shared memory about a microsecond after the X loads, and all SMs take a
// weight slice.  The MMAs swap roles: the weight is the 16-row A operand (up
// to three 16-channel tiles per slice) and the codes of X the 8-column B
// operand, one column per token, so no MMA row is spent on padding tokens.
// Each tile has its own weight barrier, and the MMA warps take the tiles in
// the order the producer put them in flight.
// ---------------------------------------------------------------------------

constexpr int kLocMaxT = 8;                     // tokens of a dec_local call, at most
constexpr int kLocTiles = (kDecMaxRows + 15) / 16;  // 16-channel tiles of a slice
constexpr int kLocRedStride = kLocTiles * 4 + 1;    // words per lane in the reduction (odd)
static_assert(kDecodeMaxK <= kDecConsumers * 8, "one 8-column vector per consumer thread");
static_assert(kDecodeMaxK / kDecWarps <= kDecChunkK, "one K-range sums exactly in fp32");
static_assert(kDecWarps * 32 * kLocRedStride * 4 <= kDecRedBytes, "reduction fits the weight region");

struct DecLocSmall {
  uint64_t wbar[kLocTiles];  // tile i of the weight slice has landed
  uint64_t wobar;            // W16 at the first outlier columns is in wos
  uint64_t lbar;             // the outlier list (oc, nO) is complete (or a wait gave up)
  uint64_t never;            // completed by nothing (forced-timeout test option)
  // [j][row][8]: W16[n0 + row, 8 (O[j] / 8) .. + 8), one TMA box per outlier column j
  alignas(128) uint16_t wos[kDecOutSmall][kDecMaxRows][8];
  uint32_t wcnt[kDecWarps];            // outliers of each warp's 256 columns
  uint32_t sxb[kLocMaxT];              // row maxima (16-bit magnitude bits; shared atomic max)
  uint32_t nO;
  uint32_t xo[kLocMaxT * kDecOutSmall];  // [t][j] X at the first outlier columns (16-bit bits)
  uint32_t oc[kDecOutSmall];             // the first outlier columns
  uint16_t bias[kDecMaxRows];            // the slice's 16-bit bias (0 without one)
};

// kWq: only the int8 weight is kept (W16 null); kBf: X, W16, bias and Y are
// bf16; kMT: the call's tokens at most (1, 2, 4, 6 or kLocMaxT).  The
// activation pass's loops over the rows are unrolled that far, and the
// smaller code is what a decode call spends its first microseconds fetching:
// measured at K = N = 4096, T 1 took 6.28 us with kMT 4 against 7.32 us with
// kMT 8.
template <bool kWq, bool kBf, int kMT>
__global__ void __launch_bounds__(kDecThreads, 1)
    dec_local_kernel(const __grid_constant__ CUtensorMap tm_w16, const DecArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int64_t K = p.K, pitch = dec_pitch(K), range = dec_range(K);
  uint8_t *ws = smem;                                        // [rows][pitch] weight codes
  uint8_t *xs = smem + p.wregion;                            // [8][pitch] activation codes
  uint16_t *ocols = reinterpret_cast<uint16_t *>(xs + kLocMaxT * pitch);  // outlier columns
  __shared__ DecLocSmall sm;
  uint32_t *red = reinterpret_cast<uint32_t *>(smem);  // [16 warps][32][13], after the MMAs

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T;
  const int64_t n0 = p.n_base + (int64_t)blockIdx.x * p.rows_per_cta;
  const int64_t rows = min(p.n_end, n0 + p.rows_per_cta) - n0;  // 1 .. 40
  const int nt = (int)((rows + 15) / 16);                    // weight tiles

  if (warp == kDecWarps && lane == 0) {
#pragma unroll
    for (int i = 0; i < kLocTiles; i++) mbar_init(&sm.wbar[i], 1);
    mbar_init(&sm.wobar, 1);
    mbar_init(&sm.lbar, 1);
    mbar_init(&sm.never, 1);
    mbar_init_fence();
  }
  if (threadIdx.x < kLocMaxT) sm.sxb[threadIdx.x] = 0u;
  __syncthreads();
  pdl_trigger();  // the next kernel on the stream may launch; it waits for our completion
  pdl_wait();     // X may be the output of the previous kernel on the stream
  // a wait that gives up overwrites it (a later launch of the same call keeps it)
  if (p.reset_status && blockIdx.x == 0 && threadIdx.x == 0) *p.status = kDevOk;

  const int64_t vecs = K / 8;
  if (warp == kDecWarps) {
    // The whole weight slice in flight at once, tile by tile, one bulk copy
    // per row, right behind the X loads.  Rows past `rows` and the pads past
    // K are never written: the MMA warps read row rows - 1 in place of the
    // former and zero the codes of X at the latter.
    named_bar_sync(2, kDecThreads);  // X loads issued
    uint16_t bv[2] = {0, 0};
    if (p.bias)
#pragma unroll
      for (int i = 0; i < 2; i++)
        if (lane + 32 * i < rows) bv[i] = __ldg(p.bias + n0 + lane + 32 * i);
    if (lane < nt) mbar_expect_tx(&sm.wbar[lane], (uint32_t)(min((int64_t)16, rows - 16 * lane) * K));
    __syncwarp();
    const uint64_t pol = l2_evict_first_policy();  // the slice is read once per call
    for (int64_t r = lane; r < rows; r += 32)
      bulk_g2s_once(ws + r * pitch, p.Wq + (n0 + r) * K, (uint32_t)K, &sm.wbar[r / 16], pol);
#pragma unroll
    for (int i = 0; i < 2; i++)
      if (lane + 32 * i < kDecMaxRows) sm.bias[lane + 32 * i] = bv[i];
    __syncwarp();  // lane 0's arrival on wobar below publishes the bias to the epilogue
    // W16 at the first outlier columns, one TMA box (8 columns x the slice's
    // channels) per column, once the consumers have listed them
    const bool ok = mbar_wait_bounded(&sm.lbar, 0, p.status);
    const int32_t nsmall = ok ? min((int32_t)sm.nO, kDecOutSmall) : 0;
    const bool fetch = !kWq && nsmall > 0;
    if (lane == 0) mbar_expect_tx(&sm.wobar, fetch ? (uint32_t)(nsmall * 16 * p.rows_per_cta) : 0u);
    __syncwarp();
    if (fetch && lane < nsmall)
      tma_load_2d(&sm.wos[lane][0][0], &tm_w16, (int32_t)(sm.oc[lane] & ~7u), (int32_t)n0,
                  &sm.wobar);
    // no copy outlives the CTA
    for (int i = 0; i < nt; i++) (void)mbar_wait_bounded(&sm.wbar[i], 0, p.status);
    (void)mbar_wait_bounded(&sm.wobar, 0, p.status);
    return;
  }

  // ---- activation pass: thread v owns columns [8v, 8v + 8) of every row ----
  const int64_t v = threadIdx.x;
  const bool live = v < vecs;
  uint4 x[kMT];
#pragma unroll
  for (int t = 0; t < kMT; t++)  // all loads in flight before any is used
    x[t] = (t < T && live) ? __ldg(p.X + t * vecs + v) : make_uint4(0, 0, 0, 0);
  named_bar_arrive(2, kDecThreads);
  // a column is an outlier if any of the call's rows has |x| >= tau there
  uint32_t flags = 0;
#pragma unroll
  for (int t = 0; t < kMT; t++) {
    if (t < T) {
      const uint32_t w[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
#pragma unroll
      for (int i = 0; i < 4; i++) {
        flags |= (uint32_t)(abs_bits_lo(w[i]) >= p.thr) << (2 * i);
        flags |= (uint32_t)(abs_bits_hi(w[i]) >= p.thr) << (2 * i + 1);
      }
    }
  }
  if (!live) flags = 0;
  // each row's maximum over the non-outlier columns, and the outlier count
#pragma unroll
  for (int t = 0; t < kMT; t++) {
    if (t < T) {
      const uint32_t w[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        if (!((flags >> (2 * i)) & 1)) m = max(m, abs_bits_lo(w[i]));
        if (!((flags >> (2 * i + 1)) & 1)) m = max(m, abs_bits_hi(w[i]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) atomicMax(&sm.sxb[t], m);
    }
  }
  const uint32_t pc = __popc(flags);
  uint32_t incl = pc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.wcnt[warp] = incl;
  named_bar_sync(1, kDecConsumers);
  // The row maxima are final (shared atomic max); every warp sums the 16
  // warps' outlier counts itself (lane w reads warp w's), and lane t builds
  // row t's code rule (its one division) for the warp.
  const uint32_t lc = lane < kDecWarps ? sm.wcnt[lane] : 0u;
  uint32_t before = lane < warp ? lc : 0u, nO = lc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    nO += __shfl_xor_sync(0xffffffffu, nO, o);
  }
  if (threadIdx.x == 0) sm.nO = nO;  // for the producer warp
  const RowCode<kBf> rc_lane(e2f<kBf>(lane < T ? sm.sxb[lane] : 0u));
  // codes rint(fl32(127 x) / sx) of the non-outlier columns, 0 at the outliers
#pragma unroll
  for (int t = 0; t < kMT; t++) {
    if (t < T) {
      RowCode<kBf> rc;
      rc.a = __shfl_sync(0xffffffffu, rc_lane.a, t);
      rc.r = __shfl_sync(0xffffffffu, rc_lane.r, t);
      rc.s1 = kBf ? __shfl_sync(0xffffffffu, rc_lane.s1, t) : 1.0f;
      rc.s2 = kBf ? __shfl_sync(0xffffffffu, rc_lane.s2, t) : 1.0f;
      const uint32_t w[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
      uint32_t p0, p1;
      rc.codes8(w, flags, p0, p1);
      if (live) *reinterpret_cast<uint2 *>(xs + t * pitch + 8 * v) = make_uint2(p0, p1);
    }
  }
  // the ascending outlier list (thread order is column order), and X at the
  // first kDecOutSmall of them
  if (flags) {
    uint32_t j = before + incl - pc;
    for (int b = 0; b < 8; b++)
      if ((flags >> b) & 1) {
        const uint32_t col = (uint32_t)(8 * v + b);
        ocols[j] = (uint16_t)col;
        if (blockIdx.x == 0) p.O_out[j] = (int32_t)col;
        if (j < (uint32_t)kDecOutSmall) {
          sm.oc[j] = col;
#pragma unroll
          for (int t = 0; t < kMT; t++)
            if (t < T) sm.xo[t * kDecOutSmall + j] = ((&x[t].x)[b >> 1] >> (16 * (b & 1))) & 0xffffu;
        }
        ++j;
      }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.nO_out = nO;
  bool have = true;
  // forced-timeout test option: one thread of CTA 0 waits on a barrier
  // nothing completes and gives up, so that CTA's consumers take the timeout
  // path below
  if (p.force_timeout && blockIdx.x == 0 && threadIdx.x == 0 &&
      !mbar_wait_bounded(&sm.never, 0, p.status, kForcedWaitNs))
    have = false;
  // codes, outlier list and X values in place (the same outcome for every
  // consumer thread)
  have = named_bar_and(1, kDecConsumers, have);
  if (threadIdx.x == 0) mbar_arrive(&sm.lbar);  // the producer may fetch W16's columns
  if (blockIdx.x == 0) {  // the activation pass's results, for the debug entry point
    if (threadIdx.x < T) p.sx_out[threadIdx.x] = e2f<kBf>(sm.sxb[threadIdx.x]);
    if (p.dbg_xq)
      for (int64_t i = threadIdx.x; i < (int64_t)T * vecs; i += kDecConsumers) {
        const int64_t t = i / vecs, vv = i - t * vecs;
        reinterpret_cast<uint2 *>(p.dbg_xq)[i] = *reinterpret_cast<const uint2 *>(xs + t * pitch + 8 * vv);
      }
  }
  if (!have) return;  // the producer still waits for every copy before it exits

  // ---- MMA warps: K-range [k0, k1) of every tile, A = weight, B = codes of X ----
  const int g = lane >> 2, q = lane & 3;
  // epilogue item of this thread: accumulator word idx = i / 32 of lane i % 32
  // (tile idx / 4, word idx % 4: channel 16 tile + g' + 8 (word / 2), token
  // 2 q' + word % 2); the channel scale is loaded while the MMAs run
  const int el = threadIdx.x & 31, eidx = threadIdx.x >> 5;
  const bool eitem = eidx < 4 * kLocTiles;
  const int e_n = (eidx >> 2) * 16 + (el >> 2) + 8 * ((eidx & 3) >> 1);
  const int e_t = 2 * (el & 3) + (eidx & 1);
  const bool e_live = eitem && e_n < rows && e_t < T;
  const float e_sw = e_live ? __ldg(p.sw + n0 + e_n) : 0.f;

  const int64_t k0 = warp * range, k1 = min(K, k0 + range);
  const int nkb = k1 > k0 ? (int)((k1 - k0 + 63) / 64) : 0;  // <= 4
  uint32_t xg[4][8];  // token g's codes of this warp's blocks, widened (0 past K)
#pragma unroll
  for (int b = 0; b < 4; b++) {
    const int64_t kb = k0 + 64 * b;
    if (b < nkb && kb + 16 * q < k1) {
      widen16(*reinterpret_cast<const uint4 *>(xs + g * pitch + kb + 16 * q), xg[b]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; i++) xg[b][i] = 0u;
    }
  }
  int acc[kLocTiles][4] = {};
  bool landed = true;
#pragma unroll
  for (int ti = 0; ti < kLocTiles; ti++) {
    if (ti < nt) {
      landed = mbar_wait_bounded(&sm.wbar[ti], 0, p.status) && landed;
      const uint8_t *wa = ws + min((int64_t)(16 * ti + g), rows - 1) * pitch + 16 * q;
      const uint8_t *wb = ws + min((int64_t)(16 * ti + g + 8), rows - 1) * pitch + 16 * q;
      float f[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int b = 0; b < 4; b++) {
        if (b < nkb) {
          const int64_t kb = k0 + 64 * b;
          uint32_t ha[8], hb[8];
          widen16(*reinterpret_cast<const uint4 *>(wa + kb), ha);
          widen16(*reinterpret_cast<const uint4 *>(wb + kb), hb);
#pragma unroll
          for (int mm = 0; mm < 4; mm++)
            mma_f16_16x8x16(f, ha[2 * mm], hb[2 * mm], ha[2 * mm + 1], hb[2 * mm + 1],
                            xg[b][2 * mm], xg[b][2 * mm + 1]);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; j++) acc[ti][j] = __float2int_rn(f[j]);
    }
  }
  // Only the int8 weight kept (W16 null): the outlier weights are the slice's
  // own codes, Wq sw / 127, with sw / 127 applied in the epilogue; they are
  // read before the reduction reuses the weight region.
  const int nsmall = nO < (uint32_t)kDecOutSmall ? (int)nO : kDecOutSmall;
  float e_out = 0.f;
  if (kWq) {
    bool all = true;
    for (int ti = 0; ti < nt; ti++) all = mbar_wait_bounded(&sm.wbar[ti], 0, p.status) && all;
    if (all && e_live)
      for (int j = 0; j < nsmall; j++)
        e_out = fmaf(e2f<kBf>(sm.xo[e_t * kDecOutSmall + j]),
                     (float)(int8_t)ws[e_n * pitch + sm.oc[j]], e_out);
  }
  // outlier columns beyond the first kDecOutSmall: split over the warps
  const bool big = nO > (uint32_t)kDecOutSmall;  // the same in every warp
  float o[kLocTiles][4] = {};
  for (uint32_t j = kDecOutSmall + warp; big && j < nO; j += kDecWarps) {
    const int64_t k = ocols[j];
    const float x0 = 2 * q < T ? e2f<kBf>(__ldg(p.X16 + (int64_t)(2 * q) * K + k)) : 0.f;
    const float x1 = 2 * q + 1 < T ? e2f<kBf>(__ldg(p.X16 + (int64_t)(2 * q + 1) * K + k)) : 0.f;
#pragma unroll
    for (int ti = 0; ti < kLocTiles; ti++) {
      if (ti < nt) {
        const int64_t ra = min((int64_t)(16 * ti + g), rows - 1);
        const int64_t rb = min((int64_t)(16 * ti + g + 8), rows - 1);
        const float wa = kWq ? (float)(int8_t)ws[ra * pitch + k]
                             : e2f<kBf>(__ldg(p.W16 + (n0 + ra) * K + k));
        const float wb = kWq ? (float)(int8_t)ws[rb * pitch + k]
                             : e2f<kBf>(__ldg(p.W16 + (n0 + rb) * K + k));
        o[ti][0] = fmaf(wa, x0, o[ti][0]);
        o[ti][1] = fmaf(wa, x1, o[ti][1]);
        o[ti][2] = fmaf(wb, x0, o[ti][2]);
        o[ti][3] = fmaf(wb, x1, o[ti][3]);
      }
    }
  }
  // cross-warp reduction in the weight region, once every warp is past its MMAs
  named_bar_sync(1, kDecConsumers);
  uint32_t *mine = red + (warp * 32 + lane) * kLocRedStride;
#pragma unroll
  for (int ti = 0; ti < kLocTiles; ti++)
#pragma unroll
    for (int j = 0; j < 4; j++) mine[ti * 4 + j] = (uint32_t)acc[ti][j];
  named_bar_sync(1, kDecConsumers);
  int e_acc = 0;
  if (eitem)
#pragma unroll
    for (int w = 0; w < kDecWarps; w++) e_acc += (int)red[(w * 32 + el) * kLocRedStride + eidx];
  if (big) {
    named_bar_sync(1, kDecConsumers);
#pragma unroll
    for (int ti = 0; ti < kLocTiles; ti++)
#pragma unroll
      for (int j = 0; j < 4; j++) mine[ti * 4 + j] = __float_as_uint(o[ti][j]);
    named_bar_sync(1, kDecConsumers);
    if (eitem)
#pragma unroll
      for (int w = 0; w < kDecWarps; w++)
        e_out += __uint_as_float(red[(w * 32 + el) * kLocRedStride + eidx]);
  }
  // the first outlier columns: X from the activation pass, W16 from the TMA boxes
  const bool ok_o = mbar_wait_bounded(&sm.wobar, 0, p.status);
  if (!kWq && e_live)
    for (int j = 0; j < nsmall; j++)
      e_out = fmaf(e2f<kBf>(sm.xo[e_t * kDecOutSmall + j]),
                   e2f<kBf>(sm.wos[j][e_n][sm.oc[j] & 7u]), e_out);
  if (e_live && ok_o && landed) {
    const int64_t n = n0 + e_n;
    const float st = e2f<kBf>(sm.sxb[e_t]) / 127.0f, sn = e_sw / 127.0f;
    const float b = e2f<kBf>(sm.bias[e_n]);  // 0 without a bias
    const float y = kWq ? fmaf(fmaf((float)e_acc, st, e_out), sn, b)
                        : fmaf((float)e_acc * st, sn, e_out + b);
    p.Y[e_t * p.N + n] = f2e<kBf>(y);
    if (p.dbg_acc) p.dbg_acc[e_t * p.N + n] = e_acc;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

// dec_local's four forms (kWq, kBf) for a token bound
#define DEC_LOCAL_FORMS(mt)                                                          \
  dec_local_kernel<false, false, mt>, dec_local_kernel<true, false, mt>,             \
      dec_local_kernel<false, true, mt>, dec_local_kernel<true, true, mt>

// the kernels built (index into DecCfg::ctas): dec_fused in clusters of 8, 16
// or 4 CTAs, and dec_local (1: no cluster)
constexpr int kDecClusterSizes[4] = {8, 16, 4, 1};
constexpr int kDecLocal = 3;
// Order of preference over kDecClusterSizes, measured per call in 16-layer
// CUDA graphs at N 3900 (both sizes hold it): 16-CTA clusters are 3-8 %
// faster than 8-CTA ones while T K <= 32768 (every T <= 16 at K 2048, T <= 8
// at K 4096), 8-CTA ones faster beyond (6 % at T 16, K 4096; 2 % at T 16,
// K 3072).  4-CTA clusters were the slowest everywhere.
constexpr int64_t kDecSmallWork = 32768;
constexpr int kDecPreferSmall[3] = {1, 0, 2};  // T K <= kDecSmallWork: 16, 8, 4
constexpr int kDecPreferLarge[3] = {0, 1, 2};  // otherwise: 8, 16, 4
// dec_local comes first for T <= dec_local_first(K), and serves T <= kLocMaxT
// where no cluster size holds the call.  Its activation pass costs every CTA
// the whole T x K codes, the clustered kernel's exchange grows with K.
// Measured per call (16-layer CUDA graphs, N 4096) against 16-CTA clusters:
// at K 4096, 5.94 / 7.81 / 8.57 / 9.08 / 9.88 / 10.37 us at T 1 / 4 / 5 / 6 /
// 7 / 8 against 9.54 / 9.61 / 9.83 / 9.85 / 9.90 / 10.14; at K 2048, 4.92 /
// 7.04 / 7.81 / 8.32 at T 1 / 4 / 5 / 6 against 7.98 / 8.19 / 8.08 / 8.25.
constexpr int64_t dec_local_first(int64_t K) { return K > 2048 ? 6 : 5; }

// CTAs of dec_fused<kC> resident at once, in whole clusters (0 if the query
// fails); also opens the kernel's shared-memory limit to `dyn_max`.
template <int kC>
int dec_resident_ctas(int dyn_max) {
  for (auto *f : {dec_fused_kernel<kC, false, false>, dec_fused_kernel<kC, true, false>,
                  dec_fused_kernel<kC, false, true>, dec_fused_kernel<kC, true, true>}) {
    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max) !=
        cudaSuccess)
      return 0;
    if (kC > 8 &&
        cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kC * 16);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = decode_smem_bytes(kDecodeMaxK, 32);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int least = 1 << 30;
  for (auto *f : {dec_fused_kernel<kC, false, false>, dec_fused_kernel<kC, true, false>,
                  dec_fused_kernel<kC, false, true>, dec_fused_kernel<kC, true, true>}) {
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) n = 0;
    least = n < least ? n : least;  // every form must fit
  }
  return least * kC;
}

// CTAs of dec_local resident at once (0 if the query fails); also opens the
// kernel's shared-memory limit to `dyn_max`.
int dec_local_ctas(int dev, int dyn_max) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  int least = 1 << 30;
  for (auto *f : {DEC_LOCAL_FORMS(1), DEC_LOCAL_FORMS(2), DEC_LOCAL_FORMS(4),
                  DEC_LOCAL_FORMS(6), DEC_LOCAL_FORMS(kLocMaxT)}) {
    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max) !=
        cudaSuccess)
      return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, f, kDecThreads, decode_smem_bytes(kDecodeMaxK, 32, kLocMaxT)) != cudaSuccess)
      n = 0;
    least = n < least ? n : least;  // every form must fit
  }
  return least * sms;
}

struct DecCfg {
  int ctas[4];  // resident CTAs for each entry of kDecClusterSizes (0: not available)
  int dyn_max;  // dynamic shared memory a CTA may use
};

// Queried once per device; the nominal B300 figures when no device answers.
DecCfg decode_cfg(int dev) {
  static std::atomic<int> cache[64][6];  // ctas[0..3], dyn_max, valid
  if (dev >= 0 && dev < 64 && cache[dev][5].load(std::memory_order_acquire) == 1) {
    DecCfg r;
    for (int i = 0; i < 4; i++) r.ctas[i] = cache[dev][i].load(std::memory_order_relaxed);
    r.dyn_max = cache[dev][4].load(std::memory_order_relaxed);
    return r;
  }
  int optin = 0;
  cudaFuncAttributes fa = {}, fl = {};
  DecCfg r{{0, 0, 0, 0}, 0};
  const int qdev = dev < 0 ? 0 : dev;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, qdev) ==
          cudaSuccess &&
      cudaFuncGetAttributes(&fa, dec_fused_kernel<8, false, false>) == cudaSuccess &&
      cudaFuncGetAttributes(&fl, dec_local_kernel<false, false, kLocMaxT>) == cudaSuccess) {
    r.dyn_max = optin - (int)(fa.sharedSizeBytes > fl.sharedSizeBytes ? fa.sharedSizeBytes
                                                                       : fl.sharedSizeBytes);
    r.ctas[0] = dec_resident_ctas<8>(r.dyn_max);
    r.ctas[1] = dec_resident_ctas<16>(r.dyn_max);
    r.ctas[2] = dec_resident_ctas<4>(r.dyn_max);
    r.ctas[3] = dec_local_ctas(qdev, r.dyn_max);
  }
  (void)cudaGetLastError();  // a failed query is not a launch error
  if (r.ctas[0] + r.ctas[1] + r.ctas[2] + r.ctas[3] == 0)
    return DecCfg{{0, 0, kB300Sms / 4 * 4, 0}, (int)decode_smem_bytes(kDecodeMaxK, 32)};
  if (dev >= 0 && dev < 64) {
    for (int i = 0; i < 4; i++) cache[dev][i].store(r.ctas[i], std::memory_order_relaxed);
    cache[dev][4].store(r.dyn_max, std::memory_order_relaxed);
    cache[dev][5].store(1, std::memory_order_release);
  }
  return r;
}

// Output channels a CTA can hold at this K (at most kDecMaxRows).
int64_t dec_rows_cap(const DecCfg &c, int64_t K, int64_t xrows = 16) {
  int64_t rows = kDecMaxRows;
  while (rows > 8 && decode_smem_bytes(K, rows, xrows) > (size_t)c.dyn_max) rows--;
  return rows;
}

// Whether the resident CTAs of kernel i (index into kDecClusterSizes) hold
// N output channels in one wave.
// Output channels one launch of kernel i (index into kDecClusterSizes) holds
// in one wave of its resident CTAs; 0 where the kernel does not apply.
int64_t decode_wave(const DecCfg &c, int i, int64_t T, int64_t K) {
  if (i == kDecLocal && T > kLocMaxT) return 0;
  return (int64_t)c.ctas[i] * dec_rows_cap(c, K, i == kDecLocal ? kLocMaxT : dec_xrows(T));
}

// Launches of kernel i a call of N channels takes (one wave each); a large
// number where the kernel does not apply.
int64_t decode_launches(const DecCfg &c, int i, int64_t T, int64_t N, int64_t K) {
  const int64_t w = decode_wave(c, i, T, K);
  return w > 0 ? (N + w - 1) / w : (int64_t)1 << 40;
}

// The decode path splits the channels over at most this many launches (each
// runs the activation pass again); beyond it the GEMM's 32-token tile is
// faster.  Measured at T 16, K 4096: N 11008 in three launches, 31.5 us
// against 41 us on the GEMM.
constexpr int64_t kDecMaxLaunches = 3;

// The index (into kDecClusterSizes) of the kernel a call runs: the first, in
// the order of preference for T and K, that takes the call in one launch;
// otherwise the one with the fewest launches (at most kDecMaxLaunches; ties
// in that order); -1 if none.  A call may ask for a cluster size (`want`, 0 =
// no preference; 1 = dec_local), taken whenever it holds the call in one
// launch.
int decode_pick(const DecCfg &c, int64_t T, int64_t N, int64_t K, int want) {
  for (int i = 0; i < 4; i++)
    if (want != 0 && kDecClusterSizes[i] == want && decode_launches(c, i, T, N, K) == 1) return i;
  int order[4], n = 0;
  const bool local_first = T <= dec_local_first(K);
  if (local_first) order[n++] = kDecLocal;
  const int *pref = T * K <= kDecSmallWork ? kDecPreferSmall : kDecPreferLarge;
  for (int j = 0; j < 3; j++) order[n++] = pref[j];
  if (!local_first) order[n++] = kDecLocal;
  int best = -1;
  for (int j = 0; j < n; j++) {
    const int64_t l = decode_launches(c, order[j], T, N, K);
    if (l == 1) return order[j];
    if (l <= kDecMaxLaunches && (best < 0 || l < decode_launches(c, best, T, N, K))) best = order[j];
  }
  return best;
}

}  // namespace

// Output channels the decode path takes at this T and K: what the resident
// CTAs of the best-covered kernel hold in kDecMaxLaunches launches.
int64_t decode_max_n(int dev, int64_t T, int64_t K) {
  const DecCfg c = decode_cfg(dev);
  int64_t n = 0;
  for (int i = 0; i < 4; i++) {
    const int64_t w = decode_wave(c, i, T, K);
    n = w > n ? w : n;
  }
  return kDecMaxLaunches * n;
}

int decode_cluster_size(int dev, int64_t T, int64_t N, int64_t K) {
  const int pick = decode_pick(decode_cfg(dev), T, N, K, 0);
  return pick < 0 ? 0 : kDecClusterSizes[pick];
}

cudaError_t launch_decode(const void *X, int64_t T, int64_t K, uint32_t thr, const int8_t *Wq,
                          const float *sw, const void *W16, const void *bias, int64_t N,
                          bool bf16, void *Y, const Workspace &ws, int8_t *dbg_xq,
                          int32_t *dbg_acc, uint32_t opts, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const DecCfg dc = decode_cfg(dev);
  const int pick = decode_pick(dc, T, N, K, (int)((opts >> 8) & 0xffu));
  if (pick < 0) return cudaErrorInvalidValue;  // the host routes only shapes that fit here
  const bool local = pick == kDecLocal;
  const int kc = kDecClusterSizes[pick];
  const int form = (W16 == nullptr ? 1 : 0) | (bf16 ? 2 : 0);
  using Kern = void (*)(CUtensorMap, DecArgs);
  static const Kern kerns[4][4] = {
      {dec_fused_kernel<8, false, false>, dec_fused_kernel<8, true, false>,
       dec_fused_kernel<8, false, true>, dec_fused_kernel<8, true, true>},
      {dec_fused_kernel<16, false, false>, dec_fused_kernel<16, true, false>,
       dec_fused_kernel<16, false, true>, dec_fused_kernel<16, true, true>},
      {dec_fused_kernel<4, false, false>, dec_fused_kernel<4, true, false>,
       dec_fused_kernel<4, false, true>, dec_fused_kernel<4, true, true>},
      {DEC_LOCAL_FORMS(kLocMaxT)}};
  // the kernel without clusters, by the call's tokens at most
  static const Kern kerns_local[4][4] = {
      {DEC_LOCAL_FORMS(1)}, {DEC_LOCAL_FORMS(2)}, {DEC_LOCAL_FORMS(4)}, {DEC_LOCAL_FORMS(6)}};
  const int mt = T <= 1 ? 0 : T <= 2 ? 1 : T <= 4 ? 2 : T <= 6 ? 3 : 4;
  const Kern kern = local && mt < 4 ? kerns_local[mt][form] : kerns[pick][form];
  DecArgs a;
  a.X = reinterpret_cast<const uint4 *>(X);
  a.X16 = reinterpret_cast<const unsigned short *>(X);
  a.T = (int)T;
  a.K = K;
  a.N = N;
  a.thr = thr;
  a.xrows = local ? kLocMaxT : (int)dec_xrows(T);
  a.Wq = Wq;
  a.sw = sw;
  a.W16 = reinterpret_cast<const unsigned short *>(W16);
  a.bias = reinterpret_cast<const unsigned short *>(bias);
  a.Y = reinterpret_cast<uint16_t *>(Y);
  a.sx_out = ws.sx;
  a.O_out = ws.O;
  a.nO_out = ws.counters + 1;
  a.dbg_xq = dbg_xq;
  a.dbg_acc = dbg_acc;
  a.status = ws.status;
  a.force_timeout = (opts & BNB_OPT_FORCE_TIMEOUT) ? 1 : 0;
  // One launch per wave of the resident CTAs, each over an equal share of
  // the channels (every launch runs the activation pass; each later one
  // waits for the one before through programmatic dependent launch).
  const int64_t wave = decode_wave(dc, pick, T, K);
  const int64_t nl = (N + wave - 1) / wave;
  const int64_t share = (N + nl - 1) / nl;
  cudaError_t e = cudaSuccess;
  for (int64_t nb = 0; nb < N && e == cudaSuccess; nb += share) {
    const int64_t nn = min(share, N - nb);
    a.n_base = nb;
    a.n_end = nb + nn;
    a.reset_status = nb == 0 ? 1 : 0;
    // the resident CTAs (whole clusters) share the channels evenly, with no
    // more CTAs than one per 8 channels (rounded up to whole clusters)
    const int64_t want = min((int64_t)dc.ctas[pick], ((nn + 7) / 8 + kc - 1) / kc * kc);
    a.rows_per_cta = (nn + want - 1) / want;
    const int64_t used = (nn + a.rows_per_cta - 1) / a.rows_per_cta;
    const int64_t ctas = (used + kc - 1) / kc * kc;
    a.wregion = dec_wregion(K, a.rows_per_cta);
    // W16 in boxes of 8 columns x one slice's channels (outlier columns only,
    // so no L2 promotion beyond the sector)
    // (without W16 the map is never read: it then describes Wq)
    CUtensorMap tm;
    const bool enc = W16 ? encode_2d(&tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, W16, (uint64_t)K,
                                     (uint64_t)N, (uint64_t)K * 2, 8, (uint32_t)a.rows_per_cta,
                                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE)
                         : encode_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, (uint64_t)K,
                                     (uint64_t)N, (uint64_t)K, 16, (uint32_t)a.rows_per_cta,
                                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    if (!enc) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = decode_smem_bytes(K, a.rows_per_cta, a.xrows);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (!local) {
      attr[na].id = cudaLaunchAttributeClusterDimension;
      attr[na].val.clusterDim.x = (unsigned)kc;
      attr[na].val.clusterDim.y = 1;
      attr[na].val.clusterDim.z = 1;
      na++;
    }
    if (!(opts & BNB_OPT_NO_PDL)) {
      attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[na].val.programmaticStreamSerializationAllowed = 1;
      na++;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, tm, a);
    note_launch();
  }
  return e;
}

}  // namespace bnb
