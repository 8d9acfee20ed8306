// Internal launch interface between the C-ABI host layer and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace bnb {

// Process-wide count of kernel launches issued by this library.
void note_launch();

// Tensor map of a 2-D row-major tensor [outer x inner] with `row_bytes`
// between rows, loaded in boxes of box_outer x box_inner elements (false if
// the driver entry point is missing or rejects the layout).
bool encode_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swz, CUtensorMapL2promotion l2);

cudaError_t launch_quantize_weight(const void *W16, int64_t N, int64_t K, bool bf16, int8_t *Wq,
                                   float *sw, cudaStream_t stream);

// S2 + S3.  code_mode 0: int8 codes, 1: fp16 integer codes.  with_xo: write
// the padded fp16 outlier block.  pdl: launch the row pass with programmatic
// dependent launch behind the column scan.
cudaError_t launch_act_pass(const void *X, int64_t T, int64_t K, uint32_t thr_bits,
                            const Workspace &ws, int code_mode, bool with_xo, const void *W16,
                            const int8_t *Wq, int64_t N, bool bf16, int8_t *dbg_xq,
                            int num_sms, cudaStream_t stream, bool pdl);

// The blockwise 8-bit codec (blocks of B values, B a power of two in
// [64, 2048]): fp32 -> int8 codes + per-block absmax, and back.
cudaError_t launch_quantize_blockwise(const float *x, int64_t n, int B, int8_t *codes,
                                      float *absmax, int num_sms, cudaStream_t stream);
cudaError_t launch_dequantize_blockwise(const int8_t *codes, const float *absmax, int64_t n,
                                        int B, float *y, int num_sms, cudaStream_t stream);

// The whole layer for T <= 16, K <= kDecodeMaxK, N <= decode_max_n(dev, T, K)
// in one kernel launch per wave of channels, at most three (activation pass
// fused into the GEMV: shared by clusters of CTAs, or repeated by every CTA
// for T <= 5, T <= 6 at K > 2048), launched with programmatic dependent launch unless the call's
// options turn it off.
int64_t decode_max_n(int dev, int64_t T, int64_t K);
// The cluster size launch_decode picks for this shape (1: no clusters), 0 if
// none holds it.
int decode_cluster_size(int dev, int64_t T, int64_t N, int64_t K);
cudaError_t launch_decode(const void *X, int64_t T, int64_t K, uint32_t thr, const int8_t *Wq,
                          const float *sw, const void *W16, const void *bias, int64_t N,
                          bool bf16, void *Y, const Workspace &ws, int8_t *dbg_xq,
                          int32_t *dbg_acc, uint32_t opts, cudaStream_t stream);

// S4..S6 on tcgen05 tensor cores (fp16 integer codes from the activation
// pass, code_mode 1), persistent over 256 x 256 output tiles on CTA pairs
// (T > 32; 128 x 256 on single CTAs with BNB_OPT_SINGLE_CTA) or 128 x 32
// tiles (T <= 32).
cudaError_t launch_gemm_tc(int64_t T, int64_t K, const int8_t *Wq, const float *sw,
                           const void *W16, const void *bias, int64_t N, bool bf16, void *Y,
                           const Workspace &ws, int32_t *dbg_acc, int num_sms, uint32_t opts,
                           cudaStream_t stream);

// S4..S6 with warp-level mma.sync (legacy tensor path), int8 codes.
cudaError_t launch_gemm_mma(int64_t T, int64_t K, const int8_t *Wq, const float *sw,
                            const void *W16, const void *bias, int64_t N, bool bf16, void *Y,
                            const Workspace &ws, int32_t *dbg_acc, cudaStream_t stream);

}  // namespace bnb
