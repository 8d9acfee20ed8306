// S1: per-output-channel weight quantization, run once per weight.
//
// sw[n] = max_k |W16[n,k]|, Wq[n,k] = rint(fl32(127 W16[n,k]) / sw[n]).
// The pages quantize weights "on the fly as the model loads" ("bitsandbytes"
// glossary page, introduction) and vector-wise ("bitsandbytes: GPU-Accelerated
// Inference and Training at Lower Bit Depths", section "How LLM.int8()
// quantizes weights and activations"); the vector is the output channel.
//
// HBM-bound one-off pass: one warp per row, 16-byte loads, the absmax taken on
// fp16 (or bf16) bit patterns (exact), the row read a second time (from L2)
// for codes.
#include "common.cuh"
#include "kernels.h"

namespace bnb {

template <bool kBf>
__global__ void __launch_bounds__(256) quantize_weight_kernel(
    const uint4 *__restrict__ W16, int64_t N, int64_t K, int8_t *__restrict__ Wq,
    float *__restrict__ sw) {
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x / 32);
  const int64_t vecs = K / 8;  // 16-byte vectors per row
  const uint32_t lane = threadIdx.x & 31;
  for (int64_t n = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; n < N;
       n += warps_total) {
    const uint4 *row = W16 + n * vecs;
    uint32_t m = 0;
    for (int64_t v = lane; v < vecs; v += 32) {
      uint4 q = __ldg(row + v);
      uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; i++) m = max(m, max(abs_bits_lo(w[i]), abs_bits_hi(w[i])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float a = e2f<kBf>(m);
    const RowCode<kBf> rc(a);
    if (lane == 0) sw[n] = a;
    uint2 *out = reinterpret_cast<uint2 *>(Wq + n * K);
    for (int64_t v = lane; v < vecs; v += 32) {
      uint4 q = __ldg(row + v);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
      uint32_t p0, p1;
      rc.codes8(w, 0u, p0, p1);
      out[v] = make_uint2(p0, p1);
    }
  }
}

cudaError_t launch_quantize_weight(const void *W16, int64_t N, int64_t K, bool bf16, int8_t *Wq,
                                   float *sw, cudaStream_t stream) {
  const int warps_per_block = 8;
  int64_t blocks = (N + warps_per_block - 1) / warps_per_block;
  if (blocks > 148 * 64) blocks = 148 * 64;
  (bf16 ? quantize_weight_kernel<true> : quantize_weight_kernel<false>)
      <<<(unsigned)blocks, 32 * warps_per_block, 0, stream>>>(
      reinterpret_cast<const uint4 *>(W16), N, K, Wq, sw);
  note_launch();
  return cudaGetLastError();
}

}  // namespace bnb
