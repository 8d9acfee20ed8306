// Warp-level mma.sync wrappers and the fragment convention shared by the
// decode GEMV and the warp-level GEMM.
//
// A dot product over k is exact in any order for integers (and in fp32 the
// order only moves rounding), so the physical k positions may be assigned to
// the MMA's logical k slots by any permutation that A and B share.  Both
// operands are read as one 16-byte vector per lane per 64-byte k-block:
//   lane (g = lane/4, q = lane%4) reads bytes [16q, 16q+16) of row g (and of
//   row g+8 for A); registers .x/.y feed the first MMA of the block and
//   .z/.w the second.
// For m16n8k32 (int8) the first MMA's logical k in [4q, 4q+4) is physical
// 16q + [0,4) and logical 16 + [4q, 4q+4) is physical 16q + [4,8); the second
// MMA takes physical 16q + [8,16) in the same way.  For m16n8k16 (fp16) the
// 64-byte block holds 32 halves and the same register assignment applies.
#pragma once

#include <cstdint>

namespace bnb {

__device__ __forceinline__ void mma_s8_16x8x32(int (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16x8x16(float (&d)[4], uint32_t a0, uint32_t a1,
                                                uint32_t a2, uint32_t a3, uint32_t b0,
                                                uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with bf16 operands.
__device__ __forceinline__ void mma_bf16_16x8x16(float (&d)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 64-byte k-block: xa = row g, xb = row g+8 (A); w = row g of B.
__device__ __forceinline__ void mma_s8_block(int (&d)[4], const uint4 &xa, const uint4 &xb,
                                             const uint4 &w) {
  mma_s8_16x8x32(d, xa.x, xb.x, xa.y, xb.y, w.x, w.y);
  mma_s8_16x8x32(d, xa.z, xb.z, xa.w, xb.w, w.z, w.w);
}

__device__ __forceinline__ void mma_f16_block(float (&d)[4], const uint4 &xa, const uint4 &xb,
                                              const uint4 &w) {
  mma_f16_16x8x16(d, xa.x, xb.x, xa.y, xb.y, w.x, w.y);
  mma_f16_16x8x16(d, xa.z, xb.z, xa.w, xb.w, w.z, w.w);
}
__device__ __forceinline__ void mma_bf16_block(float (&d)[4], const uint4 &xa, const uint4 &xb,
                                               const uint4 &w) {
  mma_bf16_16x8x16(d, xa.x, xb.x, xa.y, xb.y, w.x, w.y);
  mma_bf16_16x8x16(d, xa.z, xb.z, xa.w, xb.w, w.z, w.w);
}

// Accumulator element i of an m16n8 tile: row g + 8*(i/2), column 2q + (i%2).

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;\n"); }

}  // namespace bnb
