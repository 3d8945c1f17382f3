// Warp-level tensor-core fragments shared by the attention kernels:
// ldmatrix, movmatrix, mma.sync m16n8k16 (bf16 in, fp32 accumulate), the SFU
// exponential, and the swizzled layout of one KV page as the 2-D TMA copies of
// the pool deliver it.
#pragma once
#include <stdint.h>

namespace nf {

constexpr int AMMA_P = 16;  // page size the tensor-core attention kernels are built for

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// Transpose of an 8x8 b16 matrix held one pair per lane in fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// 2^x by the SFU (ex2.approx, relative error near 2^-22; 0 for -inf)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// d += a . b  (m16n8k16, bf16 inputs, fp32 accumulators)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of the 16-byte chunk `ci` (8 bf16 from dim 8*ci) of position
// `pos` inside one page block of K or V: 64-column boxes of 16 rows x 128 bytes,
// each 1024-byte half-box swizzled by (row % 8).
__device__ __forceinline__ uint32_t page_chunk_off(int pos, int ci) {
  const int box = ci >> 3, c = ci & 7;
  return static_cast<uint32_t>(box * (AMMA_P * 128) + pos * 128 + ((c ^ (pos & 7)) << 4));
}

}  // namespace nf
