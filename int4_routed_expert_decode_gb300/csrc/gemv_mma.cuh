// gemv_mma.cuh -- building blocks of the int4 GEMVs on the tensor cores
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation) shared by the decode
// kernels: 16 weight rows are the M dimension, the inputs the N columns.
#pragma once

#include <stdint.h>

namespace moe {
namespace mmag {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Codes j and j + 4 of a packed word as the bf16 pair (128 + q_j, 128 + q_j+4).
__device__ __forceinline__ uint32_t code_pair(uint32_t w, int j) {
  return ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
}

// Shared-memory layout of one tile of 16 rows for ldmatrix: rows 0-7 and
// 8-15 are two halves `half` bytes apart, each written by the TMA as column
// blocks of 8 rows x `pitch` bytes; with the 128-byte swizzle (pitch 128)
// the 16-byte piece j of row r sits at piece j ^ (r & 7).
struct TileGeom {
  uint32_t cb_stride;  // bytes between column blocks
  uint32_t pitch;      // bytes of one row in one column block (128, or less unswizzled)
  uint32_t half;       // bytes between rows r and r + 8
  bool swz;
};

}  // namespace mmag
}  // namespace moe
