// Device helpers of the f16-operand MXFP4 prefill kernel (expert_prefill_fp4.cu):
// the clamped GLU, the exact E2M1 -> f16 decode of one 32-input block into a
// 128-byte-swizzled K-major tile, and its f16 multiplier.
//
// Source: "Phase 19: MoE - gpt-oss-20b", section 2 (clamped GLU) and section 3
// (MXFP4: E2M1 codes, low nibble first, one E8M0 scale per 32 inputs).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace moe {
namespace f16op {

__device__ __forceinline__ float tanh_fast(float z) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(z));
  return r;
}

// h = (clamp(up, -L, L) + 1) * min(gate, L) * sigmoid(alpha * min(gate, L)), with
// sigmoid(z) = (1 + tanh(z / 2)) / 2 on the hardware tanh.
__device__ __forceinline__ float clamped_glu(float gt, float up, float limit, float alpha) {
  gt = fminf(gt, limit);
  up = fminf(fmaxf(up, -limit), limit);
  return (up + 1.f) * gt * fmaf(0.5f, tanh_fast(0.5f * alpha * gt), 0.5f);
}

// f16x2 of the block multiplier 2^(s - 127 - c): exact for -23 <= s - 127 - c <= 15
// (subnormal below -14), 0 below -23 (the block is flushed), NaN for s = 255.
__device__ __forceinline__ uint32_t block_mult_f16(uint32_t s, int c) {
  const int qe = (int)s - 127 - c;
  uint32_t m = qe >= -14 ? (uint32_t)(qe + 15) << 10 : (qe >= -23 ? 1u << (qe + 24) : 0u);
  if (s == 255u) m = 0x7E00u;
  return m | (m << 16);
}

// The same multiplier when every block of the row is in the plain range
// (-14 <= s - 127 - c <= 13): kr = 15 - 127 - c.
__device__ __forceinline__ uint32_t block_mult_f16_plain(uint32_t s, uint32_t kr) {
  return ((s + kr) << 10) * 0x10001u;
}

// One block (16 code bytes at codes[r][16 b], rows of 32 bytes) -> 32 f16 values
// of row r of a tile with 128-byte rows and the 128-byte swizzle (16-byte chunk j
// of row r stored at chunk j ^ (r % 8)).
__device__ __forceinline__ void dequant_block(const uint8_t* codes, uint8_t* tile, int r, int b, uint32_t m2) {
  const uint4 w = *reinterpret_cast<const uint4*>(codes + r * 32 + b * 16);
  const uint32_t wk[4] = {w.x, w.y, w.z, w.w};
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t o[4];
    e2m1x8_to_f16(wk[k], o);
    uint4 q;
    q.x = f16x2_mul(o[0], m2);
    q.y = f16x2_mul(o[1], m2);
    q.z = f16x2_mul(o[2], m2);
    q.w = f16x2_mul(o[3], m2);
    *reinterpret_cast<uint4*>(row + (((4 * b + k) ^ (r & 7)) << 4)) = q;
  }
}

// Largest magnitude of a row, accumulated as fp32 bits (atomicMax on the bits of a
// non-negative float orders like the values; a NaN wins over every number).
__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

}  // namespace f16op
}  // namespace moe
