// Device helpers shared by the MoE kernels: bf16 packing, the warp-level
// bf16 MMA, MXFP4 -> bf16 decoding and the device status word.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {

// Programmatic dependent launch: wait until the preceding kernel of the stream has
// completed and its writes are visible (a no-op when launched without the
// attribute); let the next kernel start launching once every CTA got here.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void flag_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// Two fp32 -> bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16(float v) {
  return (uint16_t)(pack_bf16x2(v, 0.0f) & 0xffffu);
}

// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col).
// Fragment layout (PTX ISA, mma.m16n8k16, .bf16): lane = 4*g + c;
//   a0 = (row g,   k 2c..2c+1)  a1 = (row g+8, k 2c..2c+1)
//   a2 = (row g,   k 2c+8..9)   a3 = (row g+8, k 2c+8..9)
//   b0 = (k 2c..2c+1, col g)    b1 = (k 2c+8..9, col g)
//   d0,d1 = (row g, col 2c, 2c+1)   d2,d3 = (row g+8, col 2c, 2c+1)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Loads are plain (non-volatile) asm so that the compiler can hoist them ahead of
// the MMAs of earlier k steps: the data they read does not change during a kernel.
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// One 32-byte store of eight fp32 values (p 32-byte aligned): a whole sector per
// thread, half the store instructions of 16-byte vectors.
__device__ __forceinline__ void stg_v8(float* p, const float* v) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]),
               "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}

// Four fp32 values added to p[0..3] (p 16-byte aligned) by one vector reduction in
// L2: the per-token sums of the prefill down projection.
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Streaming load for weights read once: skip L1, and let L2 fetch 256-byte
// granules (the following k steps of the same row are requested right after).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// ---------------------------------------------------------------- f16 operands

// Two fp32 -> f16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void unpack_f16x2(uint32_t v, float& lo, float& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi) : "r"(v));
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// D(16x8, fp32) += A(16x16, f16) * B(16x8, f16); same fragment layout as the bf16 form.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^e as fp32 for -126 <= e <= 127.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// The four code bytes of `w` (eight E2M1 values, low nibble first) as exact f16
// pairs, byte t -> o[t] with its low nibble in the low half.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// ---------------------------------------------------------------- MXFP4 decoding
//
// An E2M1 code c = s e1 e0 m (bit 3 sign, bits 2..1 exponent with bias 1, bit 0
// mantissa) placed as bf16 bits  (s << 15) | (e1 e0 m << 6)  is exactly
// value(c) * 2^-126: exponent field e and top mantissa bit m give 2^(e-127) (1 + m/2)
// for e >= 1, and the subnormal 0.5 (e = 0, m = 1) becomes bf16 subnormal 2^-127.
// Multiplying by 2^126 * 2^(scale - 127) = 2^(scale - 1) is then exact (a power of
// two), which gives value * 2^(scale - 127) as bf16 with no rounding for every
// scale byte whose result is a normal or subnormal bf16.

// Scale factor(s) for one E8M0 byte: the value multiplies a decoded pair by
// `first` and then, when `two` is set, by `second` (1.0 otherwise, so that a warp
// that takes the two-multiply form for all of its rows stays exact).
struct Fp4Scale {
  uint32_t first, second;
  bool two;
};

__device__ __forceinline__ Fp4Scale fp4_scale(uint32_t s) {
  Fp4Scale r;
  if (s <= 128u) {                       // 2^(s-1): exponent field s+126 <= 254
    uint32_t b = (s + 126u) << 7;
    r.first = b | (b << 16);
    r.second = 0x3F803F80u;              // 1.0: a caller that multiplies twice
    r.two = false;
  } else if (s < 255u) {                 // 2^126 then 2^(s-127)
    r.first = 0x7E807E80u;
    uint32_t b = s << 7;
    r.second = b | (b << 16);
    r.two = true;
  } else {                               // 0xFF is NaN in E8M0
    r.first = 0x7FC07FC0u;
    r.second = 0x3F803F80u;
    r.two = false;
  }
  return r;
}

// Byte i (0..3) of w: its low nibble -> low bf16, high nibble -> high bf16,
// both scaled.  lo = w & 0x0F0F0F0F, hi = (w >> 4) & 0x0F0F0F0F.
template <int I>
__device__ __forceinline__ uint32_t fp4_pair(uint32_t lo, uint32_t hi, const Fp4Scale& sc) {
  // output bytes: [lo.byte I, 0x00, hi.byte I, 0x00]; selector nibble 8 replicates the
  // (zero) sign bit of lo.byte 0, i.e. yields 0x00.
  constexpr uint32_t sel = (uint32_t)I | (0x8u << 4) | ((uint32_t)(4 + I) << 8) | (0x8u << 12);
  uint32_t p;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p) : "r"(lo), "r"(hi), "n"(sel));
  uint32_t bits = (p * 0x1040u) & 0x81C081C0u;   // (p << 6) | (p << 12), disjoint, masked
  uint32_t v = bf16x2_mul(bits, sc.first);
  if (sc.two) v = bf16x2_mul(v, sc.second);
  return v;
}

}  // namespace moe
