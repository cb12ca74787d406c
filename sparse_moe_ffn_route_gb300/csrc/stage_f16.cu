// Staging of the f16 token operands of the f16-operand MXFP4 kernels.
//
// An f16 operand keeps 11 significant bits but only 5 exponent bits, so every row
// (a token's x, or its h) is scaled by a power of two 2^e chosen from the row's
// largest magnitude, which then lands in [2^14, 2^15): all values of the row within
// 2^38 of its largest keep every bit they have in bf16 (x) or 11 bits (h).  The
// matching 2^-e is applied in the consumer's epilogue.
//
//   gather_rows_f16_kernel: x rows of the grouped order -> f16 (one pass, the row held
//                           in registers), rowmul[r] = 2^-e;
//                           also clears the per-row maxima that the gate_up
//                           epilogue accumulates for h, and (one warp) writes the
//                           GEMMs' item order and clears their unit counters.
//   h_fix_f16_kernel:       h rows, written by the gate_up epilogue as f16 times a
//                           fixed 2^kh with each row's largest |h|: rows whose
//                           largest |h| fits that scale keep it (hmul = 2^-kh); a row
//                           below 2^(-2 - kh) is re-staged from its fp32 copy with
//                           its own 2^e (hmul = 2^-e).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// e with m * 2^e in [2^14, 2^15) for the largest magnitude m of a row, given the
// biased exponent field of m (0 for a zero row, which then keeps e = 0; the field
// of inf / NaN also gives e = 0 so that they propagate).
__device__ __forceinline__ int row_exp_from_field(int ex, bool zero) {
  if (zero || ex == 255) return 0;
  return min(141 - ex, 126);
}

// The f16 row of bf16 values v (8 per 16-byte unit) times sc.
__device__ __forceinline__ uint4 scaled_f16x8(const uint4& v, float sc) {
  uint4 o;
  o.x = pack_f16x2(bf16_lo(v.x) * sc, bf16_hi(v.x) * sc);
  o.y = pack_f16x2(bf16_lo(v.y) * sc, bf16_hi(v.y) * sc);
  o.z = pack_f16x2(bf16_lo(v.z) * sc, bf16_hi(v.z) * sc);
  o.w = pack_f16x2(bf16_lo(v.w) * sc, bf16_hi(v.w) * sc);
  return o;
}

__device__ __forceinline__ uint32_t max_abs_bf16x8(const uint4& v) {
  const uint32_t mk = 0x7FFF7FFFu;
  return __vmaxu2(__vmaxu2(v.x & mk, v.y & mk), __vmaxu2(v.z & mk, v.w & mk));
}

// The item order of the MXFP4 grouped GEMMs, written by one warp: items of more than
// half_rows rows (two m tiles) first, in the work list's order, then the one-m-tile
// items from the end backwards.  The GEMMs' CTAs claim units in this order, so that
// the half-cost units come last and even out the CTAs' finishing times.
__device__ void order_items(const RouteState& rs, int half_rows, int32_t* __restrict__ order, int lane) {
  const int n = *rs.n_work;
  const uint32_t below = (1u << lane) - 1u;
  int nh = 0, nl = 0;
  for (int b = 0; b < n; b += 32) {
    const int i = b + lane;
    bool heavy = false;
    if (i < n) {
      const int2 w = rs.work[i];
      heavy = rs.offsets[w.x + 1] - rs.offsets[w.x] - w.y > half_rows;
    }
    const uint32_t hb = __ballot_sync(0xffffffffu, i < n && heavy);
    const uint32_t lb = __ballot_sync(0xffffffffu, i < n && !heavy);
    if (i < n) order[heavy ? nh + __popc(hb & below) : n - 1 - (nl + __popc(lb & below))] = i;
    nh += __popc(hb);
    nl += __popc(lb);
  }
}

// Warp per grouped row.  UNITS > 0: the row (at most 32 * UNITS 16-byte units) is
// loaded into registers at once (one round trip), its largest magnitude found and the
// row converted from the registers; UNITS == 0: any width, two passes over the row.
template <int UNITS>
__global__ void __launch_bounds__(256)
gather_rows_f16_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ row2slot, int S, int K,
                       int d, uint16_t* __restrict__ xp, float* __restrict__ rowmul,
                       uint32_t* __restrict__ hmax, const RouteState rs, int half_rows,
                       int32_t* __restrict__ order, int32_t* __restrict__ sched) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  if (order && blockIdx.x == 0 && threadIdx.x < 32) {
    order_items(rs, half_rows, order, lane);
    if (lane == 0) sched[0] = sched[1] = 0;
  }
  const int nvec = d / 8;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < S; r += (gridDim.x * blockDim.x) >> 5) {
    const int t = row2slot[r] / K;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)r * d);
    uint32_t m2 = 0;
    int e;
    if (UNITS > 0) {
      uint4 v[UNITS > 0 ? UNITS : 1];
#pragma unroll
      for (int j = 0; j < UNITS; ++j) {
        const int i = lane + 32 * j;
        v[j] = i < nvec ? ldg_nc_v4(src + i) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < UNITS; ++j) m2 = __vmaxu2(m2, max_abs_bf16x8(v[j]));
      const uint32_t m = __reduce_max_sync(0xffffffffu, max(m2 & 0xffffu, m2 >> 16));
      e = row_exp_from_field((int)(m >> 7), m == 0);                // bf16 exponent field
      const float sc = exp2i(e);
#pragma unroll
      for (int j = 0; j < UNITS; ++j) {
        const int i = lane + 32 * j;
        if (i < nvec) dst[i] = scaled_f16x8(v[j], sc);
      }
    } else {
      for (int i = lane; i < nvec; i += 32) m2 = __vmaxu2(m2, max_abs_bf16x8(ldg_nc_v4(src + i)));
      const uint32_t m = __reduce_max_sync(0xffffffffu, max(m2 & 0xffffu, m2 >> 16));
      e = row_exp_from_field((int)(m >> 7), m == 0);
      const float sc = exp2i(e);
      for (int i = lane; i < nvec; i += 32) dst[i] = scaled_f16x8(ldg_nc_v4(src + i), sc);
    }
    if (lane == 0) {
      rowmul[r] = exp2i(-e);
      if (hmax) hmax[r] = 0u;
    }
  }
  pdl_trigger();
}

__global__ void __launch_bounds__(256)
h_fix_f16_kernel(const float* __restrict__ hside, const uint32_t* __restrict__ hmax, int S, int ff, int kh,
                 uint16_t* __restrict__ h16, int ldh, float* __restrict__ hmul) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const float small = exp2i(-2 - kh);
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < S; r += (gridDim.x * blockDim.x) >> 5) {
    const uint32_t m = hmax[r];
    // NaN / inf compare false here and keep the fixed scale, so that they propagate
    if (!(__uint_as_float(m) < small)) {
      if (lane == 0) hmul[r] = exp2i(-kh);
      continue;
    }
    const int e = row_exp_from_field((int)(m >> 23), m == 0);       // fp32 exponent field
    const float sc = exp2i(e);
    const float4* src = reinterpret_cast<const float4*>(hside + (size_t)r * ldh);
    uint2* dst = reinterpret_cast<uint2*>(h16 + (size_t)r * ldh);
    for (int i = lane; i < ff / 4; i += 32) {
      const float4 v = src[i];
      dst[i] = make_uint2(pack_f16x2(v.x * sc, v.y * sc), pack_f16x2(v.z * sc, v.w * sc));
    }
    if (lane == 0) hmul[r] = exp2i(-e);
  }
  pdl_trigger();
}

int grid_rows(int S) {
  int blocks = (S + 7) / 8;
  if (blocks > 152 * 8) blocks = 152 * 8;
  return blocks < 1 ? 1 : blocks;
}

}  // namespace

cudaError_t launch_gather_rows_f16(const uint16_t* x, const int32_t* row2slot, int S, int K, int d, uint16_t* xp16,
                                   float* rowmul, uint32_t* hmax, const RouteState& rs, int half_rows,
                                   int32_t* order, int32_t* sched, cudaStream_t s) {
  const int units = (d / 8 + 31) / 32;   // 16-byte units per lane
  auto go = [&](auto kernel) {
    return launch_pdl(kernel, dim3(grid_rows(S)), dim3(256), 0, s, x, row2slot, S, K, d, xp16, rowmul, hmax, rs,
                      half_rows, order, sched);
  };
  if (units <= 8) return go(gather_rows_f16_kernel<8>);
  if (units <= 12) return go(gather_rows_f16_kernel<12>);
  if (units <= 16) return go(gather_rows_f16_kernel<16>);
  return go(gather_rows_f16_kernel<0>);
}

cudaError_t launch_h_fix_f16(const float* hside, const uint32_t* hmax, int S, int ff, int kh, uint16_t* h16,
                             int ldh, float* hmul, cudaStream_t s) {
  return launch_pdl(h_fix_f16_kernel, dim3(grid_rows(S)), dim3(256), 0, s, hside, hmax, S, ff, kh, h16, ldh, hmul);
}

}  // namespace moe
