// Combine: y[t] = (x[t] +) sum_j w[t, j] * Y[t*K + j] over a token's routed slots
// and, last, its shared-expert slot (weight = sigmoid gate), accumulated in fp32 in
// that fixed order (the residual first) and rounded once to bf16.  On the prefill
// path with cfg.deterministic = 0 the down projection has already added the weighted
// slots into a per-token fp32 sum, and the finish kernel only adds the residual and
// rounds.
// RMSNorm: the MoE's input RMSNorm(x) = x / sqrt(mean(x^2) + eps) * w, in bf16.
//
// Sources: "qwen35moe - Forward-Pass Design", section "Shared-expert MoE FFN"
// (out = moe_out + sgate * shexp) and "Block scaffold" (post_attention_norm; the
// residual adds the un-normalised input); "qwen35moe CPU-reference golden vectors",
// Kernel 3 (RMS = 1 / sqrt(mean(x^2) + eps)); "Phase 19: MoE - gpt-oss-20b",
// section 2 Experts (out = sum over the top-4 of scores * y_e), RMSNorm (fp32
// variance) and Decoder layer (out = h + moe(post_norm(h))).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

template <bool F32>
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ Y, const float* __restrict__ slot_w,
               const int32_t* __restrict__ slot_expert, int T, int K, int d, int E1,
               const uint16_t* __restrict__ resid, void* __restrict__ y) {
  pdl_wait();
  const int d8 = d / 8;
  const long n = (long)T * d8;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long t = i / d8;
    const int o = (int)(i - t * d8) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (resid) {
      const uint4 r = ldg_nc_v4(resid + (size_t)t * d + o);
      acc[0] = bf16_lo(r.x); acc[1] = bf16_hi(r.x); acc[2] = bf16_lo(r.y); acc[3] = bf16_hi(r.y);
      acc[4] = bf16_lo(r.z); acc[5] = bf16_hi(r.z); acc[6] = bf16_lo(r.w); acc[7] = bf16_hi(r.w);
    }
    // Slots in groups of four: every load of a group (expert, weight, Y row) is in
    // flight together, and the sums still take the slots in order.  A slot flagged by
    // the permute (expert out of range) contributes nothing: its Y row (in bounds, but
    // never written) is read and dropped by the select, not multiplied by zero.
#pragma unroll 2
    for (int j0 = 0; j0 < K; j0 += 4) {
      int v[4];
      float w[4];
      float4 a[4], b[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool in = j0 + q < K;
        const long s = t * K + (in ? j0 + q : 0);
        v[q] = in ? slot_expert[s] : -1;
        w[q] = in ? slot_w[s] : 0.f;
        const float4* src = reinterpret_cast<const float4*>(Y + (size_t)s * d + o);
        a[q] = src[0];
        b[q] = src[1];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (v[q] >= 0 && v[q] < E1) {
          acc[0] += w[q] * a[q].x; acc[1] += w[q] * a[q].y; acc[2] += w[q] * a[q].z; acc[3] += w[q] * a[q].w;
          acc[4] += w[q] * b[q].x; acc[5] += w[q] * b[q].y; acc[6] += w[q] * b[q].z; acc[7] += w[q] * b[q].w;
        }
      }
    }
    if (F32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(y) + (size_t)t * d + o);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      uint4 out;
      out.x = pack_bf16x2(acc[0], acc[1]);
      out.y = pack_bf16x2(acc[2], acc[3]);
      out.z = pack_bf16x2(acc[4], acc[5]);
      out.w = pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(y) + (size_t)t * d + o) = out;
    }
  }
  pdl_trigger();
}

// The accumulated prefill's last step: y[t] = (x[t] +) yacc[t], where yacc holds the
// token's weighted expert outputs (shared expert included) summed by the down
// projection's atomic adds.
template <bool F32>
__global__ void __launch_bounds__(256)
finish_kernel(const float* __restrict__ yacc, int T, int d, const uint16_t* __restrict__ resid,
              void* __restrict__ y) {
  pdl_wait();
  const int d8 = d / 8;
  const long n = (long)T * d8;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long t = i / d8;
    const int o = (int)(i - t * d8) * 8;
    const float4* src = reinterpret_cast<const float4*>(yacc + (size_t)t * d + o);
    const float4 a = src[0], b = src[1];
    float acc[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    if (resid) {
      const uint4 r = ldg_nc_v4(resid + (size_t)t * d + o);
      const float rv[8] = {bf16_lo(r.x), bf16_hi(r.x), bf16_lo(r.y), bf16_hi(r.y),
                           bf16_lo(r.z), bf16_hi(r.z), bf16_lo(r.w), bf16_hi(r.w)};
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = rv[j] + acc[j];
    }
    if (F32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(y) + (size_t)t * d + o);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      uint4 out;
      out.x = pack_bf16x2(acc[0], acc[1]);
      out.y = pack_bf16x2(acc[2], acc[3]);
      out.z = pack_bf16x2(acc[4], acc[5]);
      out.w = pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(y) + (size_t)t * d + o) = out;
    }
  }
  pdl_trigger();
}

// One warp per token row: sum of squares in fp32, r = 1 / sqrt(mean + eps), and
// xn = bf16(x * r * w).  Also the first kernel of a call that uses it: it clears the
// device status word.
__global__ void __launch_bounds__(256)
rmsnorm_kernel(const uint16_t* __restrict__ x, int T, int d, const uint16_t* __restrict__ w, float eps,
               uint16_t* __restrict__ xn, uint32_t* __restrict__ status) {
  pdl_wait();
  if (status && blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;
  const int lane = threadIdx.x & 31;
  const int d8 = d / 8;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    float ss = 0.f;
    for (int i = lane; i < d8; i += 32) {
      const uint4 v = ldg_nc_v4(src + i);
      const float a[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                          bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(a[j], a[j], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float r = 1.f / sqrtf(ss / (float)d + eps);
    uint4* dst = reinterpret_cast<uint4*>(xn + (size_t)t * d);
    const uint4* wv = reinterpret_cast<const uint4*>(w);
    for (int i = lane; i < d8; i += 32) {
      const uint4 v = ldg_nc_v4(src + i), g = ldg_nc_v4(wv + i);
      uint4 o;
      o.x = pack_bf16x2(bf16_lo(v.x) * r * bf16_lo(g.x), bf16_hi(v.x) * r * bf16_hi(g.x));
      o.y = pack_bf16x2(bf16_lo(v.y) * r * bf16_lo(g.y), bf16_hi(v.y) * r * bf16_hi(g.y));
      o.z = pack_bf16x2(bf16_lo(v.z) * r * bf16_lo(g.z), bf16_hi(v.z) * r * bf16_hi(g.z));
      o.w = pack_bf16x2(bf16_lo(v.w) * r * bf16_lo(g.w), bf16_hi(v.w) * r * bf16_hi(g.w));
      dst[i] = o;
    }
  }
  pdl_trigger();
}

}  // namespace

cudaError_t launch_combine(const float* Y, const float* slot_w, const int32_t* slot_expert, int T,
                           int K, int d, int E1, const uint16_t* resid, void* y, bool y_fp32,
                           cudaStream_t s) {
  const long n = (long)T * (d / 8);
  long blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (y_fp32)
    return launch_pdl(combine_kernel<true>, dim3((int)blocks), dim3(256), 0, s, Y, slot_w, slot_expert,
                      T, K, d, E1, resid, y);
  return launch_pdl(combine_kernel<false>, dim3((int)blocks), dim3(256), 0, s, Y, slot_w, slot_expert,
                    T, K, d, E1, resid, y);
}

cudaError_t launch_finish_accumulated(const float* yacc, int T, int d, const uint16_t* resid, void* y,
                                      bool y_fp32, cudaStream_t s) {
  const long n = (long)T * (d / 8);
  long blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  if (y_fp32) return launch_pdl(finish_kernel<true>, dim3((int)blocks), dim3(256), 0, s, yacc, T, d, resid, y);
  return launch_pdl(finish_kernel<false>, dim3((int)blocks), dim3(256), 0, s, yacc, T, d, resid, y);
}

cudaError_t launch_rmsnorm(const uint16_t* x, int T, int d, const uint16_t* w, float eps, uint16_t* xn,
                           uint32_t* status, cudaStream_t s) {
  int blocks = (T + 7) / 8;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  return launch_pdl(rmsnorm_kernel, dim3(blocks), dim3(256), 0, s, x, T, d, w, eps, xn, status);
}

}  // namespace moe
