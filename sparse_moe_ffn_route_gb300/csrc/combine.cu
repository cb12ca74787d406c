// Combine: y[t] = sum_j w[t, j] * Y[t*K + j] over a token's routed slots and,
// last, its shared-expert slot (weight = sigmoid gate), accumulated in fp32 in
// that fixed order and rounded once to bf16.
//
// Sources: "qwen35moe - Forward-Pass Design", section "Shared-expert MoE FFN"
// (out = moe_out + sgate * shexp); "Phase 19: MoE - gpt-oss-20b", section 2
// Experts (out = sum over the top-4 of scores * y_e).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

template <bool F32>
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ Y, const float* __restrict__ slot_w,
               const int32_t* __restrict__ slot_expert, int T, int K, int d, int E1,
               void* __restrict__ y) {
  pdl_wait();
  const int d8 = d / 8;
  const long n = (long)T * d8;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long t = i / d8;
    const int o = (int)(i - t * d8) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < K; ++j) {
      const long s = t * K + j;
      const int v = slot_expert[s];
      if (v < 0 || v >= E1) continue;          // flagged by the permute, contributes nothing
      const float w = slot_w[s];
      const float4* src = reinterpret_cast<const float4*>(Y + (size_t)s * d + o);
      const float4 a = src[0], b = src[1];
      acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
      acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
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

}  // namespace

cudaError_t launch_combine(const float* Y, const float* slot_w, const int32_t* slot_expert, int T,
                           int K, int d, int E1, void* y, bool y_fp32, cudaStream_t s) {
  const long n = (long)T * (d / 8);
  long blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (y_fp32)
    return launch_pdl(combine_kernel<true>, dim3((int)blocks), dim3(256), 0, s, Y, slot_w, slot_expert,
                      T, K, d, E1, y);
  return launch_pdl(combine_kernel<false>, dim3((int)blocks), dim3(256), 0, s, Y, slot_w, slot_expert,
                    T, K, d, E1, y);
}

}  // namespace moe
