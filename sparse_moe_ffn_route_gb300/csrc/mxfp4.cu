// Stand-alone MXFP4 -> bf16 decode (one thread per 32-input block), using the
// same decoder as the expert kernels' weight-load path.
//
// Source: "Phase 19: MoE - gpt-oss-20b", section 3 (value = fp4_lut[code] *
// 2^(e8m0 - 127)) and the section 2 tensor layout (low nibble = even input).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256)
mxfp4_to_bf16_kernel(const uint8_t* __restrict__ blocks, const uint8_t* __restrict__ scales,
                     long long n_blocks, uint16_t* __restrict__ out) {
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < n_blocks;
       b += (long long)gridDim.x * blockDim.x) {
    const uint4 w = ldg_nc_v4(blocks + b * 16);
    const Fp4Scale sc = fp4_scale(scales[b]);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = ws[i] & 0x0F0F0F0Fu, hi = (ws[i] >> 4) & 0x0F0F0F0Fu;
      o[4 * i + 0] = fp4_pair<0>(lo, hi, sc);
      o[4 * i + 1] = fp4_pair<1>(lo, hi, sc);
      o[4 * i + 2] = fp4_pair<2>(lo, hi, sc);
      o[4 * i + 3] = fp4_pair<3>(lo, hi, sc);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + b * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
  }
}

}  // namespace

cudaError_t launch_mxfp4_to_bf16(const uint8_t* blocks, const uint8_t* scales, long long rows,
                                 int n_in, uint16_t* out, cudaStream_t s) {
  const long long nb = rows * (n_in / 32);
  long long grid = (nb + 255) / 256;
  if (grid > 152 * 32) grid = 152 * 32;
  mxfp4_to_bf16_kernel<<<(int)grid, 256, 0, s>>>(blocks, scales, nb, out);
  return cudaGetLastError();
}

}  // namespace moe
