// Decode path: a weight-streaming grouped matvec over the selected experts.
//
// Each CTA owns one (active expert, tile of weight rows) pair and streams those
// rows once from HBM with 16-byte loads, applying them to all of the expert's
// tokens: weights are the MMA's A operand (16 rows), tokens its N = 8 columns,
// so a handful of tokens per expert costs the same weight traffic as one.
// Experts with no tokens are never read.
//
// Operands are loaded straight from global memory into MMA fragments.  For a
// 16-row weight tile, lane (g, c) reads 16 contiguous bytes of rows g and g+8:
//   bf16  : inputs k0 + 8c .. +7, consumed by 2 MMAs (words {0,1}, {2,3});
//   MXFP4 : the whole 32-input block k0/32 + c (16 bytes of codes + one scale),
//           decoded to bf16 pairs and consumed by 8 MMAs (bytes {2j, 2j+1}).
// The token operand is read with the same input order, so the reordering of k
// inside a step leaves every dot product unchanged.
//
// Sources: "qwen35moe - Forward-Pass Design", section "Shared-expert MoE FFN"
// (SwiGLU experts, shared expert) and "K80 GPU decode" (grouped MoE: all top-k
// experts' gate+up+SwiGLU in one launch, then a fused down pass); "Phase 19:
// MoE - gpt-oss-20b", section 2 Experts (interleaved gate_up + bias, clamped GLU,
// down + bias) and section 3 (MXFP4).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kWarps = 4;
constexpr int kChunks = 4;                       // token chunks of 8 per pass
constexpr int kTokensPerPass = 8 * kChunks;
constexpr int kGateUpFeatures = kWarps * 16;     // features per CTA (2 tiles of 8 per warp)
constexpr int kDownRows = kWarps * 32;           // output rows per CTA (2 tiles of 16 per warp)

__device__ __forceinline__ float act_swiglu(float g, float u) {
  return g / (1.f + __expf(-g)) * u;
}

__device__ __forceinline__ float act_clamped(float g, float u, float limit, float alpha) {
  g = fminf(g, limit);
  u = fminf(fmaxf(u, -limit), limit);
  return (u + 1.f) * g / (1.f + __expf(-alpha * g));
}

// One MXFP4 block word set: 16 bytes of codes split into low / high nibbles.
struct Fp4Row {
  uint32_t lo[4], hi[4];
  Fp4Scale sc;
};

__device__ __forceinline__ Fp4Row fp4_row(uint4 w, uint32_t scale) {
  Fp4Row r;
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r.lo[i] = ws[i] & 0x0F0F0F0Fu;
    r.hi[i] = (ws[i] >> 4) & 0x0F0F0F0Fu;
  }
  r.sc = fp4_scale(scale);
  return r;
}

// bf16 pair of inputs (4j, 4j+1) [B = 0] or (4j+2, 4j+3) [B = 1] of the block.
template <int J, int B>
__device__ __forceinline__ uint32_t fp4_frag(const Fp4Row& r) {
  constexpr int byte = 2 * J + B;
  return fp4_pair<byte & 3>(r.lo[byte >> 2], r.hi[byte >> 2], r.sc);
}

// ---------------------------------------------------------------- gate_up + activation
//
// Tile i of a warp covers features f = f0 + 8i + g: A rows 0..7 are their gate
// rows, rows 8..15 their up rows, so the accumulator of lane (g, c) holds gate
// (d0, d1) and up (d2, d3) of feature f for tokens 2c and 2c+1.
template <int WFMT>
__global__ void __launch_bounds__(kWarps * 32)
gateup_decode_kernel(ExpertParams p, RouteState rs, const uint16_t* __restrict__ x, int K,
                     uint16_t* __restrict__ h, int ldh, int interleaved) {
  const int a = blockIdx.y;
  if (a >= *rs.n_active) return;
  const int v = rs.active[a];
  const bool shared = (v == p.E);
  if (WFMT == MOE_WFMT_MXFP4 && shared) return;   // rejected on the host
  const int ffv = shared ? p.sff : p.ff;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int f0 = blockIdx.x * kGateUpFeatures + warp * 16;
  if (f0 >= ffv) return;
  const int d = p.d;
  const int r0 = rs.offsets[v], cnt = rs.offsets[v + 1] - r0;
  const int fa = f0 + g, fb = f0 + 8 + g;          // lane's feature in tile 0 / tile 1

  // Row pointers (bf16) or block/scale pointers (MXFP4) of the lane's 4 weight rows.
  const uint8_t* rg[2];
  const uint8_t* ru[2];
  const uint8_t* sg[2] = {nullptr, nullptr};
  const uint8_t* su[2] = {nullptr, nullptr};
  float bias_g[2] = {0.f, 0.f}, bias_u[2] = {0.f, 0.f};
  const int fs[2] = {fa, fb};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int f = fs[i];
    if (WFMT == MOE_WFMT_BF16) {
      const size_t rowb = (size_t)d * 2;   // bytes per bf16 row
      if (shared) {
        rg[i] = reinterpret_cast<const uint8_t*>(p.sh_gate) + (size_t)f * rowb;
        ru[i] = reinterpret_cast<const uint8_t*>(p.sh_up) + (size_t)f * rowb;
      } else if (interleaved) {
        rg[i] = p.gate_up + ((size_t)v * 2 * p.ff + 2 * (size_t)f) * rowb;
        ru[i] = rg[i] + rowb;
      } else {
        rg[i] = reinterpret_cast<const uint8_t*>(p.gate) + ((size_t)v * p.ff + f) * rowb;
        ru[i] = reinterpret_cast<const uint8_t*>(p.up) + ((size_t)v * p.ff + f) * rowb;
      }
    } else {
      const size_t nb = (size_t)(d / 32);
      const size_t row = (size_t)v * 2 * p.ff + 2 * (size_t)f;
      rg[i] = p.gate_up + row * nb * 16;
      ru[i] = rg[i] + nb * 16;
      sg[i] = p.gu_scales + row * nb;
      su[i] = sg[i] + nb;
    }
    if (!shared && p.gu_bias) {
      const size_t row = (size_t)v * 2 * p.ff + 2 * (size_t)f;
      bias_g[i] = bf16_to_f32(p.gu_bias[row]);
      bias_u[i] = bf16_to_f32(p.gu_bias[row + 1]);
    }
  }
  const int act = shared ? MOE_ACT_SWIGLU : p.act;
  const uint4 z = make_uint4(0, 0, 0, 0);

  for (int p0 = 0; p0 < cnt; p0 += kTokensPerPass) {
    const int nch = min(kChunks, (cnt - p0 + 7) / 8);
    const uint8_t* xr[kChunks];
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
      const int i = p0 + 8 * ch + g;
      xr[ch] = (ch < nch && i < cnt)
                   ? reinterpret_cast<const uint8_t*>(x + (size_t)(rs.row2slot[r0 + i] / K) * d)
                   : nullptr;
    }
    float acc[2][kChunks][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][ch][q] = 0.f;

    if (WFMT == MOE_WFMT_BF16) {
#pragma unroll 2
      for (int k = 0; k < d; k += 32) {
        const size_t o = (size_t)(k + 8 * c) * 2;
        const uint4 g0 = ldg_stream_v4(rg[0] + o), u0 = ldg_stream_v4(ru[0] + o);
        const uint4 g1 = ldg_stream_v4(rg[1] + o), u1 = ldg_stream_v4(ru[1] + o);
#pragma unroll
        for (int ch = 0; ch < kChunks; ++ch) {
          if (ch < nch) {
            const uint4 b = xr[ch] ? ldg_nc_v4(xr[ch] + o) : z;
            mma_bf16_16816(acc[0][ch], g0.x, u0.x, g0.y, u0.y, b.x, b.y);
            mma_bf16_16816(acc[0][ch], g0.z, u0.z, g0.w, u0.w, b.z, b.w);
            mma_bf16_16816(acc[1][ch], g1.x, u1.x, g1.y, u1.y, b.x, b.y);
            mma_bf16_16816(acc[1][ch], g1.z, u1.z, g1.w, u1.w, b.z, b.w);
          }
        }
      }
    } else {
      const int nb = d / 32;
      for (int kb = 0; kb < nb; kb += 4) {
        const int blk = kb + c;
        const bool ok = blk < nb;
        Fp4Row G[2], U[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          G[i] = fp4_row(ok ? ldg_stream_v4(rg[i] + (size_t)blk * 16) : z, ok ? sg[i][blk] : 127u);
          U[i] = fp4_row(ok ? ldg_stream_v4(ru[i] + (size_t)blk * 16) : z, ok ? su[i][blk] : 127u);
        }
        const size_t xo = (size_t)blk * 64;   // bytes of x for this block
#define MOE_FP4_STEP(J)                                                                      \
  {                                                                                          \
    const uint32_t a00 = fp4_frag<J, 0>(G[0]), a01 = fp4_frag<J, 0>(U[0]);                   \
    const uint32_t a02 = fp4_frag<J, 1>(G[0]), a03 = fp4_frag<J, 1>(U[0]);                   \
    const uint32_t a10 = fp4_frag<J, 0>(G[1]), a11 = fp4_frag<J, 0>(U[1]);                   \
    const uint32_t a12 = fp4_frag<J, 1>(G[1]), a13 = fp4_frag<J, 1>(U[1]);                   \
    _Pragma("unroll") for (int ch = 0; ch < kChunks; ++ch) {                                 \
      if (ch < nch) {                                                                        \
        uint2 b = make_uint2(0, 0);                                                          \
        if (ok && xr[ch]) b = *reinterpret_cast<const uint2*>(xr[ch] + xo + 8 * (J));         \
        mma_bf16_16816(acc[0][ch], a00, a01, a02, a03, b.x, b.y);                            \
        mma_bf16_16816(acc[1][ch], a10, a11, a12, a13, b.x, b.y);                            \
      }                                                                                      \
    }                                                                                        \
  }
        MOE_FP4_STEP(0) MOE_FP4_STEP(1) MOE_FP4_STEP(2) MOE_FP4_STEP(3)
        MOE_FP4_STEP(4) MOE_FP4_STEP(5) MOE_FP4_STEP(6) MOE_FP4_STEP(7)
#undef MOE_FP4_STEP
      }
    }

    // Epilogue: bias, activation, bf16 h rows (permuted order).
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int ti = p0 + 8 * ch + 2 * c + q;
          if (ch < nch && ti < cnt) {
            const float gv = acc[i][ch][q] + bias_g[i];
            const float uv = acc[i][ch][2 + q] + bias_u[i];
            const float hv = act == MOE_ACT_SWIGLU ? act_swiglu(gv, uv)
                                                   : act_clamped(gv, uv, p.limit, p.alpha);
            h[(size_t)(r0 + ti) * ldh + fs[i]] = f32_to_bf16(hv);
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------- down
//
// Tile i of a warp covers output rows o0 + 16i + {g, g+8}; the accumulator of
// lane (g, c) holds rows (o, o+8) for tokens 2c, 2c+1.  Results (plus the down
// bias) go to the token's slot row of Y.
template <int WFMT>
__global__ void __launch_bounds__(kWarps * 32)
down_decode_kernel(ExpertParams p, RouteState rs, const uint16_t* __restrict__ h, int ldh,
                   float* __restrict__ Y) {
  const int a = blockIdx.y;
  if (a >= *rs.n_active) return;
  const int v = rs.active[a];
  const bool shared = (v == p.E);
  if (WFMT == MOE_WFMT_MXFP4 && shared) return;
  const int Kin = shared ? p.sff : p.ff;           // inputs of the down matrix
  const int d = p.d;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int o0 = blockIdx.x * kDownRows + warp * 32;
  if (o0 >= d) return;
  const bool tile1 = o0 + 16 < d;
  const int r0 = rs.offsets[v], cnt = rs.offsets[v + 1] - r0;

  const uint8_t* ra[2][2];     // [tile][row g / g+8]
  const uint8_t* sa[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};
  float bias[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      int o = o0 + 16 * i + g + 8 * hh;
      if (o >= d) o = d - 1;                       // tile 1 beyond d: clamped, never stored
      if (WFMT == MOE_WFMT_BF16) {
        const size_t rowb = (size_t)Kin * 2;
        ra[i][hh] = shared ? reinterpret_cast<const uint8_t*>(p.sh_down) + (size_t)o * rowb
                           : p.down + ((size_t)v * d + o) * rowb;
      } else {
        const size_t nb = (size_t)(Kin / 32);
        const size_t row = (size_t)v * d + o;
        ra[i][hh] = p.down + row * nb * 16;
        sa[i][hh] = p.dn_scales + row * nb;
      }
      if (!shared && p.dn_bias) bias[i][hh] = bf16_to_f32(p.dn_bias[(size_t)v * d + o]);
    }
  }
  const uint4 z = make_uint4(0, 0, 0, 0);

  for (int p0 = 0; p0 < cnt; p0 += kTokensPerPass) {
    const int nch = min(kChunks, (cnt - p0 + 7) / 8);
    const uint8_t* hr[kChunks];
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
      const int i = p0 + 8 * ch + g;
      hr[ch] = (ch < nch && i < cnt) ? reinterpret_cast<const uint8_t*>(h + (size_t)(r0 + i) * ldh)
                                     : nullptr;
    }
    float acc[2][kChunks][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][ch][q] = 0.f;

    if (WFMT == MOE_WFMT_BF16) {
#pragma unroll 2
      for (int k = 0; k < Kin; k += 32) {
        const size_t o = (size_t)(k + 8 * c) * 2;
        const uint4 a0 = ldg_stream_v4(ra[0][0] + o), a1 = ldg_stream_v4(ra[0][1] + o);
        const uint4 a2 = tile1 ? ldg_stream_v4(ra[1][0] + o) : z;
        const uint4 a3 = tile1 ? ldg_stream_v4(ra[1][1] + o) : z;
#pragma unroll
        for (int ch = 0; ch < kChunks; ++ch) {
          if (ch < nch) {
            const uint4 b = hr[ch] ? ldg_nc_v4(hr[ch] + o) : z;
            mma_bf16_16816(acc[0][ch], a0.x, a1.x, a0.y, a1.y, b.x, b.y);
            mma_bf16_16816(acc[0][ch], a0.z, a1.z, a0.w, a1.w, b.z, b.w);
            mma_bf16_16816(acc[1][ch], a2.x, a3.x, a2.y, a3.y, b.x, b.y);
            mma_bf16_16816(acc[1][ch], a2.z, a3.z, a2.w, a3.w, b.z, b.w);
          }
        }
      }
    } else {
      const int nb = Kin / 32;
      for (int kb = 0; kb < nb; kb += 4) {
        const int blk = kb + c;
        const bool ok = blk < nb;
        Fp4Row A[2][2];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const bool okr = ok && (i == 0 || tile1);
            A[i][hh] = fp4_row(okr ? ldg_stream_v4(ra[i][hh] + (size_t)blk * 16) : z,
                               okr ? sa[i][hh][blk] : 127u);
          }
        const size_t ho = (size_t)blk * 64;
#define MOE_FP4_STEP(J)                                                                      \
  {                                                                                          \
    const uint32_t a00 = fp4_frag<J, 0>(A[0][0]), a01 = fp4_frag<J, 0>(A[0][1]);             \
    const uint32_t a02 = fp4_frag<J, 1>(A[0][0]), a03 = fp4_frag<J, 1>(A[0][1]);             \
    const uint32_t a10 = fp4_frag<J, 0>(A[1][0]), a11 = fp4_frag<J, 0>(A[1][1]);             \
    const uint32_t a12 = fp4_frag<J, 1>(A[1][0]), a13 = fp4_frag<J, 1>(A[1][1]);             \
    _Pragma("unroll") for (int ch = 0; ch < kChunks; ++ch) {                                 \
      if (ch < nch) {                                                                        \
        uint2 b = make_uint2(0, 0);                                                          \
        if (ok && hr[ch]) b = *reinterpret_cast<const uint2*>(hr[ch] + ho + 8 * (J));         \
        mma_bf16_16816(acc[0][ch], a00, a01, a02, a03, b.x, b.y);                            \
        mma_bf16_16816(acc[1][ch], a10, a11, a12, a13, b.x, b.y);                            \
      }                                                                                      \
    }                                                                                        \
  }
        MOE_FP4_STEP(0) MOE_FP4_STEP(1) MOE_FP4_STEP(2) MOE_FP4_STEP(3)
        MOE_FP4_STEP(4) MOE_FP4_STEP(5) MOE_FP4_STEP(6) MOE_FP4_STEP(7)
#undef MOE_FP4_STEP
      }
    }

#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int ti = p0 + 8 * ch + 2 * c + q;
        if (ch < nch && ti < cnt) {
          float* yrow = Y + (size_t)rs.row2slot[r0 + ti] * d;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (i == 0 || tile1) {
              const int o = o0 + 16 * i + g;
              yrow[o] = acc[i][ch][q] + bias[i][0];
              yrow[o + 8] = acc[i][ch][2 + q] + bias[i][1];
            }
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_gateup_decode(const ExpertParams& p, int wfmt, int interleaved,
                                 const RouteState& rs, const uint16_t* x, int K, uint16_t* h,
                                 int ldh, int E1, cudaStream_t s) {
  const int ffmax = p.ff > p.sff ? p.ff : p.sff;
  dim3 grid((ffmax + kGateUpFeatures - 1) / kGateUpFeatures, E1);
  if (wfmt == MOE_WFMT_BF16)
    gateup_decode_kernel<MOE_WFMT_BF16><<<grid, kWarps * 32, 0, s>>>(p, rs, x, K, h, ldh, interleaved);
  else
    gateup_decode_kernel<MOE_WFMT_MXFP4><<<grid, kWarps * 32, 0, s>>>(p, rs, x, K, h, ldh, interleaved);
  return cudaGetLastError();
}

cudaError_t launch_down_decode(const ExpertParams& p, int wfmt, const RouteState& rs,
                               const uint16_t* h, int ldh, float* Y, int E1, cudaStream_t s) {
  dim3 grid((p.d + kDownRows - 1) / kDownRows, E1);
  if (wfmt == MOE_WFMT_BF16)
    down_decode_kernel<MOE_WFMT_BF16><<<grid, kWarps * 32, 0, s>>>(p, rs, h, ldh, Y);
  else
    down_decode_kernel<MOE_WFMT_MXFP4><<<grid, kWarps * 32, 0, s>>>(p, rs, h, ldh, Y);
  return cudaGetLastError();
}

}  // namespace moe
