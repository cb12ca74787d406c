// Decode path: a weight-streaming grouped matvec over the selected experts.
//
// Each CTA owns one (work item, tile of weight rows) pair -- a work item is up to
// 8 or 32 of one expert's token rows -- and streams those weight rows once from
// HBM with 16-byte loads, applying them to all of the item's tokens: weights are
// the MMA's A operand (16 rows), tokens its N = 8 columns, so a handful of tokens
// per expert costs the same weight traffic as one.  Experts with no tokens are
// never read; an expert with many tokens (the shared expert) has many items, each
// re-reading the rows (from L2 after the first) in parallel.
//
// Operands are loaded straight from global memory into MMA fragments.  A lane
// (g, c) of a warp holds four weight rows (two 16-row tiles, rows g and g+8 of
// each) and reads 16 contiguous bytes of each per k step:
//   bf16  : inputs k0 + 8c .. +7, consumed by 2 MMAs (words {0,1}, {2,3});
//   MXFP4 : the whole 32-input block k0/32 + c (16 bytes of codes + one scale),
//           decoded to bf16 pairs and consumed by 8 MMAs (bytes {2j, 2j+1}).
// The token operand is read with the same input order, so the reordering of k
// inside a step leaves every dot product unchanged.  The weight loads run a
// fixed number of k steps ahead of the MMAs (a ring of registers), so that each
// warp keeps several kilobytes of HBM reads in flight.
//
// Sources: "qwen35moe - Forward-Pass Design", section "Shared-expert MoE FFN"
// (SwiGLU experts, shared expert) and "K80 GPU decode" (grouped MoE: all top-k
// experts' gate+up+SwiGLU in one launch, then a fused down pass); "Phase 19:
// MoE - gpt-oss-20b", section 2 Experts (interleaved gate_up + bias, clamped GLU,
// down + bias) and section 3 (MXFP4).
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxChunks = 4;                    // token chunks of 8 per pass (at most)
constexpr int kGateUpFeatures = kWarps * 16;     // features per CTA (2 tiles of 8 per warp)
constexpr int kDownRows = kWarps * 32;           // output rows per CTA (2 tiles of 16 per warp)
constexpr int kDepthBf16 = 4;                    // k steps of weight loads in flight (bf16)
constexpr int kDepthFp4 = 2;                     // k groups of weight loads in flight (MXFP4)
constexpr size_t kMaxStage = 48 * 1024;          // largest staged token-row block per CTA

__device__ __forceinline__ float act_swiglu(float g, float u) {
  return g / (1.f + __expf(-g)) * u;
}

__device__ __forceinline__ float act_clamped(float g, float u, float limit, float alpha) {
  g = fminf(g, limit);
  u = fminf(fmaxf(u, -limit), limit);
  return (u + 1.f) * g / (1.f + __expf(-alpha * g));
}

// 16 bytes of a token row: from shared memory (staged rows, generic pointer) or
// through the read-only path from global memory.
template <bool SB>
__device__ __forceinline__ uint4 ld_b16(const uint8_t* p) {
  if (SB) return *reinterpret_cast<const uint4*>(p);
  return ldg_nc_v4(p);
}

// 16 bytes from global memory through L2 only: data that other CTAs of the same
// launch wrote (the read-only path may not see them).
__device__ __forceinline__ uint4 ldg_cg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Copy `n` token rows of `rb` bytes (rows[i], global) into shared memory `dst`
// (row i at i * rb), all threads of the CTA, then synchronise.  CG: the rows were
// written during this launch.
template <bool CG = false>
__device__ __forceinline__ void stage_rows(uint8_t* dst, const uint8_t* const* rows, int n, int rb) {
  const int per = rb >> 4;
  for (int i = threadIdx.x; i < n * per; i += blockDim.x) {
    const int r = i / per, c = i - r * per;
    reinterpret_cast<uint4*>(dst + r * rb)[c] = CG ? ldg_cg_v4(rows[r] + 16 * c) : ldg_nc_v4(rows[r] + 16 * c);
  }
  __syncthreads();
}

// Bounded wait of a CTA until the counter *ctr reaches `need` (thread 0 polls with
// acquire loads; the block barrier passes the ordering on to every thread).  False,
// with STATUS_TIMEOUT set, if it gave up after the poll limit of the bounded waits
// (tc::c_wait_test, 2^20 polls by default).
__device__ __forceinline__ bool wait_count(const int32_t* ctr, int need, uint32_t* status) {
  __shared__ int ok_s;
  if (threadIdx.x == 0) {
    int ok = 0;
    const uint32_t polls = tc::c_wait_test.polls;
    for (uint32_t i = 0; i < polls; ++i) {
      int v;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= need) {
        ok = 1;
        break;
      }
      if (i > 64) __nanosleep(64);
    }
    if (!ok) flag_status(status, STATUS_TIMEOUT);
    ok_s = ok;
  }
  __syncthreads();
  return ok_s != 0;
}

// bf16 pair of the block's inputs (4j, 4j+1) [B = 0] or (4j+2, 4j+3) [B = 1].
// TWO: the scale needs the second multiply (scale byte > 128).
template <int J, int B, bool TWO>
__device__ __forceinline__ uint32_t fp4_frag(const uint4& w, const Fp4Scale& sc) {
  constexpr int byte = 2 * J + B;
  const uint32_t word = (byte >> 2) == 0 ? w.x : (byte >> 2) == 1 ? w.y : (byte >> 2) == 2 ? w.z : w.w;
  const uint32_t lo = word & 0x0F0F0F0Fu, hi = (word >> 4) & 0x0F0F0F0Fu;
  constexpr uint32_t sel = (uint32_t)(byte & 3) | (0x8u << 4) | ((uint32_t)(4 + (byte & 3)) << 8) |
                           (0x8u << 12);
  uint32_t p;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p) : "r"(lo), "r"(hi), "n"(sel));
  uint32_t v = bf16x2_mul((p * 0x1040u) & 0x81C081C0u, sc.first);
  if (TWO) v = bf16x2_mul(v, sc.second);
  return v;
}

// Eight MMAs of one MXFP4 k group for both tiles and all token chunks.
// W[0..3] are the lane's blocks of rows (tile0 row g, tile0 row g+8, tile1 row g,
// tile1 row g+8); xo is the byte offset of the block's 32 inputs in a token row.
template <bool TWO, int CH, bool LO, bool SB>
__device__ __forceinline__ void fp4_group_mma(const uint4 (&W)[4], const Fp4Scale (&S)[4],
                                              const uint8_t* const (&br)[CH], int nch,
                                              bool ok, size_t xo, float (&acc)[2][CH][4],
                                              size_t lo_off) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t a[2][4];
#define MOE_FRAGS(J)                                                                    \
  if (j == J) {                                                                         \
    a[0][0] = fp4_frag<J, 0, TWO>(W[0], S[0]); a[0][1] = fp4_frag<J, 0, TWO>(W[1], S[1]); \
    a[0][2] = fp4_frag<J, 1, TWO>(W[0], S[0]); a[0][3] = fp4_frag<J, 1, TWO>(W[1], S[1]); \
    a[1][0] = fp4_frag<J, 0, TWO>(W[2], S[2]); a[1][1] = fp4_frag<J, 0, TWO>(W[3], S[3]); \
    a[1][2] = fp4_frag<J, 1, TWO>(W[2], S[2]); a[1][3] = fp4_frag<J, 1, TWO>(W[3], S[3]); \
  }
    MOE_FRAGS(0) MOE_FRAGS(1) MOE_FRAGS(2) MOE_FRAGS(3)
    MOE_FRAGS(4) MOE_FRAGS(5) MOE_FRAGS(6) MOE_FRAGS(7)
#undef MOE_FRAGS
#pragma unroll
    for (int ch = 0; ch < CH; ++ch) {
      if (ch < nch) {
        uint2 b = make_uint2(0, 0);
        if (ok && br[ch]) b = *reinterpret_cast<const uint2*>(br[ch] + xo + 8 * j);
        mma_bf16_16816(acc[0][ch], a[0][0], a[0][1], a[0][2], a[0][3], b.x, b.y);
        mma_bf16_16816(acc[1][ch], a[1][0], a[1][1], a[1][2], a[1][3], b.x, b.y);
        if (LO) {
          uint2 l = make_uint2(0, 0);
          if (ok && br[ch]) l = *reinterpret_cast<const uint2*>(br[ch] + lo_off + xo + 8 * j);
          mma_bf16_16816(acc[0][ch], a[0][0], a[0][1], a[0][2], a[0][3], l.x, l.y);
          mma_bf16_16816(acc[1][ch], a[1][0], a[1][1], a[1][2], a[1][3], l.x, l.y);
        }
      }
    }
  }
}

// The first kDepthBf16 k steps of a bf16 weight ring: the loads a kernel issues
// before its token rows are staged, so that the weight stream does not wait on them.
__device__ __forceinline__ void prime_bf16(const uint8_t* const (&R)[4], int Kin, int c,
                                           uint4 (&W)[kDepthBf16][4]) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  const int nk = Kin >> 5;
#pragma unroll
  for (int s = 0; s < kDepthBf16; ++s)
#pragma unroll
    for (int r = 0; r < 4; ++r)
      W[s][r] = s < nk ? ldg_stream_v4(R[r] + (size_t)(s * 32 + 8 * c) * 2) : z;
}

// The streaming core shared by both kernels: acc[i][ch] += tile i (rows R[2i] /
// R[2i+1] as MMA rows g / g+8) times token chunk ch, over Kin inputs.
// R: byte pointers to the lane's 4 weight rows; Sc: their MXFP4 scale rows;
// br: byte pointers to the token rows (bf16) of the lane's B column per chunk.
// LO: the token operand is an (hi, lo) bf16 pair whose lo half sits lo_off bytes
// after the hi half in each row; both halves are multiplied by the same weights.
// SB: the token rows were staged in shared memory (br are generic pointers to it).
// W: bf16 weights, the ring as prime_bf16 left it (unused for MXFP4).
template <int WFMT, int CH, bool LO, bool SB>
__device__ __forceinline__ void stream_rows(const uint8_t* const (&R)[4],
                                            const uint8_t* const (&Sc)[4], int Kin, int c,
                                            const uint8_t* const (&br)[CH], int nch,
                                            float (&acc)[2][CH][4], size_t lo_off,
                                            uint4 (&W)[kDepthBf16][4]) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  if (WFMT == MOE_WFMT_BF16) {
    constexpr int P = kDepthBf16;
    const int nk = Kin >> 5;
    for (int k0 = 0; k0 < nk; k0 += P) {
#pragma unroll
      for (int s = 0; s < P; ++s) {
        const int kk = k0 + s;
        if (kk < nk) {
          const uint4 w0 = W[s][0], w1 = W[s][1], w2 = W[s][2], w3 = W[s][3];
          const int kn = kk + P;
          if (kn < nk) {
#pragma unroll
            for (int r = 0; r < 4; ++r) W[s][r] = ldg_stream_v4(R[r] + (size_t)(kn * 32 + 8 * c) * 2);
          }
          const size_t o = (size_t)(kk * 32 + 8 * c) * 2;
#pragma unroll
          for (int ch = 0; ch < CH; ++ch) {
            if (ch < nch) {
              const uint4 b = br[ch] ? ld_b16<SB>(br[ch] + o) : z;
              mma_bf16_16816(acc[0][ch], w0.x, w1.x, w0.y, w1.y, b.x, b.y);
              mma_bf16_16816(acc[0][ch], w0.z, w1.z, w0.w, w1.w, b.z, b.w);
              mma_bf16_16816(acc[1][ch], w2.x, w3.x, w2.y, w3.y, b.x, b.y);
              mma_bf16_16816(acc[1][ch], w2.z, w3.z, w2.w, w3.w, b.z, b.w);
              if (LO) {
                const uint4 l = br[ch] ? ld_b16<SB>(br[ch] + lo_off + o) : z;
                mma_bf16_16816(acc[0][ch], w0.x, w1.x, w0.y, w1.y, l.x, l.y);
                mma_bf16_16816(acc[0][ch], w0.z, w1.z, w0.w, w1.w, l.z, l.w);
                mma_bf16_16816(acc[1][ch], w2.x, w3.x, w2.y, w3.y, l.x, l.y);
                mma_bf16_16816(acc[1][ch], w2.z, w3.z, w2.w, w3.w, l.z, l.w);
              }
            }
          }
        }
      }
    }
  } else {
    constexpr int P = kDepthFp4;
    const int nb = Kin >> 5;                 // 32-input blocks per row
    const int ng = (nb + 3) >> 2;            // k groups of 4 blocks
    uint4 W[P][4];
    uint32_t S[P][4];
#pragma unroll
    for (int s = 0; s < P; ++s) {
      const int blk = 4 * s + c;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const bool ok = s < ng && blk < nb;
        W[s][r] = ok ? ldg_stream_v4(R[r] + (size_t)blk * 16) : z;
        S[s][r] = ok ? Sc[r][blk] : 127u;
      }
    }
    for (int g0 = 0; g0 < ng; g0 += P) {
#pragma unroll
      for (int s = 0; s < P; ++s) {
        const int gg = g0 + s;
        if (gg < ng) {
          const uint4 cw[4] = {W[s][0], W[s][1], W[s][2], W[s][3]};
          const uint32_t cs[4] = {S[s][0], S[s][1], S[s][2], S[s][3]};
          const int gn = gg + P;
          if (gn < ng) {
            const int blk = 4 * gn + c;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const bool ok = blk < nb;
              W[s][r] = ok ? ldg_stream_v4(R[r] + (size_t)blk * 16) : z;
              S[s][r] = ok ? Sc[r][blk] : 127u;
            }
          }
          const int blk = 4 * gg + c;
          const bool ok = blk < nb;
          Fp4Scale sc[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) sc[r] = fp4_scale(cs[r]);
          const bool big = (cs[0] | cs[1] | cs[2] | cs[3]) > 128u;   // any scale > 128
          if (__any_sync(0xffffffffu, big))
            fp4_group_mma<true, CH, LO, SB>(cw, sc, br, nch, ok, (size_t)blk * 64, acc, lo_off);
          else
            fp4_group_mma<false, CH, LO, SB>(cw, sc, br, nch, ok, (size_t)blk * 64, acc, lo_off);
        }
      }
    }
  }
}

// ---------------------------------------------------------------- MXFP4 x f16 tokens
//
// One-chunk MXFP4 items stage their token rows as f16, each row scaled by a power
// of two 2^e (e per token) that puts its largest magnitude in [2^14, 2^15): bf16
// rows convert exactly, and an (hi, lo) h row keeps 11 significant bits.  A weight
// code then decodes with one conversion instruction per byte (E2M1 values are
// exact in f16) and one f16 multiply by 2^(s - 127), which is exact while the
// scale byte s lies in [113, 140] (products stay normal-or-exact and below 65504).
// A k group in which some lane sees a scale outside that range takes the bf16
// decode instead and splits each f16 token value into an exact bf16 (hi, lo)
// pair.  The accumulators carry the token's 2^e; the epilogues remove it.
constexpr uint32_t kF16ScaleLo = 113, kF16ScaleSpan = 27;   // fast scale bytes: [113, 140]

// 16-byte units per staged f16 row: a multiple of 8 plus one, so that rows g of
// the 8 token columns start in different bank groups.
__host__ __device__ __forceinline__ int f16_row_units(int kin) { return (((kin >> 3) + 7) & ~7) + 1; }

// Unit u of a staged row sits at u ^ ((u >> 2) & 2): the lanes c and c + 2 of a
// quad, whose blocks are 128 bytes apart, then read different bank groups.
__device__ __forceinline__ int f16_unit(int u) { return u ^ ((u >> 2) & 2); }

// Exponent e of a token row from the bf16 bits of its largest magnitude.
__device__ __forceinline__ int token_exp(uint32_t m16) {
  const int E = (int)(m16 >> 7);
  if (m16 == 0 || E == 255) return 0;
  return min(141 - E, 126);
}

// Stage n (<= 8) token rows of kin values, one warp per row, as scaled f16 (layout
// above, row i at unit i * ru); esc[i] receives the row's exponent.  rows[i] is a
// bf16 row in global memory; PAIR: it is the hi half of an (hi, lo) pair whose lo
// half sits lo_off bytes further, and the staged value is hi + lo.
template <bool PAIR>
__device__ __forceinline__ void stage_rows_f16(uint8_t* dst, const uint8_t* const* rows, int n,
                                               int kin, int ru, size_t lo_off, int* esc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = kin >> 3;
  for (int r = warp; r < n; r += kWarps) {
    uint4* drow = reinterpret_cast<uint4*>(dst) + (size_t)r * ru;
    uint32_t m2 = 0;
    for (int u = lane; u < per; u += 32) {
      const uint4 v = ldg_nc_v4(rows[r] + 16 * u);
      drow[f16_unit(u)] = v;
      const uint32_t mask = 0x7FFF7FFFu;
      m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v.x & mask, v.y & mask), __vmaxu2(v.z & mask, v.w & mask)));
    }
    // the magnitude of lo is below half an ulp of hi: the max of hi sets e
    const int e = token_exp(__reduce_max_sync(0xffffffffu, max(m2 & 0xffffu, m2 >> 16)));
    const float s = exp2i(e);
    for (int u = lane; u < per; u += 32) {
      uint4* q = drow + f16_unit(u);
      const uint4 v = *q;                      // written by this lane above
      uint4 l = make_uint4(0, 0, 0, 0);
      if (PAIR) l = ldg_nc_v4(rows[r] + lo_off + 16 * u);
      uint4 o;
      o.x = pack_f16x2(s * (bf16_lo(v.x) + bf16_lo(l.x)), s * (bf16_hi(v.x) + bf16_hi(l.x)));
      o.y = pack_f16x2(s * (bf16_lo(v.y) + bf16_lo(l.y)), s * (bf16_hi(v.y) + bf16_hi(l.y)));
      o.z = pack_f16x2(s * (bf16_lo(v.z) + bf16_lo(l.z)), s * (bf16_hi(v.z) + bf16_hi(l.z)));
      o.w = pack_f16x2(s * (bf16_lo(v.w) + bf16_lo(l.w)), s * (bf16_hi(v.w) + bf16_hi(l.w)));
      *q = o;
    }
    if (lane == 0) esc[r] = e;
  }
  __syncthreads();
}

// Word q of a 16-byte block of codes.
__device__ __forceinline__ uint32_t word_of(const uint4& w, int q) {
  return q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w;
}

// One MXFP4 k group (the lane's block of each of its 4 rows) against the staged
// f16 token column b0 (null: empty column), fast decode: all scales in range.
// Word q of a block holds inputs 8q..8q+7 and feeds MMA j = 2q (bytes 4q, 4q+1)
// and j = 2q + 1 (bytes 4q+2, 4q+3); the token operand is the matching 16 bytes.
__device__ __forceinline__ void fp4h_group_fast(const uint4 (&W)[4], const uint32_t (&S)[4],
                                                const uint8_t* b0, const int (&qo)[4],
                                                float (&acc)[2][1][4]) {
  uint32_t sh[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t e = S[r] - 112u;           // f16 exponent field of 2^(s - 127)
    sh[r] = (e << 10) | (e << 26);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t f[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      e2m1x8_to_f16(word_of(W[r], q), f[r]);
#pragma unroll
      for (int t = 0; t < 4; ++t) f[r][t] = f16x2_mul(f[r][t], sh[r]);
    }
    const uint4 b = b0 ? *reinterpret_cast<const uint4*>(b0 + qo[q]) : make_uint4(0, 0, 0, 0);
    mma_f16_16816(acc[0][0], f[0][0], f[1][0], f[0][1], f[1][1], b.x, b.y);
    mma_f16_16816(acc[1][0], f[2][0], f[3][0], f[2][1], f[3][1], b.x, b.y);
    mma_f16_16816(acc[0][0], f[0][2], f[1][2], f[0][3], f[1][3], b.z, b.w);
    mma_f16_16816(acc[1][0], f[2][2], f[3][2], f[2][3], f[3][3], b.z, b.w);
  }
}

// bf16 pair of byte t of `word` (low nibble low), scaled (fp4_frag with a byte
// index known after unrolling).
__device__ __forceinline__ uint32_t fp4_byte_bf16(uint32_t word, int t, const Fp4Scale& sc, bool two) {
  const uint32_t lo = word & 0x0F0F0F0Fu, hi = (word >> 4) & 0x0F0F0F0Fu;
  const uint32_t sel = (uint32_t)t | (0x8u << 4) | ((uint32_t)(4 + t) << 8) | (0x8u << 12);
  uint32_t p;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p) : "r"(lo), "r"(hi), "r"(sel));
  uint32_t v = bf16x2_mul((p * 0x1040u) & 0x81C081C0u, sc.first);
  if (two) v = bf16x2_mul(v, sc.second);
  return v;
}

// The same k group when some scale is out of the fast range: bf16 weights, and
// each f16 token value split into bf16 hi + lo (exact: 11 = 8 + 3 bits).
template <bool TWO>
__device__ __forceinline__ void fp4h_group_split(const uint4 (&W)[4], const Fp4Scale (&S)[4],
                                                 const uint8_t* b0, const int (&qo)[4],
                                                 float (&acc)[2][1][4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 b = b0 ? *reinterpret_cast<const uint4*>(b0 + qo[q]) : make_uint4(0, 0, 0, 0);
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
    uint32_t bh[4], bl[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      float v0, v1;
      unpack_f16x2(bw[t], v0, v1);
      bh[t] = pack_bf16x2(v0, v1);
      bl[t] = pack_bf16x2(v0 - bf16_lo(bh[t]), v1 - bf16_hi(bh[t]));
    }
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      uint32_t a[4][2];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t w = word_of(W[r], q);
        a[r][0] = fp4_byte_bf16(w, 2 * jj, S[r], TWO);
        a[r][1] = fp4_byte_bf16(w, 2 * jj + 1, S[r], TWO);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mma_bf16_16816(acc[i][0], a[2 * i][0], a[2 * i + 1][0], a[2 * i][1], a[2 * i + 1][1],
                       bh[2 * jj], bh[2 * jj + 1]);
        mma_bf16_16816(acc[i][0], a[2 * i][0], a[2 * i + 1][0], a[2 * i][1], a[2 * i + 1][1],
                       bl[2 * jj], bl[2 * jj + 1]);
      }
    }
  }
}

// stream_rows for MXFP4 weights against one staged f16 token chunk (column b0 of
// this lane, null when empty): the same register ring of k groups.
__device__ __forceinline__ void stream_rows_fp4h(const uint8_t* const (&R)[4],
                                                 const uint8_t* const (&Sc)[4], int Kin, int c,
                                                 const uint8_t* b0, float (&acc)[2][1][4]) {
  constexpr int P = kDepthFp4;
  const uint4 z = make_uint4(0, 0, 0, 0);
  const int nb = Kin >> 5;
  const int ng = (nb + 3) >> 2;
  const int xq = c & 2;                        // the unit swizzle of this lane's blocks
  uint4 W[P][4];
  uint32_t S[P][4];
#pragma unroll
  for (int s = 0; s < P; ++s) {
    const int blk = 4 * s + c;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const bool ok = s < ng && blk < nb;
      W[s][r] = ok ? ldg_stream_v4(R[r] + (size_t)blk * 16) : z;
      S[s][r] = ok ? Sc[r][blk] : 127u;
    }
  }
  for (int g0 = 0; g0 < ng; g0 += P) {
#pragma unroll
    for (int s = 0; s < P; ++s) {
      const int gg = g0 + s;
      if (gg < ng) {
        const uint4 cw[4] = {W[s][0], W[s][1], W[s][2], W[s][3]};
        const uint32_t cs[4] = {S[s][0], S[s][1], S[s][2], S[s][3]};
        const int gn = gg + P;
        if (gn < ng) {
          const int blk = 4 * gn + c;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const bool ok = blk < nb;
            W[s][r] = ok ? ldg_stream_v4(R[r] + (size_t)blk * 16) : z;
            S[s][r] = ok ? Sc[r][blk] : 127u;
          }
        }
        const int blk = 4 * gg + c;
        // past the last block the codes are zero and the token operand must be too
        const uint8_t* bb = blk < nb ? b0 : nullptr;
        int qo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) qo[q] = 64 * blk + 16 * (q ^ xq);
        bool fast = true;
#pragma unroll
        for (int r = 0; r < 4; ++r) fast = fast && (cs[r] - kF16ScaleLo <= kF16ScaleSpan);
        if (__all_sync(0xffffffffu, fast)) {
          fp4h_group_fast(cw, cs, bb, qo, acc);
        } else {
          Fp4Scale sc[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) sc[r] = fp4_scale(cs[r]);
          const bool big = (cs[0] | cs[1] | cs[2] | cs[3]) > 128u;
          if (__any_sync(0xffffffffu, big))
            fp4h_group_split<true>(cw, sc, bb, qo, acc);
          else
            fp4h_group_split<false>(cw, sc, bb, qo, acc);
        }
      }
    }
  }
}

template <int CH>
__device__ __forceinline__ void zero_acc(float (&acc)[2][CH][4]) {
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int ch = 0; ch < CH; ++ch)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][ch][q] = 0.f;
}

// ---------------------------------------------------------------- gate_up + activation
//
// Tile i of a warp covers features f = f0 + 8i + g: its A rows 0..7 are their gate
// rows and rows 8..15 their up rows, so the accumulator of lane (g, c) holds gate
// (d0, d1) and up (d2, d3) of feature f for tokens 2c and 2c+1.
// STAGE: a one-chunk item (CH == 1) copies its token rows to shared memory first.
// One CTA's unit: work item a (below *rs.n_work), feature tile bx.
template <int WFMT, int CH, bool STAGE>
__device__ __forceinline__ void gateup_unit(const ExpertParams& p, const RouteState& rs,
                                            const uint16_t* __restrict__ x, int K, uint16_t* __restrict__ h,
                                            int ldh, int interleaved, int a, int bx) {
  const int2 item = rs.work[a];                    // (virtual expert, first row within it)
  const int v = item.x;
  const bool shared = (v == p.E);
  if (WFMT == MOE_WFMT_MXFP4 && shared) return;   // rejected on the host
  const int ffv = shared ? p.sff : p.ff;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int f0 = bx * kGateUpFeatures + warp * 16;
  // ff % 32 == 0: a warp's 16 features are all valid or all past the end; a warp
  // past the end still takes part in the row staging and its barriers.
  const bool warp_on = f0 < ffv;
  const int fclamp = warp_on ? f0 : 0;
  const int d = p.d;
  const int r0 = rs.offsets[v], cnt = min(rs.offsets[v + 1] - r0, item.y + 8 * CH);
  const int fs[2] = {fclamp + g, fclamp + 8 + g};  // lane's feature in tile 0 / tile 1

  // Byte pointers of the lane's rows: R = {gate f0+g, up f0+g, gate f0+8+g, up f0+8+g}.
  const uint8_t* R[4];
  const uint8_t* Sc[4] = {nullptr, nullptr, nullptr, nullptr};
  float bias_g[2] = {0.f, 0.f}, bias_u[2] = {0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int f = fs[i];
    if (WFMT == MOE_WFMT_BF16) {
      const size_t rowb = (size_t)d * 2;
      if (shared) {
        R[2 * i] = reinterpret_cast<const uint8_t*>(p.sh_gate) + (size_t)f * rowb;
        R[2 * i + 1] = reinterpret_cast<const uint8_t*>(p.sh_up) + (size_t)f * rowb;
      } else if (interleaved) {
        R[2 * i] = p.gate_up + ((size_t)v * 2 * p.ff + 2 * (size_t)f) * rowb;
        R[2 * i + 1] = R[2 * i] + rowb;
      } else {
        R[2 * i] = reinterpret_cast<const uint8_t*>(p.gate) + ((size_t)v * p.ff + f) * rowb;
        R[2 * i + 1] = reinterpret_cast<const uint8_t*>(p.up) + ((size_t)v * p.ff + f) * rowb;
      }
    } else {
      const size_t nb = (size_t)(d / 32);
      const size_t row = (size_t)v * 2 * p.ff + 2 * (size_t)f;
      R[2 * i] = p.gate_up + row * nb * 16;
      R[2 * i + 1] = R[2 * i] + nb * 16;
      Sc[2 * i] = p.gu_scales + row * nb;
      Sc[2 * i + 1] = Sc[2 * i] + nb;
    }
    if (!shared && p.gu_bias) {
      const size_t row = (size_t)v * 2 * p.ff + 2 * (size_t)f;
      bias_g[i] = bf16_to_f32(p.gu_bias[row]);
      bias_u[i] = bf16_to_f32(p.gu_bias[row + 1]);
    }
  }
  const int act = shared ? MOE_ACT_SWIGLU : p.act;
  uint4 W[kDepthBf16][4];
  if (WFMT == MOE_WFMT_BF16) prime_bf16(R, d, c, W);

  // MXFP4 with staged rows: f16 token operand (see "MXFP4 x f16 tokens")
  constexpr bool H16 = WFMT == MOE_WFMT_MXFP4 && STAGE;
  extern __shared__ __align__(16) uint8_t stage[];
  __shared__ int esc[8];                           // H16: token exponents
  for (int p0 = item.y; p0 < cnt; p0 += 8 * CH) {
    if (WFMT == MOE_WFMT_BF16 && p0 != item.y) prime_bf16(R, d, c, W);
    const int nch = min(CH, (cnt - p0 + 7) / 8);
    const uint8_t* br[CH];
    if (STAGE) {
      // one chunk: stage its (up to 8) x rows in shared memory for all warps
      __shared__ const uint8_t* rows[8];
      const int n = min(8, cnt - p0);
      if (threadIdx.x < n)
        rows[threadIdx.x] = reinterpret_cast<const uint8_t*>(x + (size_t)(rs.row2slot[r0 + p0 + threadIdx.x] / K) * d);
      __syncthreads();
      if (H16) {
        const int ru = f16_row_units(d);
        stage_rows_f16<false>(stage, rows, n, d, ru, 0, esc);
        br[0] = g < n ? stage + (size_t)g * ru * 16 : nullptr;
      } else {
        stage_rows(stage, rows, n, d * 2);
        br[0] = g < n ? stage + g * d * 2 : nullptr;
      }
    } else {
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) {
        const int i = p0 + 8 * ch + g;
        br[ch] = (ch < nch && i < cnt)
                     ? reinterpret_cast<const uint8_t*>(x + (size_t)(rs.row2slot[r0 + i] / K) * d)
                     : nullptr;
      }
    }
    float acc[2][CH][4];
    zero_acc(acc);
    if (!warp_on) continue;
    if constexpr (H16)
      stream_rows_fp4h(R, Sc, d, c, br[0], acc);
    else
      stream_rows<WFMT, CH, false, STAGE>(R, Sc, d, c, br, nch, acc, 0, W);
    pdl_trigger();

    // Epilogue: bias, activation, bf16 h rows (permuted order).
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int ti = p0 + 8 * ch + 2 * c + q;
          if (ch < nch && ti < cnt) {
            const float un = H16 ? exp2i(-esc[2 * c + q]) : 1.f;   // undo the token scale
            const float gv = acc[i][ch][q] * un + bias_g[i];
            const float uv = acc[i][ch][2 + q] * un + bias_u[i];
            const float hv = act == MOE_ACT_SWIGLU ? act_swiglu(gv, uv)
                                                   : act_clamped(gv, uv, p.limit, p.alpha);
            // h as a pair of bf16 (hi, lo = bf16(h - hi)): ~16 significant bits
            const uint16_t hi = f32_to_bf16(hv);
            uint16_t* hr = h + (size_t)(r0 + ti) * 2 * ldh + fs[i];
            hr[0] = hi;
            hr[ldh] = f32_to_bf16(hv - bf16_to_f32(hi));
          }
        }
      }
    }
  }
}

template <int WFMT, int CH, bool STAGE>
__global__ void __launch_bounds__(kWarps * 32, 3)
gateup_decode_kernel(ExpertParams p, RouteState rs, const uint16_t* __restrict__ x, int K,
                     uint16_t* __restrict__ h, int ldh, int interleaved) {
  pdl_wait();
  const int a = blockIdx.y;
  if (a >= *rs.n_work) return;
  gateup_unit<WFMT, CH, STAGE>(p, rs, x, K, h, ldh, interleaved, a, blockIdx.x);
}

// ---------------------------------------------------------------- down
//
// Tile i of a warp covers output rows o0 + 16i + {g, g+8}; the accumulator of
// lane (g, c) holds rows (o, o+8) for tokens 2c, 2c+1.  Results (plus the down
// bias) go to the token's slot row of Y.
// One CTA's unit: work item a (below *rs.n_work), output row tile bx.  The unit
// issues its first weight loads, then waits for its h rows: FUSED, until *ready
// reaches `need` (the fused launch, whose gate_up units count each finished item);
// otherwise for the preceding gate_up launch.
template <int WFMT, int CH, bool STAGE, bool FUSED>
__device__ __forceinline__ void down_unit(const ExpertParams& p, const RouteState& rs,
                                          const uint16_t* __restrict__ h, int ldh, float* __restrict__ Y,
                                          int a, int bx, const int32_t* ready, int need) {
  static_assert(!FUSED || (WFMT == MOE_WFMT_BF16 && CH == 1 && STAGE),
                "the fused launch reads h only through the coherent staging copy");
  const int2 item = rs.work[a];                    // (virtual expert, first row within it)
  const int v = item.x;
  const bool shared = (v == p.E);
  if (WFMT == MOE_WFMT_MXFP4 && shared) return;
  const int Kin = shared ? p.sff : p.ff;           // inputs of the down matrix
  const int d = p.d;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int o0raw = bx * kDownRows + warp * 32;
  // d % 32 == 0: both 16-row tiles of a warp are valid or both past the end; a warp
  // past the end still takes part in the row staging and its barriers.
  const bool warp_on = o0raw < d;
  const int o0 = warp_on ? o0raw : 0;
  const int r0 = rs.offsets[v], cnt = min(rs.offsets[v + 1] - r0, item.y + 8 * CH);

  // R = {o0+g, o0+8+g, o0+16+g, o0+24+g}: tile i uses rows (2i, 2i+1) as MMA rows g, g+8.
  const uint8_t* R[4];
  const uint8_t* Sc[4] = {nullptr, nullptr, nullptr, nullptr};
  float bias[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int o = o0 + 8 * r + g;
    if (WFMT == MOE_WFMT_BF16) {
      const size_t rowb = (size_t)Kin * 2;
      R[r] = shared ? reinterpret_cast<const uint8_t*>(p.sh_down) + (size_t)o * rowb
                    : p.down + ((size_t)v * d + o) * rowb;
    } else {
      const size_t nb = (size_t)(Kin / 32);
      const size_t row = (size_t)v * d + o;
      R[r] = p.down + row * nb * 16;
      Sc[r] = p.dn_scales + row * nb;
    }
    if (!shared && p.dn_bias) bias[r] = bf16_to_f32(p.dn_bias[(size_t)v * d + o]);
  }

  uint4 W[kDepthBf16][4];
  if (WFMT == MOE_WFMT_BF16) prime_bf16(R, Kin, c, W);
  // The weights and the work list (written by the grouping kernel, which every CTA
  // of the preceding gate_up launch waited for) do not depend on gate_up: only h does.
  if (FUSED) {
    if (!wait_count(ready, need, rs.status)) return;
  } else {
    pdl_wait();
  }

  constexpr bool H16 = WFMT == MOE_WFMT_MXFP4 && STAGE;
  extern __shared__ __align__(16) uint8_t stage[];
  __shared__ int esc[8];                           // H16: token exponents
  for (int p0 = item.y; p0 < cnt; p0 += 8 * CH) {
    if (WFMT == MOE_WFMT_BF16 && p0 != item.y) prime_bf16(R, Kin, c, W);
    const int nch = min(CH, (cnt - p0 + 7) / 8);
    const uint8_t* br[CH];
    size_t lo_off = (size_t)ldh * 2;
    if (H16) {
      // one chunk: stage its (up to 8) h rows as single scaled f16 rows
      __shared__ const uint8_t* rows[8];
      const int n = min(8, cnt - p0);
      if (threadIdx.x < n)
        rows[threadIdx.x] = reinterpret_cast<const uint8_t*>(h + (size_t)(r0 + p0 + threadIdx.x) * 2 * ldh);
      __syncthreads();
      const int ru = f16_row_units(Kin);
      stage_rows_f16<true>(stage, rows, n, Kin, ru, lo_off, esc);
      br[0] = g < n ? stage + (size_t)g * ru * 16 : nullptr;
    } else if (STAGE) {
      // one chunk: stage its (up to 8) h rows, hi then lo halves of Kin each
      __shared__ const uint8_t* rows[16];
      const int n = min(8, cnt - p0);
      if (threadIdx.x < 2 * n) {
        const int i = threadIdx.x >> 1;
        rows[threadIdx.x] = reinterpret_cast<const uint8_t*>(h + (size_t)(r0 + p0 + i) * 2 * ldh) +
                            (threadIdx.x & 1) * lo_off;
      }
      __syncthreads();
      stage_rows<FUSED>(stage, rows, 2 * n, Kin * 2);
      br[0] = g < n ? stage + 2 * g * Kin * 2 : nullptr;
      lo_off = (size_t)Kin * 2;
    } else {
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) {
        const int i = p0 + 8 * ch + g;
        br[ch] = (ch < nch && i < cnt) ? reinterpret_cast<const uint8_t*>(h + (size_t)(r0 + i) * 2 * ldh)
                                       : nullptr;
      }
    }
    float acc[2][CH][4];
    zero_acc(acc);
    if (!warp_on) continue;
    if constexpr (H16)
      stream_rows_fp4h(R, Sc, Kin, c, br[0], acc);
    else
      stream_rows<WFMT, CH, true, STAGE>(R, Sc, Kin, c, br, nch, acc, lo_off, W);
    pdl_trigger();

#pragma unroll
    for (int ch = 0; ch < CH; ++ch) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int ti = p0 + 8 * ch + 2 * c + q;
        if (ch < nch && ti < cnt) {
          float* yrow = Y + (size_t)rs.row2slot[r0 + ti] * d;
          const float un = H16 ? exp2i(-esc[2 * c + q]) : 1.f;     // undo the token scale
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int o = o0 + 16 * i + g;
            yrow[o] = acc[i][ch][q] * un + bias[2 * i];
            yrow[o + 8] = acc[i][ch][2 + q] * un + bias[2 * i + 1];
          }
        }
      }
    }
  }
}

template <int WFMT, int CH, bool STAGE>
__global__ void __launch_bounds__(kWarps * 32, 3)
down_decode_kernel(ExpertParams p, RouteState rs, const uint16_t* __restrict__ h, int ldh,
                   float* __restrict__ Y) {
  const int a = blockIdx.y;
  if (a >= *rs.n_work) return;
  down_unit<WFMT, CH, STAGE, false>(p, rs, h, ldh, Y, a, blockIdx.x, nullptr, 0);
}

// ---------------------------------------------------------------- gate_up + down, one launch
//
// One-chunk bf16 items: every CTA takes a ticket (rs.fuse[0]); tickets below
// n_work * gu_tiles are gate_up units in item order, the next n_work * dn_tiles are
// down units in item order, the rest exit.  A gate_up unit, once its h stores are
// fenced, adds one to its item's count (rs.fuse[1 + a]); a down unit streams its first
// weights and then waits until that count reaches gu_tiles.  Every ticket of a
// gate_up unit was taken, by a CTA already running, before the first down ticket,
// so the waits end whatever order the CTAs are scheduled in; the down units of the
// first items fill the SMs that the last gate_up units leave idle.
__global__ void __launch_bounds__(kWarps * 32, 3)
experts_decode_fused_kernel(ExpertParams p, RouteState rs, const uint16_t* __restrict__ x, int K,
                            uint16_t* __restrict__ h, int ldh, float* __restrict__ Y, int interleaved,
                            int gu_tiles, int dn_tiles) {
  pdl_wait();
  __shared__ int ticket_s, nw_s;
  if (threadIdx.x == 0) {
    ticket_s = atomicAdd(rs.fuse, 1);
    nw_s = *rs.n_work;                           // in flight with the ticket's round trip
  }
  __syncthreads();
  const int t = ticket_s, nw = nw_s;
  const int ngu = nw * gu_tiles;
  if (t < ngu) {
    const int a = t / gu_tiles;
    gateup_unit<MOE_WFMT_BF16, 1, true>(p, rs, x, K, h, ldh, interleaved, a, t - a * gu_tiles);
    __threadfence();            // this thread's h stores, before the item's count
    __syncthreads();
    // (the give-up test: the first unit withholds its count, so that item 0's down
    // units run out of polls)
    if (threadIdx.x == 0 && !tc::withheld_load(0, t == 0)) atomicAdd(rs.fuse + 1 + a, 1);
  } else if (t < ngu + nw * dn_tiles) {
    const int u = t - ngu, a = u / dn_tiles;
    down_unit<MOE_WFMT_BF16, 1, true, true>(p, rs, h, ldh, Y, a, u - a * dn_tiles, rs.fuse + 1 + a, gu_tiles);
  }
}

}  // namespace

// Dynamic shared memory of a one-chunk item: its token rows (gate_up: x rows of
// d inputs; down: h rows of the widest K).
template <class Kern>
static cudaError_t set_smem(Kern k, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t launch_gateup_decode(const ExpertParams& p, int wfmt, int interleaved,
                                 const RouteState& rs, const uint16_t* x, int K, uint16_t* h,
                                 int ldh, int max_items, int chunks, cudaStream_t s) {
  const int ffmax = p.ff > p.sff ? p.ff : p.sff;
  dim3 grid((ffmax + kGateUpFeatures - 1) / kGateUpFeatures, max_items);
  // staged x rows of a one-chunk item: bf16, or scaled f16 in padded rows (MXFP4)
  const size_t sm1 = wfmt == MOE_WFMT_BF16 ? (size_t)8 * p.d * 2 : (size_t)8 * f16_row_units(p.d) * 16;
#define MOE_GU(F, C, ST, SM)                                                                  \
  do {                                                                                        \
    cudaError_t e = set_smem(gateup_decode_kernel<F, C, ST>, SM);                            \
    if (e != cudaSuccess) return e;                                                           \
    e = launch_pdl(gateup_decode_kernel<F, C, ST>, grid, dim3(kWarps * 32), SM, s, p, rs, x, K, h, \
                   ldh, interleaved);                                                           \
    if (e != cudaSuccess) return e;                                                             \
  } while (0)
  const bool st = chunks == 1 && sm1 <= kMaxStage;
  if (wfmt == MOE_WFMT_BF16) {
    if (st) MOE_GU(MOE_WFMT_BF16, 1, true, sm1);
    else if (chunks == 1) MOE_GU(MOE_WFMT_BF16, 1, false, 0);
    else MOE_GU(MOE_WFMT_BF16, kMaxChunks, false, 0);
  } else {
    if (st) MOE_GU(MOE_WFMT_MXFP4, 1, true, sm1);
    else if (chunks == 1) MOE_GU(MOE_WFMT_MXFP4, 1, false, 0);
    else MOE_GU(MOE_WFMT_MXFP4, kMaxChunks, false, 0);
  }
#undef MOE_GU
  return cudaGetLastError();
}

// Shared memory of the fused launch: the larger staged block, x (8 rows of d bf16)
// for gate_up or h (8 (hi, lo) pairs of the wider FF) for down; 0 if over the limit.
static size_t fused_stage_bytes(int d, int ff, int sff) {
  const int fmax = ff > sff ? ff : sff;
  const size_t smx = (size_t)8 * d * 2, smh = (size_t)16 * fmax * 2;
  const size_t sm = smx > smh ? smx : smh;
  return sm <= kMaxStage ? sm : 0;
}

bool decode_fused_fits(int d, int ff, int sff) { return fused_stage_bytes(d, ff, sff) != 0; }

cudaError_t decode_set_wait_test(uint32_t polls, int withhold) { return tc::set_wait_test(polls, withhold); }

cudaError_t launch_experts_decode_fused(const ExpertParams& p, const RouteState& rs, const uint16_t* x, int K,
                                       uint16_t* h, int ldh, float* Y, int max_items, int interleaved,
                                       cudaStream_t s, bool* launched) {
  *launched = false;
  const int fmax = p.ff > p.sff ? p.ff : p.sff;
  const size_t sm = fused_stage_bytes(p.d, p.ff, p.sff);
  if (!rs.fuse || rs.fuse_n < 1 + max_items || sm == 0) return cudaSuccess;
  const int gu = (fmax + kGateUpFeatures - 1) / kGateUpFeatures, dn = (p.d + kDownRows - 1) / kDownRows;
  cudaError_t e = set_smem(experts_decode_fused_kernel, sm);
  if (e != cudaSuccess) return e;
  e = launch_pdl(experts_decode_fused_kernel, dim3((unsigned)((gu + dn) * max_items)), dim3(kWarps * 32), sm, s, p,
                 rs, x, K, h, ldh, Y, interleaved, gu, dn);
  if (e != cudaSuccess) return e;
  *launched = true;
  return cudaGetLastError();
}

cudaError_t launch_down_decode(const ExpertParams& p, int wfmt, const RouteState& rs,
                               const uint16_t* h, int ldh, float* Y, int max_items, int chunks,
                               cudaStream_t s) {
  dim3 grid((p.d + kDownRows - 1) / kDownRows, max_items);
  const int kmax = p.ff > p.sff ? p.ff : p.sff;
  // staged h rows of a one-chunk item: bf16 (hi, lo) pairs, or one scaled f16 row (MXFP4)
  const size_t sm1 = wfmt == MOE_WFMT_BF16 ? (size_t)16 * kmax * 2 : (size_t)8 * f16_row_units(kmax) * 16;
#define MOE_DN(F, C, ST, SM)                                                          \
  do {                                                                                \
    cudaError_t e = set_smem(down_decode_kernel<F, C, ST>, SM);                      \
    if (e != cudaSuccess) return e;                                                   \
    e = launch_pdl(down_decode_kernel<F, C, ST>, grid, dim3(kWarps * 32), SM, s, p, rs, h, ldh, Y); \
    if (e != cudaSuccess) return e;                                                   \
  } while (0)
  const bool st = chunks == 1 && sm1 <= kMaxStage;
  if (wfmt == MOE_WFMT_BF16) {
    if (st) MOE_DN(MOE_WFMT_BF16, 1, true, sm1);
    else if (chunks == 1) MOE_DN(MOE_WFMT_BF16, 1, false, 0);
    else MOE_DN(MOE_WFMT_BF16, kMaxChunks, false, 0);
  } else {
    if (st) MOE_DN(MOE_WFMT_MXFP4, 1, true, sm1);
    else if (chunks == 1) MOE_DN(MOE_WFMT_MXFP4, 1, false, 0);
    else MOE_DN(MOE_WFMT_MXFP4, kMaxChunks, false, 0);
  }
#undef MOE_DN
  return cudaGetLastError();
}

}  // namespace moe
