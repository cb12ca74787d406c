// Decode path for MXFP4 experts with few tokens per expert: an asynchronous weight
// stream through shared memory.
//
// One persistent CTA per SM takes a contiguous share of the units (work item of up
// to 8 token rows of one expert) x (128 weight rows; for gate_up, 64 at the ends of
// the shares, which are cut in 64-row halves so that no CTA has more than half a unit
// above the average), and re-stages its token rows only when the item changes.  Warp 16
// is the producer: one elected lane streams each unit's codes into a ring of
// shared-memory stages with TMA (two boxes of 128 rows x 128 bytes, 128-byte
// swizzle: 512 inputs of each row per stage) and the unit's E8M0 scale bytes with
// one bulk copy.  About 128 KB of weights are in flight per SM at any time, without
// holding registers.
//
// Warps 0..15 consume: warp w owns the tile pair w % 4 (rows 32 (w % 4) .. + 31 of
// the unit, two MMA tiles) and two adjacent 32-input blocks of every box (the pair
// turns with the unit).  An ldmatrix of the swizzled stage hands lane (g, c) the four
// code bytes 4c..4c+3 of one block of rows g and g+8, so both k16 MMAs of that block
// see inputs of that block only: the block's two MMAs give a fresh fp32 product that
// is scaled once by 2^(s - 127) into the output fragment.  The scale is exact in fp32
// for every byte (0 gives 2^-127, 255 NaN): a row's two scale bytes become a bf16
// pair with one hardware conversion, or, for rows of an odd number of blocks, come
// from a 256-entry table.  A block's token fragments serve both tiles of the pair.
// Codes become exact f16 pairs with cvt.rn.f16x2.e2m1x2.  The token operand is the
// item's rows staged in shared memory as f16 scaled by 2^e per token (largest
// magnitude in [2^14, 2^15)), so bf16 x is exact and h = hi + lo keeps 11 bits.
//
// At a unit's end the consumers leave their partial sums in shared memory and go on
// to the next unit.  Warps 17 and 18 (on two other schedulers, four tiles each)
// finish the unit meanwhile: they add the four block classes of each tile, remove
// 2^e, add the bias and write h (after the activation) or Y, so that this tail is
// off the consumers' path and no scheduler carries all of it.
//
// Sources: "Phase 19: MoE - gpt-oss-20b", section 2 Experts (interleaved gate_up
// with bias, clamped GLU, down with bias) and section 3 (MXFP4: E2M1 codes, low
// nibble first, one E8M0 scale per 32 inputs).
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int kTiles = 8;                         // 16-row MMA tiles per unit
constexpr int kClasses = 4;                       // block classes (adjacent block pairs of a box)
constexpr int kCW = kTiles / 2 * kClasses;        // consumer warps: one per (tile pair, block class)
constexpr int kEpiWarps = 2;                       // warp kCW produces, warps kCW + 1.. finish units
constexpr int kEpiTiles = kTiles / kEpiWarps;      // tiles finished by one epilogue warp
constexpr int kThreads = (kCW + 1 + kEpiWarps) * 32;
constexpr int kRows = 16 * kTiles;                // weight rows per unit
constexpr int kBoxBytes = kRows * 128;            // one TMA box: 128 rows x 128 bytes of codes
constexpr int kBlocksPerBox = 8;                  // 32-input blocks per box row
constexpr int kBoxes = 2;                         // boxes per ring stage
constexpr int kStageBytes = kBoxes * kBoxBytes;
constexpr int kBlocksPerStage = kBoxes * kBlocksPerBox;
constexpr int kMaxRingStages = 8;
constexpr int kTokens = 8;                        // token rows per work item
constexpr int kScaleBufs = 3;                     // scale buffers: a unit's scales land a unit ahead

// Shared memory, from a 1024-aligned base: ring stages | scale buffers (3) |
// scale table | partial sums | token rows.
struct F4Smem {
  int stages, nb;            // ring depth; 32-input blocks per weight row
  int scale_bytes;           // one scale buffer (kRows * nb, rounded to 16)
  int pitch;                 // bytes per staged token row
  int ring, scales, lut, part, tok, total;
};

__host__ __device__ inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

// Token row pitch: >= 2 * kin bytes and an odd multiple of 64, so that the rows of
// the 8 token columns read by one 8-lane phase fall in different bank groups.
__host__ __device__ inline int token_pitch(int kin) { return round_up(2 * kin, 128) + 64; }

__host__ __device__ inline F4Smem f4_smem(int kin, int stages) {
  F4Smem m;
  m.stages = stages;
  m.nb = kin / 32;
  m.scale_bytes = round_up(kRows * m.nb, 16);
  m.pitch = token_pitch(kin);
  m.ring = 0;
  m.scales = stages * kStageBytes;
  m.lut = m.scales + kScaleBufs * m.scale_bytes;
  m.part = m.lut + 256 * 4;                        // partial sums [pair][class][tile][32][4]
  m.tok = m.part + kCW * 2 * 32 * 16;
  m.total = m.tok + kTokens * m.pitch;
  return m;
}

// The activations divide with __fdividef (2 ulp): the IEEE division's slow path sits on
// the critical path at every unit's end.  A denominator that overflows to infinity
// gives 0, the limit of both functions there.
__device__ __forceinline__ float act_swiglu(float g, float u) { return __fdividef(g, 1.f + __expf(-g)) * u; }

__device__ __forceinline__ float act_clamped(float g, float u, float limit, float alpha) {
  g = fminf(g, limit);
  u = fminf(fmaxf(u, -limit), limit);
  return __fdividef((u + 1.f) * g, 1.f + __expf(-alpha * g));
}

// Barrier among the consumer warps only (the producer keeps streaming).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory");
}

// volatile: it reads shared memory that an mbarrier wait (volatile asm) made valid,
// so it must stay after that wait.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Contiguous global -> shared copy completing `bytes` of transaction count on
// `bar` (both addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Exponent e of a token row from the bf16 bits of its largest magnitude, so that
// the row times 2^e has its largest magnitude in [2^14, 2^15).
__device__ __forceinline__ int row_exp(uint32_t m16) {
  const int E = (int)(m16 >> 7);
  if (m16 == 0 || E == 255) return 0;
  return min(141 - E, 126);
}

// 16-byte units per lane kept in registers while staging (a half row of up to 192 * 8
// = 1536 inputs in one round trip; longer rows load twice).  17 warps leave 96
// registers per thread (5 warps share one scheduler's 16K registers).
constexpr int kStageUnits = 6;

__device__ __forceinline__ uint32_t max_abs_bf16x8(const uint4& v) {
  const uint32_t m = 0x7FFF7FFFu;
  return __vmaxu2(__vmaxu2(v.x & m, v.y & m), __vmaxu2(v.z & m, v.w & m));
}

__device__ __forceinline__ uint4 scaled_f16x8(const uint4& v, const uint4& l, float s) {
  uint4 o;
  o.x = pack_f16x2(s * (bf16_lo(v.x) + bf16_lo(l.x)), s * (bf16_hi(v.x) + bf16_hi(l.x)));
  o.y = pack_f16x2(s * (bf16_lo(v.y) + bf16_lo(l.y)), s * (bf16_hi(v.y) + bf16_hi(l.y)));
  o.z = pack_f16x2(s * (bf16_lo(v.z) + bf16_lo(l.z)), s * (bf16_hi(v.z) + bf16_hi(l.z)));
  o.w = pack_f16x2(s * (bf16_lo(v.w) + bf16_lo(l.w)), s * (bf16_hi(v.w) + bf16_hi(l.w)));
  return o;
}

// Stage the item's token rows (n <= 8; rows n..7 become zeros) as scaled f16: the
// two warps w and w + 8 take the halves of row w % 8.  Every lane issues all of its
// loads of a half row at once (up to kStageUnits 16-byte units), so that staging
// costs one round trip to memory for x rows and two for (hi, lo) h rows while the
// weight stream keeps the memory system busy.  rows[i] is a bf16 row of kin values in global memory; PAIR:
// the hi half of an (hi, lo) pair whose lo half is lo_off bytes further, and the
// staged value is hi + lo.  rmax[8] must be zero on entry; esc[i] receives row i's
// exponent.  Contains the consumer barriers that separate its two phases.
// pmax (PAIR only, or null): each row's largest |hi| (bf16 bits), already gathered by
// the producer of h; e then comes from it, and hi and lo load in one round trip with
// no barrier.
template <bool PAIR>
__device__ void stage_tokens(uint8_t* tok, int pitch, const uint8_t* const* rows, int n, int kin,
                             size_t lo_off, int* esc, uint32_t* rmax, int warp, int lane,
                             const uint32_t* pmax = nullptr) {
  const int r = warp % kTokens, hf = warp / kTokens;
  const int per = kin >> 3;                       // 16-byte units of bf16 input per row
  const int hu = (per + 1) >> 1;                  // units per half row
  const int ub = hf * hu, ue = min(per, ub + hu);
  const bool one = hu <= 32 * kStageUnits;        // the half row fits in registers
  uint4* drow = reinterpret_cast<uint4*>(tok + (size_t)r * pitch);
  const uint8_t* src = r < n ? rows[r] : nullptr;
  uint4 hv[kStageUnits], lv[kStageUnits];
  if (PAIR && pmax) {
    const int e = src ? row_exp(pmax[r]) : 0;
    const float s = exp2i(e);
    for (int u0 = ub; u0 < ue; u0 += 32 * kStageUnits) {
#pragma unroll
      for (int i = 0; i < kStageUnits; ++i) {
        const int u = u0 + lane + 32 * i;
        hv[i] = lv[i] = make_uint4(0, 0, 0, 0);
        if (src && u < ue) {
          hv[i] = ldg_nc_v4(src + 16 * u);
          lv[i] = ldg_nc_v4(src + lo_off + 16 * u);
        }
      }
#pragma unroll
      for (int i = 0; i < kStageUnits; ++i) {
        const int u = u0 + lane + 32 * i;
        if (u < ue) drow[u] = src ? scaled_f16x8(hv[i], lv[i], s) : make_uint4(0, 0, 0, 0);
      }
    }
    if (lane == 0 && hf == 0) esc[r] = e;
    return;
  }
  uint32_t m2 = 0;
  if (src) {
    for (int u0 = ub; u0 < ue; u0 += 32 * kStageUnits) {
#pragma unroll
      for (int i = 0; i < kStageUnits; ++i) {
        const int u = u0 + lane + 32 * i;
        hv[i] = make_uint4(0, 0, 0, 0);
        if (u < ue) hv[i] = ldg_nc_v4(src + 16 * u);
      }
#pragma unroll
      for (int i = 0; i < kStageUnits; ++i) m2 = __vmaxu2(m2, max_abs_bf16x8(hv[i]));
    }
    // |lo| is below half an ulp of hi: the largest hi sets e
    const uint32_t m = __reduce_max_sync(0xffffffffu, max(m2 & 0xffffu, m2 >> 16));
    if (lane == 0) atomicMax(&rmax[r], m);
  }
  consumers_sync();
  const int e = src ? row_exp(rmax[r]) : 0;
  const float s = exp2i(e);
  for (int u0 = ub; u0 < ue; u0 += 32 * kStageUnits) {
    // hi again when the row is longer than the registers; lo (PAIR) now
#pragma unroll
    for (int i = 0; i < kStageUnits; ++i) {
      const int u = u0 + lane + 32 * i;
      lv[i] = make_uint4(0, 0, 0, 0);
      if (src && u < ue) {
        if (!one) hv[i] = ldg_nc_v4(src + 16 * u);
        if (PAIR) lv[i] = ldg_nc_v4(src + lo_off + 16 * u);
      }
    }
#pragma unroll
    for (int i = 0; i < kStageUnits; ++i) {
      const int u = u0 + lane + 32 * i;
      if (u < ue) drow[u] = src ? scaled_f16x8(hv[i], lv[i], s) : make_uint4(0, 0, 0, 0);
    }
  }
  if (lane == 0 && hf == 0) esc[r] = e;
}

// D = A * B with a zero accumulator (f16 operands, fp32 result).
__device__ __forceinline__ void mma_f16_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// One 32-input block of one 16-row tile: wa / wb are this lane's code bytes of rows
// g and g + 8, B its token fragment, s0 / s1 the rows' block scales 2^(s - 127):
// the block's two k16 MMAs give a fresh product, which is scaled into acc.
__device__ __forceinline__ void block_mma(const uint32_t wa, const uint32_t wb, const uint4& B, float s0,
                                          float s1, float (&acc)[4]) {
  uint32_t fa[4], fb[4];
  e2m1x8_to_f16(wa, fa);
  e2m1x8_to_f16(wb, fb);
  float tt[4];
  mma_f16_zero(tt, fa[0], fb[0], fa[1], fb[1], B.x, B.y);
  mma_f16_16816(tt, fa[2], fb[2], fa[3], fb[3], B.z, B.w);
  acc[0] = fmaf(s0, tt[0], acc[0]);
  acc[1] = fmaf(s0, tt[1], acc[1]);
  acc[2] = fmaf(s1, tt[2], acc[2]);
  acc[3] = fmaf(s1, tt[3], acc[3]);
}

// Two E8M0 scale bytes (low byte first) as fp32 2^(s - 127) each, through the
// hardware conversion to a bf16 pair: exact for every byte, 0 giving 2^-127 and 255
// NaN, like the table.
__device__ __forceinline__ void e8m0x2_to_f32(uint16_t v, float& lo, float& hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.ue8m0x2 %0, %1;" : "=r"(r) : "h"(v));
  lo = __uint_as_float(r << 16);
  hi = __uint_as_float(r & 0xffff0000u);
}

// Blocks 2 qe and 2 qe + 1 (those below nblk) of one box for the two tiles of a pair:
// acc[t] += 2^(s - 127) * (block's codes x token rows), per block.  rbase: the lane's
// ldmatrix row in the box for the pair's first tile (the second's is 16 rows on);
// sc: the scale bytes of row g of the first tile; gb0: global block index of block
// 2 qe.  One x4 ldmatrix per tile hands lane (g, c) the code bytes 4c..4c+3 of rows g
// and g + 8 of both blocks; the token fragments of a block serve both tiles.
// PAIRED (an even number of blocks per row, so that gb0 and every row start are
// even): each row's two scale bytes come with one 16-bit load and one conversion;
// otherwise byte by byte through the table.
template <bool FULL, bool PAIRED>
__device__ __forceinline__ void box_pair(uint32_t rbase, int mi, int ri, int qe, const uint8_t* tg, const uint8_t* sc,
                                         int nb, const float* lut, int gb0, int nblk, float (&acc)[2][4]) {
  if (FULL) {
    // every operand first, so that their latencies overlap
    uint32_t r[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t) ldmatrix_x4(rbase + t * 16 * 128 + ((uint32_t)((2 * qe + (mi >> 1)) ^ ri) << 4), r[t]);
    uint4 B[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) B[k] = *reinterpret_cast<const uint4*>(tg + 64 * (gb0 + k));
    float sv[2][2][2];                            // [tile][block][row g / g + 8]
    if (PAIRED) {
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint16_t v = *reinterpret_cast<const uint16_t*>(sc + (16 * t + 8 * h) * nb + gb0);
          e8m0x2_to_f32(v, sv[t][0][h], sv[t][1][h]);
        }
    } else {
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
          for (int h = 0; h < 2; ++h) sv[t][k][h] = lut[sc[(16 * t + 8 * h) * nb + gb0 + k]];
    }
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int t = 0; t < 2; ++t) block_mma(r[t][2 * k], r[t][2 * k + 1], B[k], sv[t][k][0], sv[t][k][1], acc[t]);
  } else {
    if (2 * qe >= nblk) return;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      uint32_t r[4];
      ldmatrix_x4(rbase + t * 16 * 128 + ((uint32_t)((2 * qe + (mi >> 1)) ^ ri) << 4), r);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (2 * qe + k < nblk) {
          const int gb = gb0 + k;
          const uint4 B = *reinterpret_cast<const uint4*>(tg + 64 * gb);
          block_mma(r[2 * k], r[2 * k + 1], B, lut[sc[16 * t * nb + gb]], lut[sc[(16 * t + 8) * nb + gb]], acc[t]);
        }
      }
    }
  }
}

struct F4Args {
  RouteState rs;
  int R;                      // weight rows per expert: gate_up 2ff (gate, up interleaved), down d
  int kin;                    // inputs per weight row: gate_up d, down ff
  int tiles;                  // positions per work item: gate_up half units (kRows / 2 weight rows),
                              // down full units (kRows)
  int stages;                 // ring depth
  const uint8_t* scales;      // E8M0 [E, R, kin/32]
  const uint16_t* bias;       // bf16 [E, R] or null
  // gate_up: x rows in, h (hi, lo) rows out
  const uint16_t* x;
  int K;                      // slots per token (row2slot / K = token)
  uint16_t* h;
  int ldh;
  int act;
  float limit, alpha;
  // down: Y rows (slot order) out
  float* Y;
};

// The units of one CTA.  gate_up: the work is cut into half units (kRows / 2 weight rows
// of one work item) and every CTA takes an equal contiguous share of them, so that no
// CTA has more than half a unit above the average; within its share a CTA takes two
// halves of the same item, the first at an even position, as one full unit (a 128-row
// box), and a lone half at either end of the share, or the last 64 rows of an item, as
// a half unit (a 64-row box).  down: equal shares of full units (the last unit of an
// item may be short, and loads a 64-row box when it has at most 64 rows).  Every role
// of the CTA walks the same sequence.
struct UnitSeq {
  int p, end, tiles, R, ord;   // next position, end of the share, positions per item, rows per expert, units so far
  bool halves;                 // positions are half units (else full units of kRows rows)
};

struct F4Unit {
  int ai, row0, nrows, ord;    // work item, first weight row, rows (<= kRows), unit ordinal in the CTA
};

__device__ __forceinline__ bool next_unit(UnitSeq& q, F4Unit& u) {
  if (q.p >= q.end) return false;
  const int ai = q.p / q.tiles, th = q.p - ai * q.tiles;
  u.ai = ai;
  u.ord = q.ord++;
  if (!q.halves) {
    u.row0 = th * kRows;
    u.nrows = min(kRows, q.R - u.row0);
    q.p += 1;
    return true;
  }
  const bool full = (th & 1) == 0 && q.p + 1 < q.end && th + 1 < q.tiles;
  u.row0 = th * (kRows / 2);
  u.nrows = min(full ? kRows : kRows / 2, q.R - u.row0);
  q.p += full ? 2 : 1;
  return true;
}

// GATEUP: codes are gate_up [E, 2ff, d/2] bytes, tokens are x rows, output h.
// Otherwise: codes are down [E, d, ff/2], tokens are h rows, output Y.
// PAIRED: kin / 32 is even (scale bytes read two at a time).
template <bool GATEUP, bool PAIRED>
__global__ void __launch_bounds__(kThreads, 1)
fp4_stream_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW64,
                  const F4Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = tc::smem_align1024(smem_raw);
  __shared__ __align__(8) uint64_t full_bar[kMaxRingStages], empty_bar[kMaxRingStages], sfull_bar[kScaleBufs],
      sempty_bar[kScaleBufs], part_full, part_empty;
  __shared__ int abort_s;
  __shared__ int esc[2][kTokens];              // token exponents of the last two staged items
  __shared__ const uint8_t* trows[kTokens];
  __shared__ uint32_t rmax[kTokens];

  const F4Smem L = f4_smem(a.kin, a.stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = a.rs.status;
  volatile int* abort = &abort_s;
  float* lut = reinterpret_cast<float*>(smem + L.lut);

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      tc::mbar_init(tc::smem_u32(&full_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&empty_bar[i]), kCW * 32);   // every consumer lane arrives
    }
    for (int i = 0; i < kScaleBufs; ++i) {
      tc::mbar_init(tc::smem_u32(&sfull_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&sempty_bar[i]), kCW);
    }
    tc::mbar_init(tc::smem_u32(&part_full), kCW * 32);     // every consumer lane arrives
    tc::mbar_init(tc::smem_u32(&part_empty), kEpiWarps * 32);   // every epilogue lane arrives
    abort_s = 0;
    tc::fence_barrier_init();
  }
  // E8M0 byte -> 2^(s - 127) as fp32: 0 is 2^-127 (subnormal), 255 is NaN
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    lut[i] = i == 0 ? __uint_as_float(0x00400000u) : i == 255 ? __uint_as_float(0x7FC00000u) : exp2i(i - 127);
  if (warp == kCW && lane == 0) {
    tc::tma_prefetch_desc(&tmW);
    tc::tma_prefetch_desc(&tmW64);
  }
  __syncthreads();
  // gate_up: the work list comes from the grouping kernel just before.  down: the work
  // list was there before the gate_up launch let this one start (each of its CTAs
  // waited for the grouping); only h depends on gate_up, and the consumers wait for it
  // before they stage it.  The producer waits too, so that its weight stream does not
  // take bandwidth from gate_up's last units.
  if (GATEUP || warp == kCW) pdl_wait();

  const int n_items = *a.rs.n_work;
  const long long H = (long long)(n_items > 0 ? n_items : 0) * a.tiles;
  const int h0 = (int)(H * blockIdx.x / gridDim.x), h1 = (int)(H * (blockIdx.x + 1) / gridDim.x);
  const UnitSeq seq0{h0, h1, a.tiles, a.R, 0, GATEUP};
  const int nst = (L.nb + kBlocksPerStage - 1) / kBlocksPerStage;   // stages per unit

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    if (tc::elect_one()) {
      int it = 0, its = 0;                      // ring loads, scale loads issued
      int withheld = -1;                        // the load skipped by the give-up test
      int st = 0;                               // ring slot of load `it`
      uint32_t ph = 0;                          // its phase parity
      // The scale bytes of the CTA's n-th unit go to buffer n % kScaleBufs and are
      // requested a unit ahead of its codes, so that the copy has a whole unit's time to
      // land; the buffer's previous unit (n - 3) is long done by then.
      auto load_scales = [&](const F4Unit& un) -> bool {
        const int v = a.rs.work[un.ai].x;
        const int nrows = un.nrows;
        const long long grow = (long long)v * a.R + un.row0;
        const int sb = its % kScaleBufs;
        if (!tc::mbar_wait(tc::smem_u32(&sempty_bar[sb]), ((its / kScaleBufs) & 1) ^ 1, abort, status))
          return false;
        const uint32_t sbytes = (uint32_t)(nrows * L.nb);
        tc::mbar_arrive_expect_tx(tc::smem_u32(&sfull_bar[sb]), sbytes);
        bulk_load(tc::smem_u32(smem + L.scales + sb * L.scale_bytes), a.scales + grow * L.nb, sbytes,
                  tc::smem_u32(&sfull_bar[sb]));
        ++its;
        return true;
      };
      UnitSeq ahead = seq0;                     // runs one unit ahead (its scales go first)
      F4Unit un, nx;
      bool has_next = next_unit(ahead, nx);
      bool live = !has_next || load_scales(nx);
      while (live && !*abort && has_next) {
        un = nx;
        has_next = next_unit(ahead, nx);
        if (has_next && !load_scales(nx)) break;
        const int v = a.rs.work[un.ai].x;
        const long long grow = (long long)v * a.R + un.row0;
        const bool half = un.nrows <= kRows / 2;
        const CUtensorMap* wm = half ? &tmW64 : &tmW;
        const uint32_t box_bytes = half ? kBoxBytes / 2 : kBoxBytes;
        for (int s = 0; s < nst; ++s) {
          if (!tc::mbar_wait(tc::smem_u32(&empty_bar[st]), ph ^ 1, abort, status)) break;
          // A slot freed by an abort is not refilled: its last load may still be landing.
          if (*abort) break;
          if (tc::withheld_load(it, h0 == 0)) {     // the CTA that owns the first unit
            // the give-up test: this load is never issued, so its stage never fills
            withheld = it++;
            if (++st == a.stages) {
              st = 0;
              ph ^= 1;
            }
            continue;
          }
          // only the boxes that start inside the row (kin / 2 bytes)
          const int k0 = s * kBoxes * 128;
          const int nbox = min(kBoxes, (a.kin / 2 - k0 + 127) / 128);
          tc::mbar_arrive_expect_tx(tc::smem_u32(&full_bar[st]), (uint32_t)nbox * box_bytes);
          for (int j = 0; j < nbox; ++j)
            tc::tma_load_2d(tc::smem_u32(smem + st * kStageBytes + j * kBoxBytes), wm, k0 + 128 * j,
                            (int)grow, tc::smem_u32(&full_bar[st]));
          ++it;
          if (++st == a.stages) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      if (*abort) {
        // Drain: wait (bounded, regardless of the abort flag) for the most recent load
        // into every buffer, so that no copy lands after the CTA has exited.
        int zero = 0;
        volatile int* never = &zero;
        for (int i = it - a.stages > 0 ? it - a.stages : 0; i < it; ++i)
          if (i != withheld)
            tc::mbar_wait(tc::smem_u32(&full_bar[i % a.stages]), (i / a.stages) & 1, never, status);
        for (int i = its - kScaleBufs > 0 ? its - kScaleBufs : 0; i < its; ++i)
          tc::mbar_wait(tc::smem_u32(&sfull_bar[i % kScaleBufs]), (i / kScaleBufs) & 1, never, status);
      }
    }
    // no early signal to the dependent launch: the consumers give it when the CTA's
    // work is done
    return;
  }

  if (warp > kCW) {
    // ------------------------------------------------------------ epilogue warps
    // Finish every unit while the consumers stream the next one: each adds the four
    // block classes' partial sums of each tile (in class order), removes the tokens'
    // 2^e, adds the bias and writes h (gate_up, after the activation) or Y (down).
    // The partial-sum buffer is single: the consumers write a unit's sums once both
    // warps have read the previous unit's.  Lane (g, c) holds, per tile, rows g and
    // g + 8 for tokens 2c and 2c + 1.
    const int g = lane >> 2, c = lane & 3;
    const bool odd = g & 1;
    const int tile0 = (warp - kCW - 1) * kEpiTiles;   // this warp's tiles: tile0 .. + kEpiTiles - 1
    const float4* part = reinterpret_cast<const float4*>(smem + L.part) + lane;
    int cur = -1, ns = 0, nu = 0;                // staged item, items staged, units finished
    UnitSeq seq = seq0;
    F4Unit un;
    while (next_unit(seq, un)) {
      const int ai = un.ai;
      const int2 item = a.rs.work[ai];
      const int v = item.x;
      const int r0 = a.rs.offsets[v] + item.y;
      const int n = min(kTokens, a.rs.offsets[v + 1] - r0);
      if (ai != cur) {
        cur = ai;
        ++ns;
      }
      const int row0 = un.row0, nrows = un.nrows;
      // biases and output rows first, so that their round trips overlap the wait
      uint32_t bias[kEpiTiles];                  // two bf16: (gate, up) of feature f, or rows o, o + 8
#pragma unroll
      for (int i = 0; i < kEpiTiles; ++i) {
        const int tile = tile0 + i;
        bias[i] = 0;
        if (a.bias && 16 * tile < nrows) {
          const uint16_t* bp = a.bias + (size_t)v * a.R +
                               (GATEUP ? 2 * (row0 / 2 + 8 * tile + (odd ? 4 : 0) + (g >> 1)) : row0 + 16 * tile + g);
          bias[i] = (uint32_t)bp[0] | ((uint32_t)bp[GATEUP ? 1 : 8] << 16);
        }
      }
      int yslot[2] = {-1, -1};
      if (!GATEUP) {
#pragma unroll
        for (int k = 0; k < 2; ++k)
          if (2 * c + k < n) yslot[k] = a.rs.row2slot[r0 + 2 * c + k];
      }
      if (!tc::mbar_wait(tc::smem_u32(&part_full), nu & 1, abort, status)) break;
      float acc[kEpiTiles][4];
#pragma unroll
      for (int i = 0; i < kEpiTiles; ++i) {
        const int tile = tile0 + i;
        acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        if (16 * tile < nrows) {
#pragma unroll
          for (int qq = 0; qq < kClasses; ++qq) {
            const float4 o = part[(((tile >> 1) * kClasses + qq) * 2 + (tile & 1)) * 32];
            acc[i][0] += o.x;
            acc[i][1] += o.y;
            acc[i][2] += o.z;
            acc[i][3] += o.w;
          }
        }
      }
      const float un[2] = {exp2i(-esc[(ns - 1) & 1][2 * c]), exp2i(-esc[(ns - 1) & 1][2 * c + 1])};
      tc::mbar_arrive(tc::smem_u32(&part_empty));
      ++nu;
      if (*abort) break;
      uint32_t hm[2] = {0u, 0u};                 // gate_up: the largest |hi| of tokens 2c, 2c + 1
#pragma unroll
      for (int i = 0; i < kEpiTiles; ++i) {
        const int tile = tile0 + i;
        if (16 * tile >= nrows) break;
        const float b0 = bf16_to_f32((uint16_t)(bias[i] & 0xffffu)), b1 = bf16_to_f32((uint16_t)(bias[i] >> 16));
        if (GATEUP) {
          // MMA row i is memory row row0 + 16 tile + i: feature (row0 + 16 tile + i) / 2,
          // its gate when i is even.  Lanes g and g^1 (lane ^ 4) trade sums: even g
          // finishes the feature of its row g, odd g the feature of its row g + 8.
          float pr[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) pr[k] = __shfl_xor_sync(0xffffffffu, acc[i][k], 4);
          const int f = row0 / 2 + 8 * tile + (odd ? 4 : 0) + (g >> 1);
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int ti = 2 * c + k;
            if (ti < n) {
              const float gv = (odd ? pr[2 + k] : acc[i][k]) * un[k] + b0;
              const float uv = (odd ? acc[i][2 + k] : pr[k]) * un[k] + b1;
              const float hv =
                  a.act == MOE_ACT_SWIGLU ? act_swiglu(gv, uv) : act_clamped(gv, uv, a.limit, a.alpha);
              // h as a pair of bf16 (hi, lo = bf16(h - hi)), the layout both down paths read
              const uint16_t hi = f32_to_bf16(hv);
              uint16_t* hr = a.h + (size_t)(r0 + ti) * 2 * a.ldh + f;
              hr[0] = hi;
              hr[a.ldh] = f32_to_bf16(hv - bf16_to_f32(hi));
              hm[k] = max(hm[k], (uint32_t)(hi & 0x7FFFu));
            }
          }
        } else {
          const int o = row0 + 16 * tile + g;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (yslot[k] >= 0) {
              float* yrow = a.Y + (size_t)yslot[k] * a.R;
              yrow[o] = acc[i][k] * un[k] + b0;
              yrow[o + 8] = acc[i][2 + k] * un[k] + b1;
            }
          }
        }
      }
      if (GATEUP && a.rs.hmax) {
        // the unit's largest |hi| per token, over the 8 lanes (g) of each token pair,
        // into the row's maximum for the down staging (the same bf16 bits that staging
        // would find: NaN above inf above every finite value)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint32_t m = hm[k];
          m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
          m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
          m = max(m, __shfl_xor_sync(0xffffffffu, m, 16));
          if (g == 0 && 2 * c + k < n && m) atomicMax(a.rs.hmax + r0 + 2 * c + k, m);
        }
      }
    }
    pdl_trigger();
    return;
  }

  // -------------------------------------------------------------- consumers
  // Warp w owns tile pair tp = w % 4 (rows 32 tp .. 32 tp + 31 of the unit) and, in
  // every box, the two adjacent blocks of class qe = (w / 4 + unit) mod 4: a block's
  // token fragments serve both tiles.  At the unit's end every warp leaves its two
  // tiles' partial sums in shared memory for the epilogue warp and goes on.
  const int tp = warp % (kTiles / 2), q = warp / (kTiles / 2);
  const int g = lane >> 2, c = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;        // this lane's ldmatrix address: matrix, row
  uint8_t* tok = smem + L.tok;
  const uint8_t* tg = tok + g * L.pitch + 16 * c; // token column g, inputs 8c.. of each block
  float4* part = reinterpret_cast<float4*>(smem + L.part) + (tp * kClasses) * 2 * 32 + lane;
  int st = 0, its = 0, cur = -1;               // ring slot, scale loads consumed, staged item
  int ns = 0, nu = 0;                            // items staged, units handed to the epilogue warp
  uint32_t ph = 0;                               // phase parity of ring slot st
  UnitSeq seq = seq0;
  F4Unit un;
  while (next_unit(seq, un)) {
    // On abort every wait returns at once; the loop still runs to its end so that
    // all consumer warps take the same barriers.
    const int ai = un.ai;
    const int2 item = a.rs.work[ai];
    const int v = item.x;
    const int r0 = a.rs.offsets[v] + item.y;     // first permuted row of the item
    const int n = min(kTokens, a.rs.offsets[v + 1] - r0);
    if (ai != cur) {
      consumers_sync();                          // every warp is done with the old rows
      if (threadIdx.x < kTokens) {
        const int i = threadIdx.x;
        rmax[i] = 0;
        const uint8_t* p = nullptr;
        if (i < n) {
          if (GATEUP)
            p = reinterpret_cast<const uint8_t*>(a.x + (size_t)(a.rs.row2slot[r0 + i] / a.K) * a.kin);
          else
            p = reinterpret_cast<const uint8_t*>(a.h + (size_t)(r0 + i) * 2 * a.ldh);
        }
        trows[i] = p;
      }
      consumers_sync();
      // down: h is gate_up's output, the first thing here that needs it
      if (!GATEUP && ns == 0) pdl_wait();
      // the epilogue warp has read the exponents of every unit of the item two back
      stage_tokens<!GATEUP>(tok, L.pitch, trows, n, a.kin, (size_t)a.ldh * 2, esc[ns & 1], rmax, warp, lane,
                            GATEUP || !a.rs.hmax ? nullptr : a.rs.hmax + r0);
      consumers_sync();
      cur = ai;
      ++ns;
    }
    const int nrows = un.nrows;
    const bool on = 32 * tp < nrows;             // nrows is a multiple of 32
    const int sb = its % kScaleBufs;
    bool ok = tc::mbar_wait(tc::smem_u32(&sfull_bar[sb]), (its / kScaleBufs) & 1, abort, status);
    const uint8_t* sc = smem + L.scales + sb * L.scale_bytes + (32 * tp + g) * L.nb;
    float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    // the block pair this warp takes in every box turns with the unit, so that the
    // ragged last box of a row does not always fall to the same warps
    const int qe = (q + un.ord) & (kClasses - 1);
    for (int s = 0; s < nst; ++s) {
      ok = ok && tc::mbar_wait(tc::smem_u32(&full_bar[st]), ph, abort, status);
      if (ok && on) {
        const uint32_t rbase = tc::smem_u32(smem + st * kStageBytes) + (32 * tp + 8 * (mi & 1) + ri) * 128;
        const int nblk = min(kBlocksPerStage, L.nb - s * kBlocksPerStage);
#pragma unroll
        for (int j = 0; j < kBoxes; ++j) {
          const int nbj = min(kBlocksPerBox, nblk - j * kBlocksPerBox);
          const int gb0 = s * kBlocksPerStage + j * kBlocksPerBox + 2 * qe;
          if (nbj == kBlocksPerBox)
            box_pair<true, PAIRED>(rbase + j * kBoxBytes, mi, ri, qe, tg, sc, L.nb, lut, gb0, kBlocksPerBox, acc2);
          else if (nbj > 0)
            box_pair<false, PAIRED>(rbase + j * kBoxBytes, mi, ri, qe, tg, sc, L.nb, lut, gb0, nbj, acc2);
        }
      }
      // Each lane arrives once its own reads of the stage are done (its ldmatrix
      // results have been consumed), so the stage needs no warp barrier first.
      tc::mbar_arrive(tc::smem_u32(&empty_bar[st]));
      if (++st == a.stages) {
        st = 0;
        ph ^= 1;
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sempty_bar[sb]));
    ++its;
    // hand the unit's partial sums to the epilogue warp, once it has read the last ones
    ok = tc::mbar_wait(tc::smem_u32(&part_empty), (nu & 1) ^ 1, abort, status) && ok;
    if (ok && on) {
#pragma unroll
      for (int t2 = 0; t2 < 2; ++t2)
        part[(q * 2 + t2) * 32] = make_float4(acc2[t2][0], acc2[t2][1], acc2[t2][2], acc2[t2][3]);
    }
    tc::mbar_arrive(tc::smem_u32(&part_full));
    ++nu;
  }
  pdl_trigger();
}

template <bool GATEUP, bool PAIRED>
void set_fp4_smem(int bytes) {
  static int done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || done[dev] >= bytes) return;
  if (cudaFuncSetAttribute(fp4_stream_kernel<GATEUP, PAIRED>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
      cudaSuccess)
    done[dev] = bytes;
}

// Ring depth that fits next to the fixed parts for `kin` inputs (0: it does not fit).
int fp4_stream_stages(int kin) {
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const int fixed = f4_smem(kin, 0).total + 1024 + 1024;   // + base alignment + static smem
  int st = (optin - fixed) / kStageBytes;
  if (st > kMaxRingStages) st = kMaxRingStages;
  return st >= 2 ? st : 0;
}

template <bool GATEUP>
cudaError_t launch_fp4_stream(const uint8_t* codes, const F4Args& a0, int n_experts, int max_items,
                              cudaStream_t s, bool* launched) {
  *launched = false;
  F4Args a = a0;
  a.stages = fp4_stream_stages(a.kin);
  if (!a.stages) return cudaSuccess;
  if ((reinterpret_cast<uintptr_t>(a.scales) & 15) || (reinterpret_cast<uintptr_t>(codes) & 15))
    return cudaSuccess;
  CUtensorMap m, m64;   // boxes of 128 rows (full units) and 64 rows (half units) x 128 bytes
  if (!make_map(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, (uint64_t)n_experts * a.R, (uint64_t)a.kin / 2,
                (uint64_t)a.kin / 2, kRows, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m64, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, (uint64_t)n_experts * a.R, (uint64_t)a.kin / 2,
                (uint64_t)a.kin / 2, kRows / 2, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaSuccess;
  // gate_up shares are cut in half units (1440 full units of gpt-oss-20b over 152 SMs
  // leave 72 CTAs a whole unit above the rest); down keeps full units, where a CTA's
  // lone halves would cost more than its imbalance
  const int unit_rows = GATEUP ? kRows / 2 : kRows;
  a.tiles = (a.R + unit_rows - 1) / unit_rows;
  const int bytes = f4_smem(a.kin, a.stages).total + 1024;
  const long long halves = (long long)max_items * a.tiles;
  int grid = sm_count();
  if (halves < grid) grid = (int)(halves > 0 ? halves : 1);
  *launched = true;
  if ((a.kin / 32) % 2 == 0) {
    set_fp4_smem<GATEUP, true>(bytes);
    return launch_pdl(fp4_stream_kernel<GATEUP, true>, dim3(grid), dim3(kThreads), (size_t)bytes, s, m, m64, a);
  }
  set_fp4_smem<GATEUP, false>(bytes);
  return launch_pdl(fp4_stream_kernel<GATEUP, false>, dim3(grid), dim3(kThreads), (size_t)bytes, s, m, m64, a);
}

}  // namespace

cudaError_t fp4_stream_set_wait_test(uint32_t polls, int withhold) { return tc::set_wait_test(polls, withhold); }

cudaError_t launch_gateup_decode_fp4(const ExpertParams& p, const RouteState& rs, const uint16_t* x, int K,
                                     uint16_t* h, int ldh, int max_items, cudaStream_t s, bool* launched) {
  F4Args a{};
  a.rs = rs;
  a.R = 2 * p.ff;
  a.kin = p.d;
  a.scales = p.gu_scales;
  a.bias = p.gu_bias;
  a.x = x;
  a.K = K;
  a.h = h;
  a.ldh = ldh;
  a.act = p.act;
  a.limit = p.limit;
  a.alpha = p.alpha;
  return launch_fp4_stream<true>(p.gate_up, a, p.E, max_items, s, launched);
}

cudaError_t launch_down_decode_fp4(const ExpertParams& p, const RouteState& rs, const uint16_t* h, int ldh,
                                   float* Y, int max_items, cudaStream_t s, bool* launched) {
  F4Args a{};
  a.rs = rs;
  a.R = p.d;
  a.kin = p.ff;
  a.scales = p.dn_scales;
  a.bias = p.dn_bias;
  a.h = const_cast<uint16_t*>(h);
  a.ldh = ldh;
  a.Y = Y;
  return launch_fp4_stream<false>(p.down, a, p.E, max_items, s, launched);
}

}  // namespace moe
