// Prefill path: grouped GEMMs on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators) fed by TMA through an mbarrier pipeline.
//
// Per expert e with rows (tokens, in the grouped order of the permute kernel):
//   gate_up:  h[r, f] = act(X_r . G_e[f], X_r . U_e[f])       A = X rows, B = weights
//   down   :  Y[slot(r), o] = h_r . D_e[o] (+ b_e[o])
// Both are D[128 x N] = A[128 x K] . B[N x K]^T with both operands K-major, the
// natural layouts of activations and of row = output weights.
//
// One persistent CTA per SM walks the tiles (m tile of 128 rows of one expert,
// n tile of N output columns), m-tile-major so that concurrently running CTAs
// share A tiles and weight tiles through L2.  Warp roles:
//   warp 0      TMA producer: A and B tiles of 64 k (128-byte rows, 128-byte
//               swizzle) into a 4-stage shared-memory ring;
//   warp 1      owns TMEM (two accumulators of up to 256 fp32 columns) and issues
//               tcgen05.mma (M 128, N <= 256, K 16) from one thread, committing
//               each stage back to the producer and each finished tile to the
//               epilogue;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator row that their TMEM lane
//               quarter holds, bias + activation (gate_up) or bias (down), stores
//               (down and the router logits: turned around in shared memory so that
//               every store writes whole lines);
//   warps 6..   MXFP4: dequant warps (B tiles into shared memory); bf16 gate_up:
//               loader warps that copy the A rows from x by row index (cp.async)
//               instead of a TMA load of a gathered copy.
// The router logits run through the same kernel (dense mode), with the k range cut
// into parts when there are few m tiles.
// Every mbarrier wait is bounded; a wait that gives up sets the device status
// and an abort flag, the CTA drains its copies and MMAs in flight, frees TMEM and
// returns.
//
// Sources: "qwen35moe - Forward-Pass Design", sections "Shared-expert MoE FFN" and
// "Batched prefill" (expert-grouped batching: tokens that share an expert stream
// its weights once); "Phase 19: MoE - gpt-oss-20b", section 2 Experts.
#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;                         // rows per tile (MMA M)
constexpr int kBK = 64;                          // k per stage: 128 bytes of bf16
constexpr int kTileA = kBM * kBK * 2;            // 16 KiB
constexpr uint32_t kTmemCols = 512;              // two accumulators of 256 columns

// Shared-memory stage of each variant: A tile(s) | B (bf16) | MXFP4 only: packed
// codes (N x 32 bytes per 64 k) | scales (2 x N bytes: the two 32-input blocks of
// the chunk).  DUAL (the down projection): two A tiles, h_hi and h_lo, multiply the
// same B tile.  Stages are multiples of 1024 bytes so every swizzled tile starts
// 1024-aligned.  MXFP4 variants add 12 dequant warps (warps 6..17).
template <bool FP4, bool DUAL>
struct Lay {
  static constexpr int kMaxN = FP4 ? 240 : 256;
  static constexpr int kATiles = DUAL ? 2 : 1;
  static constexpr int kTileB = kMaxN * kBK * 2;
  static constexpr int kPacked = FP4 ? kMaxN * (kBK / 2) : 0;
  static constexpr int kScales = FP4 ? 512 : 0;
  static constexpr int kStageBytes =
      ((kATiles * kTileA + kTileB + kPacked + kScales + 1023) / 1024) * 1024;
  static constexpr int kStages = DUAL ? 3 : 4;
  // bf16 down and dense logits: each epilogue warp turns its 32 rows x 32 fp32
  // columns around in shared memory ([32][kEpiPitch] floats) so that its stores are
  // whole lines
  static constexpr bool kEpiStage = !FP4;
  static constexpr int kEpiPitch = 36;
  static constexpr int kEpiBytes = kEpiStage ? 4 * 32 * kEpiPitch * 4 : 0;
  static constexpr int kSmemBytes = kStages * kStageBytes + kEpiBytes + 1024;   // + alignment slack
  static constexpr int kDequantWarps = FP4 ? 12 : 0;
  // bf16 gate_up: 8 warps copy the A rows straight from x by row index (cp.async)
  static constexpr int kLoadWarps = (!FP4 && !DUAL) ? 8 : 0;
  static constexpr int kThreads = 192 + 32 * (kDequantWarps + kLoadWarps);
};
constexpr int kMaxStages = 4;

enum : int { kModeGateUpSplit = 0, kModeGateUpInterleaved = 1, kModeDown = 2, kModeDense = 3 };

struct GemmArgs {
  RouteState rs;          // offsets, work = m tiles (expert, first row), n_work, row2slot
  int E;                  // routed experts; v == E is the shared expert
  int mode;               // kMode*
  int N;                  // MMA N (B rows per tile)
  int nt_routed, nt_shared, nt_max;   // n tiles per routed / shared expert
  int k_routed, k_shared;             // reduction length (elements)
  int b_rows_routed;      // rows of one routed expert in the B tensor (gate/up: ff or 2ff; down: d)
  int nf;                 // gate_up: features per n tile (N / 2)
  int act;
  float limit, alpha;
  const uint16_t* gu_bias;    // [E, 2ff] gate_up row order, or null
  const uint16_t* dn_bias;    // [E, d] or null
  int d, ff;
  uint16_t* h;            // gate_up output [S, 2*ldh]: bf16 (hi, lo) halves, grouped row order
  int a_gather;           // gate_up (bf16): A rows copied from ax by row index, not by TMA
  const uint16_t* ax;     // x [T, d] bf16; grouped row r is token row2slot[r] / aK
  int aK;                 // slots per token
  int ldh;                // width of each half
  int dual;               // down: A = h_hi and h_lo tiles against the same B tile
  float* Y;               // down output [S, d] (slot order)
  float* yacc;            // down, when non-null: yacc[token, :] += slot_w[slot] * (row + bias) by
                          // atomic adds (token = slot / aK), in place of the Y row
  float* yzero;           // gate_up, when non-null: cleared by the epilogue warps before their
  size_t yzero_n4;        // first tile (yzero_n4 float4s): the sums the down projection adds into
  int scale_rows;         // MXFP4: rows of one expert in the transposed scales
  int scale_nblk;         // MXFP4: 32-input blocks per weight row
  // kModeDense (router logits): A = x [rows, d], B = W_r [E, d]; no routing state
  int dense_rows;         // T
  int nsplit;             // dense: the k range is cut into nsplit parts (split-K)
  int dense_vec;          // dense: logits, ldl allow 16-byte stores (the staged epilogue)
  size_t split_stride;    // dense: floats between the partial logits of two parts
  float* logits;          // [T, ldl] fp32 (part s at logits + s * split_stride)
  int ldl;
  const uint16_t* rbias;  // bf16 [E] or null
};

struct Tile {
  int v, row0, n, cnt, kk;    // expert, first row within it, n tile, rows in this tile, k
  int nkc;                    // k chunks of 64
  int kbeg, split;            // first k of the tile's range and its part (dense split-K)
  bool skip;
};

// Tiles run m-tile-major: the CTAs working at the same time take the n tiles of a
// few consecutive m tiles, so each A tile and each expert's weight tiles are read
// from HBM about once and then served to the other CTAs from L2.
__device__ __forceinline__ Tile tile_at(const GemmArgs& g, int t, int n_m) {
  Tile tl;
  const int m = t / g.nt_max;
  tl.n = t - m * g.nt_max;
  tl.kbeg = 0;
  tl.split = 0;
  if (g.mode == kModeDense) {
    // nt_max counts (k part, n tile) pairs
    const int nt = g.nt_max / g.nsplit;
    tl.split = tl.n / nt;
    tl.n -= tl.split * nt;
    const int ks = g.k_routed / kBK;
    const int kb0 = ks * tl.split / g.nsplit, kb1 = ks * (tl.split + 1) / g.nsplit;
    tl.v = 0;
    tl.row0 = m * kBM;
    tl.cnt = min(kBM, g.dense_rows - tl.row0);
    tl.kbeg = kb0 * kBK;
    tl.nkc = kb1 - kb0;
    tl.kk = tl.nkc * kBK;
    tl.skip = false;
    return tl;
  }
  const int2 w = g.rs.work[m];
  tl.v = w.x;
  tl.row0 = w.y;
  const bool sh = (tl.v == g.E);
  const int rows = g.rs.offsets[tl.v + 1] - g.rs.offsets[tl.v];
  tl.cnt = min(kBM, rows - tl.row0);
  tl.kk = sh ? g.k_shared : g.k_routed;
  tl.nkc = tl.kk / kBK;
  tl.skip = tl.n >= (sh ? g.nt_shared : g.nt_routed);
  return tl;
}

__device__ __forceinline__ float act_swiglu(float gt, float up) { return gt / (1.f + __expf(-gt)) * up; }

__device__ __forceinline__ float act_clamped(float gt, float up, float limit, float alpha) {
  gt = fminf(gt, limit);
  up = fminf(fmaxf(up, -limit), limit);
  return (up + 1.f) * gt / (1.f + __expf(-alpha * gt));
}

// MXFP4 dequant of one stage: N rows x 64 inputs from packed codes (smem, [N][32])
// and scales (smem, [2][N]) into the bf16 B tile with the 128-byte swizzle.
// Work unit = one 16-byte output chunk (8 inputs, 4 code bytes, one scale).
// Thread `tid` always takes chunk column j = tid % 8 of rows tid / 8 + step * i
// (step = nthreads / 8, a multiple of 8), so its swizzle XOR (j ^ row % 8), its
// scale row and all its addresses advance by constants.
__device__ __forceinline__ uint4 dq_chunk(uint32_t w, const Fp4Scale& sc, bool two) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
  uint4 o;
  if (!two) {
    const Fp4Scale one{sc.first, 0u, false};
    o.x = fp4_pair<0>(lo, hi, one);
    o.y = fp4_pair<1>(lo, hi, one);
    o.z = fp4_pair<2>(lo, hi, one);
    o.w = fp4_pair<3>(lo, hi, one);
  } else {
    o.x = fp4_pair<0>(lo, hi, sc);
    o.y = fp4_pair<1>(lo, hi, sc);
    o.z = fp4_pair<2>(lo, hi, sc);
    o.w = fp4_pair<3>(lo, hi, sc);
  }
  return o;
}

__device__ __forceinline__ void dequant_stage(const uint8_t* packed, const uint8_t* scales, uint8_t* btile,
                                              int N, int tid, int nthreads) {
  const int j = tid & 7, r0 = tid >> 3, step = nthreads >> 3;
  const uint8_t* pk = packed + r0 * 32 + j * 4;
  const uint8_t* sp = scales + (j >> 2) * N + r0;
  uint8_t* bt = btile + r0 * 128 + ((j ^ (r0 & 7)) << 4);
#pragma unroll 5
  for (int r = r0; r < N; r += step) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(pk);
    const uint32_t sv = *sp;
    const Fp4Scale sc = fp4_scale(sv);
    const bool two = __any_sync(0xffffffffu, sv > 128u);   // warp-uniform: 2nd multiply needed
    *reinterpret_cast<uint4*>(bt) = dq_chunk(w, sc, two);
    pk += step * 32;
    sp += step;
    bt += step * 128;
  }
}

// The staged epilogue: row index (or -1) of each of the 8 rows 4i + lane / 8 that
// this lane stores, from `r`, the row index lane l holds for row l of its warp.
__device__ __forceinline__ void turned_rows(int r, int lane, int (&ridx)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) ridx[i] = __shfl_sync(0xffffffffu, r, 4 * i + (lane >> 3));
}

// The same for a per-row value (the routing weight of the row's slot).
__device__ __forceinline__ void turned_vals(float r, int lane, float (&rv)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) rv[i] = __shfl_sync(0xffffffffu, r, 4 * i + (lane >> 3));
}

// One 32 x 32 fp32 block of a warp's rows (lane l holds row l's 32 values in v) to
// rows ridx[i] (negative: skipped) of `base`, `pitch` floats apart, columns col ..
// col + min(32, ncol) - 1, plus a bf16 bias per column when `bias` is non-null.
// The block turns around in stg ([32][PITCH] floats, conflict-free both ways) so
// that lanes 8j..8j+7 store 128 contiguous bytes of one row: each store instruction
// writes four whole lines instead of 32 partial ones.  base, pitch and col keep
// every 16-byte store aligned (pitch and col multiples of 4).
template <int PITCH>
__device__ __forceinline__ void store_turned(float* stg, const float (&v)[32], const int (&ridx)[8], float* base,
                                             size_t pitch, int col, int ncol, const uint16_t* bias, int lane) {
  float4* wr = reinterpret_cast<float4*>(stg + lane * PITCH);
#pragma unroll
  for (int i = 0; i < 8; ++i) wr[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  __syncwarp();
  const int rr = lane >> 3, cc = (lane & 7) * 4;
  if (cc < ncol) {
    float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (bias) b4 = make_float4(bf16_to_f32(bias[cc]), bf16_to_f32(bias[cc + 1]), bf16_to_f32(bias[cc + 2]),
                               bf16_to_f32(bias[cc + 3]));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (ridx[i] >= 0) {
        float4 val = *reinterpret_cast<const float4*>(stg + (4 * i + rr) * PITCH + cc);
        if (bias) {
          val.x += b4.x;
          val.y += b4.y;
          val.z += b4.z;
          val.w += b4.w;
        }
        *reinterpret_cast<float4*>(base + (size_t)ridx[i] * pitch + col + cc) = val;
      }
    }
  }
  __syncwarp();
}

// store_turned for the accumulated down projection: row i of the block (plus the
// bias) times rw[i] is added to row ridx[i] of `base` with vector atomic adds, so
// that lanes 8j..8j+7 reduce 128 contiguous bytes of one row.
template <int PITCH>
__device__ __forceinline__ void red_turned(float* stg, const float (&v)[32], const int (&ridx)[8],
                                           const float (&rw)[8], float* base, size_t pitch, int col, int ncol,
                                           const uint16_t* bias, int lane) {
  float4* wr = reinterpret_cast<float4*>(stg + lane * PITCH);
#pragma unroll
  for (int i = 0; i < 8; ++i) wr[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  __syncwarp();
  const int rr = lane >> 3, cc = (lane & 7) * 4;
  if (cc < ncol) {
    float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (bias) b4 = make_float4(bf16_to_f32(bias[cc]), bf16_to_f32(bias[cc + 1]), bf16_to_f32(bias[cc + 2]),
                               bf16_to_f32(bias[cc + 3]));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (ridx[i] >= 0) {
        const float4 val = *reinterpret_cast<const float4*>(stg + (4 * i + rr) * PITCH + cc);
        red_add_v4(base + (size_t)ridx[i] * pitch + col + cc, rw[i] * (val.x + b4.x), rw[i] * (val.y + b4.y),
                   rw[i] * (val.z + b4.z), rw[i] * (val.w + b4.w));
      }
    }
  }
  __syncwarp();
}

// FP4: B comes from MXFP4 weights (tmB0: packed codes [rows, nblk*16] bytes, tmB1:
// transposed scales [E*nblk, rows] bytes); else tmB0/tmB1 (and tmS0/tmS1 for the
// shared expert) are bf16 weight maps.
template <bool FP4, bool DUAL>
__global__ void __launch_bounds__(Lay<FP4, DUAL>::kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmS0,
                    const __grid_constant__ CUtensorMap tmS1, const GemmArgs g) {
  using L = Lay<FP4, DUAL>;
  constexpr int kStages = L::kStages;
  constexpr int kStageBytes = L::kStageBytes;
  constexpr int kTileB = L::kTileB;
  constexpr int kAB = L::kATiles * kTileA;     // offset of B in a stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = tc::smem_align1024(smem_raw);
  __shared__ __align__(8) uint64_t full_bar[kMaxStages], empty_bar[kMaxStages],
      bready_bar[kMaxStages], tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int consumed_s;     // stage loads the MMA thread has waited for

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = g.rs.status;
  volatile int* abort = &abort_s;
  pdl_wait();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(tc::smem_u32(&full_bar[s]), 1 + (g.a_gather ? 128 : 0));   // TMA + one loader half
      tc::mbar_init(tc::smem_u32(&empty_bar[s]), 1);
      tc::mbar_init(tc::smem_u32(&bready_bar[s]), L::kDequantWarps ? L::kDequantWarps : 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(tc::smem_u32(&tfull_bar[b]), 1);
      tc::mbar_init(tc::smem_u32(&tempty_bar[b]), 4);
    }
    tc::mbar_init(tc::smem_u32(&drain_bar), 1);
    abort_s = 0;
    consumed_s = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tmA);
    tc::tma_prefetch_desc(&tmB0);
    tc::tma_prefetch_desc(&tmS0);
    if (FP4 || g.mode == kModeGateUpSplit) {
      tc::tma_prefetch_desc(&tmB1);
      tc::tma_prefetch_desc(&tmS1);
    }
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&tmem_base_s), kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  // dense mode is the first kernel of a call: start a clean device status (after the
  // wait above, so that no flag of the previous call can land later)
  if (g.mode == kModeDense && status && blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;
  const int n_m = g.mode == kModeDense ? (g.dense_rows + kBM - 1) / kBM : *g.rs.n_work;
  const int total = n_m > 0 ? n_m * g.nt_max : 0;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (tc::elect_one()) {
      int s = 0, issued = 0, withheld = -1;
      uint32_t ph = 0;
      for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
        const Tile tl = tile_at(g, t, n_m);
        if (tl.skip) continue;
        const bool sh = (tl.v == g.E);
        const int a_row = (g.mode == kModeDense ? 0 : g.rs.offsets[tl.v]) + tl.row0;
        const int nb = (g.mode == kModeGateUpSplit) ? g.nf : g.N;
        const int b_row = (sh ? 0 : tl.v * g.b_rows_routed) + tl.n * nb;
        const CUtensorMap* m0 = sh ? &tmS0 : &tmB0;
        const CUtensorMap* m1 = sh ? &tmS1 : &tmB1;
        for (int kc = 0; kc < tl.nkc; ++kc) {
          if (!tc::mbar_wait(tc::smem_u32(&empty_bar[s]), ph ^ 1, abort, status)) break;
          // A slot freed by an abort is not refilled: its last load may still be landing.
          if (*abort) break;
          if (tc::withheld_load(issued, blockIdx.x == 0)) {   // CTA 0 takes tile 0
            // the give-up test: this load is never issued, so its stage never fills
            withheld = issued++;
            if (++s == kStages) {
              s = 0;
              ph ^= 1;
            }
            continue;
          }
          const uint32_t fb = tc::smem_u32(&full_bar[s]);
          const uint32_t sa = tc::smem_u32(smem + s * kStageBytes);
          const uint32_t sb = sa + kAB;
          const int k0 = tl.kbeg + kc * kBK;
          uint32_t bytes = g.a_gather ? 0u : (uint32_t)kAB;
          if (FP4) bytes += (uint32_t)g.N * 34u;          // codes (32 B) + 2 scales per row
          else bytes += (uint32_t)g.N * kBK * 2;
          tc::mbar_arrive_expect_tx(fb, bytes);
          if (!g.a_gather) tc::tma_load_2d(sa, &tmA, k0, a_row, fb);
          if (DUAL) tc::tma_load_2d(sa + kTileA, &tmA, g.ldh + k0, a_row, fb);
          if (FP4) {
            const uint32_t sp = sb + (uint32_t)kTileB, ss = sp + (uint32_t)L::kPacked;
            tc::tma_load_2d(sp, &tmB0, kc * 32, b_row, fb);
            tc::tma_load_2d(ss, &tmB1, tl.n * g.N, tl.v * g.scale_nblk + 2 * kc, fb);
          } else if (g.mode == kModeGateUpSplit) {
            tc::tma_load_2d(sb, m0, k0, b_row, fb);
            tc::tma_load_2d(sb + (uint32_t)g.nf * 128u, m1, k0, b_row, fb);
          } else {
            tc::tma_load_2d(sb, m0, k0, b_row, fb);
          }
          ++issued;
          if (++s == kStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (*abort) {
        // Drain: wait (bounded, regardless of the abort flag) for the loads still in flight.
        int zero = 0;
        volatile int* never = &zero;
        for (int i = consumed_s; i < issued; ++i)
          if (i != withheld)
            tc::mbar_wait(tc::smem_u32(&full_bar[i % kStages]), (i / kStages) & 1, never, status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (tc::elect_one()) {
      int s = 0, b = 0;
      uint32_t ph = 0, aph = 0;
      const uint32_t idesc = tc::idesc_bf16_f32(kBM, g.N);
      bool any = false;
      for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
        const Tile tl = tile_at(g, t, n_m);
        if (tl.skip) continue;
        if (!tc::mbar_wait(tc::smem_u32(&tempty_bar[b]), aph ^ 1, abort, status)) break;
        tc::tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)b * 256u;
        bool ok = true;
        for (int kc = 0; kc < tl.nkc; ++kc) {
          if (!tc::mbar_wait(tc::smem_u32(&full_bar[s]), ph, abort, status) ||
              (FP4 && !tc::mbar_wait(tc::smem_u32(&bready_bar[s]), ph, abort, status))) {
            ok = false;
            break;
          }
          consumed_s = consumed_s + 1;
          tc::tc_fence_after();
          const uint32_t sa = tc::smem_u32(smem + s * kStageBytes);
          const uint64_t ad = tc::sdesc_sw128(sa), bd = tc::sdesc_sw128(sa + kAB);
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j) {
            tc::umma_bf16(dt, ad + 2 * j, bd + 2 * j, idesc, (kc | j) != 0);
            if (DUAL) tc::umma_bf16(dt, ad + (kTileA >> 4) + 2 * j, bd + 2 * j, idesc, 1);
          }
          tc::umma_commit(tc::smem_u32(&empty_bar[s]));
          any = true;
          if (++s == kStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc::umma_commit(tc::smem_u32(&tfull_bar[b]));
        if (++b == 2) {
          b = 0;
          aph ^= 1;
        }
      }
      if (*abort && any) {
        // Let every MMA issued so far finish before TMEM is released.
        tc::umma_commit(tc::smem_u32(&drain_bar));
        int zero = 0;
        volatile int* never = &zero;
        tc::mbar_wait(tc::smem_u32(&drain_bar), 0, never, status);
      }
    }
  } else if (L::kLoadWarps && warp >= 6) {
    // ---------------------------------------------------------------- A rows by index
    // Two halves of 128 threads take alternate k steps (half h the steps of parity h,
    // counted over all of the CTA's tiles).  Thread lt of a half copies 16-byte chunk
    // c = lt % 8 of rows lt / 8 + 16 j (j < 8) of the step's A tile: tile row r is x's
    // row of the token of grouped row offsets[v] + row0 + r, stored where the 128-byte
    // swizzle puts it (rows past the tile's count are zero-filled).  A step's copies
    // are waited for when the half has issued its next step (so each half keeps two
    // steps in flight, four in all; waiting further back would tie a step's
    // announcement to the MMAs freeing the slot of a later step), then made visible to
    // the tensor core's proxy and announced on the stage's full barrier (with the TMA's
    // bytes of the weight tile).
    if (g.a_gather) {
      const int lt = (threadIdx.x - 192) & 127, half = (threadIdx.x - 192) >> 7;
      const int c = lt & 7, rq = lt >> 3;
      int step = 0, pending = -1;              // global k step; the half's unannounced step
      for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
        const Tile tl = tile_at(g, t, n_m);
        if (tl.skip) continue;
        const int base = g.rs.offsets[tl.v] + tl.row0;
        const uint16_t* src[8];
        uint32_t nb[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = rq + 16 * j;
          const bool in = r < tl.cnt;
          const int tok = in ? g.rs.row2slot[base + r] / g.aK : 0;
          src[j] = g.ax + (size_t)tok * g.d + 8 * c;
          nb[j] = in ? 16u : 0u;
        }
        bool ok = true;
        for (int kc = 0; kc < tl.nkc; ++kc, ++step) {
          if ((step & 1) != half) continue;
          const int s = step % kStages;
          if (!tc::mbar_wait(tc::smem_u32(&empty_bar[s]), ((step / kStages) & 1) ^ 1, abort, status)) {
            ok = false;
            break;
          }
          const uint32_t sa = tc::smem_u32(smem + s * kStageBytes);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = rq + 16 * j;
            tc::cp_async16(sa + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)), src[j] + kc * kBK, nb[j]);
          }
          tc::cp_async_commit();
          if (pending >= 0) {
            tc::cp_async_wait<1>();             // the half's previous step has landed
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(tc::smem_u32(&full_bar[pending % kStages]));
          }
          pending = step;
        }
        if (!ok) break;
      }
      tc::cp_async_wait_all();
      tc::fence_proxy_async_smem();
      if (pending >= 0) tc::mbar_arrive(tc::smem_u32(&full_bar[pending % kStages]));
    }
  } else if (FP4 && warp >= 6) {
    // ---------------------------------------------------------------- MXFP4 dequant
    const int dt = threadIdx.x - 192;
    constexpr int kDq = 32 * L::kDequantWarps;
    int s = 0;
    uint32_t ph = 0;
    for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
      const Tile tl = tile_at(g, t, n_m);
      if (tl.skip) continue;
      bool ok = true;
      for (int kc = 0; kc < tl.nkc; ++kc) {
        if (!tc::mbar_wait(tc::smem_u32(&full_bar[s]), ph, abort, status)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * kStageBytes;
        dequant_stage(st + kAB + kTileB, st + kAB + kTileB + L::kPacked, st + kAB, g.N, dt, kDq);
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&bready_bar[s]));
        if (++s == kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quarter this warp may read
    const int row = 32 * q + lane;
    int b = 0;
    uint32_t aph = 0;
    if (g.yzero) {
      // this CTA's share of the per-token sums of the accumulated down projection,
      // cleared while the first tile's MMAs run
      const size_t per = (g.yzero_n4 + gridDim.x - 1) / gridDim.x;
      const size_t z0 = per * blockIdx.x, z1 = min(g.yzero_n4, z0 + per);
      float4* z = reinterpret_cast<float4*>(g.yzero);
      for (size_t i = z0 + (threadIdx.x - 64); i < z1; i += 128) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
      const Tile tl = tile_at(g, t, n_m);
      if (tl.skip) continue;
      if (!tc::mbar_wait(tc::smem_u32(&tfull_bar[b]), aph, abort, status)) break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)b * 256u;
      const bool valid = row < tl.cnt;
      const int grow = (g.mode == kModeDense ? 0 : g.rs.offsets[tl.v]) + tl.row0 + row;   // grouped row
      const bool sh = (tl.v == g.E);
      if (L::kEpiStage && g.mode == kModeDense && g.dense_vec) {
        // router logits of token grow, experts n*N .. n*N + N - 1 (+ bias, in part 0)
        int ridx[8];
        turned_rows(valid ? grow : -1, lane, ridx);
        const int e0 = tl.n * g.N;
        const uint16_t* rbias = tl.split == 0 && g.rbias ? g.rbias + e0 : nullptr;
        float* base = g.logits + tl.split * g.split_stride;
        float* stg = reinterpret_cast<float*>(smem + kStages * kStageBytes) + q * 32 * L::kEpiPitch;
        for (int c0 = 0; c0 < g.N; c0 += 32) {
          float v[32];
          tc::tmem_ld32(taddr + (uint32_t)c0, v);
          store_turned<L::kEpiPitch>(stg, v, ridx, base, (size_t)g.ldl, e0 + c0, g.N - c0,
                                     rbias ? rbias + c0 : nullptr, lane);
        }
      } else if (g.mode == kModeDense) {
        // router logits of token grow, experts n*N .. n*N + N - 1 (+ bias, in part 0)
        float* lrow = valid ? g.logits + tl.split * g.split_stride + (size_t)grow * g.ldl : nullptr;
        const uint16_t* rbias = tl.split == 0 ? g.rbias : nullptr;
        const int e0 = tl.n * g.N;
        for (int c0 = 0; c0 < g.N; c0 += 32) {
          float v[32];
          tc::tmem_ld32(taddr + (uint32_t)c0, v);
          if (valid) {
            const int ncol = min(32, g.N - c0);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < ncol) lrow[e0 + c0 + i] = v[i] + (rbias ? bf16_to_f32(rbias[e0 + c0 + i]) : 0.f);
          }
        }
      } else if (L::kEpiStage && g.mode == kModeDown && g.yacc) {
        // y[token] += w(slot) * (row + bias): the weighted expert output goes straight
        // into the token's fp32 sum
        const int slot = valid ? g.rs.row2slot[grow] : -1;
        int tidx[8];
        float tw[8];
        turned_rows(slot >= 0 ? slot / g.aK : -1, lane, tidx);
        turned_vals(slot >= 0 ? g.rs.slot_w[slot] : 0.f, lane, tw);
        const int o0 = tl.n * g.N;
        const uint16_t* bp = (!sh && g.dn_bias) ? g.dn_bias + (size_t)tl.v * g.d + o0 : nullptr;
        float* stg = reinterpret_cast<float*>(smem + kStages * kStageBytes) + q * 32 * L::kEpiPitch;
        for (int c0 = 0; c0 < g.N; c0 += 32) {
          float v[32];
          tc::tmem_ld32(taddr + (uint32_t)c0, v);
          red_turned<L::kEpiPitch>(stg, v, tidx, tw, g.yacc, (size_t)g.d, o0 + c0, g.N - c0,
                                   bp ? bp + c0 : nullptr, lane);
        }
      } else if (L::kEpiStage && g.mode == kModeDown) {
        const int slot = valid ? g.rs.row2slot[grow] : -1;
        int ridx[8];
        turned_rows(slot, lane, ridx);
        const int o0 = tl.n * g.N;
        const uint16_t* bp = (!sh && g.dn_bias) ? g.dn_bias + (size_t)tl.v * g.d + o0 : nullptr;
        float* stg = reinterpret_cast<float*>(smem + kStages * kStageBytes) + q * 32 * L::kEpiPitch;
        for (int c0 = 0; c0 < g.N; c0 += 32) {
          float v[32];
          tc::tmem_ld32(taddr + (uint32_t)c0, v);
          store_turned<L::kEpiPitch>(stg, v, ridx, g.Y, (size_t)g.d, o0 + c0, g.N - c0, bp ? bp + c0 : nullptr,
                                     lane);
        }
      } else if (g.mode == kModeDown && g.yacc) {
        const int slot = valid ? g.rs.row2slot[grow] : -1;
        float* yrow = slot >= 0 ? g.yacc + (size_t)(slot / g.aK) * g.d : nullptr;
        const float wt = slot >= 0 ? g.rs.slot_w[slot] : 0.f;
        const int o0 = tl.n * g.N;
        for (int c0 = 0; c0 < g.N; c0 += 32) {
          float v[32];
          tc::tmem_ld32(taddr + (uint32_t)c0, v);
          if (yrow) {
            const int ncol = min(32, g.N - c0);
            if (!sh && g.dn_bias) {
              const uint16_t* bp = g.dn_bias + (size_t)tl.v * g.d + o0 + c0;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < ncol) v[i] += bf16_to_f32(bp[i]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (4 * i < ncol)
                red_add_v4(yrow + o0 + c0 + 4 * i, wt * v[4 * i], wt * v[4 * i + 1], wt * v[4 * i + 2],
                           wt * v[4 * i + 3]);
          }
        }
      } else if (g.mode == kModeDown) {
        float* yrow = valid ? g.Y + (size_t)g.rs.row2slot[grow] * g.d : nullptr;
        const int o0 = tl.n * g.N;
        for (int c0 = 0; c0 < g.N; c0 += 32) {
          float v[32];
          tc::tmem_ld32(taddr + (uint32_t)c0, v);
          if (valid) {
            const int ncol = min(32, g.N - c0);
            if (!sh && g.dn_bias) {
              const uint16_t* bp = g.dn_bias + (size_t)tl.v * g.d + o0 + c0;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < ncol) v[i] += bf16_to_f32(bp[i]);
            }
            // 32-byte stores: d is a multiple of 32 and o0 + c0 of 16
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (8 * i < ncol) stg_v8(yrow + o0 + c0 + 8 * i, v + 8 * i);
          }
        }
      } else {
        const int f0 = tl.n * g.nf;
        const int act = sh ? MOE_ACT_SWIGLU : g.act;
        uint16_t* hrow = g.h + (size_t)grow * 2 * g.ldh;
        const uint16_t* bias = (!sh && g.gu_bias) ? g.gu_bias + (size_t)tl.v * 2 * g.ff : nullptr;
        if (g.mode == kModeGateUpSplit) {
          // columns [0, nf) gate, [nf, 2nf) up: 32 features per step
          for (int j0 = 0; j0 < g.nf; j0 += 32) {
            float gv[32], uv[32];
            tc::tmem_ld32(taddr + (uint32_t)j0, gv);
            tc::tmem_ld32(taddr + (uint32_t)(g.nf + j0), uv);
            if (valid) {
              uint32_t packed[16], plo[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float h0, h1;
                const int f = f0 + j0 + 2 * i;
                float ga = gv[2 * i], ua = uv[2 * i], gb = gv[2 * i + 1], ub = uv[2 * i + 1];
                if (bias) {
                  ga += bf16_to_f32(bias[2 * f]); ua += bf16_to_f32(bias[2 * f + 1]);
                  gb += bf16_to_f32(bias[2 * f + 2]); ub += bf16_to_f32(bias[2 * f + 3]);
                }
                h0 = act == MOE_ACT_SWIGLU ? act_swiglu(ga, ua) : act_clamped(ga, ua, g.limit, g.alpha);
                h1 = act == MOE_ACT_SWIGLU ? act_swiglu(gb, ub) : act_clamped(gb, ub, g.limit, g.alpha);
                packed[i] = pack_bf16x2(h0, h1);
                plo[i] = pack_bf16x2(h0 - bf16_lo(packed[i]), h1 - bf16_hi(packed[i]));
              }
              uint4* dst = reinterpret_cast<uint4*>(hrow + f0 + j0);
              uint4* dlo = reinterpret_cast<uint4*>(hrow + g.ldh + f0 + j0);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                dlo[i] = make_uint4(plo[4 * i], plo[4 * i + 1], plo[4 * i + 2], plo[4 * i + 3]);
              }
            }
          }
        } else {
          // interleaved: column 2j gate, 2j+1 up: 16 features per step
          for (int c0 = 0; c0 < g.N; c0 += 32) {
            float v[32];
            tc::tmem_ld32(taddr + (uint32_t)c0, v);
            if (valid) {
              uint32_t packed[8], plo[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int f = f0 + c0 / 2 + 2 * i;
                float ga = v[4 * i], ua = v[4 * i + 1], gb = v[4 * i + 2], ub = v[4 * i + 3];
                if (bias) {
                  ga += bf16_to_f32(bias[2 * f]); ua += bf16_to_f32(bias[2 * f + 1]);
                  gb += bf16_to_f32(bias[2 * f + 2]); ub += bf16_to_f32(bias[2 * f + 3]);
                }
                const float h0 = act == MOE_ACT_SWIGLU ? act_swiglu(ga, ua) : act_clamped(ga, ua, g.limit, g.alpha);
                const float h1 = act == MOE_ACT_SWIGLU ? act_swiglu(gb, ub) : act_clamped(gb, ub, g.limit, g.alpha);
                packed[i] = pack_bf16x2(h0, h1);
                plo[i] = pack_bf16x2(h0 - bf16_lo(packed[i]), h1 - bf16_hi(packed[i]));
              }
              uint4* dst = reinterpret_cast<uint4*>(hrow + f0 + c0 / 2);
              dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
              dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
              uint4* dlo = reinterpret_cast<uint4*>(hrow + g.ldh + f0 + c0 / 2);
              dlo[0] = make_uint4(plo[0], plo[1], plo[2], plo[3]);
              dlo[1] = make_uint4(plo[4], plo[5], plo[6], plo[7]);
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&tempty_bar[b]));
      if (++b == 2) {
        b = 0;
        aph ^= 1;
      }
    }
  }

  pdl_trigger();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// Copy the x row of every grouped row into Xp (the A operand of gate_up).
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ row2slot, int S,
                   int K, int d, uint16_t* __restrict__ xp) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int nvec = d / 8;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < S; r += (gridDim.x * blockDim.x) >> 5) {
    const int t = row2slot[r] / K;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)r * d);
    for (int i = lane; i < nvec; i += 32) dst[i] = ldg_nc_v4(src + i);
  }
  pdl_trigger();
}

// MXFP4 scales [E, rows, nblk] -> [E, nblk, rows], so that the scales of one
// 64-input chunk for a tile's consecutive rows are contiguous (a TMA box).
__global__ void __launch_bounds__(256)
transpose_scales_kernel(const uint8_t* __restrict__ src, int E, int rows, int nblk,
                        uint8_t* __restrict__ dst) {
  pdl_wait();
  pdl_trigger();
  const long long n = (long long)E * rows * nblk;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i % rows;
    const long long vb = i / rows;            // v * nblk + blk
    const long long v = vb / nblk, blk = vb - v * nblk;
    dst[i] = src[(v * rows + r) * nblk + blk];
  }
}

}  // namespace

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace {
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}
}  // namespace

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

// 2D map over a row-major matrix [rows, cols] (row stride in bytes) with a box of
// box_rows x box_cols elements.
bool make_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t rows,
              uint64_t cols, uint64_t stride, uint32_t box_rows, uint32_t box_cols,
              CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !base) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {stride};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, type, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// bf16 matrix, box of box_rows x 64 columns, 128-byte swizzle (operand tiles).
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t stride,
                   uint32_t box_rows) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rows, cols, stride, box_rows, kBK,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

// byte matrix, box of box_rows x box_cols bytes, no swizzle (MXFP4 codes, scales).
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 uint32_t box_cols) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rows, cols, cols, box_rows, box_cols,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}


// Largest N (multiple of 16, at most max_n) that divides `rows`; 0 if none.
int tile_n(int rows, int max_n) {
  for (int n = max_n; n >= 16; n -= 16)
    if (rows % n == 0) return n;
  return 0;
}

// gate_up features per n tile: N = 2 nf <= max_n with nf a multiple of 16 (of 32 for
// separate gate/up, whose epilogue reads 32 gate and 32 up columns at a time),
// dividing ff and, with a shared expert, sff.  0 if none.
int gateup_nf(int ff, int sff, int interleaved, int max_n) {
  const int step = interleaved ? 16 : 32;
  for (int f = (max_n / 2) / step * step; f >= step; f -= step)
    if (ff % f == 0 && (sff == 0 || sff % f == 0)) return f;
  return 0;
}

template <bool FP4, bool DUAL>
void set_smem_attr() {
  static bool done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || done[dev]) return;
  cudaFuncSetAttribute(grouped_gemm_kernel<FP4, DUAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       Lay<FP4, DUAL>::kSmemBytes);
  done[dev] = true;
}

template <bool FP4, bool DUAL>
cudaError_t launch_gemm(const CUtensorMap& tA, const CUtensorMap& tB0, const CUtensorMap& tB1,
                        const CUtensorMap& tS0, const CUtensorMap& tS1, const GemmArgs& g,
                        int max_mtiles, cudaStream_t s) {
  set_smem_attr<FP4, DUAL>();
  const long long tiles = (long long)max_mtiles * g.nt_max;
  int grid = sm_count();
  if (tiles < grid) grid = (int)(tiles > 0 ? tiles : 1);
  return launch_pdl(grouped_gemm_kernel<FP4, DUAL>, dim3(grid), dim3(Lay<FP4, DUAL>::kThreads),
                    Lay<FP4, DUAL>::kSmemBytes, s, tA, tB0, tB1, tS0, tS1, g);
}

}  // namespace

bool prefill_supported(int d, int ff, int sff, int wfmt, int interleaved) {
  const bool fp4 = wfmt == MOE_WFMT_MXFP4;
  const int max_n = fp4 ? Lay<true, false>::kMaxN : Lay<false, false>::kMaxN;
  if (d % kBK || ff % kBK || (sff && sff % kBK)) return false;
  if (fp4 && (!interleaved || sff)) return false;
  if (!gateup_nf(ff, sff, interleaved, max_n)) return false;
  if (!tile_n(d, max_n)) return false;
  if (sff && interleaved) return false;   // the shared expert has separate gate/up maps
  return true;
}

size_t prefill_scales_bytes(const ExpertParams& p, int wfmt) {
  if (wfmt != MOE_WFMT_MXFP4) return 0;
  return (size_t)p.E * 2 * p.ff * (p.d / 32) + (size_t)p.E * p.d * (p.ff / 32);
}

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* row2slot, int S, int K, int d,
                               uint16_t* xp, cudaStream_t s) {
  int blocks = (S + 7) / 8;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  return launch_pdl(gather_rows_kernel, dim3(blocks), dim3(256), 0, s, x, row2slot, S, K, d, xp);
}

cudaError_t launch_transpose_scales(const ExpertParams& p, uint8_t* scratch, cudaStream_t s) {
  const long long n1 = (long long)p.E * 2 * p.ff * (p.d / 32);
  const long long n2 = (long long)p.E * p.d * (p.ff / 32);
  (void)n2;
  cudaError_t e = launch_pdl(transpose_scales_kernel, dim3(152 * 4), dim3(256), 0, s, p.gu_scales, p.E,
                             2 * p.ff, p.d / 32, scratch);
  if (e != cudaSuccess) return e;
  return launch_pdl(transpose_scales_kernel, dim3(152 * 4), dim3(256), 0, s, p.dn_scales, p.E, p.d,
                    p.ff / 32, scratch + n1);
}

cudaError_t launch_gateup_prefill(const ExpertParams& p, int wfmt, int interleaved,
                                  const RouteState& rs, const uint16_t* xp, int S, const uint16_t* x, int T,
                                  int K, uint16_t* h, int ldh, const uint8_t* scalesT, int max_mtiles,
                                  float* yzero, size_t yzero_floats, cudaStream_t s) {
  const bool fp4 = wfmt == MOE_WFMT_MXFP4;
  const int nf = gateup_nf(p.ff, p.sff, interleaved, fp4 ? Lay<true, false>::kMaxN : Lay<false, false>::kMaxN);
  GemmArgs g{};
  g.rs = rs;
  g.yzero = yzero;
  g.yzero_n4 = yzero_floats / 4;
  g.E = p.E;
  g.mode = interleaved ? kModeGateUpInterleaved : kModeGateUpSplit;
  g.N = 2 * nf;
  g.nf = nf;
  g.nt_routed = p.ff / nf;
  g.nt_shared = p.sff ? p.sff / nf : 0;
  g.nt_max = g.nt_routed > g.nt_shared ? g.nt_routed : g.nt_shared;
  g.k_routed = p.d;
  g.k_shared = p.d;
  g.b_rows_routed = interleaved ? 2 * p.ff : p.ff;
  g.act = p.act;
  g.limit = p.limit;
  g.alpha = p.alpha;
  g.gu_bias = p.gu_bias;
  g.d = p.d;
  g.ff = p.ff;
  g.h = h;
  g.ldh = ldh;
  g.scale_rows = 2 * p.ff;
  g.scale_nblk = p.d / 32;
  CUtensorMap tA, tB0, tB1, tS0, tS1;
  std::memset(&tB1, 0, sizeof(tB1));
  const uint64_t rowb = (uint64_t)p.d * 2;
  // bf16 weights: the A rows come straight from x by row index (no gathered copy);
  // MXFP4: from the gathered rows xp by TMA
  g.a_gather = fp4 ? 0 : 1;
  g.ax = x;
  g.aK = K;
  if (fp4 ? !make_map_bf16(&tA, xp, (uint64_t)S, p.d, rowb, kBM)
          : !make_map_bf16(&tA, x, (uint64_t)T, p.d, rowb, kBM))
    return cudaErrorInvalidValue;
  if (fp4) {
    const uint64_t rows = (uint64_t)p.E * 2 * p.ff;
    if (!make_map_u8(&tB0, p.gate_up, rows, (uint64_t)(p.d / 32) * 16, g.N, kBK / 2))
      return cudaErrorInvalidValue;
    if (!make_map_u8(&tB1, scalesT, (uint64_t)p.E * (p.d / 32), 2 * (uint64_t)p.ff, 2, g.N))
      return cudaErrorInvalidValue;
    return launch_gemm<true, false>(tA, tB0, tB1, tB0, tB1, g, max_mtiles, s);
  }
  if (interleaved) {
    if (!make_map_bf16(&tB0, p.gate_up, (uint64_t)p.E * 2 * p.ff, p.d, rowb, g.N)) return cudaErrorInvalidValue;
    tB1 = tB0;
  } else {
    if (!make_map_bf16(&tB0, p.gate, (uint64_t)p.E * p.ff, p.d, rowb, nf)) return cudaErrorInvalidValue;
    if (!make_map_bf16(&tB1, p.up, (uint64_t)p.E * p.ff, p.d, rowb, nf)) return cudaErrorInvalidValue;
  }
  if (p.sff) {
    if (!make_map_bf16(&tS0, p.sh_gate, p.sff, p.d, rowb, nf)) return cudaErrorInvalidValue;
    if (!make_map_bf16(&tS1, p.sh_up, p.sff, p.d, rowb, nf)) return cudaErrorInvalidValue;
  } else {
    tS0 = tB0;
    tS1 = tB1;
  }
  return launch_gemm<false, false>(tA, tB0, tB1, tS0, tS1, g, max_mtiles, s);
}

bool router_gemm_supported(int T, int d, int E) {
  return T >= kBM && d % kBK == 0 && E % 16 == 0 && tile_n(E, Lay<false, false>::kMaxN) != 0;
}

// N of the router GEMM: the largest divisor of E (a multiple of 16, at most 256) that
// still gives every SM a tile, else 16 (the router GEMM is small; keeping all SMs
// busy matters more than the MMA shape).
int router_n(int T, int E) {
  const int m_tiles = (T + kBM - 1) / kBM, sms = sm_count();
  int best = 16;
  for (int n = 16; n <= Lay<false, false>::kMaxN && n <= E; n += 16)
    if (E % n == 0 && (long long)m_tiles * (E / n) >= sms) best = n;
  return best;
}

cudaError_t launch_router_gemm(const uint16_t* x, int T, int d, const uint16_t* w_r, const uint16_t* bias,
                               int E, float* logits, int ldl, float* parts, size_t part_floats, int* nsplit,
                               int* ppitch, uint32_t* status, cudaStream_t s) {
  GemmArgs g{};
  g.rs.status = status;
  g.E = 1;
  g.mode = kModeDense;
  // Where there is room, the logits go to `parts` with a row pitch of E rounded up to
  // 4 (whole-line stores from the staged epilogue).  Few m tiles: then one n tile as
  // wide as possible (x is read once per k part) and the k range cut into parts until
  // every SM has a tile; the select kernel adds the parts in order.  Otherwise the n
  // tiles give the parallelism.
  const int m_tiles = (T + kBM - 1) / kBM, sms = sm_count(), ks = d / kBK;
  const int nwide = tile_n(E, Lay<false, false>::kMaxN);
  const int ldp = (E + 3) / 4 * 4;
  const bool use_parts = parts && (reinterpret_cast<uintptr_t>(parts) & 15) == 0 &&
                         (size_t)T * ldp <= part_floats;
  int ns = 1;
  g.N = router_n(T, E);
  if (use_parts && nwide && (long long)m_tiles * (E / nwide) < sms) {
    int want = min(sms / (m_tiles * (E / nwide)), min(8, ks));
    while (want > 1 && (size_t)want * T * ldp > part_floats) --want;
    if (want > 1) {
      ns = want;
      g.N = nwide;
    }
  }
  *nsplit = ns;
  *ppitch = use_parts ? ldp : 0;
  g.nsplit = ns;
  g.nt_routed = E / g.N;
  g.nt_max = g.nt_routed * ns;
  g.k_routed = d;
  g.dense_rows = T;
  g.logits = use_parts ? parts : logits;
  g.ldl = use_parts ? ldp : ldl;
  g.split_stride = (size_t)T * g.ldl;
  g.dense_vec = use_parts ? 1 : 0;
  g.rbias = bias;
  CUtensorMap tA, tB;
  if (!make_map_bf16(&tA, x, (uint64_t)T, d, (uint64_t)d * 2, kBM)) return cudaErrorInvalidValue;
  if (!make_map_bf16(&tB, w_r, (uint64_t)E, d, (uint64_t)d * 2, g.N)) return cudaErrorInvalidValue;
  return launch_gemm<false, false>(tA, tB, tB, tB, tB, g, (T + kBM - 1) / kBM, s);
}

cudaError_t prefill_set_wait_test(uint32_t polls, int withhold) { return tc::set_wait_test(polls, withhold); }

cudaError_t launch_down_prefill(const ExpertParams& p, int wfmt, const RouteState& rs,
                                const uint16_t* h, int ldh, int S, float* Y, float* yacc, int K,
                                const uint8_t* scalesT, int max_mtiles, cudaStream_t s) {
  const bool fp4 = wfmt == MOE_WFMT_MXFP4;
  GemmArgs g{};
  g.rs = rs;
  g.yacc = yacc;
  g.aK = K;
  g.E = p.E;
  g.mode = kModeDown;
  g.N = tile_n(p.d, fp4 ? Lay<true, false>::kMaxN : Lay<false, false>::kMaxN);
  g.nt_routed = p.d / g.N;
  g.nt_shared = p.sff ? p.d / g.N : 0;
  g.nt_max = g.nt_routed;
  g.k_routed = p.ff;
  g.k_shared = p.sff;
  g.b_rows_routed = p.d;
  g.dn_bias = p.dn_bias;
  g.d = p.d;
  g.Y = Y;
  g.ldh = ldh;
  g.dual = 1;
  g.scale_rows = p.d;
  g.scale_nblk = p.ff / 32;
  CUtensorMap tA, tB0, tB1, tS0;
  if (!make_map_bf16(&tA, h, (uint64_t)S, 2 * (uint64_t)ldh, (uint64_t)ldh * 4, kBM))
    return cudaErrorInvalidValue;
  if (fp4) {
    const uint8_t* sT = scalesT + (size_t)p.E * 2 * p.ff * (p.d / 32);
    if (!make_map_u8(&tB0, p.down, (uint64_t)p.E * p.d, (uint64_t)(p.ff / 32) * 16, g.N, kBK / 2))
      return cudaErrorInvalidValue;
    if (!make_map_u8(&tB1, sT, (uint64_t)p.E * (p.ff / 32), (uint64_t)p.d, 2, g.N))
      return cudaErrorInvalidValue;
    return launch_gemm<true, true>(tA, tB0, tB1, tB0, tB1, g, max_mtiles, s);
  }
  if (!make_map_bf16(&tB0, p.down, (uint64_t)p.E * p.d, p.ff, (uint64_t)p.ff * 2, g.N))
    return cudaErrorInvalidValue;
  if (p.sff) {
    if (!make_map_bf16(&tS0, p.sh_down, p.d, p.sff, (uint64_t)p.sff * 2, g.N)) return cudaErrorInvalidValue;
  } else {
    tS0 = tB0;
  }
  return launch_gemm<false, true>(tA, tB0, tB0, tS0, tS0, g, max_mtiles, s);
}

}  // namespace moe
