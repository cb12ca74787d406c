// Prefill path for MXFP4 experts with the clamped GLU: grouped GEMMs on tcgen05
// with f16 operands, each weight tile decoded once for two m tiles.
//
// Per expert e with rows (tokens, in the grouped order of the permute kernel):
//   gate_up:  gu[r, n] = X_r . W_gu,e[n] + b[n];  h = (clamp(up) + 1) * min(gate, L) * sigmoid(a * min(gate, L))
//   down   :  Y[slot(r), o] = h_r . W_d,e[o] + b_d[o]
//
// Operands.  Both MMA operands are f16 (kind::f16, fp32 accumulation in TMEM):
//   - x rows are staged as f16 times 2^e per row (largest magnitude in
//     [2^14, 2^15)), which holds every bf16 value of the row exactly except those
//     more than 2^38 below its largest; rowmul[r] = 2^-e undoes it in the epilogue.
//   - h is bounded by the clamps, |h| <= (L + 1) * max(L, 1 / alpha), so the gate_up
//     epilogue stores it as f16 times a fixed 2^kh (the bound lands below 2^15) and
//     records each row's largest |h|.  A row whose largest |h| is below 2^(-2 - kh)
//     would lose bits to f16 subnormals: for such rows (all of whose 8-feature
//     chunks are then small too) the epilogue also writes each small chunk in fp32,
//     and h_fix_f16_kernel (stage_f16.cu) re-stages the row with its own power of
//     two.  The down projection thus takes one f16 MMA per k step and h keeps 11
//     significant bits at any magnitude.
//   - weights: an E2M1 code converts exactly to f16 with cvt.rn.f16x2.e2m1x2; the
//     block scale 2^(s - 127) is split into 2^(s - 127 - c_n) * 2^c_n, with c_n per
//     weight row n chosen (fp4_prep_kernel) so that the largest finite block scale
//     of the row maps to 2^13.  Every block whose scale byte is within 36 of the row's
//     largest then decodes exactly in f16 (6 * 2^13 <= 65504, 0.5 * 2^-23 = 2^-24);
//     a block more than 2^36 below the row's largest decodes to zero (its products
//     are below fp32 rounding of the row's dot product).  colmul[n] = 2^c_n is
//     applied in the epilogue.  Scale byte 255 (NaN) stays NaN.
//
// Tiling.  A work item is up to 256 rows of one expert (two m tiles of 128); a
// unit is (work item, n tile of N <= 240 weight rows).  The dequantised B tile of
// a k step feeds the MMAs of both m tiles, which accumulate into two TMEM
// accumulators (columns 0 and 256).  One persistent CTA per SM; the CTAs claim units
// from a counter (the n tiles of an item in turn, the two-m-tile items first), so
// that they finish within about one unit of each other.  Warp roles:
//   warp 0        TMA producer: claims the units and hands them to the other roles
//                 through a small queue; per 64-input k step, the A tile of each m
//                 tile (128 x 64 f16, 128-byte swizzle) and the codes (N x 32 bytes)
//                 into a 4-stage ring;
//   warp 1        TMEM owner and MMA issuer (M 128, N, K 16, one elected thread);
//   warps 2..9    epilogue: two warps per TMEM lane quarter, each half of the columns;
//   warps 10..17  dequant: codes -> f16 B tile (128-byte swizzle) in a 2-deep ring;
//                 each thread reads the scale bytes of its rows for the next k step
//                 from global memory (the E8M0 layout as given) while it converts
//                 the current one.
// Every mbarrier wait is bounded; a wait that gives up sets the device status and
// an abort flag, the CTA drains its copies and MMAs in flight, frees TMEM, returns.
//
// Sources: "Phase 19: MoE - gpt-oss-20b", section 2 (Experts: interleaved gate_up
// with bias, clamped GLU, down with bias) and section 3 (MXFP4: E2M1 codes, low
// nibble first, one E8M0 scale per 32 inputs); "qwen35moe - Forward-Pass Design",
// "Batched prefill" (expert-grouped batching).
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "fp4_f16.cuh"
#include "internal.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;                          // rows per m tile (MMA M)
constexpr int kBK = 64;                           // inputs per k step: 128 bytes of f16
constexpr int kG = 2;                             // m tiles per unit (share one B tile)
constexpr int kMaxN = 240;                        // weight rows per unit (MMA N)
constexpr int kTileA = kBM * kBK * 2;             // 16 KiB
constexpr int kTileB = kMaxN * kBK * 2;           // 30 KiB
constexpr int kCodes = kMaxN * (kBK / 2);         // 7680 B
constexpr int kLoadStage = ((kG * kTileA + kCodes + 1023) / 1024) * 1024;
constexpr int kLoadStages = 4;
constexpr int kBStages = 2;
constexpr int kEpiConst = 2 * kMaxN * 4;         // per-unit column multipliers and biases (fp32)
constexpr int kSmemBytes = kLoadStages * kLoadStage + kBStages * kTileB + kEpiConst + 1024;
constexpr int kEpiWarps = 8;
constexpr int kDqWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps + kDqWarps);
constexpr uint32_t kTmemCols = 512;               // accumulators at columns 0 and 256
constexpr int kQ = 4;                             // unit queue: claimed units on their way to the roles
constexpr int kQTakers = 1 + kDqWarps + 1;        // MMA thread, dequant warps, epilogue thread 0

static_assert(kTileB % 1024 == 0, "B tiles must stay 1024-aligned");

struct F4Gemm {
  RouteState rs;              // work items of up to kG * kBM rows
  int E, R, nb;               // experts; weight rows per expert; 32-input blocks per row
  int N, nt, nkc;             // n tile width, n tiles per expert, k steps
  const float* colmul;        // [E * R] 2^c_n
  const int32_t* cinfo;       // [E * R] c_n in the low 16 bits (signed); bit 16: a block of the
                              // row needs the general multiplier (subnormal, flushed or NaN)
  const uint8_t* scales;      // E8M0 [E, R, nb]
  const float* rowmul;        // [S] 2^-e_r of the staged x rows (gate_up) or null
  const uint16_t* bias;       // bf16 [E, R] or null
  int gateup;                 // 1: gate_up (h out), 0: down (Y out)
  uint16_t* h16;              // f16 [S, ldh]: h * 2^kh
  float* hside;               // fp32 [S, ldh]: chunks of 8 features whose largest |h| < hsmall
  int ldh;
  float hboost, hsmall;       // 2^kh, 2^(-2 - kh)
  uint32_t* hmax;             // [S] largest |h| of each row (fp32 bits), accumulated
  float limit, alpha;
  float* Y;                   // fp32 [S, d] in slot order
  float* yacc;                // down, when non-null: yacc[slot / K] += slot_w[slot] * row (atomic
                              // adds) in place of the Y row
  float* yzero;               // gate_up, when non-null: cleared by the epilogue warps before their
  size_t yzero_n4;            // first unit (yzero_n4 float4s): the sums the down projection adds into
  int K;                      // slots per token
  int d;
  int* sched;                 // unit counter, zero at launch: CTAs claim units from it
  const int32_t* order;       // [work items] the order in which items are claimed
};

struct Unit {
  int v, row0, cnt, n;        // expert, first row within it, rows (<= 256), n tile
};

__device__ __forceinline__ Unit unit_at(const F4Gemm& g, int t) {
  Unit u;
  const int m = t / g.nt;
  u.n = t - m * g.nt;
  const int2 w = g.rs.work[m];
  u.v = w.x;
  u.row0 = w.y;
  const int rows = g.rs.offsets[u.v + 1] - g.rs.offsets[u.v];
  u.cnt = min(kG * kBM, rows - u.row0);
  return u;
}

// A dequant thread converts whole 32-input blocks: segment sg = tid + 256 i is block
// sg % 2 of the k step for weight row sg / 2.
constexpr int kDqThreads = 32 * kDqWarps;
constexpr int kSegs = (2 * kMaxN + kDqThreads - 1) / kDqThreads;

// Barrier among the epilogue warps only (named barrier 1).
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
}

// One 16-column chunk of the accumulated down projection.  Lane l holds v = 16
// accumulator columns of its row; the row's value is v * colmul * rm + bias, times
// the row's routing weight rw, added into the token's sum at ybase[dst] (dst = the
// token's row offset plus the unit's first column, ~0 for no row).  The four rows of
// a lane quad turn around by shuffles (a 4 x 4 transpose of float4 chunks, in two
// exchange steps) so that lane j of the quad adds chunk j of each of the four rows:
// one vector reduction instruction then covers 64 contiguous bytes of each of 8
// rows instead of 16 bytes of each of 32.  Every lane of the warp must call it.
__device__ __forceinline__ void red_chunk_turned(float (&v)[16], const float* cm, const float* bi, float rm,
                                                 size_t dst, float rw, float* ybase, int lane) {
  const float4* cm4 = reinterpret_cast<const float4*>(cm);
  const float4* bi4 = reinterpret_cast<const float4*>(bi);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = cm4[i], b = bi4[i];
    v[4 * i] = rw * fmaf(v[4 * i], f.x * rm, b.x);
    v[4 * i + 1] = rw * fmaf(v[4 * i + 1], f.y * rm, b.y);
    v[4 * i + 2] = rw * fmaf(v[4 * i + 2], f.z * rm, b.z);
    v[4 * i + 3] = rw * fmaf(v[4 * i + 3], f.w * rm, b.w);
  }
  const int j = lane & 3;
  // step 1 (lanes j, j ^ 2): the off-diagonal 2 x 2 blocks of chunks trade places
  {
    const bool hi = j & 2;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float send = hi ? v[e] : v[8 + e];          // chunks 0, 1 or chunks 2, 3
      const float got = __shfl_xor_sync(0xffffffffu, send, 2);
      if (hi) v[e] = got;
      else v[8 + e] = got;
    }
  }
  // step 2 (lanes j, j ^ 1): each 2 x 2 block transposes
  {
    const bool odd = j & 1;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c0 = 8 * blk + e, c1 = 8 * blk + 4 + e;   // element e of chunks 2 blk, 2 blk + 1
        const float send = odd ? v[c0] : v[c1];
        const float got = __shfl_xor_sync(0xffffffffu, send, 1);
        if (odd) v[c0] = got;
        else v[c1] = got;
      }
    }
  }
  // lane j now holds chunk j of the quad's rows 0..3 (as its chunks 0..3)
  const int base = lane & ~3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const unsigned long long dk = __shfl_sync(0xffffffffu, (unsigned long long)dst, base + k);
    if (dk != ~0ull)
      red_add_v4(ybase + dk + 4 * j, v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
fp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmC,
                const F4Gemm g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = tc::smem_align1024(smem_raw);
  uint8_t* bring = smem + kLoadStages * kLoadStage;
  __shared__ __align__(8) uint64_t full_bar[kLoadStages], empty_bar[kLoadStages], bfull_bar[kBStages],
      bempty_bar[kBStages], tfull_bar, tempty_bar, drain_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int consumed_s;     // loads the MMA thread has waited for
  // The producer claims each unit (atomicAdd on g.sched, mapped through g.order) and
  // hands it to the other roles through this queue; -1 ends the work.
  __shared__ __align__(8) uint64_t q_full[kQ], q_empty[kQ];
  __shared__ int unit_q[kQ];
  __shared__ int epi_unit_s;     // the unit the epilogue warps work on

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = g.rs.status;
  volatile int* abort = &abort_s;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLoadStages; ++s) {
      tc::mbar_init(tc::smem_u32(&full_bar[s]), 1);
      tc::mbar_init(tc::smem_u32(&empty_bar[s]), 1 + kDqWarps);   // MMA commit + dequant warps
    }
    for (int b = 0; b < kBStages; ++b) {
      tc::mbar_init(tc::smem_u32(&bfull_bar[b]), kDqWarps);
      tc::mbar_init(tc::smem_u32(&bempty_bar[b]), 1);
    }
    tc::mbar_init(tc::smem_u32(&tfull_bar), 1);
    tc::mbar_init(tc::smem_u32(&tempty_bar), kEpiWarps);
    tc::mbar_init(tc::smem_u32(&drain_bar), 1);
    for (int i = 0; i < kQ; ++i) {
      tc::mbar_init(tc::smem_u32(&q_full[i]), 1);
      tc::mbar_init(tc::smem_u32(&q_empty[i]), kQTakers);
    }
    abort_s = 0;
    consumed_s = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tmA);
    tc::tma_prefetch_desc(&tmC);
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&tmem_base_s), kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  pdl_wait();
  const int n_m = *g.rs.n_work;
  const int total = n_m > 0 ? n_m * g.nt : 0;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (tc::elect_one()) {
      int s = 0, issued = 0, qs = 0;
      uint32_t ph = 0, qph = 0;
      while (!*abort) {
        // Claim the next unit: the n tiles of each item in turn, items in g.order.  The
        // claim is made once this CTA's loads of its current unit are issued, a few k
        // steps before its MMAs run dry, so that the CTAs finish within about one unit.
        const int tk = atomicAdd(g.sched, 1);
        const int t = tk < total ? g.order[tk / g.nt] * g.nt + tk % g.nt : -1;
        if (!tc::mbar_wait(tc::smem_u32(&q_empty[qs]), qph ^ 1, abort, status)) break;
        unit_q[qs] = t;
        tc::mbar_arrive(tc::smem_u32(&q_full[qs]));
        if (++qs == kQ) {
          qs = 0;
          qph ^= 1;
        }
        if (t < 0) break;
        const Unit u = unit_at(g, t);
        const int a_row = g.rs.offsets[u.v] + u.row0;
        const int b_row = u.v * g.R + u.n * g.N;
        const int gm = u.cnt > kBM ? 2 : 1;
        const uint32_t bytes = (uint32_t)(gm * kTileA + g.N * 32);
        for (int kc = 0; kc < g.nkc; ++kc) {
          if (!tc::mbar_wait(tc::smem_u32(&empty_bar[s]), ph ^ 1, abort, status)) break;
          // A slot freed by an abort is not refilled: its last load may still be landing.
          if (*abort) break;
          const uint32_t fb = tc::smem_u32(&full_bar[s]);
          const uint32_t sa = tc::smem_u32(smem + s * kLoadStage);
          tc::mbar_arrive_expect_tx(fb, bytes);
          tc::tma_load_2d(sa, &tmA, kc * kBK, a_row, fb);
          if (gm == 2) tc::tma_load_2d(sa + kTileA, &tmA, kc * kBK, a_row + kBM, fb);
          tc::tma_load_2d(sa + kG * kTileA, &tmC, kc * 32, b_row, fb);
          ++issued;
          if (++s == kLoadStages) {
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
          tc::mbar_wait(tc::smem_u32(&full_bar[i % kLoadStages]), (i / kLoadStages) & 1, never, status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (tc::elect_one()) {
      int s = 0, bs = 0;
      uint32_t ph = 0, bph = 0, aph = 0;
      const uint32_t idesc = tc::idesc_f16_f32(kBM, g.N);
      bool any = false;
      int qs = 0;
      uint32_t qph = 0;
      while (!*abort) {
        if (!tc::mbar_wait(tc::smem_u32(&q_full[qs]), qph, abort, status)) break;
        const int t = *reinterpret_cast<volatile int*>(&unit_q[qs]);
        tc::mbar_arrive(tc::smem_u32(&q_empty[qs]));
        if (++qs == kQ) {
          qs = 0;
          qph ^= 1;
        }
        if (t < 0) break;
        const Unit u = unit_at(g, t);
        const int gm = u.cnt > kBM ? 2 : 1;
        if (!tc::mbar_wait(tc::smem_u32(&tempty_bar), aph ^ 1, abort, status)) break;
        tc::tc_fence_after();
        bool ok = true;
        for (int kc = 0; kc < g.nkc; ++kc) {
          if (!tc::mbar_wait(tc::smem_u32(&full_bar[s]), ph, abort, status) ||
              !tc::mbar_wait(tc::smem_u32(&bfull_bar[bs]), bph, abort, status)) {
            ok = false;
            break;
          }
          consumed_s = consumed_s + 1;
          tc::tc_fence_after();
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(smem + s * kLoadStage));
          const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(bring + bs * kTileB));
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j) {
            tc::umma_bf16(tmem, ad + 2 * j, bd + 2 * j, idesc, (kc | j) != 0);
            if (gm == 2) tc::umma_bf16(tmem + 256u, ad + (kTileA >> 4) + 2 * j, bd + 2 * j, idesc, (kc | j) != 0);
          }
          tc::umma_commit(tc::smem_u32(&empty_bar[s]));
          tc::umma_commit(tc::smem_u32(&bempty_bar[bs]));
          any = true;
          if (++s == kLoadStages) {
            s = 0;
            ph ^= 1;
          }
          if (++bs == kBStages) {
            bs = 0;
            bph ^= 1;
          }
        }
        if (!ok) break;
        tc::umma_commit(tc::smem_u32(&tfull_bar));
        aph ^= 1;
      }
      if (*abort && any) {
        // Let every MMA issued so far finish before TMEM is released.
        tc::umma_commit(tc::smem_u32(&drain_bar));
        int zero = 0;
        volatile int* never = &zero;
        tc::mbar_wait(tc::smem_u32(&drain_bar), 0, never, status);
      }
    }
  } else if (warp >= 2 + kEpiWarps) {
    // ---------------------------------------------------------------- MXFP4 dequant
    const int tid = threadIdx.x - 32 * (2 + kEpiWarps);
    int s = 0, bs = 0, qs = 0;
    uint32_t ph = 0, bph = 0, qph = 0;
    while (!*abort) {
      if (!tc::mbar_wait(tc::smem_u32(&q_full[qs]), qph, abort, status)) break;
      const int t = *reinterpret_cast<volatile int*>(&unit_q[qs]);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&q_empty[qs]));
      if (++qs == kQ) {
        qs = 0;
        qph ^= 1;
      }
      if (t < 0) break;
      const Unit u = unit_at(g, t);
      const size_t row0 = (size_t)u.v * g.R + (size_t)u.n * g.N;
      int c[kSegs], kr[kSegs];
      bool general = false;
      const uint8_t* sp[kSegs];
      uint32_t sb[kSegs];
#pragma unroll
      for (int i = 0; i < kSegs; ++i) {
        const int sg = min(tid + kDqThreads * i, 2 * g.N - 1);
        const int r = sg >> 1;
        const int ci = g.cinfo[row0 + r];
        c[i] = (int)(int16_t)(ci & 0xFFFF);
        kr[i] = 15 - 127 - c[i];
        general |= (ci >> 16) & 1;
        sp[i] = g.scales + (row0 + r) * g.nb + (sg & 1);
        sb[i] = sp[i][0];
      }
      // every row of the warp's segments in the plain range: multiplier = (s + kr) << 10
      general = __any_sync(0xffffffffu, general);
      bool ok = true;
      for (int kc = 0; kc < g.nkc; ++kc) {
        // the next step's scale bytes, read while this one converts
        uint32_t nx[kSegs];
        const int kn = min(kc + 1, g.nkc - 1);
#pragma unroll
        for (int i = 0; i < kSegs; ++i) nx[i] = __ldg(sp[i] + 2 * kn);
        if (!tc::mbar_wait(tc::smem_u32(&full_bar[s]), ph, abort, status) ||
            !tc::mbar_wait(tc::smem_u32(&bempty_bar[bs]), bph ^ 1, abort, status)) {
          ok = false;
          break;
        }
        const uint8_t* codes = smem + s * kLoadStage + kG * kTileA;
        uint8_t* bt = bring + bs * kTileB;
#pragma unroll
        for (int i = 0; i < kSegs; ++i) {
          const int sg = tid + kDqThreads * i;
          if (sg < 2 * g.N) {
            uint32_t m2;
            if (!general) m2 = f16op::block_mult_f16_plain(sb[i], (uint32_t)kr[i]);
            else m2 = f16op::block_mult_f16(sb[i], c[i]);
            f16op::dequant_block(codes, bt, sg >> 1, sg & 1, m2);
          }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(tc::smem_u32(&bfull_bar[bs]));
          tc::mbar_arrive(tc::smem_u32(&empty_bar[s]));
        }
#pragma unroll
        for (int i = 0; i < kSegs; ++i) sb[i] = nx[i];
        if (++s == kLoadStages) {
          s = 0;
          ph ^= 1;
        }
        if (++bs == kBStages) {
          bs = 0;
          bph ^= 1;
        }
      }
      if (!ok) break;
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                      // TMEM lane quarter this warp may read
    const int half = (warp - 2) >> 2;            // which half of the 16-column chunks
    const int etid = threadIdx.x - 64;           // 0 .. 255 over the epilogue warps
    const int nch = g.N / 16;
    const int c_begin = half ? (nch + 1) / 2 : 0, c_end = half ? nch : (nch + 1) / 2;
    float* ecm = reinterpret_cast<float*>(bring + kBStages * kTileB);   // [N] 2^c_n
    float* ebi = ecm + kMaxN;                                            // [N] bias
    uint32_t aph = 0;
    if (g.yzero) {
      // this CTA's share of the per-token sums of the accumulated down projection,
      // cleared while the first unit's MMAs run
      const size_t per = (g.yzero_n4 + gridDim.x - 1) / gridDim.x;
      const size_t z0 = per * blockIdx.x, z1 = min(g.yzero_n4, z0 + per);
      float4* z = reinterpret_cast<float4*>(g.yzero);
      for (size_t i = z0 + etid; i < z1; i += 32 * kEpiWarps) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int qs = 0;
    uint32_t qph = 0;
    for (;;) {
      // Epilogue thread 0 takes the next unit from the queue (-1 at the end or on
      // give-up) and every epilogue warp reads it after the barrier: a uniform exit.
      // The barrier also ends every use of the previous unit's constants.
      if (etid == 0) {
        int t = -1;
        if (!*abort && tc::mbar_wait(tc::smem_u32(&q_full[qs]), qph, abort, status)) {
          t = *reinterpret_cast<volatile int*>(&unit_q[qs]);
          tc::mbar_arrive(tc::smem_u32(&q_empty[qs]));
          if (++qs == kQ) {
            qs = 0;
            qph ^= 1;
          }
        }
        epi_unit_s = t;
      }
      epi_sync();
      const int t = epi_unit_s;
      if (t < 0) break;
      const Unit u = unit_at(g, t);
      const int gm = u.cnt > kBM ? 2 : 1;
      const int col0 = u.n * g.N;                          // first weight row of the unit
      // The unit's column constants into shared memory and the rows' factors into
      // registers while the MMAs run.
      for (int i = etid; i < g.N; i += 32 * kEpiWarps) {
        ecm[i] = g.colmul[(size_t)u.v * g.R + col0 + i];
        ebi[i] = g.bias ? bf16_to_f32(g.bias[(size_t)u.v * g.R + col0 + i]) : 0.f;
      }
      float rm[kG], rw[kG];
      size_t dst[kG];
#pragma unroll
      for (int gi = 0; gi < kG; ++gi) {
        const int row = gi * kBM + 32 * q + lane;
        const int grow = g.rs.offsets[u.v] + u.row0 + row;
        const bool valid = gi < gm && row < u.cnt;
        rm[gi] = (valid && g.rowmul) ? g.rowmul[grow] : 1.f;
        const int slot = (valid && !g.gateup) ? g.rs.row2slot[grow] : 0;
        rw[gi] = (valid && g.yacc) ? g.rs.slot_w[slot] : 1.f;
        dst[gi] = !valid ? ~size_t(0)
                  : g.gateup ? (size_t)grow * g.ldh + col0 / 2
                  : g.yacc   ? (size_t)(slot / g.K) * g.d + col0
                             : (size_t)slot * g.d + col0;
      }
      epi_sync();
      // On give-up the abort flag is set, and thread 0 then ends the loop.
      if (!tc::mbar_wait(tc::smem_u32(&tfull_bar), aph, abort, status)) continue;
      tc::tc_fence_after();
      for (int gi = 0; gi < gm; ++gi) {
        const bool valid = dst[gi] != ~size_t(0);
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(256 * gi);
        uint32_t hm = 0;                                   // largest |h| of this row here
        for (int c = c_begin; c < c_end; ++c) {
          float v[16];
          tc::tmem_ld16(taddr + (uint32_t)(16 * c), v);
          if (g.yacc) {
            // down, accumulated (every lane of the warp takes part: the shuffles)
            red_chunk_turned(v, ecm + 16 * c, ebi + 16 * c, valid ? rm[gi] : 1.f, valid ? dst[gi] : ~size_t(0),
                             rw[gi], g.yacc + 16 * c, lane);
            continue;
          }
          if (!valid) continue;
          const float4* cm4 = reinterpret_cast<const float4*>(ecm + 16 * c);
          const float4* bi4 = reinterpret_cast<const float4*>(ebi + 16 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 f = cm4[i], b = bi4[i];
            v[4 * i] = fmaf(v[4 * i], f.x * rm[gi], b.x);
            v[4 * i + 1] = fmaf(v[4 * i + 1], f.y * rm[gi], b.y);
            v[4 * i + 2] = fmaf(v[4 * i + 2], f.z * rm[gi], b.z);
            v[4 * i + 3] = fmaf(v[4 * i + 3], f.w * rm[gi], b.w);
          }
          if (g.gateup) {
            // columns 2i (gate) and 2i + 1 (up) of feature 8c + i
            float hv[8];
            uint32_t cmax = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              hv[i] = f16op::clamped_glu(v[2 * i], v[2 * i + 1], g.limit, g.alpha);
              cmax = max(cmax, f16op::abs_bits(hv[i]));
            }
            hm = max(hm, cmax);
            uint32_t hp[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) hp[i] = pack_f16x2(hv[2 * i] * g.hboost, hv[2 * i + 1] * g.hboost);
            *reinterpret_cast<uint4*>(g.h16 + dst[gi] + 8 * c) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
            if (__uint_as_float(cmax) < g.hsmall) {
              float4* sp = reinterpret_cast<float4*>(g.hside + dst[gi] + 8 * c);
              sp[0] = make_float4(hv[0], hv[1], hv[2], hv[3]);
              sp[1] = make_float4(hv[4], hv[5], hv[6], hv[7]);
            }
          } else {
            // Y rows are d fp32 apart with d a multiple of 32, and 16 c + col0 is a
            // multiple of 16: both halves of the chunk start on 32 bytes.
            stg_v8(g.Y + dst[gi] + 16 * c, v);
            stg_v8(g.Y + dst[gi] + 16 * c + 8, v + 8);
          }
        }
        if (g.gateup && valid) atomicMax(g.hmax + (dst[gi] - col0 / 2) / g.ldh, hm);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&tempty_bar));
      aph ^= 1;
    }
  }

  pdl_trigger();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

constexpr int kPrepRows = 128;                     // weight rows per prep CTA (one per thread)

// One matrix of weight-row scales [rows, nb blocks] and its per-row outputs.
struct PrepMat {
  const uint8_t* scales;
  long long rows;
  int nb;
  float* colmul;
  int32_t* cinfo;
};

// Per weight row n of each matrix (gate_up, then down): c_n from the row's largest
// finite scale byte (that block's multiplier becomes 2^13), colmul[n] = 2^c_n, and
// cinfo[n] = c_n | general << 16, where `general` marks a row with a block whose
// multiplier is not a normal f16 (scale byte more than 27 below the largest, or 255).
// One CTA per 128 weight rows (the first blocks0 CTAs take matrix 0), one thread per
// row, the rows staged in shared memory.
__global__ void __launch_bounds__(256)
fp4_prep_kernel(const PrepMat m0, const PrepMat m1, int blocks0) {
  extern __shared__ uint8_t tile[];               // kPrepRows rows of nb scale bytes
  pdl_wait();
  pdl_trigger();
  const bool second = (int)blockIdx.x >= blocks0;
  const PrepMat& m = second ? m1 : m0;
  const uint8_t* __restrict__ scales = m.scales;
  const long long rows = m.rows;
  const int nb = m.nb;
  float* __restrict__ colmul = m.colmul;
  int32_t* __restrict__ cinfo = m.cinfo;
  const long long r0 = (long long)(second ? blockIdx.x - blocks0 : blockIdx.x) * kPrepRows;
  const int nrows = (int)min((long long)kPrepRows, rows - r0);
  const int bytes = nrows * nb;
  // The tile's rows are contiguous: copy them with 16-byte loads (r0 * nb is a
  // multiple of 16), the ragged end byte by byte.
  const uint8_t* src = scales + r0 * nb;
  const int nvec = bytes / 16;
  for (int i = threadIdx.x; i < nvec; i += blockDim.x)
    reinterpret_cast<uint4*>(tile)[i] = ldg_nc_v4(src + 16 * i);
  for (int i = 16 * nvec + threadIdx.x; i < bytes; i += blockDim.x) tile[i] = src[i];
  __syncthreads();
  const int t = threadIdx.x;
  if (t < nrows) {
    const uint8_t* sr = tile + t * nb;
    int smax = -1, smin = 256;
    for (int b = 0; b < nb; ++b) {
      const int sv = sr[b];
      if (sv != 255) smax = max(smax, sv);
      smin = min(smin, sv == 255 ? -1000 : sv);
    }
    const int c = smax < 0 ? 0 : smax - 140;
    const int general = (smax < 0 || smin < smax - 27) ? 1 : 0;
    cinfo[r0 + t] = (c & 0xFFFF) | (general << 16);
    colmul[r0 + t] = ldexpf(1.f, c);
  }
}

// Largest N (multiple of 16, at most max_n) that divides `rows`; 0 if none.
int tile_n16(int rows, int max_n) {
  for (int n = max_n; n >= 16; n -= 16)
    if (rows % n == 0) return n;
  return 0;
}

void set_fp4_gemm_smem() {
  static bool done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || done[dev]) return;
  cudaFuncSetAttribute(fp4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  done[dev] = true;
}

struct Fp4Scratch {
  float* colmul_gu;     // [E * 2ff]
  float* colmul_dn;     // [E * d]
  int32_t* cinfo_gu;    // [E * 2ff]
  int32_t* cinfo_dn;    // [E * d]
  float* rowmul;        // [S] 2^-e of the staged x rows
  uint32_t* hmax;       // [S] largest |h| per row
  float* hmul;          // [S] 2^-e of the staged h rows
  int32_t* order;       // [max items] the order in which the GEMMs' CTAs claim work items
  int32_t* sched;       // [2] unit counters of gate_up and down
};

size_t carve_off(const ExpertParams& p, int S, Fp4Scratch* sc, uint8_t* base) {
  auto a256 = [](size_t v) { return (v + 255) & ~size_t(255); };
  const size_t Rg = 2 * (size_t)p.ff * p.E, Rd = (size_t)p.d * p.E;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* q = base ? base + off : nullptr;
    off = a256(off + bytes);
    return q;
  };
  uint8_t* a = take(4 * Rg);
  uint8_t* b = take(4 * Rd);
  uint8_t* c = take(4 * Rg);
  uint8_t* d = take(4 * Rd);
  uint8_t* e = take(4 * (size_t)S);
  uint8_t* f = take(4 * (size_t)S);
  uint8_t* h = take(4 * (size_t)S);
  uint8_t* o = take(4 * ((size_t)p.E + ((size_t)S + 2 * kBM - 1) / (2 * kBM)));
  uint8_t* q = take(8);
  if (sc) {
    sc->colmul_gu = reinterpret_cast<float*>(a);
    sc->colmul_dn = reinterpret_cast<float*>(b);
    sc->cinfo_gu = reinterpret_cast<int32_t*>(c);
    sc->cinfo_dn = reinterpret_cast<int32_t*>(d);
    sc->rowmul = reinterpret_cast<float*>(e);
    sc->hmax = reinterpret_cast<uint32_t*>(f);
    sc->hmul = reinterpret_cast<float*>(h);
    sc->order = reinterpret_cast<int32_t*>(o);
    sc->sched = reinterpret_cast<int32_t*>(q);
  }
  return off;
}

Fp4Scratch carve(const ExpertParams& p, uint8_t* base, int S) {
  Fp4Scratch sc;
  carve_off(p, S, &sc, base);
  return sc;
}

cudaError_t launch_fp4_gemm(const CUtensorMap& tA, const CUtensorMap& tC, const F4Gemm& g, int max_items,
                            cudaStream_t s) {
  set_fp4_gemm_smem();
  const long long units = (long long)max_items * g.nt;
  int grid = sm_count();
  if (units < grid) grid = (int)(units > 0 ? units : 1);
  return launch_pdl(fp4_gemm_kernel, dim3(grid), dim3(kThreads), kSmemBytes, s, tA, tC, g);
}

}  // namespace

bool prefill_fp4_supported(const ExpertParams& p, int wfmt, int interleaved) {
  if (wfmt != MOE_WFMT_MXFP4 || !interleaved || p.sff || p.act != MOE_ACT_CLAMPED_GLU) return false;
  if (p.d % kBK || p.ff % kBK) return false;
  // h must stay well inside the f16 range: |h| <= (L + 1) * max(L, 1 / alpha).
  if (!(p.limit >= 0.f) || !(p.alpha > 0.f)) return false;
  const double bound = ((double)p.limit + 1.0) * fmax((double)p.limit, 1.0 / (double)p.alpha);
  if (!(bound <= 16384.0)) return false;
  // gate_up N: a multiple of 16 (so gate, up pairs never straddle a tile) dividing 2ff.
  return tile_n16(2 * p.ff, kMaxN) != 0 && tile_n16(p.d, kMaxN) != 0;
}

size_t prefill_fp4_scratch_bytes(const ExpertParams& p, int S) { return carve_off(p, S, nullptr, nullptr); }

int h_stage_exp(float limit, float alpha) {
  const double bound = ((double)limit + 1.0) * fmax((double)limit, 1.0 / (double)alpha);
  int kh = 0;
  while (kh < 24 && bound * std::ldexp(1.0, kh + 1) < 32768.0) ++kh;
  return kh;
}

cudaError_t launch_prefill_fp4_prep(const ExpertParams& p, uint8_t* scratch, int S, cudaStream_t s) {
  const Fp4Scratch sc = carve(p, scratch, S);
  const long long rg = (long long)p.E * 2 * p.ff, rd = (long long)p.E * p.d;
  const int nbg = p.d / 32, nbd = p.ff / 32;
  const int smem = kPrepRows * (nbg > nbd ? nbg : nbd);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(fp4_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return cudaErrorInvalidValue;
  const PrepMat gu{p.gu_scales, rg, nbg, sc.colmul_gu, sc.cinfo_gu};
  const PrepMat dn{p.dn_scales, rd, nbd, sc.colmul_dn, sc.cinfo_dn};
  const int bg = (int)((rg + kPrepRows - 1) / kPrepRows), bd = (int)((rd + kPrepRows - 1) / kPrepRows);
  return launch_pdl(fp4_prep_kernel, dim3((unsigned)(bg + bd)), dim3(kPrepRows), (size_t)smem, s, gu, dn, bg);
}

Fp4Rows prefill_fp4_rows(const ExpertParams& p, uint8_t* scratch, int S) {
  const Fp4Scratch sc = carve(p, scratch, S);
  return Fp4Rows{sc.rowmul, sc.hmax, sc.hmul, sc.order, sc.sched};
}

cudaError_t launch_gateup_prefill_fp4(const ExpertParams& p, const RouteState& rs, const uint16_t* xp16, int S,
                                      uint16_t* h16, float* hside, int ldh, int kh, uint8_t* scratch,
                                      int max_items, float* yzero, size_t yzero_floats, cudaStream_t s) {
  const Fp4Scratch sc = carve(p, scratch, S);
  F4Gemm g{};
  g.rs = rs;
  g.yzero = yzero;
  g.yzero_n4 = yzero_floats / 4;
  g.E = p.E;
  g.R = 2 * p.ff;
  g.nb = p.d / 32;
  g.N = tile_n16(g.R, kMaxN);
  g.nt = g.R / g.N;
  g.nkc = p.d / kBK;
  g.colmul = sc.colmul_gu;
  g.cinfo = sc.cinfo_gu;
  g.scales = p.gu_scales;
  g.rowmul = sc.rowmul;
  g.bias = p.gu_bias;
  g.gateup = 1;
  g.h16 = h16;
  g.hside = hside;
  g.ldh = ldh;
  g.hboost = ldexpf(1.f, kh);
  g.hsmall = ldexpf(1.f, -2 - kh);
  g.hmax = sc.hmax;
  g.sched = sc.sched;
  g.order = sc.order;
  g.limit = p.limit;
  g.alpha = p.alpha;
  g.d = p.d;
  CUtensorMap tA, tC;
  if (!make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xp16, (uint64_t)(S > 0 ? S : 1), (uint64_t)p.d,
                (uint64_t)p.d * 2, kBM, kBK, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!make_map(&tC, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.gate_up, (uint64_t)p.E * g.R, (uint64_t)p.d / 2,
                (uint64_t)p.d / 2, (uint32_t)g.N, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  return launch_fp4_gemm(tA, tC, g, max_items, s);
}

cudaError_t prefill_fp4_set_wait_test(uint32_t polls, int withhold) { return tc::set_wait_test(polls, withhold); }

cudaError_t launch_down_prefill_fp4(const ExpertParams& p, const RouteState& rs, const uint16_t* h16, int ldh16,
                                    int S, float* Y, float* yacc, int K, uint8_t* scratch, int max_items,
                                    cudaStream_t s) {
  const Fp4Scratch sc = carve(p, scratch, S);
  F4Gemm g{};
  g.rs = rs;
  g.yacc = yacc;
  g.K = K;
  g.E = p.E;
  g.R = p.d;
  g.nb = p.ff / 32;
  g.N = tile_n16(g.R, kMaxN);
  g.nt = g.R / g.N;
  g.nkc = p.ff / kBK;
  g.colmul = sc.colmul_dn;
  g.cinfo = sc.cinfo_dn;
  g.scales = p.dn_scales;
  g.rowmul = sc.hmul;
  g.bias = p.dn_bias;
  g.gateup = 0;
  g.sched = sc.sched + 1;
  g.order = sc.order;
  g.Y = Y;
  g.d = p.d;
  CUtensorMap tA, tC;
  if (!make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, h16, (uint64_t)(S > 0 ? S : 1), (uint64_t)p.ff,
                (uint64_t)ldh16 * 2, kBM, kBK, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!make_map(&tC, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.down, (uint64_t)p.E * g.R, (uint64_t)p.ff / 2,
                (uint64_t)p.ff / 2, (uint32_t)g.N, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  return launch_fp4_gemm(tA, tC, g, max_items, s);
}

}  // namespace moe
