// Decode path for bf16 experts with few tokens per expert (work items of at most 8
// token rows): the weights stream through a TMA-fed shared-memory ring, so that the
// bytes in flight per SM do not depend on registers.
//
// One persistent CTA per SM takes an equal contiguous share of the units (work item
// x 128 weight rows, or 64 when the expected work would give the CTAs fewer than
// four units each).  Warp 16 is the producer: one elected lane streams each unit's
// rows into a ring of 32 KB stages, a stage being 64-input k chunks of the unit's
// rows (two TMA boxes of half the unit's rows x 128 bytes each, 128-byte swizzle).
//   gate_up: the rows of a unit are the gate rows then the up rows of the same
//            features (separate gate and up matrices);
//   down:    consecutive output rows of the down matrix.
// The shared expert (virtual expert E) takes its own matrices.
//
// Warps 0..15 consume: each MMA tile of 16 rows has 16 / tiles warps, which take
// the k16 steps of every chunk in turn.  An ldmatrix x4 of the swizzled stage gives
// the tile's A fragment (gate_up: rows 0..7 the gate rows and rows 8..15 the up rows
// of 8 features, so that one lane holds gate and up of the same feature; down: 16
// consecutive output rows); the item's token rows, staged in shared memory as bf16
// (h as its (hi, lo) pair), give the B fragments by ldmatrix as well.  mma.sync
// m16n8k16 with fp32 accumulation; at the unit's end the tile's warps add their
// sums in order and the first runs the epilogue.
//
// Sources: "qwen35moe - Forward-Pass Design", sections "Shared-expert MoE FFN"
// (SwiGLU experts, shared expert) and "K80 GPU decode" (grouped MoE: all selected
// experts' gate + up + SwiGLU in one launch, then the down pass).
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int kCW = 16;                           // consumer warps
constexpr int kThreads = (kCW + 1) * 32;          // + the producer warp
constexpr int kStageBytes = 32 * 1024;            // one ring stage
constexpr int kMaxRingStages = 8;
constexpr int kTokens = 8;                        // token rows per work item

// Unit geometry: TILES 16-row MMA tiles (8, or 4 when there are few units, so that
// the CTAs' shares even out); TMA boxes of 8 TILES rows x 128 bytes (64 inputs), two
// per 64-input k chunk; the consumer warps split into TILES tiles x 16 / TILES k16
// step classes.
template <int TILES>
struct Geo {
  static constexpr int kRows = 16 * TILES;                  // weight rows per unit
  static constexpr int kBoxRows = 8 * TILES;
  static constexpr int kBoxBytes = kBoxRows * 128;
  static constexpr int kChunkBytes = 2 * kBoxBytes;         // a 64-input k chunk of the unit's rows
  static constexpr int kChunks = kStageBytes / kChunkBytes;  // k chunks per ring stage
  static constexpr int kClasses = kCW / TILES;              // warps per tile (k16 step classes)
};

// Shared memory, from a 1024-aligned base: ring stages | partial sums | token rows
// (for down, the lo halves follow the hi rows).
struct RingSmem {
  int stages, pitch, ring, part, tok, total;
};

// Token row pitch: the row plus 16 bytes, so that the 8 rows read by one ldmatrix
// phase fall in different banks (kin is a multiple of 64).
__host__ __device__ inline int ring_pitch(int kin) { return 2 * kin + 16; }

__host__ __device__ inline RingSmem ring_smem(int kin, bool pair, int stages) {
  RingSmem m;
  m.stages = stages;
  m.pitch = ring_pitch(kin);
  m.ring = 0;
  m.part = stages * kStageBytes;
  m.tok = m.part + kCW * 32 * 16;                  // partial sums [tile][class][lane]
  m.total = m.tok + (pair ? 2 : 1) * kTokens * m.pitch;
  return m;
}

__device__ __forceinline__ float act_swiglu(float g, float u) { return g / (1.f + __expf(-g)) * u; }

__device__ __forceinline__ float act_clamped(float g, float u, float limit, float alpha) {
  g = fminf(g, limit);
  u = fminf(fmaxf(u, -limit), limit);
  return (u + 1.f) * g / (1.f + __expf(-alpha * g));
}

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory");
}

// Barrier among the warps of one tile (named barriers 2 .. 2 + TILES - 1).
template <int CLASSES>
__device__ __forceinline__ void tile_sync(int tile) {
  asm volatile("bar.sync %0, %1;" ::"r"(2 + tile), "n"(CLASSES * 32) : "memory");
}

// volatile: they read shared memory that an mbarrier wait or a barrier made valid.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

struct RingArgs {
  RouteState rs;
  int E;
  int R, Rs;                  // weight rows per routed / shared expert: gate_up ff / sff features, down d
  int kin, kin_s;             // inputs per weight row, routed / shared: gate_up d, down ff / sff
  int tiles;                  // units per work item: max over routed and shared
  int stages;
  const uint16_t* gu_bias;    // gate_up: [E, 2ff] (gate, up pairs) or null
  const uint16_t* dn_bias;    // down: [E, d] or null
  const uint16_t* x;          // gate_up: x rows in, h (hi, lo) rows out
  int K;
  uint16_t* h;
  int ldh;
  int act;
  float limit, alpha;
  float* Y;                   // down: Y rows (slot order) out
};

// GATEUP: the units' rows are 64 gate rows (map m0) then 64 up rows (map m1) of the
// same features; routed experts from m0 / m1, the shared expert from s0 / s1.
// Otherwise: 128 down rows from m0 (shared: s0), tokens are h (hi, lo) rows.
template <bool GATEUP, int TILES>
__global__ void __launch_bounds__(kThreads, 1)
ring_stream_kernel(const __grid_constant__ CUtensorMap m0, const __grid_constant__ CUtensorMap m1,
                   const __grid_constant__ CUtensorMap s0, const __grid_constant__ CUtensorMap s1,
                   const RingArgs a) {
  using G = Geo<TILES>;
  constexpr int kRows = G::kRows, kBoxRows = G::kBoxRows, kBoxBytes = G::kBoxBytes;
  constexpr int kChunkBytes = G::kChunkBytes, kChunks = G::kChunks, kClasses = G::kClasses;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = tc::smem_align1024(smem_raw);
  __shared__ __align__(8) uint64_t full_bar[kMaxRingStages], empty_bar[kMaxRingStages];
  __shared__ int abort_s;
  __shared__ const uint8_t* trows[kTokens];

  const int kmax = a.kin > a.kin_s ? a.kin : a.kin_s;
  const RingSmem L = ring_smem(kmax, !GATEUP, a.stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = a.rs.status;
  volatile int* abort = &abort_s;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      tc::mbar_init(tc::smem_u32(&full_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&empty_bar[i]), kCW * 32);   // every consumer lane arrives
    }
    abort_s = 0;
    tc::fence_barrier_init();
  }
  if (warp == kCW && lane == 0) {
    tc::tma_prefetch_desc(&m0);
    tc::tma_prefetch_desc(&s0);
    if (GATEUP) {
      tc::tma_prefetch_desc(&m1);
      tc::tma_prefetch_desc(&s1);
    }
  }
  __syncthreads();
  // gate_up: the work list comes from the grouping kernel just before.  down: it was
  // there before the gate_up launch let this one start (each of its CTAs waited for
  // the grouping); only h depends on gate_up, and the consumers wait for it before
  // they first stage it.  The producer waits too, so that its weight stream does not
  // take bandwidth from gate_up's last units.
  if (GATEUP || warp == kCW) pdl_wait();

  const int n_items = *a.rs.n_work;
  const long long U = (long long)(n_items > 0 ? n_items : 0) * a.tiles;
  const int u0 = (int)(U * blockIdx.x / gridDim.x), u1 = (int)(U * (blockIdx.x + 1) / gridDim.x);
  // unit u: work item u / tiles, kRows weight rows (gate_up: kRows / 2 features) number
  // u % tiles; an expert with fewer rows than the widest skips its last units
  constexpr int kUnitRows = GATEUP ? kRows / 2 : kRows;
  auto unit_on = [&](int v, int t) { return kUnitRows * t < (v == a.E ? a.Rs : a.R); };

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    if (tc::elect_one()) {
      int it = 0, st = 0;                       // ring loads issued, ring slot of the next one
      uint32_t ph = 0;
      for (int u = u0; u < u1 && !*abort; ++u) {
        const int ai = u / a.tiles, t = u - ai * a.tiles;
        const int v = a.rs.work[ai].x;
        if (!unit_on(v, t)) continue;
        const bool sh = v == a.E;
        const int nkc = (sh ? a.kin_s : a.kin) / 64;
        const CUtensorMap* mg = sh ? &s0 : &m0;
        const CUtensorMap* mu = sh ? &s1 : &m1;
        const int row = (sh ? 0 : v * a.R) + kUnitRows * t;
        for (int kc = 0; kc < nkc; kc += kChunks) {
          if (!tc::mbar_wait(tc::smem_u32(&empty_bar[st]), ph ^ 1, abort, status)) break;
          // A slot freed by an abort is not refilled: its last load may still be landing.
          if (*abort) break;
          const int nch = min(kChunks, nkc - kc);
          tc::mbar_arrive_expect_tx(tc::smem_u32(&full_bar[st]), (uint32_t)(nch * kChunkBytes));
          for (int j = 0; j < nch; ++j) {
            const uint32_t dst = tc::smem_u32(smem + st * kStageBytes + j * kChunkBytes);
            const int k0 = (kc + j) * 64;
            if (GATEUP) {
              tc::tma_load_2d(dst, mg, k0, row, tc::smem_u32(&full_bar[st]));
              tc::tma_load_2d(dst + kBoxBytes, mu, k0, row, tc::smem_u32(&full_bar[st]));
            } else {
              tc::tma_load_2d(dst, mg, k0, row, tc::smem_u32(&full_bar[st]));
              tc::tma_load_2d(dst + kBoxBytes, mg, k0, row + kBoxRows, tc::smem_u32(&full_bar[st]));
            }
          }
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
          tc::mbar_wait(tc::smem_u32(&full_bar[i % a.stages]), (i / a.stages) & 1, never, status);
      }
    }
    // no early signal to the dependent launch: the consumers give it when the CTA's
    // work is done
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tile = warp % TILES, cls = warp / TILES;
  const int g = lane >> 2, c = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;        // this lane's ldmatrix address: matrix, row
  // A: the box and row of MMA row 8 (mi & 1) + ri of the tile; k half mi >> 1
  int abox, arow;
  if (GATEUP) {
    abox = mi & 1;                               // gate rows, then up rows
    arow = 8 * tile + ri;
  } else {
    const int m = 16 * tile + 8 * (mi & 1) + ri;
    abox = m / kBoxRows;
    arow = m % kBoxRows;
  }
  const uint32_t aoff = (uint32_t)(abox * kBoxBytes + arow * 128);
  const int kh = mi >> 1;
  // B: lanes 0..15 address token row lane % 8 at k half (lane / 8) % 2 (x2 ldmatrix)
  uint8_t* tok = smem + L.tok;
  const uint32_t boff = tc::smem_u32(tok) + (uint32_t)((lane & 7) * L.pitch + ((lane >> 3) & 1) * 16);
  const uint32_t lo_off = (uint32_t)(kTokens * L.pitch);
  float4* part = reinterpret_cast<float4*>(smem + L.part) + tile * kClasses * 32 + lane;
  int st = 0, cur = -1;                          // ring slot, staged item
  uint32_t ph = 0;
  for (int u = u0; u < u1; ++u) {
    // On abort every wait returns at once; the loop still runs to its end so that
    // all consumer warps take the same barriers.
    const int ai = u / a.tiles, t = u - ai * a.tiles;
    const int2 item = a.rs.work[ai];
    const int v = item.x;
    if (!unit_on(v, t)) continue;
    const bool sh = v == a.E;
    const int r0 = a.rs.offsets[v] + item.y;     // first permuted row of the item
    const int n = min(kTokens, a.rs.offsets[v + 1] - r0);
    const int kin = sh ? a.kin_s : a.kin;
    if (ai != cur) {
      // the item's token rows as bf16 (down: hi rows, then lo rows), rows n..7 zero
      if (!GATEUP && cur < 0) pdl_wait();        // down: h is gate_up's output
      consumers_sync();                          // every warp is done with the old rows
      if (threadIdx.x < kTokens) {
        const int i = threadIdx.x;
        const uint8_t* p = nullptr;
        if (i < n) {
          if (GATEUP)
            p = reinterpret_cast<const uint8_t*>(a.x + (size_t)(a.rs.row2slot[r0 + i] / a.K) * kin);
          else
            p = reinterpret_cast<const uint8_t*>(a.h + (size_t)(r0 + i) * 2 * a.ldh);
        }
        trows[i] = p;
      }
      consumers_sync();
      {
        const int r = warp % kTokens, hf = warp / kTokens;
        const int per = kin / 8;                 // 16-byte units per row
        const uint8_t* src = trows[r];
        // every load of the lane (both halves of an h row) before any store: one round trip
        constexpr int kU = 4;                    // 16-byte units per lane and half row in flight
        uint4* drow = reinterpret_cast<uint4*>(tok + (size_t)r * L.pitch);
        uint4* drow_lo = reinterpret_cast<uint4*>(tok + lo_off + (size_t)r * L.pitch);
        for (int i0 = hf * 32 + lane; i0 < per; i0 += 64 * kU) {
          uint4 hv[kU], lv[kU];
#pragma unroll
          for (int j = 0; j < kU; ++j) {
            const int i = i0 + 64 * j;
            hv[j] = lv[j] = make_uint4(0u, 0u, 0u, 0u);
            if (src && i < per) {
              hv[j] = ldg_nc_v4(src + 16 * i);
              if (!GATEUP) lv[j] = ldg_nc_v4(src + (size_t)a.ldh * 2 + 16 * i);
            }
          }
#pragma unroll
          for (int j = 0; j < kU; ++j) {
            const int i = i0 + 64 * j;
            if (i < per) {
              drow[i] = hv[j];
              if (!GATEUP) drow_lo[i] = lv[j];
            }
          }
        }
      }
      consumers_sync();
      cur = ai;
    }
    const int nkc = kin / 64;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    bool ok = true;
    for (int kc = 0; kc < nkc; kc += kChunks) {
      ok = ok && tc::mbar_wait(tc::smem_u32(&full_bar[st]), ph, abort, status);
      if (ok) {
        const int nch = min(kChunks, nkc - kc);
        const uint32_t sbase = tc::smem_u32(smem + st * kStageBytes) + aoff;
        for (int j = 0; j < nch; ++j) {
#pragma unroll
          for (int s16 = cls; s16 < 4; s16 += kClasses) {   // this warp's k16 steps of the chunk
            const int kg = (kc + j) * 64 + 16 * s16;
            uint32_t A[4], b0, b1;
            ldsm_x4(sbase + j * kChunkBytes + ((uint32_t)((2 * s16 + kh) ^ ri) << 4), A);
            ldsm_x2(boff + (uint32_t)(2 * kg), b0, b1);
            mma_bf16_16816(acc, A[0], A[1], A[2], A[3], b0, b1);
            if (!GATEUP) {
              ldsm_x2(boff + lo_off + (uint32_t)(2 * kg), b0, b1);
              mma_bf16_16816(acc, A[0], A[1], A[2], A[3], b0, b1);
            }
          }
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
    // the tile's step classes add up in class order in the class-0 warp
    if (cls) part[cls * 32] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    tile_sync<kClasses>(tile);
    if (!cls) {
#pragma unroll
      for (int q = 1; q < kClasses; ++q) {
        const float4 o = part[q * 32];
        acc[0] += o.x;
        acc[1] += o.y;
        acc[2] += o.z;
        acc[3] += o.w;
      }
    }
    tile_sync<kClasses>(tile);                   // read before the next unit writes
    if (cls || !ok) continue;

    // ------------------------------------------------------------ epilogue
    // acc: MMA rows g (tokens 2c, 2c+1) and g + 8
    if (GATEUP) {
      const int f = kUnitRows * t + 8 * tile + g;   // row g: its gate, row g + 8: its up
      float bg = 0.f, bu = 0.f;
      if (!sh && a.gu_bias) {
        const size_t row = (size_t)v * 2 * a.R + 2 * (size_t)f;
        bg = bf16_to_f32(a.gu_bias[row]);
        bu = bf16_to_f32(a.gu_bias[row + 1]);
      }
      const int act = sh ? MOE_ACT_SWIGLU : a.act;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int ti = 2 * c + q;
        if (ti < n) {
          const float gv = acc[q] + bg, uv = acc[2 + q] + bu;
          const float hv = act == MOE_ACT_SWIGLU ? act_swiglu(gv, uv) : act_clamped(gv, uv, a.limit, a.alpha);
          // h as a pair of bf16 (hi, lo = bf16(h - hi)), the layout the down kernels read
          const uint16_t hi = f32_to_bf16(hv);
          uint16_t* hr = a.h + (size_t)(r0 + ti) * 2 * a.ldh + f;
          hr[0] = hi;
          hr[a.ldh] = f32_to_bf16(hv - bf16_to_f32(hi));
        }
      }
    } else {
      const int o = kRows * t + 16 * tile + g;   // output rows o and o + 8
      float b0 = 0.f, b1 = 0.f;
      if (!sh && a.dn_bias) {
        if (o < a.R) b0 = bf16_to_f32(a.dn_bias[(size_t)v * a.R + o]);
        if (o + 8 < a.R) b1 = bf16_to_f32(a.dn_bias[(size_t)v * a.R + o + 8]);
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int ti = 2 * c + q;
        if (ti < n) {
          float* yrow = a.Y + (size_t)a.rs.row2slot[r0 + ti] * a.R;
          if (o < a.R) yrow[o] = acc[q] + b0;
          if (o + 8 < a.R) yrow[o + 8] = acc[2 + q] + b1;
        }
      }
    }
  }
  pdl_trigger();
}

template <bool GATEUP, int TILES>
void set_ring_smem(int bytes) {
  static int done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || done[dev] >= bytes) return;
  if (cudaFuncSetAttribute(ring_stream_kernel<GATEUP, TILES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bytes) == cudaSuccess)
    done[dev] = bytes;
}

// Ring depth that fits next to the fixed parts (0: it does not fit).
int ring_stages(int kin, bool pair) {
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const int fixed = ring_smem(kin, pair, 0).total + 1024 + 1024;   // + base alignment + static smem
  int st = (optin - fixed) / kStageBytes;
  if (st > kMaxRingStages) st = kMaxRingStages;
  return st >= 2 ? st : 0;
}

// bf16 matrix [rows, cols], boxes of box_rows x 64 elements with the 128-byte swizzle.
bool ring_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rows, cols, cols * 2, box_rows, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

// The maps (box rows 8 TILES) and the launch of one geometry.  GATEUP: gate / up
// (m0, m1; shared s0, s1); else down (m0; shared s0).
template <bool GATEUP, int TILES>
cudaError_t launch_ring(const ExpertParams& p, RingArgs a, int max_items, cudaStream_t s, bool* launched) {
  using G = Geo<TILES>;
  const int kmax = a.kin > a.kin_s ? a.kin : a.kin_s;
  a.stages = ring_stages(kmax, !GATEUP);
  if (!a.stages) return cudaSuccess;
  const int unit = GATEUP ? G::kRows / 2 : G::kRows;        // features (gate_up) or rows per unit
  a.tiles = ((a.R > a.Rs ? a.R : a.Rs) + unit - 1) / unit;
  CUtensorMap m0, m1, s0, s1;
  if (GATEUP) {
    if (!ring_map(&m0, p.gate, (uint64_t)p.E * p.ff, p.d, G::kBoxRows) ||
        !ring_map(&m1, p.up, (uint64_t)p.E * p.ff, p.d, G::kBoxRows))
      return cudaSuccess;
    s0 = m0;
    s1 = m1;
    if (p.sff && (!ring_map(&s0, p.sh_gate, (uint64_t)p.sff, p.d, G::kBoxRows) ||
                  !ring_map(&s1, p.sh_up, (uint64_t)p.sff, p.d, G::kBoxRows)))
      return cudaSuccess;
  } else {
    if (!ring_map(&m0, p.down, (uint64_t)p.E * p.d, p.ff, G::kBoxRows)) return cudaSuccess;
    s0 = m0;
    if (p.sff && !ring_map(&s0, p.sh_down, (uint64_t)p.d, p.sff, G::kBoxRows)) return cudaSuccess;
    m1 = m0;
    s1 = s0;
  }
  const int bytes = ring_smem(kmax, !GATEUP, a.stages).total + 1024;
  set_ring_smem<GATEUP, TILES>(bytes);
  const long long units = (long long)max_items * a.tiles;
  int grid = sm_count();
  if (units < grid) grid = (int)(units > 0 ? units : 1);
  *launched = true;
  return launch_pdl(ring_stream_kernel<GATEUP, TILES>, dim3(grid), dim3(kThreads), (size_t)bytes, s, m0, m1, s0,
                    s1, a);
}

// Units of 128 rows unless the expected work would give the CTAs fewer than four
// each; then units of 64 rows, so that the shares even out.
bool small_units(long long units128) { return units128 < 4LL * sm_count(); }

}  // namespace

cudaError_t ring_set_wait_test(uint32_t polls, int withhold) { return tc::set_wait_test(polls, withhold); }

cudaError_t launch_gateup_decode_ring(const ExpertParams& p, const RouteState& rs, const uint16_t* x, int K,
                                      uint16_t* h, int ldh, int max_items, int expect_items, cudaStream_t s,
                                      bool* launched) {
  *launched = false;
  RingArgs a{};
  a.rs = rs;
  a.E = p.E;
  a.R = p.ff;
  a.Rs = p.sff;
  a.kin = p.d;
  a.kin_s = p.d;
  a.gu_bias = p.gu_bias;
  a.x = x;
  a.K = K;
  a.h = h;
  a.ldh = ldh;
  a.act = p.act;
  a.limit = p.limit;
  a.alpha = p.alpha;
  const long long units128 = (long long)expect_items * (((p.ff > p.sff ? p.ff : p.sff) + 63) / 64);
  if (small_units(units128)) return launch_ring<true, 4>(p, a, max_items, s, launched);
  return launch_ring<true, 8>(p, a, max_items, s, launched);
}

cudaError_t launch_down_decode_ring(const ExpertParams& p, const RouteState& rs, const uint16_t* h, int ldh,
                                    float* Y, int max_items, int expect_items, cudaStream_t s, bool* launched) {
  *launched = false;
  RingArgs a{};
  a.rs = rs;
  a.E = p.E;
  a.R = p.d;
  a.Rs = p.d;
  a.kin = p.ff;
  a.kin_s = p.sff ? p.sff : p.ff;
  a.dn_bias = p.dn_bias;
  a.h = const_cast<uint16_t*>(h);
  a.ldh = ldh;
  a.Y = Y;
  const long long units128 = (long long)expect_items * ((p.d + 127) / 128);
  if (small_units(units128)) return launch_ring<false, 4>(p, a, max_items, s, launched);
  return launch_ring<false, 8>(p, a, max_items, s, launched);
}

}  // namespace moe
