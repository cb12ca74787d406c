// The one-CTA permute (up to 2048 slots: counts, offsets, work items and the
// permuted-row -> slot map) as a block routine, shared by the permute kernel and the
// decode path's select-and-permute kernel, with the block scan it uses.  See
// permute.cu for the method.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kPermuteThreads = 1024;
constexpr int kPermuteOneCtaSlots = 2048;   // the one-CTA routine's largest S

// Block-wide exclusive scan of two ints per element pair, two elements per thread.
__device__ __forceinline__ int2 block_exclusive_scan2(int2 val, int2* warp_tot, int2* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int2 inc = val;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int ox = __shfl_up_sync(0xffffffffu, inc.x, off);
    const int oy = __shfl_up_sync(0xffffffffu, inc.y, off);
    if (lane >= off) {
      inc.x += ox;
      inc.y += oy;
    }
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int2 w = warp_tot[lane];
    int2 wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int ox = __shfl_up_sync(0xffffffffu, wi.x, off);
      const int oy = __shfl_up_sync(0xffffffffu, wi.y, off);
      if (lane >= off) {
        wi.x += ox;
        wi.y += oy;
      }
    }
    warp_tot[lane] = make_int2(wi.x - w.x, wi.y - w.y);
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int2 base = warp_tot[warp];
  return make_int2(base.x + inc.x - val.x, base.y + inc.y - val.y);
}

// Stable placement of the slots [s0, s1) (at most 2048, in a block of 1024 threads):
// warp w takes the 64 slots s0 + 64 w .. s0 + 64 w + 63, as two groups of 32 in
// order.  A slot's row within its expert v's range is base[v] + (v's slots of the
// earlier warps) + (v's slots before it in its own warp), so every expert's rows hold
// its slots in increasing slot order, whatever order the warps run in.
// tab: [E1][32] bytes of shared memory, tab[v][w] = v's slots among warp w's 64.
// slots: the slots' experts (rs.slot_expert, or a shared-memory copy).
__device__ __forceinline__ void place_slots_stable(const RouteState& rs, int s0, int s1, int S, int E1,
                                                   const int* base, uint8_t* tab, const int* slots) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* tw = reinterpret_cast<uint32_t*>(tab);
  for (int i = tid; i < E1 * 8; i += kPermuteThreads) tw[i] = 0u;
  __syncthreads();
  int v[2], r[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int s = s0 + 64 * warp + 32 * hh + lane;
    int e = s < s1 ? slots[s] : -1;
    if (e < 0 || e >= E1) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int before = e >= 0 ? (int)tab[e * 32 + warp] : 0;   // v's slots in this warp's first group
    __syncwarp();
    if (e >= 0 && rank == 0) tab[e * 32 + warp] = (uint8_t)(before + __popc(peers));
    __syncwarp();
    v[hh] = e;
    r[hh] = before + rank;
  }
  __syncthreads();
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    if (v[hh] < 0) continue;
    // v's slots in warps 0 .. warp - 1: a sum of bytes, four per word
    const uint32_t* row = tw + v[hh] * 8;
    uint32_t pre = 0;
    for (int q = 0; q < (warp >> 2); ++q) pre = __dp4a(row[q], 0x01010101u, pre);
    if (warp & 3) pre = __dp4a(row[warp >> 2] & ((1u << (8 * (warp & 3))) - 1u), 0x01010101u, pre);
    const int rrow = base[v[hh]] + (int)pre + r[hh];
    if (rrow < S)
      rs.row2slot[rrow] = s0 + 64 * warp + 32 * hh + lane;
    else
      flag_status(rs.status, STATUS_ROW_OVERFLOW);
  }
}

// Shared memory of permute_block, for up to MAXE routed experts (plus the shared one).
template <int MAXE>
struct PermuteSmemT {
  int cnt[MAXE + 2];
  int cursor[MAXE + 2];
  int2 warp_tot[32];
  int2 total;
  __align__(16) uint8_t tab[(MAXE + 1) * 32];
};
using PermuteSmem = PermuteSmemT<kMaxExperts>;

// The whole grouping by one CTA of kPermuteThreads threads, S <= 2048 slots whose
// experts `slots` holds (rs.slot_expert written by an earlier kernel, or a copy in
// shared memory written before a block barrier).
template <class Smem>
__device__ __forceinline__ void permute_block(const RouteState& rs, int S, int E1, int tpg, Smem& sm,
                                              const int* slots) {
  int* cnt = sm.cnt;
  int* cursor = sm.cursor;
  int2* warp_tot = sm.warp_tot;
  const int tid = threadIdx.x;
  for (int v = tid; v < E1; v += kPermuteThreads) cnt[v] = 0;
  if (rs.fuse)
    for (int i = tid; i < rs.fuse_n; i += kPermuteThreads) rs.fuse[i] = 0;
  __syncthreads();

  for (int s = tid; s < S; s += kPermuteThreads) {
    const int v = slots[s];
    if (v >= 0 && v < E1)
      atomicAdd(&cnt[v], 1);
    else
      flag_status(rs.status, STATUS_BAD_EXPERT_ID);
  }
  __syncthreads();

  // Exclusive scan of (rows, work items) over the virtual experts.
  const int v0 = 2 * tid, v1 = 2 * tid + 1;
  const int c0 = v0 < E1 ? cnt[v0] : 0, c1 = v1 < E1 ? cnt[v1] : 0;
  const int i0 = (c0 + tpg - 1) / tpg, i1 = (c1 + tpg - 1) / tpg;
  const int2 ex = block_exclusive_scan2(make_int2(c0 + c1, i0 + i1), warp_tot, &sm.total);
  if (v0 < E1) {
    cursor[v0] = ex.x;
    rs.offsets[v0] = ex.x;
    rs.counts[v0] = c0;
    for (int j = 0; j < i0; ++j) rs.work[ex.y + j] = make_int2(v0, j * tpg);
  }
  if (v1 < E1) {
    cursor[v1] = ex.x + c0;
    rs.offsets[v1] = ex.x + c0;
    rs.counts[v1] = c1;
    for (int j = 0; j < i1; ++j) rs.work[ex.y + i0 + j] = make_int2(v1, j * tpg);
  }
  if (tid == 0) {
    rs.offsets[E1] = sm.total.x;
    *rs.n_work = sm.total.y;
  }
  __syncthreads();

  // Scatter, stable: every expert's rows take its slots in slot order.
  place_slots_stable(rs, 0, S, S, E1, cursor, sm.tab, slots);
}

}  // namespace moe
