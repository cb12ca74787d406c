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

// Shared memory of permute_block.
struct PermuteSmem {
  int cnt[2 * kPermuteThreads];
  int cursor[2 * kPermuteThreads];
  int2 warp_tot[32];
  int2 total;
};

// The whole grouping by one CTA of kPermuteThreads threads, S <= 2048 slots whose
// slot_expert the block can read (written before a block barrier, or by an earlier
// kernel).
__device__ __forceinline__ void permute_block(const RouteState& rs, int S, int E1, int tpg, PermuteSmem& sm) {
  int* cnt = sm.cnt;
  int* cursor = sm.cursor;
  int2* warp_tot = sm.warp_tot;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int v = tid; v < E1; v += kPermuteThreads) cnt[v] = 0;
  __syncthreads();

  for (int s = tid; s < S; s += kPermuteThreads) {
    const int v = rs.slot_expert[s];
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

  // Scatter: each warp ranks its 32 slots per expert and reserves a run of rows.
  for (int s0 = 0; s0 < S; s0 += kPermuteThreads) {
    const int s = s0 + tid;
    int v = s < S ? rs.slot_expert[s] : -1;
    if (v < 0 || v >= E1) v = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, v);
    const int leader = __ffs(peers) - 1;
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int base = 0;
    if (lane == leader && v >= 0) base = atomicAdd(&cursor[v], __popc(peers));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (v >= 0) {
      const int row = base + rank;
      if (row < S)
        rs.row2slot[row] = s;
      else
        flag_status(rs.status, STATUS_ROW_OVERFLOW);
    }
  }
}

}  // namespace moe
