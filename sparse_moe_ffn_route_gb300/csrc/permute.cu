// Group token slots by expert: histogram, exclusive scan, the work list of the
// expert kernels and the permuted-row -> slot map.  Up to 2048 slots: one CTA does
// it all in one launch.  More: three launches, per-chunk histograms (many CTAs),
// one scan (one CTA), and the scatter (many CTAs).
//
// Work items split each expert's rows into groups of at most `tpg` rows, so that
// an expert chosen by many tokens (the shared expert is chosen by all of them) is
// spread over many CTAs instead of one CTA making many passes over its weights.
//
// This is the "expert-grouped batching" that the qwen35moe forward-pass design
// ("Batched prefill", remaining levers) names as the way for tokens that share
// an expert to stream its weights once.
//
// The grouping is stable: expert v's rows hold the slots routed to v in increasing
// slot order (t k + j), so the grouped order, the work items and the tokens each
// item holds follow from the routing alone and are the same in every run.
#include "common.cuh"
#include "internal.h"
#include "permute_core.cuh"

namespace moe {
namespace {

// All of it in one CTA, for a single chunk of slots (decode sizes): one launch.
__global__ void __launch_bounds__(kPermuteThreads)
permute_one_cta_kernel(RouteState rs, int S, int E1, int tpg) {
  __shared__ PermuteSmem sm;
  pdl_wait();
  permute_block(rs, S, E1, tpg, sm, rs.slot_expert);
  pdl_trigger();
}

// The slots are split into chunks of kSlotsPerCta; chunk c is counted and later
// scattered by CTA c.  hist[c][v] = slots of chunk c routed to v.
constexpr int kSlotsPerCta = kPermuteOneCtaSlots;

// Rows of chunk c per virtual expert (shared-memory histogram).
__global__ void __launch_bounds__(kPermuteThreads)
perm_count_kernel(RouteState rs, int S, int E1, int* __restrict__ hist) {
  __shared__ int cnt[kMaxExperts + 1];
  const int tid = threadIdx.x;
  pdl_wait();
  for (int v = tid; v < E1; v += kPermuteThreads) cnt[v] = 0;
  __syncthreads();
  const int s0 = blockIdx.x * kSlotsPerCta, s1 = min(S, s0 + kSlotsPerCta);
  for (int s = s0 + tid; s < s1; s += kPermuteThreads) {
    const int v = rs.slot_expert[s];
    if (v >= 0 && v < E1)
      atomicAdd(&cnt[v], 1);
    else
      flag_status(rs.status, STATUS_BAD_EXPERT_ID);
  }
  __syncthreads();
  int* h = hist + (size_t)blockIdx.x * E1;
  for (int v = tid; v < E1; v += kPermuteThreads) h[v] = cnt[v];
  pdl_trigger();
}

// One CTA: hist[c][v] becomes the first row of chunk c within expert v's range (an
// exclusive scan over chunks), then counts, offsets and the work list as before.
__global__ void __launch_bounds__(kPermuteThreads)
perm_scan_kernel(RouteState rs, int E1, int tpg, int* __restrict__ hist, int nchunk) {
  __shared__ int tot[kMaxExperts + 1];
  __shared__ int2 warp_tot[32];
  __shared__ int2 total;
  const int tid = threadIdx.x;
  pdl_wait();
  for (int v = tid; v < E1; v += kPermuteThreads) {
    // chunks in groups of 8 whose loads are all in flight before the running sum
    int run = 0;
    for (int c0 = 0; c0 < nchunk; c0 += 8) {
      int n[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) n[j] = c0 + j < nchunk ? hist[(size_t)(c0 + j) * E1 + v] : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (c0 + j < nchunk) hist[(size_t)(c0 + j) * E1 + v] = run;
        run += n[j];
      }
    }
    tot[v] = run;
  }
  __syncthreads();
  // Exclusive scan of (rows, work items) over the virtual experts, two per thread.
  const int v0 = 2 * tid, v1 = 2 * tid + 1;
  const int c0 = v0 < E1 ? tot[v0] : 0, c1 = v1 < E1 ? tot[v1] : 0;
  const int i0 = (c0 + tpg - 1) / tpg, i1 = (c1 + tpg - 1) / tpg;
  const int2 ex = block_exclusive_scan2(make_int2(c0 + c1, i0 + i1), warp_tot, &total);
  if (v0 < E1) {
    rs.offsets[v0] = ex.x;
    rs.counts[v0] = c0;
    for (int j = 0; j < i0; ++j) rs.work[ex.y + j] = make_int2(v0, j * tpg);
  }
  if (v1 < E1) {
    rs.offsets[v1] = ex.x + c0;
    rs.counts[v1] = c1;
    for (int j = 0; j < i1; ++j) rs.work[ex.y + i0 + j] = make_int2(v1, j * tpg);
  }
  if (tid == 0) {
    rs.offsets[E1] = total.x;
    *rs.n_work = total.y;
  }
  pdl_trigger();
}

// Chunk c's slots to rows: offsets[v] + hist[c][v] + the slot's rank among chunk c's
// slots of v, in slot order (place_slots_stable).
__global__ void __launch_bounds__(kPermuteThreads)
perm_scatter_kernel(RouteState rs, int S, int E1, const int* __restrict__ hist) {
  __shared__ int cursor[kMaxExperts + 1];
  __shared__ __align__(16) uint8_t tab[(kMaxExperts + 1) * 32];
  const int tid = threadIdx.x;
  pdl_wait();
  const int* h = hist + (size_t)blockIdx.x * E1;
  for (int v = tid; v < E1; v += kPermuteThreads) cursor[v] = rs.offsets[v] + h[v];
  const int s0 = blockIdx.x * kSlotsPerCta, s1 = min(S, s0 + kSlotsPerCta);
  place_slots_stable(rs, s0, s1, S, E1, cursor, tab, rs.slot_expert);   // (its first barrier orders cursor)
  pdl_trigger();
}

}  // namespace

size_t permute_scratch_bytes(int S, int E1) {
  const size_t nchunk = (size_t)(S + kSlotsPerCta - 1) / kSlotsPerCta;
  return (nchunk > 0 ? nchunk : 1) * (size_t)E1 * sizeof(int);
}

cudaError_t launch_permute(const RouteState& rs, int S, int E1, int tpg, int* hist, cudaStream_t s) {
  const int nchunk = S > 0 ? (S + kSlotsPerCta - 1) / kSlotsPerCta : 1;
  if (nchunk == 1)
    return launch_pdl(permute_one_cta_kernel, dim3(1), dim3(kPermuteThreads), 0, s, rs, S, E1, tpg);
  cudaError_t e = launch_pdl(perm_count_kernel, dim3(nchunk), dim3(kPermuteThreads), 0, s, rs, S, E1, hist);
  if (e != cudaSuccess) return e;
  e = launch_pdl(perm_scan_kernel, dim3(1), dim3(kPermuteThreads), 0, s, rs, E1, tpg, hist, nchunk);
  if (e != cudaSuccess) return e;
  return launch_pdl(perm_scatter_kernel, dim3(nchunk), dim3(kPermuteThreads), 0, s, rs, S, E1,
                    static_cast<const int*>(hist));
}

}  // namespace moe
