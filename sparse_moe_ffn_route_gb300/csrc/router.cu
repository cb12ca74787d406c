// Router: logits on the tensor cores (warp-level bf16 MMA), then a warp per
// token for the top-k selection and the routing weights.
//
// Sources: "qwen35moe CPU-reference golden vectors", Kernel 4 (softmax over the
// 256 logits, selection sort with first-seen tie-break, norm_topk_prob times
// expert_weights_scale, sigmoid shared gate); "Phase 19: MoE - gpt-oss-20b",
// section 2 Router (logits + bias, top-k, softmax over the chosen k).
#include "common.cuh"
#include "internal.h"
#include "permute_core.cuh"

namespace moe {
namespace {

// Router logits kernel, one CTA per (16*MT tokens) x (8*NT experts) tile.  Its
// WARPS warps split the 32-wide k steps (warp w takes steps w, w+WARPS, ...) and
// each accumulates the whole tile, reusing every loaded fragment MT or NT times;
// the partial sums are then added in shared memory in a fixed order, so logits
// are bit-reproducible.  A warp issues the loads of up to STEPS of its k steps
// before its first MMA, which at decode sizes covers all of them.
//
// Operands go straight from global memory into MMA fragments: lane (g, c) loads
// the 16 bytes at k + 8c of its rows, and the two MMAs of a k step consume words
// {0,1} and {2,3} of those bytes (the same reordering of k on both operands, so
// the dot products are unchanged).
template <int MT, int NT, int WARPS, int STEPS>
__global__ void __launch_bounds__(WARPS * 32)
router_logits_kernel(const uint16_t* __restrict__ x, int T, int d, const uint16_t* __restrict__ w_r,
                     const uint16_t* __restrict__ bias, const uint16_t* __restrict__ wsh, int E,
                     float* __restrict__ logits, int ldl, int nsplit, size_t nstride,
                     uint32_t* __restrict__ status) {
  constexpr int TM = 16 * MT, TN = 8 * NT;
  __shared__ float part[WARPS][TM][TN + 1];
  pdl_wait();
  pdl_trigger();
  // the first kernel of a call: start a clean device status
  if (status && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) *status = 0u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int t0 = blockIdx.x * TM;
  const int e0 = blockIdx.y * TN;
  const int E1 = E + (wsh ? 1 : 0);

  const uint16_t* xr[MT][2];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int t = t0 + 16 * m + 8 * hh + g;
      xr[m][hh] = t < T ? x + (size_t)t * d : nullptr;
    }
  const uint16_t* wrow[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int e = e0 + 8 * n + g;
    wrow[n] = e < E ? w_r + (size_t)e * d : (e == E && wsh ? wsh : nullptr);
  }

  float acc[MT][NT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[m][n][q] = 0.f;
  const uint4 z = make_uint4(0, 0, 0, 0);
  // split-K: part blockIdx.z of nsplit takes the contiguous k steps [kb, nk)
  const int nk_all = d >> 5;
  const int kb = (int)((long long)nk_all * blockIdx.z / nsplit);
  const int nk = (int)((long long)nk_all * (blockIdx.z + 1) / nsplit);
  for (int s0 = kb + warp; s0 < nk; s0 += WARPS * STEPS) {
    uint4 A[STEPS][MT][2], B[STEPS][NT];
#pragma unroll
    for (int s = 0; s < STEPS; ++s) {
      const int ks = s0 + s * WARPS;
      const int o = ks * 32 + 8 * c;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) A[s][m][hh] = (ks < nk && xr[m][hh]) ? ldg_nc_v4(xr[m][hh] + o) : z;
#pragma unroll
      for (int n = 0; n < NT; ++n) B[s][n] = (ks < nk && wrow[n]) ? ldg_nc_v4(wrow[n] + o) : z;
    }
#pragma unroll
    for (int s = 0; s < STEPS; ++s)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const uint4 &a0 = A[s][m][0], &a1 = A[s][m][1], &b = B[s][n];
          mma_bf16_16816(acc[m][n], a0.x, a1.x, a0.y, a1.y, b.x, b.y);
          mma_bf16_16816(acc[m][n], a0.z, a1.z, a0.w, a1.w, b.z, b.w);
        }
  }
  // acc[m][n]: (token 16m+g, expert 8n+2c), (.., 8n+2c+1), (16m+g+8, 8n+2c), (.., 8n+2c+1)
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      part[warp][16 * m + g][8 * n + 2 * c] = acc[m][n][0];
      part[warp][16 * m + g][8 * n + 2 * c + 1] = acc[m][n][1];
      part[warp][16 * m + g + 8][8 * n + 2 * c] = acc[m][n][2];
      part[warp][16 * m + g + 8][8 * n + 2 * c + 1] = acc[m][n][3];
    }
  __syncthreads();
  for (int i = threadIdx.x; i < TM * TN; i += WARPS * 32) {
    const int tt = i / TN, ee = i % TN;
    const int t = t0 + tt, e = e0 + ee;
    if (t < T && e < E1) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) v += part[w][tt][ee];
      if (e < E && bias && blockIdx.z == 0) v += bf16_to_f32(bias[e]);
      logits[blockIdx.z * nstride + (size_t)t * ldl + e] = v;
    }
  }
}

constexpr int kSelectWarps = 8;

// Order-preserving unsigned key of a non-NaN logit: a > b exactly when key(a) >
// key(b), and -0 takes +0's key (they compare equal).  Key 0 (a NaN's) is below
// every logit and marks an absent or taken entry.
__device__ __forceinline__ uint32_t logit_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Warp per token.  Lane l holds logits l, l+32, ... (EPL per lane) and keeps the
// best untaken one among them.  Each of the k rounds takes the largest untaken
// logit, lowest index on equal values (the selection sort's first-seen rule): one
// warp max over the lanes' best keys, one warp min over the indices that reach it;
// the lane that gave up its entry then finds its next best.  Lane j keeps the j-th
// pick.  (NaN logits are outside the routing's contract.)
// The selection for token t by one warp (lane = its lane).
struct SelectArgs {
  const float* logits;
  int ldl, nsplit;
  size_t nstride;
  float* lsum;
  int ldsum, T, E, k, norm_topk_prob;
  float scale;
  int has_shared;
  int32_t* ids_out;
  float* w_out;
  float* sgate_out;
  int32_t* slot_expert;
  float* slot_w;
  const uint16_t* x;
  int d;
  const uint16_t* wsh;
};

// DOT: the shared-gate dot x_t . wsh may be asked for (else the gate is column E).
// sm_slots (shared memory, or null): the slots' experts also go there, for a grouping
// in the same block.
template <int EPL, bool DOT>
__device__ __forceinline__ void select_token(const SelectArgs& a, int t, int lane, int* sm_slots = nullptr) {
  const float* __restrict__ logits = a.logits;
  const int ldl = a.ldl, nsplit = a.nsplit;
  const size_t nstride = a.nstride;
  float* __restrict__ lsum = a.lsum;
  const int ldsum = a.ldsum, E = a.E, k = a.k, norm_topk_prob = a.norm_topk_prob;
  const float scale = a.scale;
  const int has_shared = a.has_shared;
  int32_t* __restrict__ ids_out = a.ids_out;
  float* __restrict__ w_out = a.w_out;
  float* __restrict__ sgate_out = a.sgate_out;
  int32_t* __restrict__ slot_expert = a.slot_expert;
  float* __restrict__ slot_w = a.slot_w;
  const uint16_t* __restrict__ x = a.x;
  const int d = a.d;
  const uint16_t* __restrict__ wsh = a.wsh;
  const float* row = logits + (size_t)t * ldl;
  float v[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : 0.f;
  }
  if (nsplit > 1) {
    // partial logits of the k parts, added in part order (three parts' loads at once)
    for (int p0 = 1; p0 < nsplit; p0 += 3) {
      float pv[3][EPL];
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const float* rp = row + (size_t)(p0 + q) * nstride;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const int e = lane + 32 * i;
          pv[q][i] = (p0 + q < nsplit && e < E) ? rp[e] : 0.f;
        }
      }
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        if (p0 + q >= nsplit) break;
#pragma unroll
        for (int i = 0; i < EPL; ++i) v[i] += pv[q][i];
      }
    }
  }
  if (lsum) {   // the logits themselves, when they were read from scratch
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) lsum[(size_t)t * ldsum + e] = v[i];
    }
  }
  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) key[i] = lane + 32 * i < E ? logit_key(v[i]) : 0u;
  // this lane's best: the largest key, the lowest slot i on equal keys
  uint32_t bk = 0u;
  int bi = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (key[i] > bk) {
      bk = key[i];
      bi = i;
    }
  int my_id = -1;
  float my_val = 0.f, top_val = 0.f;
  for (int j = 0; j < k; ++j) {
    const uint32_t gk = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t gi = __reduce_min_sync(0xffffffffu, bk == gk ? (uint32_t)(lane + 32 * bi) : 0xffffffffu);
    const float gv = key_logit(gk);
    if (lane == j) {
      my_id = (int)gi;
      my_val = gv;
    }
    if (j == 0) top_val = gv;   // the largest logit overall
    if ((int)(gi & 31u) == lane) {
      // this lane's entry gi >> 5 is taken: its next best
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == (int)(gi >> 5)) key[i] = 0u;
      bk = 0u;
      bi = 0;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (key[i] > bk) {
          bk = key[i];
          bi = i;
        }
    }
  }
  // Routing weights.  Renormalised softmax over the chosen k equals
  // exp(l_j - l_top) / sum_chosen exp(l_i - l_top) (the full softmax's
  // denominator cancels); this is also the gpt-oss softmax over the chosen k.
  float ex = (lane < k) ? expf(my_val - top_val) : 0.f;
  float den = ex;
  if (!norm_topk_prob) {   // plain softmax probability of each chosen expert
    den = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) den += expf(v[i] - top_val);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  const float w = ex / den * scale;
  const int K = k + has_shared;
  if (lane < k) {
    if (ids_out) ids_out[(size_t)t * k + lane] = my_id;
    if (w_out) w_out[(size_t)t * k + lane] = w;
    if (slot_expert) {
      slot_expert[(size_t)t * K + lane] = my_id;
      slot_w[(size_t)t * K + lane] = w;
    }
    if (sm_slots) sm_slots[t * K + lane] = my_id;
  }
  float sl = 0.f;   // the shared-gate logit: column E of the logits, or w_sh . x here
  if (DOT && has_shared && wsh) {
    // pieces i = lane, lane + 32, ... in order, eight pieces' loads in flight at once
    constexpr int kDotBatch = 8;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const uint4* wr = reinterpret_cast<const uint4*>(wsh);
    for (int i0 = 0; 32 * i0 < d / 8; i0 += kDotBatch) {
      uint4 xa[kDotBatch], wb[kDotBatch];
#pragma unroll
      for (int q = 0; q < kDotBatch; ++q) {
        const int i = lane + 32 * (i0 + q);
        xa[q] = wb[q] = make_uint4(0u, 0u, 0u, 0u);
        if (i < d / 8) {
          xa[q] = ldg_nc_v4(xr + i);
          wb[q] = ldg_nc_v4(wr + i);
        }
      }
#pragma unroll
      for (int q = 0; q < kDotBatch; ++q) {
        if (lane + 32 * (i0 + q) >= d / 8) break;
        const uint4 a = xa[q], b = wb[q];
        sl = fmaf(bf16_lo(a.x), bf16_lo(b.x), sl); sl = fmaf(bf16_hi(a.x), bf16_hi(b.x), sl);
        sl = fmaf(bf16_lo(a.y), bf16_lo(b.y), sl); sl = fmaf(bf16_hi(a.y), bf16_hi(b.y), sl);
        sl = fmaf(bf16_lo(a.z), bf16_lo(b.z), sl); sl = fmaf(bf16_hi(a.z), bf16_hi(b.z), sl);
        sl = fmaf(bf16_lo(a.w), bf16_lo(b.w), sl); sl = fmaf(bf16_hi(a.w), bf16_hi(b.w), sl);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sl += __shfl_xor_sync(0xffffffffu, sl, off);
  } else if (has_shared) {
    sl = row[E];
    for (int p = 1; p < nsplit; ++p) sl += row[(size_t)p * nstride + E];   // in part order
  }
  if (has_shared && lane == 0) {
    const float sg = 1.f / (1.f + expf(-sl));
    if (sgate_out) sgate_out[t] = sg;
    if (slot_expert) {
      slot_expert[(size_t)t * K + k] = E;
      slot_w[(size_t)t * K + k] = sg;
    }
    if (sm_slots) sm_slots[t * K + k] = E;
  }
}

template <int EPL>
__global__ void __launch_bounds__(kSelectWarps * 32) router_select_kernel(const SelectArgs a) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * kSelectWarps + (threadIdx.x >> 5);
  if (t < a.T) select_token<EPL, true>(a, t, threadIdx.x & 31);
}

// Decode sizes: the selection of every token (a warp per token, in turn) and then
// the grouping by expert in one CTA, one launch instead of two.
template <int EPL>
__global__ void __launch_bounds__(kPermuteThreads) select_permute_kernel(const SelectArgs a, RouteState rs,
                                                                         int S, int E1, int tpg) {
  __shared__ PermuteSmemT<256> sm;               // the fused kernel takes at most 256 experts
  __shared__ int slots[kPermuteOneCtaSlots];     // the slots' experts, for the grouping
  pdl_wait();
  pdl_trigger();
  for (int t = threadIdx.x >> 5; t < a.T; t += kPermuteThreads / 32)
    select_token<EPL, false>(a, t, threadIdx.x & 31, slots);
  __syncthreads();   // the slots are written: the grouping reads them from shared memory
  permute_block(rs, S, E1, tpg, sm, slots);
}

__global__ void ingest_routing_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w,
                                      const float* __restrict__ sgate, int T, int E, int k,
                                      int has_shared, int32_t* __restrict__ slot_expert,
                                      float* __restrict__ slot_w, uint32_t* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  // the first kernel of a call: start a clean device status
  if (status && blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;
  const int K = k + has_shared;
  const long n = (long)T * K;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long t = i / K;
    const int j = (int)(i - t * K);
    if (j < k) {
      // A routed id outside [0, E) becomes -1: the permute flags it and every
      // later kernel skips the slot (E itself would alias the shared expert).
      const int id = ids[t * k + j];
      slot_expert[i] = (id >= 0 && id < E) ? id : -1;
      if (slot_w) slot_w[i] = w[t * k + j];
    } else {
      slot_expert[i] = E;
      slot_w[i] = sgate[t];
    }
  }
}

}  // namespace

cudaError_t launch_router_logits(const uint16_t* x, int T, int d, const uint16_t* w_r,
                                 const uint16_t* bias, const uint16_t* wsh, int E, float* logits,
                                 int ldl, float* parts, size_t part_floats, int* nsplit, int* ppitch,
                                 uint32_t* status, bool* gate_in_logits, cudaStream_t s) {
  *gate_in_logits = wsh != nullptr;
  *nsplit = 1;
  *ppitch = 0;
  const int E1 = E + (wsh ? 1 : 0);
  if (T > 256 && router_gemm_supported(T, d, E)) {
    // a dense GEMM on tcgen05 over the routed experts; the shared-gate dot is left to
    // the select kernel
    *gate_in_logits = false;
    return launch_router_gemm(x, T, d, w_r, bias, E, logits, ldl, parts, part_floats, nsplit, ppitch, status,
                              s);
  }
  if (T <= 256) {
    // Latency-bound: many small CTAs, all loads of a warp in flight at once.  When the
    // (token, expert) tiles are too few to fill the SMs, d is split as well (parts of
    // at least 16 k steps of 32) and the select kernel adds the parts in order.
    dim3 grid((T + 15) / 16, (E1 + 15) / 16, 1);
    const int tiles = (int)(grid.x * grid.y);
    int ns = sm_count() / tiles;
    if (ns > (d >> 5) / 16) ns = (d >> 5) / 16;
    if (ns > 8) ns = 8;
    if (parts && ns > 1 && (size_t)ns * (size_t)T * (size_t)E1 <= part_floats) {
      grid.z = ns;
      *nsplit = ns;
      *ppitch = E1;
      return launch_pdl(router_logits_kernel<1, 2, 16, 6>, grid, dim3(16 * 32), 0, s, x, T, d, w_r,
                        bias, wsh, E, parts, E1, ns, (size_t)T * E1, status);
    }
    return launch_pdl(router_logits_kernel<1, 2, 16, 6>, grid, dim3(16 * 32), 0, s, x, T, d, w_r,
                      bias, wsh, E, logits, ldl, 1, (size_t)0, status);
  } else {          // throughput-bound: larger tiles, fewer re-reads of x and W_r from L2
    dim3 grid((T + 63) / 64, (E1 + 31) / 32);
    return launch_pdl(router_logits_kernel<4, 4, 4, 2>, grid, dim3(4 * 32), 0, s, x, T, d, w_r, bias,
                      wsh, E, logits, ldl, 1, (size_t)0, status);
  }
}

cudaError_t launch_router_select(const float* logits, int ldl, int nsplit, size_t nstride, float* lsum,
                                 int ldsum, int T, int E, int k, int norm_topk_prob, float scale,
                                 int has_shared,
                                 int32_t* ids_out, float* w_out, float* sgate_out,
                                 int32_t* slot_expert, float* slot_w, const uint16_t* x, int d,
                                 const uint16_t* wsh, const RouteState* rs, int S, int E1, int tpg,
                                 cudaStream_t s) {
  const SelectArgs a{logits, ldl, nsplit, nstride, lsum, ldsum, T, E, k, norm_topk_prob, scale, has_shared,
                     ids_out, w_out, sgate_out, slot_expert, slot_w, x, d, wsh};
  const int epl = (E + 31) / 32;
  // rs: also group the slots by expert in the same launch (one CTA); the shared gate
  // must then come as logit column E
  if (rs) {
    // at most 256 experts (the widths that fit the 64 registers of a 1024-thread CTA)
    if (wsh || S > kPermuteOneCtaSlots || epl > 8) return cudaErrorInvalidValue;
#define MOE_SELECT(N) \
  return launch_pdl(select_permute_kernel<N>, dim3(1), dim3(kPermuteThreads), 0, s, a, *rs, S, E1, tpg)
    if (epl <= 1) MOE_SELECT(1);
    else if (epl <= 4) MOE_SELECT(4);
    else MOE_SELECT(8);
#undef MOE_SELECT
  }
  dim3 grid((T + kSelectWarps - 1) / kSelectWarps);
#define MOE_SELECT(N) return launch_pdl(router_select_kernel<N>, grid, dim3(kSelectWarps * 32), 0, s, a)
  if (epl <= 1) MOE_SELECT(1);
  else if (epl <= 2) MOE_SELECT(2);
  else if (epl <= 4) MOE_SELECT(4);
  else if (epl <= 8) MOE_SELECT(8);
  else if (epl <= 16) MOE_SELECT(16);
  else MOE_SELECT(32);
#undef MOE_SELECT
  return cudaGetLastError();
}

cudaError_t launch_ingest_routing(const int32_t* ids, const float* w, const float* sgate, int T,
                                  int E, int k, int has_shared, int32_t* slot_expert,
                                  float* slot_w, uint32_t* status, cudaStream_t s) {
  const long n = (long)T * (k + has_shared);
  int blocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  if (blocks < 1) blocks = 1;   // (T = 0 still clears the status word)
  return launch_pdl(ingest_routing_kernel, dim3(blocks), dim3(256), 0, s, ids, w, sgate, T, E, k,
                    has_shared, slot_expert, slot_w, status);
}

}  // namespace moe
