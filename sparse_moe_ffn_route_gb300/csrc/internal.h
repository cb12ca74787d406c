// Internal contract between the C-ABI host code (moe_abi.cu) and the kernel
// translation units: parameter blocks and launcher declarations.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// Launch with programmatic stream serialization: the kernel may begin launching
// while its predecessor on the stream finishes; it calls pdl_wait() before reading
// anything the predecessor wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Bits of the device status word kept at the start of the workspace.
enum : uint32_t {
  STATUS_BAD_EXPERT_ID = 1u << 0,   // a routing id outside [0, E) was seen and skipped
  STATUS_ROW_OVERFLOW = 1u << 1,    // a row index fell outside the permuted-row range
  STATUS_TILE_OVERFLOW = 1u << 2,   // the prefill tile list would exceed its capacity
  STATUS_TIMEOUT = 1u << 8,         // a bounded wait on an mbarrier gave up
};

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;

// Expert weights as the kernels see them.  Virtual expert index v in [0, E) is a
// routed expert; v == E is the shared expert (bf16, separate gate/up, SwiGLU).
struct ExpertParams {
  // routed experts
  const uint16_t* gate;       // bf16 [E, ff, d]            (separate layout)
  const uint16_t* up;         // bf16 [E, ff, d]            (separate layout)
  const uint8_t* gate_up;     // bf16 [E, 2ff, d] or MXFP4 blocks [E, 2ff, d/32, 16]
  const uint8_t* gu_scales;   // MXFP4 [E, 2ff, d/32]
  const uint16_t* gu_bias;    // bf16 [E, 2ff] or null
  const uint8_t* down;        // bf16 [E, d, ff] or MXFP4 blocks [E, d, ff/32, 16]
  const uint8_t* dn_scales;   // MXFP4 [E, d, ff/32]
  const uint16_t* dn_bias;    // bf16 [E, d] or null
  // shared expert
  const uint16_t* sh_gate;    // bf16 [sff, d]
  const uint16_t* sh_up;      // bf16 [sff, d]
  const uint16_t* sh_down;    // bf16 [d, sff]
  int E, d, ff, sff;
  int act;                    // MOE_ACT_* of routed experts
  float limit, alpha;
};

// Routing state in the workspace.  S = T * K slots, K = k + (shared ? 1 : 0);
// slot t*K + j is token t's j-th expert (j == k: the shared expert, id E).
struct RouteState {
  int32_t* slot_expert;  // [S]
  float* slot_w;         // [S]
  int32_t* counts;       // [E1]
  int32_t* offsets;      // [E1 + 1]  permuted-row ranges per virtual expert
  int2* work;            // [E1 + S]  work items (virtual expert, first row within it); each
                         //           covers up to `tpg` of that expert's rows
  int32_t* n_work;       // [1]
  int32_t* row2slot;     // [S]       permuted row -> slot
  uint32_t* status;      // device status word
  // [fuse_n] per-call counters that the one-CTA grouping zeroes: for the fused decode
  // launch a ticket counter and one count of finished gate_up units per work item,
  // then hmax.  Null where the layout has none.
  int32_t* fuse = nullptr;
  int fuse_n = 0;
  // [S], the last S entries of fuse: per permuted row, the largest |hi| of its h row
  // (bf16 bits), gathered by the MXFP4 decode ring's gate_up epilogue for its down
  // staging.  Null unless the one-CTA grouping zeroes it (S <= 2048).
  uint32_t* hmax = nullptr;
};

// ---------------------------------------------------------------- host helpers
// 2D TMA map over a row-major matrix [rows, cols] of `type` (row stride in bytes)
// with a box of box_rows x box_cols elements; false if the driver rejects it.
bool make_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t rows,
              uint64_t cols, uint64_t stride, uint32_t box_rows, uint32_t box_cols,
              CUtensorMapSwizzle swz);
int sm_count();   // SMs of the current device

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.

// MXFP4 decode with one-chunk work items (at most 8 rows each): the asynchronous
// weight-stream kernels.  *launched is false (and nothing is enqueued) when the
// shapes or alignments do not suit them; the caller then uses the register-stream
// kernels below.
cudaError_t launch_gateup_decode_fp4(const ExpertParams& p, const RouteState& rs, const uint16_t* x, int K,
                                     uint16_t* h, int ldh, int max_items, cudaStream_t s, bool* launched);
cudaError_t launch_down_decode_fp4(const ExpertParams& p, const RouteState& rs, const uint16_t* h, int ldh,
                                   float* Y, int max_items, cudaStream_t s, bool* launched);

// logits[t, e] (row stride ldl) = x_t . W_r[e] (+ bias[e]) for e < E, and, when
// *gate_in_logits comes back true, x_t . wsh for e == E (else the select kernel
// computes that dot itself).  The first kernel of a call: it clears *status.
// With many tokens the logits may come back in `parts` (part_floats floats of
// scratch): when *ppitch > 0, as *nsplit partial sums at parts + i * T * *ppitch
// (row pitch *ppitch), which the select kernel adds in order; else in logits.
cudaError_t launch_router_logits(const uint16_t* x, int T, int d, const uint16_t* w_r,
                                 const uint16_t* bias, const uint16_t* wsh, int E, float* logits,
                                 int ldl, float* parts, size_t part_floats, int* nsplit, int* ppitch,
                                 uint32_t* status, bool* gate_in_logits, cudaStream_t s);
// Router logits of many tokens as a dense tcgen05 GEMM (expert_prefill.cu).
bool router_gemm_supported(int T, int d, int E);
cudaError_t launch_router_gemm(const uint16_t* x, int T, int d, const uint16_t* w_r, const uint16_t* bias,
                               int E, float* logits, int ldl, float* parts, size_t part_floats, int* nsplit,
                               int* ppitch, uint32_t* status, cudaStream_t s);

// Top-k + routing weights from logits [T, ldl] (first E columns), given as nsplit
// partial sums nstride floats apart that are added in order (lsum [T, ldsum], when
// non-null, receives the sums).  With has_shared, the shared-gate logit is column
// E, or, when wsh is non-null, x_t . wsh computed here (x bf16 [T, d]).  Writes any
// non-null output.  rs non-null (S = T * K <= 2048 slots, E1 virtual experts, work
// items of tpg rows): the same launch then groups the slots by expert, in place of
// launch_permute.
cudaError_t launch_router_select(const float* logits, int ldl, int nsplit, size_t nstride, float* lsum,
                                 int ldsum, int T, int E, int k, int norm_topk_prob, float scale,
                                 int has_shared,
                                 int32_t* ids_out, float* w_out, float* sgate_out,
                                 int32_t* slot_expert, float* slot_w, const uint16_t* x, int d,
                                 const uint16_t* wsh, const RouteState* rs, int S, int E1, int tpg,
                                 cudaStream_t s);

// Copy caller routing into the slot arrays (routed entry point).
cudaError_t launch_ingest_routing(const int32_t* ids, const float* w, const float* sgate, int T,
                                  int E, int k, int has_shared, int32_t* slot_expert,
                                  float* slot_w, uint32_t* status, cudaStream_t s);

// Histogram, offsets, work list (items of up to tpg rows) and row -> slot map; hist is
// scratch of permute_scratch_bytes(S, E1).
size_t permute_scratch_bytes(int S, int E1);
cudaError_t launch_permute(const RouteState& rs, int S, int E1, int tpg, int* hist, cudaStream_t s);

// Decode path: weight-streaming grouped matvec on mma.sync.  One CTA row per work
// item; chunks = token chunks of 8 per item (1 or 4, so tpg = 8 * chunks);
// max_items bounds the work list (grid size).
cudaError_t launch_gateup_decode(const ExpertParams& p, int wfmt, int interleaved,
                                 const RouteState& rs, const uint16_t* x, int K, uint16_t* h,
                                 int ldh, int max_items, int chunks, cudaStream_t s);
cudaError_t launch_down_decode(const ExpertParams& p, int wfmt, const RouteState& rs,
                               const uint16_t* h, int ldh, float* Y, int max_items, int chunks,
                               cudaStream_t s);
// Both of the above in one launch, for bf16 weights and one-chunk items whose token
// rows fit the staging copy, when rs carries the fused counters (zeroed by the one-CTA
// grouping that precedes it); *launched comes back false (nothing enqueued) otherwise.
cudaError_t launch_experts_decode_fused(const ExpertParams& p, const RouteState& rs, const uint16_t* x, int K,
                                       uint16_t* h, int ldh, float* Y, int max_items, int interleaved,
                                       cudaStream_t s, bool* launched);
// Whether the fused launch's staged rows fit for these sizes (host).
bool decode_fused_fits(int d, int ff, int sff);

// Decode path, bf16 weights in the separate gate / up layout (d, ff, sff multiples
// of 64), one-chunk items (at most 8 token rows): the weights stream through a
// TMA-fed shared-memory ring (expert_decode_ring.cu).  *launched comes back false
// when the ring does not fit the device (the caller then runs the kernels above).
// expect_items: the expected number of work items (the unit size follows from it).
cudaError_t launch_gateup_decode_ring(const ExpertParams& p, const RouteState& rs, const uint16_t* x, int K,
                                      uint16_t* h, int ldh, int max_items, int expect_items, cudaStream_t s,
                                      bool* launched);
cudaError_t launch_down_decode_ring(const ExpertParams& p, const RouteState& rs, const uint16_t* h, int ldh,
                                    float* Y, int max_items, int expect_items, cudaStream_t s, bool* launched);

// Prefill path: grouped GEMMs on tcgen05 (see expert_prefill.cu).  The work list
// must hold 128-row m tiles (permute with tpg = 128).
bool prefill_supported(int d, int ff, int sff, int wfmt, int interleaved);
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* row2slot, int S, int K, int d,
                               uint16_t* xp, cudaStream_t s);
// MXFP4: bytes of the transposed-scale scratch, and the kernel that fills it.
size_t prefill_scales_bytes(const ExpertParams& p, int wfmt);
cudaError_t launch_transpose_scales(const ExpertParams& p, uint8_t* scratch, cudaStream_t s);
// gate_up over the grouped rows: A rows come from xp (the gathered x rows, MXFP4
// weights) or, with bf16 weights, straight from x [T, d] by row index (grouped row r
// is token row2slot[r] / K), so that no gathered copy is needed.
// yzero non-null: the kernel's epilogue warps also clear yzero [yzero_floats] fp32 (the
// per-token sums the accumulated down projection adds into), before their first tile.
cudaError_t launch_gateup_prefill(const ExpertParams& p, int wfmt, int interleaved,
                                  const RouteState& rs, const uint16_t* xp, int S, const uint16_t* x, int T,
                                  int K, uint16_t* h, int ldh, const uint8_t* scalesT, int max_mtiles,
                                  float* yzero, size_t yzero_floats, cudaStream_t s);
// yacc non-null: instead of the Y rows, yacc[t] += slot_w * (row + bias) for slot
// t * K + j, by atomic adds (yacc [T, d] fp32, zeroed before the call's down step).
cudaError_t launch_down_prefill(const ExpertParams& p, int wfmt, const RouteState& rs,
                                const uint16_t* h, int ldh, int S, float* Y, float* yacc, int K,
                                const uint8_t* scalesT, int max_mtiles, cudaStream_t s);

// f16 token operands (stage_f16.cu).  Per grouped row: rowmul = 2^-e of the staged
// x row, hmax = largest |h| (fp32 bits, accumulated by the gate_up epilogue), hmul =
// 2^-e of the staged h row.
// The grouped GEMMs of expert_prefill_fp4.cu claim their units from a counter
// (sched[0] gate_up, sched[1] down) in the item order `order` [work items].
struct Fp4Rows {
  float* rowmul;
  uint32_t* hmax;
  float* hmul;
  int32_t* order;
  int32_t* sched;
};
// x rows of the grouped order as f16 times 2^e per row (largest magnitude in
// [2^14, 2^15)), rowmul[r] = 2^-e; clears hmax[r] when hmax is non-null.  When
// order is non-null it also writes the GEMMs' item order (items of more than
// half_rows rows first, in the work list's order, then the others) and clears the
// two unit counters sched[0..1].
cudaError_t launch_gather_rows_f16(const uint16_t* x, const int32_t* row2slot, int S, int K, int d, uint16_t* xp16,
                                   float* rowmul, uint32_t* hmax, const RouteState& rs, int half_rows,
                                   int32_t* order, int32_t* sched, cudaStream_t s);
// h rows staged by the gate_up epilogue as f16 times 2^kh: hmul[r] = 2^-kh, except
// rows whose largest |h| (hmax) is below 2^(-2 - kh), which are re-staged from their
// fp32 copy (hside [S, ldh]) with their own power of two.
cudaError_t launch_h_fix_f16(const float* hside, const uint32_t* hmax, int S, int ff, int kh, uint16_t* h16,
                             int ldh, float* hmul, cudaStream_t s);
// kh of the f16 h staging: the clamped GLU's bound on |h| times 2^kh stays below 2^15.
int h_stage_exp(float limit, float alpha);

// Prefill path for MXFP4 experts with the clamped GLU (expert_prefill_fp4.cu): f16
// operands, weights decoded once per two m tiles.  The work list must hold items of
// up to 256 rows (permute with tpg = 256).  Scratch (prefill_fp4_scratch_bytes):
// per weight row shifts and multipliers, and the per grouped row arrays.
bool prefill_fp4_supported(const ExpertParams& p, int wfmt, int interleaved);
size_t prefill_fp4_scratch_bytes(const ExpertParams& p, int S);
Fp4Rows prefill_fp4_rows(const ExpertParams& p, uint8_t* scratch, int S);
cudaError_t launch_prefill_fp4_prep(const ExpertParams& p, uint8_t* scratch, int S, cudaStream_t s);
cudaError_t launch_gateup_prefill_fp4(const ExpertParams& p, const RouteState& rs, const uint16_t* xp16, int S,
                                      uint16_t* h16, float* hside, int ldh, int kh, uint8_t* scratch,
                                      int max_items, float* yzero, size_t yzero_floats, cudaStream_t s);
// yacc non-null: as for launch_down_prefill.
cudaError_t launch_down_prefill_fp4(const ExpertParams& p, const RouteState& rs, const uint16_t* h16, int ldh16,
                                    int S, float* Y, float* yacc, int K, uint8_t* scratch, int max_items,
                                    cudaStream_t s);

// The bounded-wait limits of each translation unit with TMA-fed kernels (see
// tc::WaitTest): the poll limit, and whether CTA 0's producer withholds its first load
// (the grouped GEMMs of expert_prefill.cu and the MXFP4 decode ring read it).
cudaError_t prefill_set_wait_test(uint32_t polls, int withhold);
cudaError_t decode_set_wait_test(uint32_t polls, int withhold);
cudaError_t prefill_fp4_set_wait_test(uint32_t polls, int withhold);
cudaError_t ring_set_wait_test(uint32_t polls, int withhold);
cudaError_t fp4_stream_set_wait_test(uint32_t polls, int withhold);

// MXFP4 [rows, n_in/32, 16] + scales -> bf16 [rows, n_in].
cudaError_t launch_mxfp4_to_bf16(const uint8_t* blocks, const uint8_t* scales, long long rows,
                                 int n_in, uint16_t* out, cudaStream_t s);

// y[t] = (resid[t] +) yacc[t] (bf16 or fp32 out): the end of the accumulated prefill.
cudaError_t launch_finish_accumulated(const float* yacc, int T, int d, const uint16_t* resid, void* y,
                                      bool y_fp32, cudaStream_t s);
// y[t] = (resid[t] +) sum_j slot_w[t,j] * Y[t*K + j]  (fp32 accumulation; bf16 or fp32 out).
cudaError_t launch_combine(const float* Y, const float* slot_w, const int32_t* slot_expert, int T,
                           int K, int d, int E1, const uint16_t* resid, void* y, bool y_fp32,
                           cudaStream_t s);
// xn = bf16(x * w / sqrt(mean(x^2) + eps)) per token row; clears *status (the first
// kernel of a call that normalises).
cudaError_t launch_rmsnorm(const uint16_t* x, int T, int d, const uint16_t* w, float eps, uint16_t* xn,
                           uint32_t* status, cudaStream_t s);

}  // namespace moe
