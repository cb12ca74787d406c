// C-ABI host layer of libmoe.so: argument validation, workspace carving and the
// stream-ordered launch sequence of each entry point (see include/moe.h).
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "permute_core.cuh"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
constexpr int kDecodeTokensPerExpert = 16;   // AUTO: decode path below this mean load

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Layout {
  int K, E1, S, ldl, ldh;
  bool prefill;             // the expert phase runs the tcgen05 grouped GEMMs
  bool prefill_fp4;         // ... in their f16-operand MXFP4 form (expert_prefill_fp4.cu)
  bool accumulate;          // prefill, not deterministic: down adds w * Y into yacc with atomics
  size_t status, counts, offsets, work, n_work, slot_expert, slot_w, row2slot, hist, logits, h, Y, xn,
      xp, scalesT, xstage, ystage, yacc, fuse, total;
  int fuse_n;               // decode: counters of the fused expert launch (ticket + one per work item)
};

int path_for(const moe_cfg_t* c, int T);

int validate_cfg(const moe_cfg_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->d_model <= 0 || c->n_experts < 1 || c->n_experts > kMaxExperts || c->top_k < 1 ||
      c->top_k > c->n_experts || c->top_k > kMaxTopK || c->expert_ff <= 0 || c->shared_ff < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->gating < 0 || c->gating > 1 || c->act < 0 || c->act > 1 || c->wfmt < 0 || c->wfmt > 1 ||
      c->interleaved_gate_up < 0 || c->interleaved_gate_up > 1 || c->norm_topk_prob < 0 ||
      c->norm_topk_prob > 1 || c->path < 0 || c->path > MOE_PATH_DECODE_REGISTERS || c->y_fp32 < 0 || c->y_fp32 > 1)
    return MOE_ERR_INVALID_ARG;
  for (int r : c->reserved)
    if (r != 0) return MOE_ERR_INVALID_ARG;
  if (c->rms_norm < 0 || c->rms_norm > 1 || c->residual < 0 || c->residual > 1 || c->deterministic < 0 ||
      c->deterministic > 1 ||
      !std::isfinite(c->rms_eps) || c->rms_eps < 0.f)
    return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->expert_weights_scale) || !std::isfinite(c->glu_limit) ||
      !std::isfinite(c->glu_alpha))
    return MOE_ERR_INVALID_ARG;
  if (c->d_model % 32 || c->expert_ff % 32 || c->shared_ff % 32) return MOE_ERR_UNSUPPORTED;
  if (c->wfmt == MOE_WFMT_MXFP4 && (!c->interleaved_gate_up || c->shared_ff > 0))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool make_layout(const moe_cfg_t* c, int T, Layout* L) {
  const int has_sh = c->shared_ff > 0;
  L->K = c->top_k + has_sh;
  L->E1 = c->n_experts + has_sh;
  const long long S = (long long)T * L->K;
  if (T < 0 || S > (1LL << 30)) return false;
  L->S = (int)S;
  L->ldl = L->E1;
  L->ldh = c->expert_ff > c->shared_ff ? c->expert_ff : c->shared_ff;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  const size_t Tz = (size_t)T, Sz = (size_t)S, d = (size_t)c->d_model;
  L->status = take(64);
  L->counts = take(4 * (size_t)L->E1);
  L->offsets = take(4 * ((size_t)L->E1 + 1));
  L->work = take(8 * ((size_t)L->E1 + Sz));
  L->n_work = take(4);
  L->slot_expert = take(4 * Sz);
  L->slot_w = take(4 * Sz);
  L->row2slot = take(4 * Sz);
  L->hist = take(permute_scratch_bytes(L->S, L->E1));
  L->logits = take(4 * Tz * (size_t)L->ldl);
  L->h = take(4 * Sz * (size_t)L->ldh);   // (hi, lo) bf16 halves
  L->Y = take(4 * Sz * (d > (size_t)L->ldh ? d : (size_t)L->ldh));   // also h's fp32 side copies
  L->prefill = path_for(c, T) == MOE_PATH_PREFILL &&
               prefill_supported(c->d_model, c->expert_ff, c->shared_ff, c->wfmt,
                                 c->interleaved_gate_up);
  L->xp = take(L->prefill && c->wfmt == MOE_WFMT_MXFP4 ? 2 * Sz * d : 0);   // gathered x rows (MXFP4)
  {
    ExpertParams sp{};
    sp.E = c->n_experts;
    sp.d = c->d_model;
    sp.ff = c->expert_ff;
    sp.sff = c->shared_ff;
    sp.act = c->act;
    sp.limit = c->glu_limit;
    sp.alpha = c->glu_alpha;
    L->prefill_fp4 = L->prefill && prefill_fp4_supported(sp, c->wfmt, c->interleaved_gate_up);
    L->scalesT = take(!L->prefill      ? 0
                      : L->prefill_fp4 ? prefill_fp4_scratch_bytes(sp, L->S)
                                       : prefill_scales_bytes(sp, c->wfmt));
  }
  L->accumulate = L->prefill && !c->deterministic;
  // a ticket counter and one count per one-chunk work item (at most E1 + S / 8 items),
  // then the largest |hi| of each permuted row's h
  L->fuse_n = L->prefill ? 0 : 1 + L->E1 + (int)((S + 7) / 8) + (int)S;
  L->fuse = take(4 * (size_t)L->fuse_n);
  L->yacc = take(L->accumulate ? 4 * Tz * d : 0);   // per-token fp32 sums of the weighted expert outputs
  L->xn = take(c->rms_norm ? 2 * Tz * d : 0);   // RMSNorm(x), the MoE's input
  L->xstage = take(2 * Tz * d);
  L->ystage = take(4 * Tz * d);
  L->total = off;
  return true;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

RouteState route_state(void* ws, const Layout& L) {
  RouteState rs;
  rs.slot_expert = at<int32_t>(ws, L.slot_expert);
  rs.slot_w = at<float>(ws, L.slot_w);
  rs.counts = at<int32_t>(ws, L.counts);
  rs.offsets = at<int32_t>(ws, L.offsets);
  rs.work = at<int2>(ws, L.work);
  rs.n_work = at<int32_t>(ws, L.n_work);
  rs.row2slot = at<int32_t>(ws, L.row2slot);
  rs.status = at<uint32_t>(ws, L.status);
  rs.fuse = L.fuse_n ? at<int32_t>(ws, L.fuse) : nullptr;
  rs.fuse_n = L.fuse_n;
  rs.hmax = L.fuse_n && L.S <= kPermuteOneCtaSlots ? reinterpret_cast<uint32_t*>(rs.fuse + L.fuse_n - L.S) : nullptr;
  return rs;
}

int check_ws(const moe_cfg_t* c, int T, void* ws, size_t ws_bytes, Layout* L) {
  if (!make_layout(c, T, L)) return MOE_ERR_UNSUPPORTED;
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < L->total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// Pointer checks for the expert and shared weights of cfg.
int check_experts(const moe_cfg_t* c, const moe_experts_t* e, const moe_shared_t* sh) {
  if (!e) return MOE_ERR_INVALID_ARG;
  const void* need[4] = {nullptr, nullptr, nullptr, nullptr};
  if (c->wfmt == MOE_WFMT_MXFP4) {
    need[0] = e->gate_up; need[1] = e->gate_up_scales; need[2] = e->down; need[3] = e->down_scales;
    for (const void* p : need)
      if (!p) return MOE_ERR_INVALID_ARG;
  } else if (c->interleaved_gate_up) {
    if (!e->gate_up || !e->down) return MOE_ERR_INVALID_ARG;
  } else {
    if (!e->gate || !e->up || !e->down) return MOE_ERR_INVALID_ARG;
    if (e->gate_up_bias) return MOE_ERR_UNSUPPORTED;   // bias is defined in gate_up row order
  }
  const void* all[8] = {e->gate, e->up, e->gate_up, e->gate_up_scales, e->gate_up_bias, e->down,
                        e->down_scales, e->down_bias};
  for (const void* p : all)
    if (p && !aligned16(p)) return MOE_ERR_ALIGNMENT;
  if (c->shared_ff > 0) {
    if (!sh || !sh->gate || !sh->up || !sh->down || !sh->gate_inp) return MOE_ERR_INVALID_ARG;
    const void* s4[4] = {sh->gate, sh->up, sh->down, sh->gate_inp};
    for (const void* p : s4)
      if (!aligned16(p)) return MOE_ERR_ALIGNMENT;
  }
  return MOE_OK;
}

int check_router(const moe_cfg_t* c, const moe_router_t* r) {
  if (!r || !r->w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(r->w) || (r->bias && !aligned16(r->bias))) return MOE_ERR_ALIGNMENT;
  if (c->rms_norm) {
    if (!r->norm_w) return MOE_ERR_INVALID_ARG;
    if (!aligned16(r->norm_w)) return MOE_ERR_ALIGNMENT;
  }
  return MOE_OK;
}

ExpertParams expert_params(const moe_cfg_t* c, const moe_experts_t* e, const moe_shared_t* sh) {
  ExpertParams p;
  std::memset(&p, 0, sizeof(p));
  p.gate = static_cast<const uint16_t*>(e->gate);
  p.up = static_cast<const uint16_t*>(e->up);
  p.gate_up = static_cast<const uint8_t*>(e->gate_up);
  p.gu_scales = static_cast<const uint8_t*>(e->gate_up_scales);
  p.gu_bias = static_cast<const uint16_t*>(e->gate_up_bias);
  p.down = static_cast<const uint8_t*>(e->down);
  p.dn_scales = static_cast<const uint8_t*>(e->down_scales);
  p.dn_bias = static_cast<const uint16_t*>(e->down_bias);
  if (c->shared_ff > 0) {
    p.sh_gate = static_cast<const uint16_t*>(sh->gate);
    p.sh_up = static_cast<const uint16_t*>(sh->up);
    p.sh_down = static_cast<const uint16_t*>(sh->down);
  }
  p.E = c->n_experts;
  p.d = c->d_model;
  p.ff = c->expert_ff;
  p.sff = c->shared_ff;
  p.act = c->act;
  p.limit = c->glu_limit;
  p.alpha = c->glu_alpha;
  return p;
}

int path_for(const moe_cfg_t* c, int T) {
  if (c->path != MOE_PATH_AUTO) return c->path;
  return (long long)T * c->top_k < (long long)kDecodeTokensPerExpert * c->n_experts
             ? MOE_PATH_DECODE
             : MOE_PATH_PREFILL;
}

// Decode path: token chunks of 8 per work item, one while experts average at most 4
// tokens, else four.
int decode_chunks(const moe_cfg_t* c, int T) {
  return 4LL * T * c->top_k <= 16LL * c->n_experts ? 1 : 4;
}

// Decode path, expected work items for T tokens: the distinct routed experts (at most
// T k or E), plus the shared expert's items of 8 rows.
int expect_items(const moe_cfg_t* c, int T) {
  const long long tk = (long long)T * c->top_k;
  return (int)(tk < c->n_experts ? tk : c->n_experts) + (c->shared_ff > 0 ? (T + 7) / 8 : 0);
}

// Decode path: one-chunk items take the TMA-fed ring kernels (which fall back to the
// register-stream ones only if the device lacks the shared memory they need): MXFP4
// weights; bf16 weights in the separate gate / up layout with d, ff, sff multiples
// of 64 while the down projection has fewer than kRingUnits units of 128 rows (16
// per SM of a 152-SM GB300).  Past that the register-stream kernels, in their
// one-launch form, are faster (Qwen3.5-mini T=64: 0.234 against 0.244 ms a step with
// the ring); below it the two are level (T=8: 0.0915 against 0.0909 ms).
constexpr long long kRingUnits = 16LL * 152;
bool decode_ring(const moe_cfg_t* c, int T) {
  if (c->path == MOE_PATH_DECODE_REGISTERS) return false;
  if (c->wfmt == MOE_WFMT_MXFP4) return true;
  return c->wfmt == MOE_WFMT_BF16 && !c->interleaved_gate_up && c->d_model % 64 == 0 &&
         c->expert_ff % 64 == 0 && c->shared_ff % 64 == 0 &&
         (long long)expect_items(c, T) * ((c->d_model + 127) / 128) < kRingUnits;
}

// Decode, bf16 weights, one-chunk items on the register-stream kernels (not the
// ring): gate_up and down run as one launch when the one-CTA grouping, which zeroes
// the launch's counters, precedes it and the staged rows fit.  The two-launch form
// stays for moe_test_set_decode_fusion(0).
bool g_decode_fusion = true;
bool decode_fused(const moe_cfg_t* c, const Layout& L, int T) {
  return g_decode_fusion && !L.prefill && c->wfmt == MOE_WFMT_BF16 && decode_chunks(c, T) == 1 &&
         !decode_ring(c, T) && L.S <= kPermuteOneCtaSlots &&
         decode_fused_fits(c->d_model, c->expert_ff, c->shared_ff);
}

// Caller-owned events recorded at phase boundaries (moe_set_phase_events).
// With two events only the start ([0]) and the end ([6]) of the call are recorded,
// which leaves consecutive kernels free to overlap their launches.
thread_local void* const* g_phase_events = nullptr;
thread_local int g_phase_n = 0;

inline cudaError_t mark_phase(int i, cudaStream_t s) {
  if (!g_phase_events) return cudaSuccess;
  if (g_phase_n == 2) {
    if (i != 0 && i != 6) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(g_phase_events[i == 0 ? 0 : 1]), s);
  }
  return cudaEventRecord(static_cast<cudaEvent_t>(g_phase_events[i]), s);
}

#define MOE_CUDA(call)                          \
  do {                                          \
    if ((call) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// Router -> slots (the routing state in the workspace), optional caller copies.
// Decode sizes (up to 32 tokens, one per warp of the CTA, and 256 experts): the
// select kernel also groups the slots by expert, so that the layer takes one launch
// fewer (gpt-oss T=32: 114.4 -> 108.5 us per step).  With two tokens per warp in turn
// (T = 64) the separate kernels are faster.
bool select_permutes(const moe_cfg_t* c, const Layout& L, int T) {
  return !L.prefill && L.S <= kPermuteOneCtaSlots && T <= kPermuteThreads / 32 && c->n_experts <= 256;
}

int run_router(const moe_cfg_t* c, const void* x, int T, const moe_router_t* r,
               const moe_shared_t* sh, const Layout& L, void* ws, int32_t* ids_out, float* w_out,
               float* sgate_out, float* logits_out, bool fill_slots, cudaStream_t s) {
  const int has_sh = (c->shared_ff > 0 && sh) ? 1 : 0;
  const uint16_t* wsh = has_sh ? static_cast<const uint16_t*>(sh->gate_inp) : nullptr;
  // Logits go straight to the caller's buffer when it has the same row layout.
  float* lg = at<float>(ws, L.logits);
  int ldl = c->n_experts + has_sh;
  if (logits_out && !has_sh) {
    lg = logits_out;
    ldl = c->n_experts;
  }
  if (fill_slots) MOE_CUDA(mark_phase(0, s));
  // The MoE's input: RMSNorm(x) when cfg.rms_norm (that kernel then clears the status).
  const uint16_t* xr = static_cast<const uint16_t*>(x);
  uint32_t* status = at<uint32_t>(ws, L.status);
  if (c->rms_norm) {
    uint16_t* xn = at<uint16_t>(ws, L.xn);
    MOE_CUDA(launch_rmsnorm(xr, T, c->d_model, static_cast<const uint16_t*>(r->norm_w), c->rms_eps, xn,
                            status, s));
    xr = xn;
    status = nullptr;
  }
  bool gate_in_logits = false;
  // The expert outputs' region is free while routing runs: it may hold the router
  // GEMM's partial logits (split-K over d).
  const size_t part_floats = (size_t)L.S * (size_t)(c->d_model > L.ldh ? c->d_model : L.ldh);
  int nsplit = 1, ppitch = 0;
  MOE_CUDA(launch_router_logits(xr, T, c->d_model, static_cast<const uint16_t*>(r->w),
                                static_cast<const uint16_t*>(r->bias), wsh, c->n_experts, lg, ldl,
                                at<float>(ws, L.Y), part_floats, &nsplit, &ppitch, status, &gate_in_logits,
                                s));
  if (fill_slots) MOE_CUDA(mark_phase(1, s));
  const int norm = c->gating == MOE_GATING_TOPK_SOFTMAX ? 1 : c->norm_topk_prob;
  int32_t* slot_e = fill_slots ? at<int32_t>(ws, L.slot_expert) : nullptr;
  float* slot_w = fill_slots ? at<float>(ws, L.slot_w) : nullptr;
  // Logits in the scratch (possibly as partial sums): the select kernel adds them and
  // writes the logits where the caller asked for them.
  const bool scratch = ppitch > 0;
  const RouteState rs = route_state(ws, L);
  MOE_CUDA(launch_router_select(scratch ? at<float>(ws, L.Y) : lg, scratch ? ppitch : ldl, nsplit,
                                (size_t)T * ppitch, scratch && logits_out ? lg : nullptr, ldl, T,
                                c->n_experts, c->top_k, norm,
                                c->expert_weights_scale, has_sh, ids_out, w_out, sgate_out, slot_e,
                                slot_w, xr, c->d_model, gate_in_logits ? nullptr : wsh,
                                fill_slots && select_permutes(c, L, T) ? &rs : nullptr, L.S, L.E1,
                                8 * decode_chunks(c, T), s));
  if (fill_slots) MOE_CUDA(mark_phase(2, s));
  if (logits_out && has_sh)
    MOE_CUDA(cudaMemcpy2DAsync(logits_out, sizeof(float) * c->n_experts, lg, sizeof(float) * ldl,
                               sizeof(float) * c->n_experts, T, cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

// Permute, experts, combine.  The slots must already hold the routing.
// permuted: the router's select kernel already grouped the slots (select_permutes).
int run_experts(const moe_cfg_t* c, const void* x_layer, int T, const moe_experts_t* e,
                const moe_shared_t* sh, void* y, const Layout& L, void* ws, bool permuted, cudaStream_t s) {
  const RouteState rs = route_state(ws, L);
  // The experts run on the MoE's input (RMSNorm(x) when cfg.rms_norm, written by the
  // router step); the residual adds the un-normalised layer input.
  const void* x = c->rms_norm ? static_cast<const void*>(at<uint16_t>(ws, L.xn)) : x_layer;
  const uint16_t* resid = c->residual ? static_cast<const uint16_t*>(x_layer) : nullptr;
  const ExpertParams p = expert_params(c, e, sh);
  uint16_t* h = at<uint16_t>(ws, L.h);
  float* Y = at<float>(ws, L.Y);
  // Prefill, not deterministic: the down projection adds each weighted expert output
  // into yacc (cleared by the gate_up kernel's epilogue warps) and the finish kernel
  // adds the residual and rounds; otherwise the combine gathers the Y rows in slot
  // order.
  float* yacc = L.accumulate ? at<float>(ws, L.yacc) : nullptr;
  const size_t yacc_floats = L.accumulate ? (size_t)T * c->d_model : 0;
  auto finish = [&](const float* Yv, const float* ya) {
    return ya ? launch_finish_accumulated(ya, T, c->d_model, resid, y, c->y_fp32 != 0, s)
              : launch_combine(Yv, rs.slot_w, rs.slot_expert, T, L.K, c->d_model, L.E1, resid, y,
                               c->y_fp32 != 0, s);
  };
  if (L.prefill_fp4) {
    // MXFP4 with the clamped GLU: f16-operand grouped GEMMs over work items of 256 rows
    // (two m tiles per dequantised weight tile).
    constexpr int kItemRows = 256;
    const int max_items = L.E1 + (L.S + kItemRows - 1) / kItemRows;
    uint16_t* xp16 = at<uint16_t>(ws, L.xp);          // x rows as f16
    uint8_t* scratch = at<uint8_t>(ws, L.scalesT);
    const Fp4Rows rows = prefill_fp4_rows(p, scratch, L.S);
    uint16_t* h16 = at<uint16_t>(ws, L.h);            // h rows as f16 [S, ldh]
    float* hside = Y;                                 // fp32 copies of small h chunks (Y is free until down)
    const int kh = h_stage_exp(c->glu_limit, c->glu_alpha);
    MOE_CUDA(launch_prefill_fp4_prep(p, scratch, L.S, s));
    MOE_CUDA(launch_permute(rs, L.S, L.E1, kItemRows, at<int>(ws, L.hist), s));
    MOE_CUDA(launch_gather_rows_f16(static_cast<const uint16_t*>(x), rs.row2slot, L.S, L.K, c->d_model, xp16,
                                    rows.rowmul, rows.hmax, rs, kItemRows / 2, rows.order, rows.sched, s));
    MOE_CUDA(mark_phase(3, s));
    MOE_CUDA(launch_gateup_prefill_fp4(p, rs, xp16, L.S, h16, hside, L.ldh, kh, scratch, max_items, yacc,
                                       yacc_floats, s));
    MOE_CUDA(mark_phase(4, s));
    MOE_CUDA(launch_h_fix_f16(hside, rows.hmax, L.S, c->expert_ff, kh, h16, L.ldh, rows.hmul, s));
    MOE_CUDA(launch_down_prefill_fp4(p, rs, h16, L.ldh, L.S, Y, yacc, L.K, scratch, max_items, s));
    MOE_CUDA(mark_phase(5, s));
    MOE_CUDA(finish(Y, yacc));
    MOE_CUDA(mark_phase(6, s));
    return MOE_OK;
  }
  if (L.prefill) {
    // Grouped GEMMs on tcgen05: m tiles of 128 rows.  With MXFP4 weights the A rows of
    // gate_up are gathered first; bf16 gate_up reads them from x by row index.
    constexpr int kTileRows = 128;
    const int max_mtiles = L.E1 + (L.S + kTileRows - 1) / kTileRows;
    const bool fp4 = c->wfmt == MOE_WFMT_MXFP4;
    uint16_t* xp = at<uint16_t>(ws, L.xp);
    uint8_t* scalesT = at<uint8_t>(ws, L.scalesT);
    if (fp4) MOE_CUDA(launch_transpose_scales(p, scalesT, s));
    MOE_CUDA(launch_permute(rs, L.S, L.E1, kTileRows, at<int>(ws, L.hist), s));
    if (fp4)
      MOE_CUDA(launch_gather_rows(static_cast<const uint16_t*>(x), rs.row2slot, L.S, L.K,
                                  c->d_model, xp, s));
    MOE_CUDA(mark_phase(3, s));
    MOE_CUDA(launch_gateup_prefill(p, c->wfmt, c->interleaved_gate_up, rs, xp, L.S,
                                   static_cast<const uint16_t*>(x), T, L.K, h, L.ldh, scalesT,
                                   max_mtiles, yacc, yacc_floats, s));
    MOE_CUDA(mark_phase(4, s));
    MOE_CUDA(launch_down_prefill(p, c->wfmt, rs, h, L.ldh, L.S, Y, yacc, L.K, scalesT, max_mtiles, s));
    MOE_CUDA(mark_phase(5, s));
    MOE_CUDA(finish(Y, yacc));
    MOE_CUDA(mark_phase(6, s));
    return MOE_OK;
  }
  const int chunks = decode_chunks(c, T);
  const int tpg = 8 * chunks;
  const int max_items = L.E1 + (L.S + tpg - 1) / tpg;
  if (!permuted) MOE_CUDA(launch_permute(rs, L.S, L.E1, tpg, at<int>(ws, L.hist), s));
  MOE_CUDA(mark_phase(3, s));
  // One-chunk items: the TMA-fed shared-memory weight stream when it applies.
  const bool ring = chunks == 1 && decode_ring(c, T);
  const bool fp4 = c->wfmt == MOE_WFMT_MXFP4;
  const int items = expect_items(c, T);
  bool done = false;
  if (ring && fp4)
    MOE_CUDA(launch_gateup_decode_fp4(p, rs, static_cast<const uint16_t*>(x), L.K, h, L.ldh, max_items,
                                      s, &done));
  else if (ring)
    MOE_CUDA(launch_gateup_decode_ring(p, rs, static_cast<const uint16_t*>(x), L.K, h, L.ldh, max_items,
                                       items, s, &done));
  // the per-row maxima of h exist only when the MXFP4 ring's gate_up wrote them
  RouteState rs_dn = rs;
  if (!(ring && fp4 && done)) rs_dn.hmax = nullptr;
  // bf16 one-chunk items on the register-stream kernels: gate_up and down in one
  // launch (the grouping that zeroes its counters is the one-CTA routine here).
  bool fused = false;
  if (!done && !ring && decode_fused(c, L, T))
    MOE_CUDA(launch_experts_decode_fused(p, rs, static_cast<const uint16_t*>(x), L.K, h, L.ldh, Y, max_items,
                                         c->interleaved_gate_up, s, &fused));
  if (!done && !fused)
    MOE_CUDA(launch_gateup_decode(p, c->wfmt, c->interleaved_gate_up, rs,
                                  static_cast<const uint16_t*>(x), L.K, h, L.ldh, max_items, chunks,
                                  s));
  MOE_CUDA(mark_phase(4, s));
  done = fused;
  if (!fused && ring && fp4)
    MOE_CUDA(launch_down_decode_fp4(p, rs_dn, h, L.ldh, Y, max_items, s, &done));
  else if (!fused && ring)
    MOE_CUDA(launch_down_decode_ring(p, rs, h, L.ldh, Y, max_items, items, s, &done));
  if (!done) MOE_CUDA(launch_down_decode(p, c->wfmt, rs, h, L.ldh, Y, max_items, chunks, s));
  MOE_CUDA(mark_phase(5, s));
  MOE_CUDA(launch_combine(Y, rs.slot_w, rs.slot_expert, T, L.K, c->d_model, L.E1, resid, y,
                          c->y_fp32 != 0, s));
  MOE_CUDA(mark_phase(6, s));
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const moe_cfg_t* cfg, int32_t T) {
  if (validate_cfg(cfg) != MOE_OK || T < 0) return 0;
  Layout L;
  if (!make_layout(cfg, T, &L)) return 0;
  return L.total;
}

int moe_select_path(const moe_cfg_t* cfg, int32_t T) {
  const int st = validate_cfg(cfg);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  return path_for(cfg, T);
}

int moe_kernel_plan(const moe_cfg_t* cfg, int32_t T) {
  const int st = validate_cfg(cfg);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(cfg, T, &L)) return MOE_ERR_UNSUPPORTED;
  if (L.prefill_fp4) return MOE_PLAN_PREFILL_F16;
  if (L.prefill) return MOE_PLAN_PREFILL_BF16;
  if (decode_fused(cfg, L, T)) return MOE_PLAN_DECODE_FUSED;
  return decode_chunks(cfg, T) == 1 && decode_ring(cfg, T) ? MOE_PLAN_DECODE_RING : MOE_PLAN_DECODE_WARP;
}

int moe_route(const moe_cfg_t* cfg, const void* x, int32_t T, const moe_router_t* router,
              const moe_shared_t* shared, int32_t* topk_ids, float* topk_w, float* sgate,
              float* logits, void* ws, size_t ws_bytes, void* stream) {
  int st = validate_cfg(cfg);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if ((st = check_router(cfg, router)) != MOE_OK) return st;
  // The shared gate is computed when the layer has a shared expert (shared_ff > 0).
  const bool has_sh = cfg->shared_ff > 0;
  if (has_sh && (!shared || !shared->gate_inp)) return MOE_ERR_INVALID_ARG;
  if (sgate && !has_sh) return MOE_ERR_INVALID_ARG;
  if (has_sh && !aligned16(shared->gate_inp)) return MOE_ERR_ALIGNMENT;
  if (!aligned16(x) || !aligned16(topk_ids) || !aligned16(topk_w) || (sgate && !aligned16(sgate)) ||
      (logits && !aligned16(logits)))
    return MOE_ERR_ALIGNMENT;
  Layout L;
  if ((st = check_ws(cfg, T, ws, ws_bytes, &L)) != MOE_OK) return st;
  return run_router(cfg, x, T, router, shared, L, ws, topk_ids, topk_w, sgate, logits, false,
                    static_cast<cudaStream_t>(stream));
}

int moe_topk_from_logits(const moe_cfg_t* cfg, const float* logits, int32_t T, int32_t* topk_ids,
                         float* topk_w, void* stream) {
  const int st = validate_cfg(cfg);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w)) return MOE_ERR_ALIGNMENT;
  const int norm = cfg->gating == MOE_GATING_TOPK_SOFTMAX ? 1 : cfg->norm_topk_prob;
  if (launch_router_select(logits, cfg->n_experts, 1, 0, nullptr, 0, T, cfg->n_experts, cfg->top_k, norm,
                           cfg->expert_weights_scale, 0, topk_ids, topk_w, nullptr, nullptr,
                           nullptr, nullptr, 0, nullptr, nullptr, 0, 0, 0,
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_group_by_expert(const moe_cfg_t* cfg, const int32_t* topk_ids, int32_t T, int32_t* counts,
                        int32_t* offsets, int32_t* perm, void* ws, size_t ws_bytes, void* stream) {
  int st = validate_cfg(cfg);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !perm)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(counts) || !aligned16(offsets) || (topk_ids && !aligned16(topk_ids)) ||
      (perm && !aligned16(perm)))
    return MOE_ERR_ALIGNMENT;
  Layout L;
  if ((st = check_ws(cfg, T, ws, ws_bytes, &L)) != MOE_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The routed slots only (no shared expert): S = T k slots over E experts, written
  // straight into the caller's arrays; the work list stays in the workspace.
  RouteState rs = route_state(ws, L);
  rs.counts = counts;
  rs.offsets = offsets;
  rs.row2slot = perm;
  const int S = T * cfg->top_k;
  MOE_CUDA(launch_ingest_routing(topk_ids, nullptr, nullptr, T, cfg->n_experts, cfg->top_k, 0, rs.slot_expert,
                                 nullptr, rs.status, s));
  MOE_CUDA(launch_permute(rs, S, cfg->n_experts, 128, at<int>(ws, L.hist), s));
  return MOE_OK;
}

int moe_ffn_forward(const moe_cfg_t* cfg, const void* x, int32_t T, const moe_router_t* router,
                    const moe_experts_t* experts, const moe_shared_t* shared, void* y,
                    int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  int st = validate_cfg(cfg);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !y) return MOE_ERR_INVALID_ARG;
  if ((st = check_router(cfg, router)) != MOE_OK) return st;
  if ((st = check_experts(cfg, experts, shared)) != MOE_OK) return st;
  if (!aligned16(x) || !aligned16(y) || (topk_ids && !aligned16(topk_ids)) ||
      (topk_w && !aligned16(topk_w)))
    return MOE_ERR_ALIGNMENT;
  Layout L;
  if ((st = check_ws(cfg, T, ws, ws_bytes, &L)) != MOE_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = run_router(cfg, x, T, router, shared, L, ws, topk_ids, topk_w, nullptr, nullptr, true,
                       s)) != MOE_OK)
    return st;
  return run_experts(cfg, x, T, experts, shared, y, L, ws, select_permutes(cfg, L, T), s);
}

int moe_ffn_forward_routed(const moe_cfg_t* cfg, const void* x, int32_t T,
                           const int32_t* topk_ids, const float* topk_w, const float* sgate,
                           const moe_experts_t* experts, const moe_shared_t* shared, void* y,
                           void* ws, size_t ws_bytes, void* stream) {
  int st = validate_cfg(cfg);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !y || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (cfg->shared_ff > 0 && !sgate) return MOE_ERR_INVALID_ARG;
  // The norm weight lives in the router description, which this entry point does not
  // take: callers that route themselves pass the MoE's input (already normalised).
  if (cfg->rms_norm) return MOE_ERR_UNSUPPORTED;
  if ((st = check_experts(cfg, experts, shared)) != MOE_OK) return st;
  if (!aligned16(x) || !aligned16(y) || !aligned16(topk_ids) || !aligned16(topk_w) ||
      (sgate && !aligned16(sgate)))
    return MOE_ERR_ALIGNMENT;
  Layout L;
  if ((st = check_ws(cfg, T, ws, ws_bytes, &L)) != MOE_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_CUDA(mark_phase(0, s));
  MOE_CUDA(launch_ingest_routing(topk_ids, topk_w, sgate, T, cfg->n_experts, cfg->top_k,
                                 cfg->shared_ff > 0, at<int32_t>(ws, L.slot_expert),
                                 at<float>(ws, L.slot_w), at<uint32_t>(ws, L.status), s));
  MOE_CUDA(mark_phase(1, s));
  MOE_CUDA(mark_phase(2, s));
  return run_experts(cfg, x, T, experts, shared, y, L, ws, false, s);
}

namespace {

// The host entry's work on one stream, without the final synchronisation: x in,
// the layer, y out (or y written across the host link by the combine kernel).
int host_step(const moe_cfg_t* cfg, const void* x_host, int32_t T, const moe_router_t* router,
              const moe_experts_t* experts, const moe_shared_t* shared, void* y_host, void* ydirect,
              void* ws, size_t ws_bytes, const Layout& L, cudaStream_t s) {
  void* xd = at<void>(ws, L.xstage);
  void* yd = at<void>(ws, L.ystage);
  const size_t bytes = (size_t)T * cfg->d_model * 2;
  const size_t ybytes = (size_t)T * cfg->d_model * (cfg->y_fp32 ? 4 : 2);
  MOE_CUDA(cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, s));
  const int st = moe_ffn_forward(cfg, xd, T, router, experts, shared, ydirect ? ydirect : yd, nullptr,
                                 nullptr, ws, ws_bytes, s);
  if (st != MOE_OK) return st;
  if (!ydirect) MOE_CUDA(cudaMemcpyAsync(y_host, yd, ybytes, cudaMemcpyDeviceToHost, s));
  return MOE_OK;
}

// Repeated host-entry calls with the same arguments replay one CUDA graph of the
// step (captured on a private stream, launched on the caller's): one launch per step
// instead of one per kernel and copy, and no gaps between the kernels.  The key is
// every argument (the tensors' contents are read when the graph runs, as in a plain
// call).  Used when both host buffers are page-locked.
struct HostGraphKey {
  moe_cfg_t cfg;
  moe_router_t router;
  moe_experts_t experts;
  moe_shared_t shared;
  const void* x_host;
  void* y_host;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  int32_t T, has_shared, device;
};

constexpr int kHostGraphs = 4;
struct HostGraph {
  bool used;
  HostGraphKey key;
  cudaGraphExec_t exec;
};
std::mutex g_host_graph_mu;
HostGraph g_host_graphs[kHostGraphs];   // not destroyed at exit: the driver reclaims them
int g_host_graph_next = 0;
cudaStream_t g_capture_stream[64] = {};

bool page_locked(const void* p) {
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return pa.type == cudaMemoryTypeHost;
}

// Launches this call's cached graph on s (captured on first use; the launch happens
// under the cache's lock, so that no other thread can retire the graph meanwhile).
// cudaErrorNotReady: run the call directly instead (phase events set, the caller's
// stream capturing, pageable buffers, or any failure to build the graph, which then
// leaves no error behind).
cudaError_t launch_host_graph(const moe_cfg_t* cfg, const void* x_host, int32_t T, const moe_router_t* router,
                              const moe_experts_t* experts, const moe_shared_t* shared, void* y_host,
                              void* ydirect, void* ws, size_t ws_bytes, const Layout& L, cudaStream_t s) {
  constexpr cudaError_t kDirect = cudaErrorNotReady;
  if (g_phase_events) return kDirect;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    (void)cudaGetLastError();
    return kDirect;
  }
  if (!page_locked(x_host) || !page_locked(y_host)) return kDirect;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kDirect;
  HostGraphKey key;
  std::memset(&key, 0, sizeof(key));
  key.cfg = *cfg;
  key.router = *router;
  key.experts = *experts;
  if (shared) key.shared = *shared;
  key.has_shared = shared != nullptr;
  key.x_host = x_host;
  key.y_host = y_host;
  key.ws = ws;
  key.ws_bytes = ws_bytes;
  key.stream = s;
  key.T = T;
  key.device = dev;
  std::lock_guard<std::mutex> lock(g_host_graph_mu);
  for (HostGraph& g : g_host_graphs)
    if (g.used && std::memcmp(&g.key, &key, sizeof(key)) == 0) return cudaGraphLaunch(g.exec, s);
  if (!g_capture_stream[dev] &&
      cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking) != cudaSuccess) {
    (void)cudaGetLastError();
    g_capture_stream[dev] = nullptr;
    return kDirect;
  }
  const cudaStream_t cap = g_capture_stream[dev];
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    (void)cudaGetLastError();
    return kDirect;
  }
  const int st = host_step(cfg, x_host, T, router, experts, shared, y_host, ydirect, ws, ws_bytes, L, cap);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cap, &graph);
  cudaGraphExec_t exec = nullptr;
  if (st == MOE_OK && ec == cudaSuccess && graph &&
      cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
    exec = nullptr;
  if (graph) cudaGraphDestroy(graph);
  (void)cudaGetLastError();
  if (!exec) return kDirect;
  HostGraph& slot = g_host_graphs[g_host_graph_next];
  g_host_graph_next = (g_host_graph_next + 1) % kHostGraphs;
  if (slot.used) cudaGraphExecDestroy(slot.exec);   // launches still in flight complete
  slot.used = true;
  slot.key = key;
  slot.exec = exec;
  return cudaGraphLaunch(exec, s);
}

}  // namespace

int moe_ffn_forward_host(const moe_cfg_t* cfg, const void* x_host, int32_t T,
                         const moe_router_t* router, const moe_experts_t* experts,
                         const moe_shared_t* shared, void* y_host, void* ws, size_t ws_bytes,
                         void* stream) {
  int st = validate_cfg(cfg);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  if ((st = check_router(cfg, router)) != MOE_OK) return st;
  if ((st = check_experts(cfg, experts, shared)) != MOE_OK) return st;
  Layout L;
  if ((st = check_ws(cfg, T, ws, ws_bytes, &L)) != MOE_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Page-locked y_host with a device address (cudaHostAlloc, or cudaHostRegister
  // with mapping) takes the layer's output directly: the combine kernel writes it
  // across the host link, in place of a device staging buffer and a second copy.
  // Pageable memory reports cudaMemoryTypeUnregistered and takes the staged copy.
  void* ydirect = nullptr;
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, y_host) == cudaSuccess) {
    if (pa.type == cudaMemoryTypeHost && pa.devicePointer && aligned16(pa.devicePointer))
      ydirect = pa.devicePointer;
  } else {
    (void)cudaGetLastError();
  }
  const cudaError_t eg =
      launch_host_graph(cfg, x_host, T, router, experts, shared, y_host, ydirect, ws, ws_bytes, L, s);
  if (eg == cudaErrorNotReady) {
    st = host_step(cfg, x_host, T, router, experts, shared, y_host, ydirect, ws, ws_bytes, L, s);
    if (st != MOE_OK) return st;
  } else {
    MOE_CUDA(eg);
  }
  MOE_CUDA(cudaStreamSynchronize(s));
  return MOE_OK;
}

int moe_mxfp4_to_bf16(const void* blocks, const void* scales, int64_t rows, int32_t n_in,
                      void* out, void* stream) {
  if (!blocks || !scales || !out || rows < 0 || n_in <= 0) return MOE_ERR_INVALID_ARG;
  if (n_in % 32) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(blocks) || !aligned16(out)) return MOE_ERR_ALIGNMENT;
  if (rows == 0) return MOE_OK;
  MOE_CUDA(launch_mxfp4_to_bf16(static_cast<const uint8_t*>(blocks),
                                static_cast<const uint8_t*>(scales), rows, n_in,
                                static_cast<uint16_t*>(out), static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_set_phase_events(void* const* events, int32_t n_events) {
  if (events && n_events != 2 && n_events < 7) return MOE_ERR_INVALID_ARG;
  const int need = n_events == 2 ? 2 : 7;
  if (events)
    for (int i = 0; i < need; ++i)
      if (!events[i]) return MOE_ERR_INVALID_ARG;
  g_phase_events = events;
  g_phase_n = events ? need : 0;
  return MOE_OK;
}

int moe_test_set_wait_limit(uint32_t max_polls, int32_t withhold_first_load) {
  if (max_polls == 0 || withhold_first_load < 0 || withhold_first_load > 1) return MOE_ERR_INVALID_ARG;
  const int w = withhold_first_load;
  MOE_CUDA(prefill_set_wait_test(max_polls, w));
  MOE_CUDA(prefill_fp4_set_wait_test(max_polls, w));
  MOE_CUDA(ring_set_wait_test(max_polls, w));
  MOE_CUDA(fp4_stream_set_wait_test(max_polls, w));
  MOE_CUDA(decode_set_wait_test(max_polls, w));
  return MOE_OK;
}

int moe_test_set_decode_fusion(int32_t enable) {
  if (enable < 0 || enable > 1) return MOE_ERR_INVALID_ARG;
  g_decode_fusion = enable != 0;
  return MOE_OK;
}

int moe_device_status(void* ws, void* stream, uint32_t* detail) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  MOE_CUDA(cudaStreamSynchronize(s));
  MOE_CUDA(cudaMemcpy(&bits, ws, sizeof(bits), cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemset(ws, 0, sizeof(bits)));
  if (detail) *detail = bits;
  if (bits & STATUS_TIMEOUT) return MOE_ERR_TIMEOUT;
  return bits ? MOE_ERR_DEVICE_CHECK : MOE_OK;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case MOE_ERR_CUDA: return "CUDA launch or runtime error";
    case MOE_ERR_DEVICE_CHECK: return "device-side bounds check fired";
    case MOE_ERR_TIMEOUT: return "device-side bounded wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
