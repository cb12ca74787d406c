/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse Mixture-of-Experts FFN forward pass.
 *
 * One shared library, libmoe.so, computes the forward pass of a sparse MoE FFN
 * layer on the GPU in two gating conventions:
 *
 *   Qwen3.5-MoE  ("qwen35moe - Forward-Pass Design (Pantheon port)", section
 *                "Shared-expert MoE FFN (every layer)"; "qwen35moe CPU-reference
 *                golden vectors", section "Kernel 4 - MoE routing"):
 *       l = x W_r^T;  p = softmax(l);  ids = top-k(p) by selection sort with
 *       first-seen tie-break;  w_j = p_ids_j / sum_j p_ids_j * expert_weights_scale;
 *       moe = sum_j w_j * down_e(silu(gate_e x) * up_e x);
 *       y = moe + sigmoid(gate_inp_shexp . x) * SwiGLU_shexp(x).
 *
 *   gpt-oss      ("Phase 19: MoE - gpt-oss-20b", section 2, Router and Experts;
 *                section 3, MXFP4 dequantisation):
 *       l = x W_r^T + b;  ids = top-k(l);  s = softmax(l[ids]);
 *       gu = x W_gu,e^T + b_gu,e;  gate = gu[0::2], up = gu[1::2];
 *       gate = min(gate, limit);  up = clamp(up, -limit, limit);
 *       h = (up + 1) * gate * sigmoid(alpha * gate);
 *       y = sum_j s_j * (h W_d,e^T + b_d,e),
 *       with MXFP4 expert weights: per 32 inputs, 16 bytes of E2M1 codes (low
 *       nibble = even input) and one E8M0 scale byte, value = code * 2^(scale-127).
 *
 * Conventions shared by every entry point
 *   - Pointers named as device pointers must be device memory of the current
 *     CUDA device; the caller owns every buffer.  The library allocates nothing
 *     and never synchronises, except where an entry point says otherwise.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued on it in stream order; results are valid once the
 *     stream has reached the end of the call's work.
 *   - bf16 tensors are raw IEEE bfloat16 bit patterns (uint16), row-major.
 *     Weight matrices are stored row = output, column = input (y = x W^T).
 *   - T == 0 is a no-op that returns MOE_OK (data pointers may then be NULL).
 *   - Every tensor pointer must be 16-byte aligned (MOE_ERR_ALIGNMENT).
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_* code.  On error nothing
 *     has been enqueued unless the code is MOE_ERR_CUDA (a launch failed).
 *   - Scratch memory comes from the caller's workspace `ws` of at least
 *     moe_workspace_bytes(cfg, T) bytes (16-byte aligned).  Calls that share a
 *     workspace must be ordered on one stream.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status codes */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)   /* null pointer, T < 0, k > E, unknown enum value, ... */
#define MOE_ERR_UNSUPPORTED (-2)   /* well-formed but outside what the kernels implement */
#define MOE_ERR_WORKSPACE (-3)     /* ws_bytes < moe_workspace_bytes(cfg, T) */
#define MOE_ERR_ALIGNMENT (-4)     /* a pointer is not 16-byte aligned */
#define MOE_ERR_CUDA (-5)          /* a CUDA runtime call or kernel launch failed */
#define MOE_ERR_DEVICE_CHECK (-6)  /* a kernel's bounds check fired (see moe_device_status) */
#define MOE_ERR_TIMEOUT (-7)       /* a bounded device-side wait gave up */

/* ------------------------------------------------------------------ configuration */
enum {
  MOE_GATING_SOFTMAX_TOPK_RENORM = 0, /* Qwen: softmax over E, top-k, renormalise x scale */
  MOE_GATING_TOPK_SOFTMAX = 1         /* gpt-oss: top-k on logits, softmax over the k chosen */
};
enum {
  MOE_ACT_SWIGLU = 0,     /* h = silu(gate) * up */
  MOE_ACT_CLAMPED_GLU = 1 /* h = (clamp(up,+-limit) + 1) * min(gate,limit) * sigmoid(alpha*min(gate,limit)) */
};
enum {
  MOE_WFMT_BF16 = 0,  /* bf16 expert weights */
  MOE_WFMT_MXFP4 = 1  /* MXFP4 blocks u8 [rows, in/32, 16] + E8M0 scales u8 [rows, in/32] */
};
enum {
  MOE_PATH_AUTO = 0,    /* pick by mean tokens per expert, T*k/E */
  MOE_PATH_DECODE = 1,  /* weight-streaming grouped matvec (mma.sync); when experts have
                           at most 4 tokens on average, MXFP4 weights, and bf16 weights
                           in the separate gate / up layout (d, ff, sff multiples of 64)
                           for small batches, stream through a TMA-fed shared-memory
                           ring */
  MOE_PATH_PREFILL = 2, /* grouped GEMM on tcgen05 / TMEM fed by TMA */
  MOE_PATH_DECODE_REGISTERS = 3  /* MOE_PATH_DECODE with every weight load going straight
                                    to registers (no shared-memory ring); same results to
                                    within rounding, kept for comparison and tests */
};

typedef struct {
  int32_t d_model;              /* hidden size d; multiple of 32 */
  int32_t n_experts;            /* E, 1..1024 */
  int32_t top_k;                /* k, 1..min(E, 32) */
  int32_t expert_ff;            /* routed expert FF width; multiple of 32 */
  int32_t shared_ff;            /* shared expert FF width (multiple of 32); 0 = none */
  int32_t gating;               /* MOE_GATING_* */
  int32_t act;                  /* MOE_ACT_* of the routed experts (shared expert: SwiGLU) */
  int32_t wfmt;                 /* MOE_WFMT_* of the routed experts (shared expert: bf16) */
  int32_t interleaved_gate_up;  /* 1: one gate_up matrix, gate = even rows, up = odd rows
                                   (required for MXFP4); 0: separate gate and up matrices */
  int32_t norm_topk_prob;       /* softmax gating: 1 = divide chosen probabilities by their sum */
  float expert_weights_scale;   /* multiplies every routing weight (Qwen 1.0; gpt-oss 1.0) */
  float glu_limit;              /* clamped GLU limit (gpt-oss 7.0) */
  float glu_alpha;              /* clamped GLU sigmoid slope (gpt-oss 1.702) */
  int32_t path;                 /* MOE_PATH_* */
  int32_t y_fp32;               /* 0: y is bf16 [T, d] (RNE of the fp32 result); 1: y is fp32 [T, d] */
  /* Steps either side of the MoE ("qwen35moe - Forward-Pass Design", "Block
   * scaffold": post_attention_norm, then the residual adds the un-normalised input;
   * "Phase 19: MoE - gpt-oss-20b", section 2, "Decoder layer": out = h + moe(post_norm(h))). */
  int32_t rms_norm;             /* 1: route and run the experts on RMSNorm(x) = x / sqrt(mean(x^2) +
                                   rms_eps) * router.norm_w (fp32 statistics, rounded to bf16) */
  float rms_eps;                /* Qwen 1e-6, gpt-oss 1e-5; finite and >= 0 */
  int32_t residual;             /* 1: y = x + MoE(...) (x un-normalised), summed in fp32 */
  int32_t deterministic;        /* 1: a token's expert outputs are summed in a fixed order by a
                                   gather over its slots, so y is bit-identical run to run.
                                   0: on the prefill path the down projection adds each weighted
                                   expert output into a per-token fp32 sum with atomic adds in its
                                   epilogue (no round trip of the [T*k, d] expert outputs through
                                   memory); the order of those adds varies, so the last bits of y
                                   may differ between runs.  The decode path always takes the
                                   fixed order. */
  int32_t reserved[2];          /* must be zero */
} moe_cfg_t;

/* Router: w bf16 [E, d] (row e = expert e's logit weights); bias bf16 [E] or NULL;
 * norm_w bf16 [d], the RMSNorm weight (required when cfg.rms_norm, else ignored). */
typedef struct {
  const void* w;
  const void* bias;
  const void* norm_w;
} moe_router_t;

/* Routed experts (device pointers; unused members NULL).
 *   bf16, separate:     gate bf16 [E, ff, d], up bf16 [E, ff, d]
 *   bf16, interleaved:  gate_up bf16 [E, 2ff, d] (row 2f = gate f, row 2f+1 = up f)
 *   MXFP4:              gate_up u8 [E, 2ff, d/32, 16] blocks, gate_up_scales u8 [E, 2ff, d/32]
 *   gate_up_bias        bf16 [E, 2ff] in gate_up row order (interleaved layouts only) or NULL
 *   down                bf16 [E, d, ff]  |  MXFP4 u8 [E, d, ff/32, 16], down_scales u8 [E, d, ff/32]
 *   down_bias           bf16 [E, d] or NULL */
typedef struct {
  const void* gate;
  const void* up;
  const void* gate_up;
  const void* gate_up_scales;
  const void* gate_up_bias;
  const void* down;
  const void* down_scales;
  const void* down_bias;
} moe_experts_t;

/* Shared expert, always on (bf16): gate/up [sff, d], down [d, sff], gate_inp [d]
 * ("qwen35moe - Forward-Pass Design", section "Shared-expert MoE FFN": ffn_*_shexp
 * and ffn_gate_inp_shexp). */
typedef struct {
  const void* gate;
  const void* up;
  const void* down;
  const void* gate_inp;
} moe_shared_t;

/* ------------------------------------------------------------------ entry points */

/* Bytes of workspace that moe_route / moe_ffn_forward / moe_ffn_forward_routed /
 * moe_ffn_forward_host need for T tokens with this configuration.  Returns 0
 * if cfg is invalid.  Pure host function, no CUDA calls. */
size_t moe_workspace_bytes(const moe_cfg_t* cfg, int32_t T);

/* Which expert path MOE_PATH_AUTO takes for T tokens (MOE_PATH_DECODE or
 * MOE_PATH_PREFILL), or a negative MOE_ERR_* if cfg is invalid. */
int moe_select_path(const moe_cfg_t* cfg, int32_t T);

/* The kernel family the expert phase of moe_ffn_forward runs for T tokens: */
enum {
  MOE_PLAN_DECODE_WARP = 1,     /* weight-streaming grouped matvec on warp MMAs, weights
                                   loaded straight into registers */
  MOE_PLAN_DECODE_RING = 2,     /* the same, weights streaming through a TMA-fed
                                   shared-memory ring (items of at most 8 tokens; MXFP4,
                                   or bf16 in the separate gate / up layout while the
                                   down projection has fewer than 16 x 152 units of
                                   128 rows) */
  MOE_PLAN_PREFILL_BF16 = 3,    /* tcgen05 grouped GEMMs with bf16 operands (bf16 weights,
                                   or MXFP4 decoded to bf16 in shared memory) */
  MOE_PLAN_PREFILL_F16 = 4,     /* tcgen05 grouped GEMMs with f16 operands: MXFP4 with the
                                   clamped GLU, each decoded weight tile shared by two
                                   128-row tiles */
  MOE_PLAN_DECODE_FUSED = 5     /* MOE_PLAN_DECODE_WARP's kernels as one launch (bf16
                                   weights, items of at most 8 tokens, at most 2048 slots
                                   when not on the ring): each CTA takes a ticket, gate_up
                                   units first, and a down unit waits for its item's
                                   gate_up units through a counter */
};
/* Returns one of MOE_PLAN_* (a host-side decision from cfg and T alone; no device
 * work), or a negative MOE_ERR_* if cfg is invalid or T < 0. */
int moe_kernel_plan(const moe_cfg_t* cfg, int32_t T);

/* Router: logits, top-k selection and routing weights, and the shared-expert gate.
 * Defined by: "qwen35moe CPU-reference golden vectors", Kernel 4 (softmax,
 * selection sort with first-seen tie-break, norm_topk_prob x expert_weights_scale,
 * sigmoid(gate_w . x)); "Phase 19: MoE - gpt-oss-20b", section 2 Router
 * (logits + bias, top-k, softmax over the chosen k).
 *   x         bf16 [T, d] device
 *   router    router weights (device)
 *   shared    NULL, or a shared expert whose gate_inp [d] is used for sgate
 *   topk_ids  int32 [T, k] device, out: chosen experts in selection order
 *             (descending logit; equal logits: lower index first)
 *   topk_w    fp32 [T, k] device, out: routing weights
 *   sgate     fp32 [T] device or NULL, out: sigmoid(gate_inp . x) (needs shared)
 *   logits    fp32 [T, E] device or NULL, out: router logits (bias included)
 * Logits accumulate bf16 x bf16 products in fp32; selection compares the fp32
 * logits (softmax is strictly increasing, so the order equals the order of the
 * probabilities).  T == 0 is a no-op. */
int moe_route(const moe_cfg_t* cfg, const void* x, int32_t T, const moe_router_t* router,
              const moe_shared_t* shared, int32_t* topk_ids, float* topk_w, float* sgate,
              float* logits, void* ws, size_t ws_bytes, void* stream);

/* Top-k selection and routing weights from caller-given fp32 logits [T, E]
 * (device), with the same rule as moe_route.  Needs no workspace. */
int moe_topk_from_logits(const moe_cfg_t* cfg, const float* logits, int32_t T, int32_t* topk_ids,
                         float* topk_w, void* stream);

/* Group token slots by expert: the permute step of the layer, on caller routing.
 * Defined by "qwen35moe - Forward-Pass Design", section "Batched prefill"
 * (expert-grouped batching: tokens that share an expert stream its weights once).
 *   topk_ids  int32 [T, k] device: slot s = t * k + j chose expert topk_ids[t, j]
 *   counts    int32 [E] device, out: slots routed to each expert
 *   offsets   int32 [E + 1] device, out: offsets[e] = sum of counts[0 .. e - 1]
 *   perm      int32 [T * k] device, out: perm[offsets[e] .. offsets[e + 1] - 1] are the
 *             slots routed to e in increasing slot order (the grouping is stable:
 *             the order the expert kernels of moe_ffn_forward see)
 * A slot whose id lies outside [0, E) is left out of counts, offsets and perm (its
 * entries of perm past offsets[E] are not written) and flags the device status word
 * in ws (moe_device_status then returns MOE_ERR_DEVICE_CHECK).  ws: at least
 * moe_workspace_bytes(cfg, T) bytes. */
int moe_group_by_expert(const moe_cfg_t* cfg, const int32_t* topk_ids, int32_t T, int32_t* counts,
                        int32_t* offsets, int32_t* perm, void* ws, size_t ws_bytes, void* stream);

/* The whole layer: route, group tokens by expert, run the selected experts (and
 * the shared expert), combine.  y bf16 [T, d] device, out.  topk_ids [T, k] /
 * topk_w [T, k] device or NULL: if given, the routing is also written there.
 * The combine accumulates in fp32; with cfg->y_fp32 = 0, y holds that fp32 result
 * rounded to bf16 (round to nearest even), with y_fp32 = 1 the fp32 result itself.
 * With cfg->rms_norm the router and the experts see RMSNorm(x) (router->norm_w);
 * with cfg->residual, y = x + MoE(...).  moe_route applies the same norm.
 * Defined by the two conventions in the header comment above. */
int moe_ffn_forward(const moe_cfg_t* cfg, const void* x, int32_t T, const moe_router_t* router,
                    const moe_experts_t* experts, const moe_shared_t* shared, void* y,
                    int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, void* stream);

/* The layer with caller-given routing (no router): topk_ids int32 [T, k] and
 * topk_w fp32 [T, k] device; sgate fp32 [T] device, required when the layer has
 * a shared expert.  Out-of-range ids are caught on the device: the call still
 * returns MOE_OK and moe_device_status() then reports MOE_ERR_DEVICE_CHECK
 * (rows with a bad id contribute nothing).  cfg->residual applies; cfg->rms_norm
 * returns MOE_ERR_UNSUPPORTED (the norm weight belongs to the router, which this
 * entry point does not take: pass the normalised input instead). */
int moe_ffn_forward_routed(const moe_cfg_t* cfg, const void* x, int32_t T,
                           const int32_t* topk_ids, const float* topk_w, const float* sgate,
                           const moe_experts_t* experts, const moe_shared_t* shared, void* y,
                           void* ws, size_t ws_bytes, void* stream);

/* moe_ffn_forward from and to HOST memory: x_host bf16 [T, d] and y_host bf16
 * [T, d] (fp32 with cfg->y_fp32) are host pointers (pinned memory gives full copy
 * speed); the weights stay device pointers.  Copies x into the workspace, runs the
 * layer and synchronises `stream` before returning, so y_host is ready on return.
 * A page-locked y_host that has a device address (cudaHostAlloc, or cudaHostRegister
 * with mapping) and is 16-byte aligned is written by the last kernel directly;
 * other memory receives y through a workspace buffer and a device-to-host copy.
 * When x_host and y_host are both page-locked, the call's work (copies and kernels)
 * is captured once as a CUDA graph and replayed by later calls with the same
 * arguments (every pointer, cfg, T, ws and stream; the buffers' contents are read
 * when the graph runs, as in a plain call); the library keeps the last four such
 * graphs.  A stream that is itself being captured, or phase events set with
 * moe_set_phase_events, take the plain path. */
int moe_ffn_forward_host(const moe_cfg_t* cfg, const void* x_host, int32_t T,
                         const moe_router_t* router, const moe_experts_t* experts,
                         const moe_shared_t* shared, void* y_host, void* ws, size_t ws_bytes,
                         void* stream);

/* Size of the device array that moe_ffn_forward_noalloc uses as its workspace. */
#define MOE_NOALLOC_WORKSPACE_BYTES ((size_t)8 << 20)

/* MOE_NOALLOC_WORKSPACE_BYTES as built into the library (for bindings that cannot
 * read the header's macro).  Pure host function. */
size_t moe_noalloc_workspace_bytes(void);

/* moe_ffn_forward for callers that cannot allocate device memory.  (The pages
 * have no counterpart: this is an interface addition.)
 *
 * Some callers are given only their input and output buffers: a plug-in inside
 * a host program or serving framework that owns all device memory through its
 * own pool, where a cudaMalloc would fail or take memory the pool has reserved,
 * or a latency-critical loop that must not make a call which may synchronise
 * the device.  They cannot provide the workspace moe_ffn_forward needs, so this
 * entry point takes it from a device array of MOE_NOALLOC_WORKSPACE_BYTES
 * (8 MiB) held by the library; it calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *   - Arguments and results are those of moe_ffn_forward without ws/ws_bytes.
 *   - Returns MOE_ERR_WORKSPACE when moe_workspace_bytes(cfg, T) exceeds the
 *     array: the largest batches that fit are 79 tokens of the Qwen3.5-mini
 *     layer and 76 of gpt-oss-20b (76 and 72 with cfg.rms_norm, whose
 *     normalised copy of x also lives in the workspace).
 *   - Every GPU that loads the library holds the array until the process exits.
 *   - The array has its own device address in every CUDA context.  The first
 *     call in a context (the device's primary context, a driver-API context the
 *     host program made current, or the primary context re-created after
 *     cudaDeviceReset) looks that address up (cudaGetSymbolAddress) and keeps it
 *     under the context's unique id; make that first call before any stream
 *     capture begins.  Up to 16 contexts are remembered at once.
 *   - All calls in a context share the one array and it keeps the last call's
 *     contents (the kernels rewrite all scratch they read, and the call's first
 *     kernel clears the status word): calls that overlap on the GPU -- on
 *     different streams or from different host threads without ordering -- race
 *     and corrupt each other.
 *   - Device-side checks of the call (a bounds check, a bounded wait that gave
 *     up) are read with moe_noalloc_device_status. */
int moe_ffn_forward_noalloc(const moe_cfg_t* cfg, const void* x, int32_t T,
                            const moe_router_t* router, const moe_experts_t* experts,
                            const moe_shared_t* shared, void* y, int32_t* topk_ids, float* topk_w,
                            void* stream);

/* moe_device_status for moe_ffn_forward_noalloc: synchronises `stream`, then
 * returns MOE_OK, MOE_ERR_DEVICE_CHECK or MOE_ERR_TIMEOUT according to the status
 * word in the library's array for the current context, and clears it; *detail (if
 * not NULL) receives the raw bits.  Reports the last noalloc call in this context
 * that the stream has completed. */
int moe_noalloc_device_status(void* stream, uint32_t* detail);

/* Decode MXFP4 weights to bf16 with the decoder the expert kernels use on their
 * weight-load path.  Defined by "Phase 19: MoE - gpt-oss-20b", section 3
 * (value = fp4_lut[code] * 2^(e8m0 - 127)) and the section 2 tensor layout (16
 * bytes per 32 inputs, low nibble = even input).
 *   blocks  u8 [rows, n_in/32, 16] device;  scales u8 [rows, n_in/32] device
 *   out     bf16 [rows, n_in] device
 * E2M1 values times a power of two are exact in bf16, so the result is exact
 * whenever it is a normal or subnormal bf16 (every scale byte 1..254 with
 * |value| < 2^128); scale byte 255 gives NaN.  n_in must be a positive multiple
 * of 32; rows >= 0. */
int moe_mxfp4_to_bf16(const void* blocks, const void* scales, int64_t rows, int32_t n_in,
                      void* out, void* stream);

/* Phase timing for benchmarks.  While enabled (events != NULL), each later
 * moe_ffn_forward / moe_ffn_forward_routed call made from this host thread
 * records events[i] on its stream at the phase boundaries:
 *   [0] start  [1] router logits done  [2] top-k done  [3] grouping done
 *   [4] gate_up + activation done  [5] down done  [6] combine done
 * (under MOE_PLAN_DECODE_FUSED gate_up and down are one launch: [4] and [5] both
 * follow it)
 * (the routed entry point records [1] and [2] together after ingesting the
 * routing).  `events` holds n_events >= 7 cudaEvent_t handles created by the
 * caller, or exactly 2: then only the start (events[0]) and the end
 * (events[1]) are recorded, which keeps the kernels free to overlap their
 * launches.  The array must stay valid while enabled.  events == NULL disables.
 * No counterpart on the pages: measurement plumbing only. */
int moe_set_phase_events(void* const* events, int32_t n_events);

/* Test hook for the give-up path of the bounded device waits (no counterpart on the
 * pages; not for production use).  Every mbarrier wait of the TMA-fed kernels, and
 * the down units' wait for their item's gate_up units under MOE_PLAN_DECODE_FUSED,
 * gives up after max_polls polls (default 2^20, about a second), sets
 * MOE_ERR_TIMEOUT in the device status word, and the CTA drains what it has in
 * flight, frees its TMEM and returns.  withhold_first_load = 1 also makes the
 * producer of the CTA that owns the first unit of work of the grouped GEMMs
 * (prefill, bf16 operands and router logits) and of the MXFP4 decode ring skip its
 * first load, and the first gate_up unit of MOE_PLAN_DECODE_FUSED withhold its
 * count, so that the wait for it runs out: the call's output is
 * then undefined and moe_device_status reports MOE_ERR_TIMEOUT.  Applies to the
 * current device, to calls enqueued after it returns; synchronises the device.
 * Restore with moe_test_set_wait_limit(1u << 20, 0).  max_polls > 0. */
int moe_test_set_wait_limit(uint32_t max_polls, int32_t withhold_first_load);

/* Test hook: enable (1, the default) or disable (0) MOE_PLAN_DECODE_FUSED, so that
 * the two-launch form of the same kernels can be checked against it.  Host-side only
 * (no device work); applies to calls made after it returns, from any thread.
 * MOE_ERR_INVALID_ARG for other values. */
int moe_test_set_decode_fusion(int32_t enable);

/* Synchronises `stream`, then returns MOE_OK, MOE_ERR_DEVICE_CHECK or
 * MOE_ERR_TIMEOUT according to the device status word kept in `ws`, and clears
 * it.  *detail (if not NULL) receives the raw status bits. */
int moe_device_status(void* ws, void* stream, uint32_t* detail);

/* Static text for a status code. */
const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
