/*
 * fp64 CPU oracle for the forward pass of a sparse Mixture-of-Experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header or table with the CUDA library.
 *
 * Every quantity is computed in fp64 from the bf16 / MXFP4-decoded inputs, with
 * no intermediate rounding, in plain loops that follow the pages' equations in
 * their order.  Sources (page title, section):
 *   [QW]  "qwen35moe - Forward-Pass Design (Pantheon port)", section
 *         "Shared-expert MoE FFN (every layer)" and the "Correctness watch-list"
 *         (norm_topk_prob = true).
 *   [GV]  "qwen35moe CPU-reference golden vectors", section "Kernel 4 - MoE
 *         routing" (softmax, selection sort with first-seen tie-break,
 *         norm_topk_prob and expert_weights_scale, sigmoid shared gate).
 *   [OSS] "Phase 19: MoE - gpt-oss-20b", section 2 "Router (GptOssTopKRouter)"
 *         and "Experts (GptOssExperts)", the measured tensor-layout listing, and
 *         section 3 "MXFP4 dequantisation".
 *   Optional steps either side of the MoE (cfg rms_norm, residual):
 *   [QW]  "Block scaffold": x -> post_attention_norm -> shared-MoE FFN -> + the
 *         un-normalised input; all norms RMS.
 *   [GV]  "Kernel 3 - QK-RMSNorm": RMS uses 1 / sqrt(mean(x^2) + eps), times the
 *         norm weight.
 *   [OSS] section 2, "RMSNorm" (standard) and "Decoder layer":
 *         out = h + moe(post_norm(h)).
 *
 * Readings taken where the pages leave a step open:
 *   - SwiGLU(x) = down(silu(gate x) * (up x)), silu(z) = z / (1 + e^-z).
 *   - Qwen selection is done on the logits: softmax is strictly increasing, so
 *     the selected set and order equal those of the probabilities in exact
 *     arithmetic, and no ties are introduced by rounding of exp.
 *   - Ties: first-seen (lowest index) wins, for both gating conventions; the
 *     output order is the selection order (descending key).
 *   - The gpt-oss down bias is added before the routing weight: s * (W_d h + b_d).
 *   - expert_weights_scale multiplies the final routing weights in both
 *     conventions (it is 1.0 for gpt-oss, whose page has no such factor).
 *   - E2M1 codes: bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa;
 *     exponent 0 is subnormal (0.5 * m).  E8M0 byte s means 2^(s-127); 255 is NaN.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int32_t d_model, n_experts, top_k, expert_ff, shared_ff;
  int32_t gating;          /* 0: softmax over all -> top-k -> renorm [QW][GV]; 1: top-k -> softmax [OSS] */
  int32_t act;             /* 0: SwiGLU [QW]; 1: clamped (up+1)*gate*sigmoid(alpha*gate) [OSS] */
  int32_t wfmt;            /* 0: bf16 weights; 1: MXFP4 blocks + E8M0 scales [OSS] */
  int32_t norm_topk_prob;  /* 1: divide the chosen probabilities by their sum [QW] */
  int32_t interleaved;     /* 1: one gate_up matrix, gate = even rows, up = odd rows [OSS] */
  double scale;            /* expert_weights_scale [GV] */
  double limit, alpha;     /* 7.0, 1.702 [OSS] */
  int32_t rms_norm;        /* 1: the MoE runs on RMSNorm(x) [QW Block scaffold; OSS Decoder layer] */
  int32_t residual;        /* 1: y = x + MoE(...) (x un-normalised) [QW; OSS] */
  double rms_eps;          /* 1e-6 [QW config], 1e-5 [OSS] */
} oracle_cfg;

typedef struct {
  const uint16_t *router_w;   /* bf16 [E, d] */
  const uint16_t *router_b;   /* bf16 [E] or NULL */
  /* bf16 experts: gate/up [E, ff, d] (or gate_up [E, 2ff, d] when interleaved), down [E, d, ff] */
  const uint16_t *gate, *up, *gate_up, *down;
  /* MXFP4 experts: gate_up blocks [E, 2ff, d/32, 16], scales [E, 2ff, d/32];
                    down blocks [E, d, ff/32, 16], scales [E, d, ff/32] */
  const uint8_t *gu_blocks, *gu_scales, *dn_blocks, *dn_scales;
  const uint16_t *gu_bias;    /* bf16 [E, 2ff] or NULL (interleaved) */
  const uint16_t *dn_bias;    /* bf16 [E, d] or NULL */
  /* shared expert (NULL when shared_ff == 0): gate/up [sff, d], down [d, sff], gate_inp [d] */
  const uint16_t *sh_gate, *sh_up, *sh_down, *sh_gate_inp;
  const uint16_t *norm_w;     /* bf16 [d]: RMSNorm weight (cfg rms_norm), else NULL */
} oracle_weights;

/* ------------------------------------------------------------------ number formats */

double oracle_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* E2M1 code (low 4 bits) -> value, from the bit definition [OSS section 3]. */
double oracle_e2m1(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* E8M0 scale byte -> 2^(s-127) [OSS section 3]. */
double oracle_e8m0(int s) { return s == 255 ? NAN : ldexp(1.0, s - 127); }

/* Element (row o, input i) of an MXFP4 matrix with n_in inputs per row: byte
   i/2 of block i/32 holds input i in its low nibble when i is even, in its high
   nibble when i is odd [OSS tensor-layout listing]; value = lut[code] * 2^(s-127). */
static double mxfp4_at(const uint8_t* blocks, const uint8_t* scales, int n_in, size_t o, int i) {
  size_t nb = (size_t)(n_in / 32);
  uint8_t byte = blocks[(o * nb + (size_t)(i / 32)) * 16 + (size_t)((i % 32) / 2)];
  int code = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);
  return oracle_e2m1(code) * oracle_e8m0(scales[o * nb + (size_t)(i / 32)]);
}

/* Decode n_rows rows of an MXFP4 matrix (n_in inputs each) to fp64. */
void oracle_mxfp4_decode(const uint8_t* blocks, const uint8_t* scales, int64_t n_rows, int n_in,
                         double* out) {
  for (int64_t o = 0; o < n_rows; ++o)
    for (int i = 0; i < n_in; ++i) out[o * n_in + i] = mxfp4_at(blocks, scales, n_in, (size_t)o, i);
}

/* ------------------------------------------------------------------ routing */

/* k rounds of a selection sort: each round scans e = 0..E-1 and keeps e if its
   key is strictly greater than the best so far, skipping taken experts, so the
   first-seen (lowest) index wins a tie [GV Kernel 4]. */
void oracle_select_topk(const double* key, int E, int k, int32_t* ids) {
  unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    double bv = 0.0;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || key[e] > bv) {
        best = e;
        bv = key[e];
      }
    }
    ids[j] = best;
    taken[best] = 1;
  }
  free(taken);
}

/* Routing of one token from its E logits: ids [k] in selection order, weights [k]. */
static void route_one(const oracle_cfg* c, const double* l, const int32_t* forced, int32_t* ids,
                      double* w) {
  int E = c->n_experts, k = c->top_k;
  if (forced)
    memcpy(ids, forced, sizeof(int32_t) * (size_t)k);
  else
    oracle_select_topk(l, E, k, ids);
  if (c->gating == 0) {
    /* softmax over all E logits [GV Kernel 4: router_softmax] */
    double mx = l[0];
    for (int e = 1; e < E; ++e) mx = l[e] > mx ? l[e] : mx;
    double Z = 0.0;
    for (int e = 0; e < E; ++e) Z += exp(l[e] - mx);
    double sel = 0.0;
    for (int j = 0; j < k; ++j) {
      w[j] = exp(l[ids[j]] - mx) / Z;
      sel += w[j];
    }
    /* norm_topk_prob, then expert_weights_scale [GV Kernel 4; QW watch-list] */
    for (int j = 0; j < k; ++j) w[j] = (c->norm_topk_prob ? w[j] / sel : w[j]) * c->scale;
  } else {
    /* softmax over the k chosen logits only [OSS Router] */
    double mx = l[ids[0]];
    for (int j = 1; j < k; ++j) mx = l[ids[j]] > mx ? l[ids[j]] : mx;
    double Z = 0.0;
    for (int j = 0; j < k; ++j) Z += exp(l[ids[j]] - mx);
    for (int j = 0; j < k; ++j) w[j] = exp(l[ids[j]] - mx) / Z * c->scale;
  }
}

/* Routing from caller-given logits [T, E] (fp64): ids [T, k], weights [T, k]. */
void oracle_route_from_logits(const oracle_cfg* c, const double* logits, int T, int32_t* ids,
                              double* w) {
#pragma omp parallel for schedule(dynamic, 16)
  for (int t = 0; t < T; ++t)
    route_one(c, logits + (size_t)t * c->n_experts, NULL, ids + (size_t)t * c->top_k,
              w + (size_t)t * c->top_k);
}

/* ------------------------------------------------------------------ experts */

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Dot of row `row` of expert e's first-layer matrix with x.  part 0 = gate, 1 = up. */
static double first_layer_dot(const oracle_cfg* c, const oracle_weights* W, int e, int part,
                              int f, const double* x) {
  int d = c->d_model, ff = c->expert_ff;
  double s = 0.0;
  if (c->wfmt == 1) {
    size_t row = (size_t)e * 2 * ff + (size_t)(2 * f + part);   /* interleaved gate/up */
    for (int i = 0; i < d; ++i) s += mxfp4_at(W->gu_blocks, W->gu_scales, d, row, i) * x[i];
  } else if (c->interleaved) {
    const uint16_t* r = W->gate_up + ((size_t)e * 2 * ff + (size_t)(2 * f + part)) * d;
    for (int i = 0; i < d; ++i) s += oracle_bf16(r[i]) * x[i];
  } else {
    const uint16_t* r = (part == 0 ? W->gate : W->up) + ((size_t)e * ff + (size_t)f) * d;
    for (int i = 0; i < d; ++i) s += oracle_bf16(r[i]) * x[i];
  }
  if (W->gu_bias) s += oracle_bf16(W->gu_bias[(size_t)e * 2 * ff + (size_t)(2 * f + part)]);
  return s;
}

/* Dot of row o of expert e's down matrix with h (ff values), plus the down bias. */
static double down_dot(const oracle_cfg* c, const oracle_weights* W, int e, int o, const double* h) {
  int d = c->d_model, ff = c->expert_ff;
  double s = 0.0;
  size_t row = (size_t)e * d + (size_t)o;
  if (c->wfmt == 1) {
    for (int f = 0; f < ff; ++f) s += mxfp4_at(W->dn_blocks, W->dn_scales, ff, row, f) * h[f];
  } else {
    const uint16_t* r = W->down + row * ff;
    for (int f = 0; f < ff; ++f) s += oracle_bf16(r[f]) * h[f];
  }
  if (W->dn_bias) s += oracle_bf16(W->dn_bias[row]);
  return s;
}

/* The expert's activation on one (gate, up) pair. */
static double activation(const oracle_cfg* c, double gate, double up) {
  if (c->act == 0) return gate * sigmoid(gate) * up;   /* silu(gate) * up [QW] */
  /* gate clamped from above only, up on both sides; (up + 1) * gate * sigmoid(alpha*gate) [OSS] */
  if (gate > c->limit) gate = c->limit;
  if (up > c->limit) up = c->limit;
  if (up < -c->limit) up = -c->limit;
  return (up + 1.0) * gate * sigmoid(c->alpha * gate);
}

/* ------------------------------------------------------------------ layer forward */

/* fp64 -> the nearest bf16 value (ties to even), returned as fp64: 8 significant
   bits, 8 exponent bits (finite, normal-range values; zero, inf and NaN pass). */
static double round_bf16(double v) {
  if (v == 0.0 || !isfinite(v)) return v;
  int e;
  double m = frexp(v, &e);          /* v = m * 2^e, 0.5 <= |m| < 1 */
  if (e < -125) e = -125;           /* below the normal range: bf16 subnormal spacing 2^-133 */
  return ldexp(nearbyint(ldexp(v, 8 - e)), e - 8);
}

/* The MoE's input from the layer input x (d values): RMSNorm(x) when cfg rms_norm,
   x / sqrt(mean(x^2) + eps) * w [GV Kernel 3; OSS RMSNorm], else x itself.  The
   normalised value is an activation in the layer's type, bf16, as x is: the
   "standard" RMSNorm of [OSS section 2] keeps its statistics in higher precision
   and returns the input's type; rounded to nearest, ties to even. */
static void moe_input(const oracle_cfg* c, const oracle_weights* W, const double* x, double* out) {
  int d = c->d_model;
  if (!c->rms_norm) {
    for (int i = 0; i < d; ++i) out[i] = x[i];
    return;
  }
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / d + c->rms_eps);
  for (int i = 0; i < d; ++i) out[i] = round_bf16(x[i] * inv * oracle_bf16(W->norm_w[i]));
}

/* Router of one token: logits x . W_r^T (+ b) [QW ffn_gate_inp; OSS Router], then
   the routing.  Returns 1 if a logit is NaN. */
static int router_one(const oracle_cfg* c, const oracle_weights* W, const double* xv, double* ll,
                      const int32_t* forced, int32_t* ids, double* w) {
  int d = c->d_model, E = c->n_experts, bad = 0;
  for (int e = 0; e < E; ++e) {
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += oracle_bf16(W->router_w[(size_t)e * d + i]) * xv[i];
    if (W->router_b) s += oracle_bf16(W->router_b[e]);
    ll[e] = s;
    if (isnan(s)) bad = 1;
  }
  route_one(c, ll, forced, ids, w);
  return bad;
}

/* Shared-expert gate sigmoid(gate_inp . x) [QW; GV Kernel 4]. */
static double shared_gate(const oracle_cfg* c, const oracle_weights* W, const double* xv) {
  double z = 0.0;
  for (int i = 0; i < c->d_model; ++i) z += oracle_bf16(W->sh_gate_inp[i]) * xv[i];
  return sigmoid(z);
}

/* Routing only, for the n_eval tokens in `tokens`: logits [n, E], ids [n, k],
   w [n, k], sgate [n] (0 without shared expert).  Returns the NaN-logit count. */
int oracle_route(const oracle_cfg* c, const oracle_weights* W, const uint16_t* x, int T,
                 const int32_t* tokens, int n_eval, int32_t* ids, double* w, double* sgate,
                 double* logits) {
  int d = c->d_model, E = c->n_experts, k = c->top_k, n_nan = 0;
  (void)T;
#pragma omp parallel for schedule(dynamic, 16) reduction(+ : n_nan)
  for (int n = 0; n < n_eval; ++n) {
    double* xin = (double*)malloc(sizeof(double) * (size_t)d);
    double* xv = (double*)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < d; ++i) xin[i] = oracle_bf16(x[(size_t)tokens[n] * d + i]);
    moe_input(c, W, xin, xv);
    n_nan += router_one(c, W, xv, logits + (size_t)n * E, NULL, ids + (size_t)n * k,
                        w + (size_t)n * k);
    sgate[n] = c->shared_ff > 0 ? shared_gate(c, W, xv) : 0.0;
    free(xin);
    free(xv);
  }
  return n_nan;
}


/*
 * Forward pass for the n_eval tokens listed in `tokens` (indices into x [T, d]).
 * Outputs, row i for token tokens[i]:
 *   y [n_eval, d], ids [n_eval, k], w [n_eval, k], sgate [n_eval] (0 without shared expert),
 *   logits [n_eval, E].
 * forced_ids (nullable) [n_eval, k]: use these experts instead of the top-k (the
 * weights still follow the gating rule, restricted to the forced set).
 * Returns the number of evaluated tokens with a NaN logit (outside the contract).
 */
int oracle_forward(const oracle_cfg* c, const oracle_weights* W, const uint16_t* x, int T,
                   const int32_t* tokens, int n_eval, const int32_t* forced_ids, double* y,
                   int32_t* ids, double* w, double* sgate, double* logits) {
  int d = c->d_model, E = c->n_experts, k = c->top_k, ff = c->expert_ff, sff = c->shared_ff;
  int n_nan = 0;
  (void)T;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : n_nan)
  for (int n = 0; n < n_eval; ++n) {
    int t = tokens[n];
    int hmax = ff > sff ? ff : sff;
    double* xin = (double*)malloc(sizeof(double) * (size_t)d);
    double* xv = (double*)malloc(sizeof(double) * (size_t)d);
    double* h = (double*)malloc(sizeof(double) * (size_t)hmax);
    double* yl = y + (size_t)n * d;
    double* ll = logits + (size_t)n * E;
    for (int i = 0; i < d; ++i) xin[i] = oracle_bf16(x[(size_t)t * d + i]);
    moe_input(c, W, xin, xv);   /* the MoE runs on RMSNorm(x) or on x */

    n_nan += router_one(c, W, xv, ll, forced_ids ? forced_ids + (size_t)n * k : NULL,
                        ids + (size_t)n * k, w + (size_t)n * k);

    /* routed experts: y = sum_j w_j * expert_{id_j}(x) [QW moe_out; OSS out] */
    for (int i = 0; i < d; ++i) yl[i] = 0.0;
    for (int j = 0; j < k; ++j) {
      int e = ids[(size_t)n * k + j];
      double wj = w[(size_t)n * k + j];
      for (int f = 0; f < ff; ++f)
        h[f] = activation(c, first_layer_dot(c, W, e, 0, f, xv), first_layer_dot(c, W, e, 1, f, xv));
      for (int o = 0; o < d; ++o) yl[o] += wj * down_dot(c, W, e, o, h);
    }

    /* shared expert: SwiGLU with the shexp weights, gated by sigmoid(gate_inp . x) [QW] */
    double sg = 0.0;
    if (sff > 0) {
      sg = shared_gate(c, W, xv);
      for (int f = 0; f < sff; ++f) {
        double gsum = 0.0, usum = 0.0;
        for (int i = 0; i < d; ++i) {
          gsum += oracle_bf16(W->sh_gate[(size_t)f * d + i]) * xv[i];
          usum += oracle_bf16(W->sh_up[(size_t)f * d + i]) * xv[i];
        }
        h[f] = gsum * sigmoid(gsum) * usum;
      }
      for (int o = 0; o < d; ++o) {
        double s = 0.0;
        for (int f = 0; f < sff; ++f) s += oracle_bf16(W->sh_down[(size_t)o * sff + f]) * h[f];
        yl[o] += sg * s;   /* out = moe_out + sgate * shexp [QW] */
      }
    }
    sgate[n] = sg;
    /* + the un-normalised layer input [QW Block scaffold; OSS Decoder layer] */
    if (c->residual)
      for (int o = 0; o < d; ++o) yl[o] += xin[o];
    free(xin);
    free(xv);
    free(h);
  }
  return n_nan;
}

/* Number of OpenMP threads the oracle runs with. */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
