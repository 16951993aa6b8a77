/*
 * CPU oracle of one MoE layer forward -- TEST INFRASTRUCTURE ONLY (see colibri_oracle.h).
 *
 * Each function is the plain definition of one step, in fp64, with no blocking,
 * fusion or reordering beyond the definition.  OpenMP only splits independent
 * tokens across threads; every per-token sum runs in index order.
 */
#include "colibri_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static int cfg_ok(const oracle_cfg_t* c) {
  return c && c->d_model > 0 && c->d_ff > 0 && c->num_experts >= 2 && c->top_k >= 1 && c->top_k <= 4 &&
         c->top_k <= c->num_experts && (c->act == ORACLE_ACT_RELU_BIAS || c->act == ORACLE_ACT_SWIGLU) &&
         (c->gate_mode == ORACLE_GATE_PAIR_SOFTMAX || c->gate_mode == ORACLE_GATE_FULL_SOFTMAX) &&
         (c->has_shared == 0 || c->has_shared == 1);
}

/* Router logits: the routing GEMM of zskr.cn article 3.2 (step 1, "no softmax yet"),
 * plus the optional router bias of news.rkmt.cn article 3.1. */
int oracle_router_logits(const oracle_cfg_t* cfg, const oracle_weights_t* w, const float* x, int32_t T,
                         double* logits) {
  if (!cfg_ok(cfg) || !w || !w->w_router || (T > 0 && (!x || !logits)) || T < 0) return -1;
  const int d = cfg->d_model, E = cfg->num_experts;
#pragma omp parallel for schedule(static)
  for (int32_t t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int j = 0; j < d; ++j) acc += (double)x[(size_t)t * d + j] * (double)w->w_router[(size_t)e * d + j];
      if (w->b_router) acc += (double)w->b_router[e];
      logits[(size_t)t * E + e] = acc;
    }
  }
  return 0;
}

/* "a ranks before b": higher logit first, equal logits -> lower expert index first. */
static int ranks_before(double la, int a, double lb, int b) { return la > lb || (la == lb && a < b); }

/* Top-k selection and gates.  Ranking: hnwysp.cn article 3.1 (top-k indices in strictly descending
 * score order); zskr.cn article 3.2 (selection is deterministic).
 * Pair mode: the softmax restricted to the selected experts, which sums to 1 as every gate pair
 * printed in hnwysp.cn article 2.2 / 4.3 does.  For k = 2 that is g_a = 1 / (1 + e^{L_b - L_a}) and
 * g_b = 1 - g_a.  Full mode: the softmax over all experts evaluated at the selected ones (the weights
 * hnwysp.cn article 3.1's code returns; news.rkmt.cn article 5.2's "softmax top-k"). */
int oracle_topk(const oracle_cfg_t* cfg, const double* logits, int32_t T, int32_t* idx, double* gate) {
  if (!cfg_ok(cfg) || T < 0 || (T > 0 && (!logits || !idx || !gate))) return -1;
  const int E = cfg->num_experts, k = cfg->top_k;
  if (E > 64) return -1;
  for (int32_t t = 0; t < T; ++t) {
    const double* L = logits + (size_t)t * E;
    /* insertion sort of the expert ids by the ranking above (stable, plainly correct) */
    int order[64];
    for (int e = 0; e < E; ++e) order[e] = e;
    for (int i = 1; i < E; ++i) {
      int cur = order[i], j = i - 1;
      while (j >= 0 && ranks_before(L[cur], cur, L[order[j]], order[j])) {
        order[j + 1] = order[j];
        --j;
      }
      order[j + 1] = cur;
    }
    int32_t* it = idx + (size_t)t * k;
    double* gt = gate + (size_t)t * k;
    for (int j = 0; j < k; ++j) it[j] = order[j];
    const double top = L[order[0]];
    if (cfg->gate_mode == ORACLE_GATE_PAIR_SOFTMAX && k == 2) {
      gt[0] = 1.0 / (1.0 + exp(L[order[1]] - top));
      gt[1] = 1.0 - gt[0];
    } else {
      double den = 0.0;
      const int n = cfg->gate_mode == ORACLE_GATE_PAIR_SOFTMAX ? k : E;
      for (int j = 0; j < n; ++j) den += exp(L[order[j]] - top);
      for (int j = 0; j < k; ++j) gt[j] = exp(L[order[j]] - top) / den;
    }
  }
  return 0;
}

/* Dispatch: per-expert counts and offsets (zskr.cn article 3.2, "expert_counts ... dispatch
 * offsets"), tokens grouped by expert (zskr.cn article 2.1, Dispatch stage), each group in
 * ascending token order (a counting sort). */
int oracle_dispatch(const oracle_cfg_t* cfg, const int32_t* idx, int32_t T, int32_t* counts,
                    int32_t* offsets_raw, int32_t* row_of, int32_t* token_of_row) {
  if (!cfg_ok(cfg) || T < 0 || !counts || !offsets_raw) return -1;
  const int E = cfg->num_experts, k = cfg->top_k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < (int64_t)k * T; ++i) {
    int e = idx[i];
    if (e < 0 || e >= E) return -1;
    counts[e] += 1;
  }
  offsets_raw[0] = 0;
  for (int e = 0; e < E; ++e) offsets_raw[e + 1] = offsets_raw[e] + counts[e];
  int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  if (!fill) return -1;
  for (int32_t t = 0; t < T; ++t) {
    for (int s = 0; s < k; ++s) {
      int e = idx[(size_t)k * t + s];
      int32_t row = offsets_raw[e] + fill[e];
      fill[e] += 1;
      if (row_of) row_of[(size_t)k * t + s] = row;
      if (token_of_row) token_of_row[row] = t;
    }
  }
  free(fill);
  return 0;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* One expert on one token.  Affine expert layers out = in * W^T + b with W stored [out, in]
 * (hnwysp.cn article 3.2); two layers per expert W1 | b1 | W2 | b2 (m.nxbn.cn article 3.1).  SwiGLU:
 * h = silu(W_gate x) * (W_up x), y = W_down h. */
static int ffn(const oracle_cfg_t* cfg, const float* W1, const float* W3, const float* W2, const float* B1,
               const float* B2, const float* x_t, double* y) {
  const int d = cfg->d_model, f = cfg->d_ff;
  double* h = (double*)malloc((size_t)f * sizeof(double));
  if (!h) return -1;
  for (int i = 0; i < f; ++i) {
    double u = 0.0;
    for (int j = 0; j < d; ++j) u += (double)W1[(size_t)i * d + j] * (double)x_t[j];
    if (cfg->act == ORACLE_ACT_RELU_BIAS) {
      if (B1) u += (double)B1[i];
      h[i] = u > 0.0 ? u : 0.0;
    } else {
      double v = 0.0;
      for (int j = 0; j < d; ++j) v += (double)W3[(size_t)i * d + j] * (double)x_t[j];
      h[i] = silu(u) * v;
    }
  }
  for (int kk = 0; kk < d; ++kk) {
    double acc = 0.0;
    for (int i = 0; i < f; ++i) acc += (double)W2[(size_t)kk * f + i] * h[i];
    if (cfg->act == ORACLE_ACT_RELU_BIAS && B2) acc += (double)B2[kk];
    y[kk] = acc;
  }
  free(h);
  return 0;
}

int oracle_expert_ffn(const oracle_cfg_t* cfg, const oracle_weights_t* w, int32_t e, const float* x_t, double* y) {
  if (!cfg_ok(cfg) || !w || !x_t || !y || e < 0 || e >= cfg->num_experts) return -1;
  return ffn(cfg, w->w1[e], w->w3 ? w->w3[e] : NULL, w->w2[e], w->b1 ? w->b1[e] : NULL, w->b2 ? w->b2[e] : NULL,
             x_t, y);
}

/* The shared expert: same shape as a routed expert, applied to every token (news.rkmt.cn 5.2). */
int oracle_shared_ffn(const oracle_cfg_t* cfg, const oracle_weights_t* w, const float* x_t, double* y) {
  if (!cfg_ok(cfg) || !w || !x_t || !y || !cfg->has_shared || !w->ws1 || !w->ws2) return -1;
  if (cfg->act == ORACLE_ACT_SWIGLU && !w->ws3) return -1;
  return ffn(cfg, w->ws1, w->ws3, w->ws2, w->bs1, w->bs2, x_t, y);
}

static int weights_ok(const oracle_cfg_t* cfg, const oracle_weights_t* w) {
  if (!w || !w->w_router || !w->w1 || !w->w2) return 0;
  if (cfg->act == ORACLE_ACT_SWIGLU && !w->w3) return 0;
  for (int e = 0; e < cfg->num_experts; ++e) {
    if (!w->w1[e] || !w->w2[e]) return 0;
    if (cfg->act == ORACLE_ACT_SWIGLU && !w->w3[e]) return 0;
    if (cfg->act == ORACLE_ACT_RELU_BIAS && ((w->b1 && !w->b1[e]) || (w->b2 && !w->b2[e]))) return 0;
  }
  if (cfg->has_shared && (!w->ws1 || !w->ws2 || (cfg->act == ORACLE_ACT_SWIGLU && !w->ws3))) return 0;
  return 1;
}

/* Output of one token: gate-weighted sum of its k experts (m.nxbn.cn article 3.3) in slot order, then
 * the shared expert's output with weight 1. */
static int token_output(const oracle_cfg_t* cfg, const oracle_weights_t* w, const float* x_t, const int32_t* idx_t,
                        const double* gate_t, double* out_t, double* y) {
  const int d = cfg->d_model;
  for (int k = 0; k < d; ++k) out_t[k] = 0.0;
  for (int s = 0; s < cfg->top_k; ++s) {
    if (oracle_expert_ffn(cfg, w, idx_t[s], x_t, y)) return -1;
    for (int k = 0; k < d; ++k) out_t[k] += gate_t[s] * y[k];
  }
  if (cfg->has_shared) {
    if (oracle_shared_ffn(cfg, w, x_t, y)) return -1;
    for (int k = 0; k < d; ++k) out_t[k] += y[k];
  }
  return 0;
}

int oracle_forward_rows(const oracle_cfg_t* cfg, const oracle_weights_t* w, const float* x, int32_t T,
                        const int32_t* idx, const double* gate, const int32_t* tokens, int32_t n,
                        double* out_rows) {
  if (!cfg_ok(cfg) || !weights_ok(cfg, w) || n < 0 || (n > 0 && (!x || !idx || !gate || !tokens || !out_rows)))
    return -1;
  const int d = cfg->d_model, k = cfg->top_k;
  int bad = 0;
#pragma omp parallel
  {
    double* y = (double*)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(dynamic, 1)
    for (int32_t i = 0; i < n; ++i) {
      int32_t t = tokens[i];
      if (!y || t < 0 || t >= T ||
          token_output(cfg, w, x + (size_t)t * d, idx + (size_t)k * t, gate + (size_t)k * t,
                       out_rows + (size_t)i * d, y)) {
#pragma omp atomic write
        bad = 1;
      }
    }
    free(y);
  }
  return bad ? -1 : 0;
}

int oracle_forward(const oracle_cfg_t* cfg, const oracle_weights_t* w, const float* x, int32_t T, double* out,
                   int32_t* idx, double* gate, int32_t* counts, int32_t* offsets_raw, int32_t* row_of,
                   double* logits) {
  if (!cfg_ok(cfg) || !weights_ok(cfg, w) || T < 0 || (T > 0 && (!x || !out))) return -1;
  const int E = cfg->num_experts, k = cfg->top_k;
  int rc = -1;
  double* L = logits ? logits : (double*)malloc(((size_t)T * E + 1) * sizeof(double));
  int32_t* I = idx ? idx : (int32_t*)malloc(((size_t)k * T + 1) * sizeof(int32_t));
  double* G = gate ? gate : (double*)malloc(((size_t)k * T + 1) * sizeof(double));
  int32_t* C = counts ? counts : (int32_t*)malloc((size_t)E * sizeof(int32_t));
  int32_t* O = offsets_raw ? offsets_raw : (int32_t*)malloc(((size_t)E + 1) * sizeof(int32_t));
  int32_t* tok = (int32_t*)malloc(((size_t)T + 1) * sizeof(int32_t));
  if (!L || !I || !G || !C || !O || !tok) goto done;
  if (oracle_router_logits(cfg, w, x, T, L)) goto done;
  if (oracle_topk(cfg, L, T, I, G)) goto done;
  if (oracle_dispatch(cfg, I, T, C, O, row_of, NULL)) goto done;
  for (int32_t t = 0; t < T; ++t) tok[t] = t;
  rc = oracle_forward_rows(cfg, w, x, T, I, G, tok, T, out);
done:
  if (!logits) free(L);
  if (!idx) free(I);
  if (!gate) free(G);
  if (!counts) free(C);
  if (!offsets_raw) free(O);
  free(tok);
  return rc;
}
