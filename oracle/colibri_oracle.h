/*
 * CPU oracle of one Mixture-of-Experts layer forward: TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 reference of what the layer computes.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the product
 * library never links or calls it.  It shares no code with the CUDA path.
 *
 * Sources (Colibri MoE engine articles; section numbers are the articles' own):
 *   zskr.cn/news/2272131 "Colibri: a lightweight C MoE inference engine for edge
 *     devices", 2.1 (stages Route -> Dispatch -> Compute), 3.2 (routing logits
 *     GEMM, top-k, per-expert counts and dispatch offsets)
 *   hnwysp.cn/news/30485, 2.2 (gate-weighted sum, gate pair like [0.6, 0.4]),
 *     3.1 (softmax over experts, then top-k in descending score order),
 *     3.2 (expert = affine map out = in * W^T + b, W stored [out_dim, in_dim])
 *   m.nxbn.cn/news/48047, 3.1 (per-expert parameters W1 | b1 | W2 | b2),
 *     3.3 (output aggregation: sum of expert outputs weighted by gating score)
 *   news.rkmt.cn/news/2271114, 3.1 (optional router bias)
 *
 * Readings where the articles are silent or disagree:
 *   - selection is made on the logits; softmax is monotone so it selects the
 *     same experts;
 *   - default gates: the softmax over the selected experts (they sum to 1; the
 *     "linear" top-k of news.rkmt.cn 5.2, Mixtral-style); gate_mode 1: the full
 *     softmax over all experts evaluated at the selected ones (the unnormalised
 *     weights of hnwysp.cn 3.1's code, "softmax top-k", DeepSeek-style);
 *   - top_k from 1 to 4 (hnwysp.cn 3.1: TOP_K is a compile-time 2, "change it to
 *     1 or 4 and recompile");
 *   - optional shared expert (news.rkmt.cn 5.2: Qwen2-MoE, 1 shared + 15 routed
 *     experts): an always-on expert of the same shape whose output is added to
 *     the gated mixture with weight 1;
 *   - equal logits: the lower expert index ranks first;
 *   - rows of one expert are ordered by ascending token index;
 *   - SwiGLU experts h = silu(W_gate x) * (W_up x), y = W_down h, no biases;
 *     ReLU experts h = max(W1 x + b1, 0), y = W2 h + b2;
 *   - no residual add: the layer returns the mixture only.
 *
 * All arrays are host, row-major, fp32 inputs (bf16 data widened to fp32);
 * every accumulation is fp64.  Functions return 0, or -1 on a bad argument.
 */
#ifndef COLIBRI_ORACLE_H
#define COLIBRI_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_ACT_RELU_BIAS = 0, ORACLE_ACT_SWIGLU = 1 };

enum { ORACLE_GATE_PAIR_SOFTMAX = 0, ORACLE_GATE_FULL_SOFTMAX = 1 };

typedef struct {
  int32_t d_model;      /* d */
  int32_t d_ff;         /* f */
  int32_t num_experts;  /* E (routed) */
  int32_t top_k;        /* k, 1..4 */
  int32_t act;          /* ORACLE_ACT_* */
  int32_t gate_mode;    /* ORACLE_GATE_* */
  int32_t has_shared;   /* 0/1: shared expert present */
} oracle_cfg_t;

typedef struct {
  const float* w_router;   /* [E, d] */
  const float* b_router;   /* [E] or NULL */
  const float* const* w1;  /* E x [f, d]: W1 (ReLU) or W_gate (SwiGLU) */
  const float* const* w3;  /* E x [f, d]: W_up (SwiGLU), NULL for ReLU */
  const float* const* w2;  /* E x [d, f]: W2 / W_down */
  const float* const* b1;  /* E x [f] (ReLU) or NULL */
  const float* const* b2;  /* E x [d] (ReLU) or NULL */
  const float* ws1;        /* shared expert [f, d] (has_shared) */
  const float* ws3;        /* shared expert [f, d] (SwiGLU) */
  const float* ws2;        /* shared expert [d, f] */
  const float* bs1;        /* shared expert [f] (ReLU) */
  const float* bs2;        /* shared expert [d] (ReLU) */
} oracle_weights_t;

/* logits[t, e] = sum_j x[t, j] * W_r[e, j] (+ b_r[e]), fp64. */
int oracle_router_logits(const oracle_cfg_t* cfg, const oracle_weights_t* w, const float* x, int32_t T,
                         double* logits);

/* Per token: experts ranked by (logit descending, index ascending); idx[t, 0..k-1] the first k.
 * Gates (gate[t, 0..k-1]): pair mode, k == 2: gate[t,0] = 1 / (1 + exp(L_b - L_a)), gate[t,1] = 1 - gate[t,0];
 * pair mode, other k: exp(L_j - L_a) / sum over the selected i of exp(L_i - L_a);
 * full mode: exp(L_j - L_a) / sum over all experts i of exp(L_i - L_a). */
int oracle_topk(const oracle_cfg_t* cfg, const double* logits, int32_t T, int32_t* idx, double* gate);

/* counts[e] = number of (t, s) with idx[t, s] == e (routed experts); offsets_raw = exclusive prefix sum
 * of counts (E + 1 entries); row_of[t, s] = offsets_raw[e] + rank of t among tokens routed to e
 * (ascending t); token_of_row[row] = t (k*T entries). */
int oracle_dispatch(const oracle_cfg_t* cfg, const int32_t* idx, int32_t T, int32_t* counts,
                    int32_t* offsets_raw, int32_t* row_of, int32_t* token_of_row);

/* y[d] = expert e applied to one token row x_t[d] (fp64 output). */
int oracle_expert_ffn(const oracle_cfg_t* cfg, const oracle_weights_t* w, int32_t e, const float* x_t, double* y);

/* Shared expert (has_shared) applied to one token row. */
int oracle_shared_ffn(const oracle_cfg_t* cfg, const oracle_weights_t* w, const float* x_t, double* y);

/* Full layer: out[t, :] = sum_j gate[t,j] * y_{idx[t,j]}(x_t)  (+ y_shared(x_t)).
 * Any of idx, gate, counts, offsets_raw, row_of, logits may be NULL. */
int oracle_forward(const oracle_cfg_t* cfg, const oracle_weights_t* w, const float* x, int32_t T, double* out,
                   int32_t* idx, double* gate, int32_t* counts, int32_t* offsets_raw, int32_t* row_of,
                   double* logits);

/* The layer output for the n tokens listed in `tokens` only (out_rows[n, d]), given that batch's
 * routing (idx, gate from oracle_topk).  Used to check large batches on a sample of rows. */
int oracle_forward_rows(const oracle_cfg_t* cfg, const oracle_weights_t* w, const float* x, int32_t T,
                        const int32_t* idx, const double* gate, const int32_t* tokens, int32_t n,
                        double* out_rows);

#ifdef __cplusplus
}
#endif
#endif
