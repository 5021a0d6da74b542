/*
 * CPU oracle for the latency-oriented MoE decode step.
 *
 * TEST INFRASTRUCTURE ONLY. This is a plain, slow restatement of what one
 * decode step of a pre-norm MoE transformer computes, written so that a reader can check it
 * against its definition by eye. Only the test suite, the smoke check and the benchmark's CPU
 * baseline may call it. The GPU engine never links, loads or calls it, and the two share no
 * code, tables or constants.
 *
 * Sources (web pages on latency-oriented decode):
 *  - "Ultra-High Interactivity on NVIDIA GPUs? TileRT on InferenceX", section "But What Exactly
 *    is TileRT?": the persistent engine kernel forwards intermediates on chip; the result is the
 *    one the unfused chain of operators would give, so the oracle is that chain.
 *  - "vLLM's Kimi K3 Backend Hits 842 Tokens per Second", section "Four changes drive the gains":
 *    attention input projection, output projection + residual, router scores, shared expert,
 *    routed experts.
 *  - "Kimi K3: The Manos, The Mythos, The Legendos": GQA attention; the FFN expert modelled as
 *    SwiGLU (6 d m flops per token); top-k over router scores; the residual x_{l+1} = x_l + f(x_l).
 * The pages do not define RMSNorm, RoPE, the router normalisation or the FP8 block layout; those
 * follow the model configuration (FP8-E4M3 weights with 128x128 fp32 block scales, bf16
 * activations, sigmoid router with top-k normalised gates, one shared expert, RoPE) under the
 * plainest readings listed with each function in oracle.c.
 *
 * Arithmetic: every sum, product, exp and sqrt is in double. Values are rounded to bf16 (round
 * to nearest even) only where the method stores a bf16 activation: the normalised GEMV inputs,
 * q/k/v, the attention output, the SwiGLU product h, and the residual stream.
 */
#ifndef ORC_ORACLE_H
#define ORC_ORACLE_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* An FP8-E4M3 matrix W[n][k], row-major, with fp32 block scales S[ceil(n/128)][ceil(k/128)].
   The real value of element (r, c) is S[r/128][c/128] * e4m3(W[r][c]). */
typedef struct {
  const uint8_t* w;
  const float* s;
  int32_t n, k;
} orc_mat;

typedef struct {
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim;
  int32_t n_experts, top_k, moe_inter, n_shared;
  int32_t dense_ffn; /* > 0: a dense SwiGLU FFN replaces the MoE block */
  int32_t vocab;     /* 0: no embedding table and no LM head */
  double rms_eps, rope_theta;
} orc_cfg;

typedef struct {
  const uint16_t* attn_norm; /* bf16 [hidden] */
  orc_mat wq, wk, wv, wo;
  const uint16_t* ffn_norm; /* bf16 [hidden] */
  orc_mat router;           /* [n_experts][hidden] */
  const orc_mat* gate;      /* [n_experts], each [moe_inter][hidden] */
  const orc_mat* up;        /* [n_experts], each [moe_inter][hidden] */
  const orc_mat* down;      /* [n_experts], each [hidden][moe_inter] */
  const orc_mat* sgate;     /* [n_shared] */
  const orc_mat* sup;
  const orc_mat* sdown;
  orc_mat fgate, fup, fdown; /* dense FFN */
} orc_layer;

typedef struct {
  orc_cfg cfg;
  const uint16_t* embed;      /* bf16 [vocab][hidden] */
  const uint16_t* final_norm; /* bf16 [hidden] */
  orc_mat lm_head;            /* [vocab][hidden] */
  const orc_layer* layers;    /* [n_layers] */
} orc_model;

/* One sequence's KV cache: k and v are bf16 [n_layers][n_kv_heads][max_ctx][head_dim]. */
typedef struct {
  uint16_t* k;
  uint16_t* v;
  int32_t max_ctx;
} orc_kv;

/* Optional per-layer observations of one decode step (any pointer may be NULL). */
typedef struct {
  double* layer_out;   /* [n_layers][hidden] residual stream after each layer (bf16 values) */
  int32_t* topk_idx;   /* [n_layers][top_k] selected experts, score-descending */
  double* topk_gate;   /* [n_layers][top_k] normalised gates */
  double* router_score;/* [n_layers][n_experts] sigmoid scores */
  double* attn_out;    /* [n_layers][n_heads*head_dim] attention output o (bf16 values) */
} orc_trace;

/* ---- element codecs ---- */
double orc_e4m3_value(uint8_t code);
double orc_bf16_value(uint16_t bits);
uint16_t orc_bf16_bits(double v); /* round to nearest even, IEEE-style overflow to inf */
double orc_bf16_round(double v);  /* orc_bf16_value(orc_bf16_bits(v)) */

/* ---- building blocks ---- */
void orc_gemv(const orc_mat* m, const double* x, double* y);
void orc_rmsnorm(const double* x, const uint16_t* w, int32_t n, double eps, double* out);
void orc_rope(double* v, int32_t head_dim, int32_t pos, double theta);
void orc_attention_head(const double* q, const uint16_t* k, const uint16_t* v, int32_t n_keys,
                        int32_t head_dim, double* o);
void orc_router_topk(const double* logits, int32_t n_experts, int32_t top_k, int32_t* idx,
                     double* gate, double* score);
void orc_swiglu_expert(const orc_mat* gate, const orc_mat* up, const orc_mat* down,
                       const double* xn, double* y);

/* ---- whole steps ---- */
/* One decoder layer for one sequence at position pos: x (bf16 values) is updated in place, the
   layer's k/v for pos are written into kv. */
int32_t orc_layer_step(const orc_model* m, int32_t layer, double* x, int32_t pos, orc_kv* kv,
                       orc_trace* tr);
/* One decode step for one sequence. Input: hidden (bf16 bits) when given, else the embedding row
   of token (vocab > 0); the engine's hidden_in path starts from a hidden state the same way.
   Outputs: logits [vocab] (may be NULL), hidden_out [hidden] final residual stream as bf16 bits
   (may be NULL). Returns the greedy token (lowest id among equal maxima), or -1 if vocab == 0. */
int32_t orc_decode_step(const orc_model* m, int32_t token, const uint16_t* hidden, int32_t pos,
                        orc_kv* kv, double* logits, uint16_t* hidden_out, orc_trace* tr);
/* Recompute the last position of tokens[0..n) from scratch, layer by layer over all positions
   (no cache carried between calls). logits [vocab] of position n-1. Returns its argmax. */
int32_t orc_full_recompute(const orc_model* m, const int32_t* tokens, int32_t n, double* logits);
/* argmax with ties to the lowest index */
int32_t orc_argmax(const double* v, int32_t n);

/* Host threads for the rows of a matrix-vector product (bit-identical results for any count;
   1 when built without OpenMP). */
void orc_set_threads(int32_t n);
int32_t orc_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
