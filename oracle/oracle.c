/*
 * CPU oracle for the latency-oriented MoE decode step. TEST INFRASTRUCTURE ONLY: see oracle.h.
 * Plain C, double arithmetic; bf16 rounding only at the stored activations. The rows of a
 * matrix-vector product may run on several host threads (OpenMP), with bit-identical results.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Host threads for the independent rows of a matrix-vector product (1 unless the library was
   built with OpenMP). Each row's sum runs in the same order on one thread, so every result is
   bit-identical for any thread count. */
void orc_set_threads(int32_t n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : 1);
#else
  (void)n;
#endif
}

int32_t orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------------------------ */
/* Element codecs                                                                              */
/* ------------------------------------------------------------------------------------------ */

/* OCP 8-bit floating point, E4M3 ("fn": no infinities, one NaN pattern S.1111.111):
   bias 7; normal (-1)^s * 2^(e-7) * (1 + m/8); subnormal (e == 0) (-1)^s * 2^-6 * (m/8). */
double orc_e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* bf16 is the upper half of an IEEE binary32. */
double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double straight to bf16 (8 significant bits, exponent range of binary32), ties to
   even, without passing through binary32 (which would round twice). */
uint16_t orc_bf16_bits(double v) {
  if (isnan(v)) return 0x7FC0;
  int neg = signbit(v) ? 1 : 0;
  double a = fabs(v);
  uint16_t out;
  if (a == 0.0) {
    out = 0;
  } else if (isinf(a)) {
    out = 0x7F80;
  } else {
    int ex;
    frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1): unbiased exponent ex - 1 */
    int unb = ex - 1;
    int q = (unb < -126) ? -133 : unb - 7; /* exponent of one unit in the last place */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r >= ldexp(1.0, 128)) {
      out = 0x7F80;
    } else {
      float f = (float)r; /* exact: r has at most 8 significant bits */
      uint32_t u;
      memcpy(&u, &f, 4);
      out = (uint16_t)(u >> 16);
    }
  }
  return (uint16_t)(out | (neg ? 0x8000 : 0));
}

double orc_bf16_round(double v) { return orc_bf16_value(orc_bf16_bits(v)); }

/* ------------------------------------------------------------------------------------------ */
/* Building blocks                                                                             */
/* ------------------------------------------------------------------------------------------ */

static double g_e4m3[256];
static int g_e4m3_ready = 0;

static void e4m3_table(void) {
  if (g_e4m3_ready) return;
  for (int c = 0; c < 256; ++c) g_e4m3[c] = orc_e4m3_value((uint8_t)c);
  g_e4m3_ready = 1;
}

/* FP8 block-scaled matrix-vector product: y[r] = sum_b S[r/128][b] * sum_{c in block b}
   e4m3(W[r][c]) * x[c]. The block scale multiplies the block's partial sum, which equals
   scaling every element of the block. */
void orc_gemv(const orc_mat* m, const double* x, double* y) {
  e4m3_table();
  int kb_n = (m->k + 127) / 128;
#pragma omp parallel for schedule(static) if (m->n >= 256)
  for (int r = 0; r < m->n; ++r) {
    const uint8_t* row = m->w + (size_t)r * m->k;
    double acc = 0.0;
    for (int b = 0; b < kb_n; ++b) {
      int c0 = b * 128, c1 = c0 + 128 < m->k ? c0 + 128 : m->k;
      double part = 0.0;
      for (int c = c0; c < c1; ++c) part += g_e4m3[row[c]] * x[c];
      acc += (double)m->s[(size_t)(r / 128) * kb_n + b] * part;
    }
    y[r] = acc;
  }
}

/* RMSNorm with a bf16 weight, output rounded to bf16: out = bf16((x / sqrt(mean(x^2) + eps)) * w).
   (Plainest reading: the normalised GEMV input is a bf16 activation.) */
void orc_rmsnorm(const double* x, const uint16_t* w, int32_t n, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; ++i) out[i] = orc_bf16_round((x[i] * inv) * orc_bf16_value(w[i]));
}

/* Rotary position embedding, half-split ("rotate half") pairing: element i pairs with
   i + head_dim/2, angle pos * theta^(-2i/head_dim). (Plainest reading; the pages do not fix the
   variant.) */
void orc_rope(double* v, int32_t head_dim, int32_t pos, double theta) {
  int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = pow(theta, -2.0 * (double)i / (double)head_dim);
    double ang = (double)pos * inv_freq;
    double c = cos(ang), s = sin(ang);
    double a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = b * c + a * s;
  }
}

/* One query head against n_keys cached keys/values (bf16 rows of head_dim):
   o = softmax(q . K^T / sqrt(head_dim)) V, softmax with the maximum subtracted. Unrounded. */
void orc_attention_head(const double* q, const uint16_t* k, const uint16_t* v, int32_t n_keys,
                        int32_t head_dim, double* o) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
  double scale = 1.0 / sqrt((double)head_dim);
  double mx = -INFINITY;
  for (int j = 0; j < n_keys; ++j) {
    double d = 0.0;
    for (int i = 0; i < head_dim; ++i) d += q[i] * orc_bf16_value(k[(size_t)j * head_dim + i]);
    s[j] = d * scale;
    if (s[j] > mx) mx = s[j];
  }
  double l = 0.0;
  for (int j = 0; j < n_keys; ++j) {
    s[j] = exp(s[j] - mx);
    l += s[j];
  }
  for (int i = 0; i < head_dim; ++i) {
    double acc = 0.0;
    for (int j = 0; j < n_keys; ++j) acc += s[j] * orc_bf16_value(v[(size_t)j * head_dim + i]);
    o[i] = n_keys > 0 ? acc / l : 0.0;
  }
  free(s);
}

/* Sigmoid router: score = 1 / (1 + exp(-logit)); the top_k experts by score (descending, ties
   to the lower expert index); gates = score / sum of the selected scores. No score bias, no
   group limit, routed scaling 1 (plainest reading). */
void orc_router_topk(const double* logits, int32_t n_experts, int32_t top_k, int32_t* idx,
                     double* gate, double* score) {
  double* sc = (double*)malloc(sizeof(double) * (size_t)n_experts);
  char* taken = (char*)calloc((size_t)n_experts, 1);
  for (int e = 0; e < n_experts; ++e) sc[e] = 1.0 / (1.0 + exp(-logits[e]));
  double sum = 0.0;
  for (int j = 0; j < top_k; ++j) {
    int best = -1;
    for (int e = 0; e < n_experts; ++e)
      if (!taken[e] && (best < 0 || sc[e] > sc[best])) best = e;
    taken[best] = 1;
    idx[j] = best;
    sum += sc[best];
  }
  for (int j = 0; j < top_k; ++j) gate[j] = sc[idx[j]] / sum;
  if (score)
    for (int e = 0; e < n_experts; ++e) score[e] = sc[e];
  free(sc);
  free(taken);
}

/* SwiGLU expert: h = bf16(silu(W_gate x) * (W_up x)), silu(a) = a / (1 + exp(-a)); y = W_down h. */
void orc_swiglu_expert(const orc_mat* gate, const orc_mat* up, const orc_mat* down,
                       const double* xn, double* y) {
  int inter = gate->n;
  double* a = (double*)malloc(sizeof(double) * (size_t)inter);
  double* b = (double*)malloc(sizeof(double) * (size_t)inter);
  double* h = (double*)malloc(sizeof(double) * (size_t)inter);
  orc_gemv(gate, xn, a);
  orc_gemv(up, xn, b);
  for (int j = 0; j < inter; ++j) h[j] = orc_bf16_round((a[j] / (1.0 + exp(-a[j]))) * b[j]);
  orc_gemv(down, h, y);
  free(a);
  free(b);
  free(h);
}

int32_t orc_argmax(const double* v, int32_t n) {
  int best = 0;
  for (int i = 1; i < n; ++i)
    if (v[i] > v[best]) best = i;
  return best;
}

/* ------------------------------------------------------------------------------------------ */
/* Decoder layer                                                                               */
/* ------------------------------------------------------------------------------------------ */

static size_t kv_index(const orc_cfg* c, int max_ctx, int layer, int g, int pos) {
  return (((size_t)layer * c->n_kv_heads + g) * (size_t)max_ctx + pos) * c->head_dim;
}

/* Attention input: RMSNorm, q/k/v projections, RoPE on q and k, bf16 rounding of q, k, v.
   Outputs bf16 values: q [n_heads*head_dim], k and v [n_kv_heads*head_dim]. */
static void qkv_project(const orc_model* m, int layer, const double* x, int pos, double* q,
                        double* k, double* v) {
  const orc_cfg* c = &m->cfg;
  const orc_layer* L = &m->layers[layer];
  int d = c->hidden, hd = c->head_dim;
  double* xn = (double*)malloc(sizeof(double) * (size_t)d);
  orc_rmsnorm(x, L->attn_norm, d, c->rms_eps, xn);
  orc_gemv(&L->wq, xn, q);
  orc_gemv(&L->wk, xn, k);
  orc_gemv(&L->wv, xn, v);
  for (int h = 0; h < c->n_heads; ++h) orc_rope(q + (size_t)h * hd, hd, pos, c->rope_theta);
  for (int g = 0; g < c->n_kv_heads; ++g) orc_rope(k + (size_t)g * hd, hd, pos, c->rope_theta);
  for (int i = 0; i < c->n_heads * hd; ++i) q[i] = orc_bf16_round(q[i]);
  for (int i = 0; i < c->n_kv_heads * hd; ++i) {
    k[i] = orc_bf16_round(k[i]);
    v[i] = orc_bf16_round(v[i]);
  }
  free(xn);
}

/* The rest of the layer for one position whose keys/values 0..n_keys-1 sit in kc/vc
   (layer-local, [n_kv_heads][ctx][head_dim] with row stride ctx): GQA attention, output
   projection + residual, RMSNorm, FFN (dense SwiGLU or routed top-k + shared experts) +
   residual. x is updated in place (bf16 values). */
static void attn_and_ffn(const orc_model* m, int layer, double* x, const double* q,
                         const uint16_t* kc, const uint16_t* vc, int ctx, int n_keys,
                         orc_trace* tr) {
  const orc_cfg* c = &m->cfg;
  const orc_layer* L = &m->layers[layer];
  int d = c->hidden, hd = c->head_dim, hq = c->n_heads, hkv = c->n_kv_heads;
  int group = hq / hkv;
  double* o = (double*)malloc(sizeof(double) * (size_t)hq * hd);
  double* a = (double*)malloc(sizeof(double) * (size_t)d);
  double* xn = (double*)malloc(sizeof(double) * (size_t)d);
  double* y = (double*)calloc((size_t)d, sizeof(double));
  double* ye = (double*)malloc(sizeof(double) * (size_t)d);

  for (int h = 0; h < hq; ++h) {
    int g = h / group; /* query head h reads KV head h / (n_heads / n_kv_heads) */
    orc_attention_head(q + (size_t)h * hd, kc + (size_t)g * ctx * hd, vc + (size_t)g * ctx * hd,
                       n_keys, hd, o + (size_t)h * hd);
  }
  for (int i = 0; i < hq * hd; ++i) o[i] = orc_bf16_round(o[i]);
  if (tr && tr->attn_out) memcpy(tr->attn_out + (size_t)layer * hq * hd, o, sizeof(double) * hq * hd);

  orc_gemv(&L->wo, o, a);
  for (int i = 0; i < d; ++i) x[i] = orc_bf16_round(x[i] + a[i]);

  orc_rmsnorm(x, L->ffn_norm, d, c->rms_eps, xn);
  if (c->dense_ffn > 0) {
    orc_swiglu_expert(&L->fgate, &L->fup, &L->fdown, xn, y);
  } else {
    int E = c->n_experts, K = c->top_k;
    double* r = (double*)malloc(sizeof(double) * (size_t)E);
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
    double* gt = (double*)malloc(sizeof(double) * (size_t)K);
    double* sc = (double*)malloc(sizeof(double) * (size_t)E);
    orc_gemv(&L->router, xn, r);
    orc_router_topk(r, E, K, idx, gt, sc);
    if (tr && tr->topk_idx) memcpy(tr->topk_idx + (size_t)layer * K, idx, sizeof(int32_t) * K);
    if (tr && tr->topk_gate) memcpy(tr->topk_gate + (size_t)layer * K, gt, sizeof(double) * K);
    if (tr && tr->router_score) memcpy(tr->router_score + (size_t)layer * E, sc, sizeof(double) * E);
    for (int j = 0; j < K; ++j) {
      int e = idx[j];
      orc_swiglu_expert(&L->gate[e], &L->up[e], &L->down[e], xn, ye);
      for (int i = 0; i < d; ++i) y[i] += gt[j] * ye[i];
    }
    for (int s = 0; s < c->n_shared; ++s) {
      orc_swiglu_expert(&L->sgate[s], &L->sup[s], &L->sdown[s], xn, ye);
      for (int i = 0; i < d; ++i) y[i] += ye[i];
    }
    free(r);
    free(idx);
    free(gt);
    free(sc);
  }
  for (int i = 0; i < d; ++i) x[i] = orc_bf16_round(x[i] + y[i]);
  if (tr && tr->layer_out) memcpy(tr->layer_out + (size_t)layer * d, x, sizeof(double) * d);

  free(o);
  free(a);
  free(xn);
  free(y);
  free(ye);
}

int32_t orc_layer_step(const orc_model* m, int32_t layer, double* x, int32_t pos, orc_kv* kv,
                       orc_trace* tr) {
  const orc_cfg* c = &m->cfg;
  int hd = c->head_dim;
  if (pos < 0 || pos >= kv->max_ctx) return -1;
  double* q = (double*)malloc(sizeof(double) * (size_t)c->n_heads * hd);
  double* k = (double*)malloc(sizeof(double) * (size_t)c->n_kv_heads * hd);
  double* v = (double*)malloc(sizeof(double) * (size_t)c->n_kv_heads * hd);
  qkv_project(m, layer, x, pos, q, k, v);
  for (int g = 0; g < c->n_kv_heads; ++g)
    for (int i = 0; i < hd; ++i) {
      size_t at = kv_index(c, kv->max_ctx, layer, g, pos) + i;
      kv->k[at] = orc_bf16_bits(k[(size_t)g * hd + i]);
      kv->v[at] = orc_bf16_bits(v[(size_t)g * hd + i]);
    }
  attn_and_ffn(m, layer, x, q, kv->k + kv_index(c, kv->max_ctx, layer, 0, 0),
               kv->v + kv_index(c, kv->max_ctx, layer, 0, 0), kv->max_ctx, pos + 1, tr);
  free(q);
  free(k);
  free(v);
  return 0;
}

static void final_logits(const orc_model* m, const double* x, double* logits) {
  const orc_cfg* c = &m->cfg;
  double* xn = (double*)malloc(sizeof(double) * (size_t)c->hidden);
  orc_rmsnorm(x, m->final_norm, c->hidden, c->rms_eps, xn);
  orc_gemv(&m->lm_head, xn, logits);
  free(xn);
}

int32_t orc_decode_step(const orc_model* m, int32_t token, const uint16_t* hidden, int32_t pos,
                        orc_kv* kv, double* logits, uint16_t* hidden_out, orc_trace* tr) {
  const orc_cfg* c = &m->cfg;
  int d = c->hidden;
  double* x = (double*)malloc(sizeof(double) * (size_t)d);
  for (int i = 0; i < d; ++i)
    x[i] = hidden ? orc_bf16_value(hidden[i]) : orc_bf16_value(m->embed[(size_t)token * d + i]);
  for (int l = 0; l < c->n_layers; ++l)
    if (orc_layer_step(m, l, x, pos, kv, tr) != 0) {
      free(x);
      return -2;
    }
  if (hidden_out)
    for (int i = 0; i < d; ++i) hidden_out[i] = orc_bf16_bits(x[i]);
  int32_t tok = -1;
  if (c->vocab > 0) {
    double* lg = logits ? logits : (double*)malloc(sizeof(double) * (size_t)c->vocab);
    final_logits(m, x, lg);
    tok = orc_argmax(lg, c->vocab);
    if (!logits) free(lg);
  }
  free(x);
  return tok;
}

/* Layer-major recomputation: every layer runs over all n positions before the next layer, with
   a fresh layer-local cache. Each position sees exactly the keys 0..p, so the result must equal
   the incremental (position-major) decode. */
int32_t orc_full_recompute(const orc_model* m, const int32_t* tokens, int32_t n, double* logits) {
  const orc_cfg* c = &m->cfg;
  int d = c->hidden, hd = c->head_dim, hq = c->n_heads, hkv = c->n_kv_heads;
  double* X = (double*)malloc(sizeof(double) * (size_t)n * d);
  double* Q = (double*)malloc(sizeof(double) * (size_t)n * hq * hd);
  double* kk = (double*)malloc(sizeof(double) * (size_t)hkv * hd);
  double* vv = (double*)malloc(sizeof(double) * (size_t)hkv * hd);
  uint16_t* kc = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)hkv * n * hd);
  uint16_t* vc = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)hkv * n * hd);
  for (int p = 0; p < n; ++p)
    for (int i = 0; i < d; ++i) X[(size_t)p * d + i] = orc_bf16_value(m->embed[(size_t)tokens[p] * d + i]);
  for (int l = 0; l < c->n_layers; ++l) {
    for (int p = 0; p < n; ++p) {
      qkv_project(m, l, X + (size_t)p * d, p, Q + (size_t)p * hq * hd, kk, vv);
      for (int g = 0; g < hkv; ++g)
        for (int i = 0; i < hd; ++i) {
          kc[((size_t)g * n + p) * hd + i] = orc_bf16_bits(kk[(size_t)g * hd + i]);
          vc[((size_t)g * n + p) * hd + i] = orc_bf16_bits(vv[(size_t)g * hd + i]);
        }
    }
    for (int p = 0; p < n; ++p)
      attn_and_ffn(m, l, X + (size_t)p * d, Q + (size_t)p * hq * hd, kc, vc, n, p + 1, NULL);
  }
  final_logits(m, X + (size_t)(n - 1) * d, logits);
  int32_t tok = orc_argmax(logits, c->vocab);
  free(X);
  free(Q);
  free(kk);
  free(vv);
  free(kc);
  free(vc);
  return tok;
}
