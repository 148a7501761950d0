/*
 * CPU oracle for the Grok-1 top-2-of-8 Mixture-of-Experts feed-forward layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * of the package entry file and the CPU-baseline leg of the benchmark may load
 * or run this file.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only through the arrays of the seeded input generator.
 *
 * What it computes, written as plain loops in the order the sources give it:
 *
 *   xn   = RMSNorm_pre(x)                      pre-MoE RMSNorm
 *   l_e  = <xn, G_e> (+ b_e)                   router logits, e = 0..7
 *   p    = softmax(l)                          router probabilities
 *   i0, i1 = top_k(p, 2)                       ties go to the lower index
 *   o_r  = W1_e (GELU(W_e xn) * (Wv_e xn))     GeGLU expert FFN, e = i_r
 *   m    = p_i0 o_0 + p_i1 o_1                 probability-weighted combine
 *   y    = x + RMSNorm_post(m)                 post-MoE RMSNorm, residual add
 *
 * Sources (page title, section):
 *  - "Jah-yee/grok" README, architecture diagram: MoE FFN with 8 experts and
 *    top-2 routing, expert form GELU(x W) (*) (x Wv) followed by an output
 *    projection; RMSNorm; list item "Gated GELU".
 *  - "Grok-1: 314B Total Parameters, 25B Active Per Token (MoE Explained)"
 *    (oneruby-dev blog), section "Expert Routing Details": the
 *    router applies softmax to the gate logits and takes jax.lax.top_k(k=2) of
 *    the softmax outputs, returning those gates unrenormalised; the gating
 *    noise is for training only.  Section "How MoE Works in Practice": each
 *    expert output is multiplied by its gate weight and the results summed.
 *    Section "Why JAX Instead of PyTorch" (block listing): normalised input to
 *    the MoE sublayer, then x + sublayer output.
 *  - "TevunahAi/Grok-1-BF16" model card, "Grok-1 Specific Behaviors": four
 *    norms per layer, pre-MoE and post-MoE among them; "Weight Verification":
 *    expert tensors linear / linear_v [32768, 6144] and linear_1 [6144, 32768]
 *    in PyTorch [out, in] order, gate [8, 6144], norm scales [6144];
 *    "Conversion Details": int8 weights times bf16 scales with grouped scale
 *    broadcasting, scale shapes (1,N), (8,N), (8,1,N), (8,8,N), transposed from
 *    JAX [in, out] to PyTorch [out, in].
 *
 * Readings where the sources are silent:
 *  - GELU is the tanh approximation 0.5 u (1 + tanh(sqrt(2/pi)(u + 0.044715 u^3))).
 *  - RMSNorm(v) = v / sqrt(mean(v^2) + eps) * scale, scale applied as is.
 *  - The router sees the unrounded pre-norm output; ties in top-2 go to the
 *    lower expert index; no capacity limit, no token dropping.
 *  - The top-2 decision is taken on the probabilities rounded to fp32 (the
 *    precision the GPU kernel decides in); every value is otherwise computed in
 *    fp64 and the combine weights are the fp64 probabilities.
 *  - Grouped scale rule for a weight viewed in JAX order [E, K_in, N] with scale
 *    shape (E_s, G, N): w[e,k,n] = q[e,k,n] * s[E_s > 1 ? e : 0, k / (K_in/G), n].
 *    The int8 x bf16 product is exact in fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_W_BF16 0
#define ORACLE_W_INT8 1

static inline float bf16_bits_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Threads the OpenMP loops of this file use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* One expert-stacked weight tensor, stored [E, N, K] (PyTorch [out, in]). */
typedef struct {
  int32_t dtype;          /* ORACLE_W_BF16 or ORACLE_W_INT8 */
  const void* q;          /* bf16 bits (uint16) or int8, [E, N, K] */
  const uint16_t* scale;  /* int8 only: bf16 bits, logical shape (scale_E, scale_G, N) */
  int32_t scale_E;        /* 1 (shared by experts) or E */
  int32_t scale_G;        /* number of groups along K_in; 1 = one scale per output channel */
  int64_t N, K;
} oracle_weight_t;

/* Dequantised weight element w[e, n, k] ("Conversion Details": int8 x bf16 scale,
 * grouped broadcasting).  The fp32 product of an 8-bit integer and an 8-bit-
 * mantissa bf16 is exact. */
static inline double weight_at(const oracle_weight_t* W, int64_t e, int64_t n, int64_t k) {
  int64_t off = (e * W->N + n) * W->K + k;
  if (W->dtype == ORACLE_W_BF16) return (double)bf16_bits_to_float(((const uint16_t*)W->q)[off]);
  int64_t es = (W->scale_E > 1) ? e : 0;
  int64_t g = k / (W->K / W->scale_G);
  float s = bf16_bits_to_float(W->scale[(es * W->scale_G + g) * W->N + n]);
  float v = (float)((const int8_t*)W->q)[off] * s;
  return (double)v;
}

/* Full dequantisation of one weight tensor to fp32 [E, N, K] (for checks). */
void oracle_dequant(int32_t dtype, const void* q, const uint16_t* scale, int32_t scale_E, int32_t scale_G,
                    int64_t E, int64_t N, int64_t K, float* out) {
  oracle_weight_t W = {dtype, q, scale, scale_E, scale_G, N, K};
  for (int64_t e = 0; e < E; ++e)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t k = 0; k < K; ++k) out[(e * N + n) * K + k] = (float)weight_at(&W, e, n, k);
}

/* GELU, tanh approximation ("Jah-yee/grok" README: gated GELU; the tanh form is
 * the reading taken where the page names only "GELU"). */
double oracle_gelu_tanh(double u) {
  const double c = 0.79788456080286535588; /* sqrt(2/pi) */
  return 0.5 * u * (1.0 + tanh(c * (u + 0.044715 * u * u * u)));
}

/* RMSNorm: out_j = v_j / sqrt(mean_i v_i^2 + eps) * s_j. */
void oracle_rmsnorm(int64_t n, const double* v, const double* s, double eps, double* out) {
  double ss = 0.0;
  for (int64_t j = 0; j < n; ++j) ss += v[j] * v[j];
  double r = 1.0 / sqrt(ss / (double)n + eps);
  for (int64_t j = 0; j < n; ++j) out[j] = v[j] * r * s[j];
}

/* Router for one token: pre-norm, logits, softmax, top-2 ("Expert Routing
 * Details": softmax(gate(x)), then top_k(k=2) of the softmax outputs). */
static void route_one(int64_t d, int64_t E, const uint16_t* x_row, const float* gate, const float* bias,
                      const float* s_pre, double eps, double* xn, double* p, int32_t* idx2, double* w2) {
  double ss = 0.0;
  for (int64_t j = 0; j < d; ++j) {
    double xj = (double)bf16_bits_to_float(x_row[j]);
    ss += xj * xj;
  }
  double r = 1.0 / sqrt(ss / (double)d + eps);
  for (int64_t j = 0; j < d; ++j) xn[j] = (double)bf16_bits_to_float(x_row[j]) * r * (double)s_pre[j];

  double l[64]; /* E <= 64 */
  for (int64_t e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int64_t j = 0; j < d; ++j) acc += xn[j] * (double)gate[e * d + j];
    l[e] = acc + (bias ? (double)bias[e] : 0.0);
  }
  double mx = l[0];
  for (int64_t e = 1; e < E; ++e)
    if (l[e] > mx) mx = l[e];
  double Z = 0.0;
  for (int64_t e = 0; e < E; ++e) {
    p[e] = exp(l[e] - mx);
    Z += p[e];
  }
  for (int64_t e = 0; e < E; ++e) p[e] /= Z;

  /* top-2 on the fp32-rounded probabilities, ties to the lower index */
  int32_t i0 = 0;
  for (int64_t e = 1; e < E; ++e)
    if ((float)p[e] > (float)p[i0]) i0 = (int32_t)e;
  int32_t i1 = (i0 == 0) ? 1 : 0;
  for (int64_t e = 0; e < E; ++e)
    if (e != i0 && (float)p[e] > (float)p[i1]) i1 = (int32_t)e;
  idx2[0] = i0;
  idx2[1] = i1;
  w2[0] = p[i0];
  w2[1] = p[i1];
}

/* Router over all T tokens.  xn_out [T, d] may be NULL. */
void oracle_route(int64_t T, int64_t d, int64_t E, const uint16_t* x, const float* gate, const float* bias,
                  const float* s_pre, double eps, double* xn_out, double* p_out, int32_t* idx_out, double* w_out) {
#pragma omp parallel
  {
    double* xn_local = (double*)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      double* xn = xn_out ? xn_out + t * d : xn_local;
      route_one(d, E, x + t * d, gate, bias, s_pre, eps, xn, p_out + t * E, idx_out + 2 * t, w_out + 2 * t);
    }
    free(xn_local);
  }
}

/* Routing diagnostics over T tokens ("Jah-yee/grok" README, list "New metrics
 * track MoE-specific grokking signals" (routing entropy, collapse index) and the
 * --demo block "[3] MoE routing (layer 0)", which prints one weight per expert
 * and the routing entropy against its maximum):
 *   out[e]     = (1/T) sum_t p[t, e]              mean router probability of expert e
 *   out[E]     = -sum_e out[e] ln out[e]          routing entropy in nats (max ln E)
 *   out[E + 1] = 1 - out[E] / ln E                collapse index (reading: 0 uniform,
 *                                                 1 when one expert takes all)
 * Terms with out[e] == 0 contribute 0 to the entropy. */
void oracle_routing_stats(int64_t T, int64_t E, const double* p, double* out) {
  for (int64_t e = 0; e < E; ++e) {
    double s = 0.0;
    for (int64_t t = 0; t < T; ++t) s += p[t * E + e];
    out[e] = s / (double)T;
  }
  double h = 0.0;
  for (int64_t e = 0; e < E; ++e)
    if (out[e] > 0.0) h -= out[e] * log(out[e]);
  out[E] = h;
  out[E + 1] = 1.0 - h / log((double)E);
}

/* One GeGLU expert on one token ("Jah-yee/grok" README: GELU(x W) (*) (x Wv),
 * then the output projection; shapes from the model card's weight listing).
 *   h_n = sum_k W[e,n,k] xn_k,  v_n = sum_k Wv[e,n,k] xn_k,  a_n = GELU(h_n) v_n,
 *   o_j = sum_n W1[e,j,n] a_n.
 * h, v, a are [F] and o is [d]; h, v may be NULL. */
static void expert_ffn(int64_t d, int64_t F, int64_t e, const double* xn, const oracle_weight_t* W,
                       const oracle_weight_t* Wv, const oracle_weight_t* W1, double* h, double* v, double* a,
                       double* o) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < F; ++n) {
    double hn = 0.0, vn = 0.0;
    for (int64_t k = 0; k < d; ++k) {
      hn += weight_at(W, e, n, k) * xn[k];
      vn += weight_at(Wv, e, n, k) * xn[k];
    }
    if (h) h[n] = hn;
    if (v) v[n] = vn;
    a[n] = oracle_gelu_tanh(hn) * vn;
  }
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < d; ++j) {
    double oj = 0.0;
    for (int64_t n = 0; n < F; ++n) oj += weight_at(W1, e, j, n) * a[n];
    o[j] = oj;
  }
}

static void fill_weights(int32_t dtype, int64_t d, int64_t F, const void* w, const void* wv, const void* w1,
                         const uint16_t* sw, const uint16_t* swv, const uint16_t* sw1, int32_t scale_E,
                         int32_t scale_G_up, int32_t scale_G_down, oracle_weight_t* W, oracle_weight_t* Wv,
                         oracle_weight_t* W1) {
  oracle_weight_t a = {dtype, w, sw, scale_E, scale_G_up, F, d};
  oracle_weight_t b = {dtype, wv, swv, scale_E, scale_G_up, F, d};
  oracle_weight_t c = {dtype, w1, sw1, scale_E, scale_G_down, d, F};
  *W = a;
  *Wv = b;
  *W1 = c;
}

/* One expert's FFN intermediates for one pre-normed token vector xn [d]. */
void oracle_expert_ffn(int64_t d, int64_t F, int64_t e, const double* xn, int32_t dtype, const void* w,
                       const void* wv, const void* w1, const uint16_t* sw, const uint16_t* swv,
                       const uint16_t* sw1, int32_t scale_E, int32_t scale_G_up, int32_t scale_G_down, double* h,
                       double* v, double* a, double* o) {
  oracle_weight_t W, Wv, W1;
  fill_weights(dtype, d, F, w, wv, w1, sw, swv, sw1, scale_E, scale_G_up, scale_G_down, &W, &Wv, &W1);
  expert_ffn(d, F, e, xn, &W, &Wv, &W1, h, v, a, o);
}

/* The whole layer for a list of tokens (any subset of the T rows of x).
 * Outputs, per listed token i: y [n, d] = x + RMSNorm_post(m), m [n, d] (may be
 * NULL), idx [n, 2], w [n, 2] (combine weights), p [n, E] (probabilities).
 * scratch must hold 2 * F + 3 * d doubles. */
void oracle_moe_tokens(int64_t n_tok, const int64_t* tok, int64_t d, int64_t F, int64_t E, const uint16_t* x,
                       const float* gate, const float* bias, const float* s_pre, const float* s_post, double eps,
                       int32_t dtype, const void* w, const void* wv, const void* w1, const uint16_t* sw,
                       const uint16_t* swv, const uint16_t* sw1, int32_t scale_E, int32_t scale_G_up,
                       int32_t scale_G_down, double* y, double* m_out, int32_t* idx, double* wts, double* p,
                       double* scratch) {
  oracle_weight_t W, Wv, W1;
  fill_weights(dtype, d, F, w, wv, w1, sw, swv, sw1, scale_E, scale_G_up, scale_G_down, &W, &Wv, &W1);
  double* a = scratch;       /* [F] */
  double* xn = a + F;        /* [d] */
  double* o = xn + d;        /* [d] */
  double* m = o + d;         /* [d] */
  for (int64_t i = 0; i < n_tok; ++i) {
    int64_t t = tok[i];
    const uint16_t* x_row = x + t * d;
    route_one(d, E, x_row, gate, bias, s_pre, eps, xn, p + i * E, idx + 2 * i, wts + 2 * i);
    for (int64_t j = 0; j < d; ++j) m[j] = 0.0;
    for (int r = 0; r < 2; ++r) {
      int64_t e = idx[2 * i + r];
      expert_ffn(d, F, e, xn, &W, &Wv, &W1, NULL, NULL, a, o);
      for (int64_t j = 0; j < d; ++j) m[j] += wts[2 * i + r] * o[j];
    }
    if (m_out)
      for (int64_t j = 0; j < d; ++j) m_out[i * d + j] = m[j];
    /* y = x + RMSNorm_post(m) */
    double ss = 0.0;
    for (int64_t j = 0; j < d; ++j) ss += m[j] * m[j];
    double rr = 1.0 / sqrt(ss / (double)d + eps);
    for (int64_t j = 0; j < d; ++j)
      y[i * d + j] = (double)bf16_bits_to_float(x_row[j]) + m[j] * rr * (double)s_post[j];
  }
}

/* ===================================================================== */
/* Attention half of a Grok-1 decoder layer (the block before the MoE one).
 *
 * Sources (page title, section): "Jah-yee/grok" README, architecture diagram
 * (GQA with 48 query and 8 key/value heads, rotary position embeddings,
 * RMSNorm) and references (Su et al., "RoFormer: Enhanced Transformer with
 * Rotary Position Embedding"); "TevunahAi/Grok-1-BF16" model card, "Grok-1
 * Specific Behaviors" (attention logits hard-clamped to [-30, 30] before the
 * softmax; pre- and post-attention norms) and "Weight Verification" (q_proj
 * [6144, 6144], k_proj and v_proj [1024, 6144], o_proj [6144, 6144] in
 * PyTorch [out, in] order, so the head dimension is 6144 / 48 = 128).
 *
 * For one causal sequence x [T, d] and every requested token t:
 *   xn_t  = RMSNorm_pre(x_t)
 *   q_t   = RoPE_t(Wq xn_t),  k_j = RoPE_j(Wk xn_j),  v_j = Wv xn_j   (per head)
 *   s_hj  = clamp(<q_t,h, k_j,g(h)> / sqrt(Dh), -c, c),  j = 0..t,  g(h) = h / (Hq / Hkv)
 *   ctx_h = sum_j softmax_j(s_h) v_j,g(h)
 *   y_t   = x_t + RMSNorm_post(Wo ctx_t)
 * Readings where the pages are silent: RoPE as in RoFormer, rotating the
 * pairs (2i, 2i + 1) of each head by angle pos * base^(-2i / Dh), base 10000;
 * logits scaled by 1/sqrt(Dh) before the clamp; a causal mask; query head h
 * uses key/value head h / (Hq / Hkv); head h is rows [Dh h, Dh (h + 1)) of the
 * projection; the residual around the post-norm as in the MoE half. */

/* RoPE of one head vector v [Dh] at position pos, in place. */
void oracle_rope(int64_t Dh, double* v, int64_t pos, double base) {
  for (int64_t i = 0; i < Dh / 2; ++i) {
    const double theta = pow(base, -2.0 * (double)i / (double)Dh);
    const double a = (double)pos * theta;
    const double c = cos(a), s = sin(a);
    const double x0 = v[2 * i], x1 = v[2 * i + 1];
    v[2 * i] = x0 * c - x1 * s;
    v[2 * i + 1] = x0 * s + x1 * c;
  }
}

/* xn = x_row / sqrt(mean(x_row^2) + eps) * s  (x_row bf16 bits) */
static void rmsnorm_bf16_row(int64_t d, const uint16_t* x_row, const float* s, double eps, double* xn) {
  double ss = 0.0;
  for (int64_t j = 0; j < d; ++j) {
    const double v = (double)bf16_bits_to_float(x_row[j]);
    ss += v * v;
  }
  const double r = 1.0 / sqrt(ss / (double)d + eps);
  for (int64_t j = 0; j < d; ++j) xn[j] = (double)bf16_bits_to_float(x_row[j]) * r * (double)s[j];
}

/* out[n] = sum_k W[n, k] v[k] for a bf16 matrix W [N, K] */
static void matvec_bf16(int64_t N, int64_t K, const uint16_t* W, const double* v, double* out) {
  for (int64_t n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += (double)bf16_bits_to_float(W[n * K + k]) * v[k];
    out[n] = acc;
  }
}

/* y [n_tok, d] of the attention block for the tokens tok[] of the sequence x [T, d];
 * ctx_out [n_tok, Hq Dh] (attention output before o_proj) may be NULL. */
void oracle_attn_tokens(int64_t n_tok, const int64_t* tok, int64_t T, int64_t d, int64_t Hq, int64_t Hkv,
                        int64_t Dh, const uint16_t* x, const float* s_pre, const float* s_post, double eps,
                        const uint16_t* wq, const uint16_t* wk, const uint16_t* wv, const uint16_t* wo,
                        double rope_base, double clamp_c, double* y, double* ctx_out) {
  (void)T;
  int64_t tmax = 0;
  for (int64_t i = 0; i < n_tok; ++i)
    if (tok[i] > tmax) tmax = tok[i];
  const int64_t nk = tmax + 1, kvw = Hkv * Dh, qw = Hq * Dh, group = Hq / Hkv;
  double* K = (double*)malloc((size_t)(nk * kvw) * sizeof(double));
  double* V = (double*)malloc((size_t)(nk * kvw) * sizeof(double));
#pragma omp parallel
  {
    double* xn = (double*)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(static)
    for (int64_t t = 0; t < nk; ++t) {
      rmsnorm_bf16_row(d, x + t * d, s_pre, eps, xn);
      matvec_bf16(kvw, d, wk, xn, K + t * kvw);
      matvec_bf16(kvw, d, wv, xn, V + t * kvw);
      for (int64_t g = 0; g < Hkv; ++g) oracle_rope(Dh, K + t * kvw + g * Dh, t, rope_base);
    }
    free(xn);
  }
#pragma omp parallel
  {
    double* xn = (double*)malloc((size_t)d * sizeof(double));
    double* q = (double*)malloc((size_t)qw * sizeof(double));
    double* ctx = (double*)malloc((size_t)qw * sizeof(double));
    double* sc = (double*)malloc((size_t)nk * sizeof(double));
    double* o = (double*)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_tok; ++i) {
      const int64_t t = tok[i];
      rmsnorm_bf16_row(d, x + t * d, s_pre, eps, xn);
      matvec_bf16(qw, d, wq, xn, q);
      for (int64_t h = 0; h < Hq; ++h) oracle_rope(Dh, q + h * Dh, t, rope_base);
      for (int64_t h = 0; h < Hq; ++h) {
        const int64_t g = h / group;
        double mx = -INFINITY;
        for (int64_t j = 0; j <= t; ++j) {
          double s = 0.0;
          for (int64_t c = 0; c < Dh; ++c) s += q[h * Dh + c] * K[j * kvw + g * Dh + c];
          s /= sqrt((double)Dh);
          if (s > clamp_c) s = clamp_c;
          if (s < -clamp_c) s = -clamp_c;
          sc[j] = s;
          if (s > mx) mx = s;
        }
        double z = 0.0;
        for (int64_t j = 0; j <= t; ++j) {
          sc[j] = exp(sc[j] - mx);
          z += sc[j];
        }
        for (int64_t c = 0; c < Dh; ++c) {
          double acc = 0.0;
          for (int64_t j = 0; j <= t; ++j) acc += sc[j] * V[j * kvw + g * Dh + c];
          ctx[h * Dh + c] = acc / z;
        }
      }
      if (ctx_out)
        for (int64_t c = 0; c < qw; ++c) ctx_out[i * qw + c] = ctx[c];
      matvec_bf16(d, qw, wo, ctx, o);
      double ss = 0.0;
      for (int64_t n = 0; n < d; ++n) ss += o[n] * o[n];
      const double rr = 1.0 / sqrt(ss / (double)d + eps);
      for (int64_t n = 0; n < d; ++n)
        y[i * d + n] = (double)bf16_bits_to_float(x[t * d + n]) + o[n] * rr * (double)s_post[n];
    }
    free(xn);
    free(q);
    free(ctx);
    free(sc);
    free(o);
  }
  free(K);
  free(V);
}
