/* oracle.c -- plain, slow, obviously correct CPU decoder for the batch-1 decode step.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * this code. The CUDA library never links, calls or includes it, and it includes nothing of the
 * CUDA library. Inputs come from the seeded generators in synth/, or from the tests themselves.
 *
 * What it computes, and where the method is stated:
 *   - one token through every layer, each weight read once
 *       ("Decoding in tiles" (TileInfer), section 2 "Why decode has a lower bound", Figure 3;
 *        "One launch per token", section "The oracle, then the kernels")
 *   - RMSNorm                         ("LLAMA 1B Optimizing Kernels", section "RMSNorm")
 *   - GEMV y = W x                    ("How I built an LLM inference engine from scratch in CUDA"
 *                                      (tinyinfer), section "The speed limit is memory, not math")
 *   - symmetric int4, zero point 8, one scale per group along the input dimension
 *                                     (tinyinfer, same section: one fp16 scale per 64 weights)
 *   - NEOX half-split RoPE            (flint, the RoPE convention note under the chat demo)
 *   - grouped-query attention, one KV head per group of query heads
 *                                     ("Decoding in tiles", section 2; "LLAMA 1B Optimizing
 *                                      Kernels", section "Grouped Query Attention (GQA)")
 *   - split-K flash-decode partials and their log-sum-exp merge
 *                                     ("One launch per token", section "The attention trap";
 *                                      tinyinfer, "Round 2: attention when eight heads share one K/V")
 *   - SwiGLU MLP and residual adds    ("One launch per token", section "The oracle, then the
 *                                      kernels"; "LLAMA 1B Optimizing Kernels", "Kernel Fusion")
 *   - greedy argmax, lowest token id among ties, error on a non-finite logit
 *                                     ("Decoding in tiles", section 5 "One token, end to end")
 *
 * Readings where the pages are silent or garbled are listed in the design notes and restated in
 * each function below. Loops follow the definitions directly: no blocking, no fusion, every sum in
 * index order, accumulated in orc_real (double by default).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_real_bytes(void) { return (int)sizeof(orc_real); }

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------- scalar formats */

/* bf16 is the top half of an IEEE binary32: the value is exact in double. */
double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* IEEE 754 binary16 from its definition: sign, 5-bit exponent (bias 15), 10-bit fraction. */
double orc_fp16_value(uint16_t bits) {
  int sign = bits >> 15, e = (bits >> 10) & 0x1F, frac = bits & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
  else if (e == 31) v = frac ? NAN : INFINITY;
  else v = ldexp((double)(frac + 1024), e - 25);            /* (1 + frac/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* Round a double to the nearest bf16, ties to even, in one step (no detour through float, which
 * would round twice). bf16: 8-bit significand, exponent range of binary32. */
uint16_t orc_round_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  frexp(a, &e);                             /* a = m * 2^e, m in [0.5, 1) */
  double q = rint(ldexp(a, 8 - e));          /* significand scaled to [128, 256], ties to even */
  if (q == 256.0) { q = 128.0; e += 1; }
  int biased = (e - 1) + 127;                /* a ~= (q/128) * 2^(e-1) */
  if (biased >= 255) return sign | 0x7F80;
  if (biased <= 0) {                         /* subnormal: multiples of 2^-133 */
    double s = rint(ldexp(a, 133));
    return sign | (uint16_t)s;               /* s == 128 lands on the smallest normal */
  }
  return sign | (uint16_t)((biased << 7) | ((int)q - 128));
}

/* ---------------------------------------------------------------- building blocks */

/* RMSNorm: y = x / sqrt(mean(x^2) + eps) * g, gain applied after normalising ("LLAMA 1B
 * Optimizing Kernels", section "RMSNorm"; the formula is the standard Llama one, which the pages
 * name but do not print). */
void orc_rmsnorm(const orc_real* x, const uint16_t* gain, int n, double eps, orc_real* y) {
  orc_real ss = 0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  orc_real inv = (orc_real)(1.0 / sqrt((double)(ss / (orc_real)n) + eps));
  for (int i = 0; i < n; ++i) y[i] = x[i] * inv * (orc_real)orc_bf16_value(gain[i]);
}

/* y[r] = sum_c W[r][c] * x[c], W in bf16 (tinyinfer, "The speed limit is memory, not math"). */
void orc_gemv_bf16(const uint16_t* w, int rows, int cols, const orc_real* x, orc_real* y) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    const uint16_t* row = w + (size_t)r * cols;
    orc_real acc = 0;
    for (int c = 0; c < cols; ++c) acc += (orc_real)orc_bf16_value(row[c]) * x[c];
    y[r] = acc;
  }
}

static double int4_weight(const uint8_t* wq, const uint16_t* scales, int scale_is_bf16, int cols,
                          int group, int r, int c) {
  uint8_t byte = wq[(size_t)r * (cols / 2) + c / 2];
  int q = (c & 1) ? (byte >> 4) : (byte & 0xF);
  uint16_t sb = scales[(size_t)r * (cols / group) + c / group];
  double s = scale_is_bf16 ? orc_bf16_value(sb) : orc_fp16_value(sb);
  return (double)(q - 8) * s;  /* exact: 4-bit integer times an 11- or 8-bit significand */
}

/* Symmetric int4 with zero point 8 and one scale per `group` consecutive inputs of a row
 * (tinyinfer, "The speed limit is memory, not math": 4 bits plus one fp16 scale per 64 weights). */
void orc_dequant_int4(const uint8_t* wq, const uint16_t* scales, int scale_is_bf16, int rows,
                      int cols, int group, orc_real* w_out) {
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < cols; ++c)
      w_out[(size_t)r * cols + c] =
          (orc_real)int4_weight(wq, scales, scale_is_bf16, cols, group, r, c);
}

void orc_gemv_int4(const uint8_t* wq, const uint16_t* scales, int scale_is_bf16, int rows, int cols,
                   int group, const orc_real* x, orc_real* y) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    orc_real acc = 0;
    for (int c = 0; c < cols; ++c)
      acc += (orc_real)int4_weight(wq, scales, scale_is_bf16, cols, group, r, c) * x[c];
    y[r] = acc;
  }
}

/* NEOX half-split rotary embedding (flint, RoPE convention note). For i < d/2 the pair
 * (v[i], v[i+d/2]) is rotated by theta_i = pos * base^(-2i/d):
 *   v[i]     <- v[i] cos - v[i+d/2] sin
 *   v[i+d/2] <- v[i+d/2] cos + v[i] sin
 * The angle, cosine and sine are computed in double. */
void orc_rope(orc_real* v, int head_dim, int pos, double theta) {
  int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)head_dim);
    orc_real c = (orc_real)cos(ang), s = (orc_real)sin(ang);
    orc_real a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = b * c + a * s;
  }
}

/* softmax with the maximum subtracted first */
void orc_softmax(const orc_real* s, int n, orc_real* p) {
  orc_real m = -INFINITY;
  for (int i = 0; i < n; ++i) if (s[i] > m) m = s[i];
  orc_real sum = 0;
  for (int i = 0; i < n; ++i) { p[i] = (orc_real)exp((double)(s[i] - m)); sum += p[i]; }
  for (int i = 0; i < n; ++i) p[i] /= sum;
}

/* KV head used by query head h: contiguous groups of n_heads/n_kv_heads query heads share one KV
 * head ("Decoding in tiles" section 2: 32 query heads share 8 K/V heads). */
static int kv_head_of(int h, int n_heads, int n_kv_heads) {
  return (int)(((long long)h * n_kv_heads) / n_heads);
}

/* Grouped-query attention for one query position over cache slots [0, n_ctx): for each query
 * head h with KV head j, s_t = q_h . K[j][t] / sqrt(d), p = softmax(s), out_h = sum_t p_t V[j][t].
 * k and v point at one layer: [n_kv_heads][ctx_stride][head_dim] bf16. */
void orc_attention(const orc_real* q, const uint16_t* k, const uint16_t* v, int n_heads,
                   int n_kv_heads, int head_dim, int n_ctx, int ctx_stride, orc_real* out) {
  orc_real* s = (orc_real*)malloc(sizeof(orc_real) * (size_t)n_ctx);
  orc_real* p = (orc_real*)malloc(sizeof(orc_real) * (size_t)n_ctx);
  orc_real scale = (orc_real)(1.0 / sqrt((double)head_dim));
  for (int h = 0; h < n_heads; ++h) {
    int j = kv_head_of(h, n_heads, n_kv_heads);
    const orc_real* qh = q + (size_t)h * head_dim;
    for (int t = 0; t < n_ctx; ++t) {
      const uint16_t* kt = k + ((size_t)j * ctx_stride + t) * head_dim;
      orc_real acc = 0;
      for (int i = 0; i < head_dim; ++i) acc += qh[i] * (orc_real)orc_bf16_value(kt[i]);
      s[t] = acc * scale;
    }
    orc_softmax(s, n_ctx, p);
    for (int i = 0; i < head_dim; ++i) {
      orc_real acc = 0;
      for (int t = 0; t < n_ctx; ++t)
        acc += p[t] * (orc_real)orc_bf16_value(v[((size_t)j * ctx_stride + t) * head_dim + i]);
      out[(size_t)h * head_dim + i] = acc;
    }
  }
  free(s);
  free(p);
}

/* Split-K flash-decode, pass 1 ("One launch per token", "The attention trap"; tinyinfer,
 * "Round 2"). Chunk c covers slots [c*chunk_len, min((c+1)*chunk_len, n_ctx)). Per query head h
 * and chunk c: m = max_t s_t, l = sum_t e^(s_t - m), o = sum_t e^(s_t - m) V_t (unnormalised).
 * An empty chunk (past the current length) gives m = -inf, l = 0, o = 0.
 * Outputs: m, l [n_heads][n_chunks]; o [n_heads][n_chunks][head_dim]. */
void orc_attention_partials(const orc_real* q, const uint16_t* k, const uint16_t* v, int n_heads,
                            int n_kv_heads, int head_dim, int n_ctx, int ctx_stride,
                            int chunk_len, int n_chunks, orc_real* m, orc_real* l, orc_real* o) {
  orc_real scale = (orc_real)(1.0 / sqrt((double)head_dim));
  orc_real* s = (orc_real*)malloc(sizeof(orc_real) * (size_t)(chunk_len > 0 ? chunk_len : 1));
  for (int h = 0; h < n_heads; ++h) {
    int j = kv_head_of(h, n_heads, n_kv_heads);
    const orc_real* qh = q + (size_t)h * head_dim;
    for (int c = 0; c < n_chunks; ++c) {
      int t0 = c * chunk_len, t1 = t0 + chunk_len;
      if (t1 > n_ctx) t1 = n_ctx;
      size_t hc = (size_t)h * n_chunks + c;
      orc_real* oc = o + hc * head_dim;
      orc_real mc = -INFINITY, lc = 0;
      for (int i = 0; i < head_dim; ++i) oc[i] = 0;
      for (int t = t0; t < t1; ++t) {
        const uint16_t* kt = k + ((size_t)j * ctx_stride + t) * head_dim;
        orc_real acc = 0;
        for (int i = 0; i < head_dim; ++i) acc += qh[i] * (orc_real)orc_bf16_value(kt[i]);
        s[t - t0] = acc * scale;
        if (s[t - t0] > mc) mc = s[t - t0];
      }
      for (int t = t0; t < t1; ++t) {
        orc_real e = (orc_real)exp((double)(s[t - t0] - mc));
        lc += e;
        const uint16_t* vt = v + ((size_t)j * ctx_stride + t) * head_dim;
        for (int i = 0; i < head_dim; ++i) oc[i] += e * (orc_real)orc_bf16_value(vt[i]);
      }
      m[hc] = mc;
      l[hc] = lc;
    }
  }
  free(s);
}

/* Split-K pass 2, the log-sum-exp merge: M = max_c m_c, w_c = e^(m_c - M) (exactly 0 for an empty
 * chunk, which is skipped so that -inf - (-inf) never occurs), out = sum_c w_c o_c / sum_c w_c l_c
 * ("One launch per token", "The attention trap"). */
void orc_attention_combine(const orc_real* m, const orc_real* l, const orc_real* o, int n_heads,
                           int head_dim, int n_chunks, orc_real* out) {
  for (int h = 0; h < n_heads; ++h) {
    const orc_real* mh = m + (size_t)h * n_chunks;
    orc_real M = -INFINITY;
    for (int c = 0; c < n_chunks; ++c) if (mh[c] > M) M = mh[c];
    orc_real den = 0;
    orc_real* oh = out + (size_t)h * head_dim;
    for (int i = 0; i < head_dim; ++i) oh[i] = 0;
    for (int c = 0; c < n_chunks; ++c) {
      if (mh[c] == -INFINITY) continue;
      orc_real w = (orc_real)exp((double)(mh[c] - M));
      den += w * l[(size_t)h * n_chunks + c];
      const orc_real* oc = o + ((size_t)h * n_chunks + c) * head_dim;
      for (int i = 0; i < head_dim; ++i) oh[i] += w * oc[i];
    }
    for (int i = 0; i < head_dim; ++i) oh[i] /= den;
  }
}

/* a = silu(gate) * up, silu(z) = z / (1 + e^-z) */
void orc_swiglu(const orc_real* gate, const orc_real* up, int n, orc_real* a) {
  for (int i = 0; i < n; ++i) {
    orc_real z = gate[i];
    a[i] = z / ((orc_real)1 + (orc_real)exp(-(double)z)) * up[i];
  }
}

/* Greedy choice: the largest logit, the lowest index among ties; any NaN or infinity is an error
 * ("Decoding in tiles", section 5). On error *idx = -1. */
int orc_argmax(const orc_real* logits, int n, int* idx) {
  int best = -1;
  orc_real bv = 0;
  for (int i = 0; i < n; ++i) {
    if (!isfinite((double)logits[i])) { *idx = -1; return ORC_ERR_NONFINITE; }
    if (best < 0 || logits[i] > bv) { best = i; bv = logits[i]; }
  }
  *idx = best;
  return ORC_OK;
}

/* ---------------------------------------------------------------- the decode step */

static void gemv_any(const orc_model* m, const void* w, const uint16_t* s, int rows, int cols,
                     const orc_real* x, orc_real* y) {
  if (m->weight_format == ORC_INT4)
    orc_gemv_int4((const uint8_t*)w, s, m->scale_is_bf16, rows, cols, m->group_size, x, y);
  else
    orc_gemv_bf16((const uint16_t*)w, rows, cols, x, y);
}

/* One decode step at position `pos` (0-based) for token `token`:
 *   x = E[token]
 *   per layer: n = rmsnorm(x, g1); q,k,v = Wq n (+bq), Wk n (+bk), Wv n (+bv);
 *              RoPE(q_h, pos), RoPE(k_j, pos); K[pos] = bf16(k), V[pos] = bf16(v);
 *              o = attention(q, K[0..pos], V[0..pos]); x += Wo o;
 *              n2 = rmsnorm(x, g2); x += Wd (silu(Wg n2) * (Wu n2))
 *   n_f = rmsnorm(x, g_final); logits = W_lm n_f; argmax.
 * ("Decoding in tiles", section 2, Figure 3; "One launch per token", "The oracle, then the
 * kernels"). The cache must hold slots [0, pos) already. */
/* Gathered-expert SwiGLU MLP ("One launch per token", "The same trick, sparser: a 64-expert MoE"):
 * for each chosen expert i in order, its gate and up projections of x, the SwiGLU of the two, its
 * down projection of that, scaled by weight[i] and added to y. Weights stay in their stored format
 * and are decoded exactly per row, as in the dense linears. */
static void orc_linear(int fmt, int group, int scale_is_bf16, const void* w, const uint16_t* s,
                       size_t expert, int rows, int cols, const orc_real* x, orc_real* y) {
  if (fmt == ORC_INT4)
    orc_gemv_int4((const uint8_t*)w + expert * (size_t)rows * (cols / 2),
                  s + expert * (size_t)rows * (cols / group), scale_is_bf16, rows, cols, group, x, y);
  else
    orc_gemv_bf16((const uint16_t*)w + expert * (size_t)rows * cols, rows, cols, x, y);
}

void orc_moe_mlp(int weight_format, int group, int scale_is_bf16, int hidden, int ffn_e,
                 const void* wg, const uint16_t* sg, const void* wu, const uint16_t* su,
                 const void* wd, const uint16_t* sd, int top_k, const int32_t* ids,
                 const orc_real* weights, const orc_real* x, orc_real* y) {
  orc_real* g = (orc_real*)malloc(sizeof(orc_real) * (size_t)ffn_e);
  orc_real* u = (orc_real*)malloc(sizeof(orc_real) * (size_t)ffn_e);
  orc_real* a = (orc_real*)malloc(sizeof(orc_real) * (size_t)ffn_e);
  orc_real* d = (orc_real*)malloc(sizeof(orc_real) * (size_t)hidden);
  for (int o = 0; o < hidden; ++o) y[o] = 0;
  for (int i = 0; i < top_k; ++i) {
    const size_t e = (size_t)ids[i];
    orc_linear(weight_format, group, scale_is_bf16, wg, sg, e, ffn_e, hidden, x, g);
    orc_linear(weight_format, group, scale_is_bf16, wu, su, e, ffn_e, hidden, x, u);
    orc_swiglu(g, u, ffn_e, a);
    orc_linear(weight_format, group, scale_is_bf16, wd, sd, e, hidden, ffn_e, a, d);
    for (int o = 0; o < hidden; ++o) y[o] += weights[i] * d[o];
  }
  free(g);
  free(u);
  free(a);
  free(d);
}

int orc_decode_step(const orc_model* m, int token, int pos, uint16_t* kcache, uint16_t* vcache,
                    orc_real* logits, int* argmax, orc_real* trace_x) {
  const int H = m->hidden, nq = m->n_heads, nkv = m->n_kv_heads, d = m->head_dim;
  const int F = m->ffn, V = m->vocab, C = m->max_ctx;
  if (token < 0 || token >= V || pos < 0 || pos >= C || nq % nkv != 0 || d % 2 != 0)
    return ORC_ERR_INVALID;
  const int qd = nq * d, kvd = nkv * d;
  orc_real* x = (orc_real*)malloc(sizeof(orc_real) * H);
  orc_real* n = (orc_real*)malloc(sizeof(orc_real) * H);
  orc_real* q = (orc_real*)malloc(sizeof(orc_real) * qd);
  orc_real* k = (orc_real*)malloc(sizeof(orc_real) * kvd);
  orc_real* v = (orc_real*)malloc(sizeof(orc_real) * kvd);
  orc_real* att = (orc_real*)malloc(sizeof(orc_real) * qd);
  orc_real* y = (orc_real*)malloc(sizeof(orc_real) * H);
  orc_real* g = (orc_real*)malloc(sizeof(orc_real) * F);
  orc_real* u = (orc_real*)malloc(sizeof(orc_real) * F);
  orc_real* a = (orc_real*)malloc(sizeof(orc_real) * F);

  for (int i = 0; i < H; ++i) x[i] = (orc_real)orc_bf16_value(m->embed[(size_t)token * H + i]);

  for (int li = 0; li < m->n_layers; ++li) {
    const orc_layer* L = &m->layers[li];
    orc_rmsnorm(x, L->g1, H, m->rms_eps, n);
    gemv_any(m, L->wq, L->sq, qd, H, n, q);
    gemv_any(m, L->wk, L->sk, kvd, H, n, k);
    gemv_any(m, L->wv, L->sv, kvd, H, n, v);
    if (m->qkv_bias) {
      for (int i = 0; i < qd; ++i) q[i] += (orc_real)orc_bf16_value(L->bq[i]);
      for (int i = 0; i < kvd; ++i) k[i] += (orc_real)orc_bf16_value(L->bk[i]);
      for (int i = 0; i < kvd; ++i) v[i] += (orc_real)orc_bf16_value(L->bv[i]);
    }
    for (int h = 0; h < nq; ++h) orc_rope(q + (size_t)h * d, d, pos, m->rope_theta);
    for (int j = 0; j < nkv; ++j) orc_rope(k + (size_t)j * d, d, pos, m->rope_theta);

    uint16_t* Kl = kcache + (size_t)li * nkv * C * d;
    uint16_t* Vl = vcache + (size_t)li * nkv * C * d;
    for (int j = 0; j < nkv; ++j)
      for (int i = 0; i < d; ++i) {
        Kl[((size_t)j * C + pos) * d + i] = orc_round_bf16((double)k[(size_t)j * d + i]);
        Vl[((size_t)j * C + pos) * d + i] = orc_round_bf16((double)v[(size_t)j * d + i]);
      }
    orc_attention(q, Kl, Vl, nq, nkv, d, pos + 1, C, att);

    gemv_any(m, L->wo, L->so, H, qd, att, y);
    for (int i = 0; i < H; ++i) x[i] += y[i];

    orc_rmsnorm(x, L->g2, H, m->rms_eps, n);
    gemv_any(m, L->wg, L->sg, F, H, n, g);
    gemv_any(m, L->wu, L->su, F, H, n, u);
    orc_swiglu(g, u, F, a);
    gemv_any(m, L->wd, L->sd, H, F, a, y);
    for (int i = 0; i < H; ++i) x[i] += y[i];
    if (trace_x) memcpy(trace_x + (size_t)li * H, x, sizeof(orc_real) * H);
  }

  orc_rmsnorm(x, m->final_norm, H, m->rms_eps, n);
  orc_gemv_bf16(m->lm_head, V, H, n, logits);
  int rc = orc_argmax(logits, V, argmax);

  free(x); free(n); free(q); free(k); free(v); free(att); free(y); free(g); free(u); free(a);
  return rc;
}
