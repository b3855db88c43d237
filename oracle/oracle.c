/* CPU oracle for the 4-bit decode step — TEST INFRASTRUCTURE ONLY.
 *
 * Plain C, fp64 everywhere except where the pages fix a storage precision:
 *   - weights are group-64 4-bit codes with fp16 scale and min, w = scale*q + min
 *     (llmopt page, "packed group-64 W4A16 linear kernels"); dequantised exactly
 *     in fp64;
 *   - the KV cache holds bf16 keys and values appended from f32 (zynfer page,
 *     M4: "bf16 KV cache (append from f32 Q/K/V; attention widens to f32)"),
 *     so k and v are rounded fp64 -> fp32 -> bf16 before they are stored and
 *     every position (the current one included) is read back from the cache;
 *   - the greedy choice is taken on fp32-rounded logits, the precision the GPU
 *     path decides in; lowest index wins a tie;
 *   - optionally the cache holds K/V as grouped int8 (llmopt page, "grouped-Q8
 *     attention/recurrent state"; the q8_0 block of GGUF files): groups of 32,
 *     an fp16 scale amax/127 and round-to-nearest codes, all decided in fp32
 *     (the precision the pages append from).
 * Pipeline and per-architecture variants follow the aot-llm page (sequence
 * diagram, "static pipeline", Qwen3 per-head q/k RMSNorm before RoPE, NEOX
 * pairing (i, i + rot_dim/2) versus adjacent pairs); GQA grouping and the
 * bottom-right causal alignment follow the pytensor-ml issue ("Already here"
 * table: k_idx <= q_idx + (sk - sq), _repeat_kv). OpenMP only splits output
 * rows; every sum runs in index order.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int32_t g_mut = ORC_MUT_NONE;
static int32_t g_kv_q8 = 0;

void orc_set_kv_q8(int32_t on) { g_kv_q8 = on; }

void orc_set_mutation(int32_t m) { g_mut = m; }

int32_t orc_num_threads(void) {
#ifdef _OPENMP
  return (int32_t)omp_get_max_threads();
#else
  return 1;
#endif
}

/* IEEE binary16 -> double, exact. */
double orc_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)f, -24);
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp((double)(1024 + f), e - 25);
  return sign ? -v : v;
}

double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

float orc_f32_from_double(double x) { return (float)x; }

/* Round to bf16: first to fp32 (the precision the pages append from), then to
   8 significant bits with ties to even. */
uint16_t orc_bf16_from_double(double x) {
  float f = (float)x;
  double d = (double)f, r;
  uint32_t u;
  if (isnan(d)) return 0x7FC0;
  if (d == 0.0 || isinf(d)) {
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
  }
  if (fabs(d) < ldexp(1.0, -126)) {
    r = ldexp(nearbyint(ldexp(d, 133)), -133);      /* bf16 subnormal spacing */
  } else {
    int e;
    double m = frexp(d, &e);                          /* d = m * 2^e, |m| in [0.5,1) */
    r = ldexp(nearbyint(ldexp(m, 8)), e - 8);         /* 8 significant bits */
  }
  f = (float)r;                                       /* exact, or inf on overflow */
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* w[r][c] = scale * q + min for one row, q read from the canonical nibble. */
void orc_dequant_row(const orc_q4* w, int64_t r, double* out) {
  const int64_t cols = w->cols, groups = cols / 64;
  const uint8_t* cr = w->codes + r * (cols / 2);
  const int swap_nibbles = (g_mut == ORC_MUT_NIBBLE_ORDER);
  for (int64_t g = 0; g < groups; ++g) {
    double s = orc_half_to_double(w->scales[r * groups + g]);
    double m = orc_half_to_double(w->mins[r * groups + g]);
    if (g_mut == ORC_MUT_SCALE_MIN_SWAP) { double t = s; s = m; m = t; }
    for (int64_t c = g * 64; c < g * 64 + 64; ++c) {
      uint8_t byte = cr[c / 2];
      int hi = (int)(c & 1) ^ swap_nibbles;
      int q = hi ? (byte >> 4) : (byte & 15);
      out[c] = s * (double)q + m;
    }
  }
}

/* y = W x with fp64 sums over the full input, rows in parallel. */
void orc_matvec(const orc_q4* w, const double* x, double* y) {
  const int64_t rows = w->rows, cols = w->cols;
#pragma omp parallel
  {
    double* row = (double*)malloc((size_t)cols * sizeof(double));
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      orc_dequant_row(w, r, row);
      double acc = 0.0;
      for (int64_t c = 0; c < cols; ++c) acc += row[c] * x[c];
      y[r] = acc;
    }
    free(row);
  }
}

/* RMSNorm, Llama form: x / sqrt(mean(x^2) + eps) * w. */
void orc_rmsnorm(const double* x, const float* w, int32_t n, double eps, double* out) {
  double ss = 0.0;
  for (int32_t i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int32_t i = 0; i < n; ++i) out[i] = x[i] * inv * (double)w[i];
}

/* Rotary embedding of one head at position pos: theta_i = base^(-2i/hd),
   pairs (2i, 2i+1) or, NEOX layout, (i, i + hd/2). */
void orc_rope(double* v, int32_t hd, int32_t pos, double theta, int32_t neox) {
  if (g_mut == ORC_MUT_ROPE_PAIRING) neox = !neox;
  const int32_t half = hd / 2;
  for (int32_t i = 0; i < half; ++i) {
    double inv_freq = pow(theta, -2.0 * (double)i / (double)hd);
    double ang = (double)pos * inv_freq;
    double c = cos(ang), s = sin(ang);
    if (g_mut == ORC_MUT_ROPE_SIGN) s = -s;
    int32_t a = neox ? i : 2 * i;
    int32_t b = neox ? i + half : 2 * i + 1;
    double x0 = v[a], x1 = v[b];
    v[a] = x0 * c - x1 * s;
    v[b] = x0 * s + x1 * c;
  }
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

void orc_silu_mul(const double* g, const double* u, int32_t n, double* out) {
  for (int32_t i = 0; i < n; ++i) out[i] = silu(g[i]) * u[i];
}

/* softmax(q . k_t / sqrt(hd)) weighted sum of v_t over t = 0..n_pos-1. */
void orc_attend(const double* q, const uint16_t* k, const uint16_t* v, int32_t n_pos,
                int32_t hd, double* out) {
  const double scale = 1.0 / sqrt((double)hd);
  double* s = (double*)malloc((size_t)(n_pos > 0 ? n_pos : 1) * sizeof(double));
  double mx = -INFINITY, l = 0.0;
  for (int32_t t = 0; t < n_pos; ++t) {
    double dot = 0.0;
    for (int32_t d = 0; d < hd; ++d) dot += q[d] * orc_bf16_to_double(k[(int64_t)t * hd + d]);
    s[t] = dot * scale;
    if (s[t] > mx) mx = s[t];
  }
  for (int32_t d = 0; d < hd; ++d) out[d] = 0.0;
  for (int32_t t = 0; t < n_pos; ++t) {
    double p = exp(s[t] - mx);
    l += p;
    for (int32_t d = 0; d < hd; ++d) out[d] += p * orc_bf16_to_double(v[(int64_t)t * hd + d]);
  }
  for (int32_t d = 0; d < hd; ++d) out[d] /= l;
  free(s);
}

/* fp32 -> IEEE binary16, round to nearest even (11 significant bits; subnormal
   spacing 2^-24; overflow to infinity). */
uint16_t orc_half_from_float(float f) {
  const double x = (double)f;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x), r;
  if (isnan(x)) return 0x7E00;
  if (a < ldexp(1.0, -14)) {
    r = ldexp(nearbyint(ldexp(a, 24)), -24);
  } else {
    int e;
    double m = frexp(a, &e);                          /* a = m * 2^e, m in [0.5, 1) */
    r = ldexp(nearbyint(ldexp(m, 11)), e - 11);
  }
  if (r >= 65520.0 || isinf(a)) return (uint16_t)(sign | 0x7C00);
  if (r < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)nearbyint(ldexp(r, 24)));
  int e;
  double m = frexp(r, &e);                            /* r = m * 2^e exactly */
  const int E = e - 1 + 15;                           /* biased exponent of 1.f * 2^(e-1) */
  const int F = (int)nearbyint(ldexp(m, 11)) - 1024;  /* 10 fraction bits */
  return (uint16_t)(sign | (E << 10) | F);
}

void orc_q8_quantize(const double* x, int32_t n, int8_t* q, uint16_t* d) {
  for (int32_t g = 0; g < n / ORC_Q8_GROUP; ++g) {
    float xf[ORC_Q8_GROUP], amax = 0.0f;
    for (int32_t i = 0; i < ORC_Q8_GROUP; ++i) {
      xf[i] = (float)x[g * ORC_Q8_GROUP + i];
      if (fabsf(xf[i]) > amax) amax = fabsf(xf[i]);
    }
    d[g] = orc_half_from_float(amax / 127.0f);
    const float dq = (float)orc_half_to_double(d[g]);
    for (int32_t i = 0; i < ORC_Q8_GROUP; ++i) {
      float c = dq == 0.0f ? 0.0f : roundf(xf[i] / dq);
      c = c > 127.0f ? 127.0f : (c < -127.0f ? -127.0f : c);
      q[g * ORC_Q8_GROUP + i] = (int8_t)c;
    }
  }
}

double orc_q8_value(int8_t q, uint16_t d) { return (double)q * orc_half_to_double(d); }

void orc_attend_q8(const double* q, const int8_t* k, const uint16_t* ks, const int8_t* v,
                   const uint16_t* vs, int32_t n_pos, int32_t hd, double* out) {
  const double scale = 1.0 / sqrt((double)hd);
  const int32_t ng = hd / ORC_Q8_GROUP;
  double* s = (double*)malloc((size_t)(n_pos > 0 ? n_pos : 1) * sizeof(double));
  double mx = -INFINITY, l = 0.0;
  for (int32_t t = 0; t < n_pos; ++t) {
    double dot = 0.0;
    for (int32_t d = 0; d < hd; ++d)
      dot += q[d] * orc_q8_value(k[(int64_t)t * hd + d], ks[(int64_t)t * ng + d / ORC_Q8_GROUP]);
    s[t] = dot * scale;
    if (s[t] > mx) mx = s[t];
  }
  for (int32_t d = 0; d < hd; ++d) out[d] = 0.0;
  for (int32_t t = 0; t < n_pos; ++t) {
    double p = exp(s[t] - mx);
    l += p;
    for (int32_t d = 0; d < hd; ++d)
      out[d] += p * orc_q8_value(v[(int64_t)t * hd + d], vs[(int64_t)t * ng + d / ORC_Q8_GROUP]);
  }
  for (int32_t d = 0; d < hd; ++d) out[d] /= l;
  free(s);
}

/* Greedy choice on fp32-rounded logits; lowest index wins a tie; -1 on NaN. */
int32_t orc_argmax_f32(const double* logits, int64_t n) {
  int64_t best = -1;
  float bv = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float f = (float)logits[i];
    if (isnan(f)) return -1;
    if (best < 0 || f > bv) { best = i; bv = f; }
  }
  return (int32_t)best;
}

static void embed_row(const orc_model* m, int32_t tok, double* x) {
  const int32_t d = m->cfg.dim;
  if (m->cfg.embed_bf16) {
    const uint16_t* e = (const uint16_t*)m->embed + (int64_t)tok * d;
    for (int32_t i = 0; i < d; ++i) x[i] = orc_bf16_to_double(e[i]);
  } else {
    const float* e = (const float*)m->embed + (int64_t)tok * d;
    for (int32_t i = 0; i < d; ++i) x[i] = (double)e[i];
  }
}

static void lm_head(const orc_model* m, const double* xn, double* logits) {
  const int32_t d = m->cfg.dim;
  if (m->cfg.tied) {
    const uint16_t* e = (const uint16_t*)m->embed;
    const int64_t V = m->cfg.vocab;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < V; ++r) {
      double acc = 0.0;
      for (int32_t c = 0; c < d; ++c) acc += orc_bf16_to_double(e[r * d + c]) * xn[c];
      logits[r] = acc;
    }
  } else {
    orc_matvec(&m->lm_head, xn, logits);
  }
}

/* Per-head q/k RMSNorm (Qwen3), then RoPE, for one position's q and k. */
static void qk_prepare(const orc_model* m, const orc_layer* L, double* q, double* k, int32_t pos) {
  const orc_config* c = &m->cfg;
  const int32_t hd = c->head_dim;
  double* tmp = (double*)malloc((size_t)hd * sizeof(double));
  for (int32_t h = 0; h < c->n_heads; ++h) {
    if (c->qk_norm) {
      orc_rmsnorm(q + (int64_t)h * hd, L->q_norm, hd, c->norm_eps, tmp);
      memcpy(q + (int64_t)h * hd, tmp, (size_t)hd * sizeof(double));
    }
    orc_rope(q + (int64_t)h * hd, hd, pos, c->rope_theta, c->rope_neox);
  }
  for (int32_t h = 0; h < c->n_kv_heads; ++h) {
    if (c->qk_norm) {
      orc_rmsnorm(k + (int64_t)h * hd, L->k_norm, hd, c->norm_eps, tmp);
      memcpy(k + (int64_t)h * hd, tmp, (size_t)hd * sizeof(double));
    }
    orc_rope(k + (int64_t)h * hd, hd, pos, c->rope_theta, c->rope_neox);
  }
  free(tmp);
}

static int32_t kv_head_of(const orc_config* c, int32_t h) {
  if (g_mut == ORC_MUT_GQA_MAP) return h % c->n_kv_heads;
  return h / (c->n_heads / c->n_kv_heads);
}

/* Residual add x += y (the planted mistake replaces it by x = y). */
static void residual(double* x, const double* y, int32_t n) {
  for (int32_t i = 0; i < n; ++i) x[i] = (g_mut == ORC_MUT_NO_RESIDUAL) ? y[i] : x[i] + y[i];
}

/* SwiGLU feed-forward of one position, added to x. */
static void ffn(const orc_model* m, const orc_layer* L, double* x) {
  const orc_config* c = &m->cfg;
  const int32_t d = c->dim, F = c->ffn_dim;
  double* xn = (double*)malloc((size_t)d * sizeof(double));
  double* g = (double*)malloc((size_t)F * sizeof(double));
  double* u = (double*)malloc((size_t)F * sizeof(double));
  double* a = (double*)malloc((size_t)F * sizeof(double));
  double* y = (double*)malloc((size_t)d * sizeof(double));
  orc_rmsnorm(x, L->ffn_norm, d, c->norm_eps, xn);
  orc_matvec(&L->wg, xn, g);
  orc_matvec(&L->wu, xn, u);
  orc_silu_mul(g, u, F, a);
  orc_matvec(&L->wd, a, y);
  residual(x, y, d);
  free(xn); free(g); free(u); free(a); free(y);
}

int32_t orc_step(const orc_model* m, orc_cache* cache, int32_t tok, double* logits, double* hidden) {
  const orc_config* c = &m->cfg;
  const int32_t d = c->dim, hd = c->head_dim, Hq = c->n_heads, Hkv = c->n_kv_heads;
  const int32_t qd = Hq * hd, kd = Hkv * hd;
  const int32_t pos = cache->len;
  if (pos >= cache->cap || tok < 0 || tok >= c->vocab) return -1;
  double* x = (double*)malloc((size_t)d * sizeof(double));
  double* xn = (double*)malloc((size_t)d * sizeof(double));
  double* q = (double*)malloc((size_t)qd * sizeof(double));
  double* k = (double*)malloc((size_t)kd * sizeof(double));
  double* v = (double*)malloc((size_t)kd * sizeof(double));
  double* o = (double*)malloc((size_t)qd * sizeof(double));
  double* y = (double*)malloc((size_t)d * sizeof(double));
  embed_row(m, tok, x);
  if (hidden) memcpy(hidden, x, (size_t)d * sizeof(double));
  for (int32_t l = 0; l < c->n_layers; ++l) {
    const orc_layer* L = &m->layers[l];
    orc_rmsnorm(x, L->attn_norm, d, c->norm_eps, xn);
    orc_matvec(&L->wq, xn, q);
    orc_matvec(&L->wk, xn, k);
    orc_matvec(&L->wv, xn, v);
    qk_prepare(m, L, q, k, pos);
    /* append this position's K and V (bf16, or grouped int8) to the cache */
    for (int32_t g = 0; g < Hkv; ++g) {
      int64_t base = (((int64_t)l * Hkv + g) * cache->cap + pos) * hd;
      if (cache->k8) {
        const int64_t sbase = base / ORC_Q8_GROUP;
        orc_q8_quantize(k + (int64_t)g * hd, hd, cache->k8 + base, cache->ks + sbase);
        orc_q8_quantize(v + (int64_t)g * hd, hd, cache->v8 + base, cache->vs + sbase);
        continue;
      }
      for (int32_t i = 0; i < hd; ++i) {
        cache->k[base + i] = orc_bf16_from_double(k[(int64_t)g * hd + i]);
        cache->v[base + i] = orc_bf16_from_double(v[(int64_t)g * hd + i]);
      }
    }
    /* the query attends to cached positions 0..pos, itself included */
    int32_t n_att = pos + 1;
    if (g_mut == ORC_MUT_CACHE_FRONTIER && pos > 0) n_att = pos;
#pragma omp parallel for schedule(static)
    for (int32_t h = 0; h < Hq; ++h) {
      int32_t g = kv_head_of(c, h);
      int64_t base = ((int64_t)l * Hkv + g) * cache->cap * hd;
      if (cache->k8)
        orc_attend_q8(q + (int64_t)h * hd, cache->k8 + base, cache->ks + base / ORC_Q8_GROUP, cache->v8 + base,
                      cache->vs + base / ORC_Q8_GROUP, n_att, hd, o + (int64_t)h * hd);
      else
        orc_attend(q + (int64_t)h * hd, cache->k + base, cache->v + base, n_att, hd,
                   o + (int64_t)h * hd);
    }
    orc_matvec(&L->wo, o, y);
    residual(x, y, d);
    ffn(m, L, x);
    if (hidden) memcpy(hidden + (int64_t)(l + 1) * d, x, (size_t)d * sizeof(double));
  }
  if (logits) {
    orc_rmsnorm(x, m->final_norm, d, c->norm_eps, xn);
    lm_head(m, xn, logits);
  }
  cache->len = pos + 1;
  free(x); free(xn); free(q); free(k); free(v); free(o); free(y);
  return 0;
}

int32_t orc_full_prefix(const orc_model* m, const int32_t* toks, int32_t n, double* logits,
                        double* hidden) {
  const orc_config* c = &m->cfg;
  const int32_t d = c->dim, hd = c->head_dim, Hq = c->n_heads, Hkv = c->n_kv_heads;
  const int32_t qd = Hq * hd, kd = Hkv * hd;
  if (n <= 0) return -1;
  double* H = (double*)malloc((size_t)n * d * sizeof(double));
  double* Q = (double*)malloc((size_t)n * qd * sizeof(double));
  double* K = (double*)malloc((size_t)n * kd * sizeof(double));
  double* Vv = (double*)malloc((size_t)n * kd * sizeof(double));
  double* Kb = (double*)malloc((size_t)n * kd * sizeof(double));   /* K/V as read back from storage */
  double* Vb = (double*)malloc((size_t)n * kd * sizeof(double));
  int8_t q8[512];
  uint16_t d8[512 / ORC_Q8_GROUP];
  double* xn = (double*)malloc((size_t)d * sizeof(double));
  double* o = (double*)malloc((size_t)qd * sizeof(double));
  double* y = (double*)malloc((size_t)d * sizeof(double));
  double* s = (double*)malloc((size_t)n * sizeof(double));
  const double scale = 1.0 / sqrt((double)hd);
  for (int32_t t = 0; t < n; ++t) {
    if (toks[t] < 0 || toks[t] >= c->vocab) return -1;
    embed_row(m, toks[t], H + (int64_t)t * d);
  }
  if (hidden) memcpy(hidden, H, (size_t)n * d * sizeof(double));
  for (int32_t l = 0; l < c->n_layers; ++l) {
    const orc_layer* L = &m->layers[l];
    /* projections of every position of this layer */
    for (int32_t t = 0; t < n; ++t) {
      orc_rmsnorm(H + (int64_t)t * d, L->attn_norm, d, c->norm_eps, xn);
      orc_matvec(&L->wq, xn, Q + (int64_t)t * qd);
      orc_matvec(&L->wk, xn, K + (int64_t)t * kd);
      orc_matvec(&L->wv, xn, Vv + (int64_t)t * kd);
      qk_prepare(m, L, Q + (int64_t)t * qd, K + (int64_t)t * kd, t);
    }
    /* keys and values as read back from the storage type (bf16 or grouped
       int8): [kv_head][t][hd] */
    for (int32_t t = 0; t < n; ++t)
      for (int32_t g = 0; g < Hkv; ++g) {
        double* kr = Kb + ((int64_t)g * n + t) * hd;
        double* vr = Vb + ((int64_t)g * n + t) * hd;
        if (g_kv_q8) {
          orc_q8_quantize(K + (int64_t)t * kd + g * hd, hd, q8, d8);
          for (int32_t i = 0; i < hd; ++i) kr[i] = orc_q8_value(q8[i], d8[i / ORC_Q8_GROUP]);
          orc_q8_quantize(Vv + (int64_t)t * kd + g * hd, hd, q8, d8);
          for (int32_t i = 0; i < hd; ++i) vr[i] = orc_q8_value(q8[i], d8[i / ORC_Q8_GROUP]);
          continue;
        }
        for (int32_t i = 0; i < hd; ++i) {
          kr[i] = orc_bf16_to_double(orc_bf16_from_double(K[(int64_t)t * kd + g * hd + i]));
          vr[i] = orc_bf16_to_double(orc_bf16_from_double(Vv[(int64_t)t * kd + g * hd + i]));
        }
      }
    /* causal attention, bottom-right aligned: key j visible to query t iff
       j <= t + (sk - sq); here sq == sk == n */
    for (int32_t t = 0; t < n; ++t) {
      for (int32_t h = 0; h < Hq; ++h) {
        int32_t g = kv_head_of(c, h);
        const double* kg = Kb + (int64_t)g * n * hd;
        const double* vg = Vb + (int64_t)g * n * hd;
        double mx = -INFINITY, lsum = 0.0;
        double* out = o + (int64_t)h * hd;
        for (int32_t j = 0; j < n; ++j) {
          int visible = (g_mut == ORC_MUT_MASK_POLARITY) ? (j >= t) : (j <= t + (n - n));
          if (!visible) continue;
          double dot = 0.0;
          if (g_mut == ORC_MUT_QK_ORIENTATION) {
            /* planted: the roles of query and key rows exchanged */
            const double* qj = Q + (int64_t)j * qd + (int64_t)h * hd;
            for (int32_t i = 0; i < hd; ++i) dot += qj[i] * kg[(int64_t)t * hd + i];
          } else {
            const double* qt = Q + (int64_t)t * qd + (int64_t)h * hd;
            for (int32_t i = 0; i < hd; ++i) dot += qt[i] * kg[(int64_t)j * hd + i];
          }
          s[j] = dot * scale;
          if (s[j] > mx) mx = s[j];
        }
        for (int32_t i = 0; i < hd; ++i) out[i] = 0.0;
        for (int32_t j = 0; j < n; ++j) {
          int visible = (g_mut == ORC_MUT_MASK_POLARITY) ? (j >= t) : (j <= t + (n - n));
          if (!visible) continue;
          double p = exp(s[j] - mx);
          lsum += p;
          for (int32_t i = 0; i < hd; ++i) out[i] += p * vg[(int64_t)j * hd + i];
        }
        for (int32_t i = 0; i < hd; ++i) out[i] /= lsum;
      }
      orc_matvec(&L->wo, o, y);
      residual(H + (int64_t)t * d, y, d);
    }
    for (int32_t t = 0; t < n; ++t) ffn(m, L, H + (int64_t)t * d);
    if (hidden) memcpy(hidden + (int64_t)(l + 1) * n * d, H, (size_t)n * d * sizeof(double));
  }
  if (logits) {
    for (int32_t t = 0; t < n; ++t) {
      orc_rmsnorm(H + (int64_t)t * d, m->final_norm, d, c->norm_eps, xn);
      lm_head(m, xn, logits + (int64_t)t * c->vocab);
    }
  }
  free(H); free(Q); free(K); free(Vv); free(Kb); free(Vb); free(xn); free(o); free(y); free(s);
  return 0;
}
