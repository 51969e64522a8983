/*
 * qtts_oracle.c -- plain CPU oracle for one lockstep multi-codebook codec
 * frame (see qtts_oracle.h for the pages this follows).
 *
 * TEST INFRASTRUCTURE: never linked into, loaded by or called from the CUDA
 * product path. Everything here is written out in the order the model is
 * described, with no blocking, fusion or reordering. Sessions are processed
 * one after another (the lockstep batch changes no arithmetic), and inside a
 * session the Code Predictor runs one position at a time.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math:
 * the binary32 sampler and quantiser must be plain IEEE operations).
 */
#include "qtts_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 storage format                                                 */
/* ------------------------------------------------------------------ */

double orc_from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), directly from double. */
uint16_t orc_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  if (isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
  int e;
  frexp(x, &e);                 /* |x| = m * 2^e, m in [0.5, 1) */
  int qe = e - 8;               /* bf16 keeps 8 significant bits */
  if (qe < -133) qe = -133;     /* bf16 subnormal quantum 2^-133 */
  double r = nearbyint(ldexp(x, -qe)); /* exact scaling, round half even */
  r = ldexp(r, qe);
  float f = (float)r;           /* exact, or +-inf on overflow */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* Transformer pieces (double)                                         */
/* ------------------------------------------------------------------ */

/* RMSNorm: out = x / sqrt(mean(x^2) + eps) * g */
void orc_rmsnorm(const double* x, const uint16_t* g, int n, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < n; i++) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; i++) out[i] = x[i] * r * orc_from_bf16(g[i]);
}

/* Rotate-half RoPE at position pos: within each head, element i pairs with
 * element i + d/2 and the pair is turned by angle pos * theta^(-2i/d). */
void orc_rope(double* v, int n_heads, int head_dim, int pos, double theta) {
  int half = head_dim / 2;
  for (int h = 0; h < n_heads; h++) {
    double* e = v + (size_t)h * head_dim;
    for (int i = 0; i < half; i++) {
      double inv_freq = pow(theta, -2.0 * (double)i / (double)head_dim);
      double ang = (double)pos * inv_freq;
      double c = cos(ang), s = sin(ang);
      double a = e[i], b = e[i + half];
      e[i] = a * c - b * s;
      e[i + half] = b * c + a * s;
    }
  }
}

/* y[n] = sum_k W[n,k] x[k]; INT8: y[n] = scale[n] * sum_k q[n,k] x[k]. */
void orc_linear(const double* x, orc_lin W, int use_int8, int N, int K, double* y) {
  if (use_int8 && W.q) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
      const int8_t* row = W.q + (size_t)n * K;
      double acc = 0.0;
      for (int k = 0; k < K; k++) acc += (double)row[k] * x[k];
      y[n] = (double)W.s[n] * acc;
    }
  } else {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
      const uint16_t* row = W.w + (size_t)n * K;
      double acc = 0.0;
      for (int k = 0; k < K; k++) acc += orc_from_bf16(row[k]) * x[k];
      y[n] = acc;
    }
  }
}

/* Decode attention for one query position over n_pos cached positions.
 * q: [n_q_heads][d]; caches: [n_pos][n_kv_heads][d] bf16. Query head h reads
 * kv group h / (n_q_heads / n_kv_heads). Softmax is max-subtracted. */
void orc_attention(const double* q, const uint16_t* k_cache, const uint16_t* v_cache,
                   int n_pos, int n_q_heads, int n_kv_heads, int head_dim, double* out) {
  int group = n_q_heads / n_kv_heads;
  double scale = 1.0 / sqrt((double)head_dim);
  double* sc = (double*)malloc(sizeof(double) * (size_t)(n_pos > 0 ? n_pos : 1));
  for (int h = 0; h < n_q_heads; h++) {
    int g = h / group;
    const double* qh = q + (size_t)h * head_dim;
    double mx = -INFINITY;
    for (int i = 0; i < n_pos; i++) {
      const uint16_t* kr = k_cache + ((size_t)i * n_kv_heads + g) * head_dim;
      double dot = 0.0;
      for (int t = 0; t < head_dim; t++) dot += qh[t] * orc_from_bf16(kr[t]);
      sc[i] = dot * scale;
      if (sc[i] > mx) mx = sc[i];
    }
    double den = 0.0;
    for (int i = 0; i < n_pos; i++) {
      sc[i] = exp(sc[i] - mx);
      den += sc[i];
    }
    double* oh = out + (size_t)h * head_dim;
    for (int t = 0; t < head_dim; t++) oh[t] = 0.0;
    for (int i = 0; i < n_pos; i++) {
      const uint16_t* vr = v_cache + ((size_t)i * n_kv_heads + g) * head_dim;
      double p = sc[i] / den;
      for (int t = 0; t < head_dim; t++) oh[t] += p * orc_from_bf16(vr[t]);
    }
  }
  free(sc);
}

double orc_silu(double a) { return a / (1.0 + exp(-a)); }

/* ------------------------------------------------------------------ */
/* INT8 weight-only quantiser (binary32, exact integer rule)           */
/* ------------------------------------------------------------------ */

/* Per output channel (row): m = max|w|, scale = m / 127 (IEEE binary32
 * division), q = round-half-even(w / scale) clamped to [-127, 127].
 * A zero row gets scale 0 and q = 0. */
void orc_quantize_rows(const uint16_t* w, int N, int K, int8_t* q, float* scale) {
  for (int n = 0; n < N; n++) {
    const uint16_t* row = w + (size_t)n * K;
    float m = 0.0f;
    for (int k = 0; k < K; k++) {
      float a = fabsf((float)orc_from_bf16(row[k]));
      if (a > m) m = a;
    }
    float s = m / 127.0f;
    scale[n] = s;
    for (int k = 0; k < K; k++) {
      int8_t v = 0;
      if (s != 0.0f) {
        float t = (float)orc_from_bf16(row[k]) / s;
        float r = nearbyintf(t); /* default rounding mode: ties to even */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        v = (int8_t)r;
      }
      q[(size_t)n * K + k] = v;
    }
  }
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11)                    */
/* ------------------------------------------------------------------ */

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; round++) {
    if (round > 0) { /* Weyl key schedule between rounds */
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* ------------------------------------------------------------------ */
/* Natural log in binary32, written for this project so that two        */
/* independent implementations give identical bits:                     */
/*   x = m * 2^k with m in (sqrt(1/2), sqrt(2)],                        */
/*   log m = 2 atanh(s), s = (m-1)/(m+1), atanh series up to s^11.      */
/* Every operation is one IEEE binary32 operation, in this order.       */
/* ------------------------------------------------------------------ */

float orc_logf(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  int k = 0;
  if (((u >> 23) & 0xFFu) == 0u) { /* subnormal: scale by 2^25 (exact) */
    x = x * 0x1p25f;
    memcpy(&u, &x, 4);
    k = -25;
  }
  k += (int)((u >> 23) & 0xFFu) - 127;
  uint32_t mb = (u & 0x007FFFFFu) | 0x3F800000u; /* m in [1, 2) */
  if (mb > 0x3FB504F3u) {                          /* m > sqrt(2): halve */
    mb = (u & 0x007FFFFFu) | 0x3F000000u;
    k += 1;
  }
  float m;
  memcpy(&m, &mb, 4);
  float num = m - 1.0f;
  float den = m + 1.0f;
  float s = num / den;
  float s2 = s * s;
  float t = 0x1.745d18p-4f;          /* 1/11 */
  t = t * s2; t = t + 0x1.c71c72p-4f; /* 1/9 */
  t = t * s2; t = t + 0x1.24924ap-3f; /* 1/7 */
  t = t * s2; t = t + 0x1.99999ap-3f; /* 1/5 */
  t = t * s2; t = t + 0x1.555556p-2f; /* 1/3 */
  t = t * s2; t = t + 1.0f;
  float two_s = s + s;
  float lm = two_s * t;
  float kl = (float)k * 0x1.62e430p-1f; /* k * ln 2 */
  return kl + lm;
}

/* Uniform in (0,1) for vocabulary id v of codebook j at frame frame_ctr:
 * word v&3 of Philox4x32-10(key, ctr = (v>>2, j, frame_ctr, 0)),
 * top 23 bits, u = (bits + 0.5) * 2^-23 (exact in binary32). */
float orc_uniform(uint32_t key0, uint32_t key1, int codebook, uint32_t frame_ctr, int v) {
  uint32_t ctr[4] = {(uint32_t)v >> 2, (uint32_t)codebook, frame_ctr, 0u};
  uint32_t key[2] = {key0, key1};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  uint32_t bits = out[v & 3] >> 9;
  float f = (float)bits;
  f = f + 0.5f;
  return f * 0x1p-23f;
}

/* ------------------------------------------------------------------ */
/* Sampler                                                              */
/* ------------------------------------------------------------------ */

typedef struct { float z; int id; } orc_cand;

static int cand_cmp(const void* a, const void* b) {
  const orc_cand* x = (const orc_cand*)a;
  const orc_cand* y = (const orc_cand*)b;
  if (x->z > y->z) return -1; /* larger z first */
  if (x->z < y->z) return 1;
  return (x->id < y->id) ? -1 : (x->id > y->id); /* equal z: smaller id first */
}

/* One code from one row of raw logits:
 *  1. codebook 0: ids >= n_codes other than eos_id -> -inf; eos_id -> -inf
 *     unless eos_allowed; repetition penalty on every id in the seen set
 *     (positive logit divided by r, otherwise multiplied by r).
 *  2. greedy (temperature 0 or top_k 1): argmax, lowest id on ties.
 *  3. z = l / T; keep the top_k ids by (z desc, id asc).
 *  4. Gumbel-max: argmax over kept ids of z + (-log(-log u)), lowest id on ties. */
int32_t orc_sample(const float* logits, int V, int codebook, const orc_session* s,
                   uint32_t key0, uint32_t key1, uint32_t frame_ctr, const uint32_t* seen,
                   int eos_id, int n_codes) {
  float* lp = (float*)malloc(sizeof(float) * (size_t)V);
  for (int v = 0; v < V; v++) lp[v] = logits[v];
  float T;
  int k;
  if (codebook == 0) {
    for (int v = 0; v < V; v++) {
      if (v >= n_codes && v != eos_id) lp[v] = -INFINITY;
      if (v == eos_id && !s->eos_allowed) lp[v] = -INFINITY;
    }
    float r = s->rep_penalty;
    for (int v = 0; v < V; v++) {
      if (seen && ((seen[v >> 5] >> (v & 31)) & 1u)) lp[v] = (lp[v] > 0.0f) ? lp[v] / r : lp[v] * r;
    }
    T = s->temperature;
    k = s->top_k;
  } else {
    T = s->cp_temperature;
    k = s->cp_top_k;
  }
  int32_t best = 0;
  if (T == 0.0f || k == 1) {
    for (int v = 1; v < V; v++)
      if (lp[v] > lp[best]) best = v;
    free(lp);
    return best;
  }
  if (k <= 0 || k > V) k = V;
  orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)V);
  for (int v = 0; v < V; v++) {
    float z = lp[v] / T;
    if (z == 0.0f) z = 0.0f; /* one zero: -0 and +0 order as equal values */
    c[v].z = z;
    c[v].id = v;
  }
  qsort(c, (size_t)V, sizeof(orc_cand), cand_cmp);
  /* kept set, visited in id order so that ties go to the lowest id */
  unsigned char* keep = (unsigned char*)calloc((size_t)V, 1);
  float* zz = (float*)malloc(sizeof(float) * (size_t)V);
  for (int i = 0; i < k; i++) {
    keep[c[i].id] = 1;
    zz[c[i].id] = c[i].z;
  }
  int have = 0;
  float best_val = 0.0f;
  for (int v = 0; v < V; v++) {
    if (!keep[v]) continue;
    float u = orc_uniform(key0, key1, codebook, frame_ctr, v);
    float l1 = orc_logf(u);
    float a = -l1;
    float l2 = orc_logf(a);
    float g = -l2;
    float val = zz[v] + g;
    if (!have || val > best_val) {
      have = 1;
      best_val = val;
      best = v;
    }
  }
  free(keep);
  free(zz);
  free(c);
  free(lp);
  return best;
}

/* ------------------------------------------------------------------ */
/* One transformer layer at one position                                */
/* ------------------------------------------------------------------ */

typedef struct {
  int H, nq, nkv, d, F;
  double eps, theta;
} layer_dims;

/* x: [H] residual stream, updated. kc, vc: this layer's caches
 * [cap][nkv][d] bf16; position pos is written, positions 0..pos are read. */
static void run_layer(const orc_layer* L, const layer_dims* ld, int use_int8, double* x, int pos,
                      uint16_t* kc, uint16_t* vc) {
  int H = ld->H, nq = ld->nq, nkv = ld->nkv, d = ld->d, F = ld->F;
  double* n = (double*)malloc(sizeof(double) * (size_t)H);
  double* q = (double*)malloc(sizeof(double) * (size_t)nq * d);
  double* k = (double*)malloc(sizeof(double) * (size_t)nkv * d);
  double* v = (double*)malloc(sizeof(double) * (size_t)nkv * d);
  double* a = (double*)malloc(sizeof(double) * (size_t)nq * d);
  double* o = (double*)malloc(sizeof(double) * (size_t)H);
  double* g = (double*)malloc(sizeof(double) * (size_t)F);
  double* u = (double*)malloc(sizeof(double) * (size_t)F);

  /* attention block */
  orc_rmsnorm(x, L->in_norm, H, ld->eps, n);
  orc_linear(n, L->wq, use_int8, nq * d, H, q);
  orc_linear(n, L->wk, use_int8, nkv * d, H, k);
  orc_linear(n, L->wv, use_int8, nkv * d, H, v);
  orc_rope(q, nq, d, pos, ld->theta);
  orc_rope(k, nkv, d, pos, ld->theta);
  for (int i = 0; i < nkv * d; i++) {
    kc[(size_t)pos * nkv * d + i] = orc_to_bf16(k[i]);
    vc[(size_t)pos * nkv * d + i] = orc_to_bf16(v[i]);
  }
  orc_attention(q, kc, vc, pos + 1, nq, nkv, d, a);
  orc_linear(a, L->wo, use_int8, H, nq * d, o);
  for (int i = 0; i < H; i++) x[i] += o[i];

  /* SwiGLU MLP block */
  orc_rmsnorm(x, L->post_norm, H, ld->eps, n);
  orc_linear(n, L->wg, use_int8, F, H, g);
  orc_linear(n, L->wu, use_int8, F, H, u);
  for (int i = 0; i < F; i++) g[i] = orc_silu(g[i]) * u[i];
  orc_linear(g, L->wd, use_int8, H, F, o);
  for (int i = 0; i < H; i++) x[i] += o[i];

  free(n); free(q); free(k); free(v); free(a); free(o); free(g); free(u);
}

static void to_float_row(const double* src, int n, float* dst) {
  for (int i = 0; i < n; i++) dst[i] = (float)src[i];
}

/* projection into the Code Predictor: P(v) = Wp v (+ b) */
static void project(const orc_model* m, const double* v, double* out) {
  const orc_dims* D = &m->d;
  orc_linear(v, m->proj, m->use_int8, D->cp_hidden, D->hidden, out);
  if (D->proj_bias && m->proj_b)
    for (int i = 0; i < D->cp_hidden; i++) out[i] += orc_from_bf16(m->proj_b[i]);
}

int orc_frame_step(const orc_model* m, int B, orc_session* sess, uint16_t* const* kv, int kv_cap,
                   const uint16_t* in_embeds, uint32_t* rng, uint32_t* seen, const int32_t* forced,
                   int32_t* codes_out, uint8_t* eos_out, double* logits_out) {
  const orc_dims* D = &m->d;
  const int H = D->hidden, Hc = D->cp_hidden, V0 = D->vocab0, Vc = D->cp_vocab;
  const int NCB = D->n_codebooks;
  const int seen_words = (V0 + 31) / 32;
  layer_dims tl = {H, D->n_q_heads, D->n_kv_heads, D->head_dim, D->ffn, D->rms_eps, D->rope_theta};
  layer_dims cl = {Hc, D->cp_n_q_heads, D->cp_n_kv_heads, D->cp_head_dim, D->cp_ffn, D->rms_eps,
                   D->cp_rope_theta};
  const size_t t_tok = (size_t)D->n_kv_heads * D->head_dim;       /* one token, one of K/V */
  const size_t c_tok = (size_t)D->cp_n_kv_heads * D->cp_head_dim;

  for (int b = 0; b < B; b++) {
    if (sess[b].kv_len < 0 || sess[b].kv_len >= kv_cap) return -1;
  }

  double* x = (double*)malloc(sizeof(double) * (size_t)H);
  double* h = (double*)malloc(sizeof(double) * (size_t)H);
  double* e = (double*)malloc(sizeof(double) * (size_t)H);
  double* y = (double*)malloc(sizeof(double) * (size_t)Hc);
  double* yn = (double*)malloc(sizeof(double) * (size_t)Hc);
  double* lg = (double*)malloc(sizeof(double) * (size_t)(V0 > Vc ? V0 : Vc));
  float* lf = (float*)malloc(sizeof(float) * (size_t)(V0 > Vc ? V0 : Vc));
  /* Code-Predictor cache for one frame: [cp_layers][2][n_codebooks][nkv][d] */
  uint16_t* ckv = (uint16_t*)calloc((size_t)D->cp_layers * 2 * NCB * c_tok, sizeof(uint16_t));

  for (int b = 0; b < B; b++) {
    orc_session* S = &sess[b];
    uint32_t key0 = rng[4 * b + 0], key1 = rng[4 * b + 1], fctr = rng[4 * b + 2];
    uint32_t* sb = seen ? seen + (size_t)b * seen_words : NULL;
    int pos = S->kv_len;

    /* Talker step */
    for (int i = 0; i < H; i++) x[i] = orc_from_bf16(in_embeds[(size_t)b * H + i]);
    for (int l = 0; l < D->n_layers; l++) {
      uint16_t* base = kv[b] + (size_t)l * 2 * kv_cap * t_tok;
      run_layer(&m->talker[l], &tl, m->use_int8, x, pos, base, base + (size_t)kv_cap * t_tok);
    }
    orc_rmsnorm(x, m->final_norm, H, D->rms_eps, h); /* h_t */
    orc_linear(h, m->head0, m->use_int8, V0, H, lg);
    if (logits_out)
      for (int v = 0; v < V0; v++) logits_out[((size_t)b * NCB + 0) * V0 + v] = lg[v];
    to_float_row(lg, V0, lf);
    int32_t c = orc_sample(lf, V0, 0, S, key0, key1, fctr, sb, D->eos_id, D->n_codes);
    codes_out[(size_t)b * NCB + 0] = c;
    eos_out[b] = (uint8_t)(c == D->eos_id);
    int32_t committed = forced ? forced[(size_t)b * NCB + 0] : c;
    if (sb) sb[committed >> 5] |= 1u << (committed & 31);

    /* Code Predictor: position 0 carries P(h_t); position j (1..15) carries
     * P(E_{j-1}[c_{j-1}]) and its output row gives the logits of codebook j. */
    for (int p = 0; p < NCB; p++) {
      if (p == 0) {
        project(m, h, y);
      } else {
        const uint16_t* E = m->embed[p - 1];
        for (int i = 0; i < H; i++) e[i] = orc_from_bf16(E[(size_t)committed * H + i]);
        project(m, e, y);
      }
      for (int l = 0; l < D->cp_layers; l++) {
        uint16_t* base = ckv + (size_t)l * 2 * NCB * c_tok;
        run_layer(&m->cp[l], &cl, m->use_int8, y, p, base, base + (size_t)NCB * c_tok);
      }
      if (p == 0) continue;
      orc_rmsnorm(y, m->cp_final_norm, Hc, D->rms_eps, yn);
      orc_linear(yn, m->cp_head[p], m->use_int8, Vc, Hc, lg);
      if (logits_out)
        for (int v = 0; v < Vc; v++) logits_out[((size_t)b * NCB + p) * V0 + v] = lg[v];
      to_float_row(lg, Vc, lf);
      int32_t cj = orc_sample(lf, Vc, p, S, key0, key1, fctr, NULL, D->eos_id, D->n_codes);
      codes_out[(size_t)b * NCB + p] = cj;
      committed = forced ? forced[(size_t)b * NCB + p] : cj;
    }

    S->kv_len += 1;
    rng[4 * b + 2] = fctr + 1u;
  }
  free(x); free(h); free(e); free(y); free(yn); free(lg); free(lf); free(ckv);
  return 0;
}

/* Talker prefill (header): the decode step's Talker layers, one prompt token
 * after another, which is the causal prompt pass the pages describe the
 * serving stacks running before the first frame. Always on the BF16 weights:
 * with INT8 decode enabled, prefill stays BF16 ("Qwen3-TTS Native v0.3.0",
 * "What changed"). */
int orc_talker_prefill(const orc_model* m, int B, orc_session* sess, uint16_t* const* kv, int kv_cap,
                       const uint16_t* embeds, int n_tok) {
  const orc_dims* D = &m->d;
  const int H = D->hidden;
  layer_dims tl = {H, D->n_q_heads, D->n_kv_heads, D->head_dim, D->ffn, D->rms_eps, D->rope_theta};
  const size_t t_tok = (size_t)D->n_kv_heads * D->head_dim;
  for (int b = 0; b < B; b++)
    if (sess[b].kv_len < 0 || sess[b].kv_len + n_tok > kv_cap) return -1;
  double* x = (double*)malloc(sizeof(double) * (size_t)H);
  for (int b = 0; b < B; b++) {
    for (int t = 0; t < n_tok; t++) {
      const int pos = sess[b].kv_len + t;
      for (int i = 0; i < H; i++) x[i] = orc_from_bf16(embeds[((size_t)t * B + b) * H + i]);
      for (int l = 0; l < D->n_layers; l++) {
        uint16_t* kc = kv[b] + (size_t)l * 2 * kv_cap * t_tok;
        run_layer(&m->talker[l], &tl, 0, x, pos, kc, kc + (size_t)kv_cap * t_tok);
      }
    }
    sess[b].kv_len += n_tok;
  }
  free(x);
  return 0;
}

void orc_feedback(const orc_model* m, int B, const int32_t* codes, const uint16_t* text, double* out) {
  const int H = m->d.hidden, NCB = m->d.n_codebooks;
  for (int b = 0; b < B; b++) {
    for (int i = 0; i < H; i++) {
      double s = orc_from_bf16(text[(size_t)b * H + i]);
      for (int j = 0; j < NCB; j++) s += orc_from_bf16(m->embed[j][(size_t)codes[(size_t)b * NCB + j] * H + i]);
      out[(size_t)b * H + i] = s;
    }
  }
}
