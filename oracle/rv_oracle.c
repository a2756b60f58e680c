/*
 * CPU oracle for the River-LLM token-level early-exit decode path.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  Plain loops in
 * fp64; no blocking, fusion or reordering beyond the method's own steps.
 *
 * Sources (page title and section):
 *  - paperlayer.ai "River-LLM" summary, section 4 "KV-Shared Exit Layer":
 *    each exit layer is a copy of the backbone layer with the same index,
 *    4-bit weight-only quantized, using the backbone's KV addressing and a
 *    16-bit KV cache.
 *  - same page, section 4 "Inference with Seamless Exit": once the exit
 *    criterion holds, the remaining layers run as exit layers and then the
 *    original LM head produces the logits; prefill uses a sequence-level exit,
 *    generation a token-level exit.
 *  - same page, section 3 "Sequence-level Exit": one exit layer per
 *    sequence, set by the latest-exiting token.
 *  - aitrends.kr article, paragraph on the state transition similarity:
 *    s(l) = cos(h(l-1), h(l)) between the input and output of layer l; exit
 *    when s(l) is greater than tau.
 *  - aitrends.kr article, paragraph on the exit layers: the backbone block's
 *    weights are copied and quantized to W4A16.
 * Readings where the pages are silent are listed beside each function.
 */
#include "rv_oracle.h"

#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define RV_OK 0
#define RV_EINVAL (-1)
#define RV_ENOMEM (-2)
#define RV_ECAPACITY (-4)
#define RV_ESTATE (-5)

#define KV_SENTINEL 0x7FFFu
#define TIE_S 1e-3
#define TIE_LOGIT 1e-2

enum { P_Q = 0, P_K, P_V, P_O, P_G, P_U, P_D, N_PROJ };

typedef struct {
  const uint16_t *attn_norm, *w[N_PROJ], *mlp_norm;
  /* river copy (canonical packing) */
  uint32_t *rq[N_PROJ];
  uint16_t *rs[N_PROJ], *rz[N_PROJ];
} ora_layer;

struct ora_model {
  ora_config c;
  int nthreads;
  const uint16_t *embed, *final_norm, *lm_head;
  ora_layer *layers;
  int group, entry, has_river;
  int cap;      /* last backbone layer kept (L = all): exits are capped there */
  int quantizer; /* river quantizer: 0 RTN, 1 HQQ */
  uint16_t *kv; /* [L][2][max_batch][Hkv][max_seq][hd] */
  int32_t *len; /* [max_batch] */
};

/* ------------------------------------------------------------------ */
/* 16-bit formats                                                      */
/* ------------------------------------------------------------------ */

static void fmt_params(int act, int *p, int *emin, int *emax) {
  if (act == 1) { *p = 8; *emin = -126; *emax = 127; }  /* bf16 */
  else { *p = 11; *emin = -14; *emax = 15; }           /* fp16 */
}

/* Round to the nearest value of the 16-bit format, ties to even. */
double ora_act16_round(double x, int act) {
  if (x == 0.0 || !isfinite(x)) return x;
  int p, emin, emax;
  fmt_params(act, &p, &emin, &emax);
  double a = fabs(x);
  int e;
  frexp(a, &e);
  int E = e - 1;
  if (E < emin) E = emin;
  double quantum = ldexp(1.0, E - p + 1);
  double r = nearbyint(a / quantum) * quantum;
  if (r >= ldexp(1.0, emax + 1)) r = INFINITY;
  return copysign(r, x);
}

uint16_t ora_act16_encode(double x, int act) {
  int p, emin, emax;
  fmt_params(act, &p, &emin, &emax);
  int ebits = act == 1 ? 8 : 5, bias = act == 1 ? 127 : 15;
  uint16_t sign = signbit(x) ? (uint16_t)0x8000u : 0;
  if (isnan(x)) return (uint16_t)(act == 1 ? 0x7FC0 : 0x7E00);
  double r = ora_act16_round(x, act);
  double a = fabs(r);
  if (isinf(a)) return (uint16_t)(sign | (((1u << ebits) - 1u) << (p - 1)));
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);
  int E = e - 1;
  if (E < emin) {
    uint32_t mant = (uint32_t)(a / ldexp(1.0, emin - p + 1));
    return (uint16_t)(sign | mant);
  }
  uint32_t mant = (uint32_t)(a / ldexp(1.0, E - p + 1)) - (1u << (p - 1));
  return (uint16_t)(sign | ((uint32_t)(E + bias) << (p - 1)) | mant);
}

static double decode_bits(uint16_t b, int act) {
  double sign = (b & 0x8000u) ? -1.0 : 1.0;
  if (act == 1) {
    int ex = (b >> 7) & 0xFF, man = b & 0x7F;
    if (ex == 0xFF) return man ? NAN : sign * INFINITY;
    if (ex == 0) return sign * ldexp((double)man, -133);
    return sign * ldexp((double)(128 + man), ex - 134);
  }
  int ex = (b >> 10) & 0x1F, man = b & 0x3FF;
  if (ex == 0x1F) return man ? NAN : sign * INFINITY;
  if (ex == 0) return sign * ldexp((double)man, -24);
  return sign * ldexp((double)(1024 + man), ex - 25);
}

/* Lookup tables of decode_bits for all 65536 patterns of each type. */
static double g_decode_tab[2][65536];
static pthread_once_t g_decode_once = PTHREAD_ONCE_INIT;

static void build_decode_tab(void) {
  for (int a = 0; a < 2; ++a)
    for (int b = 0; b < 65536; ++b) g_decode_tab[a][b] = decode_bits((uint16_t)b, a);
}

double ora_act16_decode(uint16_t b, int act) {
  pthread_once(&g_decode_once, build_decode_tab);
  return g_decode_tab[act == 1][b];
}

/* ------------------------------------------------------------------ */
/* Threads: split [0, n) into contiguous chunks                         */
/* ------------------------------------------------------------------ */

typedef void (*range_fn)(void *ctx, int lo, int hi);
typedef struct { range_fn fn; void *ctx; int lo, hi; } par_job;

static void *par_worker(void *p) {
  par_job *j = (par_job *)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void par_for(int nthreads, int n, range_fn fn, void *ctx) {
  if (n <= 0) return;
  if (nthreads > n) nthreads = n;
  if (nthreads <= 1) { fn(ctx, 0, n); return; }
  pthread_t th[256];
  par_job jobs[256];
  if (nthreads > 256) nthreads = 256;
  int chunk = (n + nthreads - 1) / nthreads, started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].fn = fn; jobs[t].ctx = ctx;
    jobs[t].lo = t * chunk;
    jobs[t].hi = jobs[t].lo + chunk < n ? jobs[t].lo + chunk : n;
    if (jobs[t].lo >= jobs[t].hi) break;
    if (pthread_create(&th[t], NULL, par_worker, &jobs[t]) != 0) { fn(ctx, jobs[t].lo, jobs[t].hi); continue; }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* Primitives                                                          */
/* ------------------------------------------------------------------ */

/* s(l) = cos(h(l-1), h(l)) (aitrends.kr, state transition similarity).
 * Reading: the denominator is floored at 1e-8 so a zero vector gives 0. */
double ora_cosine(const double *a, const double *b, int n) {
  double dot = 0, na = 0, nb = 0;
  for (int i = 0; i < n; ++i) { dot += a[i] * b[i]; na += a[i] * a[i]; nb += b[i] * b[i]; }
  double den = sqrt(na) * sqrt(nb);
  if (den < 1e-8) den = 1e-8;
  return dot / den;
}

/* RMSNorm as in the Llama decoder: h / sqrt(mean(h^2) + eps) * gamma,
 * rounded to the 16-bit activation type because it feeds a matrix product
 * (W4A16 / 16-bit backbone: activations are 16-bit). */
void ora_rmsnorm(const double *h, const uint16_t *gamma, int d, double eps, int act, double *out) {
  double ss = 0;
  for (int i = 0; i < d; ++i) ss += h[i] * h[i];
  double r = 1.0 / sqrt(ss / d + eps);
  for (int i = 0; i < d; ++i) out[i] = ora_act16_round(h[i] * r * ora_act16_decode(gamma[i], act), act);
}

/* Rotary embedding, rotate-half pairing (i, i + hd/2), angle pos * theta^(-2i/hd). */
void ora_rope(double *v, int hd, int pos, double theta) {
  int half = hd / 2;
  for (int i = 0; i < half; ++i) {
    double inv = pow(theta, -2.0 * (double)i / (double)hd);
    double ang = (double)pos * inv;
    double c = cos(ang), s = sin(ang);
    double a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = a * s + b * c;
  }
}

/* One query head over T cached positions: softmax(q.K^T / sqrt(hd)) V. */
void ora_attention(const double *q, const uint16_t *K, const uint16_t *V, int T, int hd, int act, double *out) {
  double *sc = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
  double scale = 1.0 / sqrt((double)hd), mx = -INFINITY;
  for (int t = 0; t < T; ++t) {
    double dot = 0;
    for (int i = 0; i < hd; ++i) dot += q[i] * ora_act16_decode(K[(size_t)t * hd + i], act);
    sc[t] = dot * scale;
    if (sc[t] > mx) mx = sc[t];
  }
  double den = 0;
  for (int t = 0; t < T; ++t) { sc[t] = exp(sc[t] - mx); den += sc[t]; }
  for (int i = 0; i < hd; ++i) out[i] = 0;
  for (int t = 0; t < T; ++t) {
    double p = sc[t] / den;
    for (int i = 0; i < hd; ++i) out[i] += p * ora_act16_decode(V[(size_t)t * hd + i], act);
  }
  free(sc);
}

/* Greedy pick: largest value, lowest index on ties. */
int ora_argmax(const double *v, int n) {
  int best = 0;
  for (int i = 1; i < n; ++i)
    if (v[i] > v[best]) best = i;
  return best;
}

double ora_silu(double g) { return g / (1.0 + exp(-g)); }

/* ------------------------------------------------------------------ */
/* River construction: round-to-nearest int4, asymmetric, per group    */
/* ------------------------------------------------------------------ */

static float f16_bits_to_float(uint16_t b) { return (float)ora_act16_decode(b, 0); }

/* One group of n weights (aitrends.kr: copy the backbone weights, quantize to
 * 4 bits).  Reading (classic asymmetric RTN, fp32 IEEE arithmetic):
 *   mn, mx = group min, max;  s = fp16_rn((mx - mn) / 15);
 *   s == 0  ->  s = 1, z = 0 (degenerate group);  s = inf -> error;
 *   z = clamp(rint(-mn / s), 0, 15);  q = clamp(rint(w / s) + z, 0, 15);
 *   dequantized weight = (q - z) * s.  rint rounds half to even. */
int ora_rtn_group(const uint16_t *w, int n, int act, uint8_t *q, uint16_t *s_out, uint16_t *z_out) {
  float mn = INFINITY, mx = -INFINITY;
  for (int i = 0; i < n; ++i) {
    float v = (float)ora_act16_decode(w[i], act);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  volatile float range = mx - mn;
  volatile float sf = range / 15.0f;
  uint16_t s16 = ora_act16_encode((double)sf, 0);
  float s = f16_bits_to_float(s16);
  if (isinf(s) || isnan(s)) return RV_EINVAL;
  float z;
  if (s == 0.0f) {
    s16 = 0x3C00; /* 1.0 */
    s = 1.0f;
    z = 0.0f;
  } else {
    volatile float t = -mn / s;
    z = rintf(t);
    if (z <= 0.0f) z = 0.0f; /* also maps -0 to +0 */
    if (z > 15.0f) z = 15.0f;
  }
  for (int i = 0; i < n; ++i) {
    volatile float v = (float)ora_act16_decode(w[i], act);
    volatile float t = v / s;
    float r = rintf(t) + z;
    if (r < 0.0f) r = 0.0f;
    if (r > 15.0f) r = 15.0f;
    q[i] = (uint8_t)r;
  }
  *s_out = s16;
  *z_out = ora_act16_encode((double)z, 0);
  return RV_OK;
}

/* HQQ (Badri and Shaji, "Half-Quadratic Quantization of Large Machine
 * Learning Models", 2023; the pages' river quantizer, paperlayer.ai appendix
 * A.1): the scale stays the min/max one, s = fp16_rn((mx - mn) / 15), and the
 * float zero z (start: -mn / s) minimises the lp norm (p = 0.7) of the
 * dequantization error by half-quadratic splitting.  Per iteration, in this
 * order: q = clamp(rint(w / s + z), 0, 15); w_r = (q - z) s;
 * e = shrink(w - w_r, beta) with shrink(x) = sign(x) max(|x| - |x|^(p-1) / beta, 0);
 * z = mean(q - (w - e) / s); beta = beta * kappa; the mean |w - w_r| must keep
 * falling, else stop (the zero of the stopping iteration is kept).  beta = 10,
 * kappa = 1.01, at most 20 iterations.  Reading of the pages' storage: the
 * final zero is rounded to fp16 and the codes are taken again with it, so
 * (q - z) s is the stored dequantization.  Degenerate groups as in RTN.
 * Every step is one IEEE fp32 operation; |x|^(p-1) = 2^((p-1) log2 x) with
 * log2 from the atanh series on the mantissa, log2(m) = (2 / ln 2)(u + u^3/3
 * + ... + u^11/11), u = (m - 1)/(m + 1), and 2^f = e^(f ln 2) from its Taylor
 * series to degree 8, so the GPU quantizer can repeat it bit for bit. */
static float hqq_pow_pm1(float a) { /* a^(p - 1), p = 0.7, a > 0 finite */
  uint32_t b;
  memcpy(&b, &a, 4);
  int ex = (int)(b >> 23);
  if (ex == 0) { /* subnormal: scale by 2^64 */
    float t = a * 18446744073709551616.0f;
    memcpy(&b, &t, 4);
    ex = (int)(b >> 23) - 64;
  }
  ex -= 127;
  const uint32_t mb = (b & 0x7FFFFFu) | 0x3F800000u;
  float m;
  memcpy(&m, &mb, 4);
  const float u = (m - 1.0f) / (m + 1.0f), u2 = u * u;
  float ser = 1.0f / 11.0f;
  ser = ser * u2 + 1.0f / 9.0f;
  ser = ser * u2 + 1.0f / 7.0f;
  ser = ser * u2 + 1.0f / 5.0f;
  ser = ser * u2 + 1.0f / 3.0f;
  ser = ser * u2 + 1.0f;
  const float lg = (float)ex + (ser * u) * 2.88539008f;
  const float y = -0.3f * lg;
  const float fi = floorf(y), f = y - fi;
  const float t = f * 0.693147182f;
  float ep = 1.0f / 40320.0f;
  ep = ep * t + 1.0f / 5040.0f;
  ep = ep * t + 1.0f / 720.0f;
  ep = ep * t + 1.0f / 120.0f;
  ep = ep * t + 1.0f / 24.0f;
  ep = ep * t + 1.0f / 6.0f;
  ep = ep * t + 0.5f;
  ep = ep * t + 1.0f;
  ep = ep * t + 1.0f;
  const int i = (int)fi;
  const uint32_t pb = (uint32_t)(i + 127) << 23;
  float p2;
  memcpy(&p2, &pb, 4);
  return ep * p2;
}

/* The |x|^(p-1) step alone, for its pin against the mathematical power. */
float ora_hqq_pow_pm1(float a) { return hqq_pow_pm1(a); }

int ora_hqq_group(const uint16_t *w, int n, int act, uint8_t *q, uint16_t *s_out, uint16_t *z_out) {
  float mn = INFINITY, mx = -INFINITY;
  for (int i = 0; i < n; ++i) {
    float v = (float)ora_act16_decode(w[i], act);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  float range = mx - mn;
  float sf = range / 15.0f;
  uint16_t s16 = ora_act16_encode((double)sf, 0);
  float s = f16_bits_to_float(s16);
  if (isinf(s) || isnan(s)) return RV_EINVAL;
  if (s == 0.0f) return ora_rtn_group(w, n, act, q, s_out, z_out); /* degenerate: s = 1, z = 0 */
  float z = -mn / s, beta = 10.0f, best = INFINITY;
  for (int it = 0; it < 20; ++it) {
    float zsum = 0.0f, esum = 0.0f;
    for (int i = 0; i < n; ++i) {
      const float v = (float)ora_act16_decode(w[i], act);
      float r = rintf(v / s + z);
      if (r < 0.0f) r = 0.0f;
      if (r > 15.0f) r = 15.0f;
      const float wr = (r - z) * s, res = v - wr;
      float e = 0.0f;
      if (res != 0.0f) {
        const float a = fabsf(res), sh = a - hqq_pow_pm1(a) / beta;
        if (sh > 0.0f) e = res < 0.0f ? -sh : sh;
      }
      zsum = zsum + (r - (v - e) / s);
      esum = esum + fabsf(res);
    }
    z = zsum / (float)n;
    beta = beta * 1.01f;
    const float err = esum / (float)n;
    if (err < best) best = err;
    else break;
  }
  const uint16_t z16 = ora_act16_encode((double)z, 0);
  const float zq = f16_bits_to_float(z16);
  for (int i = 0; i < n; ++i) {
    const float v = (float)ora_act16_decode(w[i], act);
    float r = rintf(v / s + zq);
    if (r < 0.0f) r = 0.0f;
    if (r > 15.0f) r = 15.0f;
    q[i] = (uint8_t)r;
  }
  *s_out = s16;
  *z_out = z16;
  return RV_OK;
}

static void proj_dims(const ora_config *c, int proj, int *N, int *K) {
  int d = c->d_model, qd = c->n_heads * c->head_dim, kvd = c->n_kv_heads * c->head_dim;
  switch (proj) {
    case P_Q: *N = qd; *K = d; break;
    case P_K: case P_V: *N = kvd; *K = d; break;
    case P_O: *N = d; *K = qd; break;
    case P_G: case P_U: *N = c->ffn; *K = d; break;
    default: *N = d; *K = c->ffn; break;
  }
}

typedef struct { ora_model *m; ora_layer *ly; int proj, N, K, G, err; } quant_ctx;

static void quant_rows(void *p, int lo, int hi) {
  quant_ctx *qc = (quant_ctx *)p;
  const ora_model *m = qc->m;
  int K = qc->K, G = qc->G, g = m->group;
  uint8_t *qq = (uint8_t *)malloc((size_t)K);
  for (int n = lo; n < hi; ++n) {
    const uint16_t *row = qc->ly->w[qc->proj] + (size_t)n * K;
    for (int gi = 0; gi < G; ++gi) {
      int k0 = gi * g, cnt = K - k0 < g ? K - k0 : g;
      int (*quant)(const uint16_t *, int, int, uint8_t *, uint16_t *, uint16_t *) =
          m->quantizer == 1 ? ora_hqq_group : ora_rtn_group;
      if (quant(row + k0, cnt, m->c.act_dtype, qq + k0, &qc->ly->rs[qc->proj][(size_t)n * G + gi],
                &qc->ly->rz[qc->proj][(size_t)n * G + gi]) != RV_OK)
        qc->err = 1;
    }
    /* canonical packing: word w of row n holds q[n][8w + j] in bits 4j..4j+3 */
    uint32_t *dst = qc->ly->rq[qc->proj] + (size_t)n * (K / 8);
    for (int w = 0; w < K / 8; ++w) {
      uint32_t word = 0;
      for (int j = 0; j < 8; ++j) word |= (uint32_t)qq[8 * w + j] << (4 * j);
      dst[w] = word;
    }
  }
  free(qq);
}

int ora_quantize_river(ora_model *m, int group, int entry_layer) {
  if (!m || group < 8 || group % 8 || entry_layer < 1 || entry_layer > m->c.n_layers) return RV_EINVAL;
  m->group = group;
  m->entry = entry_layer;
  for (int l = 0; l < m->c.n_layers; ++l) {
    ora_layer *ly = &m->layers[l];
    for (int p = 0; p < N_PROJ; ++p) {
      int N, K;
      proj_dims(&m->c, p, &N, &K);
      int G = (K + group - 1) / group;
      free(ly->rq[p]); free(ly->rs[p]); free(ly->rz[p]);
      ly->rq[p] = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)N * (K / 8));
      ly->rs[p] = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)N * G);
      ly->rz[p] = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)N * G);
      if (!ly->rq[p] || !ly->rs[p] || !ly->rz[p]) return RV_ENOMEM;
      quant_ctx qc = {m, ly, p, N, K, G, 0};
      par_for(m->nthreads, N, quant_rows, &qc);
      if (qc.err) return RV_EINVAL;
    }
  }
  m->has_river = 1;
  return RV_OK;
}

int ora_export_river(const ora_model *m, int layer, int proj, uint32_t *q, uint16_t *s, uint16_t *z) {
  if (!m || !m->has_river || layer < 1 || layer > m->c.n_layers || proj < 0 || proj >= N_PROJ) return RV_EINVAL;
  int N, K;
  proj_dims(&m->c, proj, &N, &K);
  int G = (K + m->group - 1) / m->group;
  const ora_layer *ly = &m->layers[layer - 1];
  if (q) memcpy(q, ly->rq[proj], sizeof(uint32_t) * (size_t)N * (K / 8));
  if (s) memcpy(s, ly->rs[proj], sizeof(uint16_t) * (size_t)N * G);
  if (z) memcpy(z, ly->rz[proj], sizeof(uint16_t) * (size_t)N * G);
  return RV_OK;
}

/* ------------------------------------------------------------------ */
/* Matrix product Y[t][n] = sum_k W[n][k] X[t][k]                      */
/* W is either the 16-bit backbone matrix or the river copy, whose     */
/* element is (q - z) * s.                                             */
/* ------------------------------------------------------------------ */

typedef struct {
  const ora_model *m;
  const ora_layer *ly;
  int proj, river, N, K, ntok;
  const double *X;
  double *Y;
} mm_ctx;

static void mm_rows(void *p, int lo, int hi) {
  mm_ctx *c = (mm_ctx *)p;
  int K = c->K, act = c->m->c.act_dtype;
  double *w = (double *)malloc(sizeof(double) * (size_t)K);
  for (int n = lo; n < hi; ++n) {
    if (!c->river) {
      const uint16_t *row = c->ly->w[c->proj] + (size_t)n * K;
      for (int k = 0; k < K; ++k) w[k] = ora_act16_decode(row[k], act);
    } else {
      int g = c->m->group, G = (K + g - 1) / g;
      const uint32_t *qrow = c->ly->rq[c->proj] + (size_t)n * (K / 8);
      for (int gi = 0; gi < G; ++gi) {
        double s = ora_act16_decode(c->ly->rs[c->proj][(size_t)n * G + gi], 0);
        double z = ora_act16_decode(c->ly->rz[c->proj][(size_t)n * G + gi], 0);
        for (int k = gi * g; k < K && k < (gi + 1) * g; ++k) {
          int qv = (int)((qrow[k / 8] >> (4 * (k % 8))) & 0xFu);
          w[k] = ((double)qv - z) * s;
        }
      }
    }
    for (int t = 0; t < c->ntok; ++t) {
      const double *x = c->X + (size_t)t * K;
      double acc = 0;
      for (int k = 0; k < K; ++k) acc += w[k] * x[k];
      c->Y[(size_t)t * c->N + n] = acc;
    }
  }
  free(w);
}

static void matmul(const ora_model *m, const ora_layer *ly, int proj, int river, int ntok, const double *X, double *Y) {
  mm_ctx c;
  c.m = m; c.ly = ly; c.proj = proj; c.river = river; c.ntok = ntok; c.X = X; c.Y = Y;
  proj_dims(&m->c, proj, &c.N, &c.K);
  par_for(m->nthreads, c.N, mm_rows, &c);
}

/* ------------------------------------------------------------------ */
/* KV cache: one set shared by backbone and river layers               */
/* (paperlayer.ai section 4 and appendix A.3: a single KV-cache set;   */
/*  aitrends.kr: the same KV addressing for backbone and exit layers)  */
/* ------------------------------------------------------------------ */

static size_t kv_index(const ora_model *m, int l0, int kv01, int b, int g, int p) {
  const ora_config *c = &m->c;
  return (((((size_t)l0 * 2 + kv01) * c->max_batch + b) * c->n_kv_heads + g) * c->max_seq + p) * c->head_dim;
}

size_t ora_kv_bytes(const ora_model *m) {
  const ora_config *c = &m->c;
  return (size_t)c->n_layers * 2 * c->max_batch * c->n_kv_heads * (size_t)c->max_seq * c->head_dim * 2;
}

/* ------------------------------------------------------------------ */
/* One decoder layer (backbone or its river copy) over a list of       */
/* tokens that share the path.  Tokens of one row come in position     */
/* order; every token writes its K/V into slot (l, row, pos).          */
/* ------------------------------------------------------------------ */

typedef struct {
  const ora_model *m;
  int l0, ntok;
  const int *row, *pos;
  const double *Q; /* [ntok][H*hd], act16-rounded after RoPE */
  double *O;       /* [ntok][H*hd] */
} attn_ctx;

static void attn_tokens(void *p, int lo, int hi) {
  attn_ctx *a = (attn_ctx *)p;
  const ora_config *c = &a->m->c;
  int H = c->n_heads, hd = c->head_dim, grp = c->n_heads / c->n_kv_heads;
  double *o = (double *)malloc(sizeof(double) * (size_t)hd);
  for (int i = lo; i < hi; ++i) {
    int t = i / H, h = i % H, g = h / grp;
    const uint16_t *K = a->m->kv + kv_index(a->m, a->l0, 0, a->row[t], g, 0);
    const uint16_t *V = a->m->kv + kv_index(a->m, a->l0, 1, a->row[t], g, 0);
    ora_attention(a->Q + (size_t)t * H * hd + (size_t)h * hd, K, V, a->pos[t] + 1, hd, c->act_dtype, o);
    for (int j = 0; j < hd; ++j) a->O[(size_t)t * H * hd + (size_t)h * hd + j] = ora_act16_round(o[j], c->act_dtype);
  }
  free(o);
}

static void layer_apply(ora_model *m, int l0, int river, int ntok, const int *row, const int *pos, double *Hs) {
  const ora_config *c = &m->c;
  const ora_layer *ly = &m->layers[l0];
  int d = c->d_model, hd = c->head_dim, H = c->n_heads, Hkv = c->n_kv_heads, F = c->ffn, act = c->act_dtype;
  int qd = H * hd, kvd = Hkv * hd;
  size_t nt = (size_t)ntok;
  double *X = (double *)malloc(sizeof(double) * nt * (d > F ? d : F));
  double *Q = (double *)malloc(sizeof(double) * nt * qd);
  double *Kx = (double *)malloc(sizeof(double) * nt * kvd);
  double *Vx = (double *)malloc(sizeof(double) * nt * kvd);
  double *O = (double *)malloc(sizeof(double) * nt * qd);
  double *Y = (double *)malloc(sizeof(double) * nt * d);
  double *G = (double *)malloc(sizeof(double) * nt * F);
  double *U = (double *)malloc(sizeof(double) * nt * F);

  /* attention sub-block */
  for (int t = 0; t < ntok; ++t) ora_rmsnorm(Hs + (size_t)t * d, ly->attn_norm, d, c->rms_eps, act, X + (size_t)t * d);
  matmul(m, ly, P_Q, river, ntok, X, Q);
  matmul(m, ly, P_K, river, ntok, X, Kx);
  matmul(m, ly, P_V, river, ntok, X, Vx);
  for (int t = 0; t < ntok; ++t) {
    for (int h = 0; h < H; ++h) {
      double *q = Q + (size_t)t * qd + (size_t)h * hd;
      ora_rope(q, hd, pos[t], c->rope_theta);
      for (int j = 0; j < hd; ++j) q[j] = ora_act16_round(q[j], act);
    }
    for (int g = 0; g < Hkv; ++g) {
      double *k = Kx + (size_t)t * kvd + (size_t)g * hd;
      const double *v = Vx + (size_t)t * kvd + (size_t)g * hd;
      ora_rope(k, hd, pos[t], c->rope_theta);
      uint16_t *ks = m->kv + kv_index(m, l0, 0, row[t], g, pos[t]);
      uint16_t *vs = m->kv + kv_index(m, l0, 1, row[t], g, pos[t]);
      for (int j = 0; j < hd; ++j) { ks[j] = ora_act16_encode(k[j], act); vs[j] = ora_act16_encode(v[j], act); }
    }
  }
  attn_ctx ac = {m, l0, ntok, row, pos, Q, O};
  par_for(m->nthreads, ntok * H, attn_tokens, &ac);
  matmul(m, ly, P_O, river, ntok, O, Y);
  for (size_t i = 0; i < nt * d; ++i) Hs[i] += Y[i];

  /* MLP sub-block (SwiGLU) */
  for (int t = 0; t < ntok; ++t) ora_rmsnorm(Hs + (size_t)t * d, ly->mlp_norm, d, c->rms_eps, act, X + (size_t)t * d);
  matmul(m, ly, P_G, river, ntok, X, G);
  matmul(m, ly, P_U, river, ntok, X, U);
  for (size_t i = 0; i < nt * F; ++i) X[i] = ora_act16_round(ora_silu(G[i]) * U[i], act);
  matmul(m, ly, P_D, river, ntok, X, Y);
  for (size_t i = 0; i < nt * d; ++i) Hs[i] += Y[i];

  free(X); free(Q); free(Kx); free(Vx); free(O); free(Y); free(G); free(U);
}

/* ------------------------------------------------------------------ */
/* LM head: the original head of the backbone (never quantized)        */
/* ------------------------------------------------------------------ */

typedef struct { const ora_model *m; const double *y; double *logits; } head_ctx;

static void head_rows(void *p, int lo, int hi) {
  head_ctx *hc = (head_ctx *)p;
  const ora_config *c = &hc->m->c;
  int d = c->d_model;
  for (int v = lo; v < hi; ++v) {
    const uint16_t *row = hc->m->lm_head + (size_t)v * d;
    double acc = 0;
    for (int k = 0; k < d; ++k) acc += ora_act16_decode(row[k], c->act_dtype) * hc->y[k];
    hc->logits[v] = acc;
  }
}

/* Returns the next id; *forced is set when the oracle took the GPU's id. */
static int lm_head_pick(ora_model *m, const double *h, double *logits, int tf_id, int *forced) {
  const ora_config *c = &m->c;
  double *y = (double *)malloc(sizeof(double) * (size_t)c->d_model);
  ora_rmsnorm(h, m->final_norm, c->d_model, c->rms_eps, c->act_dtype, y);
  head_ctx hc = {m, y, logits};
  par_for(m->nthreads, c->vocab, head_rows, &hc);
  free(y);
  int best = ora_argmax(logits, c->vocab);
  double second = -INFINITY;
  for (int v = 0; v < c->vocab; ++v)
    if (v != best && logits[v] > second) second = logits[v];
  *forced = 0;
  if (tf_id >= 0 && tf_id < c->vocab && logits[best] - second < TIE_LOGIT && tf_id != best) {
    *forced = 1;
    return tf_id;
  }
  return best;
}

/* ------------------------------------------------------------------ */
/* Prefill: sequence-level exit                                        */
/* ------------------------------------------------------------------ */

/* Backbone offloading (paperlayer.ai section 4, Backbone Offloading): only
 * backbone layers 1..cap stay; a row still in the backbone after layer cap
 * continues in the river.  cap in 1..L; needs the river. */
int ora_set_exit_cap(ora_model *m, int cap) {
  if (!m || cap < 1 || cap > m->c.n_layers) return RV_EINVAL;
  if (!m->has_river && cap < m->c.n_layers) return RV_ESTATE;
  m->cap = cap;
  return RV_OK;
}

/* Host threads the row loops are split over (1..256); results do not depend
 * on it (every row's sums run in one thread, in a fixed order). */
int ora_set_threads(ora_model *m, int nthreads) {
  if (!m || nthreads < 1 || nthreads > 256) return RV_EINVAL;
  m->nthreads = nthreads;
  return RV_OK;
}

/* River quantizer for the next ora_quantize_river: 0 RTN, 1 HQQ. */
int ora_set_quantizer(ora_model *m, int method) {
  if (!m || (method != 0 && method != 1)) return RV_EINVAL;
  m->quantizer = method;
  return RV_OK;
}

int ora_prefill(ora_model *m, const int32_t *tokens, int B, int T0, double tau, int fixed_exit,
                const int32_t *tf_exit, const int32_t *tf_ids, int32_t *next_ids, int32_t *exit_layer,
                double *dbg_smin, double *dbg_hidden_last, double *dbg_logits, int32_t *n_forced) {
  if (!m || !tokens || B < 1 || B > m->c.max_batch || T0 < 1 || T0 > m->c.max_seq) return RV_EINVAL;
  const ora_config *c = &m->c;
  int L = c->n_layers, d = c->d_model;
  if (fixed_exit > L || fixed_exit < -1) return RV_EINVAL;
  if (fixed_exit > m->cap) return RV_EINVAL;
  if (!m->has_river && fixed_exit != L) return RV_ESTATE;
  for (int i = 0; i < B * T0; ++i)
    if (tokens[i] < 0 || tokens[i] >= c->vocab) return RV_EINVAL;
  if (n_forced) { n_forced[0] = 0; n_forced[1] = 0; }
  double *Hs = (double *)malloc(sizeof(double) * (size_t)T0 * d);
  double *Hin = (double *)malloc(sizeof(double) * (size_t)T0 * d);
  double *logits = (double *)malloc(sizeof(double) * (size_t)c->vocab);
  int *row = (int *)malloc(sizeof(int) * (size_t)T0), *pos = (int *)malloc(sizeof(int) * (size_t)T0);
  for (int b = 0; b < B; ++b) {
    for (int t = 0; t < T0; ++t) {
      row[t] = b; pos[t] = t;
      for (int i = 0; i < d; ++i)
        Hs[(size_t)t * d + i] = ora_act16_decode(m->embed[(size_t)tokens[b * T0 + t] * d + i], c->act_dtype);
    }
    if (dbg_hidden_last)
      memcpy(dbg_hidden_last + (size_t)b * d, Hs + (size_t)(T0 - 1) * d, sizeof(double) * d);
    int river = fixed_exit == 0;
    int e_seq = fixed_exit >= 0 ? fixed_exit : L;
    for (int l = 1; l <= L; ++l) {
      memcpy(Hin, Hs, sizeof(double) * (size_t)T0 * d);
      layer_apply(m, l - 1, river, T0, row, pos, Hs);
      if (dbg_hidden_last)
        memcpy(dbg_hidden_last + ((size_t)l * B + b) * d, Hs + (size_t)(T0 - 1) * d, sizeof(double) * d);
      if (dbg_smin) dbg_smin[(size_t)(l - 1) * B + b] = NAN;
      if (river) continue;
      if (fixed_exit >= 0) {
        if (l == fixed_exit) river = 1;
      } else if (l >= m->entry && l <= L - 1) {
        /* the latest-exiting token sets the depth: exit when every token's
         * similarity exceeds tau, i.e. when the minimum does */
        double smin = INFINITY;
        for (int t = 0; t < T0; ++t) {
          double s = ora_cosine(Hin + (size_t)t * d, Hs + (size_t)t * d, d);
          if (s < smin) smin = s;
        }
        if (dbg_smin) dbg_smin[(size_t)(l - 1) * B + b] = smin;
        int go = smin > tau;
        if (tf_exit && fabs(smin - tau) <= TIE_S) {
          int g2 = tf_exit[b] == l;
          if (g2 != go && n_forced) n_forced[0]++;
          go = g2;
        }
        if (go) { e_seq = l; river = 1; }
      }
      /* backbone offloading: layers after the cap exist only in the river */
      if (!river && l >= m->cap && l < L) { e_seq = l; river = 1; }
    }
    m->len[b] = T0;
    int forced = 0;
    next_ids[b] = lm_head_pick(m, Hs + (size_t)(T0 - 1) * d, logits, tf_ids ? tf_ids[b] : -1, &forced);
    if (forced && n_forced) n_forced[1]++;
    if (dbg_logits) memcpy(dbg_logits + (size_t)b * c->vocab, logits, sizeof(double) * c->vocab);
    exit_layer[b] = e_seq;
  }
  free(Hs); free(Hin); free(logits); free(row); free(pos);
  return RV_OK;
}

/* ------------------------------------------------------------------ */
/* Decode step: token-level exit                                       */
/* ------------------------------------------------------------------ */

int ora_decode_step(ora_model *m, const int32_t *tokens, int B, double tau, const int32_t *forced,
                    const int32_t *tf_exit, const int32_t *tf_ids, int32_t *next_ids, int32_t *exit_layer,
                    double *dbg_hidden, double *dbg_s, double *dbg_logits, int32_t *n_forced) {
  if (!m || !tokens || B < 1 || B > m->c.max_batch) return RV_EINVAL;
  const ora_config *c = &m->c;
  int L = c->n_layers, d = c->d_model;
  for (int b = 0; b < B; ++b) {
    if (tokens[b] < 0 || tokens[b] >= c->vocab) return RV_EINVAL;
    if (forced && (forced[b] < 0 || forced[b] > L || forced[b] > m->cap)) return RV_EINVAL;
    if (forced && forced[b] < L && !m->has_river) return RV_ESTATE;
  }
  if (!forced && !m->has_river) return RV_ESTATE;
  for (int b = 0; b < B; ++b)
    if (m->len[b] >= c->max_seq) return RV_ECAPACITY;
  if (n_forced) { n_forced[0] = 0; n_forced[1] = 0; }
  double *Hs = (double *)malloc(sizeof(double) * (size_t)B * d);
  double *Hin = (double *)malloc(sizeof(double) * (size_t)B * d);
  double *Hsub = (double *)malloc(sizeof(double) * (size_t)B * d);
  double *logits = (double *)malloc(sizeof(double) * (size_t)c->vocab);
  int *river = (int *)calloc((size_t)B, sizeof(int));
  int *row = (int *)malloc(sizeof(int) * (size_t)B), *pos = (int *)malloc(sizeof(int) * (size_t)B);
  for (int b = 0; b < B; ++b) {
    for (int i = 0; i < d; ++i)
      Hs[(size_t)b * d + i] = ora_act16_decode(m->embed[(size_t)tokens[b] * d + i], c->act_dtype);
    river[b] = forced ? forced[b] == 0 : 0;
    exit_layer[b] = river[b] ? 0 : L;
  }
  if (dbg_hidden) memcpy(dbg_hidden, Hs, sizeof(double) * (size_t)B * d);
  for (int l = 1; l <= L; ++l) {
    memcpy(Hin, Hs, sizeof(double) * (size_t)B * d);
    /* rows on the same path go through the layer together; both paths
     * write slot (l, row, len[row]) of the one cache */
    for (int path = 0; path < 2; ++path) {
      int n = 0;
      for (int b = 0; b < B; ++b)
        if (river[b] == path) {
          row[n] = b; pos[n] = m->len[b];
          memcpy(Hsub + (size_t)n * d, Hs + (size_t)b * d, sizeof(double) * d);
          n++;
        }
      if (!n) continue;
      layer_apply(m, l - 1, path, n, row, pos, Hsub);
      for (int i = 0; i < n; ++i) memcpy(Hs + (size_t)row[i] * d, Hsub + (size_t)i * d, sizeof(double) * d);
    }
    if (dbg_hidden) memcpy(dbg_hidden + (size_t)l * B * d, Hs, sizeof(double) * (size_t)B * d);
    for (int b = 0; b < B; ++b) {
      if (dbg_s) dbg_s[(size_t)(l - 1) * B + b] = NAN;
      if (river[b]) continue;
      double s = ora_cosine(Hin + (size_t)b * d, Hs + (size_t)b * d, d);
      if (dbg_s) dbg_s[(size_t)(l - 1) * B + b] = s;
      if (forced) {
        if (l == forced[b] && l < L) { river[b] = 1; exit_layer[b] = l; }
      } else if (l >= m->entry && l <= L - 1) {
        int go = s > tau;
        if (tf_exit && fabs(s - tau) <= TIE_S) {
          int g2 = tf_exit[b] == l;
          if (g2 != go && n_forced) n_forced[0]++;
          go = g2;
        }
        if (go) { river[b] = 1; exit_layer[b] = l; }
      }
      /* backbone offloading: layers after the cap exist only in the river */
      if (!river[b] && l >= m->cap && l < L) { river[b] = 1; exit_layer[b] = l; }
    }
  }
  for (int b = 0; b < B; ++b) {
    int f = 0;
    next_ids[b] = lm_head_pick(m, Hs + (size_t)b * d, logits, tf_ids ? tf_ids[b] : -1, &f);
    if (f && n_forced) n_forced[1]++;
    if (dbg_logits) memcpy(dbg_logits + (size_t)b * c->vocab, logits, sizeof(double) * c->vocab);
    m->len[b] += 1;
  }
  free(Hs); free(Hin); free(Hsub); free(logits); free(river); free(row); free(pos);
  return RV_OK;
}

/* ------------------------------------------------------------------ */
/* Single layer / head entry points (for layer-by-layer checks)        */
/* ------------------------------------------------------------------ */

int ora_layer_forward(ora_model *m, int layer, int B, const int32_t *river, const double *h_in, double *h_out) {
  if (!m || !river || !h_in || !h_out || layer < 1 || layer > m->c.n_layers || B < 1 || B > m->c.max_batch)
    return RV_EINVAL;
  const int d = m->c.d_model;
  for (int b = 0; b < B; ++b) {
    if (river[b] && !m->has_river) return RV_ESTATE;
    if (m->len[b] >= m->c.max_seq) return RV_ECAPACITY;
  }
  double *Hsub = (double *)malloc(sizeof(double) * (size_t)B * d);
  int *row = (int *)malloc(sizeof(int) * (size_t)B), *pos = (int *)malloc(sizeof(int) * (size_t)B);
  for (int path = 0; path < 2; ++path) {
    int n = 0;
    for (int b = 0; b < B; ++b)
      if ((river[b] != 0) == path) {
        row[n] = b; pos[n] = m->len[b];
        memcpy(Hsub + (size_t)n * d, h_in + (size_t)b * d, sizeof(double) * d);
        n++;
      }
    if (!n) continue;
    layer_apply(m, layer - 1, path, n, row, pos, Hsub);
    for (int i = 0; i < n; ++i) memcpy(h_out + (size_t)row[i] * d, Hsub + (size_t)i * d, sizeof(double) * d);
  }
  free(Hsub); free(row); free(pos);
  return RV_OK;
}

int ora_head(ora_model *m, int B, const double *h, double *logits, int32_t *ids) {
  if (!m || !h || !logits || !ids || B < 1) return RV_EINVAL;
  for (int b = 0; b < B; ++b) {
    int f = 0;
    ids[b] = lm_head_pick(m, h + (size_t)b * m->c.d_model, logits + (size_t)b * m->c.vocab, -1, &f);
  }
  return RV_OK;
}

/* ------------------------------------------------------------------ */
/* Model lifetime and cache access                                     */
/* ------------------------------------------------------------------ */

int ora_create(const ora_config *cfg, const uint16_t *const *weights, int nthreads, ora_model **out) {
  if (!cfg || !weights || !out) return RV_EINVAL;
  const ora_config *c = cfg;
  if (c->n_layers < 1 || c->d_model < 2 || c->n_heads < 1 || c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads ||
      c->head_dim < 2 || c->head_dim % 2 || c->ffn < 1 || c->vocab < 2 || c->max_batch < 1 || c->max_seq < 1 ||
      (c->act_dtype != 0 && c->act_dtype != 1) || c->d_model % 8 || c->ffn % 8 ||
      (c->n_heads * c->head_dim) % 8)
    return RV_EINVAL;
  ora_model *m = (ora_model *)calloc(1, sizeof(ora_model));
  if (!m) return RV_ENOMEM;
  m->c = *cfg;
  m->nthreads = nthreads < 1 ? 1 : nthreads;
  m->embed = weights[0];
  m->final_norm = weights[1];
  m->lm_head = c->tied_embed ? weights[0] : weights[2];
  m->entry = 1;
  m->cap = c->n_layers;
  m->layers = (ora_layer *)calloc((size_t)c->n_layers, sizeof(ora_layer));
  for (int l = 0; l < c->n_layers; ++l) {
    const uint16_t *const *w = weights + 3 + 9 * l;
    ora_layer *ly = &m->layers[l];
    ly->attn_norm = w[0];
    ly->w[P_Q] = w[1]; ly->w[P_K] = w[2]; ly->w[P_V] = w[3]; ly->w[P_O] = w[4];
    ly->mlp_norm = w[5];
    ly->w[P_G] = w[6]; ly->w[P_U] = w[7]; ly->w[P_D] = w[8];
  }
  size_t nkv = ora_kv_bytes(m) / 2;
  m->kv = (uint16_t *)malloc(nkv * 2);
  m->len = (int32_t *)calloc((size_t)c->max_batch, sizeof(int32_t));
  if (!m->kv || !m->len || !m->layers) { ora_free(m); return RV_ENOMEM; }
  for (size_t i = 0; i < nkv; ++i) m->kv[i] = KV_SENTINEL;
  *out = m;
  return RV_OK;
}

void ora_free(ora_model *m) {
  if (!m) return;
  if (m->layers)
    for (int l = 0; l < m->c.n_layers; ++l)
      for (int p = 0; p < N_PROJ; ++p) { free(m->layers[l].rq[p]); free(m->layers[l].rs[p]); free(m->layers[l].rz[p]); }
  free(m->layers);
  free(m->kv);
  free(m->len);
  free(m);
}

int ora_kv_reset(ora_model *m, const int32_t *rows, int n_rows) {
  if (!m) return RV_EINVAL;
  const ora_config *c = &m->c;
  int n = rows ? n_rows : c->max_batch;
  for (int i = 0; i < n; ++i) {
    int b = rows ? rows[i] : i;
    if (b < 0 || b >= c->max_batch) return RV_EINVAL;
  }
  for (int i = 0; i < n; ++i) {
    int b = rows ? rows[i] : i;
    m->len[b] = 0;
    for (int l = 0; l < c->n_layers; ++l)
      for (int kv = 0; kv < 2; ++kv)
        for (int g = 0; g < c->n_kv_heads; ++g) {
          uint16_t *p = m->kv + kv_index(m, l, kv, b, g, 0);
          for (size_t j = 0; j < (size_t)c->max_seq * c->head_dim; ++j) p[j] = KV_SENTINEL;
        }
  }
  return RV_OK;
}

int ora_get_kv(const ora_model *m, uint16_t *dst, size_t bytes) {
  if (!m || !dst || bytes != ora_kv_bytes(m)) return RV_EINVAL;
  memcpy(dst, m->kv, bytes);
  return RV_OK;
}

int ora_set_kv(ora_model *m, const uint16_t *src, size_t bytes, const int32_t *lens) {
  if (!m || !src || !lens || bytes != ora_kv_bytes(m)) return RV_EINVAL;
  for (int b = 0; b < m->c.max_batch; ++b)
    if (lens[b] < 0 || lens[b] > m->c.max_seq) return RV_EINVAL;
  memcpy(m->kv, src, bytes);
  memcpy(m->len, lens, sizeof(int32_t) * (size_t)m->c.max_batch);
  return RV_OK;
}

int ora_get_lens(const ora_model *m, int32_t *lens) {
  if (!m || !lens) return RV_EINVAL;
  memcpy(lens, m->len, sizeof(int32_t) * (size_t)m->c.max_batch);
  return RV_OK;
}
