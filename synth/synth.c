/*
 * Seeded synthetic inputs for the River-LLM decode path (weights, prompts,
 * forced exit layers).  This module holds none of the method's arithmetic:
 * it only draws numbers.  The oracle and the CUDA library both receive the
 * arrays it writes as plain inputs.
 *
 * Generator: splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used counter-style: draw n of stream k is
 * mix(key_k + (n + 1) * 0x9E3779B97F4A7C15), where mix is the splitmix64
 * output function.  Uniforms take the top 53 bits.  Normals use the
 * Box-Muller transform (cosine branch) in double, are scaled by the standard
 * deviation, rounded to fp32 and then to the 16-bit activation type with
 * round-to-nearest-even.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Key of stream (seed, tensor id). */
static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
  return mix64(seed * GOLDEN + mix64(tid + 0x632BE59BD9B4E019ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t n) { return mix64(key + (n + 1) * GOLDEN); }

static inline double u53(uint64_t r) { return (double)(r >> 11) * (1.0 / 9007199254740992.0); }

/* fp32 -> bf16 / fp16 bit patterns, round to nearest even. */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static uint16_t f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t sign = (u >> 16) & 0x8000u;
  uint32_t ex = (u >> 23) & 0xFFu;
  uint32_t man = u & 0x007FFFFFu;
  if (ex == 0xFF) return (uint16_t)(sign | 0x7C00u | (man ? 0x200u : 0u));
  int e = (int)ex - 127;
  if (e > 15) return (uint16_t)(sign | 0x7C00u);
  if (e >= -14) { /* normal half */
    uint32_t m = man | 0x800000u;            /* 24-bit significand */
    uint32_t keep = m >> 13, rem = m & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (keep & 1u))) keep++;
    uint32_t he = (uint32_t)(e + 15);
    if (keep == 0x800u) { keep = 0x400u; he++; }
    if (he >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (he << 10) | (keep & 0x3FFu));
  }
  if (e < -25) return (uint16_t)sign;
  /* subnormal half: value = m * 2^-24 */
  uint32_t m = man | 0x800000u; /* value = m * 2^(e-23) */
  int shift = -e - 1;            /* (e-23) -> -24 : divide by 2^(-24-(e-23)) = 2^(-1-e) */
  uint32_t keep = m >> shift, rem = m & ((1u << shift) - 1u), half = 1u << (shift - 1);
  if (rem > half || (rem == half && (keep & 1u))) keep++;
  return (uint16_t)(sign | keep);
}

typedef struct {
  uint64_t key;
  double stdv;
  int64_t lo, hi;
  int dtype; /* 0 fp16, 1 bf16 */
  uint16_t *out;
} norm_job;

static void *norm_worker(void *p) {
  norm_job *j = (norm_job *)p;
  const double two_pi = 6.283185307179586476925286766559;
  for (int64_t i = j->lo; i < j->hi; ++i) {
    double u1 = u53(draw(j->key, 2 * (uint64_t)i));
    double u2 = u53(draw(j->key, 2 * (uint64_t)i + 1));
    double z = sqrt(-2.0 * log(1.0 - u1)) * cos(two_pi * u2);
    float f = (float)(j->stdv * z);
    j->out[i] = j->dtype ? f32_to_bf16(f) : f32_to_f16(f);
  }
  return NULL;
}

/* n draws of N(0, stdv^2) rounded to the 16-bit type, stream (seed, tid). */
int synth_normal_act16(uint64_t seed, uint64_t tid, double stdv, int64_t n, int dtype,
                       uint16_t *out, int nthreads) {
  if (n < 0 || !out) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < 65536) nthreads = 1;
  pthread_t th[256];
  norm_job jobs[256];
  uint64_t key = stream_key(seed, tid);
  int64_t chunk = (n + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].key = key;
    jobs[t].stdv = stdv;
    jobs[t].lo = (int64_t)t * chunk;
    jobs[t].hi = jobs[t].lo + chunk < n ? jobs[t].lo + chunk : n;
    jobs[t].dtype = dtype;
    jobs[t].out = out;
    if (jobs[t].lo >= jobs[t].hi) break;
    if (nthreads == 1) { norm_worker(&jobs[t]); started = 0; break; }
    pthread_create(&th[t], NULL, norm_worker, &jobs[t]);
    started++;
  }
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  return 0;
}

/* n uniform integers in [0, vocab), stream (seed, tid). */
int synth_uniform_ids(uint64_t seed, uint64_t tid, int64_t n, int32_t vocab, int32_t *out) {
  if (n < 0 || vocab <= 0 || !out) return -1;
  uint64_t key = stream_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) {
    int64_t v = (int64_t)(u53(draw(key, (uint64_t)i)) * (double)vocab);
    out[i] = (int32_t)(v < vocab ? v : vocab - 1);
  }
  return 0;
}

/* Forced exit layers for one decode step: per row, with probability 0.55 a
 * layer uniform in 1..min(5,L), otherwise uniform in 6..L (only the first
 * branch exists when L < 6).  Stream (seed, step). */
int synth_forced_exits(uint64_t seed, uint64_t step, int32_t batch, int32_t n_layers, int32_t *out) {
  if (batch < 0 || n_layers < 1 || !out) return -1;
  uint64_t key = stream_key(seed, 0x4000000000ULL + step);
  int lo_hi = n_layers < 5 ? n_layers : 5;
  for (int32_t b = 0; b < batch; ++b) {
    double c = u53(draw(key, 2 * (uint64_t)b));
    double u = u53(draw(key, 2 * (uint64_t)b + 1));
    int e;
    if (c < 0.55 || n_layers < 6) {
      e = 1 + (int)(u * lo_hi);
      if (e > lo_hi) e = lo_hi;
    } else {
      int span = n_layers - 5;
      e = 6 + (int)(u * span);
      if (e > n_layers) e = n_layers;
    }
    out[b] = e;
  }
  return 0;
}

/* Fill n 16-bit values with one bit pattern (e.g. the RMSNorm gains, 1.0). */
int synth_fill_u16(int64_t n, uint16_t value, uint16_t *out) {
  if (n < 0 || !out) return -1;
  for (int64_t i = 0; i < n; ++i) out[i] = value;
  return 0;
}
