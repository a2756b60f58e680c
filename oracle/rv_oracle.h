/*
 * CPU oracle for the River-LLM token-level early-exit decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the slow, plain reference that
 * the CUDA path is checked against.  Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark load it; the product path never does.
 * It shares no code with the CUDA library.
 *
 * Method source: "River-LLM: Large Language Model Seamless Exit Based on KV
 * Share" (Shen, Zou), as summarised on paperlayer.ai (sections 3 and 4) and
 * aitrends.kr.  Arithmetic is fp64 except where the method fixes a 16-bit
 * storage type (weights, the FP16/BF16 KV cache, 16-bit activations entering
 * a matrix product) or where the quantizer's reading fixes fp32 (see
 * ora_rtn_group).
 */
#ifndef RV_ORACLE_H
#define RV_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ora_config {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int tied_embed; /* 1: LM head is the embedding matrix */
  int act_dtype;  /* 0 = fp16, 1 = bf16 */
  double rms_eps, rope_theta;
  int max_batch, max_seq;
} ora_config;

typedef struct ora_model ora_model;

/* weights: 3 + 9*L pointers to 16-bit arrays (see synth tensor order); the
 * arrays are referenced, not copied, and must outlive the model. */
int ora_create(const ora_config *cfg, const uint16_t *const *weights, int nthreads, ora_model **out);
void ora_free(ora_model *m);

int ora_quantize_river(ora_model *m, int group, int entry_layer);
int ora_export_river(const ora_model *m, int layer, int proj, uint32_t *q, uint16_t *s, uint16_t *z);

/* River quantizer for the next ora_quantize_river: 0 RTN, 1 HQQ. */
int ora_set_quantizer(ora_model *m, int method);
/* One group of n 16-bit weights by HQQ: codes, fp16 scale and zero. */
int ora_hqq_group(const uint16_t *w, int n, int act, uint8_t *q, uint16_t *s_out, uint16_t *z_out);
float ora_hqq_pow_pm1(float a); /* a^(p - 1), p = 0.7, the HQQ shrink's power */
/* Backbone offloading: keep backbone layers 1..cap; exits are capped at cap. */
int ora_set_exit_cap(ora_model *m, int cap);
int ora_set_threads(ora_model *m, int nthreads);
int ora_prefill(ora_model *m, const int32_t *tokens, int B, int T0, double tau, int fixed_exit,
                const int32_t *tf_exit, const int32_t *tf_ids, int32_t *next_ids, int32_t *exit_layer,
                double *dbg_smin, double *dbg_hidden_last, double *dbg_logits, int32_t *n_forced);

int ora_decode_step(ora_model *m, const int32_t *tokens, int B, double tau, const int32_t *forced,
                    const int32_t *tf_exit, const int32_t *tf_ids, int32_t *next_ids, int32_t *exit_layer,
                    double *dbg_hidden, double *dbg_s, double *dbg_logits, int32_t *n_forced);

/* One decoder layer (1-based `layer`) for rows 0..B-1 at their current
 * positions len[b] (len is not advanced): river[b] selects the river copy.
 * Writes the rows' K/V slot of that layer.  h_in, h_out: [B][d]. */
int ora_layer_forward(ora_model *m, int layer, int B, const int32_t *river, const double *h_in, double *h_out);

/* Final RMSNorm + original LM head + greedy pick for rows 0..B-1 (h: [B][d]). */
int ora_head(ora_model *m, int B, const double *h, double *logits, int32_t *ids);

int ora_kv_reset(ora_model *m, const int32_t *rows, int n_rows);
int ora_get_kv(const ora_model *m, uint16_t *dst, size_t bytes);
int ora_set_kv(ora_model *m, const uint16_t *src, size_t bytes, const int32_t *lens);
int ora_get_lens(const ora_model *m, int32_t *lens);
size_t ora_kv_bytes(const ora_model *m);

/* Primitives, exported for the oracle's own pins. */
double ora_act16_round(double x, int act_dtype);
uint16_t ora_act16_encode(double x, int act_dtype);
double ora_act16_decode(uint16_t bits, int act_dtype);
double ora_cosine(const double *a, const double *b, int n);
void ora_rmsnorm(const double *h, const uint16_t *gamma, int d, double eps, int act_dtype, double *out);
void ora_rope(double *v, int head_dim, int pos, double theta);
void ora_attention(const double *q, const uint16_t *K, const uint16_t *V, int T, int head_dim, int act_dtype,
                   double *out);
int ora_argmax(const double *v, int n);
int ora_rtn_group(const uint16_t *w, int n, int act_dtype, uint8_t *q, uint16_t *s, uint16_t *z);
double ora_silu(double g);

#ifdef __cplusplus
}
#endif
#endif
