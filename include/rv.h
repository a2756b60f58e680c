/*
 * rv.h - C ABI of the River-LLM token-level early-exit decode library
 * (librv.so, CUDA, sm_103a).
 *
 * The method: "River-LLM: Large Language Model Seamless Exit Based on KV
 * Share" (Shen, Zou).  Page summaries used as the definition:
 *   - paperlayer.ai summary, section 4 "KV-Shared Exit Layer": every exit
 *     layer is a plug-in copy of the backbone layer with the same index,
 *     4-bit weight-only quantized, addressing the backbone's KV cache.
 *   - same page, section 4 "Inference with Seamless Exit": exit layers run
 *     in series from a predefined entry layer; after an exit the remaining
 *     layers run as exit layers and the original LM head gives the logits;
 *     prefill uses one sequence-level exit, generation a token-level exit.
 *   - aitrends.kr article: s(l) = cos(h(l-1), h(l)) between the input and
 *     output of layer l; a token exits when s(l) is greater than tau; the
 *     exit layers are W4A16 copies of the backbone blocks.
 *
 * Conventions
 *   - Every call returns an int status (RV_OK or a negative RV_E* code) and
 *     records a message readable with rv_last_error() on the calling thread.
 *     No call throws, aborts the process or traps on the device.
 *   - The library owns all device memory behind the opaque rv_model handle:
 *     backbone weights, river copies, the KV cache, activations, scratch.
 *   - The caller owns every array passed in.  Pointers are HOST pointers
 *     unless the function name ends in _dev, in which case they are DEVICE
 *     pointers on the model's device and the call is asynchronous on the
 *     model's stream.
 *   - Layers are numbered 1..L.  An exit layer e in 1..L means layers 1..e
 *     ran in the backbone and e+1..L in the river; e = L means the token never
 *     left the backbone; e = 0 (forced mode only) means every layer ran in the
 *     river.
 *   - 16-bit types: act_dtype 0 = fp16, 1 = bf16.  Weights, the KV cache and
 *     every activation that enters a matrix product use it; the residual
 *     stream, accumulations, norms, softmax and s(l) are fp32.
 */
#ifndef RV_H
#define RV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RV_OK 0
#define RV_EINVAL (-1)     /* bad argument (range, pointer, shape) */
#define RV_ENOMEM (-2)     /* device or pinned host allocation failed; nothing leaked */
#define RV_ECUDA (-3)      /* a CUDA runtime call failed */
#define RV_ECAPACITY (-4)  /* a row's KV cache is full (len == max_seq); nothing changed */
#define RV_ESTATE (-5)     /* call out of order, e.g. tau-rule decode before rv_quantize_river */
#define RV_ETIMEOUT (-6)   /* a bounded device wait gave up (persistent engine, tensor-core GEMM) */

/* Projection ids of a decoder layer (for rv_export_river). */
#define RV_PROJ_Q 0
#define RV_PROJ_K 1
#define RV_PROJ_V 2
#define RV_PROJ_O 3
#define RV_PROJ_GATE 4
#define RV_PROJ_UP 5
#define RV_PROJ_DOWN 6

/* What rv_debug_dump copies out (all host layouts, row-major). */
#define RV_DUMP_HIDDEN 0  /* float [L+1][B][d]: residual stream after layers 0..L of the last step */
#define RV_DUMP_S 1       /* float [L][B]: s(l) of the last step, NaN where not evaluated */
#define RV_DUMP_LOGITS 2  /* float [B][V]: logits of the last step */
#define RV_DUMP_KV 3      /* uint16 [L][2][max_batch][Hkv][max_seq][hd]: the whole cache */
#define RV_DUMP_LENS 4    /* int32 [max_batch]: cached positions per row */

typedef struct rv_model rv_model; /* opaque */

/* Decoder shape (Llama-style: RMSNorm, GQA with rotate-half RoPE, SwiGLU).
 * max_batch and max_seq size the KV cache once, at load. */
typedef struct rv_config {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int tied_embed; /* 1: the LM head is the embedding matrix */
  int act_dtype;  /* 0 = fp16, 1 = bf16 */
  float rms_eps, rope_theta;
  int max_batch, max_seq;
} rv_config;

/* Last error message of the calling thread ("" if none). */
const char *rv_last_error(void);

/* Load a backbone.  weights holds 3 + 9*L host pointers to 16-bit arrays in
 * this order: embedding [V][d], final norm [d], LM head [V][d] (NULL when
 * tied_embed), then per layer: attention norm [d], W_q [H*hd][d],
 * W_k [Hkv*hd][d], W_v [Hkv*hd][d], W_o [d][H*hd], MLP norm [d],
 * W_gate [F][d], W_up [F][d], W_down [d][F].  The arrays are copied to the
 * device; the caller may free them afterwards.  stream is a cudaStream_t
 * (NULL: the library creates its own).  Allocates the one KV cache for
 * max_batch x max_seq positions, filled with the sentinel 0x7FFF (a NaN in
 * both 16-bit types).  Requires d_model, ffn and H*hd multiples of 8 and
 * head_dim in {64, 128}.  On failure nothing stays allocated. */
int rv_load_model(const rv_config *cfg, const void *const *weights, void *stream, rv_model **out);

/* Build the river: for every layer, copy the 7 projection matrices and
 * quantize them to int4 by round-to-nearest, asymmetric, per output row and
 * per group of group_size consecutive input columns, with an fp16 scale and
 * an fp16 (integer-valued) zero point; the exit layers share the backbone's
 * RMSNorm gains, RoPE and KV cache and allocate no KV memory.
 * entry_layer (1..L) is the first layer after which a token may exit by the
 * tau rule.  group_size: a multiple of 32.  Returns RV_EINVAL if a group's
 * scale overflows fp16.  May be called again (rebuilds the river). */
int rv_quantize_river(rv_model *m, int group_size, int entry_layer);

/* Copy one river matrix out in the canonical layout: q as uint32
 * [N][K/8] with element k of a row in bits 4*(k%8).. of word k/8, scales and
 * zeros as fp16 [N][ceil(K/group)].  layer in 1..L, proj an RV_PROJ_* id.
 * Any of the three pointers may be NULL. */
int rv_export_river(const rv_model *m, int layer, int proj, void *q_packed, void *scales, void *zeros);

/* Prefill rows 0..B-1 with tokens [B][T0] (row-major int32), starting each
 * row over at position 0, and return the first generated id per row.
 * Sequence-level exit: with fixed_exit_layer = -1 a row's exit layer is the
 * first l in [entry, L-1] at which s_t(l) > tau for every prompt token t
 * (else L); with fixed_exit_layer in 0..L it is that layer.  exit_layer[b]
 * receives it.  Cache slots at positions >= T0 keep their contents (use
 * rv_kv_reset first to restore the sentinel). */
int rv_prefill(rv_model *m, const int32_t *tokens, int B, int T0, float tau, int fixed_exit_layer,
               int32_t *next_ids, int32_t *exit_layer);

/* One decode step for rows 0..B-1: token b enters at position len_b, every
 * layer 1..L writes its K and V into slot (l, b, len_b) whichever path the
 * row takes, then len_b += 1.  Token-level exit: a row leaves the backbone
 * after the first layer l in [entry, L-1] with s(l) > tau and finishes in the
 * river.  forced_exit (NULL for the tau rule) gives each row's exit layer
 * 0..L instead.  next_ids[b] is the greedy id (lowest index on ties),
 * exit_layer[b] the row's exit layer.  RV_ECAPACITY if any row has
 * len_b == max_seq (nothing is changed). */
int rv_decode_step(rv_model *m, const int32_t *tokens, int B, float tau, const int32_t *forced_exit,
                   int32_t *next_ids, int32_t *exit_layer);

/* rv_decode_step with device pointers, asynchronous on the model's stream.
 * Arguments are checked on the host except token values and forced exit
 * values, which the device checks: an out-of-range value sets a device error
 * flag (reported by rv_sync_status) and is treated as token 0 / exit L. */
int rv_decode_step_dev(rv_model *m, const int32_t *d_tokens, int B, float tau, const int32_t *d_forced_exit,
                       int32_t *d_next_ids, int32_t *d_exit_layer);

/* Wait for the model's stream and report any device-side error flag. */
int rv_sync_status(rv_model *m);

/* Forget the cached positions of the given rows (NULL: all rows) and refill
 * their cache slots with the sentinel. */
int rv_kv_reset(rv_model *m, const int32_t *rows, int n_rows);

/* Keep per-step debug copies (hidden states per layer, s(l), logits) when
 * enable != 0.  Costs extra device writes; off by default. */
int rv_set_debug(rv_model *m, int enable);

/* Copy a debug buffer or the cache out (see RV_DUMP_*).  bytes must equal
 * the buffer's size for max_batch rows (hidden, s, logits use B = max_batch). */
int rv_debug_dump(rv_model *m, int what, void *dst, size_t bytes);

/* Options (rv_set_option).  RV_OPT_DECODE_ENGINE selects how a batch-1
 * decode step runs: RV_ENGINE_CHAIN (default) = a captured graph of one
 * kernel per GEMV / attention, chained by programmatic dependent launch;
 * RV_ENGINE_PERSISTENT = one cooperative launch of a persistent kernel with
 * every block resident and grid barriers between the phases of a layer.
 * Both compute the same step.  Returns RV_EINVAL for an unknown option or
 * value, RV_ESTATE if the persistent kernel cannot be made resident. */
#define RV_OPT_DECODE_ENGINE 0
#define RV_ENGINE_CHAIN 0
#define RV_ENGINE_PERSISTENT 1
/* RV_OPT_QUANTIZER selects how the next rv_quantize_river builds the river,
 * in the same packed format: RV_QUANT_RTN (default, integer fp16 zero) or
 * RV_QUANT_HQQ (the pages' quantizer, paperlayer.ai appendix A.1: the same
 * min/max scale, a float zero (stored as fp16) minimising the lp (p = 0.7)
 * norm of the error by half-quadratic splitting: beta 10, kappa 1.01, at
 * most 20 iterations, stopping when the mean absolute error stops falling;
 * deterministic, bit-identical to the oracle). */
#define RV_OPT_QUANTIZER 1
#define RV_QUANT_RTN 0
#define RV_QUANT_HQQ 1
/* RV_OPT_WAIT_LIMIT_US: the limit, in microseconds, of every bounded device
 * wait of the persistent kernel (grid barriers, weight-ring stages, route
 * hand-offs); 0 restores the default of two seconds.  A wait that runs out
 * sets an error flag; the kernel finishes its control flow without waiting,
 * lets its copies land, returns, and the step reports RV_ETIMEOUT without
 * advancing the cached positions.  A limit of a few microseconds makes
 * waits run out on purpose (a test of that path). */
#define RV_OPT_WAIT_LIMIT_US 2
int rv_set_option(rv_model *m, int option, int value);

/* Test hook: make a device allocation of this library fail.  after >= 0:
 * the next `after` allocations (cudaMalloc) succeed and the one after them
 * fails as if the device were out of memory (once); after < 0 turns the hook
 * off.  Process-wide; returns RV_OK.  The failing call returns RV_ENOMEM and
 * frees what it had allocated. */
int rv_debug_fail_alloc(int after);

/* Kernel timing for roofline reports: launch one batch-1 GEMV kernel of the
 * decode step `iters` times back to back on the model's stream (outside the
 * step graph) and return its mean device time per launch in *ms_per_launch
 * (CUDA events) and its algorithmic HBM bytes per launch in *bytes (weights,
 * the activation vector read, the outputs written).
 * kind: RV_TIME_GATEUP (RMSNorm + gate/up + SwiGLU of `layer`), RV_TIME_O
 * (O projection + residual), RV_TIME_LMHEAD (final norm + LM head + argmax),
 * RV_TIME_ATTN (the decode attention of row 0 in `layer` at its current
 * position; bytes = the K/V it reads).  river selects the int4 copy
 * (gate/up, O).  Leaves the KV cache and the cached positions untouched;
 * the step's activation buffers are overwritten. */
#define RV_TIME_GATEUP 0
#define RV_TIME_O 1
#define RV_TIME_LMHEAD 2
#define RV_TIME_ATTN 3
int rv_time_kernel(rv_model *m, int kind, int layer, int river, int iters, float *ms_per_launch, double *bytes);

/* Launch plan of the decode attention (host arithmetic only, no device
 * work; the pages have no counterpart: the plan is how this library splits
 * the attention over a single token's K/V, the "Memory Efficiency" long
 * contexts of paperlayer.ai section 5 included).  For `batch` rows with
 * n_kv_heads KV heads each, on a GPU of n_sm SMs whose largest launchable
 * cluster is max_cluster (a power of two <= 16), the longest context being
 * `context` positions: returns 0 for the cluster plan (the splits of a
 * (row, KV head) form one thread-block cluster and merge through
 * distributed shared memory; *splits = the cluster size: the largest power
 * of two <= max_cluster with splits x n_kv_heads x batch <= 2 n_sm) when
 * each warp of a split has at most 4 tiles of 32 positions, or when the
 * rows alone fill the GPU (n_sm / (n_kv_heads x batch) < 2); else 1 for the
 * global-merge plan (*splits = min(n_sm / (n_kv_heads x batch),
 * max_splits, 128) blocks per (row, KV head), merged through global
 * memory).  The decode step keys its captured graph by this plan.
 * RV_EINVAL for a null splits, batch, n_kv_heads, n_sm or max_splits below
 * 1, a negative context, or max_cluster not a power of two in 1..16. */
int rv_decode_attention_plan(int batch, int n_kv_heads, int n_sm, int max_cluster, int max_splits, int context,
                             int *splits);

/* Greedy LM head without allocation: final RMSNorm (gain d_final_norm, eps
 * rms_eps) of the fp32 vector d_h [d_model], the LM-head GEMV against
 * d_lm_head [vocab][d_model] (16-bit, act_dtype 0 = fp16, 1 = bf16) and the
 * argmax (lowest index on ties) into d_next_id[0]; d_logits [vocab] (fp32)
 * receives the logits when not NULL.  All pointers are device pointers; the
 * call is asynchronous on `stream` (a cudaStream_t, NULL = default stream).
 * The pages have no counterpart: this entry point exists for callers that
 * must not allocate device memory (a runtime that owns the whole memory
 * budget, or code that cannot afford the implicit synchronization of
 * cudaMalloc/cudaFree).  It runs the decode step's LM-head kernel with its
 * cross-block scratch (per-block results for at most 1024 blocks, ~8 KB) in
 * an array compiled into the library, which every GPU that loads the library
 * holds until the process exits; it calls no allocator.  The first call on a
 * device looks the array's address up (cudaGetSymbolAddress), so make that
 * first call before any stream capture.  All calls share the one array:
 * calls whose executions overlap on the GPU (other streams, other threads)
 * race and must be serialized by the caller.  Returns RV_EINVAL, before
 * any GPU work, for vocab not a positive multiple of 4, d_model not a
 * positive multiple of 8, d_model above the maximum of 16384, vocab x
 * d_model above 2^32 - 1, or d_lm_head, d_final_norm or d_h not 16-byte
 * aligned (the kernel reads them with 16-byte loads). */
int rv_greedy_head_noalloc(const void *d_lm_head, const void *d_final_norm, const float *d_h, int vocab,
                           int d_model, int act_dtype, float rms_eps, int32_t *d_next_id, float *d_logits,
                           void *stream);

/* Backbone offloading (paperlayer.ai section 4, "Backbone Offloading": with
 * most tokens leaving the backbone after a few layers, only the first
 * backbone layers need to stay on the device next to the river).  Frees the
 * 16-bit matrices of backbone layers keep_layers+1..L on the device (their
 * RMSNorm gains stay: the river shares them) and caps every exit at
 * keep_layers: a row still in the backbone after layer keep_layers
 * continues in the river, in decode and in prefill.  Needs the river
 * (RV_ESTATE otherwise); keep_layers in 1..L (RV_EINVAL), not above an
 * earlier call's value (RV_ESTATE: freed layers cannot come back without
 * reloading the model); keep_layers = L changes nothing.  Afterwards forced
 * and fixed exits above keep_layers are RV_EINVAL and rv_param_bytes(m, 0)
 * counts only the resident backbone. */
int rv_offload_backbone(rv_model *m, int keep_layers);

/* Sizes, for callers that allocate dump buffers.  rv_param_bytes: which = 0,
 * the 16-bit parameters resident on the device (embedding, LM head, norms,
 * backbone layers 1..keep_layers); which = 1, the river (codes and
 * (scale, zero) words). */
size_t rv_kv_bytes(const rv_model *m);
size_t rv_param_bytes(const rv_model *m, int which);

/* Free everything the model owns. */
void rv_free_model(rv_model *m);

#ifdef __cplusplus
}
#endif
#endif
