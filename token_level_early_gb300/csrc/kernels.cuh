// Kernel argument blocks and host launchers of librv (internal header).
#pragma once

#include "common.cuh"

namespace rv {

enum { PRO_NORM = 0, PRO_VEC = 1 };
enum { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_DOWN = 3, EPI_LOGITS = 4 };

// Arguments of the batch-1 GEMV kernels (see decode_b1.cu).
struct GemvArgs {
  Mat m;
  int units;   // unused: the launcher derives the work from the matrix and epilogue
  int s4, s16; // K splits per row quad for the int4 / 16-bit path (set by the launcher)
  // prologue
  const float *h;         // PRO_NORM: residual stream [K]
  const uint16_t *gamma;  // PRO_NORM: RMSNorm gain [K]
  float eps;
  const float *vec;       // PRO_VEC: activation [K]
  // epilogue
  const float *h_base;  // EPI_RESID / EPI_DOWN: residual added to
  float *h_out;         // EPI_RESID / EPI_DOWN
  const float *h_in;    // EPI_DOWN: layer input, for s(l)
  float *out_vec;       // EPI_QKV: q [H*hd]; EPI_SWIGLU: a [F]
  KVGeom kv;
  int layer;            // 0-based
  int L, H, Hkv, hd;
  const float2 *rope_cs;  // [max_seq][hd/2] (cos, sin)
  float *partials;
  unsigned *counter;
  float *dbg_h;       // EPI_DOWN: hidden dump for this layer (row 0) or NULL
  float *dbg_s;       // s dump of the decided layer or NULL
  // batch-1 chain, EPI_QKV / EPI_LOGITS: the exit decision of layer
  // decide_layer1 (1-based; 0 = none), from its input h_prev and output h
  const float *h_prev;
  int decide_layer1;
  float *dbg_logits;  // EPI_LOGITS: logits dump or NULL
  StepState st;
};

// Exit decision for row b after layer layer1 (1-based) from the three sums
// sum(h_in*h_out), sum(h_in^2), sum(h_out^2), for a row whose route before
// the decision is route_now.  s = dot / max(|h_in| |h_out|, 1e-8); strict
// s > tau (aitrends.kr); river rows do not evaluate s (NaN).
struct Decision {
  int route;
  bool exited;
  float s;
};
// The step's decision inputs for row b, read once: a kernel of the batch-1
// chain loads them before its dependency wait (they are written before the
// step's first layer kernel), so the decision itself waits on no memory.
struct DecideScalars {
  int mode, forced, entry, cap;
  float tau;
};
__device__ __forceinline__ DecideScalars load_decide_scalars(const StepState &st, int b) {
  DecideScalars p;
  p.mode = *st.mode;
  p.forced = st.forced[b];
  p.entry = *st.entry;
  p.cap = *st.cap;
  p.tau = *st.tau;
  return p;
}
__device__ __forceinline__ Decision decide(const DecideScalars &p, int route_now, int layer1, int L, float dot,
                                           float n1, float n2) {
  Decision d{route_now, false, __int_as_float(0x7fc00000)};
  if (route_now != 0) return d;
  const float den = fmaxf(sqrtf(n1) * sqrtf(n2), 1e-8f);
  d.s = dot / den;
  if (p.mode == 1) {
    int f = p.forced;
    if (f < 0 || f > L) f = L;
    d.exited = layer1 == f && layer1 < L;
  } else {
    d.exited = layer1 >= p.entry && layer1 <= L - 1 && d.s > p.tau;
  }
  // backbone offloading: the layers after the cap exist only in the river
  if (layer1 >= p.cap && layer1 < L) d.exited = true;
  if (d.exited) d.route = 1;
  return d;
}
__device__ __forceinline__ Decision decide(const StepState &st, int b, int route_now, int layer1, int L, float dot,
                                           float n1, float n2) {
  if (route_now != 0) return Decision{route_now, false, __int_as_float(0x7fc00000)};
  return decide(load_decide_scalars(st, b), route_now, layer1, L, dot, n1, n2);
}
// Record a decision in the step state (one thread).
__device__ __forceinline__ void commit_decision(const StepState &st, int b, int layer1, const Decision &d,
                                                float *dbg_s) {
  if (dbg_s) dbg_s[b] = d.s;
  if (d.exited) {
    st.route[b] = 1;
    st.exit_layer[b] = layer1;
  }
}
__device__ __forceinline__ void decide_row(const StepState &st, int b, int layer1, int L, float dot, float n1,
                                           float n2, float *dbg_s) {
  commit_decision(st, b, layer1, decide(st, b, st.route[b], layer1, L, dot, n1, n2), dbg_s);
}

cudaError_t launch_gemv_b1(int act, int pro, int epi, const GemvArgs &a, int grid, cudaStream_t s, int pdl = 0);

// ---------------------------------------------------------------- attention
struct AttnArgs {
  KVGeom kv;
  int layer, H, Hkv, hd, act;
  const float *q;      // [B][H*hd] (act16-rounded, after RoPE)
  float *o;            // [B][H*hd] output (act16-rounded)
  const int32_t *len;  // [B]: the token being decoded sits at position len[b]
  int splits;
  float *part;         // [B][Hkv][splits][H / Hkv][hd + 2] (global merge)
  unsigned *counter;   // [B][Hkv], zero between launches (global merge)
  int global_merge;    // 0: the splits form a cluster; 1: they merge through part / counter
};
constexpr int kAttnMaxSplits = 128;
cudaError_t launch_attn_decode(const AttnArgs &a, int B, cudaStream_t s, int pdl = 0);
// Largest cluster size (power of two <= 16) launch_attn_decode can use; 0 if none.
int attn_dec_max_cluster(int hd, int grp, int act);
// Launch plan for B rows whose longest context is pmax positions: returns
// AttnArgs::global_merge and sets *splits.
int attn_dec_plan(int B, int Hkv, int n_sm, int max_cluster, int max_splits, int pmax, int *splits);

// Causal attention for token rows of the general path: row m of the list
// attends to positions 0..pos(m) of its sequence.
struct AttnRowsArgs {
  KVGeom kv;
  int layer, H, Hkv, hd, act;
  const float *q;  // [M][H*hd]
  float *o;        // [M][H*hd]
  const int32_t *list;
  const int32_t *count;
  int tokens_per_row;    // T: token m belongs to sequence m / T, position base + m % T
  const int32_t *base;   // [B] position of the row's first token (decode: len; prefill: NULL = 0)
};
cudaError_t launch_attn_rows(const AttnRowsArgs &a, int max_rows, cudaStream_t s);

// ---------------------------------------------------------------- general path
cudaError_t launch_embed(const uint16_t *E, int d, int act, const int32_t *tokens, int M, int vocab, float *H,
                         float *dbg_h, int32_t *err, cudaStream_t s, int pdl = 0);
cudaError_t launch_step_init(const StepState &st, int B, int L, cudaStream_t s);
cudaError_t launch_route_lists(const int32_t *route, int B, int T, int32_t *lists, int list_stride,
                               int32_t *counts, cudaStream_t s);
cudaError_t launch_rmsnorm_rows(const float *H, const uint16_t *gamma, int d, float eps, int act, float *X,
                                const int32_t *list, const int32_t *count, int max_rows, cudaStream_t s);
// Tensor-core (tcgen05) rows GEMM for 16-bit matrices: gathers the listed
// rows of X into xb [max_rows][K] (16-bit) and writes Y[list[r]][n];
// K % 8 == 0.  Sets bit 16 of *err if a bounded wait gave up.
bool gemm_tc_available();
// The driver's cuTensorMapEncodeTiled (a PFN_cuTensorMapEncodeTiled_v12000), or NULL.
void *tensor_map_encoder();
cudaError_t launch_gemm_tc(const Mat &m, int act, const float *X, float *Y, const int32_t *list, const int32_t *count,
                           int max_rows, uint16_t *xb, int32_t *err, cudaStream_t s);
// The same for an int4 river matrix: split into 16-bit hi + lo (whi, wlo:
// [N][K] each, exact), then Y = X hi^T + X lo^T.
cudaError_t launch_gemm_tc_river(const Mat &m, int act, const float *X, float *Y, const int32_t *list,
                                 const int32_t *count, int max_rows, uint16_t *xb, uint16_t *whi, uint16_t *wlo,
                                 int32_t *err, cudaStream_t s);
// Batched decode rows on the tensor pipe (mma.sync): Y[list[i]] = W X[list[i]]
// for the river copy ((q - z) s, groups of 32, 64, 128 or 256; fewer than 256
// rows) or the 16-bit matrix (at most 64 rows).
bool rows_i4_supported(const Mat &m);
bool rows_b16_supported(const Mat &m);
cudaError_t launch_rows_i4(const Mat &m, int act, const float *X, float *Y, const int32_t *list,
                           const int32_t *count, int max_rows, int n_sm, cudaStream_t s);
// amax (optional, [rows]): each row's greedy pick as a key (largest value,
// lowest column on ties), for launch_pick_finish; zero before the launch.
cudaError_t launch_rows_b16(const Mat &m, int act, const float *X, float *Y, const int32_t *list,
                            const int32_t *count, int max_rows, int n_sm, cudaStream_t s,
                            unsigned long long *amax = nullptr);
cudaError_t launch_pick_finish(unsigned long long *amax, int B, StepState st, int bump_len, int set_len,
                               cudaStream_t s);
cudaError_t launch_gemm_rows(const Mat &m, int river, int act, const float *X, float *Y, const int32_t *list,
                             const int32_t *count, int max_rows, cudaStream_t s);
struct RopeRowsArgs {
  KVGeom kv;
  int layer, H, Hkv, hd, act;
  const float *Y;  // [M][(H+2Hkv)*hd]
  float *q;        // [M][H*hd]
  const float2 *rope_cs;
  const int32_t *list, *count;
  int tokens_per_row;
  const int32_t *base;
};
cudaError_t launch_rope_rows(const RopeRowsArgs &a, int max_rows, cudaStream_t s);
cudaError_t launch_resid_rows(float *H, const float *Y, int d, const int32_t *list, const int32_t *count,
                              int max_rows, cudaStream_t s);
cudaError_t launch_swiglu_rows(const float *Y, int F, int act, float *A, const int32_t *list,
                               const int32_t *count, int max_rows, cudaStream_t s);
cudaError_t launch_decide_rows(const StepState &st, const float *Hin, const float *H, int d, int B, int layer1,
                               int L, float *dbg_s, cudaStream_t s);
// smin: B unsigned words, all 0xFFFFFFFF before the first call (each call leaves them so).
cudaError_t launch_seq_decide(const StepState &st, const float *Hin, const float *H, int d, int B, int T,
                              int layer1, int L, int fixed_exit, unsigned *smin, float *dbg_smin, cudaStream_t s);
cudaError_t launch_argmax_rows(const float *logits, int V, int B, StepState st, int bump_len, int set_len,
                               cudaStream_t s);
cudaError_t launch_copy_rows(const float *src, int src_stride, float *dst, int dst_stride, int d, int B,
                             cudaStream_t s);

// ---------------------------------------------------------------- river construction
cudaError_t launch_hqq_quantize(const uint16_t *W, int N, int K, int act, int g, int Kp, uint32_t *q, __half2 *sz,
                                int32_t *err, cudaStream_t s);
cudaError_t launch_rtn_quantize(const uint16_t *W, int N, int K, int act, int g, int Kp, uint32_t *q, __half2 *sz,
                                int32_t *err, cudaStream_t s);
cudaError_t launch_rope_table(float2 *cs, int T, int hd, double theta, cudaStream_t s);
cudaError_t launch_fill_u16(uint16_t *p, size_t n, uint16_t v, cudaStream_t s);

// Sets the calling thread's message returned by rv_last_error().
void set_error_message(const char *msg);

}  // namespace rv
