// Host runtime of librv: the C ABI declared in include/rv.h.
//
// Owns the device copy of the backbone, the river copies, the one shared KV
// cache and all activations; runs prefill (sequence-level exit) and decode
// steps (token-level exit) on the model's stream.  Decode steps are captured
// once per batch size in a CUDA graph: every per-step value (tokens, tau,
// forced exits, positions, routes) lives in device memory, so a step is one
// host-to-device copy, one graph launch and one device-to-host copy.  The
// batch-1 chain is launched with programmatic dependent launch, so each
// kernel's launch and weight prefetch overlap its predecessor's tail.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <map>
#include <string>
#include <algorithm>
#include <vector>

#include "../../include/rv.h"
#include "common.cuh"
#include "gemv_core.cuh"
#include "kernels.cuh"
#include "stream.cuh"

using namespace rv;

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define RV_CK(call)                                                                               \
  do {                                                                                            \
    cudaError_t e_ = (call);                                                                      \
    if (e_ != cudaSuccess) {                                                                      \
      return fail(e_ == cudaErrorMemoryAllocation ? RV_ENOMEM : RV_ECUDA, "%s failed: %s", #call, \
                  cudaGetErrorString(e_));                                                        \
    }                                                                                             \
  } while (0)

constexpr uint16_t KV_SENTINEL = 0x7FFF;
enum { MAT_QKV = 0, MAT_O = 1, MAT_GU = 2, MAT_D = 3, N_MAT = 4 };

struct RiverDev {
  uint32_t *q = nullptr;
  __half2 *sz = nullptr;
  int Kp = 0, G = 0, Gs = 0;  // Gs: row stride of sz (G padded to a multiple of 4)
};

struct LayerDev {
  uint16_t *attn_norm = nullptr, *mlp_norm = nullptr;
  uint16_t *w[N_MAT] = {nullptr, nullptr, nullptr, nullptr};
  RiverDev r[N_MAT];
};

inline int round32(int k) { return (k + 31) & ~31; }

}  // namespace

struct rv_model {
  rv_config c{};
  int act = 1, L = 0, d = 0, H = 0, Hkv = 0, hd = 0, F = 0, V = 0, Bmax = 0, Tmax = 0;
  int qd = 0, kvd = 0, qkv_n = 0;
  int dev = 0, n_sm = 0;
  cudaStream_t stream = nullptr;
  bool own_stream = false;

  std::vector<void *> allocs;  // every device allocation (freed at rv_free_model)
  void *pinned = nullptr;

  uint16_t *embed = nullptr, *final_norm = nullptr, *lm_head = nullptr;
  std::vector<LayerDev> layers;
  int group = 0, entry = 1;
  int cap = 0;  // last backbone layer on the device (L = all; set by rv_offload_backbone)
  int quantizer = RV_QUANT_RTN;  // river quantizer of the next rv_quantize_river
  bool has_river = false;
  std::vector<void *> river_allocs;

  KVGeom kv{};
  size_t kv_bytes = 0;
  float2 *rope_cs = nullptr;

  // device state block (int32 words), see state_layout()
  int32_t *d_state = nullptr;
  int in_words = 0, out_words = 0;
  StepState st{};
  int32_t *d_counts = nullptr, *d_nrows = nullptr, *d_ident = nullptr;
  std::vector<int32_t> h_len;

  // batch-1 activations
  float *hbuf[2] = {nullptr, nullptr}, *hmid = nullptr, *qbuf = nullptr, *obuf = nullptr, *abuf = nullptr;
  float *partials = nullptr;
  unsigned *seq_min = nullptr;  // [Bmax] prefill sequence-exit minima (order-preserving encoding)
  unsigned *counters = nullptr;
  int attn_splits_max = 1, attn_cluster = 1;
  float *attn_part = nullptr;
  unsigned *attn_counter = nullptr;
  unsigned long long *head_keys = nullptr;  // [Bmax] greedy-pick keys of the batched LM head (zero between steps)

  // general-path workspace (grown on demand)
  long ws_rows = 0;
  std::vector<void *> ws_allocs;
  float *gH = nullptr, *gHin = nullptr, *gX = nullptr, *gY = nullptr, *gY2 = nullptr, *gQ = nullptr, *gO = nullptr;
  int32_t *gLists = nullptr, *gTokens = nullptr;
  float *gHf = nullptr, *gXf = nullptr, *gLogits = nullptr;
  uint16_t *gXb = nullptr;  // 16-bit staging of GEMM rows for the tensor-core path
  uint16_t *gWhi = nullptr, *gWlo = nullptr;  // a river matrix split into 16-bit hi + lo (tensor-core rows path)
  bool tc_gemm = false;     // tcgen05 rows GEMM usable on this device

  // debug copies
  bool debug = false;
  float *dbg_h = nullptr, *dbg_s = nullptr, *dbg_logits = nullptr;

  // graphs
  std::map<int, cudaGraphExec_t> graphs;

  // persistent batch-1 step (stream.cu)
  int engine = RV_ENGINE_CHAIN;
  int wait_us = 0;  // RV_OPT_WAIT_LIMIT_US (0: the kernel's default)
  bool stream_ready = false;
  int stream_grid = 0;
  LayerDesc *d_layers = nullptr;
  CUtensorMap *d_tmaps = nullptr;  // [12 L + 1]: per layer and matrix the 16-bit, code and scale maps; LM head
  unsigned *bar = nullptr;
  StreamArgs sargs{};
};

namespace {

// Test hook (rv_debug_fail_alloc): allocations left before one fails; < 0 off.
std::atomic<long> g_fail_after{-1};

int dalloc(rv_model *m, std::vector<void *> &list, void **p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) bytes = 16;
  if (g_fail_after.load() >= 0 && g_fail_after.fetch_sub(1) == 0)
    return fail(RV_ENOMEM, "cudaMalloc(%zu bytes) failed: injected by rv_debug_fail_alloc", bytes);
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return fail(RV_ENOMEM, "cudaMalloc(%zu bytes) failed: %s", bytes, cudaGetErrorString(e));
  }
  list.push_back(*p);
  return RV_OK;
}

#define RV_ALLOC(list, ptr, bytes)                                              \
  do {                                                                          \
    int rc_ = dalloc(m, list, reinterpret_cast<void **>(&(ptr)), (bytes));      \
    if (rc_ != RV_OK) return rc_;                                               \
  } while (0)

// Weight matrices get kWeightPad zeroed bytes past their end: the persistent
// engine's tensor copies move whole boxes, and a row's last box may run past
// the row (and, for the last row, past the matrix) when K is not a multiple
// of the box; the extra values only ever meet zero activations.
constexpr size_t kWeightPad = 256;
#define RV_ALLOC_W(list, ptr, bytes)                                                               \
  do {                                                                                             \
    const size_t b_ = (bytes);                                                                     \
    RV_ALLOC(list, ptr, b_ + kWeightPad);                                                          \
    RV_CK(cudaMemsetAsync(reinterpret_cast<char *>(ptr) + b_, 0, kWeightPad, m->stream));           \
  } while (0)

void free_list(std::vector<void *> &list) {
  for (void *p : list) cudaFree(p);
  list.clear();
}

void drop_graphs(rv_model *m) {
  for (auto &kv : m->graphs) cudaGraphExecDestroy(kv.second);
  m->graphs.clear();
}

// int32 state block: [in: tokens B | forced B | mode | tau | entry | nrows]
//                    [out: next B | exit B | err | pad] [route B | len B | counts 2 | cap | pad]
void state_layout(rv_model *m) {
  const int B = m->Bmax;
  m->in_words = 2 * B + 4;
  m->out_words = 2 * B + 2;
  int32_t *s = m->d_state;
  StepState &st = m->st;
  st.tokens = s;
  st.forced = s + B;
  st.mode = s + 2 * B;
  st.tau = reinterpret_cast<const float *>(s + 2 * B + 1);
  st.entry = s + 2 * B + 2;
  m->d_nrows = s + 2 * B + 3;
  int32_t *o = s + m->in_words;
  st.next_ids = o;
  st.exit_layer = o + B;
  st.err = o + 2 * B;
  int32_t *r = o + m->out_words;
  st.route = r;
  st.len = r + B;
  m->d_counts = r + 2 * B;
  st.cap = r + 2 * B + 2;
}

size_t state_words(int B) { return (size_t)(2 * B + 4) + (2 * B + 2) + (2 * B + 4); }

int32_t *pin_in(rv_model *m) { return static_cast<int32_t *>(m->pinned); }
int32_t *pin_out(rv_model *m) { return static_cast<int32_t *>(m->pinned) + m->in_words; }

Mat make_mat(const rv_model *m, const LayerDev &ly, int which) {
  Mat mt{};
  mt.w = ly.w[which];
  switch (which) {
    case MAT_QKV: mt.N = m->qkv_n; mt.K = m->d; break;
    case MAT_O: mt.N = m->d; mt.K = m->qd; break;
    case MAT_GU: mt.N = 2 * m->F; mt.K = m->d; break;
    default: mt.N = m->d; mt.K = m->F; break;
  }
  if (m->has_river) {
    mt.r.q = ly.r[which].q;
    mt.r.sz = ly.r[which].sz;
    mt.r.Kp = ly.r[which].Kp;
    mt.r.G = ly.r[which].G;
    mt.r.Gs = ly.r[which].Gs;
    mt.r.g = m->group;
  }
  return mt;
}

// Upper bound on a batch-1 GEMV grid: the reduction scratch holds 4 blocks
// per SM (the launcher also caps the grid at one resident wave).
int gemv_grid(const rv_model *m, int) { return 4 * m->n_sm; }

// Decode-attention plan for rows 0..B-1 at their current positions (the
// captured step of batch B is keyed by it).
int attn_plan(const rv_model *m, int B, AttnArgs *at) {
  int pmax = 0;
  for (int b = 0; b < B && b < (int)m->h_len.size(); ++b) pmax = m->h_len[b] > pmax ? m->h_len[b] : pmax;
  int splits = 1;
  const int gm = attn_dec_plan(B, m->Hkv, m->n_sm, m->attn_cluster, m->attn_splits_max, pmax, &splits);
  if (at) {
    at->global_merge = gm;
    at->splits = splits;
  }
  return gm;
}

// -------------------------------------------------------------- batch-1 step

int enqueue_step_b1(rv_model *m, cudaStream_t s) {
  const int L = m->L, B = m->Bmax;
  RV_CK(cudaMemsetAsync(m->st.err, 0, sizeof(int32_t), s));
  RV_CK(launch_step_init(m->st, 1, L, s));
  RV_CK(launch_embed(m->embed, m->d, m->act, m->st.tokens, 1, m->V, m->hbuf[0], m->debug ? m->dbg_h : nullptr,
                     m->st.err, s, 1));
  for (int l = 0; l < L; ++l) {
    const LayerDev &ly = m->layers[l];
    float *hin = m->hbuf[l & 1], *hout = m->hbuf[(l + 1) & 1];
    GemvArgs a{};
    a.st = m->st;
    a.kv = m->kv;
    a.layer = l;
    a.L = L; a.H = m->H; a.Hkv = m->Hkv; a.hd = m->hd;
    a.eps = m->c.rms_eps;
    a.rope_cs = m->rope_cs;
    a.partials = m->partials;

    // exit decision of layer l (1-based) -> RMSNorm -> QKV -> RoPE -> K/V append
    a.m = make_mat(m, ly, MAT_QKV);
    a.units = m->qkv_n / 2;
    a.h = hin; a.gamma = ly.attn_norm; a.out_vec = m->qbuf;
    if (l > 0) {
      a.h_prev = m->hbuf[(l - 1) & 1];
      a.decide_layer1 = l;
      a.dbg_s = m->debug ? m->dbg_s + (size_t)(l - 1) * B : nullptr;
    }
    RV_CK(launch_gemv_b1(m->act, PRO_NORM, EPI_QKV, a, gemv_grid(m, a.units), s, 1));
    a.h_prev = nullptr;
    a.decide_layer1 = 0;
    a.dbg_s = nullptr;

    AttnArgs at{};
    at.kv = m->kv; at.layer = l; at.H = m->H; at.Hkv = m->Hkv; at.hd = m->hd; at.act = m->act;
    at.q = m->qbuf; at.o = m->obuf; at.len = m->st.len;
    at.part = m->attn_part; at.counter = m->attn_counter;
    attn_plan(m, 1, &at);
    RV_CK(launch_attn_decode(at, 1, s, 1));

    // O projection + residual
    a.m = make_mat(m, ly, MAT_O);
    a.units = m->d;
    a.vec = m->obuf; a.h_base = hin; a.h_out = m->hmid;
    RV_CK(launch_gemv_b1(m->act, PRO_VEC, EPI_RESID, a, gemv_grid(m, a.units), s, 1));

    // MLP in: RMSNorm -> gate/up -> SwiGLU
    a.m = make_mat(m, ly, MAT_GU);
    a.units = m->F;
    a.h = m->hmid; a.gamma = ly.mlp_norm; a.out_vec = m->abuf;
    RV_CK(launch_gemv_b1(m->act, PRO_NORM, EPI_SWIGLU, a, gemv_grid(m, a.units), s, 1));

    // down projection + residual (its exit decision is made by the next kernel)
    a.m = make_mat(m, ly, MAT_D);
    a.units = m->d;
    a.vec = m->abuf; a.h_base = m->hmid; a.h_in = hin; a.h_out = hout;
    a.dbg_h = m->debug ? m->dbg_h + (size_t)(l + 1) * B * m->d : nullptr;
    RV_CK(launch_gemv_b1(m->act, PRO_VEC, EPI_DOWN, a, gemv_grid(m, a.units), s, 1));
  }
  // (s(L) for the debug dump) final RMSNorm + LM head + greedy argmax
  GemvArgs a{};
  a.st = m->st;
  a.L = L;
  a.m.w = m->lm_head; a.m.N = m->V; a.m.K = m->d;
  a.units = m->V;
  a.h = m->hbuf[L & 1]; a.gamma = m->final_norm; a.eps = m->c.rms_eps;
  if (m->debug) {  // no exit after the last layer: only the dump needs s(L)
    a.h_prev = m->hbuf[(L - 1) & 1];
    a.decide_layer1 = L;
    a.dbg_s = m->dbg_s + (size_t)(L - 1) * B;
  }
  a.partials = m->partials;
  a.counter = m->counters + L;
  a.dbg_logits = m->debug ? m->dbg_logits : nullptr;
  RV_CK(launch_gemv_b1(m->act, PRO_NORM, EPI_LOGITS, a, gemv_grid(m, a.units), s, 1));
  return RV_OK;
}

// -------------------------------------------------------------- general path

// Rows GEMM: the tcgen05 kernel for 16-bit matrices where the device has it;
// river copies: fewer than 256 rows on the tensor pipe straight from the int4
// codes, more through the matrix's 16-bit hi + lo copies on tcgen05.
// River rows take the tcgen05 path (the matrix split into exact 16-bit hi +
// lo, two GEMMs) from this many rows up; below it the int4 kernel, which
// reads a quarter of the bytes of either 16-bit copy, is the faster one.
constexpr long kRiverTcRows = 256;
constexpr int kRowsMmaMax16 = 64;

static cudaError_t gemm_rows(rv_model *m, const Mat &mt, int river, const float *X, float *Y, const int32_t *list,
                             const int32_t *count, int max_rows, cudaStream_t s) {
  // up to 64 rows of a 16-bit matrix: the mma.sync rows kernel splits K over
  // clusters, where the tcgen05 GEMM would run one 128-row tile per 128
  // columns of N and leave most SMs idle
  if (!river && max_rows <= kRowsMmaMax16 && rows_b16_supported(mt))
    return launch_rows_b16(mt, m->act, X, Y, list, count, max_rows, m->n_sm, s);
  if (m->tc_gemm && mt.K % 8 == 0 && max_rows <= m->ws_rows) {
    if (!river) return launch_gemm_tc(mt, m->act, X, Y, list, count, max_rows, m->gXb, m->st.err, s);
    if (max_rows >= kRiverTcRows && m->gWhi)
      return launch_gemm_tc_river(mt, m->act, X, Y, list, count, max_rows, m->gXb, m->gWhi, m->gWlo, m->st.err, s);
  }
  if (river && max_rows < kRiverTcRows && rows_i4_supported(mt))
    return launch_rows_i4(mt, m->act, X, Y, list, count, max_rows, m->n_sm, s);
  return launch_gemm_rows(mt, river, m->act, X, Y, list, count, max_rows, s);
}

int ensure_ws(rv_model *m, long rows) {
  if (rows <= m->ws_rows) return RV_OK;
  // captured graphs hold workspace pointers: drop them before reallocating
  RV_CK(cudaStreamSynchronize(m->stream));
  drop_graphs(m);
  free_list(m->ws_allocs);
  m->ws_rows = 0;
  const size_t d = m->d, F = m->F, qd = m->qd;
  size_t xw = d > F ? d : F;
  if (qd > xw) xw = qd;
  size_t yw = (size_t)m->qkv_n;
  if (2 * F > yw) yw = 2 * F;
  if (d > yw) yw = d;
  auto &L = m->ws_allocs;
  RV_ALLOC(L, m->gH, sizeof(float) * rows * d);
  RV_ALLOC(L, m->gHin, sizeof(float) * rows * d);
  RV_ALLOC(L, m->gX, sizeof(float) * rows * xw);
  RV_ALLOC(L, m->gXb, sizeof(uint16_t) * rows * (xw > (size_t)m->d ? xw : (size_t)m->d));
  m->gWhi = m->gWlo = nullptr;
  if (m->tc_gemm && rows >= kRiverTcRows) {
    size_t wmax = (size_t)m->qkv_n * d;
    if ((size_t)d * qd > wmax) wmax = (size_t)d * qd;
    if (2 * F * d > wmax) wmax = 2 * F * d;
    if ((size_t)d * F > wmax) wmax = (size_t)d * F;
    RV_ALLOC(L, m->gWhi, sizeof(uint16_t) * wmax);
    RV_ALLOC(L, m->gWlo, sizeof(uint16_t) * wmax);
  }
  RV_ALLOC(L, m->gY, sizeof(float) * rows * yw);
  RV_ALLOC(L, m->gY2, sizeof(float) * rows * d);
  RV_ALLOC(L, m->gQ, sizeof(float) * rows * qd);
  RV_ALLOC(L, m->gO, sizeof(float) * rows * qd);
  RV_ALLOC(L, m->gLists, sizeof(int32_t) * rows * 2);
  RV_ALLOC(L, m->gTokens, sizeof(int32_t) * rows);
  m->ws_rows = rows;
  return RV_OK;
}

// One decoder layer over all rows of the general path; rows are split by
// route into two lists and each projection runs once per path.
int enqueue_layer_rows(rv_model *m, int l, int B, int T, const int32_t *base, cudaStream_t s) {
  const LayerDev &ly = m->layers[l];
  const long M = (long)B * T;
  const int32_t *lists[2] = {m->gLists, m->gLists + M};
  const int32_t *cnt[2] = {m->d_counts, m->d_counts + 1};
  const int act = m->act, d = m->d;
  const int npath = m->has_river ? 2 : 1;
  RV_CK(launch_copy_rows(m->gH, d, m->gHin, d, d, (int)M, s));  // a kernel, so the layer's launches chain by PDL
  RV_CK(launch_route_lists(m->st.route, B, T, m->gLists, (int)M, m->d_counts, s));
  // attention sub-block
  RV_CK(launch_rmsnorm_rows(m->gH, ly.attn_norm, d, m->c.rms_eps, act, m->gX, nullptr, m->d_nrows, (int)M, s));
  for (int p = 0; p < npath; ++p)
    if (p == 1 || ly.w[MAT_QKV]) RV_CK(gemm_rows(m, make_mat(m, ly, MAT_QKV), p, m->gX, m->gY, lists[p], cnt[p], (int)M, s));
  RopeRowsArgs ra{};
  ra.kv = m->kv; ra.layer = l; ra.H = m->H; ra.Hkv = m->Hkv; ra.hd = m->hd; ra.act = act;
  ra.Y = m->gY; ra.q = m->gQ; ra.rope_cs = m->rope_cs; ra.list = nullptr; ra.count = m->d_nrows;
  ra.tokens_per_row = T; ra.base = base;
  RV_CK(launch_rope_rows(ra, (int)M, s));
  if (T == 1) {
    AttnArgs at{};
    at.kv = m->kv; at.layer = l; at.H = m->H; at.Hkv = m->Hkv; at.hd = m->hd; at.act = act;
    at.q = m->gQ; at.o = m->gO; at.len = base;
    at.part = m->attn_part; at.counter = m->attn_counter;
    attn_plan(m, B, &at);
    RV_CK(launch_attn_decode(at, B, s, 1));
  } else {
    AttnRowsArgs ar{};
    ar.kv = m->kv; ar.layer = l; ar.H = m->H; ar.Hkv = m->Hkv; ar.hd = m->hd; ar.act = act;
    ar.q = m->gQ; ar.o = m->gO; ar.tokens_per_row = T; ar.base = base;
    RV_CK(launch_attn_rows(ar, (int)M, s));
  }
  for (int p = 0; p < npath; ++p)
    if (p == 1 || ly.w[MAT_O]) RV_CK(gemm_rows(m, make_mat(m, ly, MAT_O), p, m->gO, m->gY2, lists[p], cnt[p], (int)M, s));
  RV_CK(launch_resid_rows(m->gH, m->gY2, d, nullptr, m->d_nrows, (int)M, s));
  // MLP sub-block
  RV_CK(launch_rmsnorm_rows(m->gH, ly.mlp_norm, d, m->c.rms_eps, act, m->gX, nullptr, m->d_nrows, (int)M, s));
  for (int p = 0; p < npath; ++p)
    if (p == 1 || ly.w[MAT_GU]) RV_CK(gemm_rows(m, make_mat(m, ly, MAT_GU), p, m->gX, m->gY, lists[p], cnt[p], (int)M, s));
  RV_CK(launch_swiglu_rows(m->gY, m->F, act, m->gX, nullptr, m->d_nrows, (int)M, s));
  for (int p = 0; p < npath; ++p)
    if (p == 1 || ly.w[MAT_D]) RV_CK(gemm_rows(m, make_mat(m, ly, MAT_D), p, m->gX, m->gY2, lists[p], cnt[p], (int)M, s));
  RV_CK(launch_resid_rows(m->gH, m->gY2, d, nullptr, m->d_nrows, (int)M, s));
  return RV_OK;
}

// Final norm + LM head + argmax over rows Hf [B][d].
int enqueue_head_rows(rv_model *m, int B, int bump_len, int set_len, cudaStream_t s) {
  RV_CK(launch_rmsnorm_rows(m->gHf, m->final_norm, m->d, m->c.rms_eps, m->act, m->gXf, nullptr, m->d_nrows, B, s));
  Mat lm{};
  lm.w = m->lm_head; lm.N = m->V; lm.K = m->d;
  if (B <= kRowsMmaMax16 && rows_b16_supported(lm)) {
    // the greedy pick rides on the LM-head kernel (one key per row)
    RV_CK(launch_rows_b16(lm, m->act, m->gXf, m->gLogits, nullptr, m->d_nrows, B, m->n_sm, s, m->head_keys));
    RV_CK(launch_pick_finish(m->head_keys, B, m->st, bump_len, set_len, s));
  } else {
    RV_CK(gemm_rows(m, lm, 0, m->gXf, m->gLogits, nullptr, m->d_nrows, B, s));
    RV_CK(launch_argmax_rows(m->gLogits, m->V, B, m->st, bump_len, set_len, s));
  }
  if (m->debug)
    RV_CK(cudaMemcpyAsync(m->dbg_logits, m->gLogits, sizeof(float) * B * m->V, cudaMemcpyDeviceToDevice, s));
  return RV_OK;
}

int enqueue_step_rows(rv_model *m, int B, cudaStream_t s) {
  const int L = m->L;
  RV_CK(cudaMemsetAsync(m->st.err, 0, sizeof(int32_t), s));
  RV_CK(launch_step_init(m->st, B, L, s));
  RV_CK(launch_embed(m->embed, m->d, m->act, m->st.tokens, B, m->V, m->gH, m->debug ? m->dbg_h : nullptr, m->st.err,
                     s));
  for (int l = 0; l < L; ++l) {
    int rc = enqueue_layer_rows(m, l, B, 1, m->st.len, s);
    if (rc) return rc;
    RV_CK(launch_decide_rows(m->st, m->gHin, m->gH, m->d, B, l + 1, L,
                             m->debug ? m->dbg_s + (size_t)l * m->Bmax : nullptr, s));
    if (m->debug)
      RV_CK(cudaMemcpyAsync(m->dbg_h + (size_t)(l + 1) * m->Bmax * m->d, m->gH, sizeof(float) * B * m->d,
                            cudaMemcpyDeviceToDevice, s));
  }
  RV_CK(cudaMemcpyAsync(m->gHf, m->gH, sizeof(float) * B * m->d, cudaMemcpyDeviceToDevice, s));
  return enqueue_head_rows(m, B, 1, -1, s);
}

// (Re)build the persistent kernel's argument block: layer descriptors (with
// the river copies when built), activations, scratch, debug pointers, and the
// size of its activation region (the largest staged vector of any phase, or
// the attention's K/V tiles).
int build_stream(rv_model *m) {
  m->stream_ready = false;
  const int grp = m->H / m->Hkv;
  if (!stream_supported(m->hd, grp, m->act, m->has_river ? m->group : 0)) return RV_OK;
  std::vector<LayerDesc> h(m->L);
  std::vector<CUtensorMap> tm(12 * (size_t)m->L + 1);
  int xb = 0;
  for (int l = 0; l < m->L; ++l) {
    for (int i = 0; i < N_MAT; ++i) {
      const Mat mt = make_mat(m, m->layers[l], i);
      h[l].m[i] = mt;
      CUtensorMap *t = &tm[(size_t)12 * l + 3 * i];
      const CUtensorMap *dt = m->d_tmaps + (size_t)12 * l + 3 * i;
      h[l].tw[i] = h[l].tq[i] = h[l].ts[i] = nullptr;
      if (mt.w) {
        if (!stream_map_w16(&t[0], mt.w, mt.N, mt.K, m->act)) return RV_OK;  // no tensor maps: the chain serves
        h[l].tw[i] = dt;
        xb = std::max(xb, x_geom(mt, 0).bytes);
      }
      if (m->has_river) {
        if (!stream_map_q(&t[1], mt.r.q, mt.N, mt.r.Kp) || !stream_map_sz(&t[2], mt.r.sz, mt.N, mt.r.Gs, mt.r.g))
          return RV_OK;
        h[l].tq[i] = dt + 1;
        h[l].ts[i] = dt + 2;
        xb = std::max(xb, x_geom(mt, 1).bytes);
      }
    }
    h[l].attn_norm = m->layers[l].attn_norm;
    h[l].mlp_norm = m->layers[l].mlp_norm;
  }
  Mat lm{};
  lm.w = m->lm_head; lm.N = m->V; lm.K = m->d;
  if (!stream_map_w16(&tm[(size_t)12 * m->L], lm.w, lm.N, lm.K, m->act)) return RV_OK;
  xb = std::max(xb, x_geom(lm, 0).bytes);
  // attention: two K/V tiles of 32 positions (K rows padded by 16 bytes) + q of a group as 16-bit
  xb = std::max(xb, 2 * sk::ATILE * (m->hd * 2 + 16 + m->hd * 2) + grp * m->hd * 2);
  xb = (xb + 127) & ~127;
  RV_CK(cudaMemcpy(m->d_layers, h.data(), sizeof(LayerDesc) * m->L, cudaMemcpyHostToDevice));
  RV_CK(cudaMemcpy(m->d_tmaps, tm.data(), sizeof(CUtensorMap) * tm.size(), cudaMemcpyHostToDevice));
  StreamArgs &A = m->sargs;
  A = StreamArgs{};
  A.layers = m->d_layers;
  A.embed = m->embed; A.final_norm = m->final_norm; A.lm_head = m->lm_head;
  A.t_head = m->d_tmaps + (size_t)12 * m->L;
  A.L = m->L; A.d = m->d; A.H = m->H; A.Hkv = m->Hkv; A.hd = m->hd; A.F = m->F; A.V = m->V; A.act = m->act;
  A.Bmax = m->Bmax;
  A.eps = m->c.rms_eps;
  A.kv = m->kv;
  A.rope_cs = m->rope_cs;
  A.st = m->st;
  A.h[0] = m->hbuf[0]; A.h[1] = m->hbuf[1]; A.hmid = m->hmid; A.q = m->qbuf; A.o = m->obuf; A.a = m->abuf;
  A.attn_part = m->attn_part;
  A.attn_counter = m->attn_counter;
  int sp = m->n_sm / m->Hkv;
  if (sp > m->attn_splits_max) sp = m->attn_splits_max;
  A.att_splits = sp < 1 ? 1 : sp;
  A.partials = m->partials;
  A.bar = m->bar;
  A.dbg_h = m->debug ? m->dbg_h : nullptr;
  A.dbg_s = m->debug ? m->dbg_s : nullptr;
  A.dbg_logits = m->debug ? m->dbg_logits : nullptr;
  A.xbytes = xb;
  A.wait_ns = (unsigned long long)m->wait_us * 1000ull;
  A.nstages = 0;  // set by stream_prepare from the device's shared memory
  int grid = 0;
  cudaError_t e = stream_prepare(A, m->n_sm, &grid);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RV_OK;  // not resident on this device: the kernel chain serves
  }
  m->stream_grid = grid;
  m->stream_ready = true;
  return RV_OK;
}

// Launch one decode step (persistent kernel for batch 1 when selected, else
// the captured graph for batch B, captured once per batch size).
int launch_step(rv_model *m, int B) {
  if (B == 1 && m->engine == RV_ENGINE_PERSISTENT && m->stream_ready) {
    RV_CK(cudaMemsetAsync(m->st.err, 0, sizeof(int32_t), m->stream));
    RV_CK(cudaMemsetAsync(m->bar, 0, sizeof(unsigned) * 2, m->stream));  // fresh barrier every step
    RV_CK(stream_launch(m->sargs, m->stream_grid, m->stream));
    return RV_OK;
  }
  const int key = 2 * B + attn_plan(m, B, nullptr);
  auto it = m->graphs.find(key);
  if (it == m->graphs.end()) {
    if (B > 1) {
      int rc = ensure_ws(m, m->Bmax);
      if (rc) return rc;
    }
    cudaGraph_t g = nullptr;
    RV_CK(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal));
    int rc = B == 1 ? enqueue_step_b1(m, m->stream) : enqueue_step_rows(m, B, m->stream);
    cudaError_t ec = cudaStreamEndCapture(m->stream, &g);
    if (rc != RV_OK) {
      if (g) cudaGraphDestroy(g);
      return rc;
    }
    if (ec != cudaSuccess) return fail(RV_ECUDA, "graph capture failed: %s", cudaGetErrorString(ec));
    cudaGraphExec_t ge = nullptr;
    cudaError_t ei = cudaGraphInstantiate(&ge, g, 0);
    cudaGraphDestroy(g);
    if (ei != cudaSuccess) return fail(RV_ECUDA, "graph instantiate failed: %s", cudaGetErrorString(ei));
    it = m->graphs.emplace(key, ge).first;
  }
  RV_CK(cudaGraphLaunch(it->second, m->stream));
  return RV_OK;
}

int check_common(rv_model *m) {
  if (!m) return fail(RV_EINVAL, "null model");
  return RV_OK;
}

int set_scalars(rv_model *m, int mode, float tau, int nrows) {
  int32_t *in = pin_in(m);
  const int B = m->Bmax;
  in[2 * B] = mode;
  memcpy(&in[2 * B + 1], &tau, sizeof(float));
  in[2 * B + 2] = m->entry;
  in[2 * B + 3] = nrows;
  return RV_OK;
}

// Scalars of the state block written in stream order (device-pointer API).
__global__ void k_set_scalars(int32_t *in, int Bmax, int mode, float tau, int entry, int nrows) {
  in[2 * Bmax] = mode;
  in[2 * Bmax + 1] = __float_as_int(tau);
  in[2 * Bmax + 2] = entry;
  in[2 * Bmax + 3] = nrows;
}

}  // namespace

namespace rv {
void set_error_message(const char *msg) { g_err = msg ? msg : ""; }
}  // namespace rv

// ==================================================================== C ABI

extern "C" {

const char *rv_last_error(void) { return g_err.c_str(); }

void rv_free_model(rv_model *m) {
  if (!m) return;
  if (m->stream) cudaStreamSynchronize(m->stream);
  drop_graphs(m);
  free_list(m->ws_allocs);
  free_list(m->river_allocs);
  free_list(m->allocs);
  if (m->pinned) cudaFreeHost(m->pinned);
  if (m->own_stream && m->stream) cudaStreamDestroy(m->stream);
  delete m;
}

static int load_impl(rv_model *m, const rv_config *cfg, const void *const *weights) {
  const rv_config &c = *cfg;
  m->c = c;
  m->act = c.act_dtype;
  m->L = c.n_layers; m->d = c.d_model; m->H = c.n_heads; m->Hkv = c.n_kv_heads; m->hd = c.head_dim;
  m->F = c.ffn; m->V = c.vocab; m->Bmax = c.max_batch; m->Tmax = c.max_seq;
  m->qd = m->H * m->hd; m->kvd = m->Hkv * m->hd; m->qkv_n = m->qd + 2 * m->kvd;
  RV_CK(cudaGetDevice(&m->dev));
  RV_CK(cudaDeviceGetAttribute(&m->n_sm, cudaDevAttrMultiProcessorCount, m->dev));
  m->tc_gemm = gemm_tc_available();
  const size_t e2 = 2;
  const int d = m->d, F = m->F, V = m->V;
  auto &A = m->allocs;
  auto up = [&](uint16_t *dst, const void *src, size_t n) -> int {
    RV_CK(cudaMemcpyAsync(dst, src, n * e2, cudaMemcpyHostToDevice, m->stream));
    return RV_OK;
  };
#define RV_UP(dst, src, n)           \
  do {                               \
    int rc_ = up((dst), (src), (n)); \
    if (rc_) return rc_;             \
  } while (0)
  RV_ALLOC_W(A, m->embed, e2 * V * d);
  RV_UP(m->embed, weights[0], (size_t)V * d);
  RV_ALLOC(A, m->final_norm, e2 * d);
  RV_UP(m->final_norm, weights[1], d);
  if (c.tied_embed) {
    m->lm_head = m->embed;
  } else {
    RV_ALLOC_W(A, m->lm_head, e2 * V * d);
    RV_UP(m->lm_head, weights[2], (size_t)V * d);
  }
  m->layers.resize(m->L);
  for (int l = 0; l < m->L; ++l) {
    const void *const *w = weights + 3 + 9 * l;
    LayerDev &ly = m->layers[l];
    RV_ALLOC(A, ly.attn_norm, e2 * d);
    RV_UP(ly.attn_norm, w[0], d);
    RV_ALLOC(A, ly.mlp_norm, e2 * d);
    RV_UP(ly.mlp_norm, w[5], d);
    RV_ALLOC_W(A, ly.w[MAT_QKV], e2 * m->qkv_n * d);
    RV_UP(ly.w[MAT_QKV], w[1], (size_t)m->qd * d);
    RV_UP(ly.w[MAT_QKV] + (size_t)m->qd * d, w[2], (size_t)m->kvd * d);
    RV_UP(ly.w[MAT_QKV] + (size_t)(m->qd + m->kvd) * d, w[3], (size_t)m->kvd * d);
    RV_ALLOC_W(A, ly.w[MAT_O], e2 * d * m->qd);
    RV_UP(ly.w[MAT_O], w[4], (size_t)d * m->qd);
    RV_ALLOC_W(A, ly.w[MAT_GU], e2 * 2 * F * d);
    RV_UP(ly.w[MAT_GU], w[6], (size_t)F * d);
    RV_UP(ly.w[MAT_GU] + (size_t)F * d, w[7], (size_t)F * d);
    RV_ALLOC_W(A, ly.w[MAT_D], e2 * d * F);
    RV_UP(ly.w[MAT_D], w[8], (size_t)d * F);
  }
  // the one KV cache, filled with the sentinel
  m->kv.B = m->Bmax; m->kv.Hkv = m->Hkv; m->kv.T = m->Tmax; m->kv.hd = m->hd;
  m->kv_bytes = (size_t)m->L * 2 * m->Bmax * m->Hkv * (size_t)m->Tmax * m->hd * e2;
  RV_ALLOC(A, m->kv.base, m->kv_bytes);
  RV_CK(launch_fill_u16(m->kv.base, m->kv_bytes / 2, KV_SENTINEL, m->stream));
  RV_ALLOC(A, m->rope_cs, sizeof(float2) * (size_t)m->Tmax * (m->hd / 2));
  RV_CK(launch_rope_table(m->rope_cs, m->Tmax, m->hd, (double)c.rope_theta, m->stream));
  // step state
  RV_ALLOC(A, m->d_state, sizeof(int32_t) * state_words(m->Bmax));
  RV_CK(cudaMemsetAsync(m->d_state, 0, sizeof(int32_t) * state_words(m->Bmax), m->stream));
  state_layout(m);
  {
    const int32_t cap = m->L;  // every backbone layer resident
    m->cap = cap;
    RV_CK(cudaMemcpyAsync(const_cast<int32_t *>(m->st.cap), &cap, sizeof(int32_t), cudaMemcpyHostToDevice, m->stream));
    RV_CK(cudaStreamSynchronize(m->stream));
  }
  {
    cudaError_t e = cudaMallocHost(&m->pinned, sizeof(int32_t) * (m->in_words + m->out_words + 2 * (size_t)m->Bmax));
    if (e != cudaSuccess) {
      m->pinned = nullptr;
      return fail(RV_ENOMEM, "cudaMallocHost failed: %s", cudaGetErrorString(e));
    }
    memset(m->pinned, 0, sizeof(int32_t) * (m->in_words + m->out_words));
  }
  m->h_len.assign(m->Bmax, 0);
  // batch-1 activations and reduction scratch
  RV_ALLOC(A, m->hbuf[0], sizeof(float) * d);
  RV_ALLOC(A, m->hbuf[1], sizeof(float) * d);
  RV_ALLOC(A, m->hmid, sizeof(float) * d);
  RV_ALLOC(A, m->qbuf, sizeof(float) * m->qd);
  RV_ALLOC(A, m->obuf, sizeof(float) * m->qd);
  RV_ALLOC(A, m->abuf, sizeof(float) * F);
  RV_ALLOC(A, m->partials, sizeof(float) * 3 * 4 * (size_t)m->n_sm);
  RV_ALLOC(A, m->seq_min, sizeof(unsigned) * (size_t)m->Bmax);
  RV_CK(cudaMemsetAsync(m->seq_min, 0xFF, sizeof(unsigned) * (size_t)m->Bmax, m->stream));
  RV_ALLOC(A, m->counters, sizeof(unsigned) * (m->L + 4));
  RV_CK(cudaMemsetAsync(m->counters, 0, sizeof(unsigned) * (m->L + 4), m->stream));
  int sp = (2 * m->n_sm + m->Hkv - 1) / m->Hkv;
  const int tiles = (m->Tmax + 31) / 32;
  if (sp > tiles) sp = tiles;
  if (sp > kAttnMaxSplits) sp = kAttnMaxSplits;
  if (sp < 1) sp = 1;
  m->attn_splits_max = sp;  // split count of the persistent kernel's attention
  // decode attention: one cluster of splits per (row, kv head)
  m->attn_cluster = attn_dec_max_cluster(m->hd, m->H / m->Hkv, m->act);
  if (m->attn_cluster < 1) return fail(RV_ECUDA, "decode attention cannot be launched on this device");
  RV_ALLOC(A, m->attn_part, sizeof(float) * (size_t)m->Bmax * m->H * sp * (m->hd + 2));
  RV_ALLOC(A, m->attn_counter, sizeof(unsigned) * (size_t)m->Bmax * m->Hkv);
  RV_ALLOC(A, m->head_keys, sizeof(unsigned long long) * (size_t)m->Bmax);
  RV_CK(cudaMemsetAsync(m->head_keys, 0, sizeof(unsigned long long) * (size_t)m->Bmax, m->stream));
  RV_CK(cudaMemsetAsync(m->attn_counter, 0, sizeof(unsigned) * (size_t)m->Bmax * m->Hkv, m->stream));
  // head rows for the general path, identity list
  RV_ALLOC(A, m->gHf, sizeof(float) * (size_t)m->Bmax * d);
  RV_ALLOC(A, m->gXf, sizeof(float) * (size_t)m->Bmax * d);
  RV_ALLOC(A, m->gLogits, sizeof(float) * (size_t)m->Bmax * V);
  RV_ALLOC(A, m->d_layers, sizeof(LayerDesc) * (size_t)m->L);
  RV_ALLOC(A, m->d_tmaps, sizeof(CUtensorMap) * (size_t)(12 * m->L + 1));
  RV_ALLOC(A, m->bar, sizeof(unsigned) * 2);
  RV_CK(cudaMemsetAsync(m->bar, 0, sizeof(unsigned) * 2, m->stream));
  RV_CK(cudaStreamSynchronize(m->stream));
  return build_stream(m);
}

int rv_load_model(const rv_config *cfg, const void *const *weights, void *stream, rv_model **out) {
  g_err.clear();
  if (!cfg || !weights || !out) return fail(RV_EINVAL, "null argument");
  *out = nullptr;
  const rv_config &c = *cfg;
  if (c.n_layers < 1 || c.d_model < 8 || c.n_heads < 1 || c.n_kv_heads < 1 || c.n_heads % c.n_kv_heads ||
      (c.head_dim != 64 && c.head_dim != 128) || c.ffn < 8 || c.vocab < 2 || c.max_batch < 1 || c.max_seq < 1 ||
      (c.act_dtype != 0 && c.act_dtype != 1) || c.d_model % 32 || c.ffn % 16 ||
      (c.n_heads / c.n_kv_heads) > 8 || !(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f))
    return fail(RV_EINVAL, "unsupported configuration (d_model %% 32, ffn %% 16, head_dim 64/128, H/Hkv <= 8)");
  if ((long)c.max_batch * c.max_seq > (1L << 31) || c.max_batch > 4096)
    return fail(RV_EINVAL, "max_batch x max_seq too large");
  {
    // the batch-1 GEMV keeps element offsets of a matrix in 32 bits
    const uint64_t qkv = (uint64_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
    const uint64_t big = std::max({(uint64_t)c.vocab, qkv, 2 * (uint64_t)c.ffn}) * (uint64_t)c.d_model;
    if (big > 0xFFFFFFFFull || (uint64_t)c.d_model * c.ffn > 0xFFFFFFFFull)
      return fail(RV_EINVAL, "a weight matrix above 2^32 - 1 elements");
  }
  const int nw = 3 + 9 * c.n_layers;
  for (int i = 0; i < nw; ++i)
    if (!weights[i] && !(i == 2 && c.tied_embed)) return fail(RV_EINVAL, "weight %d is NULL", i);
  rv_model *m = new (std::nothrow) rv_model();
  if (!m) return fail(RV_ENOMEM, "host allocation failed");
  if (stream) {
    m->stream = static_cast<cudaStream_t>(stream);
  } else {
    cudaError_t e = cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
      delete m;
      return fail(RV_ECUDA, "cudaStreamCreate failed: %s", cudaGetErrorString(e));
    }
    m->own_stream = true;
  }
  int rc = load_impl(m, cfg, weights);
  if (rc != RV_OK) {
    std::string msg = g_err;
    rv_free_model(m);
    g_err = msg;
    return rc;
  }
  *out = m;
  return RV_OK;
}

int rv_quantize_river(rv_model *m, int group_size, int entry_layer) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  if (group_size < 32 || group_size % 32) return fail(RV_EINVAL, "group_size must be a positive multiple of 32");
  if (entry_layer < 1 || entry_layer > m->L) return fail(RV_EINVAL, "entry_layer must be in 1..L");
  RV_CK(cudaStreamSynchronize(m->stream));
  drop_graphs(m);
  free_list(m->river_allocs);
  m->has_river = false;
  m->stream_ready = false;
  m->group = group_size;
  for (LayerDev &ly : m->layers)
    for (int i = 0; i < N_MAT; ++i) ly.r[i] = RiverDev{};
  RV_CK(cudaMemsetAsync(m->st.err, 0, sizeof(int32_t), m->stream));
  for (LayerDev &ly : m->layers) {
    for (int i = 0; i < N_MAT; ++i) {
      Mat mt = make_mat(m, ly, i);
      RiverDev &r = ly.r[i];
      r.Kp = round32(mt.K);
      r.G = (mt.K + group_size - 1) / group_size;
      r.Gs = pad_groups(r.G);
      auto &A = m->river_allocs;
      RV_ALLOC_W(A, r.q, sizeof(uint32_t) * (size_t)mt.N * (r.Kp / 8));
      RV_ALLOC(A, r.sz, sizeof(__half2) * (size_t)mt.N * r.Gs);
      if (r.Gs != r.G) RV_CK(cudaMemsetAsync(r.sz, 0, sizeof(__half2) * (size_t)mt.N * r.Gs, m->stream));
      if (m->quantizer == RV_QUANT_HQQ)
        RV_CK(launch_hqq_quantize(mt.w, mt.N, mt.K, m->act, group_size, r.Kp, r.q, r.sz, m->st.err, m->stream));
      else
        RV_CK(launch_rtn_quantize(mt.w, mt.N, mt.K, m->act, group_size, r.Kp, r.q, r.sz, m->st.err, m->stream));
    }
  }
  int32_t err = 0;
  RV_CK(cudaMemcpyAsync(&err, m->st.err, sizeof(int32_t), cudaMemcpyDeviceToHost, m->stream));
  RV_CK(cudaStreamSynchronize(m->stream));
  if (err & 4) {
    free_list(m->river_allocs);
    build_stream(m);
    return fail(RV_EINVAL, "a group's scale overflows fp16");
  }
  m->has_river = true;
  m->entry = entry_layer;
  return build_stream(m);
}

int rv_export_river(const rv_model *m, int layer, int proj, void *q_packed, void *scales, void *zeros) {
  g_err.clear();
  if (!m) return fail(RV_EINVAL, "null model");
  if (!m->has_river) return fail(RV_ESTATE, "river not built");
  if (layer < 1 || layer > m->L || proj < 0 || proj > 6) return fail(RV_EINVAL, "bad layer or projection");
  int mat, row0, rows, K;
  switch (proj) {
    case RV_PROJ_Q: mat = MAT_QKV; row0 = 0; rows = m->qd; K = m->d; break;
    case RV_PROJ_K: mat = MAT_QKV; row0 = m->qd; rows = m->kvd; K = m->d; break;
    case RV_PROJ_V: mat = MAT_QKV; row0 = m->qd + m->kvd; rows = m->kvd; K = m->d; break;
    case RV_PROJ_O: mat = MAT_O; row0 = 0; rows = m->d; K = m->qd; break;
    case RV_PROJ_GATE: mat = MAT_GU; row0 = 0; rows = m->F; K = m->d; break;
    case RV_PROJ_UP: mat = MAT_GU; row0 = m->F; rows = m->F; K = m->d; break;
    default: mat = MAT_D; row0 = 0; rows = m->d; K = m->F; break;
  }
  const RiverDev &r = m->layers[layer - 1].r[mat];
  if (q_packed)
    RV_CK(cudaMemcpy2D(q_packed, sizeof(uint32_t) * (K / 8), r.q + (size_t)row0 * (r.Kp / 8), sizeof(uint32_t) * (r.Kp / 8),
                       sizeof(uint32_t) * (K / 8), rows, cudaMemcpyDeviceToHost));
  // (scale, zero) pairs are interleaved on the device in rows padded to Gs
  // pairs: copy the rows, then pick each half on the host
  if (scales || zeros) {
    std::vector<__half2> tmp((size_t)rows * r.Gs);
    RV_CK(cudaMemcpy(tmp.data(), r.sz + (size_t)row0 * r.Gs, sizeof(__half2) * tmp.size(), cudaMemcpyDeviceToHost));
    uint16_t *so = static_cast<uint16_t *>(scales), *zo = static_cast<uint16_t *>(zeros);
    for (int n = 0; n < rows; ++n)
      for (int gi = 0; gi < r.G; ++gi) {
        const __half2 v = tmp[(size_t)n * r.Gs + gi];
        if (so) so[(size_t)n * r.G + gi] = __half_as_ushort(__low2half(v));
        if (zo) zo[(size_t)n * r.G + gi] = __half_as_ushort(__high2half(v));
      }
  }
  return RV_OK;
}

static int validate_step(rv_model *m, int B, const int32_t *forced_host, bool forced_given) {
  if (B < 1 || B > m->Bmax) return fail(RV_EINVAL, "B must be in 1..max_batch");
  if (!forced_given && !m->has_river) return fail(RV_ESTATE, "tau-rule decode needs rv_quantize_river first");
  if (forced_host)
    for (int b = 0; b < B; ++b) {
      if (forced_host[b] < 0 || forced_host[b] > m->L) return fail(RV_EINVAL, "forced exit out of range");
      if (forced_host[b] < m->L && !m->has_river) return fail(RV_ESTATE, "forced exit below L needs the river");
      if (forced_host[b] > m->cap) return fail(RV_EINVAL, "forced exit %d beyond the resident backbone layers (%d)", forced_host[b], m->cap);
    }
  for (int b = 0; b < B; ++b)
    if (m->h_len[b] >= m->Tmax) return fail(RV_ECAPACITY, "row %d: KV cache full (%d positions)", b, m->Tmax);
  return RV_OK;
}

// Device error flags -> status: 8 = a persistent-kernel grid barrier gave up
// waiting, 16 = a tensor-core GEMM wait gave up, 32 = a persistent-kernel
// stage or route wait gave up; the other bits flag invalid inputs (token,
// forced exit, quantization).
static int device_status(int32_t err) {
  if (err & 8) return fail(RV_ETIMEOUT, "a grid barrier of the persistent decode kernel timed out (0x%x)", err);
  if (err & 16) return fail(RV_ETIMEOUT, "a bounded wait of the tensor-core GEMM gave up (0x%x)", err);
  if (err & 32) return fail(RV_ETIMEOUT, "a bounded wait of the persistent decode kernel's weight ring gave up (0x%x)", err);
  return fail(RV_EINVAL, "device flagged an invalid input (0x%x)", err);
}

int rv_decode_step(rv_model *m, const int32_t *tokens, int B, float tau, const int32_t *forced_exit,
                   int32_t *next_ids, int32_t *exit_layer) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  if (!tokens || !next_ids || !exit_layer) return fail(RV_EINVAL, "null pointer");
  int rc = validate_step(m, B, forced_exit, forced_exit != nullptr);
  if (rc) return rc;
  for (int b = 0; b < B; ++b)
    if (tokens[b] < 0 || tokens[b] >= m->V) return fail(RV_EINVAL, "token %d out of range", tokens[b]);
  if (!(tau == tau)) return fail(RV_EINVAL, "tau is NaN");
  int32_t *in = pin_in(m);
  memcpy(in, tokens, sizeof(int32_t) * B);
  if (forced_exit) memcpy(in + m->Bmax, forced_exit, sizeof(int32_t) * B);
  set_scalars(m, forced_exit ? 1 : 0, tau, B);
  RV_CK(cudaMemcpyAsync(m->d_state, in, sizeof(int32_t) * m->in_words, cudaMemcpyHostToDevice, m->stream));
  rc = launch_step(m, B);
  if (rc) return rc;
  int32_t *out = pin_out(m);
  RV_CK(cudaMemcpyAsync(out, m->st.next_ids, sizeof(int32_t) * m->out_words, cudaMemcpyDeviceToHost, m->stream));
  RV_CK(cudaStreamSynchronize(m->stream));
  if (out[2 * m->Bmax]) return device_status(out[2 * m->Bmax]);
  memcpy(next_ids, out, sizeof(int32_t) * B);
  memcpy(exit_layer, out + m->Bmax, sizeof(int32_t) * B);
  for (int b = 0; b < B; ++b) m->h_len[b] += 1;
  return RV_OK;
}

int rv_decode_step_dev(rv_model *m, const int32_t *d_tokens, int B, float tau, const int32_t *d_forced_exit,
                       int32_t *d_next_ids, int32_t *d_exit_layer) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  if (!d_tokens || !d_next_ids || !d_exit_layer) return fail(RV_EINVAL, "null pointer");
  int rc = validate_step(m, B, nullptr, d_forced_exit != nullptr);
  if (rc) return rc;
  if (d_forced_exit && !m->has_river) return fail(RV_ESTATE, "forced exits need the river");
  if (!(tau == tau)) return fail(RV_EINVAL, "tau is NaN");
  RV_CK(cudaMemcpyAsync(m->d_state, d_tokens, sizeof(int32_t) * B, cudaMemcpyDeviceToDevice, m->stream));
  if (d_forced_exit)
    RV_CK(cudaMemcpyAsync(m->d_state + m->Bmax, d_forced_exit, sizeof(int32_t) * B, cudaMemcpyDeviceToDevice,
                          m->stream));
  k_set_scalars<<<1, 1, 0, m->stream>>>(m->d_state, m->Bmax, d_forced_exit ? 1 : 0, tau, m->entry, B);
  RV_CK(cudaGetLastError());
  rc = launch_step(m, B);
  if (rc) return rc;
  RV_CK(cudaMemcpyAsync(d_next_ids, m->st.next_ids, sizeof(int32_t) * B, cudaMemcpyDeviceToDevice, m->stream));
  RV_CK(cudaMemcpyAsync(d_exit_layer, m->st.exit_layer, sizeof(int32_t) * B, cudaMemcpyDeviceToDevice, m->stream));
  for (int b = 0; b < B; ++b) m->h_len[b] += 1;
  return RV_OK;
}

int rv_sync_status(rv_model *m) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  int32_t err = 0;
  RV_CK(cudaMemcpyAsync(&err, m->st.err, sizeof(int32_t), cudaMemcpyDeviceToHost, m->stream));
  RV_CK(cudaStreamSynchronize(m->stream));
  if (err) return device_status(err);
  return RV_OK;
}

int rv_prefill(rv_model *m, const int32_t *tokens, int B, int T0, float tau, int fixed_exit_layer,
               int32_t *next_ids, int32_t *exit_layer) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  if (!tokens || !next_ids || !exit_layer) return fail(RV_EINVAL, "null pointer");
  if (B < 1 || B > m->Bmax || T0 < 1 || T0 > m->Tmax) return fail(RV_EINVAL, "B or T0 out of range");
  if (fixed_exit_layer < -1 || fixed_exit_layer > m->L) return fail(RV_EINVAL, "fixed_exit_layer out of range");
  if (!m->has_river && fixed_exit_layer != m->L) return fail(RV_ESTATE, "prefill with exits needs the river");
  if (fixed_exit_layer > m->cap) return fail(RV_EINVAL, "fixed exit beyond the resident backbone layers (%d)", m->cap);
  if (!(tau == tau)) return fail(RV_EINVAL, "tau is NaN");
  const long M = (long)B * T0;
  if (M > (1L << 24)) return fail(RV_EINVAL, "B x T0 too large");
  for (long i = 0; i < M; ++i)
    if (tokens[i] < 0 || tokens[i] >= m->V) return fail(RV_EINVAL, "token %d out of range", tokens[i]);
  RV_CK(cudaStreamSynchronize(m->stream));
  int rc = ensure_ws(m, M > m->Bmax ? M : m->Bmax);
  if (rc) return rc;
  cudaStream_t s = m->stream;
  RV_CK(cudaMemcpy(m->gTokens, tokens, sizeof(int32_t) * M, cudaMemcpyHostToDevice));
  int32_t *in = pin_in(m);
  for (int b = 0; b < B; ++b) in[m->Bmax + b] = fixed_exit_layer;
  set_scalars(m, fixed_exit_layer >= 0 ? 1 : 0, tau, (int)M);
  RV_CK(cudaMemcpyAsync(m->d_state, in, sizeof(int32_t) * m->in_words, cudaMemcpyHostToDevice, s));
  RV_CK(cudaMemsetAsync(m->st.err, 0, sizeof(int32_t), s));
  RV_CK(launch_step_init(m->st, B, m->L, s));
  RV_CK(launch_embed(m->embed, m->d, m->act, m->gTokens, (int)M, m->V, m->gH, nullptr, m->st.err, s));
  if (m->debug) RV_CK(launch_copy_rows(m->gH + (size_t)(T0 - 1) * m->d, T0 * m->d, m->dbg_h, m->d, m->d, B, s));
  for (int l = 0; l < m->L; ++l) {
    rc = enqueue_layer_rows(m, l, B, T0, nullptr, s);
    if (rc) return rc;
    RV_CK(launch_seq_decide(m->st, m->gHin, m->gH, m->d, B, T0, l + 1, m->L, fixed_exit_layer, m->seq_min,
                            m->debug ? m->dbg_s + (size_t)l * m->Bmax : nullptr, s));
    if (m->debug)
      RV_CK(launch_copy_rows(m->gH + (size_t)(T0 - 1) * m->d, T0 * m->d, m->dbg_h + (size_t)(l + 1) * m->Bmax * m->d,
                             m->d, m->d, B, s));
  }
  RV_CK(launch_copy_rows(m->gH + (size_t)(T0 - 1) * m->d, T0 * m->d, m->gHf, m->d, m->d, B, s));
  // the head runs over B rows: nrows = B (written in-stream; the pinned block may still be in flight)
  k_set_scalars<<<1, 1, 0, s>>>(m->d_state, m->Bmax, fixed_exit_layer >= 0 ? 1 : 0, tau, m->entry, B);
  RV_CK(cudaGetLastError());
  rc = enqueue_head_rows(m, B, 0, T0, s);
  if (rc) return rc;
  int32_t *out = pin_out(m);
  RV_CK(cudaMemcpyAsync(out, m->st.next_ids, sizeof(int32_t) * m->out_words, cudaMemcpyDeviceToHost, s));
  RV_CK(cudaStreamSynchronize(s));
  if (out[2 * m->Bmax]) return device_status(out[2 * m->Bmax]);
  memcpy(next_ids, out, sizeof(int32_t) * B);
  memcpy(exit_layer, out + m->Bmax, sizeof(int32_t) * B);
  for (int b = 0; b < B; ++b) m->h_len[b] = T0;
  return RV_OK;
}

int rv_kv_reset(rv_model *m, const int32_t *rows, int n_rows) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  const int n = rows ? n_rows : m->Bmax;
  if (rows && n_rows < 0) return fail(RV_EINVAL, "n_rows < 0");
  for (int i = 0; i < n; ++i) {
    const int b = rows ? rows[i] : i;
    if (b < 0 || b >= m->Bmax) return fail(RV_EINVAL, "row %d out of range", b);
  }
  RV_CK(cudaStreamSynchronize(m->stream));
  if (!rows) {
    RV_CK(launch_fill_u16(m->kv.base, m->kv_bytes / 2, KV_SENTINEL, m->stream));
  } else {
    const size_t per = (size_t)m->Hkv * m->Tmax * m->hd;
    for (int i = 0; i < n; ++i)
      for (int l = 0; l < m->L; ++l)
        for (int kvi = 0; kvi < 2; ++kvi)
          RV_CK(launch_fill_u16(m->kv.base + m->kv.idx(l, kvi, rows[i], 0, 0), per, KV_SENTINEL, m->stream));
  }
  for (int i = 0; i < n; ++i) {
    const int b = rows ? rows[i] : i;
    m->h_len[b] = 0;
  }
  RV_CK(cudaMemcpyAsync(m->st.len, m->h_len.data(), sizeof(int32_t) * m->Bmax, cudaMemcpyHostToDevice, m->stream));
  RV_CK(cudaStreamSynchronize(m->stream));
  return RV_OK;
}

int rv_set_debug(rv_model *m, int enable) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  RV_CK(cudaStreamSynchronize(m->stream));
  if (enable && !m->dbg_h) {
    auto &A = m->allocs;
    RV_ALLOC(A, m->dbg_h, sizeof(float) * (size_t)(m->L + 1) * m->Bmax * m->d);
    RV_ALLOC(A, m->dbg_s, sizeof(float) * (size_t)m->L * m->Bmax);
    RV_ALLOC(A, m->dbg_logits, sizeof(float) * (size_t)m->Bmax * m->V);
    RV_CK(cudaMemset(m->dbg_h, 0, sizeof(float) * (size_t)(m->L + 1) * m->Bmax * m->d));
    RV_CK(cudaMemset(m->dbg_s, 0xff, sizeof(float) * (size_t)m->L * m->Bmax));
    RV_CK(cudaMemset(m->dbg_logits, 0, sizeof(float) * (size_t)m->Bmax * m->V));
  }
  if ((bool)enable != m->debug) drop_graphs(m);
  m->debug = enable != 0;
  return build_stream(m);
}

int rv_set_option(rv_model *m, int option, int value) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  if (option == RV_OPT_QUANTIZER) {
    if (value != RV_QUANT_RTN && value != RV_QUANT_HQQ) return fail(RV_EINVAL, "unknown quantizer %d", value);
    m->quantizer = value;  // used by the next rv_quantize_river
    return RV_OK;
  }
  if (option == RV_OPT_WAIT_LIMIT_US) {
    if (value < 0) return fail(RV_EINVAL, "wait limit must be >= 0");
    RV_CK(cudaStreamSynchronize(m->stream));
    m->wait_us = value;
    m->sargs.wait_ns = (unsigned long long)value * 1000ull;
    return RV_OK;
  }
  if (option != RV_OPT_DECODE_ENGINE) return fail(RV_EINVAL, "unknown option %d", option);
  if (value != RV_ENGINE_CHAIN && value != RV_ENGINE_PERSISTENT) return fail(RV_EINVAL, "unknown engine %d", value);
  if (value == RV_ENGINE_PERSISTENT && !m->stream_ready)
    return fail(RV_ESTATE, "the persistent decode kernel cannot be made resident on this device");
  RV_CK(cudaStreamSynchronize(m->stream));
  m->engine = value;
  return RV_OK;
}

int rv_debug_dump(rv_model *m, int what, void *dst, size_t bytes) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  if (!dst) return fail(RV_EINVAL, "null dst");
  RV_CK(cudaStreamSynchronize(m->stream));
  const void *src = nullptr;
  size_t need = 0;
  switch (what) {
    case RV_DUMP_HIDDEN: src = m->dbg_h; need = sizeof(float) * (size_t)(m->L + 1) * m->Bmax * m->d; break;
    case RV_DUMP_S: src = m->dbg_s; need = sizeof(float) * (size_t)m->L * m->Bmax; break;
    case RV_DUMP_LOGITS: src = m->dbg_logits; need = sizeof(float) * (size_t)m->Bmax * m->V; break;
    case RV_DUMP_KV: src = m->kv.base; need = m->kv_bytes; break;
    case RV_DUMP_LENS:
      if (bytes != sizeof(int32_t) * m->Bmax) return fail(RV_EINVAL, "size mismatch");
      RV_CK(cudaMemcpy(dst, m->st.len, bytes, cudaMemcpyDeviceToHost));
      return RV_OK;
    default: return fail(RV_EINVAL, "unknown dump id");
  }
  if (!src) return fail(RV_ESTATE, "debug buffers not enabled (rv_set_debug)");
  if (bytes != need) return fail(RV_EINVAL, "size mismatch: need %zu bytes", need);
  RV_CK(cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost));
  return RV_OK;
}

int rv_time_kernel(rv_model *m, int kind, int layer, int river, int iters, float *ms_per_launch, double *bytes) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  if (!ms_per_launch || !bytes || iters < 1 || kind < 0 || kind > 3) return fail(RV_EINVAL, "bad argument");
  if (layer < 1 || layer > m->L) return fail(RV_EINVAL, "layer out of range");
  if (kind == RV_TIME_ATTN) {
    // the decode attention of row 0 at its current position len: reads the
    // K/V of positions 0..len of the layer (q and the output are the step's
    // own buffers, whatever they hold)
    cudaStream_t s = m->stream;
    RV_CK(cudaStreamSynchronize(s));
    AttnArgs at{};
    at.kv = m->kv; at.layer = layer - 1; at.H = m->H; at.Hkv = m->Hkv; at.hd = m->hd; at.act = m->act;
    at.q = m->qbuf; at.o = m->obuf; at.len = m->st.len;
    at.part = m->attn_part; at.counter = m->attn_counter;
    attn_plan(m, 1, &at);
    *bytes = 2.0 * m->Hkv * m->hd * 2.0 * (double)(m->h_len[0] + 1);
    cudaEvent_t e0, e1;
    RV_CK(cudaEventCreate(&e0));
    RV_CK(cudaEventCreate(&e1));
    RV_CK(launch_attn_decode(at, 1, s));  // warm launch
    RV_CK(cudaEventRecord(e0, s));
    for (int i = 0; i < iters; ++i) RV_CK(launch_attn_decode(at, 1, s));
    RV_CK(cudaEventRecord(e1, s));
    RV_CK(cudaEventSynchronize(e1));
    float ms = 0.f;
    RV_CK(cudaEventElapsedTime(&ms, e0, e1));
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    *ms_per_launch = ms / iters;
    return RV_OK;
  }
  if (river && (!m->has_river || kind == RV_TIME_LMHEAD)) return fail(RV_ESTATE, "no river copy for this kernel");
  if (!river && kind != RV_TIME_LMHEAD && layer > m->cap) return fail(RV_ESTATE, "backbone layer %d is offloaded", layer);
  cudaStream_t s = m->stream;
  RV_CK(cudaStreamSynchronize(s));
  const int32_t route = river ? 1 : 0;
  RV_CK(cudaMemcpy(m->st.route, &route, sizeof(int32_t), cudaMemcpyHostToDevice));
  const LayerDev &ly = m->layers[layer - 1];
  GemvArgs a{};
  a.st = m->st;
  a.kv = m->kv;
  a.layer = layer - 1;
  a.L = m->L; a.H = m->H; a.Hkv = m->Hkv; a.hd = m->hd;
  a.eps = m->c.rms_eps;
  a.rope_cs = m->rope_cs;
  a.partials = m->partials;
  int pro, epi;
  if (kind == RV_TIME_GATEUP) {
    a.m = make_mat(m, ly, MAT_GU);
    a.h = m->hbuf[0]; a.gamma = ly.mlp_norm; a.out_vec = m->abuf;
    pro = PRO_NORM; epi = EPI_SWIGLU;
  } else if (kind == RV_TIME_O) {
    a.m = make_mat(m, ly, MAT_O);
    a.vec = m->obuf; a.h_base = m->hbuf[0]; a.h_out = m->hmid;
    pro = PRO_VEC; epi = EPI_RESID;
  } else {
    a.m.w = m->lm_head; a.m.N = m->V; a.m.K = m->d;
    a.h = m->hbuf[0]; a.gamma = m->final_norm;
    a.counter = m->counters + m->L + 1;
    pro = PRO_NORM; epi = EPI_LOGITS;
  }
  const double N = a.m.N, K = a.m.K;
  double wbytes;
  if (river) {
    const int G = (a.m.K + m->group - 1) / m->group;
    wbytes = N * (K / 2.0) + N * G * 4.0;
  } else {
    wbytes = N * K * 2.0;
  }
  // weights + the activation vector read + one fp32 output per row written
  const double out_rows = epi == EPI_SWIGLU ? N / 2 : (epi == EPI_LOGITS ? 0 : N);
  *bytes = wbytes + K * 4.0 + out_rows * 4.0;
  cudaEvent_t e0, e1;
  RV_CK(cudaEventCreate(&e0));
  RV_CK(cudaEventCreate(&e1));
  RV_CK(launch_gemv_b1(m->act, pro, epi, a, gemv_grid(m, 0), s));  // warm launch
  RV_CK(cudaEventRecord(e0, s));
  for (int i = 0; i < iters; ++i) RV_CK(launch_gemv_b1(m->act, pro, epi, a, gemv_grid(m, 0), s));
  RV_CK(cudaEventRecord(e1, s));
  RV_CK(cudaEventSynchronize(e1));
  float ms = 0.f;
  RV_CK(cudaEventElapsedTime(&ms, e0, e1));
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  *ms_per_launch = ms / iters;
  // the LM head's argmax advanced len[0]; restore the host's view
  RV_CK(cudaMemcpy(m->st.len, m->h_len.data(), sizeof(int32_t) * m->Bmax, cudaMemcpyHostToDevice));
  return RV_OK;
}

size_t rv_kv_bytes(const rv_model *m) { return m ? m->kv_bytes : 0; }

int rv_debug_fail_alloc(int after) {
  g_fail_after.store(after < 0 ? -1 : after);
  return RV_OK;
}

int rv_decode_attention_plan(int batch, int n_kv_heads, int n_sm, int max_cluster, int max_splits, int context,
                             int *splits) {
  g_err.clear();
  if (!splits) return fail(RV_EINVAL, "null pointer");
  if (batch < 1 || n_kv_heads < 1 || n_sm < 1 || max_splits < 1 || context < 0)
    return fail(RV_EINVAL, "bad argument");
  if (max_cluster < 1 || max_cluster > 16 || (max_cluster & (max_cluster - 1)))
    return fail(RV_EINVAL, "max_cluster must be a power of two <= 16");
  return attn_dec_plan(batch, n_kv_heads, n_sm, max_cluster, max_splits, context, splits);
}

int rv_offload_backbone(rv_model *m, int keep_layers) {
  g_err.clear();
  if (check_common(m)) return RV_EINVAL;
  if (!m->has_river) return fail(RV_ESTATE, "offloading needs the river (rv_quantize_river)");
  if (keep_layers < 1 || keep_layers > m->L) return fail(RV_EINVAL, "keep_layers must be in 1..L");
  if (keep_layers > m->cap) return fail(RV_ESTATE, "backbone layers above %d were already offloaded", m->cap);
  if (keep_layers == m->cap) return RV_OK;
  RV_CK(cudaStreamSynchronize(m->stream));
  drop_graphs(m);  // captured steps hold the matrices' pointers
  for (int l = keep_layers; l < m->L; ++l)
    for (int i = 0; i < N_MAT; ++i) {
      void *p = m->layers[l].w[i];
      if (!p) continue;
      auto it = std::find(m->allocs.begin(), m->allocs.end(), p);
      if (it != m->allocs.end()) m->allocs.erase(it);
      RV_CK(cudaFree(p));
      m->layers[l].w[i] = nullptr;
    }
  const int32_t cap = keep_layers;
  RV_CK(cudaMemcpy(const_cast<int32_t *>(m->st.cap), &cap, sizeof(int32_t), cudaMemcpyHostToDevice));
  m->cap = keep_layers;
  return build_stream(m);
}

size_t rv_param_bytes(const rv_model *m, int which) {
  if (!m) return 0;
  size_t t = 0;
  if (which == 0) {  // resident 16-bit parameters: embedding, LM head, norms, backbone layers 1..cap
    const size_t d = m->d;
    t = 2 * ((size_t)m->V * d * (m->c.tied_embed ? 1 : 2) + d);
    t += (size_t)m->L * 2 * (2 * d);
    t += (size_t)m->cap * 2 * ((size_t)m->qkv_n * d + d * m->qd + 2 * (size_t)m->F * d + d * m->F);
    return t;
  }
  if (!m->has_river) return 0;
  for (const LayerDev &ly : m->layers)
    for (int i = 0; i < N_MAT; ++i) {
      const int N = i == MAT_QKV ? m->qkv_n : i == MAT_GU ? 2 * m->F : m->d;
      t += (size_t)N * (ly.r[i].Kp / 2) + 2 * sizeof(__half) * (size_t)N * ly.r[i].G;
    }
  return t;
}

}  // extern "C"
