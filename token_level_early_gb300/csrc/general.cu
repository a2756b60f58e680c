// Multi-row kernels: prefill over B x T0 prompt tokens and decode steps with
// B > 1 rows.  Rows that share a path (backbone or river) are gathered
// through a device-side index list, so one launch per path and per
// projection serves a batch in which rows exit at different layers; both
// paths write the same KV cache slots.
//
// Method: "River-LLM: Large Language Model Seamless Exit Based on KV Share",
// paperlayer.ai summary section 2 (token-level vs sequence-level exit),
// section 3 (Sequence-level Exit: the latest-exiting token sets the depth) and
// section 4 (phase-adaptive: sequence-level exit in prefill, token-level in
// generation).
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

// A launch whose error returns from the enclosing launcher.
#define RV_CK_LAUNCH(call)                     \
  do {                                         \
    const cudaError_t e_ = (call);             \
    if (e_ != cudaSuccess) return e_;          \
  } while (0)

namespace rv {

static inline int cdiv(long a, long b) { return (int)((a + b - 1) / b); }

// ------------------------------------------------------------------ embed / init

__global__ void k_embed(const uint16_t *E, int d, int act, const int32_t *tokens, int vocab, float *H,
                        float *dbg_h, int32_t *err) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x;
  int tok = tokens[m];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) atomicOr(err, 1);
    tok = 0;
  }
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float v = act_to_f(E[(size_t)tok * d + i], act);
    H[(size_t)m * d + i] = v;
    if (dbg_h) dbg_h[(size_t)m * d + i] = v;
  }
}

cudaError_t launch_embed(const uint16_t *E, int d, int act, const int32_t *tokens, int M, int vocab, float *H,
                         float *dbg_h, int32_t *err, cudaStream_t s, int pdl) {
  if (M <= 0) return cudaSuccess;
  return launch_k(k_embed, dim3(M), dim3(256), 0, s, pdl, E, d, act, tokens, vocab, H, dbg_h, err);
}

// Route state at the start of a step (forced mode: exit 0 = all river).
__global__ void k_step_init(StepState st, int B, int L) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  if (*st.mode == 1) {
    int f = st.forced[b];
    if (f < 0 || f > L) { atomicOr(st.err, 2); f = L; }
    st.route[b] = f == 0;
    st.exit_layer[b] = f == 0 ? 0 : L;
  } else {
    st.route[b] = 0;
    st.exit_layer[b] = L;
  }
}

cudaError_t launch_step_init(const StepState &st, int B, int L, cudaStream_t s) {
  RV_CK_LAUNCH(launch_k(k_step_init, dim3(cdiv(B, 128)), dim3(128), 0, s, 1, st, B, L));
  return cudaGetLastError();
}

// Index lists of the token rows on each path: lists[p * stride + i].
__global__ void k_route_lists(const int32_t *route, int B, int T, int32_t *lists, int stride, int32_t *counts) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  extern __shared__ int off[];  // [B]
  if (threadIdx.x == 0) {
    int c0 = 0, c1 = 0;
    for (int b = 0; b < B; ++b) {
      if (route[b] == 0) { off[b] = c0; c0 += T; }
      else { off[b] = c1; c1 += T; }
    }
    counts[0] = c0;
    counts[1] = c1;
  }
  __syncthreads();
  const long total = (long)B * T;
  for (long i = threadIdx.x; i < total; i += blockDim.x) {
    const int b = (int)(i / T), t = (int)(i % T), p = route[b] != 0;
    lists[(long)p * stride + off[b] + t] = (int32_t)i;
  }
}

cudaError_t launch_route_lists(const int32_t *route, int B, int T, int32_t *lists, int list_stride,
                               int32_t *counts, cudaStream_t s) {
  RV_CK_LAUNCH(launch_k(k_route_lists, dim3(1), dim3(1024), sizeof(int) * B, s, 1, route, B, T, lists, list_stride, counts));
  return cudaGetLastError();
}

// ------------------------------------------------------------------ row-wise ops

__global__ void k_rmsnorm_rows(const float *H, const uint16_t *gamma, int d, float eps, int act, float *X,
                               const int32_t *list, const int32_t *count) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  __shared__ float red[32];
  for (int idx = blockIdx.x; idx < *count; idx += gridDim.x) {
    const int m = list ? list[idx] : idx;
    const float *h = H + (size_t)m * d;
    float ss = 0.f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) ss = fmaf(h[i], h[i], ss);
    ss = block_sum(ss, red);
    const float r = 1.0f / sqrtf(ss / (float)d + eps);
    for (int i = threadIdx.x; i < d; i += blockDim.x)
      X[(size_t)m * d + i] = round_act(h[i] * r * act_to_f(gamma[i], act), act);
    __syncthreads();
  }
}

cudaError_t launch_rmsnorm_rows(const float *H, const uint16_t *gamma, int d, float eps, int act, float *X,
                                const int32_t *list, const int32_t *count, int max_rows, cudaStream_t s) {
  if (max_rows <= 0) return cudaSuccess;
  RV_CK_LAUNCH(launch_k(k_rmsnorm_rows, dim3(min(max_rows, 4096)), dim3(256), 0, s, 1, H, gamma, d, eps, act, X, list, count));
  return cudaGetLastError();
}

__global__ void k_resid_rows(float *H, const float *Y, int d, const int32_t *list, const int32_t *count) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  const long total = (long)(*count) * d;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int idx = (int)(i / d), c = (int)(i % d);
    const int m = list ? list[idx] : idx;
    H[(size_t)m * d + c] += Y[(size_t)m * d + c];
  }
}

cudaError_t launch_resid_rows(float *H, const float *Y, int d, const int32_t *list, const int32_t *count,
                              int max_rows, cudaStream_t s) {
  if (max_rows <= 0) return cudaSuccess;
  RV_CK_LAUNCH(launch_k(k_resid_rows, dim3(min(cdiv((long)max_rows * d, 256), 8192)), dim3(256), 0, s, 1, H, Y, d, list, count));
  return cudaGetLastError();
}

// a = round16(silu(gate) * up); Y rows hold [gate (F) | up (F)].
__global__ void k_swiglu_rows(const float *Y, int F, int act, float *A, const int32_t *list, const int32_t *count) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  const long total = (long)(*count) * F;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int idx = (int)(i / F), c = (int)(i % F);
    const int m = list ? list[idx] : idx;
    const float g = Y[(size_t)m * 2 * F + c], u = Y[(size_t)m * 2 * F + F + c];
    A[(size_t)m * F + c] = round_act(g / (1.0f + expf(-g)) * u, act);
  }
}

cudaError_t launch_swiglu_rows(const float *Y, int F, int act, float *A, const int32_t *list,
                               const int32_t *count, int max_rows, cudaStream_t s) {
  if (max_rows <= 0) return cudaSuccess;
  RV_CK_LAUNCH(launch_k(k_swiglu_rows, dim3(min(cdiv((long)max_rows * F, 256), 8192)), dim3(256), 0, s, 1, Y, F, act, A, list, count));
  return cudaGetLastError();
}

// RoPE on q and k, K/V into the cache slot (layer, sequence, position).
__global__ void k_rope_rows(RopeRowsArgs a) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  const int half = a.hd / 2, qkv = (a.H + 2 * a.Hkv) * a.hd;
  for (int idx = blockIdx.x; idx < *a.count; idx += gridDim.x) {
    const int m = a.list ? a.list[idx] : idx;
    const int b = m / a.tokens_per_row;
    const int pos = (a.base ? a.base[b] : 0) + m % a.tokens_per_row;
    const float *y = a.Y + (size_t)m * qkv;
    for (int u = threadIdx.x; u < (a.H + 2 * a.Hkv) * half; u += blockDim.x) {
      const int slot = u / half, r = u % half;
      const float y0 = y[slot * a.hd + r], y1 = y[slot * a.hd + r + half];
      if (slot < a.H + a.Hkv) {
        const float2 cs = a.rope_cs[(size_t)pos * half + r];
        const float o0 = y0 * cs.x - y1 * cs.y, o1 = y0 * cs.y + y1 * cs.x;
        if (slot < a.H) {
          a.q[(size_t)m * a.H * a.hd + slot * a.hd + r] = round_act(o0, a.act);
          a.q[(size_t)m * a.H * a.hd + slot * a.hd + r + half] = round_act(o1, a.act);
        } else {
          uint16_t *k = a.kv.base + a.kv.idx(a.layer, 0, b, slot - a.H, pos);
          k[r] = f_to_act(o0, a.act);
          k[r + half] = f_to_act(o1, a.act);
        }
      } else {
        uint16_t *v = a.kv.base + a.kv.idx(a.layer, 1, b, slot - a.H - a.Hkv, pos);
        v[r] = f_to_act(y0, a.act);
        v[r + half] = f_to_act(y1, a.act);
      }
    }
  }
}

cudaError_t launch_rope_rows(const RopeRowsArgs &a, int max_rows, cudaStream_t s) {
  if (max_rows <= 0) return cudaSuccess;
  RV_CK_LAUNCH(launch_k(k_rope_rows, dim3(min(max_rows, 8192)), dim3(256), 0, s, 1, a));
  return cudaGetLastError();
}

// Token-level decision for each decode row (one block per row).
__global__ void k_decide_rows(StepState st, const float *Hin, const float *H, int d, int layer1, int L,
                              float *dbg_s) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  __shared__ float red[96];
  const int b = blockIdx.x;
  float dot = 0.f, n1 = 0.f, n2 = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float x = Hin[(size_t)b * d + i], y = H[(size_t)b * d + i];
    dot = fmaf(x, y, dot);
    n1 = fmaf(x, x, n1);
    n2 = fmaf(y, y, n2);
  }
  dot = block_sum(dot, red);
  n1 = block_sum(n1, red + 32);
  n2 = block_sum(n2, red + 64);
  if (threadIdx.x == 0) decide_row(st, b, layer1, L, dot, n1, n2, dbg_s);
}

cudaError_t launch_decide_rows(const StepState &st, const float *Hin, const float *H, int d, int B, int layer1,
                               int L, float *dbg_s, cudaStream_t s) {
  RV_CK_LAUNCH(launch_k(k_decide_rows, dim3(B), dim3(256), 0, s, 1, st, Hin, H, d, layer1, L, dbg_s));
  return cudaGetLastError();
}

// Sequence-level decision for prefill: exit when min over the sequence's
// tokens of s_t(l) exceeds tau (the latest-exiting token sets the depth).
// Pass 1 spreads the tokens over the GPU (a warp per token, the same sums in
// the same order as a single-block pass would take) and folds each block's
// minimum into smin[b], a float in an order-preserving unsigned encoding (min
// is exact, so the result does not depend on the order of the atomics).
// Pass 2 decides and re-arms smin[b] for the next layer.
__device__ __forceinline__ unsigned f2ord(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord2f(unsigned o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

constexpr int SEQ_TOK_PER_BLOCK = 64;

__global__ void k_seq_smin(StepState st, const float *Hin, const float *H, int d, int T, unsigned *smin) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  __shared__ float wmin[32];
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (st.route[b] != 0) return;
  const int t0 = blockIdx.x * SEQ_TOK_PER_BLOCK, t1 = min(T, t0 + SEQ_TOK_PER_BLOCK);
  float mn = INFINITY;
  for (int t = t0 + warp; t < t1; t += nw) {
    const float *x = Hin + ((size_t)b * T + t) * d, *y = H + ((size_t)b * T + t) * d;
    float dot = 0.f, n1 = 0.f, n2 = 0.f;
    for (int i = lane; i < d; i += 32) {
      dot = fmaf(x[i], y[i], dot);
      n1 = fmaf(x[i], x[i], n1);
      n2 = fmaf(y[i], y[i], n2);
    }
    dot = warp_sum(dot);
    n1 = warp_sum(n1);
    n2 = warp_sum(n2);
    const float s = dot / fmaxf(sqrtf(n1) * sqrtf(n2), 1e-8f);
    mn = fminf(mn, s);
  }
  if (lane == 0) wmin[warp] = mn;
  __syncthreads();
  if (threadIdx.x != 0) return;
  for (int w = 1; w < nw; ++w) mn = fminf(mn, wmin[w]);
  mn = fminf(mn, wmin[0]);
  atomicMin(smin + b, f2ord(mn));
}

__global__ void k_seq_decide(StepState st, int B, int layer1, int L, int fixed_exit, unsigned *smin,
                             float *dbg_smin) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const unsigned o = smin[b];
  smin[b] = 0xFFFFFFFFu;  // re-armed for the next layer
  if (st.route[b] != 0) {
    if (dbg_smin) dbg_smin[b] = __int_as_float(0x7fc00000);
    return;
  }
  const float mn = o == 0xFFFFFFFFu ? INFINITY : ord2f(o);  // no token: as the empty minimum
  if (dbg_smin) dbg_smin[b] = mn;
  bool go;
  if (fixed_exit >= 0)
    go = layer1 == fixed_exit && layer1 < L;
  else
    go = layer1 >= *st.entry && layer1 <= L - 1 && mn > *st.tau;
  if (layer1 >= *st.cap && layer1 < L) go = true;  // backbone offloaded past the cap
  if (go) {
    st.route[b] = 1;
    st.exit_layer[b] = layer1;
  }
}

cudaError_t launch_seq_decide(const StepState &st, const float *Hin, const float *H, int d, int B, int T,
                              int layer1, int L, int fixed_exit, unsigned *smin, float *dbg_smin, cudaStream_t s) {
  if (T > 0) {
    RV_CK_LAUNCH(launch_k(k_seq_smin, dim3(dim3((T + SEQ_TOK_PER_BLOCK - 1) / SEQ_TOK_PER_BLOCK, B)), dim3(256), 0, s, 1, st, Hin, H, d, T, smin));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  RV_CK_LAUNCH(launch_k(k_seq_decide, dim3((B + 127) / 128), dim3(128), 0, s, 1, st, B, layer1, L, fixed_exit, smin, dbg_smin));
  return cudaGetLastError();
}

// Greedy pick per row: largest logit, lowest index on ties.
__global__ void k_argmax_rows(const float *logits, int V, StepState st, int bump_len, int set_len) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  __shared__ float bv[32];
  __shared__ int bi[32];
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  float best = -INFINITY;
  int besti = 0x7fffffff;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float x = logits[(size_t)b * V + v];
    if (x > best) { best = x; besti = v; }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, besti, o);
    if (ov > best || (ov == best && oi < besti)) { best = ov; besti = oi; }
  }
  if (lane == 0) { bv[warp] = best; bi[warp] = besti; }
  __syncthreads();
  if (threadIdx.x == 0) {
    best = bv[0]; besti = bi[0];
    for (int w = 1; w < nw; ++w)
      if (bv[w] > best || (bv[w] == best && bi[w] < besti)) { best = bv[w]; besti = bi[w]; }
    st.next_ids[b] = besti == 0x7fffffff ? 0 : besti;
    if (bump_len) st.len[b] += 1;
    if (set_len >= 0) st.len[b] = set_len;
  }
}

cudaError_t launch_argmax_rows(const float *logits, int V, int B, StepState st, int bump_len, int set_len,
                               cudaStream_t s) {
  RV_CK_LAUNCH(launch_k(k_argmax_rows, dim3(B), dim3(1024), 0, s, 1, logits, V, st, bump_len, set_len));
  return cudaGetLastError();
}

__global__ void k_copy_rows(const float *src, int src_stride, float *dst, int dst_stride, int d) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < d; i += blockDim.x) dst[(size_t)b * dst_stride + i] = src[(size_t)b * src_stride + i];
}

cudaError_t launch_copy_rows(const float *src, int src_stride, float *dst, int dst_stride, int d, int B,
                             cudaStream_t s) {
  RV_CK_LAUNCH(launch_k(k_copy_rows, dim3(B), dim3(256), 0, s, 1, src, src_stride, dst, dst_stride, d));
  return cudaGetLastError();
}

// ------------------------------------------------------------------ GEMM
// Y[m][n] = sum_k W[n][k] X[m][k] for the listed rows m, W either the 16-bit
// backbone matrix or the river copy whose element is (q - z) * s (exact in
// fp32).  CUDA-core tiles of 64 rows x 64 outputs x 16 columns.

constexpr int GBM = 64, GBN = 64, GBK = 16;

__global__ void __launch_bounds__(256) k_gemm_rows(Mat mt, int river, int act, const float *X, float *Y,
                                                   const int32_t *list, const int32_t *count) {
  pdl_wait();  // griddepcontrol.wait: the previous kernel's results are visible
  pdl_trigger();
  __shared__ float Xs[GBK][GBM + 4];
  __shared__ float Ws[GBK][GBN + 4];
  __shared__ int rows[GBM];
  const int cnt = *count;
  const int r0 = blockIdx.y * GBM;
  if (r0 >= cnt) return;
  const int n0 = blockIdx.x * GBN;
  const int N = mt.N, K = mt.K;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  if (tid < GBM) rows[tid] = (r0 + tid < cnt) ? (list ? list[r0 + tid] : r0 + tid) : -1;
  __syncthreads();
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  const int lr = tid / 4, lk = (tid % 4) * 4;  // loader: row/col lr, k offset lk
  for (int k0 = 0; k0 < K; k0 += GBK) {
    // X tile
    {
      const int m = rows[lr];
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m >= 0 && k0 + lk < K) v = *reinterpret_cast<const float4 *>(X + (size_t)m * K + k0 + lk);
      Xs[lk + 0][lr] = v.x; Xs[lk + 1][lr] = v.y; Xs[lk + 2][lr] = v.z; Xs[lk + 3][lr] = v.w;
    }
    // W tile
    {
      const int n = n0 + lr;
      float w[4] = {0.f, 0.f, 0.f, 0.f};
      if (n < N && k0 + lk < K) {
        const int k = k0 + lk;
        if (!river) {
          const uint2 raw = *reinterpret_cast<const uint2 *>(mt.w + (size_t)n * K + k);
          const uint16_t *p = reinterpret_cast<const uint16_t *>(&raw);
#pragma unroll
          for (int j = 0; j < 4; ++j) w[j] = act_to_f(p[j], act);
        } else {
          const RiverMat &R = mt.r;
          const uint32_t word = R.q[(size_t)n * (R.Kp >> 3) + (k >> 3)];
          const int gi = k / R.g;
          const float2 szf = __half22float2(R.sz[(size_t)n * R.Gs + gi]);
          const float s = szf.x, z = szf.y;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float q = (float)((word >> (4 * ((k + j) & 7))) & 0xFu);
            w[j] = (q - z) * s;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) Ws[lk + j][lr] = w[j];
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < GBK; ++kk) {
      const float4 a4 = *reinterpret_cast<const float4 *>(&Xs[kk][ty * 4]);
      const float4 b4 = *reinterpret_cast<const float4 *>(&Ws[kk][tx * 4]);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bw[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = rows[ty * 4 + i];
    if (m < 0) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) Y[(size_t)m * N + n] = acc[i][j];
    }
  }
}

cudaError_t launch_gemm_rows(const Mat &m, int river, int act, const float *X, float *Y, const int32_t *list,
                             const int32_t *count, int max_rows, cudaStream_t s) {
  if (max_rows <= 0) return cudaSuccess;
  dim3 grid(cdiv(m.N, GBN), cdiv(max_rows, GBM));
  if (grid.y > 65535) return cudaErrorInvalidValue;
  RV_CK_LAUNCH(launch_k(k_gemm_rows, dim3(grid), dim3(256), 0, s, 1, m, river, act, X, Y, list, count));
  return cudaGetLastError();
}

}  // namespace rv
