// Single-row (batch 1) decode kernels of the River-LLM token-level early exit.
//
// One decode step at batch 1 is a chain of GEMV kernels per layer:
//   qkv  : RMSNorm(h) -> [q;k;v] = W_qkv x -> RoPE -> K/V into slot (l, 0, p)
//   attn : split-KV GQA decode attention (attention.cu)
//   o    : h_mid = h + W_o o
//   gu   : RMSNorm(h_mid) -> a = silu(W_g x) * (W_u x)
//   down : h_out = h_mid + W_d a, s(l) = cos(h, h_out), exit decision
// and a final LM-head GEMV with a fused greedy argmax.  Every GEMV reads the
// row's route flag on the device and streams either the 16-bit backbone
// matrix or its int4 river copy (same kernel, same grid), so a step needs no
// host round trip per layer and is captured once in a CUDA graph.
//
// GEMV engine.  A warp owns 4 output rows (a "quad") and a subset of the K
// chunks; the 8 warps of a block split K (S ways) and cover 8/S quads.  A
// lane's activation chunk sits in registers and serves the 4 rows; lanes
// stream 16-byte weight pieces (a coalesced 512-byte run per row and warp).
// Partial sums are reduced across lanes by a transpose-reduce and across the
// K splits through shared memory; the epilogue then runs once per row.
//
// int4 inner loop.  A code q becomes the float 1 + q/16 (nibble rotated into
// mantissa bits 19..22 and the exponent of 1.0 OR-ed in) or 1 + q/256 (bits
// 15..18): one funnel rotate per pair of codes and one LOP3 per code.  The
// matching activation is pre-scaled by 16 or 256, so (1 + q/16)(16 x) =
// 16 x + q x, and the constant sum of the pre-scaled activations is removed
// once per 32 codes.  Products and sums are fp32 (packed fma.rn.f32x2), the
// products exact.  Per 32 codes of a row: sum w x = s (sum q x - z sum x).
//
// Method: "River-LLM: Large Language Model Seamless Exit Based on KV Share",
// paperlayer.ai summary section 4 (KV-Shared Exit Layer; Inference with
// Seamless Exit) and aitrends.kr (s(l) = cos(h(l-1), h(l)) > tau; W4A16 exit
// layers copied from the backbone blocks).
#include "common.cuh"
#include "kernels.cuh"

namespace rv {

constexpr int NW = 8;      // warps per block
constexpr int CH4 = 1024;  // int4 chunk: 32 lanes x 32 codes
constexpr int CH16 = 256;  // 16-bit chunk: 32 lanes x 8 values

typedef unsigned long long u64;

// 128-bit streaming load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ u64 pack2(float lo, float hi) {
  return ((u64)__float_as_uint(hi) << 32) | (u64)__float_as_uint(lo);
}

__device__ __forceinline__ float sum2(u64 v) {
  return __uint_as_float((uint32_t)v) + __uint_as_float((uint32_t)(v >> 32));
}

// d = a * b + c on two fp32 lanes at once.
__device__ __forceinline__ u64 ffma2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint32_t rotl(uint32_t x, int s) { return __funnelshift_l(x, x, s); }

// One word of 8 codes (canonical nibble order) against its 4 activation
// pairs.  Pair p holds (16 x[even nibble], 256 x[odd nibble]) for the nibble
// pairs (0,7), (2,1), (4,3), (6,5), which rotations by 19, 11, 3 and 27 bring
// to bits 19..22 and 15..18.
__device__ __forceinline__ u64 word_fma(uint32_t w, const u64 *xp, u64 acc) {
  const int rot[4] = {19, 11, 3, 27};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t u = rotl(w, rot[p]);
    const uint32_t fh = (u & 0x00780000u) | 0x3F800000u;  // 1 + q/16
    const uint32_t fl = (u & 0x00078000u) | 0x3F800000u;  // 1 + q/256
    acc = ffma2(((u64)fl << 32) | fh, xp[p], acc);
  }
  return acc;
}

// Two 16-bit weights of a word times their activations (packed fp32 FMA).
template <int ACT>
__device__ __forceinline__ u64 pair16_fma(uint32_t w, u64 x, u64 acc) {
  u64 f;
  if (ACT == 1) {
    f = ((u64)(w & 0xFFFF0000u) << 32) | (u64)(w << 16);
  } else {
    const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&w));
    f = pack2(v.x, v.y);
  }
  return ffma2(f, x, acc);
}

// Rows of quad qd by epilogue; pairs (0,2) and (1,3) stay together where the
// epilogue combines two rows (RoPE pairs i, i + hd/2; gate/up pairs).
template <int EPI>
__device__ __forceinline__ void quad_rows(const GemvArgs &a, int qd, int *rows) {
  if (EPI == EPI_QKV) {
    const int hq = a.hd >> 2, slot = qd / hq, rr = (qd - slot * hq) * 2;
    const int base = slot * a.hd + rr, half = a.hd >> 1;
    rows[0] = base; rows[1] = base + 1; rows[2] = base + half; rows[3] = base + half + 1;
  } else if (EPI == EPI_SWIGLU) {
    const int u = qd * 2, F = a.m.N >> 1;
    rows[0] = u; rows[1] = u + 1; rows[2] = F + u; rows[3] = F + u + 1;
  } else {
    rows[0] = 4 * qd; rows[1] = 4 * qd + 1; rows[2] = 4 * qd + 2; rows[3] = 4 * qd + 3;
  }
}

__host__ __device__ __forceinline__ int split_of(int nk) { return nk >= 8 ? 8 : nk >= 4 ? 4 : nk >= 2 ? 2 : 1; }

// Transpose-reduce of 4 per-lane values over the warp: the total of v[r]
// ends in lane 8 * r.
__device__ __forceinline__ float quad_reduce(const float *v, int lane) {
  const bool b4 = lane & 16, b3 = lane & 8;
  const float s0 = b4 ? v[0] : v[2], s1 = b4 ? v[1] : v[3];
  const float k0 = (b4 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, s0, 16);
  const float k1 = (b4 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, s1, 16);
  float m = (b3 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, b3 ? k0 : k1, 8);
  m += __shfl_xor_sync(0xffffffffu, m, 4);
  m += __shfl_xor_sync(0xffffffffu, m, 2);
  m += __shfl_xor_sync(0xffffffffu, m, 1);
  return m;
}

// Last-block-done: true in exactly one block once every block has published
// its partials; the counter is left at zero for the next launch.
__device__ __forceinline__ bool last_block(unsigned *counter) {
  __shared__ bool am_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned t = atomicAdd(counter, 1u);
    am_last = (t == gridDim.x - 1);
    if (am_last) *counter = 0u;
  }
  __syncthreads();
  if (am_last) __threadfence();
  return am_last;
}

struct Geo {
  int K, Kp, nk4, nk16, words, G;
};

__host__ __device__ __forceinline__ Geo geo_of(const Mat &m) {
  Geo g;
  g.K = m.K;
  g.Kp = m.r.Kp > 0 ? m.r.Kp : ((m.K + 31) & ~31);
  g.nk4 = (g.Kp + CH4 - 1) / CH4;
  g.nk16 = (m.K + CH16 - 1) / CH16;
  g.words = g.Kp >> 3;
  g.G = m.r.G;
  return g;
}

// Shared memory (floats): activations in the lane layout of the larger path,
// then 256 floats of reduction scratch.
__host__ __device__ __forceinline__ size_t smem_floats(const Geo &g) {
  const size_t river = (size_t)g.nk4 * (8 * 32 * 4 + 32 * 2);
  const size_t b16 = (size_t)g.nk16 * (2 * 32 * 4);
  return (river > b16 ? river : b16) + 256;
}

template <int ACT, int PRO>
__device__ __forceinline__ float x_at(const GemvArgs &a, int k, float r) {
  if (PRO == PRO_NORM) return round_act(a.h[k] * r * act_to_f(a.gamma[k], ACT), ACT);
  return a.vec[k];
}

template <int ACT, int PRO, int EPI>
__global__ void __launch_bounds__(NW * 32, 3) k_gemv_b1(GemvArgs a) {
  extern __shared__ __align__(16) float smem[];
  const Geo g = geo_of(a.m);
  const int river = (EPI == EPI_LOGITS) ? 0 : a.st.route[0];
  const int nk = river ? g.nk4 : g.nk16;
  float *red = smem + (smem_floats(g) - 256);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- prologue: x = round16(RMSNorm(h) * gamma) or x = vec, in the lane layout
  float rs = 0.f;
  if (PRO == PRO_NORM) {
    float ss = 0.f;
    for (int i = tid; i < g.K; i += blockDim.x) ss = fmaf(a.h[i], a.h[i], ss);
    ss = block_sum(ss, red);
    rs = 1.0f / sqrtf(ss / (float)g.K + a.eps);
  }
  if (river) {
    float4 *xq = reinterpret_cast<float4 *>(smem);                    // [nk][8][32]
    float2 *cx = reinterpret_cast<float2 *>(smem + nk * 8 * 32 * 4);  // [nk][32] (C, X)
    for (int t = tid; t < nk * 32; t += blockDim.x) {
      const int c = t >> 5, ln = t & 31, base = c * CH4 + ln * 32;
      float C = 0.f, X = 0.f;
      const int ev[4] = {0, 2, 4, 6}, od[4] = {7, 1, 3, 5};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float e[4][2];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int ke = base + 8 * i + ev[p], ko = base + 8 * i + od[p];
          const float xe = ke < g.K ? x_at<ACT, PRO>(a, ke, rs) : 0.f;
          const float xo = ko < g.K ? x_at<ACT, PRO>(a, ko, rs) : 0.f;
          e[p][0] = 16.f * xe;
          e[p][1] = 256.f * xo;
          C += e[p][0] + e[p][1];
          X += xe + xo;
        }
        xq[(c * 8 + 2 * i) * 32 + ln] = make_float4(e[0][0], e[0][1], e[1][0], e[1][1]);
        xq[(c * 8 + 2 * i + 1) * 32 + ln] = make_float4(e[2][0], e[2][1], e[3][0], e[3][1]);
      }
      cx[c * 32 + ln] = make_float2(C, X);
    }
  } else {
    float4 *xb = reinterpret_cast<float4 *>(smem);  // [nk][2][32]
    for (int t = tid; t < nk * 32; t += blockDim.x) {
      const int c = t >> 5, ln = t & 31, base = c * CH16 + ln * 8;
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = base + j < g.K ? x_at<ACT, PRO>(a, base + j, rs) : 0.f;
      xb[(c * 2) * 32 + ln] = make_float4(v[0], v[1], v[2], v[3]);
      xb[(c * 2 + 1) * 32 + ln] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
  __syncthreads();

  const int S = split_of(nk), RG = NW / S, rg = warp / S, sp = warp % S;
  const int nquads = a.m.N >> 2;
  const int pos = (EPI == EPI_QKV) ? a.st.len[0] : 0;
  float p_dot = 0.f, p_n1 = 0.f, p_n2 = 0.f;
  float best = -INFINITY;
  int best_i = 0x7fffffff;

  for (int base_q = blockIdx.x * RG; base_q < nquads; base_q += gridDim.x * RG) {
    const int qd = base_q + rg;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (qd < nquads) {
      int rows[4];
      quad_rows<EPI>(a, qd, rows);
      if (river) {
        const float4 *xq = reinterpret_cast<const float4 *>(smem);
        const float2 *cx = reinterpret_cast<const float2 *>(smem + nk * 8 * 32 * 4);
        const RiverMat &R = a.m.r;
#pragma unroll 1
        for (int c = sp; c < nk; c += S) {
          const int k0 = c * CH4 + lane * 32;
          if (k0 >= g.Kp) continue;
          uint4 w[4];
          __half2 szh[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            w[r] = ld_stream(R.q + (size_t)rows[r] * g.words + (k0 >> 3));
            szh[r] = R.sz[(size_t)rows[r] * g.G + k0 / R.g];
          }
          u64 xp[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 f = xq[(c * 8 + i) * 32 + lane];
            xp[2 * i] = pack2(f.x, f.y);
            xp[2 * i + 1] = pack2(f.z, f.w);
          }
          const float2 cxv = cx[c * 32 + lane];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            u64 acc = 0ull;
            acc = word_fma(w[r].x, xp + 0, acc);
            acc = word_fma(w[r].y, xp + 4, acc);
            acc = word_fma(w[r].z, xp + 8, acc);
            acc = word_fma(w[r].w, xp + 12, acc);
            const float2 sz = __half22float2(szh[r]);
            v[r] = fmaf(sz.x, sum2(acc) - fmaf(sz.y, cxv.y, cxv.x), v[r]);
          }
        }
      } else {
        const float4 *xb = reinterpret_cast<const float4 *>(smem);
        u64 acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll 2
        for (int c = sp; c < nk; c += S) {
          const int k0 = c * CH16 + lane * 8;
          if (k0 >= g.K) continue;
          uint4 w[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) w[r] = ld_stream(a.m.w + (size_t)rows[r] * g.K + k0);
          const float4 f0 = xb[(c * 2) * 32 + lane], f1 = xb[(c * 2 + 1) * 32 + lane];
          const u64 x0 = pack2(f0.x, f0.y), x1 = pack2(f0.z, f0.w), x2 = pack2(f1.x, f1.y),
                    x3 = pack2(f1.z, f1.w);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            acc[r] = pair16_fma<ACT>(w[r].x, x0, acc[r]);
            acc[r] = pair16_fma<ACT>(w[r].y, x1, acc[r]);
            acc[r] = pair16_fma<ACT>(w[r].z, x2, acc[r]);
            acc[r] = pair16_fma<ACT>(w[r].w, x3, acc[r]);
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) v[r] = sum2(acc[r]);
      }
    }
    const float m = quad_reduce(v, lane);
    if ((lane & 7) == 0) red[(rg * S + sp) * 4 + (lane >> 3)] = m;
    __syncthreads();
    if (tid < RG * 4) {
      const int rgt = tid >> 2, r = tid & 3, q2 = base_q + rgt;
      if (q2 < nquads) {
        int rows[4];
        quad_rows<EPI>(a, q2, rows);
        float y = 0.f;
        for (int s2 = 0; s2 < S; ++s2) y += red[(rgt * S + s2) * 4 + r];
        if (EPI == EPI_QKV || EPI == EPI_SWIGLU) {
          // pairs (0,2) and (1,3): thread r < 2 combines rows r and r + 2
          if (r < 2) {
            float y2 = 0.f;
            for (int s2 = 0; s2 < S; ++s2) y2 += red[(rgt * S + s2) * 4 + r + 2];
            if (EPI == EPI_SWIGLU) {
              const float sg = y / (1.0f + expf(-y));
              a.out_vec[rows[r]] = round_act(sg * y2, ACT);
            } else {
              const int half = a.hd >> 1, slot = rows[r] / a.hd, i = rows[r] - slot * a.hd;
              if (slot < a.H + a.Hkv) {
                const float2 cs = a.rope_cs[(size_t)pos * half + i];
                const float o0 = y * cs.x - y2 * cs.y, o1 = y * cs.y + y2 * cs.x;
                if (slot < a.H) {
                  a.out_vec[slot * a.hd + i] = round_act(o0, ACT);
                  a.out_vec[slot * a.hd + i + half] = round_act(o1, ACT);
                } else {
                  uint16_t *kp = a.kv.base + a.kv.idx(a.layer, 0, 0, slot - a.H, pos);
                  kp[i] = f_to_act(o0, ACT);
                  kp[i + half] = f_to_act(o1, ACT);
                }
              } else {
                uint16_t *vp = a.kv.base + a.kv.idx(a.layer, 1, 0, slot - a.H - a.Hkv, pos);
                vp[i] = f_to_act(y, ACT);
                vp[i + half] = f_to_act(y2, ACT);
              }
            }
          }
        } else if (EPI == EPI_RESID) {
          a.h_out[rows[r]] = a.h_base[rows[r]] + y;
        } else if (EPI == EPI_DOWN) {
          const int u = rows[r];
          const float hn = a.h_base[u] + y, hi = a.h_in[u];
          a.h_out[u] = hn;
          if (a.dbg_h) a.dbg_h[u] = hn;
          p_dot = fmaf(hi, hn, p_dot);
          p_n1 = fmaf(hi, hi, p_n1);
          p_n2 = fmaf(hn, hn, p_n2);
        } else if (EPI == EPI_LOGITS) {
          const int u = rows[r];
          if (a.dbg_logits) a.dbg_logits[u] = y;
          if (y > best || (y == best && u < best_i)) { best = y; best_i = u; }
        }
      }
    }
    __syncthreads();
  }

  if (EPI == EPI_DOWN) {
    p_dot = block_sum(p_dot, red);
    p_n1 = block_sum(p_n1, red + 32);
    p_n2 = block_sum(p_n2, red + 64);
    if (tid == 0) {
      a.partials[blockIdx.x * 3 + 0] = p_dot;
      a.partials[blockIdx.x * 3 + 1] = p_n1;
      a.partials[blockIdx.x * 3 + 2] = p_n2;
    }
    if (!last_block(a.counter)) return;
    float t0 = 0.f, t1 = 0.f, t2 = 0.f;
    for (int i = tid; i < (int)gridDim.x; i += blockDim.x) {
      t0 += a.partials[i * 3 + 0];
      t1 += a.partials[i * 3 + 1];
      t2 += a.partials[i * 3 + 2];
    }
    t0 = block_sum(t0, red);
    t1 = block_sum(t1, red + 32);
    t2 = block_sum(t2, red + 64);
    if (tid == 0) decide_row(a.st, 0, a.layer + 1, a.L, t0, t1, t2, a.dbg_s);
  } else if (EPI == EPI_LOGITS) {
    // block argmax (lowest index on ties) over the epilogue threads
    __shared__ float bv[NW * 32];
    __shared__ int bi[NW * 32];
    bv[tid] = best;
    bi[tid] = best_i;
    __syncthreads();
    if (tid == 0) {
      float vb = bv[0];
      int ib = bi[0];
      for (int t = 1; t < RG * 4; ++t)
        if (bv[t] > vb || (bv[t] == vb && bi[t] < ib)) { vb = bv[t]; ib = bi[t]; }
      a.partials[blockIdx.x * 2] = vb;
      reinterpret_cast<int *>(a.partials)[blockIdx.x * 2 + 1] = ib;
    }
    if (!last_block(a.counter)) return;
    if (tid == 0) {
      float vb = -INFINITY;
      int ib = 0x7fffffff;
      for (int b = 0; b < (int)gridDim.x; ++b) {
        const float bvv = a.partials[b * 2];
        const int bii = reinterpret_cast<const int *>(a.partials)[b * 2 + 1];
        if (bvv > vb || (bvv == vb && bii < ib)) { vb = bvv; ib = bii; }
      }
      a.st.next_ids[0] = ib == 0x7fffffff ? 0 : ib;
      a.st.len[0] += 1;
    }
  }
}

// ------------------------------------------------------------------ launch

template <int ACT, int PRO, int EPI>
static cudaError_t launch_t(const GemvArgs &a, int max_grid, cudaStream_t s) {
  const Geo g = geo_of(a.m);
  const size_t smem = sizeof(float) * smem_floats(g);
  auto fn = k_gemv_b1<ACT, PRO, EPI>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // Quad groups per block-iteration depend on the path (the K split
  // differs): size the grid for the path with more groups, never beyond one
  // resident wave; the grid-stride loop covers the rest.
  const int nq = a.m.N / 4;
  const int nk_max = g.nk4 > g.nk16 ? g.nk4 : g.nk16;
  const int RG = NW / split_of(nk_max);
  int grid = (nq + RG - 1) / RG;
  int per_sm = 0, dev = 0, n_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, NW * 32, smem);
  if (e != cudaSuccess) return e;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (per_sm < 1) per_sm = 1;
  if (grid > per_sm * n_sm) grid = per_sm * n_sm;
  if (grid > max_grid) grid = max_grid;
  fn<<<grid, NW * 32, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gemv_b1(int act, int pro, int epi, const GemvArgs &a, int max_grid, cudaStream_t s) {
  if (a.m.N % 4) return cudaErrorInvalidValue;
#define RV_DISPATCH(PRO_, EPI_)                                                                     \
  if (pro == PRO_ && epi == EPI_)                                                                   \
    return act ? launch_t<1, PRO_, EPI_>(a, max_grid, s) : launch_t<0, PRO_, EPI_>(a, max_grid, s);
  RV_DISPATCH(PRO_NORM, EPI_QKV)
  RV_DISPATCH(PRO_VEC, EPI_RESID)
  RV_DISPATCH(PRO_NORM, EPI_SWIGLU)
  RV_DISPATCH(PRO_VEC, EPI_DOWN)
  RV_DISPATCH(PRO_NORM, EPI_LOGITS)
#undef RV_DISPATCH
  return cudaErrorInvalidValue;
}

}  // namespace rv
