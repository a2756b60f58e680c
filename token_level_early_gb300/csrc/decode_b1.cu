// Single-row (batch 1) decode kernels of the River-LLM token-level early exit.
//
// One decode step at batch 1 is a chain of GEMV kernels per layer:
//   qkv  : RMSNorm(h) -> [q;k;v] = W_qkv x -> RoPE -> K/V into slot (l, 0, p)
//   attn : split-KV GQA decode attention (kernels in attention.cu)
//   o    : h_mid = h + W_o o
//   gu   : RMSNorm(h_mid) -> a = silu(W_g x) * (W_u x)
//   down : h_out = h_mid + W_d a, s(l) = cos(h, h_out), exit decision
// and a final LM-head GEMV with a fused greedy argmax.  Every GEMV reads the
// row's route flag on the device and streams either the 16-bit backbone
// matrix or its int4 river copy (the same kernel, the same grid), so the step
// needs no host round trip per layer and is captured once in a CUDA graph.
//
// Method: "River-LLM: Large Language Model Seamless Exit Based on KV Share",
// paperlayer.ai summary section 4 (KV-Shared Exit Layer; Inference with
// Seamless Exit) and aitrends.kr (s(l) = cos(h(l-1), h(l)) > tau; W4A16 exit
// layers copied from the backbone blocks).
#include "common.cuh"
#include "kernels.cuh"

namespace rv {

// 128-bit streaming load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 8 16-bit weights (one uint4) times 8 fp32 activations.
template <int ACT>
__device__ __forceinline__ float dot8(uint4 w, float4 xa, float4 xb, float acc) {
  if (ACT == 1) {
    acc = fmaf(__uint_as_float(w.x << 16), xa.x, acc);
    acc = fmaf(__uint_as_float(w.x & 0xFFFF0000u), xa.y, acc);
    acc = fmaf(__uint_as_float(w.y << 16), xa.z, acc);
    acc = fmaf(__uint_as_float(w.y & 0xFFFF0000u), xa.w, acc);
    acc = fmaf(__uint_as_float(w.z << 16), xb.x, acc);
    acc = fmaf(__uint_as_float(w.z & 0xFFFF0000u), xb.y, acc);
    acc = fmaf(__uint_as_float(w.w << 16), xb.z, acc);
    acc = fmaf(__uint_as_float(w.w & 0xFFFF0000u), xb.w, acc);
  } else {
    float2 f;
    f = __half22float2(*reinterpret_cast<__half2 *>(&w.x));
    acc = fmaf(f.x, xa.x, acc); acc = fmaf(f.y, xa.y, acc);
    f = __half22float2(*reinterpret_cast<__half2 *>(&w.y));
    acc = fmaf(f.x, xa.z, acc); acc = fmaf(f.y, xa.w, acc);
    f = __half22float2(*reinterpret_cast<__half2 *>(&w.z));
    acc = fmaf(f.x, xb.x, acc); acc = fmaf(f.y, xb.y, acc);
    f = __half22float2(*reinterpret_cast<__half2 *>(&w.w));
    acc = fmaf(f.x, xb.z, acc); acc = fmaf(f.y, xb.w, acc);
  }
  return acc;
}

// 32 int4 codes (one uint4, canonical nibble order) times 32 activations:
// returns sum q_k x_k.  A code becomes an exact float through the 2^23
// magic-number trick: bits 0x4B000000 | q are the float 8388608 + q.
__device__ __forceinline__ float qdot32(uint4 w, const float *x) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 xa = *reinterpret_cast<const float4 *>(x + 8 * i);
    const float4 xb = *reinterpret_cast<const float4 *>(x + 8 * i + 4);
    const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float q = __uint_as_float(0x4B000000u | ((ws[i] >> (4 * j)) & 0xFu)) - 8388608.f;
      acc = fmaf(q, xv[j], acc);
    }
  }
  return acc;
}

// Dot products of NR weight rows with the activation vector in shared memory.
// Every lane ends with the full sums.
template <int ACT, int NR>
__device__ __forceinline__ void warp_rows_dot(const Mat &m, const int *rows, int river, const float *xs,
                                              const float *xsum, float *acc) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < NR; ++r) acc[r] = 0.f;
  if (!river) {
    const int K = m.K;
#pragma unroll 4
    for (int k0 = lane * 8; k0 < K; k0 += 256) {
      const float4 xa = *reinterpret_cast<const float4 *>(xs + k0);
      const float4 xb = *reinterpret_cast<const float4 *>(xs + k0 + 4);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        uint4 w = ld_stream(m.w + (size_t)rows[r] * K + k0);
        acc[r] = dot8<ACT>(w, xa, xb, acc[r]);
      }
    }
  } else {
    const RiverMat &R = m.r;
    const int Kp = R.Kp, G = R.G, words = Kp >> 3;
#pragma unroll 2
    for (int k0 = lane * 32; k0 < Kp; k0 += 1024) {
      const int gi = k0 / R.g;
      const float xsc = xsum[k0 >> 5];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const size_t row = (size_t)rows[r];
        uint4 w = ld_stream(R.q + row * words + (k0 >> 3));
        float s = __half2float(R.s[row * G + gi]);
        float z = __half2float(R.z[row * G + gi]);
        float d = qdot32(w, xs + k0);
        acc[r] = fmaf(s, d - z * xsc, acc[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) acc[r] = warp_sum(acc[r]);
}

// Activation prologue: x = round16(RMSNorm(h) * gamma) or x = vec, zero padded
// to Kp, plus per-32-column sums of x for the int4 path.
template <int ACT, int PRO>
__device__ __forceinline__ void load_x(const GemvArgs &a, int K, int Kp, float *xs, float *xsum, float *red) {
  if (PRO == PRO_NORM) {
    float ss = 0.f;
    for (int i = threadIdx.x; i < K; i += blockDim.x) {
      float v = a.h[i];
      ss = fmaf(v, v, ss);
    }
    ss = block_sum(ss, red);
    const float r = 1.0f / sqrtf(ss / (float)K + a.eps);
    for (int i = threadIdx.x; i < Kp; i += blockDim.x)
      xs[i] = i < K ? round_act(a.h[i] * r * act_to_f(a.gamma[i], ACT), ACT) : 0.f;
  } else {
    for (int i = threadIdx.x; i < Kp; i += blockDim.x) xs[i] = i < K ? a.vec[i] : 0.f;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < (Kp >> 5); c += blockDim.x) {
    float t = 0.f;
#pragma unroll 8
    for (int j = 0; j < 32; ++j) t += xs[c * 32 + j];
    xsum[c] = t;
  }
  __syncthreads();
}

// Last-block-done: returns true in exactly one block, after every block has
// published its partials.  The counter is left at zero for the next launch.
__device__ __forceinline__ bool last_block(unsigned *counter) {
  __shared__ bool am_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned t = atomicAdd(counter, 1u);
    am_last = (t == gridDim.x - 1);
    if (am_last) *counter = 0u;
  }
  __syncthreads();
  if (am_last) __threadfence();
  return am_last;
}

template <int ACT, int PRO, int EPI, int NR>
__global__ void __launch_bounds__(256) k_gemv_b1(GemvArgs a) {
  extern __shared__ float smem[];
  const int Kp = a.m.r.Kp > 0 ? a.m.r.Kp : ((a.m.K + 31) & ~31);
  float *xs = smem;
  float *xsum = xs + Kp;
  float *red = xsum + (Kp >> 5);
  const int river = (EPI == EPI_LOGITS) ? 0 : a.st.route[0];
  load_x<ACT, PRO>(a, a.m.K, Kp, xs, xsum, red);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  float p_dot = 0.f, p_n1 = 0.f, p_n2 = 0.f;    // EPI_DOWN partials
  float best = -INFINITY;
  int best_i = 0x7fffffff;                      // EPI_LOGITS partials
  const int pos = (EPI == EPI_QKV) ? a.st.len[0] : 0;

  for (int u = blockIdx.x * nwarps + warp; u < a.units; u += gridDim.x * nwarps) {
    int rows[NR];
    if (EPI == EPI_QKV) {
      const int half = a.hd >> 1, slot = u / half, r = u - slot * half;
      rows[0] = slot * a.hd + r;
      if (NR > 1) rows[NR - 1] = rows[0] + half;
    } else if (EPI == EPI_SWIGLU) {
      rows[0] = u;
      if (NR > 1) rows[NR - 1] = u + (a.m.N >> 1);
    } else {
      rows[0] = u;
    }
    float acc[NR];
    warp_rows_dot<ACT, NR>(a.m, rows, river, xs, xsum, acc);
    if (lane != 0) continue;
    if (EPI == EPI_QKV) {
      const int half = a.hd >> 1, slot = u / half, r = u - slot * half;
      const float y0 = acc[0], y1 = acc[NR - 1];
      if (slot < a.H + a.Hkv) {  // q or k head: rotate the pair (r, r + hd/2)
        const float2 cs = a.rope_cs[(size_t)pos * half + r];
        const float o0 = y0 * cs.x - y1 * cs.y, o1 = y0 * cs.y + y1 * cs.x;
        if (slot < a.H) {
          a.out_vec[slot * a.hd + r] = round_act(o0, ACT);
          a.out_vec[slot * a.hd + r + half] = round_act(o1, ACT);
        } else {
          uint16_t *k = a.kv.base + a.kv.idx(a.layer, 0, 0, slot - a.H, pos);
          k[r] = f_to_act(o0, ACT);
          k[r + half] = f_to_act(o1, ACT);
        }
      } else {
        uint16_t *v = a.kv.base + a.kv.idx(a.layer, 1, 0, slot - a.H - a.Hkv, pos);
        v[r] = f_to_act(y0, ACT);
        v[r + half] = f_to_act(y1, ACT);
      }
    } else if (EPI == EPI_SWIGLU) {
      const float g = acc[0], up = acc[NR - 1];
      const float sg = g / (1.0f + expf(-g));
      a.out_vec[u] = round_act(sg * up, ACT);
    } else if (EPI == EPI_RESID) {
      a.h_out[u] = a.h_base[u] + acc[0];
    } else if (EPI == EPI_DOWN) {
      const float hn = a.h_base[u] + acc[0], hi = a.h_in[u];
      a.h_out[u] = hn;
      if (a.dbg_h) a.dbg_h[u] = hn;
      p_dot = fmaf(hi, hn, p_dot);
      p_n1 = fmaf(hi, hi, p_n1);
      p_n2 = fmaf(hn, hn, p_n2);
    } else if (EPI == EPI_LOGITS) {
      const float v = acc[0];
      if (a.dbg_logits) a.dbg_logits[u] = v;
      if (v > best || (v == best && u < best_i)) { best = v; best_i = u; }
    }
  }

  if (EPI == EPI_DOWN) {
    p_dot = block_sum(p_dot, red);
    p_n1 = block_sum(p_n1, red + 32);
    p_n2 = block_sum(p_n2, red + 64);
    if (threadIdx.x == 0) {
      a.partials[blockIdx.x * 3 + 0] = p_dot;
      a.partials[blockIdx.x * 3 + 1] = p_n1;
      a.partials[blockIdx.x * 3 + 2] = p_n2;
    }
    if (!last_block(a.counter)) return;
    float t0 = 0.f, t1 = 0.f, t2 = 0.f;
    for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x) {
      t0 += a.partials[i * 3 + 0];
      t1 += a.partials[i * 3 + 1];
      t2 += a.partials[i * 3 + 2];
    }
    t0 = block_sum(t0, red);
    t1 = block_sum(t1, red + 32);
    t2 = block_sum(t2, red + 64);
    if (threadIdx.x == 0) decide_row(a.st, 0, a.layer + 1, a.L, t0, t1, t2, a.dbg_s);
  } else if (EPI == EPI_LOGITS) {
    // block argmax, lowest index on ties
    __shared__ float bv[32];
    __shared__ int bi[32];
    if (lane == 0) { bv[warp] = best; bi[warp] = best_i; }
    __syncthreads();
    if (threadIdx.x == 0) {
      float v = bv[0];
      int i0 = bi[0];
      for (int w = 1; w < nwarps; ++w)
        if (bv[w] > v || (bv[w] == v && bi[w] < i0)) { v = bv[w]; i0 = bi[w]; }
      a.partials[blockIdx.x * 2] = v;
      reinterpret_cast<int *>(a.partials)[blockIdx.x * 2 + 1] = i0;
    }
    if (!last_block(a.counter)) return;
    if (threadIdx.x == 0) {
      float v = -INFINITY;
      int i0 = 0x7fffffff;
      for (int b = 0; b < (int)gridDim.x; ++b) {
        float bvv = a.partials[b * 2];
        int bii = reinterpret_cast<const int *>(a.partials)[b * 2 + 1];
        if (bvv > v || (bvv == v && bii < i0)) { v = bvv; i0 = bii; }
      }
      if (i0 == 0x7fffffff) i0 = 0;
      a.st.next_ids[0] = i0;
      a.st.len[0] += 1;
    }
  }
}

// ------------------------------------------------------------------ launch

template <int ACT, int PRO, int EPI, int NR>
static cudaError_t launch_t(const GemvArgs &a, int grid, cudaStream_t s) {
  const int Kp = a.m.r.Kp > 0 ? a.m.r.Kp : ((a.m.K + 31) & ~31);
  const size_t smem = sizeof(float) * ((size_t)Kp + (Kp >> 5) + 128);
  auto fn = k_gemv_b1<ACT, PRO, EPI, NR>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // never more blocks than can be resident at once (the grid-stride loop
  // covers the rest), so the last-block reductions see one wave
  int per_sm = 0, dev = 0, n_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 256, smem);
  if (e != cudaSuccess) return e;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (per_sm < 1) per_sm = 1;
  if (grid > per_sm * n_sm) grid = per_sm * n_sm;
  fn<<<grid, 256, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gemv_b1(int act, int pro, int epi, const GemvArgs &a, int grid, cudaStream_t s) {
#define RV_DISPATCH(PRO_, EPI_, NR_)                                                           \
  if (pro == PRO_ && epi == EPI_)                                                              \
    return act ? launch_t<1, PRO_, EPI_, NR_>(a, grid, s) : launch_t<0, PRO_, EPI_, NR_>(a, grid, s);
  RV_DISPATCH(PRO_NORM, EPI_QKV, 2)
  RV_DISPATCH(PRO_VEC, EPI_RESID, 1)
  RV_DISPATCH(PRO_NORM, EPI_SWIGLU, 2)
  RV_DISPATCH(PRO_VEC, EPI_DOWN, 1)
  RV_DISPATCH(PRO_NORM, EPI_LOGITS, 1)
#undef RV_DISPATCH
  return cudaErrorInvalidValue;
}

}  // namespace rv
