// River construction and small set-up kernels.
//
// The exit layers are copies of the backbone blocks quantized to W4A16
// (aitrends.kr, exit-layer paragraph; paperlayer.ai section 4, KV-Shared Exit
// Layer: 4-bit weight-only quantization).  Round-to-nearest, asymmetric, one
// fp16 scale and one integer-valued fp16 zero point per output row and group
// of g consecutive input columns, fp32 IEEE arithmetic:
//   s = fp16_rn((max - min) / 15)      (s = 0: s = 1, z = 0)
//   z = clamp(rint(-min / s), 0, 15)
//   q = clamp(rint(w / s) + z, 0, 15)  (rint: half to even)
// Codes are packed 8 per uint32, element k of a row in bits 4*(k%8) of word
// k/8, each row padded to Kp (a multiple of 32) with zero codes; scale and
// zero of a group are stored side by side as one half2, rows of groups
// padded to a multiple of 4 pairs (left as the allocation's zeros).
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace rv {

__global__ void k_rtn(const uint16_t *W, int N, int K, int act, int g, int Kp, uint32_t *q, __half2 *sz,
                      int32_t *err) {
  const int G = (K + g - 1) / g, Gs = pad_groups(G), words = Kp >> 3;
  const long total = (long)N * G;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int n = (int)(i / G), gi = (int)(i % G);
    const int k0 = gi * g, cnt = min(g, K - k0);
    const uint16_t *w = W + (size_t)n * K + k0;
    float mn = INFINITY, mx = -INFINITY;
    for (int j = 0; j < cnt; ++j) {
      const float v = act_to_f(w[j], act);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
    const float sf = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
    __half s16 = __float2half_rn(sf);
    float s = __half2float(s16), z = 0.f;
    if (isinf(s) || isnan(s)) {
      atomicOr(err, 4);
      s16 = __float2half_rn(1.0f);
      s = 1.0f;
    } else if (s == 0.0f) {
      s16 = __float2half_rn(1.0f);
      s = 1.0f;
    } else {
      z = rintf(__fdiv_rn(-mn, s));
      z = z <= 0.0f ? 0.0f : (z > 15.0f ? 15.0f : z);
    }
    for (int kb = k0; kb < k0 + g && kb < Kp; kb += 8) {
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int k = kb + j;
        if (k < K) {
          float r = rintf(__fdiv_rn(act_to_f(W[(size_t)n * K + k], act), s)) + z;
          r = r < 0.0f ? 0.0f : (r > 15.0f ? 15.0f : r);
          word |= ((uint32_t)r) << (4 * j);
        }
      }
      q[(size_t)n * words + (kb >> 3)] = word;
    }
    sz[(size_t)n * Gs + gi] = __halves2half2(s16, __float2half_rn(z));
  }
}

// HQQ (Badri and Shaji 2023, "Half-Quadratic Quantization of Large Machine
// Learning Models"; the river quantizer of paperlayer.ai appendix A.1): the
// min/max fp16 scale, a float zero (start -mn / s) that minimises the lp norm
// (p = 0.7) of the dequantization error by half-quadratic splitting.  Per
// iteration: q = clamp(rint(w / s + z), 0, 15); w_r = (q - z) s;
// e = shrink(w - w_r) with shrink(x) = sign(x) max(|x| - |x|^(p-1) / beta, 0);
// z = mean(q - (w - e) / s); beta *= 1.01; stop once the mean |w - w_r| no
// longer falls (beta starts at 10, at most 20 iterations).  The final zero is
// rounded to fp16 and the codes are taken again with it.  Every step is one
// correctly rounded fp32 operation (no contraction), and |x|^(p-1) =
// 2^((p-1) log2 x) comes from the atanh series of log2 on the mantissa and
// the Taylor series of 2^f, so the result is the same bit for bit on any
// IEEE fp32 machine.
__device__ __forceinline__ float hqq_pow_pm1(float a) {  // a^(p - 1), p = 0.7, a > 0 finite
  uint32_t b = __float_as_uint(a);
  int ex = (int)(b >> 23);
  if (ex == 0) {  // subnormal: scale by 2^64
    b = __float_as_uint(__fmul_rn(a, 18446744073709551616.0f));
    ex = (int)(b >> 23) - 64;
  }
  ex -= 127;
  const float m = __uint_as_float((b & 0x7FFFFFu) | 0x3F800000u);
  const float u = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f)), u2 = __fmul_rn(u, u);
  float ser = 1.0f / 11.0f;
  ser = __fadd_rn(__fmul_rn(ser, u2), 1.0f / 9.0f);
  ser = __fadd_rn(__fmul_rn(ser, u2), 1.0f / 7.0f);
  ser = __fadd_rn(__fmul_rn(ser, u2), 1.0f / 5.0f);
  ser = __fadd_rn(__fmul_rn(ser, u2), 1.0f / 3.0f);
  ser = __fadd_rn(__fmul_rn(ser, u2), 1.0f);
  const float lg = __fadd_rn((float)ex, __fmul_rn(__fmul_rn(ser, u), 2.88539008f));
  const float y = __fmul_rn(-0.3f, lg);
  const float fi = floorf(y), f = __fsub_rn(y, fi);
  const float t = __fmul_rn(f, 0.693147182f);
  float ep = 1.0f / 40320.0f;
  ep = __fadd_rn(__fmul_rn(ep, t), 1.0f / 5040.0f);
  ep = __fadd_rn(__fmul_rn(ep, t), 1.0f / 720.0f);
  ep = __fadd_rn(__fmul_rn(ep, t), 1.0f / 120.0f);
  ep = __fadd_rn(__fmul_rn(ep, t), 1.0f / 24.0f);
  ep = __fadd_rn(__fmul_rn(ep, t), 1.0f / 6.0f);
  ep = __fadd_rn(__fmul_rn(ep, t), 0.5f);
  ep = __fadd_rn(__fmul_rn(ep, t), 1.0f);
  ep = __fadd_rn(__fmul_rn(ep, t), 1.0f);
  return __fmul_rn(ep, __uint_as_float((uint32_t)((int)fi + 127) << 23));
}

__device__ __forceinline__ float clamp15(float r) { return r < 0.0f ? 0.0f : (r > 15.0f ? 15.0f : r); }

__global__ void k_hqq(const uint16_t *W, int N, int K, int act, int g, int Kp, uint32_t *q, __half2 *sz, int32_t *err) {
  const int G = (K + g - 1) / g, Gs = pad_groups(G), words = Kp >> 3;
  const long total = (long)N * G;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int n = (int)(i / G), gi = (int)(i % G);
    const int k0 = gi * g, cnt = min(g, K - k0);
    const uint16_t *w = W + (size_t)n * K + k0;
    float mn = INFINITY, mx = -INFINITY;
    for (int j = 0; j < cnt; ++j) {
      const float v = act_to_f(w[j], act);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
    __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
    float s = __half2float(s16), zq = 0.0f;
    bool hqq = true;
    if (isinf(s) || isnan(s)) {
      atomicOr(err, 4);
      s16 = __float2half_rn(1.0f);
      s = 1.0f;
      hqq = false;
    } else if (s == 0.0f) {  // degenerate group: as RTN
      s16 = __float2half_rn(1.0f);
      s = 1.0f;
      hqq = false;
    }
    if (hqq) {
      float z = __fdiv_rn(-mn, s), beta = 10.0f, best = INFINITY;
      for (int it = 0; it < 20; ++it) {
        float zsum = 0.0f, esum = 0.0f;
        for (int j = 0; j < cnt; ++j) {
          const float v = act_to_f(w[j], act);
          const float r = clamp15(rintf(__fadd_rn(__fdiv_rn(v, s), z)));
          const float wr = __fmul_rn(__fsub_rn(r, z), s), res = __fsub_rn(v, wr);
          float e = 0.0f;
          if (res != 0.0f) {
            const float a = fabsf(res), sh = __fsub_rn(a, __fdiv_rn(hqq_pow_pm1(a), beta));
            if (sh > 0.0f) e = res < 0.0f ? -sh : sh;
          }
          zsum = __fadd_rn(zsum, __fsub_rn(r, __fdiv_rn(__fsub_rn(v, e), s)));
          esum = __fadd_rn(esum, fabsf(res));
        }
        z = __fdiv_rn(zsum, (float)cnt);
        beta = __fmul_rn(beta, 1.01f);
        const float e = __fdiv_rn(esum, (float)cnt);
        if (e < best) best = e;
        else break;
      }
      const __half z16 = __float2half_rn(z);
      zq = __half2float(z16);
      sz[(size_t)n * Gs + gi] = __halves2half2(s16, z16);
    } else {
      sz[(size_t)n * Gs + gi] = __halves2half2(s16, __float2half_rn(0.0f));
    }
    for (int kb = k0; kb < k0 + g && kb < Kp; kb += 8) {
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int k = kb + j;
        if (k < K) {
          const float v = act_to_f(W[(size_t)n * K + k], act);
          const float r = hqq ? clamp15(rintf(__fadd_rn(__fdiv_rn(v, s), zq))) : clamp15(rintf(v));
          word |= ((uint32_t)r) << (4 * j);
        }
      }
      q[(size_t)n * words + (kb >> 3)] = word;
    }
  }
}

cudaError_t launch_hqq_quantize(const uint16_t *W, int N, int K, int act, int g, int Kp, uint32_t *q, __half2 *sz,
                                int32_t *err, cudaStream_t s) {
  const long total = (long)N * ((K + g - 1) / g);
  const int grid = (int)((total + 127) / 128 < 65536 ? (total + 127) / 128 : 65536);
  k_hqq<<<grid, 128, 0, s>>>(W, N, K, act, g, Kp, q, sz, err);
  return cudaGetLastError();
}

cudaError_t launch_rtn_quantize(const uint16_t *W, int N, int K, int act, int g, int Kp, uint32_t *q, __half2 *sz,
                                int32_t *err, cudaStream_t s) {
  const long total = (long)N * ((K + g - 1) / g);
  const int grid = (int)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
  k_rtn<<<grid, 256, 0, s>>>(W, N, K, act, g, Kp, q, sz, err);
  return cudaGetLastError();
}

// RoPE angle table: cs[p][i] = (cos, sin)(p * theta^(-2i/hd)), computed in
// double and rounded once to fp32 (rotate-half pairing i, i + hd/2).
__global__ void k_rope_table(float2 *cs, int T, int hd, double theta) {
  const int half = hd / 2;
  const long total = (long)T * half;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int p = (int)(i / half), j = (int)(i % half);
    const double inv = pow(theta, -2.0 * (double)j / (double)hd);
    double sn, c;
    sincos((double)p * inv, &sn, &c);
    cs[i] = make_float2((float)c, (float)sn);
  }
}

cudaError_t launch_rope_table(float2 *cs, int T, int hd, double theta, cudaStream_t s) {
  const long total = (long)T * (hd / 2);
  const int grid = (int)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
  k_rope_table<<<grid, 256, 0, s>>>(cs, T, hd, theta);
  return cudaGetLastError();
}

__global__ void k_fill_u16(uint16_t *p, size_t n, uint16_t v) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) p[i] = v;
}

cudaError_t launch_fill_u16(uint16_t *p, size_t n, uint16_t v, cudaStream_t s) {
  if (!n) return cudaSuccess;
  k_fill_u16<<<4096, 256, 0, s>>>(p, n, v);
  return cudaGetLastError();
}

}  // namespace rv
