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
// zero of a group are stored side by side as one half2.
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace rv {

__global__ void k_rtn(const uint16_t *W, int N, int K, int act, int g, int Kp, uint32_t *q, __half2 *sz,
                      int32_t *err) {
  const int G = (K + g - 1) / g, words = Kp >> 3;
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
    sz[(size_t)n * G + gi] = __halves2half2(s16, __float2half_rn(z));
  }
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
