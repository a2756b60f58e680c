// Device helpers and data layouts shared by the River-LLM CUDA kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define RV_WARP 32

namespace rv {

// ------------------------------------------------------------------ 16-bit
// act = 0: fp16, act = 1: bf16.  Values that enter a matrix product are kept
// as fp32 numbers that are exactly representable in the 16-bit type.

__device__ __forceinline__ float act_to_f(uint16_t b, int act) {
  if (act) return __uint_as_float(((uint32_t)b) << 16);
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint16_t f_to_act(float x, int act) {
  if (act) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  return __half_as_ushort(__float2half_rn(x));
}

__device__ __forceinline__ float round_act(float x, int act) { return act_to_f(f_to_act(x, act), act); }

// ------------------------------------------------------------------ launch chaining
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while its predecessor drains;
// pdl_wait() blocks until the predecessor grid has completed and its writes
// are visible, pdl_trigger() lets the next kernel in the chain launch.  Both
// are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with the programmatic stream-serialization attribute when pdl != 0.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*fn)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int pdl,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, fn, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ------------------------------------------------------------------ reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over the block; every thread gets the result.  scratch >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float *scratch) {
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch[wid] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += scratch[i];  // fixed order: deterministic
  return t;
}

// Three block sums with one pair of barriers; scratch holds 3 x 32 floats.
__device__ __forceinline__ float3 block_sum3(float a, float b, float c, float *scratch) {
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  c = warp_sum(c);
  __syncthreads();
  if (lane == 0) {
    scratch[wid] = a;
    scratch[32 + wid] = b;
    scratch[64 + wid] = c;
  }
  __syncthreads();
  float3 t = make_float3(0.f, 0.f, 0.f);
  for (int i = 0; i < nw; ++i) {  // fixed order: deterministic
    t.x += scratch[i];
    t.y += scratch[32 + i];
    t.z += scratch[64 + i];
  }
  return t;
}

// ------------------------------------------------------------------ weights

// River copy of one projection in the device layout: canonical packing with
// the row stride padded to Kp (a multiple of 32) nibbles; fp16 scale and zero
// per (row, group of g columns), interleaved as one half2 (scale, zero), each
// row of groups padded to Gs = a multiple of 4 (16 bytes) with zero pairs.
struct RiverMat {
  const uint32_t *q;   // [N][Kp/8]
  const __half2 *sz;   // [N][Gs]
  int Kp, G, g, Gs;
};
__host__ __device__ __forceinline__ int pad_groups(int G) { return (G + 3) & ~3; }

// One projection: backbone 16-bit matrix [N][K] and its river copy.
struct Mat {
  const uint16_t *w;
  RiverMat r;
  int N, K;
};

// Per-step device state (all pointers into one device block).
struct StepState {
  const int32_t *tokens;  // [B]
  const int32_t *forced;  // [B] forced exit layers (mode 1)
  int32_t *route;         // [B] 0 backbone, 1 river
  int32_t *exit_layer;    // [B]
  int32_t *len;           // [B] cached positions (position of the token being decoded)
  int32_t *next_ids;      // [B]
  const float *tau;       // scalar
  const int32_t *mode;    // scalar: 0 tau rule, 1 forced exits
  const int32_t *entry;   // scalar: first layer eligible for the tau rule
  const int32_t *cap;     // scalar: last backbone layer kept on the device (L = all); a row still
                          // in the backbone after layer cap continues in the river
  int32_t *err;           // scalar error flags (bit 0 token, bit 1 forced value, bit 2 quant)
};

// KV cache geometry: [L][2][max_batch][Hkv][max_seq][hd] 16-bit.
struct KVGeom {
  uint16_t *base;
  int B, Hkv, T, hd;
  __host__ __device__ size_t idx(int l, int kv, int b, int g, int p) const {
    return ((((size_t)l * 2 + kv) * B + b) * Hkv + g) * (size_t)T * hd + (size_t)p * hd;
  }
};

// Relaxed gpu-scope load (a value another kernel may be updating).
__device__ __forceinline__ int ld_relaxed_i32(const int32_t *p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// cp.async: 16- and 4-byte global -> shared copies, commit groups and waits.
__device__ __forceinline__ void cp16(void *dst, const void *src) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(void *dst, const void *src) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void cp16s(unsigned dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4s(unsigned dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// c + lo16(a) * lo16(b) and c + hi16(a) * hi16(b) with 16-bit operands of
// type ACT (1 = bf16, 0 = fp16) and an fp32 accumulator.
template <int ACT>
__device__ __forceinline__ float fma_lo16(uint32_t a, uint32_t b, float c) {
  float d;
  if (ACT == 1)
    asm("{.reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2; fma.rn.f32.bf16 %0, al, bl, %3;}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
  else
    asm("{.reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2; fma.rn.f32.f16 %0, al, bl, %3;}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}
template <int ACT>
__device__ __forceinline__ float fma_hi16(uint32_t a, uint32_t b, float c) {
  float d;
  if (ACT == 1)
    asm("{.reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2; fma.rn.f32.bf16 %0, ah, bh, %3;}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
  else
    asm("{.reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2; fma.rn.f32.f16 %0, ah, bh, %3;}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

}  // namespace rv
