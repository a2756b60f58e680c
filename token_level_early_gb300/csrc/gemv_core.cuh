// Batch-1 GEMV core shared by the per-kernel decode chain (decode_b1.cu) and
// the persistent decode-step kernel (mega.cu).  Internal header.
//
// A warp owns 4 output rows (a "quad") and, when a matrix has too few quads to
// fill the GPU, one of S splits of its K chunks (S warps of a block per quad).
// Weights stream into a per-warp ring of shared-memory stages by cp.async
// (16-byte pieces, a coalesced 512-byte run per row and stage), NST - 1 work
// items ahead of the math.  A lane's activation chunk is read from shared
// memory and serves the 4 rows.  Partial sums are reduced across lanes by a
// transpose-reduce and, for S > 1, across the splits through shared memory;
// the epilogue runs in the warp that owns the quad.
//
// int4 inner loop.  A code q becomes the float 1 + q/16 (nibble rotated into
// mantissa bits 19..22 and the exponent of 1.0 OR-ed in) or 1 + q/256 (bits
// 15..18): one funnel rotate per pair of codes and one LOP3 per code.  The
// matching activation is pre-scaled by 16 or 256, so (1 + q/16)(16 x) =
// 16 x + q x, and the constant sum of the pre-scaled activations is removed
// once per 32 codes.  Products and sums are fp32 (packed fma.rn.f32x2), the
// products exact.  Per 32 codes of a row: sum w x = s (sum q x - z sum x).
#pragma once

#include "common.cuh"
#include "kernels.cuh"

namespace rv {

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
// pairs (0,7), (2,1), (4,3), (6,5).  Shifts bring each pair to mantissa bits
// 19..22 (even) and 15..18 (odd): left shifts by 3 and 11 for (4,3) and
// (2,1), a right shift by 5 for (6,5), and for (0,7) a left shift by 19 and a
// right shift by 13.  Left shifts and the high half of a multiply (the right
// shifts) run on the FMA pipe, leaving one LOP3 per code on the ALU pipe.
__device__ __forceinline__ u64 word_fma(uint32_t w, const u64 *xp, u64 acc) {
#ifdef RV_UNPACK_ROTATE
  const int rot[4] = {19, 11, 3, 27};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t u = rotl(w, rot[p]);
    const uint32_t fh = (u & 0x00780000u) | 0x3F800000u;  // 1 + q/16
    const uint32_t fl = (u & 0x00078000u) | 0x3F800000u;  // 1 + q/256
    acc = ffma2(((u64)fl << 32) | fh, xp[p], acc);
  }
#else
  const uint32_t u0h = w << 19, u0l = __umulhi(w, 1u << 19);  // nibble 0 -> 19..22, 7 -> 15..18
  const uint32_t u1 = w << 11;                                // nibbles 2, 1
  const uint32_t u2 = w << 3;                                 // nibbles 4, 3
  const uint32_t u3 = __umulhi(w, 1u << 27);                  // nibbles 6, 5
  const uint32_t hs[4] = {u0h, u1, u2, u3}, ls[4] = {u0l, u1, u2, u3};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t fh = (hs[p] & 0x00780000u) | 0x3F800000u;  // 1 + q/16
    const uint32_t fl = (ls[p] & 0x00078000u) | 0x3F800000u;  // 1 + q/256
    acc = ffma2(((u64)fl << 32) | fh, xp[p], acc);
  }
#endif
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

// Weight staging: every warp owns a ring of NST stages; a stage holds one
// work item (one K chunk of the warp's 4 rows: 32 lanes x 16 bytes per row,
// plus the rows' (scale, zero) words on the int4 path), copied by cp.async.
constexpr int NST = 4;
constexpr int STAGE_W = 4 * 32 * 16;
constexpr int STAGE_S = 4 * 32 * 4;
constexpr int STAGE = STAGE_W + STAGE_S;

// Shared memory (bytes): activations in the lane layout of the larger path,
// 256 floats of reduction scratch, then the warps' staging rings.
__host__ __device__ __forceinline__ size_t x_floats(const Geo &g) {
  const size_t river = (size_t)g.nk4 * (8 * 32 * 4 + 32 * 2);
  const size_t b16 = (size_t)g.nk16 * (2 * 32 * 4);
  return river > b16 ? river : b16;
}
__host__ __device__ __forceinline__ size_t smem_bytes(const Geo &g, int nwarp) {
  return sizeof(float) * (x_floats(g) + 256) + (size_t)nwarp * NST * STAGE;
}

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

// Eight consecutive activations x[k0..k0+8) (k0 a multiple of 8, all < K).
template <int ACT, int PRO>
__device__ __forceinline__ void load_x8(const GemvArgs &a, int k0, float r, float *x) {
  // activations come from other blocks of the same step: read them at L2
  const float4 *src = reinterpret_cast<const float4 *>((PRO == PRO_NORM ? a.h : a.vec) + k0);
  const float4 u0 = __ldcg(src), u1 = __ldcg(src + 1);
  x[0] = u0.x; x[1] = u0.y; x[2] = u0.z; x[3] = u0.w;
  x[4] = u1.x; x[5] = u1.y; x[6] = u1.z; x[7] = u1.w;
  if (PRO == PRO_NORM) {
    const uint4 gw = *reinterpret_cast<const uint4 *>(a.gamma + k0);
    const uint16_t *gp = reinterpret_cast<const uint16_t *>(&gw);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = round_act(x[j] * r * act_to_f(gp[j], ACT), ACT);
  }
}

// K splits per row quad: the smallest power of two (<= 8, <= chunks) that
// gives at least 4096 (quad, split) tasks, so small matrices still fill the
// GPU while large ones run without cross-warp reductions.
__host__ __device__ __forceinline__ int splits_for(int nquads, int nk) {
  int S = 1;
  while (S < 8 && 2 * S <= nk && nquads * S < 4096) S *= 2;
  return S;
}

// The warp's stream of work items (quad, chunk) in consumption order: quads
// bq + rg for bq = bid * RG, + nblocks * RG, ...; chunks sp, sp + S, ...
struct ItemStream {
  int bq, c, step;
};

template <int EPI>
__device__ __forceinline__ void issue_item(const GemvArgs &a, const Geo &g, int river, int rg, int nquads, int nk,
                                           int S, int sp, int RG, ItemStream &is, char *stage, int lane) {
  if (is.bq + rg < nquads) {
    int rows[4];
    quad_rows<EPI>(a, is.bq + rg, rows);
    if (river) {
      const int k0 = is.c * CH4 + lane * 32;
      if (k0 < g.Kp) {
        const RiverMat &R = a.m.r;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          cp16(stage + (r * 32 + lane) * 16, R.q + (size_t)rows[r] * g.words + (k0 >> 3));
          cp4(stage + STAGE_W + (r * 32 + lane) * 4, R.sz + (size_t)rows[r] * g.G + k0 / R.g);
        }
      }
    } else {
      const int k0 = is.c * CH16 + lane * 8;
      if (k0 < g.K) {
#pragma unroll
        for (int r = 0; r < 4; ++r) cp16(stage + (r * 32 + lane) * 16, a.m.w + (size_t)rows[r] * g.K + k0);
      }
    }
    is.c += S;
    if (is.c >= nk) {
      is.c = sp;
      is.bq += is.step;
    }
  }
  cp_commit();  // one group per item slot, empty once the stream has ended
}


// Per-thread results of a GEMV phase that the caller combines across blocks:
// the s(l) sums of the down projection, the argmax candidate of the LM head.
struct PhaseOut {
  float p_dot, p_n1, p_n2, best;
  int best_i;
};

struct PhaseGeo {
  Geo g;
  int river, nk, S, RG, rg, sp, nquads;
};

template <int NWARP>
__device__ __forceinline__ PhaseGeo phase_geo(const GemvArgs &a, int river) {
  PhaseGeo p;
  p.g = geo_of(a.m);
  p.river = river;
  p.nk = river ? p.g.nk4 : p.g.nk16;
  p.S = river ? a.s4 : a.s16;
  p.RG = NWARP / p.S;
  const int warp = threadIdx.x >> 5;
  p.rg = warp / p.S;
  p.sp = warp % p.S;
  p.nquads = a.m.N >> 2;
  return p;
}

// Start a GEMV phase: issue the warp's first NST - 1 weight items into its
// ring.  Touches only weights (and the river flag the caller passes), so it
// may run before the phase's activations exist.
template <int NWARP, int EPI>
__device__ __forceinline__ ItemStream gemv_begin(const GemvArgs &a, int river, char *ring, int bid, int nblocks) {
  const PhaseGeo p = phase_geo<NWARP>(a, river);
  const int lane = threadIdx.x & 31;
  ItemStream is{bid * p.RG, p.sp, nblocks * p.RG};
#pragma unroll
  for (int i = 0; i < NST - 1; ++i)
    issue_item<EPI>(a, p.g, river, p.rg, p.nquads, p.nk, p.S, p.sp, p.RG, is, ring + i * STAGE, lane);
  return is;
}

// Run a GEMV phase whose first items gemv_begin issued: activation prologue
// (x = round16(RMSNorm(h) * gamma) or x = vec, into the lane layout in xs),
// the quad loop over the ring, and the epilogue in the owning warp.
// scratch: 256 floats (cross-warp partials, block sums).
template <int NWARP, int ACT, int PRO, int EPI>
__device__ __forceinline__ PhaseOut gemv_run(const GemvArgs &a, int river, float *xs, float *scratch, char *ring,
                                             ItemStream is, int bid, int nblocks) {
  const PhaseGeo p = phase_geo<NWARP>(a, river);
  const Geo &g = p.g;
  const int nk = p.nk, S = p.S, RG = p.RG, rg = p.rg, sp = p.sp, nquads = p.nquads;
  const int tid = threadIdx.x, lane = tid & 31;
  float *red = scratch;         // [2][NWARP * 4]: cross-warp partials, double-buffered
  float *bsum = scratch + 128;  // block_sum scratch (3 x 32)

  float rs = 0.f;
  if (PRO == PRO_NORM) {
    float ss = 0.f;
    for (int i = tid * 4; i < g.K; i += blockDim.x * 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.h + i));
      ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
    }
    ss = block_sum(ss, bsum);
    rs = 1.0f / sqrtf(ss / (float)g.K + a.eps);
  }
  if (river) {
    float4 *xq = reinterpret_cast<float4 *>(xs);                    // [nk][8][32]
    float2 *cx = reinterpret_cast<float2 *>(xs + nk * 8 * 32 * 4);  // [nk][32] (C, X)
    for (int t = tid; t < nk * 32; t += blockDim.x) {
      const int c = t >> 5, ln = t & 31, base = c * CH4 + ln * 32;
      float C = 0.f, X = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (base + 8 * i < g.K) load_x8<ACT, PRO>(a, base + 8 * i, rs, x);
        // pairs (even, odd) = (0,7), (2,1), (4,3), (6,5), scaled by 16 and 256
        const float e0 = 16.f * x[0], o0 = 256.f * x[7], e1 = 16.f * x[2], o1 = 256.f * x[1];
        const float e2 = 16.f * x[4], o2 = 256.f * x[3], e3 = 16.f * x[6], o3 = 256.f * x[5];
        xq[(c * 8 + 2 * i) * 32 + ln] = make_float4(e0, o0, e1, o1);
        xq[(c * 8 + 2 * i + 1) * 32 + ln] = make_float4(e2, o2, e3, o3);
        C += ((e0 + o0) + (e1 + o1)) + ((e2 + o2) + (e3 + o3));
        X += ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
      }
      cx[c * 32 + ln] = make_float2(C, X);
    }
  } else {
    float4 *xb = reinterpret_cast<float4 *>(xs);  // [nk][2][32]
    for (int t = tid; t < nk * 32; t += blockDim.x) {
      const int c = t >> 5, ln = t & 31, base = c * CH16 + ln * 8;
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (base < g.K) load_x8<ACT, PRO>(a, base, rs, x);
      xb[(c * 2) * 32 + ln] = make_float4(x[0], x[1], x[2], x[3]);
      xb[(c * 2 + 1) * 32 + ln] = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
  __syncthreads();

  const int pos = (EPI == EPI_QKV) ? a.st.len[0] : 0;
  PhaseOut out{0.f, 0.f, 0.f, -INFINITY, 0x7fffffff};
  int parity = 0, t = 0;

  for (int base_q = bid * RG; base_q < nquads; base_q += nblocks * RG, parity ^= 1) {
    const int qd = base_q + rg;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    int rows[4] = {0, 0, 0, 0};
    if (qd < nquads) {
      quad_rows<EPI>(a, qd, rows);
      u64 acc[4] = {0ull, 0ull, 0ull, 0ull};
      for (int c = sp; c < nk; c += S, ++t) {
        cp_wait<NST - 2>();  // this lane's copies of item t have landed
        issue_item<EPI>(a, g, river, rg, nquads, nk, S, sp, RG, is, ring + ((t + NST - 1) % NST) * STAGE, lane);
        const char *stg = ring + (t % NST) * STAGE;
        const uint4 *sw = reinterpret_cast<const uint4 *>(stg);
        if (river) {
          const int k0 = c * CH4 + lane * 32;
          if (k0 >= g.Kp) continue;
          const float4 *xq = reinterpret_cast<const float4 *>(xs);
          const float2 cxv = reinterpret_cast<const float2 *>(xs + nk * 8 * 32 * 4)[c * 32 + lane];
          const __half2 *ss = reinterpret_cast<const __half2 *>(stg + STAGE_W);
          u64 xp[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 f = xq[(c * 8 + i) * 32 + lane];
            xp[2 * i] = pack2(f.x, f.y);
            xp[2 * i + 1] = pack2(f.z, f.w);
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const uint4 w = sw[r * 32 + lane];
            u64 ac = word_fma(w.x, xp + 0, 0ull);
            ac = word_fma(w.y, xp + 4, ac);
            u64 ad = word_fma(w.z, xp + 8, 0ull);
            ad = word_fma(w.w, xp + 12, ad);
            const float2 sz = __half22float2(ss[r * 32 + lane]);
            v[r] = fmaf(sz.x, (sum2(ac) + sum2(ad)) - fmaf(sz.y, cxv.y, cxv.x), v[r]);
          }
        } else {
          const int k0 = c * CH16 + lane * 8;
          if (k0 >= g.K) continue;
          const float4 *xb = reinterpret_cast<const float4 *>(xs);
          const float4 f0 = xb[(c * 2) * 32 + lane], f1 = xb[(c * 2 + 1) * 32 + lane];
          const u64 x0 = pack2(f0.x, f0.y), x1 = pack2(f0.z, f0.w), x2 = pack2(f1.x, f1.y), x3 = pack2(f1.z, f1.w);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const uint4 w = sw[r * 32 + lane];
            acc[r] = pair16_fma<ACT>(w.x, x0, acc[r]);
            acc[r] = pair16_fma<ACT>(w.y, x1, acc[r]);
            acc[r] = pair16_fma<ACT>(w.z, x2, acc[r]);
            acc[r] = pair16_fma<ACT>(w.w, x3, acc[r]);
          }
        }
      }
      if (!river) {
#pragma unroll
        for (int r = 0; r < 4; ++r) v[r] = sum2(acc[r]);
      }
    }
    // row r of the quad ends in lane 8 r of every warp of the quad's group
    float m = quad_reduce(v, lane);
    if (S > 1) {
      float *rb = red + parity * (NWARP * 4);
      if ((lane & 7) == 0) rb[(rg * S + sp) * 4 + (lane >> 3)] = m;
      __syncthreads();
      if (sp == 0 && (lane & 7) == 0) {
        float tt = 0.f;
        for (int s2 = 0; s2 < S; ++s2) tt += rb[(rg * S + s2) * 4 + (lane >> 3)];
        m = tt;
      }
    }
    if (sp != 0 || qd >= nquads) continue;
    const int r = lane >> 3;
    const int row_r = r == 0 ? rows[0] : r == 1 ? rows[1] : r == 2 ? rows[2] : rows[3];
    // ---- epilogue in the owning warp: lane 8 r holds row r
    if (EPI == EPI_QKV || EPI == EPI_SWIGLU) {
      const float y2 = __shfl_down_sync(0xffffffffu, m, 16);  // rows 2, 3 -> lanes 0, 8
      if ((lane & 7) == 0 && r < 2) {
        const float y = m;
        if (EPI == EPI_SWIGLU) {
          const float sg = y / (1.0f + expf(-y));
          a.out_vec[row_r] = round_act(sg * y2, ACT);
        } else {
          const int half = a.hd >> 1, slot = row_r / a.hd, i = row_r - slot * a.hd;
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
    } else if ((lane & 7) == 0) {
      const int u = row_r;
      if (EPI == EPI_RESID) {
        a.h_out[u] = __ldcg(a.h_base + u) + m;
      } else if (EPI == EPI_DOWN) {
        const float hn = __ldcg(a.h_base + u) + m, hi = __ldcg(a.h_in + u);
        a.h_out[u] = hn;
        if (a.dbg_h) a.dbg_h[u] = hn;
        out.p_dot = fmaf(hi, hn, out.p_dot);
        out.p_n1 = fmaf(hi, hi, out.p_n1);
        out.p_n2 = fmaf(hn, hn, out.p_n2);
      } else if (EPI == EPI_LOGITS) {
        if (a.dbg_logits) a.dbg_logits[u] = m;
        if (m > out.best || (m == out.best && u < out.best_i)) { out.best = m; out.best_i = u; }
      }
    }
  }
  cp_wait<0>();  // no copy outlives the phase
  return out;
}

}  // namespace rv
