// Batch-1 GEMV core of the per-kernel decode chain (decode_b1.cu).
// Internal header.
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
// Activations are staged as 16-bit values (exact: every GEMV input is
// rounded to the model's 16-bit type) and multiplied by mixed-precision FMAs
// (16-bit operands, fp32 accumulator, exact products).  16-bit path: the two
// halves of a weight word against the two halves of an activation word.
//
// int4 inner loop.  One LOP3 turns two codes of a word into a pair of 16-bit
// floats with the code in the low mantissa bits: bf16 128 + q (mask the
// nibbles at bits 0..3 and 16..19, OR in the bits of 128.0), or fp16 1 + q/16
// (nibbles shifted to bits 6..9 and 22..25, OR in 1.0).  Each code then takes
// one mixed-precision FMA (16-bit operands, fp32 accumulator): the product of
// the code value and a 16-bit activation is exact and only the fp32 sums
// round.  Per lane run of 32 codes, with X the sum of its activations:
//   bf16: sum (q - z) x = acc - (128 + z) X;   fp16: = 16 acc - (16 + z) X,
// and the run adds s times that to the row.
#pragma once

#include "common.cuh"
#include "kernels.cuh"

namespace rv {

constexpr int CH4 = 1024;  // int4 chunk: 32 lanes x 32 codes
constexpr int CH16 = 256;  // 16-bit chunk: 32 lanes x 8 values


// d = (a & m) | c in one instruction (the compiler splits the two-constant
// form into two).
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
  return d;
}

// Code extraction constants (mask, OR-ed bits) by activation type.
template <int ACT>
struct CodeBits {
  static constexpr uint32_t mask = ACT == 1 ? 0x000F000Fu : 0x03C003C0u;
  static constexpr uint32_t one = ACT == 1 ? 0x43004300u : 0x3C003C00u;
  static constexpr float A = ACT == 1 ? 1.f : 16.f;    // sum (q - z) x = A acc - (B + z) X
  static constexpr float B = ACT == 1 ? 128.f : 16.f;
};

// One word of 8 codes (canonical nibble order: code i at bits 4i..4i+3)
// against its activation pairs xr[p] = (x[p], x[p + 4]) as 16-bit pairs.
// a0 collects codes 0..3, a1 codes 4..7.
template <int ACT>
__device__ __forceinline__ void word_mix(uint32_t w, const uint32_t *xr, float &a0, float &a1, uint32_t m,
                                         uint32_t one) {
  uint32_t u0, u1, u2, u3;
  if (ACT == 1) {
    u0 = w; u1 = w >> 4; u2 = w >> 8; u3 = w >> 12;
  } else {
    u0 = w << 6; u1 = w << 2; u2 = w >> 2; u3 = w >> 6;
  }
  const uint32_t c0 = lop3_and_or(u0, m, one), c1 = lop3_and_or(u1, m, one);
  const uint32_t c2 = lop3_and_or(u2, m, one), c3 = lop3_and_or(u3, m, one);
  a0 = fma_lo16<ACT>(c0, xr[0], a0); a1 = fma_hi16<ACT>(c0, xr[0], a1);
  a0 = fma_lo16<ACT>(c1, xr[1], a0); a1 = fma_hi16<ACT>(c1, xr[1], a1);
  a0 = fma_lo16<ACT>(c2, xr[2], a0); a1 = fma_hi16<ACT>(c2, xr[2], a1);
  a0 = fma_lo16<ACT>(c3, xr[3], a0); a1 = fma_hi16<ACT>(c3, xr[3], a1);
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

// Largest value, lowest index on ties, over the block (all threads return
// the block's pair; sv, si: one slot per warp).
__device__ __forceinline__ void block_argmax(float &v, int &i, float *sv, int *si) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();  // the slots may still be read from an earlier call
  if (lane == 0) {
    sv[warp] = v;
    si[warp] = i;
  }
  __syncthreads();
  v = sv[0];
  i = si[0];
  for (int w = 1; w < nw; ++w)
    if (sv[w] > v || (sv[w] == v && si[w] < i)) { v = sv[w]; i = si[w]; }
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
  int K, Kp, nk4, nk16, words, G, Gs;
  int gpc;  // groups per int4 chunk when the group size divides the chunk, else 0
  int spr;  // 16-byte pieces of one row's (scale, zero) words per chunk, when
            // they can be copied as such (gpc a multiple of 4; rows of groups
            // are padded to 16 bytes); else 0 and every lane copies its own
            // group's word
};

__host__ __device__ __forceinline__ Geo geo_of(const Mat &m) {
  Geo g;
  g.K = m.K;
  g.Kp = m.r.Kp > 0 ? m.r.Kp : ((m.K + 31) & ~31);
  g.nk4 = (g.Kp + CH4 - 1) / CH4;
  g.nk16 = (m.K + CH16 - 1) / CH16;
  g.words = g.Kp >> 3;
  g.G = m.r.G;
  g.Gs = m.r.Gs;
  g.gpc = (m.r.g > 0 && CH4 % m.r.g == 0) ? CH4 / m.r.g : 0;
  g.spr = (g.gpc >= 4 && g.gpc % 4 == 0) ? g.gpc / 4 : 0;
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
  const size_t river = (size_t)g.nk4 * (4 * 32 * 4 + 32);
  const size_t b16 = (size_t)g.nk16 * (32 * 4);
  return river > b16 ? river : b16;
}
__host__ __device__ __forceinline__ size_t smem_bytes(const Geo &g, int nwarp) {
  return sizeof(float) * (x_floats(g) + 256) + (size_t)nwarp * NST * STAGE;
}

// Activation prologue: x = round16(RMSNorm(h) * gamma) (PRO_NORM, r the
// reciprocal RMS) or x = vec, staged in shared memory as 16-bit pairs in the
// layout of the path.  Thread t of a pass handles the 8 activations
// x[8t..8t+8), so a warp's loads cover 1 KB of contiguous fp32.
//   16-bit path: word t (= chunk c * 32 + lane) holds x[8t..8t+8) as 4 pairs.
//   int4 path:   chunk c, lane ln, word j of the lane's 32-code run, t =
//                c * 128 + ln * 4 + j: the pairs (x[8t+p], x[8t+p+4]); and per
//                lane run the sum X of its 32 activations (4 words, summed by
//                a 4-lane shuffle).
// Word counts of the two layouts (multiples of 32, so warps stay converged).
__host__ __device__ __forceinline__ int x_words(const Geo &g, int river) { return river ? g.nk4 * 128 : g.nk16 * 32; }

// Store word t of x (8 values, already 16-bit-rounded where required).
template <int ACT>
__device__ __forceinline__ void store_xword(int river, int nk, int t, const float *x, float *xs) {
  uint4 *xw = reinterpret_cast<uint4 *>(xs);
  if (river) {
    uint32_t pr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) pr[q] = (uint32_t)f_to_act(x[q], ACT) | ((uint32_t)f_to_act(x[q + 4], ACT) << 16);
    const int c = t >> 7, ln = (t >> 2) & 31, j = t & 3;
    xw[(c * 4 + j) * 32 + ln] = make_uint4(pr[0], pr[1], pr[2], pr[3]);
    float X = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
    X += __shfl_xor_sync(0xffffffffu, X, 1);
    X += __shfl_xor_sync(0xffffffffu, X, 2);
    if (j == 0) xs[nk * 4 * 32 * 4 + c * 32 + ln] = X;
  } else {
    xw[t] = make_uint4((uint32_t)f_to_act(x[0], ACT) | ((uint32_t)f_to_act(x[1], ACT) << 16),
                       (uint32_t)f_to_act(x[2], ACT) | ((uint32_t)f_to_act(x[3], ACT) << 16),
                       (uint32_t)f_to_act(x[4], ACT) | ((uint32_t)f_to_act(x[5], ACT) << 16),
                       (uint32_t)f_to_act(x[6], ACT) | ((uint32_t)f_to_act(x[7], ACT) << 16));
  }
}

// General prologue: every thread issues the loads of SB passes before it
// converts and stores, so the L2 round trips of the passes overlap.
template <int ACT, int PRO>
__device__ __forceinline__ void stage_x(const GemvArgs &a, const Geo &g, int river, int nk, float r, float *xs) {
  constexpr int SB = 4;  // 8 for the plain vectors measured 1-2% slower (8B decode)
  const int nt = x_words(g, river);
  const float *src = PRO == PRO_NORM ? a.h : a.vec;
  const int nthr = (int)blockDim.x, lane = (int)(threadIdx.x & 31);
  for (int t0 = (int)threadIdx.x; t0 < nt; t0 += SB * nthr) {
    float4 u[SB][2];
    uint4 gw[SB];
#pragma unroll
    for (int i = 0; i < SB; ++i) {
      const int t = t0 + i * nthr;
      u[i][0] = u[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      gw[i] = make_uint4(0u, 0u, 0u, 0u);
      if (t < nt && t * 8 < g.K) {
        // activations come from other blocks of the same step: read them at L2
        const float4 *sp = reinterpret_cast<const float4 *>(src + t * 8);
        u[i][0] = __ldcg(sp);
        u[i][1] = __ldcg(sp + 1);
        if (PRO == PRO_NORM) gw[i] = *reinterpret_cast<const uint4 *>(a.gamma + t * 8);
      }
    }
#pragma unroll
    for (int i = 0; i < SB; ++i) {
      const int t = t0 + i * nthr;
      if (t - lane >= nt) break;  // the whole warp is past the end
      float x[8] = {u[i][0].x, u[i][0].y, u[i][0].z, u[i][0].w, u[i][1].x, u[i][1].y, u[i][1].z, u[i][1].w};
      if (PRO == PRO_NORM) {
        const uint16_t *gp = reinterpret_cast<const uint16_t *>(&gw[i]);
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = round_act(x[j] * r * act_to_f(gp[j], ACT), ACT);
      }
      store_xword<ACT>(river, nk, t, x, xs);
    }
  }
}

// RMSNorm prologue in one L2 round trip, for K up to NR_W * 8 * blockDim.x
// (both layouts' words fit): the thread's words t = tid + i * blockDim.x of h,
// of gamma and, where the exit decision is taken in the same prologue, of
// h_prev are loaded into registers once; the RMSNorm sum (and the decision's
// sums) come from them, then stage_norm writes x from them in the layout of
// the route the decision picked.
constexpr int NR_W = 2;
struct NormRegs {
  float4 h[NR_W][2];
  uint4 gw[NR_W];
  float ss, dot, n1;  // this thread's partial h.h, h_prev.h, h_prev.h_prev
};

__device__ __forceinline__ bool norm_fits(const Geo &g) {
  return max(x_words(g, 0), x_words(g, 1)) <= NR_W * (int)blockDim.x;
}

template <bool DEC>
__device__ __forceinline__ void norm_load(const GemvArgs &a, const Geo &g, const float *hprev, NormRegs &r) {
  r.ss = r.dot = r.n1 = 0.f;
#pragma unroll
  for (int i = 0; i < NR_W; ++i) {
    const int t = (int)threadIdx.x + i * (int)blockDim.x;
    r.h[i][0] = r.h[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    r.gw[i] = make_uint4(0u, 0u, 0u, 0u);
    float4 p0 = make_float4(0.f, 0.f, 0.f, 0.f), p1 = p0;
    if (t * 8 < g.K) {
      const float4 *sp = reinterpret_cast<const float4 *>(a.h + t * 8);
      r.h[i][0] = __ldcg(sp);
      r.h[i][1] = __ldcg(sp + 1);
      r.gw[i] = *reinterpret_cast<const uint4 *>(a.gamma + t * 8);
      if (DEC) {
        const float4 *pp = reinterpret_cast<const float4 *>(hprev + t * 8);
        p0 = __ldcg(pp);
        p1 = __ldcg(pp + 1);
      }
    }
    const float4 y0 = r.h[i][0], y1 = r.h[i][1];
    r.ss = fmaf(y0.x, y0.x, fmaf(y0.y, y0.y, fmaf(y0.z, y0.z, fmaf(y0.w, y0.w, r.ss))));
    r.ss = fmaf(y1.x, y1.x, fmaf(y1.y, y1.y, fmaf(y1.z, y1.z, fmaf(y1.w, y1.w, r.ss))));
    if (DEC) {
      r.dot = fmaf(p0.x, y0.x, fmaf(p0.y, y0.y, fmaf(p0.z, y0.z, fmaf(p0.w, y0.w, r.dot))));
      r.dot = fmaf(p1.x, y1.x, fmaf(p1.y, y1.y, fmaf(p1.z, y1.z, fmaf(p1.w, y1.w, r.dot))));
      r.n1 = fmaf(p0.x, p0.x, fmaf(p0.y, p0.y, fmaf(p0.z, p0.z, fmaf(p0.w, p0.w, r.n1))));
      r.n1 = fmaf(p1.x, p1.x, fmaf(p1.y, p1.y, fmaf(p1.z, p1.z, fmaf(p1.w, p1.w, r.n1))));
    }
  }
}

template <int ACT>
__device__ __forceinline__ void stage_norm(const Geo &g, int river, int nk, float r, const NormRegs &nr, float *xs) {
  const int nt = x_words(g, river), lane = (int)(threadIdx.x & 31);
#pragma unroll
  for (int i = 0; i < NR_W; ++i) {
    const int t = (int)threadIdx.x + i * (int)blockDim.x;
    if (t - lane >= nt) break;  // the whole warp is past the end
    const float4 y0 = nr.h[i][0], y1 = nr.h[i][1];
    float x[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
    const uint16_t *gp = reinterpret_cast<const uint16_t *>(&nr.gw[i]);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = round_act(x[j] * r * act_to_f(gp[j], ACT), ACT);
    store_xword<ACT>(river, nk, t, x, xs);
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
// bq + rg for bq = bid * RG, + nblocks * RG, ...; chunks sp, sp + S, ...  Every
// quad is two row pairs (rows[0], rows[0] + 1) and (rows[2], rows[2] + 1); the
// offsets of rows[0] and rows[2] in the quad being issued (int4 words or
// 16-bit elements, and (scale, zero) words) are cached and recomputed when the
// quad changes.
struct ItemStream {
  int bq, c, step;
  uint32_t off0, off2, soff0, soff2;
};

template <int EPI>
__device__ __forceinline__ void stream_rows(const GemvArgs &a, const Geo &g, int river, int qd, ItemStream &is) {
  int rows[4];
  quad_rows<EPI>(a, qd, rows);
  const uint32_t stride = (uint32_t)(river ? g.words : g.K);
  is.off0 = (uint32_t)rows[0] * stride;
  is.off2 = (uint32_t)rows[2] * stride;
  is.soff0 = (uint32_t)rows[0] * (uint32_t)g.Gs;
  is.soff2 = (uint32_t)rows[2] * (uint32_t)g.Gs;
}

// Copy the next item of the stream into `stage` (one commit group per call,
// empty once the stream has ended).  lane_g: the lane's group within a chunk.
template <int EPI>
__device__ __forceinline__ void issue_item(const GemvArgs &a, const Geo &g, int river, int rg, int nquads, int nk,
                                           int S, int sp, int lane_g, ItemStream &is, char *stage, int lane) {
  if (is.bq + rg < nquads) {
    const unsigned sd = (unsigned)__cvta_generic_to_shared(stage) + lane * 16;
    if (river) {
      const int k0 = is.c * CH4 + lane * 32;
      if (k0 < g.Kp) {
        const uint32_t *qb = a.m.r.q + (k0 >> 3);
        const uint32_t *q0 = qb + is.off0, *q2 = qb + is.off2;
        cp16s(sd, q0);
        cp16s(sd + 512, q0 + g.words);
        cp16s(sd + 1024, q2);
        cp16s(sd + 1536, q2 + g.words);
        if (!g.spr) {  // each lane its own group's word: row r at r * 32 + lane
          const __half2 *sb = a.m.r.sz + (g.gpc ? is.c * g.gpc + lane_g : k0 / a.m.r.g);
          const unsigned ss = (unsigned)__cvta_generic_to_shared(stage) + STAGE_W + lane * 4;
          const __half2 *s0 = sb + is.soff0, *s2 = sb + is.soff2;
          cp4s(ss, s0);
          cp4s(ss + 128, s0 + g.Gs);
          cp4s(ss + 256, s2);
          cp4s(ss + 384, s2 + g.Gs);
        }
      }
      if (g.spr && lane < 4 * g.spr) {  // the chunk's groups of the 4 rows: row r at r * gpc
        const int r = lane / g.spr, piece = lane - r * g.spr;
        if (is.c * g.gpc + piece * 4 < g.G)  // a ragged last chunk has fewer groups
          cp16s((unsigned)__cvta_generic_to_shared(stage) + STAGE_W + (r * g.gpc + piece * 4) * 4,
                a.m.r.sz + (r < 2 ? is.soff0 : is.soff2) + (r & 1) * g.Gs + is.c * g.gpc + piece * 4);
      }
    } else {
      const int k0 = is.c * CH16 + lane * 8;
      if (k0 < g.K) {
        const uint16_t *w0 = a.m.w + k0 + is.off0, *w2 = a.m.w + k0 + is.off2;
        cp16s(sd, w0);
        cp16s(sd + 512, w0 + g.K);
        cp16s(sd + 1024, w2);
        cp16s(sd + 1536, w2 + g.K);
      }
    }
    is.c += S;
    if (is.c >= nk) {
      is.c = sp;
      is.bq += is.step;
      if (is.bq + rg < nquads) stream_rows<EPI>(a, g, river, is.bq + rg, is);
    }
  }
  cp_commit();
}

// Per-thread results of a GEMV phase that the caller combines across blocks:
// the s(l) sums of the down projection, the argmax candidate of the LM head.
struct PhaseOut {
  float p_dot, p_n1, p_n2, best;
  int best_i;
};

struct PhaseGeo {
  Geo g;
  int river, nk, S, RG, rg, sp, nquads, lane_g;
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
  p.lane_g = (river && p.g.gpc) ? ((threadIdx.x & 31) * 32) / a.m.r.g : 0;
  return p;
}

// Start a GEMV phase: issue the warp's first NST - 1 weight items into its
// ring.  Touches only weights (and the river flag the caller passes), so it
// may run before the phase's activations exist.
template <int NWARP, int EPI>
__device__ __forceinline__ ItemStream gemv_begin(const GemvArgs &a, int river, char *ring, int bid, int nblocks) {
  if (!a.m.w) river = 1;  // an offloaded backbone layer exists only in the river
  const PhaseGeo p = phase_geo<NWARP>(a, river);
  const int lane = threadIdx.x & 31;
  ItemStream is;
  is.bq = bid * p.RG;
  is.c = p.sp;
  is.step = nblocks * p.RG;
  if (is.bq + p.rg < p.nquads) stream_rows<EPI>(a, p.g, river, is.bq + p.rg, is);
#pragma unroll
  for (int i = 0; i < NST - 1; ++i)
    issue_item<EPI>(a, p.g, river, p.rg, p.nquads, p.nk, p.S, p.sp, p.lane_g, is, ring + i * STAGE, lane);
  return is;
}

// Run a GEMV phase whose first items gemv_begin issued: activation prologue
// (x = round16(RMSNorm(h) * gamma) or x = vec, into the lane layout in xs),
// the quad loop over the ring, and the epilogue in the owning warp.
// scratch: 256 floats (cross-warp partials, block sums).
// ss_in: sum of h^2 when the caller already has it (PRO_NORM), else < 0;
// nrp: h already in registers (norm_load), ss_in then its block sum.
template <int NWARP, int ACT, int PRO, int EPI>
__device__ __forceinline__ PhaseOut gemv_run(const GemvArgs &a, int river, float *xs, float *scratch, char *ring,
                                             ItemStream is, int bid, int nblocks, float ss_in = -1.f,
                                             const NormRegs *nrp = nullptr) {
  if (!a.m.w) river = 1;  // an offloaded backbone layer exists only in the river
  const PhaseGeo p = phase_geo<NWARP>(a, river);
  const Geo &g = p.g;
  const int nk = p.nk, S = p.S, RG = p.RG, rg = p.rg, sp = p.sp, nquads = p.nquads;
  const int tid = threadIdx.x, lane = tid & 31;
  float *red = scratch;         // [2][NWARP * 4]: cross-warp partials, double-buffered
  float *bsum = scratch + 128;  // block_sum scratch (3 x 32)

  if (PRO == PRO_NORM && nrp) {
    // h (and the sums) already in registers: the caller took the exit decision from them
    stage_norm<ACT>(g, river, nk, 1.0f / sqrtf(ss_in / (float)g.K + a.eps), *nrp, xs);
  } else if (PRO == PRO_NORM && ss_in < 0.f && norm_fits(g)) {
    NormRegs nr;
    norm_load<false>(a, g, nullptr, nr);
    const float ss = block_sum(nr.ss, bsum);
    stage_norm<ACT>(g, river, nk, 1.0f / sqrtf(ss / (float)g.K + a.eps), nr, xs);
  } else {
    float rs = 0.f;
    if (PRO == PRO_NORM) {
      float ss = ss_in;
      if (ss < 0.f) {
        ss = 0.f;
        for (int i = tid * 4; i < g.K; i += blockDim.x * 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.h + i));
          ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
        }
        ss = block_sum(ss, bsum);
      }
      rs = 1.0f / sqrtf(ss / (float)g.K + a.eps);
    }
    stage_x<ACT, PRO>(a, g, river, nk, rs, xs);
  }
  __syncthreads();

  const int pos = (EPI == EPI_QKV) ? a.st.len[0] : 0;
  PhaseOut out{0.f, 0.f, 0.f, -INFINITY, 0x7fffffff};
  // code extraction constants in registers (a two-immediate LOP3 is split in two)
  uint32_t cm, c1;
  asm("mov.b32 %0, %1;" : "=r"(cm) : "n"(CodeBits<ACT>::mask));
  asm("mov.b32 %0, %1;" : "=r"(c1) : "n"(CodeBits<ACT>::one));
  int parity = 0, t = 0;

  for (int base_q = bid * RG; base_q < nquads; base_q += nblocks * RG, parity ^= 1) {
    const int qd = base_q + rg;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    int rows[4] = {0, 0, 0, 0};
    if (qd < nquads) {
      quad_rows<EPI>(a, qd, rows);
      float al[4] = {0.f, 0.f, 0.f, 0.f}, ah[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = sp; c < nk; c += S, ++t) {
        cp_wait<NST - 2>();  // this lane's copies of item t have landed
        issue_item<EPI>(a, g, river, rg, nquads, nk, S, sp, p.lane_g, is, ring + ((t + NST - 1) & (NST - 1)) * STAGE,
                        lane);
        const char *stg = ring + (t & (NST - 1)) * STAGE;
        const uint4 *sw = reinterpret_cast<const uint4 *>(stg);
        if (river) {
          const int k0 = c * CH4 + lane * 32;
          if (k0 >= g.Kp) continue;
          const uint4 *xq = reinterpret_cast<const uint4 *>(xs) + c * 4 * 32 + lane;
          const float X = xs[nk * 4 * 32 * 4 + c * 32 + lane];
          const __half2 *ss = reinterpret_cast<const __half2 *>(stg + STAGE_W);
          const int srow = g.spr ? g.gpc : 32, sidx = g.spr ? p.lane_g : lane;
          uint32_t xr[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 f = xq[j * 32];
            xr[4 * j] = f.x; xr[4 * j + 1] = f.y; xr[4 * j + 2] = f.z; xr[4 * j + 3] = f.w;
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const uint4 w = sw[r * 32 + lane];
            float a0 = 0.f, a1 = 0.f;
            word_mix<ACT>(w.x, xr + 0, a0, a1, cm, c1);
            word_mix<ACT>(w.y, xr + 4, a0, a1, cm, c1);
            word_mix<ACT>(w.z, xr + 8, a0, a1, cm, c1);
            word_mix<ACT>(w.w, xr + 12, a0, a1, cm, c1);
            const float2 sz = __half22float2(ss[r * srow + sidx]);
            const float run = fmaf(CodeBits<ACT>::A, a0 + a1, -(CodeBits<ACT>::B + sz.y) * X);
            v[r] = fmaf(sz.x, run, v[r]);
          }
        } else {
          const int k0 = c * CH16 + lane * 8;
          if (k0 >= g.K) continue;
          const uint4 xv = reinterpret_cast<const uint4 *>(xs)[c * 32 + lane];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const uint4 w = sw[r * 32 + lane];
            al[r] = fma_lo16<ACT>(w.x, xv.x, al[r]);
            ah[r] = fma_hi16<ACT>(w.x, xv.x, ah[r]);
            al[r] = fma_lo16<ACT>(w.y, xv.y, al[r]);
            ah[r] = fma_hi16<ACT>(w.y, xv.y, ah[r]);
            al[r] = fma_lo16<ACT>(w.z, xv.z, al[r]);
            ah[r] = fma_hi16<ACT>(w.z, xv.z, ah[r]);
            al[r] = fma_lo16<ACT>(w.w, xv.w, al[r]);
            ah[r] = fma_hi16<ACT>(w.w, xv.w, ah[r]);
          }
        }
      }
      if (!river) {
#pragma unroll
        for (int r = 0; r < 4; ++r) v[r] = al[r] + ah[r];
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
