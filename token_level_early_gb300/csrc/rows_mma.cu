// Batched decode rows on the tensor pipe (mma.sync m16n8k16), for lists of
// at most 64 rows (16-bit weights) or fewer than 256 (int4 river weights):
// Y[m][n] = sum_k X[m][k] W[n][k] over the listed rows m.  The river layer of
// a batch of decode rows is the river GEMV of paperlayer.ai section 4 applied
// to every row whose token has left the backbone; its codes, scales and zero
// points are the W4A16 copy of the backbone (aitrends.kr).
//
// Block: 8 warps x 16 weight rows = 128 rows of W, 64 listed rows of X, one
// K chunk of KC columns at a time, weights and X staged in shared memory
// (rows padded by 16 bytes so the 8 rows of an ldmatrix fall on distinct
// banks).  Each A fragment (16 weight rows x 16 columns) serves the 8 n8-tiles
// of the 64 listed rows, which enter as B fragments through ldmatrix.
//   16-bit weights: A by ldmatrix from the staged rows; X staged in natural
//     order.
//   int4 weights: one rotate and one LOP3 turn two codes of a word (codes t
//     and t + 4) into a pair of 16-bit floats 1 + q/16 (exact in fp16 and
//     bf16), so the MMA's k index runs over a word's codes in the order t,
//     t + 4; X is staged as 16-bit pairs in the same order (x[8w + t],
//     x[8w + t + 4]).  Per group of g codes the accumulator D = sum (1 +
//     q/16) x (of the size of the group's sum of |x|, so its fp32 rounding
//     stays small) is folded as
//       sum (q - z) x = 16 D - (16 + z) X_g,   X_g = sum of the group's x,
//     then scaled by s.
// The K chunks of a (weight tile, row tile) are split over a thread-block
// cluster; the blocks' partial tiles are summed in rank order through
// distributed shared memory (deterministic, no global scratch).
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.cuh"

namespace cg = cooperative_groups;

namespace rv {
namespace {

constexpr int RW = 8;        // warps per block
constexpr int RN = 16 * RW;  // weight rows per block
constexpr int RM = 64;       // listed rows per block (8 n8-tiles)

// Codes as 16-bit floats 1 + q/16 (exact): the code's nibble lands in the
// top four mantissa bits.  fp16: bits 6..9 of each half, bf16: bits 3..6.
template <int ACT>
struct CodeBits16;
template <>
struct CodeBits16<1> {  // bf16
  static constexpr uint32_t mask = 0x00780078u, one = 0x3F803F80u;
  static constexpr int sh = 3;
};
template <>
struct CodeBits16<0> {  // fp16
  static constexpr uint32_t mask = 0x03C003C0u, one = 0x3C003C00u;
  static constexpr int sh = 6;
};

// Codes t and t + 4 of word w (bits 4t.. and 4t + 16..) as the 16-bit pair
// (1 + q_t/16, 1 + q_{t+4}/16): rotate the word so both nibbles land in the
// mantissa field (rot = sh - 4t mod 32), then one LOP3 (w & mask) | one.
__device__ __forceinline__ uint32_t code_pair(uint32_t w, int rot, uint32_t m, uint32_t c) {
  const uint32_t r = __funnelshift_l(w, w, rot);
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(r), "r"(m), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int act) {
  return (uint32_t)f_to_act(lo, act) | ((uint32_t)f_to_act(hi, act) << 16);
}

__device__ __forceinline__ void ldsm4(uint32_t *r, unsigned addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

template <int ACT>
__device__ __forceinline__ void mma_16816(float *d, const uint32_t *a, const uint32_t *b) {
  if (ACT == 1)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void cp16_or_zero(unsigned dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp4_or_zero(unsigned dst, const void *src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
}

// Shared-memory layout (bytes) for a chunk of KC columns; GS = the group
// size of int4 weights, 0 for 16-bit weights.
template <int KC, int GS>
struct RowsLayout {
  static constexpr int GPC = GS ? KC / GS : 0;          // groups per chunk
  static constexpr int XR = KC * 2 + 16;                // staged X row: KC 16-bit values + pad
  static constexpr int WR = (GS ? KC / 2 : KC * 2) + 16;  // staged weight row + pad
  static constexpr int XS = 0;                          // [RM][XR]
  static constexpr int XG = XS + RM * XR;               // [RM][GPC] float group sums of x
  static constexpr int WS = XG + RM * GPC * 4;          // [RN][WR] weights
  static constexpr int SZ = WS + RN * WR;               // [RN][GPC] half2 (scale, zero)
  static constexpr int ROWS = SZ + RN * GPC * 4;        // [RM] int listed rows (-1: none)
  static constexpr int BYTES = ROWS + RM * 4;
  static_assert(RM * XR >= RM * RN * 4, "the partial tile reuses the X stage");
};

// Greedy-pick key of logit v at column n: larger keys are larger values,
// ties broken towards the lower column (order-preserving float bits above,
// the complemented column below).
__device__ __forceinline__ unsigned long long pick_key(float v, int n) {
  const uint32_t b = __float_as_uint(v == 0.f ? 0.f : v);  // -0 ties with +0
  const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)o << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)n);
}

// amax (optional): per listed row, the largest pick_key of its outputs
// (atomicMax; the caller zeroes it and reads it back with k_pick_finish).
template <int ACT, int KC, int GS>
__global__ void __launch_bounds__(RW * 32, 2) k_rows_mma(Mat mt, const float *X, float *Y, const int32_t *list,
                                                         const int32_t *count, unsigned long long *amax) {
  using LY = RowsLayout<KC, GS>;
  constexpr bool I4 = GS > 0;
  constexpr int GPC = LY::GPC, XR = LY::XR, WR = LY::WR;
  constexpr int WPR = KC / 8;  // words (8 columns) per row and chunk
  extern __shared__ __align__(16) unsigned char sm[];
  cg::cluster_group cl = cg::this_cluster();
  const int cs = (int)cl.num_blocks(), rank = (int)cl.block_rank();
  const int n0 = blockIdx.x * RN;
  const int N = mt.N, K = mt.K;
  const RiverMat &R = mt.r;
  const int Kw = I4 ? R.Kp : K;  // columns of the stored weight rows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const unsigned sbase = (unsigned)__cvta_generic_to_shared(sm);
  int *rows = reinterpret_cast<int *>(sm + LY::ROWS);
  float *xg = reinterpret_cast<float *>(sm + LY::XG);
  const __half2 *wsz = reinterpret_cast<const __half2 *>(sm + LY::SZ);

  // the warp's 16 weight rows of chunk kc (and their (scale, zero) words)
  auto stage_w = [&](int kc) {
    const int k0 = kc * KC;
    const unsigned wdst = sbase + LY::WS + warp * 16 * WR;
    constexpr int PPR = (I4 ? KC / 2 : KC * 2) / 16;  // 16-byte pieces per row
    for (int p = lane; p < 16 * PPR; p += 32) {
      const int r = p / PPR, c = p % PPR, n = n0 + warp * 16 + r;
      bool ok;
      const void *src;
      if (I4) {
        ok = n < N && k0 + 32 * c < R.Kp;
        src = R.q + (ok ? (size_t)n * (R.Kp >> 3) + (k0 >> 3) + 4 * c : 0);
      } else {
        ok = n < N && k0 + 8 * c < K;
        src = mt.w + (ok ? (size_t)n * K + k0 + 8 * c : 0);
      }
      cp16_or_zero(wdst + r * WR + 16 * c, src, ok);
    }
    if (I4) {
      const unsigned sdst = sbase + LY::SZ + warp * 16 * GPC * 4;
      for (int p = lane; p < 16 * GPC; p += 32) {
        const int r = p / (GPC ? GPC : 1), j = p % (GPC ? GPC : 1), n = n0 + warp * 16 + r;
        const int gi = k0 / (GS ? GS : 1) + j;
        const bool ok = n < N && gi < R.G;
        cp4_or_zero(sdst + p * 4, R.sz + (ok ? (size_t)n * R.Gs + gi : 0), ok);
      }
    }
    cp_commit();
  };
  const int nkc = (Kw + KC - 1) / KC;
  // the weights do not depend on the previous kernel: the first chunk's copies
  // are issued before the programmatic-dependent-launch wait
  if (rank < nkc) stage_w(rank);
  pdl_wait();
  pdl_trigger();
  const int cnt = *count;
  const int r0 = blockIdx.y * RM;
  if (r0 >= cnt) {  // the whole cluster shares blockIdx.y
    cp_wait<0>();
    return;
  }
  if (tid < RM) rows[tid] = r0 + tid < cnt ? (list ? list[r0 + tid] : r0 + tid) : -1;
  __syncthreads();

  uint32_t cmask = 0, cbits = 0;  // int4 extraction constants in registers
  if (I4) {
    asm("mov.b32 %0, %1;" : "=r"(cmask) : "n"(CodeBits16<ACT>::mask));
    asm("mov.b32 %0, %1;" : "=r"(cbits) : "n"(CodeBits16<ACT>::one));
  }
  const int rot = (CodeBits16<ACT>::sh - 4 * tq) & 31;

  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  for (int kc = rank; kc < nkc; kc += cs) {
    const int k0 = kc * KC;
    if (kc != rank) stage_w(kc);
    // X chunk as 16-bit pairs: int4 weights (x[8w + t], x[8w + t + 4]) with
    // per-group sums, 16-bit weights (x[8w + 2t], x[8w + 2t + 1]); thread:
    // word w of rows i0, i0 + RPP, ..., four rows' loads in flight before any
    // is converted
    {
      constexpr int RPP = RW * 32 / WPR;  // rows per pass
      constexpr int NB = I4 ? 4 : 8;      // rows per batch of loads
      static_assert((RM / RPP) % NB == 0, "whole batches of rows");
      const int w = tid % WPR, i0 = tid / WPR, k = k0 + 8 * w;
      const bool full = k + 8 <= K;
#pragma unroll 1
      for (int ib = i0; ib < RM; ib += NB * RPP) {
        float4 lo[NB], hi[NB];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          const int m = rows[ib + u * RPP];
          lo[u] = hi[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (m >= 0 && full) {
            lo[u] = __ldg(reinterpret_cast<const float4 *>(X + (size_t)m * K + k));
            hi[u] = __ldg(reinterpret_cast<const float4 *>(X + (size_t)m * K + k + 4));
          } else if (m >= 0) {
            float x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = k + j < K ? X[(size_t)m * K + k + j] : 0.f;
            lo[u] = make_float4(x[0], x[1], x[2], x[3]);
            hi[u] = make_float4(x[4], x[5], x[6], x[7]);
          }
        }
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          const int i = ib + u * RPP;
          uint4 v;
          if (I4) {
            v.x = pack2(lo[u].x, hi[u].x, ACT);
            v.y = pack2(lo[u].y, hi[u].y, ACT);
            v.z = pack2(lo[u].z, hi[u].z, ACT);
            v.w = pack2(lo[u].w, hi[u].w, ACT);
          } else {
            v.x = pack2(lo[u].x, lo[u].y, ACT);
            v.y = pack2(lo[u].z, lo[u].w, ACT);
            v.z = pack2(hi[u].x, hi[u].y, ACT);
            v.w = pack2(hi[u].z, hi[u].w, ACT);
          }
          *reinterpret_cast<uint4 *>(sm + LY::XS + i * XR + 16 * w) = v;
          if (I4) {
            // x is already rounded to the 16-bit type: the sum is of the values the MMA sees
            float sx = ((lo[u].x + lo[u].y) + (lo[u].z + lo[u].w)) + ((hi[u].x + hi[u].y) + (hi[u].z + hi[u].w));
#pragma unroll
            for (int o = GS / 16; o >= 1; o >>= 1) sx += __shfl_xor_sync(0xffffffffu, sx, o);
            if (w % (GS / 8 ? GS / 8 : 1) == 0) xg[i * GPC + w / (GS / 8 ? GS / 8 : 1)] = sx;
          }
        }
      }
    }
    cp_wait<0>();
    __syncthreads();

    if (I4) {
      // the warp's 16 weight rows x 64 listed rows, group by group
      const unsigned char *wr0 = sm + LY::WS + (warp * 16 + gq) * WR;
      const unsigned char *wr1 = wr0 + 8 * WR;
#pragma unroll 1
      for (int j = 0; j < GPC; ++j) {
        if constexpr (GS > 0 && GS <= 128) {
          // the group's A fragments (unpacked once), then the listed rows as
          // two halves of 4 n8-tiles: 16 registers of D instead of 32 under
          // the register budget of two blocks per SM (each tile's MMAs in the
          // same order as below; groups of 256 keep the one-pass form, whose
          // A fragments would not fit)
          uint32_t A[GS / 32 > 0 ? GS / 32 : 1][8];
#pragma unroll
          for (int s2 = 0; s2 < GS / 32; ++s2) {
            const int wd = (j * GS + 32 * s2) / 8;
            const uint4 u0 = *reinterpret_cast<const uint4 *>(wr0 + 4 * wd);
            const uint4 u1 = *reinterpret_cast<const uint4 *>(wr1 + 4 * wd);
            A[s2][0] = code_pair(u0.x, rot, cmask, cbits); A[s2][1] = code_pair(u1.x, rot, cmask, cbits);
            A[s2][2] = code_pair(u0.y, rot, cmask, cbits); A[s2][3] = code_pair(u1.y, rot, cmask, cbits);
            A[s2][4] = code_pair(u0.z, rot, cmask, cbits); A[s2][5] = code_pair(u1.z, rot, cmask, cbits);
            A[s2][6] = code_pair(u0.w, rot, cmask, cbits); A[s2][7] = code_pair(u1.w, rot, cmask, cbits);
          }
          const float2 z0 = __half22float2(wsz[(warp * 16 + gq) * GPC + j]);
          const float2 z1 = __half22float2(wsz[(warp * 16 + gq + 8) * GPC + j]);
          const float c0 = -(16.f + z0.y), c1 = -(16.f + z1.y);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            float D[4][4];
#pragma unroll
            for (int t = 0; t < 4; ++t) D[t][0] = D[t][1] = D[t][2] = D[t][3] = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < GS / 32; ++s2) {
              const int wd = (j * GS + 32 * s2) / 8;
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int nt = 4 * hf + t;
                uint32_t b[4];  // words wd .. wd + 3 of rows 8 nt .. 8 nt + 7
                ldsm4(b, sbase + LY::XS + (8 * nt + (lane & 7)) * XR + (wd + (lane >> 3)) * 16);
                mma_16816<ACT>(D[t], A[s2], b);
                mma_16816<ACT>(D[t], A[s2] + 4, b + 2);
              }
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int nt = 4 * hf + t;
              const float X0 = xg[(8 * nt + 2 * tq) * GPC + j], X1 = xg[(8 * nt + 2 * tq + 1) * GPC + j];
              acc[nt][0] = fmaf(z0.x, fmaf(c0, X0, 16.f * D[t][0]), acc[nt][0]);
              acc[nt][1] = fmaf(z0.x, fmaf(c0, X1, 16.f * D[t][1]), acc[nt][1]);
              acc[nt][2] = fmaf(z1.x, fmaf(c1, X0, 16.f * D[t][2]), acc[nt][2]);
              acc[nt][3] = fmaf(z1.x, fmaf(c1, X1, 16.f * D[t][3]), acc[nt][3]);
            }
          }
          continue;
        }
        float D[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) D[nt][0] = D[nt][1] = D[nt][2] = D[nt][3] = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < GS / 32; ++s2) {
          const int wd = (j * GS + 32 * s2) / 8;  // first of the 4 words (two k-steps)
          const uint4 u0 = *reinterpret_cast<const uint4 *>(wr0 + 4 * wd);
          const uint4 u1 = *reinterpret_cast<const uint4 *>(wr1 + 4 * wd);
          const uint32_t a0[4] = {code_pair(u0.x, rot, cmask, cbits), code_pair(u1.x, rot, cmask, cbits),
                                  code_pair(u0.y, rot, cmask, cbits), code_pair(u1.y, rot, cmask, cbits)};
          const uint32_t a1[4] = {code_pair(u0.z, rot, cmask, cbits), code_pair(u1.z, rot, cmask, cbits),
                                  code_pair(u0.w, rot, cmask, cbits), code_pair(u1.w, rot, cmask, cbits)};
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) {
            uint32_t b[4];  // words wd .. wd + 3 of rows 8 nt .. 8 nt + 7
            ldsm4(b, sbase + LY::XS + (8 * nt + (lane & 7)) * XR + (wd + (lane >> 3)) * 16);
            mma_16816<ACT>(D[nt], a0, b);
            mma_16816<ACT>(D[nt], a1, b + 2);
          }
        }
        // fold the group: rows gq / gq + 8 of the warp, listed rows 8 nt + 2 tq (+1)
        const float2 z0 = __half22float2(wsz[(warp * 16 + gq) * GPC + j]);
        const float2 z1 = __half22float2(wsz[(warp * 16 + gq + 8) * GPC + j]);
        const float c0 = -(16.f + z0.y), c1 = -(16.f + z1.y);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const float X0 = xg[(8 * nt + 2 * tq) * GPC + j], X1 = xg[(8 * nt + 2 * tq + 1) * GPC + j];
          acc[nt][0] = fmaf(z0.x, fmaf(c0, X0, 16.f * D[nt][0]), acc[nt][0]);
          acc[nt][1] = fmaf(z0.x, fmaf(c0, X1, 16.f * D[nt][1]), acc[nt][1]);
          acc[nt][2] = fmaf(z1.x, fmaf(c1, X0, 16.f * D[nt][2]), acc[nt][2]);
          acc[nt][3] = fmaf(z1.x, fmaf(c1, X1, 16.f * D[nt][3]), acc[nt][3]);
        }
      }
    } else {
      // 16-bit weights: A = rows 16 warp .. +15 by ldmatrix (matrices: rows
      // 0-7 / 8-15 x columns 0-7 / 8-15 of the k-step)
      const unsigned wa = sbase + LY::WS + (warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * WR + 16 * (lane >> 4);
#pragma unroll 2
      for (int kp = 0; kp < KC / 32; ++kp) {
        uint32_t a0[4], a1[4];
        ldsm4(a0, wa + 64 * kp);
        ldsm4(a1, wa + 64 * kp + 32);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          uint32_t b[4];  // columns 32 kp .. 32 kp + 31 of rows 8 nt .. 8 nt + 7
          ldsm4(b, sbase + LY::XS + (8 * nt + (lane & 7)) * XR + (4 * kp + (lane >> 3)) * 16);
          mma_16816<ACT>(acc[nt], a0, b);
          mma_16816<ACT>(acc[nt], a1, b + 2);
        }
      }
    }
    __syncthreads();  // the stages are rewritten by the next chunk (or the partial tile)
  }

  // partial tile [RM][RN] over the X stage, then the cluster's ranks sum it
  // in rank order, each rank writing a slice of the listed rows
  float *pt = reinterpret_cast<float *>(sm + LY::XS);
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int m0 = 8 * nt + 2 * tq, c = warp * 16 + gq;
    pt[m0 * RN + c] = acc[nt][0];
    pt[(m0 + 1) * RN + c] = acc[nt][1];
    pt[m0 * RN + c + 8] = acc[nt][2];
    pt[(m0 + 1) * RN + c + 8] = acc[nt][3];
  }
  cl.sync();
  {
    const int per = (RM + cs - 1) / cs, mb = rank * per, me = min(RM, mb + per);
    // a warp's 32 items share one listed row (RN is a multiple of 32, so the
    // trip count is warp-uniform)
    for (int it = tid; it < (me - mb) * RN; it += RW * 32) {
      const int i = mb + it / RN, c = it % RN, n = n0 + c, m = rows[i];
      const bool ok = m >= 0 && n < N;
      float v = 0.f;
      if (ok) {
        for (int r = 0; r < cs; ++r) v += cl.map_shared_rank(pt, r)[i * RN + c];
        Y[(size_t)m * N + n] = v;
      }
      if (amax) {
        unsigned long long key = ok ? pick_key(v, n) : 0ull;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
          key = other > key ? other : key;
        }
        if (lane == 0 && key) atomicMax(amax + m, key);
      }
    }
  }
  cl.sync();  // every rank's partial tile stays readable until all slices are written
}

template <int ACT, int KC, int GS>
cudaError_t launch_kc(const Mat &m, const float *X, float *Y, const int32_t *list, const int32_t *count, int max_rows,
                      int n_sm, cudaStream_t s, unsigned long long *amax = nullptr) {
  auto fn = k_rows_mma<ACT, KC, GS>;
  constexpr int bytes = RowsLayout<KC, GS>::BYTES;
  const int Kw = GS ? m.r.Kp : m.K;
  const int ntn = (m.N + RN - 1) / RN, ntm = (max_rows + RM - 1) / RM, nkc = (Kw + KC - 1) / KC;
  int cs = 1;
  while (2 * cs <= 16 && 2 * cs <= nkc && ntn * ntm * cs < 2 * n_sm) cs *= 2;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cs > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntn, ntm, cs);
  cfg.blockDim = dim3(RW * 32);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = cs;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // the kernel waits with griddepcontrol
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, fn, m, X, Y, list, count, amax);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int ACT, int GS>
cudaError_t launch_gs(const Mat &m, const float *X, float *Y, const int32_t *list, const int32_t *count, int max_rows,
                      int n_sm, cudaStream_t s) {
  // 512-column chunks unless that leaves the GPU short of blocks (small N and K)
  const int ntn = (m.N + RN - 1) / RN, ntm = (max_rows + RM - 1) / RM, nkc = (m.r.Kp + 511) / 512;
  const int most = nkc < 16 ? nkc : 16;
  if (ntn * ntm * most < 2 * n_sm) return launch_kc<ACT, 256, GS>(m, X, Y, list, count, max_rows, n_sm, s);
  return launch_kc<ACT, 512, GS>(m, X, Y, list, count, max_rows, n_sm, s);
}

}  // namespace

bool rows_i4_supported(const Mat &m) {
  const int g = m.r.g;
  return m.r.q && (g == 32 || g == 64 || g == 128 || g == 256) && m.K % 4 == 0;
}

bool rows_b16_supported(const Mat &m) { return m.w && m.K % 8 == 0; }

cudaError_t launch_rows_i4(const Mat &m, int act, const float *X, float *Y, const int32_t *list,
                           const int32_t *count, int max_rows, int n_sm, cudaStream_t s) {
  if (max_rows <= 0) return cudaSuccess;
  if (!rows_i4_supported(m) || (act != 0 && act != 1)) return cudaErrorInvalidValue;
  if ((m.N + RN - 1) / RN > 65535 || (max_rows + RM - 1) / RM > 65535) return cudaErrorInvalidValue;
#define RV_RI(A_, G_) \
  if (act == A_ && m.r.g == G_) return launch_gs<A_, G_>(m, X, Y, list, count, max_rows, n_sm, s);
  RV_RI(1, 32) RV_RI(1, 64) RV_RI(1, 128) RV_RI(1, 256)
  RV_RI(0, 32) RV_RI(0, 64) RV_RI(0, 128) RV_RI(0, 256)
#undef RV_RI
  return cudaErrorInvalidValue;
}

cudaError_t launch_rows_b16(const Mat &m, int act, const float *X, float *Y, const int32_t *list,
                            const int32_t *count, int max_rows, int n_sm, cudaStream_t s, unsigned long long *amax) {
  if (max_rows <= 0) return cudaSuccess;
  if (!rows_b16_supported(m) || (act != 0 && act != 1)) return cudaErrorInvalidValue;
  if ((m.N + RN - 1) / RN > 65535 || (max_rows + RM - 1) / RM > 65535) return cudaErrorInvalidValue;
  return act == 1 ? launch_kc<1, 256, 0>(m, X, Y, list, count, max_rows, n_sm, s, amax)
                  : launch_kc<0, 256, 0>(m, X, Y, list, count, max_rows, n_sm, s, amax);
}

// Greedy ids from the keys the LM-head rows kernel left in amax (rows
// 0..B-1), which are zeroed again for the next step; the length update of
// k_argmax_rows.
__global__ void k_pick_finish(unsigned long long *amax, int B, StepState st, int bump_len, int set_len) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const unsigned long long key = amax[b];
  amax[b] = 0ull;
  st.next_ids[b] = key ? (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull)) : 0;
  if (bump_len) st.len[b] += 1;
  if (set_len >= 0) st.len[b] = set_len;
}

cudaError_t launch_pick_finish(unsigned long long *amax, int B, StepState st, int bump_len, int set_len,
                               cudaStream_t s) {
  return launch_k(k_pick_finish, dim3((B + 127) / 128), dim3(128), 0, s, 1, amax, B, st, bump_len, set_len);
}

}  // namespace rv
