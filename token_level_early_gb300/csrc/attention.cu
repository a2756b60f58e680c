// GQA attention over the shared KV cache.
//
// One kernel serves decode and prefill: block (row m, split, kv head g)
// handles the GRP query heads that share KV head g, so each K/V tile is read
// once for all of them (grouped-query attention).  Row m is token m % T of
// sequence m / T at position base[b] + m % T and attends causally to
// positions 0..pos of its own sequence in layer `layer`.  Long rows are split
// over `splits` blocks (flash-decoding); the last block of a (row, kv head)
// merges the partial softmax states.  The single KV cache is the one every
// backbone and river layer writes (paperlayer.ai section 4 / appendix A.3;
// aitrends.kr KV Share).
//
// Decode rows use k_attn_dec: the splits of one (row, kv head) form a
// thread-block cluster.  Each split's warps stream its share of the past
// positions 0..p-1 (final before the step starts) through private
// shared-memory rings filled before the programmatic-dependent-launch wait,
// and run S = q K^T and O += P V on the tensor pipe for all the kv head's
// query heads at once; only q and the K/V of position p come from the QKV
// kernel it follows.  The warps merge in shared memory, the splits through
// distributed shared memory.
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace cg = cooperative_groups;

namespace rv {

constexpr int TILE = 32;

template <int HD, int GRP>
__global__ void __launch_bounds__(GRP * 32) k_attn(AttnArgs a, int T_per_row, const int32_t *base, int rows) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x, sp = blockIdx.y, g = blockIdx.z;
  if (m >= rows) return;
  const int b = m / T_per_row;
  const int pos = (base ? base[b] : 0) + (m % T_per_row);
  const int T = pos + 1;
  const int chunk = (T + a.splits - 1) / a.splits;
  const int t0 = sp * chunk, t1 = min(T, t0 + chunk);
  const int H = a.H, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = g * GRP + warp;
  constexpr int NT = GRP * 32;
  constexpr int PER = HD / 32;

  __shared__ float qs[GRP][HD];
  __shared__ float Ks[TILE][HD + 1];
  __shared__ float Vs[TILE][HD];

  for (int i = threadIdx.x; i < GRP * HD; i += NT) qs[i / HD][i % HD] = a.q[(size_t)m * H * HD + (size_t)g * GRP * HD + i];
  const uint16_t *Kb = a.kv.base + a.kv.idx(a.layer, 0, b, g, 0);
  const uint16_t *Vb = a.kv.base + a.kv.idx(a.layer, 1, b, g, 0);
  const float scale = 1.0f / sqrtf((float)HD);

  float mrun = -INFINITY, lrun = 0.f, o[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) o[r] = 0.f;

  for (int tile = t0; tile < t1; tile += TILE) {
    const int n = min(TILE, t1 - tile);
    __syncthreads();
    // stage K and V rows of this tile (8 values per 16-byte load)
    for (int v = threadIdx.x; v < n * (HD / 8); v += NT) {
      const int t = v / (HD / 8), c = (v % (HD / 8)) * 8;
      const uint4 kw = *reinterpret_cast<const uint4 *>(Kb + (size_t)(tile + t) * HD + c);
      const uint4 vw = *reinterpret_cast<const uint4 *>(Vb + (size_t)(tile + t) * HD + c);
      const uint16_t *kp = reinterpret_cast<const uint16_t *>(&kw);
      const uint16_t *vp = reinterpret_cast<const uint16_t *>(&vw);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        Ks[t][c + j] = act_to_f(kp[j], a.act);
        Vs[t][c + j] = act_to_f(vp[j], a.act);
      }
    }
    __syncthreads();
    float sc = -INFINITY;
    if (lane < n) {
      float d = 0.f;
#pragma unroll 8
      for (int i = 0; i < HD; ++i) d = fmaf(qs[warp][i], Ks[lane][i], d);
      sc = d * scale;
    }
    const float mt = warp_max(sc);
    const float mnew = fmaxf(mrun, mt);
    const float p = lane < n ? expf(sc - mnew) : 0.f;
    const float corr = mrun == -INFINITY ? 0.f : expf(mrun - mnew);
    lrun = lrun * corr + warp_sum(p);
#pragma unroll
    for (int r = 0; r < PER; ++r) o[r] *= corr;
    for (int t = 0; t < n; ++t) {
      const float pt = __shfl_sync(0xffffffffu, p, t);
#pragma unroll
      for (int r = 0; r < PER; ++r) o[r] = fmaf(pt, Vs[t][lane + 32 * r], o[r]);
    }
    mrun = mnew;
  }

  const size_t orow = (size_t)m * H * HD + (size_t)h * HD;
  if (a.splits == 1) {
    const float inv = 1.0f / lrun;
#pragma unroll
    for (int r = 0; r < PER; ++r) a.o[orow + lane + 32 * r] = round_act(o[r] * inv, a.act);
    return;
  }
  // publish this split's state: o (unnormalised), running max, running sum
  float *pp = a.part + (((size_t)m * H + h) * a.splits + sp) * (HD + 2);
#pragma unroll
  for (int r = 0; r < PER; ++r) pp[lane + 32 * r] = o[r];
  if (lane == 0) { pp[HD] = mrun; pp[HD + 1] = lrun; }
  __threadfence();
  __syncthreads();
  __shared__ bool last;
  if (threadIdx.x == 0) {
    unsigned *c = a.counter + (size_t)m * a.Hkv + g;
    unsigned t = atomicAdd(c, 1u);
    last = (t == (unsigned)a.splits - 1);
    if (last) *c = 0u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const float *base_p = a.part + ((size_t)m * H + h) * a.splits * (HD + 2);
  float M = -INFINITY;
  for (int s = 0; s < a.splits; ++s) M = fmaxf(M, base_p[s * (HD + 2) + HD]);
  float Lsum = 0.f, acc[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) acc[r] = 0.f;
  for (int s = 0; s < a.splits; ++s) {
    const float ms = base_p[s * (HD + 2) + HD];
    const float w = ms == -INFINITY ? 0.f : expf(ms - M);
    Lsum = fmaf(w, base_p[s * (HD + 2) + HD + 1], Lsum);
#pragma unroll
    for (int r = 0; r < PER; ++r) acc[r] = fmaf(w, base_p[s * (HD + 2) + lane + 32 * r], acc[r]);
  }
  const float inv = 1.0f / Lsum;
#pragma unroll
  for (int r = 0; r < PER; ++r) a.o[orow + lane + 32 * r] = round_act(acc[r] * inv, a.act);
}

// ---- tensor-pipe helpers (decode and prefill) ------------------------------
__device__ __forceinline__ void cp16z(unsigned dst, const void *src, bool valid) {
  const int n = valid ? 16 : 0;  // 0: zero-fill, nothing read
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t *r, unsigned addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t *r, unsigned addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
template <int ACT>
__device__ __forceinline__ void mma16816(float *d, const uint32_t *a, const uint32_t *b) {
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
__device__ __forceinline__ uint32_t pack_act2(float lo, float hi, int act) {
  return (uint32_t)f_to_act(lo, act) | ((uint32_t)f_to_act(hi, act) << 16);
}

// ---- decode: split-KV attention on the tensor pipe -------------------------
// Block (split sp, kv head g, row b) of NW warps.  The split's tiles of TT
// past positions are dealt round-robin to its warps; each warp streams its
// own tiles through a private cp.async ring of NS slots (no block barrier in
// the loop), the first ones issued before the programmatic-dependent-launch
// wait.  Per tile, one warp serves all GRP query heads of the kv head:
//   S = q K^T       m16n8k16, M = heads (rows >= GRP are zero), N = positions,
//   O^T += V^T P^T  M = head dims, N = heads, K = positions,
// so the score fragments are already the B fragments of the P V product (no
// shuffle through shared memory).  Scores are kept in the log2 domain
// (scaled by log2(e) / sqrt(hd)); P enters as two 16-bit terms hi + lo like
// the prefill kernel.  After the loop the warps' softmax states and the
// position p itself (its K/V come from the QKV kernel this kernel follows)
// merge in shared memory, then the splits merge:
//   short contexts (GM = false): the splits of a (row, kv head) form a
//     thread-block cluster and merge through distributed shared memory; one
//     ring slot per warp keeps a block small (several per SM, so clusters of
//     16 find room and the neighbouring GEMV kernels keep theirs);
//   long contexts (GM = true): no cluster, about one block per SM with a deep
//     ring, the splits' states go through global memory and the last block of
//     a (row, kv head) to finish merges them (an atomic ticket, no waiting).
// Two block shapes: short contexts (the cluster plan) 4 warps x tiles of 32
// positions x 1 ring slot per warp (a warp holds at most one tile); long
// contexts (the global-merge plan) 8 warps x tiles of 16 positions x a
// multi-slot ring, the same bytes in flight per SM with twice the warps to
// run the tile math (one warp per scheduler left the issue slots 2/3 idle).
constexpr int DTT = 32;  // positions per tile, short plan
constexpr int DNW = 4;   // warps per block, short plan
constexpr int LTT = 16;  // positions per tile, long plan
constexpr int LNW = 8;   // warps per block, long plan

template <int HD, int TT>
struct DecTile {
  static constexpr int ROW = HD * 2 + 16;      // padded row: the 8 rows of an ldmatrix hit distinct banks
  static constexpr int BYTES = 2 * TT * ROW;   // K rows then V rows
};
template <int HD>
constexpr int long_slots() { return HD == 64 ? 6 : 3; }  // ring slots per warp, long plan

// Merge-phase layout (floats, over the ring once it is drained):
//   part [GRP][HD]       the block's O (read by the other splits)
//   wpo  [NW][GRP][HD]   the warps' O
//   pm   [GRP][2]        the block's (max, sum) (read by the other splits)
//   wml  [NW][GRP][2]    the warps' (max, sum)
//   sps  [GRP]           score of position p;  spv [HD] its V row
//   gml  [splits][GRP][2] the splits' (max, sum), then the last-block flag (global merge)
template <int HD, int NW>
__host__ __device__ constexpr int dec_merge_floats(int grp) {
  return (1 + NW) * grp * HD + 2 * grp + NW * grp * 2 + grp + HD + kAttnMaxSplits * grp * 2 + 1;
}
template <int HD, int NW, int TT, int NS>
static size_t dec_smem(int grp) {
  const size_t merge = sizeof(float) * (size_t)dec_merge_floats<HD, NW>(grp);
  const size_t ring = (size_t)NW * NS * DecTile<HD, TT>::BYTES;
  return merge > ring ? merge : ring;
}

template <int HD, int GRP, int ACT, int NW, int TT, int NS, bool GM>
__global__ void __launch_bounds__(NW * 32, 1) k_attn_dec(AttnArgs a) {
  using TL = DecTile<HD, TT>;
  constexpr int KS = HD / 16, PR = HD / 8, PER = HD / 32;
  constexpr int PF = NS > 1 ? NS - 1 : 1;  // tiles a warp has in flight before its first wait
  static_assert(GRP <= 8, "one m16n8 tile holds at most 8 heads per kv head");
  extern __shared__ __align__(16) unsigned char sm[];
  int cs, sp;
  if (GM) {
    cs = (int)gridDim.x;
    sp = (int)blockIdx.x;
  } else {
    cg::cluster_group cl = cg::this_cluster();
    cs = (int)cl.num_blocks();
    sp = (int)cl.block_rank();
  }
  const int g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const bool last = sp == cs - 1;

  // The token sits at position p = len[b] (advanced by the previous step's
  // LM-head kernel, final here); positions < p were written by earlier steps.
  const int p = a.len[b];
  const int ntile = (p + TT - 1) / TT;
  const int per = (ntile + cs - 1) / cs;
  const int tb = min(ntile, sp * per), te = min(ntile, tb + per);
  const int nmine = te - tb > warp ? (te - tb - warp + NW - 1) / NW : 0;  // tiles tb + warp + NW * i
  const uint16_t *Kb = a.kv.base + a.kv.idx(a.layer, 0, b, g, 0);
  const uint16_t *Vb = a.kv.base + a.kv.idx(a.layer, 1, b, g, 0);
  const unsigned ring = (unsigned)__cvta_generic_to_shared(sm) + warp * NS * TL::BYTES;

  // the warp's i-th tile into ring slot i % NS: 32 K rows then 32 V rows,
  // rows past p zero-filled (their scores are masked; zero V keeps P V finite)
  auto issue = [&](int i) {
    if (i < nmine) {
      const int t0 = (tb + warp + NW * i) * TT, n = min(TT, p - t0);
      const unsigned st = ring + (i % NS) * TL::BYTES;
#pragma unroll 4
      for (int v = lane; v < 2 * TT * PR; v += 32) {
        const int kv = v >= TT * PR, rem = v - kv * TT * PR, t = rem / PR, c = rem % PR;
        const bool ok = t < n;
        const uint16_t *src = (kv ? Vb : Kb) + (size_t)(t0 + (ok ? t : 0)) * HD + c * 8;
        cp16z(st + (kv * TT + t) * TL::ROW + c * 16, src, ok);
      }
    }
    cp_commit();
  };
#pragma unroll
  for (int i = 0; i < PF; ++i) issue(i);

  pdl_wait();
  pdl_trigger();

  // K/V of position p (written by the QKV kernel this kernel follows), for
  // the last split: loaded now so the round trip overlaps the tile loop
  float kp[PER], vp[PER];
  if (last) {
    const uint16_t *kc = Kb + (size_t)p * HD, *vc = Vb + (size_t)p * HD;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      kp[r] = act_to_f(kc[lane + 32 * r], ACT);
      vp[r] = act_to_f(vc[lane + 32 * r], ACT);
    }
  }

  // q of the kv head's GRP query heads as the A fragments of S = q K^T
  // (row gq = head; rows 8..15 and heads >= GRP are zero; q is act-rounded
  // after RoPE, so the 16-bit pairs are exact)
  const float *qb = a.q + ((size_t)b * a.H + (size_t)g * GRP) * HD;
  uint32_t qa[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    qa[ks][0] = qa[ks][1] = qa[ks][2] = qa[ks][3] = 0u;
    if (gq < GRP) {
      const float2 lo = *reinterpret_cast<const float2 *>(qb + gq * HD + 16 * ks + 2 * tq);
      const float2 hi = *reinterpret_cast<const float2 *>(qb + gq * HD + 16 * ks + 8 + 2 * tq);
      qa[ks][0] = pack_act2(lo.x, lo.y, ACT);
      qa[ks][2] = pack_act2(hi.x, hi.y, ACT);
    }
  }
  const float sl2 = 1.4426950408889634f / sqrtf((float)HD);

  // softmax state of head gq (the same in the 4 lanes of a quad) and O^T
  // fragments: o[mt] = rows (dims) 16 mt + gq (+8) x columns (heads) 2 tq, 2 tq + 1
  float mrun = -INFINITY, lrun = 0.f;
  float o[KS][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  for (int i = 0; i < nmine; ++i) {
    if (NS > 1) {
      cp_wait<(NS > 1 ? NS - 2 : 0)>();
      __syncwarp();  // every lane's copies of tile i landed; slot (i - 1) % NS is free
      issue(i + NS - 1);
    } else {
      cp_wait<0>();
      __syncwarp();
    }
    const unsigned kt = ring + (i % NS) * TL::BYTES, vt = kt + TT * TL::ROW;
    const int n = min(TT, p - (tb + warp + NW * i) * TT);

    // S[head][t] for the tile's TT positions: n-tiles of 8
    constexpr int NT = TT / 8, KK = TT / 16;  // n-tiles of 8 positions, k-steps of 16
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kp2 = 0; kp2 < KS / 2; ++kp2) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint32_t kb[4];  // dims 32 kp2 + 8j of positions 8 nt + 0..7, j = 0..3
        ldsm_x4(kb, kt + (8 * nt + (lane & 7)) * TL::ROW + (32 * kp2 + 8 * (lane >> 3)) * 2);
        mma16816<ACT>(s[nt], qa[2 * kp2], kb);
        mma16816<ACT>(s[nt], qa[2 * kp2 + 1], kb + 2);
      }
    }
    // online softmax of head gq over positions 8 nt + 2 tq + {0, 1}
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float v = 8 * nt + 2 * tq + j < n ? s[nt][j] * sl2 : -INFINITY;
        s[nt][j] = v;
        mx = fmaxf(mx, v);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mnew = fmaxf(mrun, mx);  // finite: the tile has a position < p
    const float corr = exp2f(mrun - mnew);
    uint32_t ph[KK][2], pl[KK][2];  // P^T as B fragments: k-step kk = positions 16 kk + ...
    float ls = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float p0 = exp2f(s[nt][0] - mnew), p1 = exp2f(s[nt][1] - mnew);
      ls += p0 + p1;
      const uint32_t hw = pack_act2(p0, p1, ACT);
      ph[nt >> 1][nt & 1] = hw;
      pl[nt >> 1][nt & 1] = pack_act2(p0 - act_to_f((uint16_t)(hw & 0xffffu), ACT),
                                      p1 - act_to_f((uint16_t)(hw >> 16), ACT), ACT);
    }
    ls += __shfl_xor_sync(0xffffffffu, ls, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    lrun = fmaf(lrun, corr, ls);
    mrun = mnew;
    // rescale O^T: its columns are heads 2 tq and 2 tq + 1, whose factors sit
    // in quads 2 tq and 2 tq + 1
    const float ca = __shfl_sync(0xffffffffu, corr, 8 * tq), cb = __shfl_sync(0xffffffffu, corr, 8 * tq + 4);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      o[mt][0] *= ca;
      o[mt][1] *= cb;
      o[mt][2] *= ca;
      o[mt][3] *= cb;
    }
    // O^T += V^T P^T
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int kk = 0; kk < KK; ++kk) {
        uint32_t va[4];  // V^T rows 16 mt + 0..15 x positions 16 kk + 0..15
        ldsm_x4_t(va, vt + (16 * kk + 8 * (lane >> 4) + (lane & 7)) * TL::ROW + (16 * mt + 8 * ((lane >> 3) & 1)) * 2);
        mma16816<ACT>(o[mt], va, ph[kk]);
        mma16816<ACT>(o[mt], va, pl[kk]);
      }
    if (NS == 1) {
      __syncwarp();  // every lane is done with the slot before it is refilled
      issue(i + 1);
    }
  }
  cp_wait<0>();
  __syncthreads();  // every warp is done with its ring: the merge reuses it

  float *part = reinterpret_cast<float *>(sm);
  float *wpo = part + GRP * HD;
  float *pm = wpo + NW * GRP * HD;
  float *wml = pm + 2 * GRP;
  float *sps = wml + NW * GRP * 2;
  float *spv = sps + GRP;
  float *gml = spv + HD;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    const int d = 16 * mt + gq, h0 = 2 * tq, h1 = 2 * tq + 1;
    if (h0 < GRP) {
      wpo[(warp * GRP + h0) * HD + d] = o[mt][0];
      wpo[(warp * GRP + h0) * HD + d + 8] = o[mt][2];
    }
    if (h1 < GRP) {
      wpo[(warp * GRP + h1) * HD + d] = o[mt][1];
      wpo[(warp * GRP + h1) * HD + d + 8] = o[mt][3];
    }
  }
  if (tq == 0 && gq < GRP) {
    wml[(warp * GRP + gq) * 2] = mrun;
    wml[(warp * GRP + gq) * 2 + 1] = lrun;
  }
  if (last) {
    for (int hh = warp; hh < GRP; hh += NW) {
      float d = 0.f;
#pragma unroll
      for (int r = 0; r < PER; ++r) d = fmaf(qb[hh * HD + lane + 32 * r], kp[r], d);
      d = warp_sum(d);
      if (lane == 0) sps[hh] = d * sl2;
    }
    if (warp == 0) {
#pragma unroll
      for (int r = 0; r < PER; ++r) spv[lane + 32 * r] = vp[r];
    }
  }
  __syncthreads();

  // the block's state per head: its warps, plus position p in the last split
  for (int it = tid; it < GRP * HD; it += NW * 32) {
    const int h = it / HD, d = it - h * HD;
    float M = last ? sps[h] : -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wml[(w * GRP + h) * 2]);
    float acc = 0.f, Ls = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = wml[(w * GRP + h) * 2];
      const float wt = mw == -INFINITY ? 0.f : exp2f(mw - M);
      acc = fmaf(wt, wpo[(w * GRP + h) * HD + d], acc);
      Ls = fmaf(wt, wml[(w * GRP + h) * 2 + 1], Ls);
    }
    if (last) {
      const float wt = exp2f(sps[h] - M);
      acc = fmaf(wt, spv[d], acc);
      Ls += wt;
    }
    part[h * HD + d] = acc;
    if (d == 0) {
      pm[2 * h] = M;
      pm[2 * h + 1] = Ls;
    }
  }

  float *out = a.o + ((size_t)b * a.H + (size_t)g * GRP) * HD;
  if (GM) {
    __syncthreads();
    if (cs == 1) {  // the only split: the block's state is the result
      for (int it = tid; it < GRP * HD; it += NW * 32)
        out[it] = round_act(part[it] / pm[2 * (it / HD) + 1], ACT);
      return;
    }
    // publish (O, max, sum) of this split; the last block of (row, kv head)
    // to arrive merges every split's state
    float *gp = a.part + ((size_t)(b * a.Hkv + g) * cs) * GRP * (HD + 2);
    for (int it = tid; it < GRP * HD; it += NW * 32) {
      const int h = it / HD, d = it - h * HD;
      gp[((size_t)sp * GRP + h) * (HD + 2) + d] = part[it];
    }
    if (tid < 2 * GRP) gp[((size_t)sp * GRP + tid / 2) * (HD + 2) + HD + (tid & 1)] = pm[tid];
    __threadfence();
    __syncthreads();
    int *flag = reinterpret_cast<int *>(gml + cs * GRP * 2);
    if (tid == 0) {
      unsigned *ctr = a.counter + b * a.Hkv + g;
      const unsigned t = atomicAdd(ctr, 1u);
      const int am_last = t == (unsigned)(cs - 1);
      if (am_last) *ctr = 0u;  // left at zero for the next launch
      *flag = am_last;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    for (int it = tid; it < cs * GRP * 2; it += NW * 32)
      gml[it] = __ldcg(gp + (size_t)(it >> 1) * (HD + 2) + HD + (it & 1));
    __syncthreads();
    for (int it = tid; it < GRP * HD; it += NW * 32) {
      const int h = it / HD, d = it - h * HD;
      float M = -INFINITY;
      for (int s2 = 0; s2 < cs; ++s2) M = fmaxf(M, gml[(s2 * GRP + h) * 2]);
      float acc = 0.f, Ls = 0.f;
      for (int s2 = 0; s2 < cs; ++s2) {
        const float ms = gml[(s2 * GRP + h) * 2];
        const float wt = ms == -INFINITY ? 0.f : exp2f(ms - M);
        acc = fmaf(wt, __ldcg(gp + ((size_t)s2 * GRP + h) * (HD + 2) + d), acc);
        Ls = fmaf(wt, gml[(s2 * GRP + h) * 2 + 1], Ls);
      }
      out[it] = round_act(acc / Ls, ACT);
    }
    return;
  } else {
    // merge across the cluster: split sp combines dims [sp * HD / cs, ...) of
    // every head.  Lane l < HD / 4 reads split r = l % cs (its max, sum and 4
    // dims of O, from that block's shared memory), so all the remote loads
    // are in flight at once, and the cs lanes of a 4-dim block combine by
    // shuffles.
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();
    for (int hh = warp; hh < GRP; hh += NW) {
      const int dpc = HD / cs, r = lane % cs, d0 = sp * dpc + (lane / cs) * 4;
      const bool live = lane < HD / 4;
      float m = -INFINITY, l = 0.f;
      float4 ov = make_float4(0.f, 0.f, 0.f, 0.f);
      if (live) {
        const float *rp = cl.map_shared_rank(part, r);
        const float *rm = cl.map_shared_rank(pm, r);
        m = rm[hh * 2];
        l = rm[hh * 2 + 1];
        ov = *reinterpret_cast<const float4 *>(rp + hh * HD + d0);
      }
      float M = m;
      for (int x = 1; x < cs; x <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
      const float w = m == -INFINITY ? 0.f : exp2f(m - M);
      float Ls = w * l, o0 = w * ov.x, o1 = w * ov.y, o2 = w * ov.z, o3 = w * ov.w;
      for (int x = 1; x < cs; x <<= 1) {
        Ls += __shfl_xor_sync(0xffffffffu, Ls, x);
        o0 += __shfl_xor_sync(0xffffffffu, o0, x);
        o1 += __shfl_xor_sync(0xffffffffu, o1, x);
        o2 += __shfl_xor_sync(0xffffffffu, o2, x);
        o3 += __shfl_xor_sync(0xffffffffu, o3, x);
      }
      if (live && r == 0) {
        const float inv = 1.0f / Ls;
        float *dst = out + hh * HD + d0;
        dst[0] = round_act(o0 * inv, ACT);
        dst[1] = round_act(o1 * inv, ACT);
        dst[2] = round_act(o2 * inv, ACT);
        dst[3] = round_act(o3 * inv, ACT);
      }
    }
    cl.sync();  // every split's partials stay readable until all merges are done
  }
}

// Short-context launches whose blocks all fit two per SM reserve this much
// shared memory per block, so that at most two share an SM: the splits
// spread over twice as many SMs as at three per SM (8B decode step: tau
// 503 -> 515 tokens/s; one block per SM is slower again: clusters of 16
// then need 16 free SMs in one GPC).
constexpr size_t kDecSpreadSmem = 80 * 1024;

static int device_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n < 1) n = 1;
  }
  return n;
}

template <int HD, int GRP, int ACT, int NW, int TT, int NS, bool GM>
static cudaError_t launch_dec(const AttnArgs &a, int B, int cs, cudaStream_t s, int pdl) {
  auto fn = k_attn_dec<HD, GRP, ACT, NW, TT, NS, GM>;
  size_t smem = dec_smem<HD, NW, TT, NS>(GRP);
  if (!GM && (long)cs * a.Hkv * B <= 2L * device_sms() && smem < kDecSpreadSmem) smem = kDecSpreadSmem;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && !GM && cs > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, a.Hkv, B);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (!GM) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cs;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  e = cudaLaunchKernelEx(&cfg, fn, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Launch plan of the decode attention for B rows whose longest context is
// pmax positions: clusters of splits while each warp of a split has at most
// one tile, or while the rows alone fill the GPU (B x Hkv >= n_sm / 2: small
// blocks, many resident per SM) (returns 0, *splits = cluster size); else
// about one block per SM per (row, kv head) split, merged through global
// memory (returns 1, *splits = blocks per (row, kv head), at most
// max_splits).
int attn_dec_plan(int B, int Hkv, int n_sm, int max_cluster, int max_splits, int pmax, int *splits) {
  int cs = 1;
  while (2 * cs <= max_cluster && 2 * cs * Hkv * B <= 2 * n_sm) cs *= 2;
  const int ntile = (pmax + DTT - 1) / DTT;
  int S = n_sm / (Hkv * B);
  if ((ntile + cs - 1) / cs <= DNW || S < 2) {
    *splits = cs;
    return 0;
  }
  if (S > max_splits) S = max_splits;
  if (S > kAttnMaxSplits) S = kAttnMaxSplits;
  if (S < 1) S = 1;
  *splits = S;
  return 1;
}

// Largest cluster size (power of two, <= 16) the decode attention can be
// launched with on this device; 0 if none.
int attn_dec_max_cluster(int hd, int grp, int act) {
  for (int cs = 16; cs >= 1; cs >>= 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(DNW * 32);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaErrorInvalidValue;
#define RV_DQ(HD_, G_, A_)                                                                                   \
  if (hd == HD_ && grp == G_ && act == A_) {                                                                 \
    auto fn = k_attn_dec<HD_, G_, A_, DNW, DTT, 1, false>;                                                   \
    cfg.dynamicSmemBytes = dec_smem<HD_, DNW, DTT, 1>(G_) > kDecSpreadSmem ? dec_smem<HD_, DNW, DTT, 1>(G_) : kDecSpreadSmem; \
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.dynamicSmemBytes);    \
    if (e == cudaSuccess && cs > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1); \
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);                                  \
  }
    RV_DQ(64, 1, 0) RV_DQ(64, 2, 0) RV_DQ(64, 4, 0) RV_DQ(64, 8, 0)
    RV_DQ(128, 1, 0) RV_DQ(128, 2, 0) RV_DQ(128, 4, 0) RV_DQ(128, 8, 0)
    RV_DQ(64, 1, 1) RV_DQ(64, 2, 1) RV_DQ(64, 4, 1) RV_DQ(64, 8, 1)
    RV_DQ(128, 1, 1) RV_DQ(128, 2, 1) RV_DQ(128, 4, 1) RV_DQ(128, 8, 1)
#undef RV_DQ
    if (e == cudaSuccess && n > 0) return cs;
    cudaGetLastError();
  }
  return 0;
}

// ---- prefill: causal flash attention on the tensor pipe --------------------
// Block: 16 consecutive tokens of sequence b x the GRP query heads of kv head
// g (one warp per head), so each K/V tile serves GRP heads.  K/V tiles of 64
// positions stream through a double-buffered cp.async ring, rows padded by 16
// bytes so ldmatrix reads are conflict-free; positions past the causal bound
// are zero-filled.  S = Q K^T and O += P V run as mma.sync m16n8k16 with
// 16-bit operands and fp32 accumulators; the online softmax is fp32, and P
// enters the P V product as two 16-bit terms, P = hi + lo with hi = round16(P)
// and lo = round16(P - hi), so the product keeps about 16 significant bits
// of P.  Blocks are issued longest-first (last tokens first).
constexpr int PQ = 16;  // tokens per block (one m16 tile per warp)
constexpr int PK = 64;  // key positions per tile

template <int HD>
struct PreTile {
  static constexpr int ROW = HD * 2 + 16;
  static constexpr int KV = PK * ROW;
  static constexpr int BYTES = 2 * KV;
};

template <int HD, int GRP, int ACT>
__global__ void __launch_bounds__(GRP * 32) k_attn_prefill(AttnRowsArgs a, int T) {
  using PT = PreTile<HD>;
  constexpr int NT = GRP * 32, KS = HD / 16, DT = HD / 8, PR = HD / 8;
  extern __shared__ __align__(16) unsigned char sm[];
  const int b = blockIdx.z, g = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = g * GRP + warp, gq = lane >> 2, tq = lane & 3;
  const int base = a.base ? a.base[b] : 0;
  const int t0 = (gridDim.x - 1 - blockIdx.x) * PQ;  // first token of the block
  const int kend = base + min(T, t0 + PQ);           // keys [0, kend)
  const int ntile = (kend + PK - 1) / PK;
  const uint16_t *Kb = a.kv.base + a.kv.idx(a.layer, 0, b, g, 0);
  const uint16_t *Vb = a.kv.base + a.kv.idx(a.layer, 1, b, g, 0);
  const unsigned sb = (unsigned)__cvta_generic_to_shared(sm);

  auto issue = [&](int tile, int slot) {
    if (tile < ntile) {
      const int j0 = tile * PK;
      const unsigned st = sb + slot * PT::BYTES;
      for (int v = tid; v < 2 * PK * PR; v += NT) {
        const int kv = v >= PK * PR, rem = v - kv * PK * PR, j = rem / PR, c = rem - j * PR;
        const bool ok = j0 + j < kend;
        const uint16_t *src = (kv ? Vb : Kb) + (size_t)(ok ? j0 + j : 0) * HD + c * 8;
        cp16z(st + kv * PT::KV + j * PT::ROW + c * 16, src, ok);
      }
    }
    cp_commit();
  };
  issue(0, 0);

  // Q fragments (A operand: rows = the warp's 16 tokens, k = head dims)
  const int r0 = t0 + gq, r1 = r0 + 8;
  uint32_t qa[KS][4];
  {
    const size_t ld = (size_t)a.H * HD;
    const float *q0 = a.q + ((size_t)b * T + r0) * ld + (size_t)h * HD;
    const float *q1 = a.q + ((size_t)b * T + r1) * ld + (size_t)h * HD;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d = 16 * ks + 2 * tq;
      float2 x00 = make_float2(0.f, 0.f), x10 = x00, x01 = x00, x11 = x00;
      if (r0 < T) { x00 = *reinterpret_cast<const float2 *>(q0 + d); x01 = *reinterpret_cast<const float2 *>(q0 + d + 8); }
      if (r1 < T) { x10 = *reinterpret_cast<const float2 *>(q1 + d); x11 = *reinterpret_cast<const float2 *>(q1 + d + 8); }
      qa[ks][0] = pack_act2(x00.x, x00.y, ACT);
      qa[ks][1] = pack_act2(x10.x, x10.y, ACT);
      qa[ks][2] = pack_act2(x01.x, x01.y, ACT);
      qa[ks][3] = pack_act2(x11.x, x11.y, ACT);
    }
  }
  const int p0 = base + r0, p1 = base + r1;  // positions of the thread's two rows
  const float sl2 = 1.4426950408889634f / sqrtf((float)HD);  // softmax in base 2
  float o[DT][4];
#pragma unroll
  for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int tile = 0; tile < ntile; ++tile) {
    cp_wait<0>();
    __syncthreads();  // tile in; every warp is done with the other slot
    issue(tile + 1, (tile + 1) & 1);
    const unsigned kt = sb + (tile & 1) * PT::BYTES, vt = kt + PT::KV;
    const int j0 = tile * PK;
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    const int mi = lane >> 3;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t kb[4];
        ldsm_x4(kb, kt + (16 * np + (mi >> 1) * 8 + (lane & 7)) * PT::ROW + (16 * ks + (mi & 1) * 8) * 2);
        mma16816<ACT>(sc[2 * np], qa[ks], kb);
        mma16816<ACT>(sc[2 * np + 1], qa[ks], kb + 2);
      }
    // scale, causal mask, online softmax (rows p0: elements 0,1; p1: 2,3)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int k0 = j0 + nt * 8 + 2 * tq;
      sc[nt][0] = k0 <= p0 ? sc[nt][0] * sl2 : -INFINITY;
      sc[nt][1] = k0 + 1 <= p0 ? sc[nt][1] * sl2 : -INFINITY;
      sc[nt][2] = k0 <= p1 ? sc[nt][2] * sl2 : -INFINITY;
      sc[nt][3] = k0 + 1 <= p1 ? sc[nt][3] * sl2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);  // finite: key 0 is in the first tile
    const float c0 = exp2f(m0 - n0), c1 = exp2f(m1 - n1);
    float s0 = 0.f, s1 = 0.f;
    uint32_t pa[4][4], pl[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float e0 = exp2f(sc[nt][0] - n0), e1 = exp2f(sc[nt][1] - n0);
      const float e2 = exp2f(sc[nt][2] - n1), e3 = exp2f(sc[nt][3] - n1);
      s0 += e0 + e1;
      s1 += e2 + e3;
      const float h0 = round_act(e0, ACT), h1 = round_act(e1, ACT), h2 = round_act(e2, ACT), h3 = round_act(e3, ACT);
      pa[nt >> 1][(nt & 1) * 2] = pack_act2(h0, h1, ACT);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_act2(h2, h3, ACT);
      pl[nt >> 1][(nt & 1) * 2] = pack_act2(e0 - h0, e1 - h1, ACT);
      pl[nt >> 1][(nt & 1) * 2 + 1] = pack_act2(e2 - h2, e3 - h3, ACT);
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    l0 = l0 * c0 + s0;
    l1 = l1 * c1 + s1;
    m0 = n0;
    m1 = n1;
#pragma unroll
    for (int i = 0; i < DT; ++i) {
      o[i][0] *= c0; o[i][1] *= c0; o[i][2] *= c1; o[i][3] *= c1;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int dp = 0; dp < DT / 2; ++dp) {
        uint32_t vb[4];
        ldsm_x4_t(vb, vt + (16 * kk + (mi & 1) * 8 + (lane & 7)) * PT::ROW + (16 * dp + (mi >> 1) * 8) * 2);
        mma16816<ACT>(o[2 * dp], pa[kk], vb);
        mma16816<ACT>(o[2 * dp + 1], pa[kk], vb + 2);
        mma16816<ACT>(o[2 * dp], pl[kk], vb);
        mma16816<ACT>(o[2 * dp + 1], pl[kk], vb + 2);
      }
  }
  cp_wait<0>();

  const size_t ld = (size_t)a.H * HD;
  const float i0 = 1.0f / l0, i1 = 1.0f / l1;
#pragma unroll
  for (int i = 0; i < DT; ++i) {
    const int d = 8 * i + 2 * tq;
    if (r0 < T)
      *reinterpret_cast<float2 *>(a.o + ((size_t)b * T + r0) * ld + (size_t)h * HD + d) =
          make_float2(round_act(o[i][0] * i0, ACT), round_act(o[i][1] * i0, ACT));
    if (r1 < T)
      *reinterpret_cast<float2 *>(a.o + ((size_t)b * T + r1) * ld + (size_t)h * HD + d) =
          make_float2(round_act(o[i][2] * i1, ACT), round_act(o[i][3] * i1, ACT));
  }
}

template <int HD, int GRP, int ACT>
static cudaError_t launch_pre(const AttnRowsArgs &a, int B, int T, cudaStream_t s) {
  auto fn = k_attn_prefill<HD, GRP, ACT>;
  const int smem = 2 * PreTile<HD>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((T + PQ - 1) / PQ, a.Hkv, B);
  fn<<<grid, GRP * 32, smem, s>>>(a, T);
  return cudaGetLastError();
}

template <int HD, int GRP>
static cudaError_t launch_hg(const AttnArgs &a, int T_per_row, const int32_t *base, int rows, cudaStream_t s,
                             int pdl) {
  dim3 grid(rows, a.splits, a.Hkv);
  return launch_k(k_attn<HD, GRP>, grid, dim3(GRP * 32), 0, s, pdl, a, T_per_row, base, rows);
}

static cudaError_t launch_any(const AttnArgs &a, int T_per_row, const int32_t *base, int rows, cudaStream_t s,
                              int pdl = 0) {
  const int grp = a.H / a.Hkv;
#define RV_ATT(HD_, G_) \
  if (a.hd == HD_ && grp == G_) return launch_hg<HD_, G_>(a, T_per_row, base, rows, s, pdl);
  RV_ATT(64, 1) RV_ATT(64, 2) RV_ATT(64, 4) RV_ATT(64, 8)
  RV_ATT(128, 1) RV_ATT(128, 2) RV_ATT(128, 4) RV_ATT(128, 8)
#undef RV_ATT
  return cudaErrorInvalidValue;
}

// Decode: one row per batch entry, the token at position len[b].
// a.global_merge = 0: a.splits is the cluster size (a power of two <= 16 that
// attn_dec_max_cluster allows); 1: a.splits blocks per (row, kv head),
// 1..kAttnMaxSplits, merged through a.part / a.counter.
cudaError_t launch_attn_decode(const AttnArgs &a, int B, cudaStream_t s, int pdl) {
  const int grp = a.H / a.Hkv, cs = a.splits;
  if (a.global_merge) {
    if (cs < 1 || cs > kAttnMaxSplits) return cudaErrorInvalidValue;
  } else if (cs < 1 || cs > 16 || (cs & (cs - 1))) {
    return cudaErrorInvalidValue;
  }
#define RV_DL(HD_, G_)                                                                                   \
  if (a.hd == HD_ && grp == G_) {                                                                        \
    constexpr int NSL = long_slots<HD_>();                                                               \
    if (a.global_merge)                                                                                  \
      return a.act == 1 ? launch_dec<HD_, G_, 1, LNW, LTT, NSL, true>(a, B, cs, s, pdl)                  \
                        : launch_dec<HD_, G_, 0, LNW, LTT, NSL, true>(a, B, cs, s, pdl);                 \
    return a.act == 1 ? launch_dec<HD_, G_, 1, DNW, DTT, 1, false>(a, B, cs, s, pdl)                     \
                      : launch_dec<HD_, G_, 0, DNW, DTT, 1, false>(a, B, cs, s, pdl);                    \
  }
  RV_DL(64, 1) RV_DL(64, 2) RV_DL(64, 4) RV_DL(64, 8)
  RV_DL(128, 1) RV_DL(128, 2) RV_DL(128, 4) RV_DL(128, 8)
#undef RV_DL
  return cudaErrorInvalidValue;
}

// Prefill / general rows: T tokens per sequence starting at base (NULL = 0),
// max_rows = B * T rows.  Token rows (T > 1) run the tensor-pipe flash
// attention; the per-row kernel remains for list-driven rows.
cudaError_t launch_attn_rows(const AttnRowsArgs &r, int max_rows, cudaStream_t s) {
  const int T = r.tokens_per_row, grp = r.H / r.Hkv;
  if (T > 1 && !r.list && max_rows % T == 0) {
    const int B = max_rows / T;
#define RV_PL(HD_, G_)                                                                    \
    if (r.hd == HD_ && grp == G_)                                                         \
      return r.act == 1 ? launch_pre<HD_, G_, 1>(r, B, T, s) : launch_pre<HD_, G_, 0>(r, B, T, s);
    RV_PL(64, 1) RV_PL(64, 2) RV_PL(64, 4) RV_PL(64, 8)
    RV_PL(128, 1) RV_PL(128, 2) RV_PL(128, 4) RV_PL(128, 8)
#undef RV_PL
  }
  AttnArgs a;
  a.kv = r.kv;
  a.layer = r.layer; a.H = r.H; a.Hkv = r.Hkv; a.hd = r.hd; a.act = r.act;
  a.q = r.q; a.o = r.o; a.len = nullptr; a.splits = 1; a.part = nullptr; a.counter = nullptr;
  return launch_any(a, r.tokens_per_row, r.base, max_rows, s);
}

}  // namespace rv
