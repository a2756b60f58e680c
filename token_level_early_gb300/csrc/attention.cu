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
// thread-block cluster.  Each split streams its share of the past positions
// 0..p-1 (final before the step starts) through a shared-memory ring that it
// fills before the programmatic-dependent-launch wait; only q and the K/V of
// position p come from the QKV kernel it follows.  A split whose tiles all
// fit the ring takes its scores in one pass and one max/sum; longer ones use
// the online softmax.  The splits merge their softmax states through
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

// ---- decode: clustered split-KV attention ----------------------------------
constexpr int DTT = 32;   // positions per tile (one per lane in the score pass)
constexpr int DNST = 5;   // ring stages: a split of up to DNST - 1 tiles is in flight before the wait

template <int HD>
struct DecTile {
  static constexpr int KROW = HD * 2 + 16;  // padded K row: lane-per-row 16-byte reads hit distinct banks
  static constexpr int VROW = HD * 2;
  static constexpr int BYTES = DTT * (KROW + VROW);
};

template <int HD>
static size_t dec_smem(int grp) {
  return (size_t)DNST * DecTile<HD>::BYTES + sizeof(float) * grp * (HD + 2) + sizeof(float) * grp * DNST * DTT;
}

// q . K[row] for one position: the lane's K row (16-bit, padded) against q as
// 16-bit pairs, mixed-precision FMAs into four fp32 partial sums.
template <int HD, int ACT>
__device__ __forceinline__ float k_dot_q(const unsigned char *krow, const uint32_t *qr) {
  const uint4 *kr = reinterpret_cast<const uint4 *>(krow);
  float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
  for (int j = 0; j < HD / 8; ++j) {
    const uint4 k = kr[j];
    d0 = fma_lo16<ACT>(k.x, qr[4 * j], d0);
    d1 = fma_hi16<ACT>(k.x, qr[4 * j], d1);
    d2 = fma_lo16<ACT>(k.y, qr[4 * j + 1], d2);
    d3 = fma_hi16<ACT>(k.y, qr[4 * j + 1], d3);
    d0 = fma_lo16<ACT>(k.z, qr[4 * j + 2], d0);
    d1 = fma_hi16<ACT>(k.z, qr[4 * j + 2], d1);
    d2 = fma_lo16<ACT>(k.w, qr[4 * j + 3], d2);
    d3 = fma_hi16<ACT>(k.w, qr[4 * j + 3], d3);
  }
  return (d0 + d1) + (d2 + d3);
}

// o[r] += sum over the tile's first n positions t of p[t] * V[t][lane * PER + r],
// p broadcast from shared memory (all lanes read the same word); full tiles
// unrolled with two accumulator sets to halve the dependent FMA chains.
template <int HD, int ACT>
__device__ __forceinline__ void v_accumulate(const unsigned char *tv, const float *pw, int n, int lane, float *o) {
  constexpr int PER = HD / 32, VROW = HD * 2;
  if (n == DTT) {
    float e[PER];
#pragma unroll
    for (int r = 0; r < PER; ++r) e[r] = 0.f;
#pragma unroll
    for (int t = 0; t < DTT; t += 2) {
      const float p0 = pw[t], p1 = pw[t + 1];
      const uint16_t *v0 = reinterpret_cast<const uint16_t *>(tv + t * VROW) + lane * PER;
      const uint16_t *v1 = v0 + HD;
#pragma unroll
      for (int r = 0; r < PER; ++r) {
        o[r] = fmaf(p0, act_to_f(v0[r], ACT), o[r]);
        e[r] = fmaf(p1, act_to_f(v1[r], ACT), e[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < PER; ++r) o[r] += e[r];
  } else {
    for (int t = 0; t < n; ++t) {
      const float pt = pw[t];
      const uint16_t *vr = reinterpret_cast<const uint16_t *>(tv + t * VROW) + lane * PER;
#pragma unroll
      for (int r = 0; r < PER; ++r) o[r] = fmaf(pt, act_to_f(vr[r], ACT), o[r]);
    }
  }
}

__device__ __forceinline__ uint32_t pack_act2(float lo, float hi, int act) {
  return (uint32_t)f_to_act(lo, act) | ((uint32_t)f_to_act(hi, act) << 16);
}

template <int HD, int GRP, int ACT>
__global__ void __launch_bounds__(GRP * 32, 1) k_attn_dec(AttnArgs a) {
  using TL = DecTile<HD>;
  constexpr int NT = GRP * 32, PER = HD / 32, PR = HD / 8;
  extern __shared__ __align__(16) unsigned char sm[];
  // per head: o [GRP][HD], then (running max, sum) [GRP][2]
  float *part = reinterpret_cast<float *>(sm + DNST * TL::BYTES);
  float *pbuf = part + GRP * (HD + 2);  // [GRP][DNST * DTT]: softmax numerators of the warp's positions
  cg::cluster_group cl = cg::this_cluster();
  const int cs = (int)cl.num_blocks(), sp = (int)cl.block_rank();
  const int g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // The token sits at position p = len[b] (advanced by the previous step's
  // LM-head kernel, final here); positions < p were written by earlier steps.
  const int p = a.len[b];
  const int ntile = (p + DTT - 1) / DTT;
  const int per = (ntile + cs - 1) / cs;
  const int tb = min(ntile, sp * per), te = min(ntile, tb + per);
  const uint16_t *Kb = a.kv.base + a.kv.idx(a.layer, 0, b, g, 0);
  const uint16_t *Vb = a.kv.base + a.kv.idx(a.layer, 1, b, g, 0);
  const unsigned sbase = (unsigned)__cvta_generic_to_shared(sm);

  auto issue = [&](int tile, int slot) {
    if (tile < te) {
      const int t0 = tile * DTT, n = min(DTT, p - t0);
      const unsigned st = sbase + slot * TL::BYTES;
      for (int v = tid; v < 2 * DTT * PR; v += NT) {
        const int kv = v >= DTT * PR, rem = v - kv * DTT * PR, t = rem / PR, c = rem - t * PR;
        if (t < n) {
          const uint16_t *src = (kv ? Vb : Kb) + (size_t)(t0 + t) * HD + c * 8;
          cp16s(st + (kv ? DTT * TL::KROW + t * TL::VROW : t * TL::KROW) + c * 16, src);
        }
      }
    }
    cp_commit();
  };
#pragma unroll
  for (int i = 0; i < DNST - 1; ++i) issue(tb + i, i);

  pdl_wait();
  pdl_trigger();

  // K/V of position p itself (written by the QKV kernel this kernel follows),
  // folded in by the last split after its tiles: loaded now, with q, so the
  // round trip overlaps the tile loop
  float kp[PER], vp[PER];
  if (sp == cs - 1) {
    const uint16_t *kc = Kb + (size_t)p * HD + lane * PER, *vc = Vb + (size_t)p * HD + lane * PER;
#pragma unroll
    for (int r = 0; r < PER; ++r) {
      kp[r] = act_to_f(kc[r], ACT);
      vp[r] = act_to_f(vc[r], ACT);
    }
  }

  // q of head h as 16-bit pairs (q is act-rounded after RoPE: exact)
  const int h = g * GRP + warp;
  const float *qp = a.q + ((size_t)b * a.H + h) * HD;
  uint32_t qr[HD / 2];
#pragma unroll
  for (int i = 0; i < HD / 4; ++i) {
    const float4 v = *reinterpret_cast<const float4 *>(qp + 4 * i);
    qr[2 * i] = pack_act2(v.x, v.y, ACT);
    qr[2 * i + 1] = pack_act2(v.z, v.w, ACT);
  }
  const float scale = 1.0f / sqrtf((float)HD);
  float mrun = -INFINITY, lrun = 0.f, o[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) o[r] = 0.f;

  if (te - tb <= DNST - 1) {
    // Every tile of this split is in flight since before the wait: scores
    // of all its positions first (lane j takes position j of each tile), one
    // max and one sum, then the V pass with the final numerators.
    cp_wait<0>();
    __syncthreads();
    const int nt = te - tb;
    float sc[DNST - 1];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < DNST - 1; ++i) {
      sc[i] = -INFINITY;
      const int n = i < nt ? min(DTT, p - (tb + i) * DTT) : 0;
      if (lane < n) sc[i] = k_dot_q<HD, ACT>(sm + i * TL::BYTES + lane * TL::KROW, qr) * scale;
      mx = fmaxf(mx, sc[i]);
    }
    mx = warp_max(mx);
    float *pw = pbuf + warp * DNST * DTT;
    float ls = 0.f;
#pragma unroll
    for (int i = 0; i < DNST - 1; ++i) {
      const float pe = sc[i] == -INFINITY ? 0.f : expf(sc[i] - mx);
      pw[i * DTT + lane] = pe;
      ls += pe;
    }
    ls = warp_sum(ls);
    __syncwarp();
    for (int i = 0; i < nt; ++i)
      v_accumulate<HD, ACT>(sm + i * TL::BYTES + DTT * TL::KROW, pw + i * DTT, min(DTT, p - (tb + i) * DTT), lane, o);
    if (nt > 0) {
      mrun = mx;
      lrun = ls;
    }
  } else {
    for (int tile = tb, it = 0; tile < te; ++tile, ++it) {
      cp_wait<DNST - 2>();
      __syncthreads();  // the tile is in; every warp is done with the slot refilled next
      issue(tile + DNST - 1, (it + DNST - 1) % DNST);
      const unsigned char *tk = sm + (it % DNST) * TL::BYTES;
      const unsigned char *tv = tk + DTT * TL::KROW;
      const int n = min(DTT, p - tile * DTT);
      float sc = -INFINITY;
      if (lane < n) sc = k_dot_q<HD, ACT>(tk + lane * TL::KROW, qr) * scale;
      const float mnew = fmaxf(mrun, warp_max(sc));
      const float pe = lane < n ? expf(sc - mnew) : 0.f;
      const float corr = mrun == -INFINITY ? 0.f : expf(mrun - mnew);
      lrun = lrun * corr + warp_sum(pe);
#pragma unroll
      for (int r = 0; r < PER; ++r) o[r] *= corr;
      float *pw = pbuf + warp * DNST * DTT;
      pw[lane] = pe;
      __syncwarp();
      v_accumulate<HD, ACT>(tv, pw, n, lane, o);
      __syncwarp();  // pw is rewritten by the next tile
      mrun = mnew;
    }
  }

  // position p itself (its K/V were written by the QKV kernel this kernel
  // follows): folded in by the last split
  if (sp == cs - 1) {
    float d = 0.f;
#pragma unroll
    for (int r = 0; r < PER; ++r) d = fmaf(qp[lane * PER + r], kp[r], d);
    const float sc = warp_sum(d) * scale;
    const float mnew = fmaxf(mrun, sc);
    const float corr = mrun == -INFINITY ? 0.f : expf(mrun - mnew), pe = expf(sc - mnew);
    lrun = lrun * corr + pe;
#pragma unroll
    for (int r = 0; r < PER; ++r) o[r] = fmaf(pe, vp[r], o[r] * corr);
    mrun = mnew;
  }

  // merge across the cluster: split sp combines dims [sp * HD / cs, ...) of
  // every head.  Warp hh takes head hh; lane l < HD / 4 reads split
  // r = l % cs (its max, sum and 4 dims of o, from that block's shared
  // memory), so all the remote loads are in flight at once, and the cs lanes
  // of a 4-dim block combine by shuffles.
  float *pm = part + GRP * HD;
#pragma unroll
  for (int r = 0; r < PER; ++r) part[warp * HD + lane * PER + r] = o[r];
  if (lane == 0) {
    pm[warp * 2] = mrun;
    pm[warp * 2 + 1] = lrun;
  }
  cl.sync();
  {
    const int dpc = HD / cs, r = lane % cs, d0 = sp * dpc + (lane / cs) * 4;
    const bool live = lane < HD / 4;
    float m = -INFINITY, l = 0.f;
    float4 ov = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
      const float *rp = cl.map_shared_rank(part, r);
      m = rp[GRP * HD + warp * 2];
      l = rp[GRP * HD + warp * 2 + 1];
      ov = *reinterpret_cast<const float4 *>(rp + warp * HD + d0);
    }
    float M = m;
    for (int x = 1; x < cs; x <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
    const float w = m == -INFINITY ? 0.f : expf(m - M);
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
      float *dst = a.o + ((size_t)b * a.H + g * GRP + warp) * HD + d0;
      dst[0] = round_act(o0 * inv, ACT);
      dst[1] = round_act(o1 * inv, ACT);
      dst[2] = round_act(o2 * inv, ACT);
      dst[3] = round_act(o3 * inv, ACT);
    }
  }
  cl.sync();  // every split's partials stay readable until all merges are done
}

template <int HD, int GRP, int ACT>
static cudaError_t launch_dec(const AttnArgs &a, int B, int cs, cudaStream_t s, int pdl) {
  auto fn = k_attn_dec<HD, GRP, ACT>;
  const size_t smem = dec_smem<HD>(GRP);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && cs > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, a.Hkv, B);
  cfg.blockDim = dim3(GRP * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, fn, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Largest cluster size (power of two, <= 16) the decode attention can be
// launched with on this device; 0 if none.
int attn_dec_max_cluster(int hd, int grp, int act) {
  for (int cs = 16; cs >= 1; cs >>= 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(grp * 32);
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
    auto fn = k_attn_dec<HD_, G_, A_>;                                                                       \
    cfg.dynamicSmemBytes = dec_smem<HD_>(G_);                                                                \
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

// Decode: one row per batch entry, the token at position len[b]; a.splits is
// the cluster size (a power of two <= 16 that attn_dec_max_cluster allows).
cudaError_t launch_attn_decode(const AttnArgs &a, int B, cudaStream_t s, int pdl) {
  const int grp = a.H / a.Hkv, cs = a.splits;
  if (cs < 1 || cs > 16 || (cs & (cs - 1))) return cudaErrorInvalidValue;
#define RV_DL(HD_, G_)                                                                  \
  if (a.hd == HD_ && grp == G_)                                                         \
    return a.act == 1 ? launch_dec<HD_, G_, 1>(a, B, cs, s, pdl) : launch_dec<HD_, G_, 0>(a, B, cs, s, pdl);
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
