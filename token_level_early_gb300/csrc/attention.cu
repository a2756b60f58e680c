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
// position p come from the QKV kernel it follows.  The splits merge their
// softmax states through distributed shared memory.
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
constexpr int DNST = 4;   // ring stages

template <int HD>
struct DecTile {
  static constexpr int KROW = HD * 2 + 16;  // padded K row: lane-per-row 16-byte reads hit distinct banks
  static constexpr int VROW = HD * 2;
  static constexpr int BYTES = DTT * (KROW + VROW);
};

template <int HD>
static size_t dec_smem(int grp) {
  return (size_t)DNST * DecTile<HD>::BYTES + sizeof(float) * grp * (HD + 2);
}

__device__ __forceinline__ uint32_t pack_act2(float lo, float hi, int act) {
  return (uint32_t)f_to_act(lo, act) | ((uint32_t)f_to_act(hi, act) << 16);
}

template <int HD, int GRP, int ACT>
__global__ void __launch_bounds__(GRP * 32, 1) k_attn_dec(AttnArgs a) {
  using TL = DecTile<HD>;
  constexpr int NT = GRP * 32, PER = HD / 32, PR = HD / 8;
  extern __shared__ __align__(16) unsigned char sm[];
  float *part = reinterpret_cast<float *>(sm + DNST * TL::BYTES);  // [GRP][HD + 2]: o, running max, sum
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

  for (int tile = tb, it = 0; tile < te; ++tile, ++it) {
    cp_wait<DNST - 2>();
    __syncthreads();  // the tile is in; every warp is done with the slot refilled next
    issue(tile + DNST - 1, (it + DNST - 1) % DNST);
    const unsigned char *tk = sm + (it % DNST) * TL::BYTES;
    const unsigned char *tv = tk + DTT * TL::KROW;
    const int n = min(DTT, p - tile * DTT);
    float sc = -INFINITY;
    if (lane < n) {
      const uint4 *kr = reinterpret_cast<const uint4 *>(tk + lane * TL::KROW);
      float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
      for (int j = 0; j < PR; ++j) {
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
      sc = ((d0 + d1) + (d2 + d3)) * scale;
    }
    const float mnew = fmaxf(mrun, warp_max(sc));
    const float pe = lane < n ? expf(sc - mnew) : 0.f;
    const float corr = mrun == -INFINITY ? 0.f : expf(mrun - mnew);
    lrun = lrun * corr + warp_sum(pe);
#pragma unroll
    for (int r = 0; r < PER; ++r) o[r] *= corr;
    for (int t = 0; t < n; ++t) {
      const float pt = __shfl_sync(0xffffffffu, pe, t);
      const uint16_t *vr = reinterpret_cast<const uint16_t *>(tv + t * TL::VROW) + lane * PER;
      if constexpr (PER == 4) {
        const uint2 vv = *reinterpret_cast<const uint2 *>(vr);
        o[0] = fmaf(pt, act_to_f((uint16_t)(vv.x & 0xFFFFu), ACT), o[0]);
        o[1] = fmaf(pt, act_to_f((uint16_t)(vv.x >> 16), ACT), o[1]);
        o[2] = fmaf(pt, act_to_f((uint16_t)(vv.y & 0xFFFFu), ACT), o[2]);
        o[3] = fmaf(pt, act_to_f((uint16_t)(vv.y >> 16), ACT), o[3]);
      } else {
        const uint32_t vv = *reinterpret_cast<const uint32_t *>(vr);
        o[0] = fmaf(pt, act_to_f((uint16_t)(vv & 0xFFFFu), ACT), o[0]);
        o[1] = fmaf(pt, act_to_f((uint16_t)(vv >> 16), ACT), o[1]);
      }
    }
    mrun = mnew;
  }

  // position p itself (its K/V were written by the QKV kernel this kernel
  // follows): folded in by the last split
  if (sp == cs - 1) {
    const uint16_t *kc = Kb + (size_t)p * HD + lane * PER, *vc = Vb + (size_t)p * HD + lane * PER;
    float d = 0.f;
#pragma unroll
    for (int r = 0; r < PER; ++r) d = fmaf(qp[lane * PER + r], act_to_f(kc[r], ACT), d);
    const float sc = warp_sum(d) * scale;
    const float mnew = fmaxf(mrun, sc);
    const float corr = mrun == -INFINITY ? 0.f : expf(mrun - mnew), pe = expf(sc - mnew);
    lrun = lrun * corr + pe;
#pragma unroll
    for (int r = 0; r < PER; ++r) o[r] = fmaf(pe, act_to_f(vc[r], ACT), o[r] * corr);
    mrun = mnew;
  }

  // merge across the cluster: split sp combines dims [sp * HD / cs, ...) of every head
  float *pp = part + warp * (HD + 2);
#pragma unroll
  for (int r = 0; r < PER; ++r) pp[lane * PER + r] = o[r];
  if (lane == 0) {
    pp[HD] = mrun;
    pp[HD + 1] = lrun;
  }
  cl.sync();
  const int dpc = HD / cs;
  for (int e = tid; e < GRP * dpc; e += NT) {
    const int hh = e / dpc, dd = sp * dpc + (e - hh * dpc);
    float M = -INFINITY;
    for (int r = 0; r < cs; ++r) M = fmaxf(M, cl.map_shared_rank(part, r)[hh * (HD + 2) + HD]);
    float Ls = 0.f, O = 0.f;
    for (int r = 0; r < cs; ++r) {
      const float *rp = cl.map_shared_rank(part, r) + hh * (HD + 2);
      const float w = rp[HD] == -INFINITY ? 0.f : expf(rp[HD] - M);
      Ls = fmaf(w, rp[HD + 1], Ls);
      O = fmaf(w, rp[dd], O);
    }
    a.o[((size_t)b * a.H + g * GRP + hh) * HD + dd] = round_act(O * (1.0f / Ls), ACT);
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

// Prefill / general rows: T tokens per sequence starting at base (NULL = 0).
cudaError_t launch_attn_rows(const AttnRowsArgs &r, int max_rows, cudaStream_t s) {
  AttnArgs a;
  a.kv = r.kv;
  a.layer = r.layer; a.H = r.H; a.Hkv = r.Hkv; a.hd = r.hd; a.act = r.act;
  a.q = r.q; a.o = r.o; a.len = nullptr; a.splits = 1; a.part = nullptr; a.counter = nullptr;
  return launch_any(a, r.tokens_per_row, r.base, max_rows, s);
}

}  // namespace rv
