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
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

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
cudaError_t launch_attn_decode(const AttnArgs &a, int B, cudaStream_t s, int pdl) {
  return launch_any(a, 1, a.len, B, s, pdl);
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
