// Persistent batch-1 decode step: the whole token (embedding, every layer on
// its backbone or river path, the exit decision, the LM head and the greedy
// pick) in one cooperative launch with one resident block per SM.
//
// Phases of layer l, separated by grid barriers:
//   QKV  : RMSNorm(h) -> W_qkv (bf16 or int4) -> RoPE -> K/V into slot (l, 0, p)
//   ATTN : split-KV GQA attention over positions 0..p (one task per block)
//   COMB : merge of the splits' softmax states -> o
//   O    : h_mid = h + W_o o
//   GU   : RMSNorm(h_mid) -> a = silu(W_g x) * (W_u x)
//   DOWN : h_out = h_mid + W_d a; per-block sums of h_in.h_out, |h_in|^2, |h_out|^2
//   then every block adds the per-block sums in the same order, so all blocks
//   take the same exit decision s(l) = cos(h_in, h_out) > tau without another
//   barrier.  Before each barrier the warps already issue the next phase's
//   first weight chunks into their cp.async rings, so the weight stream keeps
//   running while blocks wait.
//
// Grid barrier: an arrival counter and an epoch word in global memory; the
// last block to arrive resets the counter and advances the epoch.  Waiting is
// bounded: after about a second without progress a block sets error bit 8 and
// every block leaves the kernel at its next barrier (copies drained first).
//
// Method: "River-LLM: Large Language Model Seamless Exit Based on KV Share",
// paperlayer.ai summary section 4 (KV-Shared Exit Layer; Inference with
// Seamless Exit) and aitrends.kr (s(l) = cos(h(l-1), h(l)) > tau; W4A16 exit
// layers copied from the backbone blocks).
#include "gemv_core.cuh"
#include "mega.cuh"

namespace rv {

constexpr int MW = 16;     // warps per block
constexpr int ATILE = 32;  // attention positions per tile

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ bool grid_barrier(unsigned *bar, unsigned &epoch, int32_t *err) {
  __shared__ int ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned target = epoch + 1;
    __threadfence();
    const unsigned prev = atomicAdd(&bar[0], 1u);
    if (prev == gridDim.x - 1) {
      atomicExch(&bar[0], 0u);
      __threadfence();
      atomicExch(&bar[1], target);
    } else {
      unsigned it = 0;
      while (ld_acquire(&bar[1]) != target) {
        if (++it > (1u << 21)) {
          atomicOr(err, 8);
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    epoch = target;
    ok = (*(volatile int32_t *)err & 8) == 0;
  }
  __syncthreads();
  return ok != 0;
}

// GEMV arguments of one phase of layer l.
__device__ __forceinline__ GemvArgs phase_args(const MegaArgs &A, int l, int which) {
  GemvArgs a{};
  const LayerDesc &ly = A.layers[l];
  a.m = ly.m[which];
  a.st = A.st;
  a.kv = A.kv;
  a.layer = l;
  a.L = A.L; a.H = A.H; a.Hkv = A.Hkv; a.hd = A.hd;
  a.eps = A.eps;
  a.rope_cs = A.rope_cs;
  const Geo g = geo_of(a.m);
  a.s4 = splits_for(a.m.N >> 2, g.nk4);
  a.s16 = splits_for(a.m.N >> 2, g.nk16);
  float *hin = A.h[l & 1], *hout = A.h[(l + 1) & 1];
  switch (which) {
    case 0: a.h = hin; a.gamma = ly.attn_norm; a.out_vec = A.q; break;
    case 1: a.vec = A.o; a.h_base = hin; a.h_out = A.hmid; break;
    case 2: a.h = A.hmid; a.gamma = ly.mlp_norm; a.out_vec = A.a; break;
    default:
      a.vec = A.a; a.h_base = A.hmid; a.h_in = hin; a.h_out = hout;
      a.dbg_h = A.dbg_h ? A.dbg_h + (size_t)(l + 1) * A.Bmax * A.d : nullptr;
      break;
  }
  return a;
}

__device__ __forceinline__ GemvArgs head_args(const MegaArgs &A) {
  GemvArgs a{};
  a.m.w = A.lm_head; a.m.N = A.V; a.m.K = A.d;
  a.st = A.st;
  a.h = A.h[A.L & 1]; a.gamma = A.final_norm; a.eps = A.eps;
  a.dbg_logits = A.dbg_logits;
  const Geo g = geo_of(a.m);
  a.s4 = splits_for(a.m.N >> 2, g.nk4);
  a.s16 = splits_for(a.m.N >> 2, g.nk16);
  return a;
}

// Split-KV attention task (kv head g, split sp of S) over positions 0..pos:
// warps 0..GRP-1 take the GRP query heads of KV head g; every warp helps to
// stage the K/V tile.  Publishes (o unnormalised, running max, running sum).
template <int HD, int GRP>
__device__ void attn_task(const MegaArgs &A, int l, int g, int sp, int S, int pos, float *tiles) {
  float *qs = tiles;                      // [GRP][HD]
  float *Ks = qs + GRP * HD;              // [ATILE][HD + 1]
  float *Vs = Ks + ATILE * (HD + 1);      // [ATILE][HD]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nt = blockDim.x;
  constexpr int PER = HD / 32;
  const int T = pos + 1, chunk = (T + S - 1) / S, t0 = sp * chunk, t1 = min(T, t0 + chunk);
  __syncthreads();  // a previous task of this block may still be reading the tiles
  for (int i = threadIdx.x; i < GRP * HD; i += nt) qs[i] = __ldcg(A.q + (size_t)g * GRP * HD + i);
  const uint16_t *Kb = A.kv.base + A.kv.idx(l, 0, 0, g, 0);
  const uint16_t *Vb = A.kv.base + A.kv.idx(l, 1, 0, g, 0);
  const float scale = 1.0f / sqrtf((float)HD);
  float mrun = -INFINITY, lrun = 0.f, o[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) o[r] = 0.f;
  for (int tile = t0; tile < t1; tile += ATILE) {
    const int n = min(ATILE, t1 - tile);
    __syncthreads();
    for (int v = threadIdx.x; v < n * (HD / 8); v += nt) {
      const int t = v / (HD / 8), c = (v % (HD / 8)) * 8;
      const uint4 kw = __ldcg(reinterpret_cast<const uint4 *>(Kb + (size_t)(tile + t) * HD + c));
      const uint4 vw = __ldcg(reinterpret_cast<const uint4 *>(Vb + (size_t)(tile + t) * HD + c));
      const uint16_t *kp = reinterpret_cast<const uint16_t *>(&kw);
      const uint16_t *vp = reinterpret_cast<const uint16_t *>(&vw);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        Ks[t * (HD + 1) + c + j] = act_to_f(kp[j], A.act);
        Vs[t * HD + c + j] = act_to_f(vp[j], A.act);
      }
    }
    __syncthreads();
    if (warp < GRP) {
      float sc = -INFINITY;
      if (lane < n) {
        float d = 0.f;
#pragma unroll 8
        for (int i = 0; i < HD; ++i) d = fmaf(qs[warp * HD + i], Ks[lane * (HD + 1) + i], d);
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
        for (int r = 0; r < PER; ++r) o[r] = fmaf(pt, Vs[t * HD + lane + 32 * r], o[r]);
      }
      mrun = mnew;
    }
  }
  if (warp < GRP) {
    const int h = g * GRP + warp;
    float *pp = A.attn_part + ((size_t)h * S + sp) * (HD + 2);
#pragma unroll
    for (int r = 0; r < PER; ++r) pp[lane + 32 * r] = o[r];
    if (lane == 0) { pp[HD] = mrun; pp[HD + 1] = lrun; }
  }
}

template <int HD, int GRP>
__device__ void attn_phase(const MegaArgs &A, int l, int S, int pos, float *tiles) {
  for (int task = blockIdx.x; task < A.Hkv * S; task += gridDim.x)
    attn_task<HD, GRP>(A, l, task / S, task % S, S, pos, tiles);
}

// Merge the S split states of every query head into o (16-bit rounded).
template <int HD>
__device__ void combine_phase(const MegaArgs &A, int S) {
  constexpr int PER = HD / 32;
  const int lane = threadIdx.x & 31;
  for (int h = blockIdx.x * MW + (threadIdx.x >> 5); h < A.H; h += gridDim.x * MW) {
    const float *base = A.attn_part + (size_t)h * S * (HD + 2);
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, __ldcg(base + s * (HD + 2) + HD));
    float Ls = 0.f, acc[PER];
#pragma unroll
    for (int r = 0; r < PER; ++r) acc[r] = 0.f;
#pragma unroll 4
    for (int s = 0; s < S; ++s) {
      const float ms = __ldcg(base + s * (HD + 2) + HD);
      const float w = ms == -INFINITY ? 0.f : expf(ms - M);
      Ls = fmaf(w, __ldcg(base + s * (HD + 2) + HD + 1), Ls);
#pragma unroll
      for (int r = 0; r < PER; ++r) acc[r] = fmaf(w, __ldcg(base + s * (HD + 2) + lane + 32 * r), acc[r]);
    }
    const float inv = 1.0f / Ls;
#pragma unroll
    for (int r = 0; r < PER; ++r) A.o[(size_t)h * HD + lane + 32 * r] = round_act(acc[r] * inv, A.act);
  }
}

template <int ACT, int HD, int GRP>
__global__ void __launch_bounds__(MW * 32, 1) k_decode_mega(MegaArgs A) {
  extern __shared__ __align__(16) float smem[];
  float *xs = smem;                      // activations / attention tiles
  float *scratch = smem + A.xs_floats;   // 256 floats
  const int tid = threadIdx.x, warp = tid >> 5, bid = blockIdx.x, nb = gridDim.x;
  char *ring = reinterpret_cast<char *>(scratch + 256) + (size_t)warp * NST * STAGE;
  unsigned epoch = 0;
  if (tid == 0) epoch = *(volatile unsigned *)&A.bar[1];
  const int L = A.L;
  const int pos = A.st.len[0];

  // ---- step start: route, embedding
  int route, exit_l;
  {
    if (*A.st.mode == 1) {
      int f = A.st.forced[0];
      if (f < 0 || f > L) {
        if (bid == 0 && tid == 0) atomicOr(A.st.err, 2);
        f = L;
      }
      route = f == 0;
      exit_l = f == 0 ? 0 : L;
    } else {
      route = 0;
      exit_l = L;
    }
    int tok = A.st.tokens[0];
    if (tok < 0 || tok >= A.V) {
      if (bid == 0 && tid == 0) atomicOr(A.st.err, 1);
      tok = 0;
    }
    for (int i = bid * blockDim.x + tid; i < A.d; i += nb * blockDim.x) {
      const float v = act_to_f(A.embed[(size_t)tok * A.d + i], ACT);
      A.h[0][i] = v;
      if (A.dbg_h) A.dbg_h[i] = v;
    }
  }
  GemvArgs a = phase_args(A, 0, 0);
  ItemStream is = gemv_begin<MW, EPI_QKV>(a, route, ring, bid, nb);
  if (!grid_barrier(A.bar, epoch, A.st.err)) { cp_wait<0>(); return; }

  const int S = A.splits;
  for (int l = 0; l < L; ++l) {
    // QKV -> RoPE -> K/V append
    gemv_run<MW, ACT, PRO_NORM, EPI_QKV>(a, route, xs, scratch, ring, is, bid, nb);
    // the O projection's weights do not depend on attention: start them now
    a = phase_args(A, l, 1);
    is = gemv_begin<MW, EPI_RESID>(a, route, ring, bid, nb);
    if (!grid_barrier(A.bar, epoch, A.st.err)) { cp_wait<0>(); return; }
    attn_phase<HD, GRP>(A, l, S, pos, xs);
    if (!grid_barrier(A.bar, epoch, A.st.err)) { cp_wait<0>(); return; }
    combine_phase<HD>(A, S);
    if (!grid_barrier(A.bar, epoch, A.st.err)) { cp_wait<0>(); return; }
    // O projection + residual
    gemv_run<MW, ACT, PRO_VEC, EPI_RESID>(a, route, xs, scratch, ring, is, bid, nb);
    a = phase_args(A, l, 2);
    is = gemv_begin<MW, EPI_SWIGLU>(a, route, ring, bid, nb);
    if (!grid_barrier(A.bar, epoch, A.st.err)) { cp_wait<0>(); return; }
    // gate/up + SwiGLU
    gemv_run<MW, ACT, PRO_NORM, EPI_SWIGLU>(a, route, xs, scratch, ring, is, bid, nb);
    a = phase_args(A, l, 3);
    is = gemv_begin<MW, EPI_DOWN>(a, route, ring, bid, nb);
    if (!grid_barrier(A.bar, epoch, A.st.err)) { cp_wait<0>(); return; }
    // down + residual, per-block s(l) sums
    {
      PhaseOut po = gemv_run<MW, ACT, PRO_VEC, EPI_DOWN>(a, route, xs, scratch, ring, is, bid, nb);
      float *bsum = scratch + 128;
      const float p0 = block_sum(po.p_dot, bsum), p1 = block_sum(po.p_n1, bsum + 32), p2 = block_sum(po.p_n2, bsum + 64);
      if (tid == 0) {
        A.partials[bid * 3 + 0] = p0;
        A.partials[bid * 3 + 1] = p1;
        A.partials[bid * 3 + 2] = p2;
      }
    }
    if (!grid_barrier(A.bar, epoch, A.st.err)) return;
    // every block derives the same decision from the same sums in the same order
    {
      __shared__ float dsum[3];
      if (warp == 0) {
        float t0 = 0.f, t1 = 0.f, t2 = 0.f;
        for (int i = (tid & 31); i < nb; i += 32) {
          t0 += __ldcg(A.partials + i * 3 + 0);
          t1 += __ldcg(A.partials + i * 3 + 1);
          t2 += __ldcg(A.partials + i * 3 + 2);
        }
        t0 = warp_sum(t0);
        t1 = warp_sum(t1);
        t2 = warp_sum(t2);
        if (tid == 0) { dsum[0] = t0; dsum[1] = t1; dsum[2] = t2; }
      }
      __syncthreads();
      const int layer1 = l + 1;
      const float s = dsum[0] / fmaxf(sqrtf(dsum[1]) * sqrtf(dsum[2]), 1e-8f);
      float *dbg_s = A.dbg_s ? A.dbg_s + (size_t)l * A.Bmax : nullptr;
      if (route == 0) {
        bool go;
        if (*A.st.mode == 1) {
          int f = A.st.forced[0];
          if (f < 0 || f > L) f = L;
          go = layer1 == f && layer1 < L;
        } else {
          go = layer1 >= *A.st.entry && layer1 <= L - 1 && s > *A.st.tau;
        }
        if (bid == 0 && tid == 0 && dbg_s) dbg_s[0] = s;
        if (go) { route = 1; exit_l = layer1; }
      } else if (bid == 0 && tid == 0 && dbg_s) {
        dbg_s[0] = __int_as_float(0x7fc00000);
      }
      __syncthreads();  // dsum is rewritten next layer
    }
    if (l + 1 < L) {
      a = phase_args(A, l + 1, 0);
      is = gemv_begin<MW, EPI_QKV>(a, route, ring, bid, nb);
    }
  }

  // ---- final norm + LM head + greedy pick
  float *head_part = A.partials + 3 * nb;
  a = head_args(A);
  is = gemv_begin<MW, EPI_LOGITS>(a, 0, ring, bid, nb);
  {
    PhaseOut po = gemv_run<MW, ACT, PRO_NORM, EPI_LOGITS>(a, 0, xs, scratch, ring, is, bid, nb);
    float *bv = xs;
    int *bi = reinterpret_cast<int *>(xs + MW * 32);
    __syncthreads();
    bv[tid] = po.best;
    bi[tid] = po.best_i;
    __syncthreads();
    if (tid == 0) {
      float vb = bv[0];
      int ib = bi[0];
      for (int q = 1; q < MW * 32; ++q)
        if (bv[q] > vb || (bv[q] == vb && bi[q] < ib)) { vb = bv[q]; ib = bi[q]; }
      // the head's results go after the s(l) sums: a slow block may still be
      // reading those for the last decision
      head_part[bid * 2] = vb;
      reinterpret_cast<int *>(head_part)[bid * 2 + 1] = ib;
    }
  }
  if (!grid_barrier(A.bar, epoch, A.st.err)) return;
  if (bid == 0 && tid == 0) {
    float vb = -INFINITY;
    int ib = 0x7fffffff;
    for (int b = 0; b < nb; ++b) {
      const float bvv = __ldcg(head_part + b * 2);
      const int bii = __ldcg(reinterpret_cast<const int *>(head_part) + b * 2 + 1);
      if (bvv > vb || (bvv == vb && bii < ib)) { vb = bvv; ib = bii; }
    }
    A.st.next_ids[0] = ib == 0x7fffffff ? 0 : ib;
    A.st.route[0] = route;
    A.st.exit_layer[0] = exit_l;
    A.st.len[0] = pos + 1;
  }
}

// ------------------------------------------------------------------ host side

size_t mega_smem_bytes(const MegaArgs &A) {
  return sizeof(float) * (A.xs_floats + 256) + (size_t)MW * NST * STAGE;
}

template <int ACT, int HD, int GRP>
static cudaError_t mega_prepare_t(MegaArgs &A, int n_sm, int *grid) {
  auto fn = k_decode_mega<ACT, HD, GRP>;
  const size_t smem = mega_smem_bytes(A);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, MW * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  *grid = n_sm;  // one resident block per SM
  return cudaSuccess;
}

template <int ACT, int HD, int GRP>
static cudaError_t mega_launch_t(const MegaArgs &A, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MW * 32);
  cfg.dynamicSmemBytes = mega_smem_bytes(A);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_decode_mega<ACT, HD, GRP>, A);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

#define RV_MEGA_DISPATCH(CALL)                                   \
  const int grp = A.H / A.Hkv;                                   \
  if (A.act == 1 && A.hd == 128 && grp == 4) return CALL(1, 128, 4); \
  if (A.act == 1 && A.hd == 64 && grp == 4) return CALL(1, 64, 4);   \
  if (A.act == 0 && A.hd == 64 && grp == 2) return CALL(0, 64, 2);   \
  if (A.act == 1 && A.hd == 64 && grp == 2) return CALL(1, 64, 2);   \
  if (A.act == 0 && A.hd == 128 && grp == 4) return CALL(0, 128, 4); \
  if (A.act == 0 && A.hd == 64 && grp == 4) return CALL(0, 64, 4);   \
  return cudaErrorNotSupported;

cudaError_t mega_prepare(MegaArgs &A, int n_sm, int *grid) {
#define RV_P(ACT_, HD_, G_) mega_prepare_t<ACT_, HD_, G_>(A, n_sm, grid)
  RV_MEGA_DISPATCH(RV_P)
#undef RV_P
}

cudaError_t mega_launch(const MegaArgs &A, int grid, cudaStream_t s) {
#define RV_L(ACT_, HD_, G_) mega_launch_t<ACT_, HD_, G_>(A, grid, s)
  RV_MEGA_DISPATCH(RV_L)
#undef RV_L
}

size_t mega_attn_tile_floats(int hd, int grp) { return (size_t)grp * hd + (size_t)ATILE * (hd + 1) + (size_t)ATILE * hd; }
int mega_warps() { return MW; }

}  // namespace rv
