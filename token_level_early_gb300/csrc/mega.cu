// Persistent batch-1 decode step: the whole token (embedding, every layer on
// its backbone or river path, the exit decision, the LM head and the greedy
// pick) in one cooperative launch with one resident block per SM.
//
// Phases of layer l, separated by grid barriers:
//   QKV  : exit decision of layer l - 1 (every block, from h(l-1) and h(l)),
//          RMSNorm(h) -> W_qkv (bf16 or int4) -> RoPE -> K/V into slot (l, 0, p)
//   ATTN : split-KV GQA attention over positions 0..p (one task per block);
//          each block starts copying its first K/V tile before the barrier
//   COMB : merge of the splits' softmax states -> o
//   O    : h_mid = h + W_o o
//   GU   : RMSNorm(h_mid) -> a = silu(W_g x) * (W_u x)
//   DOWN : h_out = h_mid + W_d a
// Every block reaches the same exit decision from the same sums in the same
// order.  Before each barrier the warps already issue the next phase's first
// weight chunks into their cp.async rings (QKV on the route before the
// decision; re-streamed in the one layer per token where it flips), so the
// weight stream keeps running while blocks wait.
//
// Grid barrier: a counter in global memory that only grows within a launch
// (the host zeroes it before each step); a block adds 1 with release
// semantics and polls with acquire loads until the counter reaches
// epoch x blocks.  Waiting is bounded: after about a second without progress
// a block sets error bit 8 and every block leaves the kernel at its next
// barrier (copies drained first).
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

__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ bool grid_barrier(unsigned *bar, unsigned &epoch, int32_t *err) {
  __shared__ int ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    epoch += 1;
    const unsigned target = epoch * gridDim.x;
    __threadfence();
    red_release_add(bar, 1u);
    unsigned it = 0;
    while ((int)(ld_acquire(bar) - target) < 0) {
      if (++it > (1u << 21)) {
        atomicOr(err, 8);
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
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

// Split-KV attention.  Task t = (kv head g, split sp of S): split sp takes
// tiles [tb, te) of the past positions 0..p-1 (tiles of ATILE positions,
// split evenly), the last split also position p.  K/V tiles are copied by
// cp.async into a 2-slot ring in the activation region (K rows padded by 16
// bytes: conflict-free row-per-lane reads); warps 0..GRP-1 take the GRP query
// heads of kv head g, scores by mixed-precision FMAs on 16-bit q and K.
// Publishes (o unnormalised, running max, running sum) per query head.
template <int HD>
struct MegaTile {
  static constexpr int KROW = HD * 2 + 16;
  static constexpr int VROW = HD * 2;
  static constexpr int BYTES = ATILE * (KROW + VROW);
};

__device__ __forceinline__ void split_tiles(int p, int S, int sp, int &tb, int &te) {
  const int ntile = (p + ATILE - 1) / ATILE, per = (ntile + S - 1) / S;
  tb = min(ntile, sp * per);
  te = min(ntile, tb + per);
}

// Copy tile `tile` (if below te) of kv head g into ring slot `slot`; one
// commit group per call.
template <int HD>
__device__ __forceinline__ void attn_issue(const MegaArgs &A, int l, int g, int tile, int te, int p, int slot,
                                           unsigned char *ring_a) {
  using TL = MegaTile<HD>;
  if (tile < te) {
    const int t0 = tile * ATILE, n = min(ATILE, p - t0);
    const uint16_t *Kb = A.kv.base + A.kv.idx(l, 0, 0, g, 0), *Vb = A.kv.base + A.kv.idx(l, 1, 0, g, 0);
    const unsigned st = (unsigned)__cvta_generic_to_shared(ring_a) + slot * TL::BYTES;
    constexpr int PR = HD / 8;
    for (int v = threadIdx.x; v < 2 * ATILE * PR; v += blockDim.x) {
      const int kv = v >= ATILE * PR, rem = v - kv * ATILE * PR, t = rem / PR, c = rem - t * PR;
      if (t < n)
        cp16s(st + (kv ? ATILE * TL::KROW + t * TL::VROW : t * TL::KROW) + c * 16,
              (kv ? Vb : Kb) + (size_t)(t0 + t) * HD + c * 8);
    }
  }
  cp_commit();
}

// qs: GRP * HD / 2 words of shared memory for q as 16-bit pairs.
template <int ACT, int HD, int GRP>
__device__ void attn_task(const MegaArgs &A, int l, int task, int S, int p, unsigned char *ring_a,
                          bool first_issued, uint32_t *qs) {
  using TL = MegaTile<HD>;
  constexpr int PER = HD / 32, PR = HD / 8;
  const int g = task / S, sp = task - g * S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int tb, te;
  split_tiles(p, S, sp, tb, te);
  if (!first_issued) attn_issue<HD>(A, l, g, tb, te, p, 0, ring_a);
  const int h = g * GRP + (warp < GRP ? warp : 0);
  const float *qp = A.q + (size_t)h * HD;
  // q of the GRP heads as 16-bit pairs (q is act-rounded after RoPE: exact)
  for (int i = threadIdx.x; i < GRP * HD / 2; i += blockDim.x) {
    const float2 v = __ldcg(reinterpret_cast<const float2 *>(A.q + (size_t)g * GRP * HD) + i);
    qs[i] = (uint32_t)f_to_act(v.x, ACT) | ((uint32_t)f_to_act(v.y, ACT) << 16);
  }
  const uint4 *q4 = reinterpret_cast<const uint4 *>(qs + (warp < GRP ? warp : 0) * (HD / 2));
  const float scale = 1.0f / sqrtf((float)HD);
  float mrun = -INFINITY, lrun = 0.f, o[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) o[r] = 0.f;
  for (int tile = tb, it = 0; tile < te; ++tile, ++it) {
    __syncthreads();  // every warp is done with the slot refilled next
    attn_issue<HD>(A, l, g, tile + 1, te, p, (it + 1) & 1, ring_a);
    cp_wait<1>();     // all but the newest group: tile `tile` (and older weight items) landed
    __syncthreads();
    if (warp < GRP) {
      const unsigned char *tk = ring_a + (it & 1) * TL::BYTES, *tv = tk + ATILE * TL::KROW;
      const int n = min(ATILE, p - tile * ATILE);
      float sc = -INFINITY;
      if (lane < n) {
        const uint4 *kr = reinterpret_cast<const uint4 *>(tk + lane * TL::KROW);
        float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
        for (int j = 0; j < PR; ++j) {
          const uint4 k = kr[j], q = q4[j];
          d0 = fma_lo16<ACT>(k.x, q.x, d0);
          d1 = fma_hi16<ACT>(k.x, q.x, d1);
          d2 = fma_lo16<ACT>(k.y, q.y, d2);
          d3 = fma_hi16<ACT>(k.y, q.y, d3);
          d0 = fma_lo16<ACT>(k.z, q.z, d0);
          d1 = fma_hi16<ACT>(k.z, q.z, d1);
          d2 = fma_lo16<ACT>(k.w, q.w, d2);
          d3 = fma_hi16<ACT>(k.w, q.w, d3);
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
#pragma unroll
        for (int r = 0; r < PER; ++r) o[r] = fmaf(pt, act_to_f(vr[r], ACT), o[r]);
      }
      mrun = mnew;
    }
  }
  if (warp < GRP) {
    if (sp == S - 1) {  // position p, written in the QKV phase
      const uint16_t *kc = A.kv.base + A.kv.idx(l, 0, 0, g, p) + lane * PER;
      const uint16_t *vc = A.kv.base + A.kv.idx(l, 1, 0, g, p) + lane * PER;
      float d = 0.f;
#pragma unroll
      for (int r = 0; r < PER; ++r) d = fmaf(__ldcg(qp + lane * PER + r), act_to_f(__ldcg(kc + r), ACT), d);
      const float sc = warp_sum(d) * scale;
      const float mnew = fmaxf(mrun, sc);
      const float corr = mrun == -INFINITY ? 0.f : expf(mrun - mnew), pe = expf(sc - mnew);
      lrun = lrun * corr + pe;
#pragma unroll
      for (int r = 0; r < PER; ++r) o[r] = fmaf(pe, act_to_f(__ldcg(vc + r), ACT), o[r] * corr);
      mrun = mnew;
    }
    float *pp = A.attn_part + ((size_t)h * S + sp) * (HD + 2);
#pragma unroll
    for (int r = 0; r < PER; ++r) pp[lane * PER + r] = o[r];
    if (lane == 0) {
      pp[HD] = mrun;
      pp[HD + 1] = lrun;
    }
  }
}

template <int ACT, int HD, int GRP>
__device__ void attn_phase(const MegaArgs &A, int l, int S, int p, unsigned char *ring_a, uint32_t *qs) {
  for (int task = blockIdx.x; task < A.Hkv * S; task += gridDim.x) {
    __syncthreads();  // a previous task may still read qs
    attn_task<ACT, HD, GRP>(A, l, task, S, p, ring_a, task == (int)blockIdx.x, qs);
  }
  cp_wait<0>();
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
      for (int r = 0; r < PER; ++r) acc[r] = fmaf(w, __ldcg(base + s * (HD + 2) + lane * PER + r), acc[r]);
    }
    const float inv = 1.0f / Ls;
#pragma unroll
    for (int r = 0; r < PER; ++r) A.o[(size_t)h * HD + lane * PER + r] = round_act(acc[r] * inv, A.act);
  }
}

template <int ACT, int HD, int GRP>
__global__ void __launch_bounds__(MW * 32, 1) k_decode_mega(MegaArgs A) {
  extern __shared__ __align__(16) float smem[];
  float *xs = smem;                      // activations / attention tiles
  float *scratch = smem + A.xs_floats;   // 256 floats
  const int tid = threadIdx.x, warp = tid >> 5, bid = blockIdx.x, nb = gridDim.x;
  char *ring = reinterpret_cast<char *>(scratch + 256) + (size_t)warp * NST * STAGE;
  unsigned epoch = 0;  // barriers passed (thread 0); the host zeroes the counter before each step
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
  unsigned char *ring_a = reinterpret_cast<unsigned char *>(xs);
  float *bsum = scratch + 128;
  for (int l = 0; l < L; ++l) {
    float ss = -1.f;  // sum of h(l)^2, shared by the decision and the RMSNorm prologue
    if (l > 0) {
      // exit decision of layer l (1-based) from its input h(l-1) and output h(l)
      const float *hp = A.h[(l - 1) & 1], *hc = A.h[l & 1];
      float dot = 0.f, n1 = 0.f, n2 = 0.f;
      for (int i = tid * 4; i < A.d; i += blockDim.x * 4) {
        const float4 x = __ldcg(reinterpret_cast<const float4 *>(hp + i));
        const float4 y = __ldcg(reinterpret_cast<const float4 *>(hc + i));
        dot = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, dot))));
        n1 = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, n1))));
        n2 = fmaf(y.x, y.x, fmaf(y.y, y.y, fmaf(y.z, y.z, fmaf(y.w, y.w, n2))));
      }
      const float3 t = block_sum3(dot, n1, n2, bsum);
      dot = t.x;
      n1 = t.y;
      n2 = t.z;
      ss = n2;
      const Decision dc = decide(A.st, 0, route, l, L, dot, n1, n2);
      if (bid == 0 && tid == 0 && A.dbg_s) A.dbg_s[(size_t)(l - 1) * A.Bmax] = dc.s;
      if (dc.exited) {
        exit_l = l;
        route = 1;
        cp_wait<0>();  // drop the backbone items streamed on the old route
        is = gemv_begin<MW, EPI_QKV>(a, route, ring, bid, nb);
      }
    }
    // QKV -> RoPE -> K/V append
    gemv_run<MW, ACT, PRO_NORM, EPI_QKV>(a, route, xs, scratch, ring, is, bid, nb, ss);
    // the first K/V tile of this block's attention task (positions < p are
    // final) and the O projection's weights do not wait for the barrier
    __syncthreads();  // the activation region is free again
    {
      const int task = bid;
      if (task < A.Hkv * S) {
        int tb, te;
        split_tiles(pos, S, task % S, tb, te);
        attn_issue<HD>(A, l, task / S, tb, te, pos, 0, ring_a);
      }
    }
    a = phase_args(A, l, 1);
    is = gemv_begin<MW, EPI_RESID>(a, route, ring, bid, nb);
    if (!grid_barrier(A.bar, epoch, A.st.err)) { cp_wait<0>(); return; }
    attn_phase<ACT, HD, GRP>(A, l, S, pos, ring_a, reinterpret_cast<uint32_t *>(scratch));
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
    // down + residual
    gemv_run<MW, ACT, PRO_VEC, EPI_DOWN>(a, route, xs, scratch, ring, is, bid, nb);
    if (l + 1 < L) {
      a = phase_args(A, l + 1, 0);
      is = gemv_begin<MW, EPI_QKV>(a, route, ring, bid, nb);
    }
    if (!grid_barrier(A.bar, epoch, A.st.err)) { cp_wait<0>(); return; }
  }

  // s(L) for the debug dump (no exit after the last layer)
  if (A.dbg_s && bid == 0) {
    const float *hp = A.h[(L - 1) & 1], *hc = A.h[L & 1];
    float dot = 0.f, n1 = 0.f, n2 = 0.f;
    for (int i = tid; i < A.d; i += blockDim.x) {
      const float x = __ldcg(hp + i), y = __ldcg(hc + i);
      dot = fmaf(x, y, dot);
      n1 = fmaf(x, x, n1);
      n2 = fmaf(y, y, n2);
    }
    dot = block_sum(dot, bsum);
    n1 = block_sum(n1, bsum + 32);
    n2 = block_sum(n2, bsum + 64);
    const Decision dc = decide(A.st, 0, route, L, L, dot, n1, n2);
    if (tid == 0) A.dbg_s[(size_t)(L - 1) * A.Bmax] = dc.s;
  }

  // ---- final norm + LM head + greedy pick
  float *head_part = A.partials;
  a = head_args(A);
  is = gemv_begin<MW, EPI_LOGITS>(a, 0, ring, bid, nb);
  {
    PhaseOut po = gemv_run<MW, ACT, PRO_NORM, EPI_LOGITS>(a, 0, xs, scratch, ring, is, bid, nb);
    float *bv = xs;
    int *bi = reinterpret_cast<int *>(xs + MW);
    float vb = po.best;
    int ib = po.best_i;
    block_argmax(vb, ib, bv, bi);
    if (tid == 0) {
      head_part[bid * 2] = vb;
      reinterpret_cast<int *>(head_part)[bid * 2 + 1] = ib;
    }
  }
  if (!grid_barrier(A.bar, epoch, A.st.err)) return;
  if (bid == 0) {
    float *bv = xs;
    int *bi = reinterpret_cast<int *>(xs + MW);
    float vb = -INFINITY;
    int ib = 0x7fffffff;
    for (int b = tid; b < nb; b += blockDim.x) {
      const float bvv = __ldcg(head_part + b * 2);
      const int bii = __ldcg(reinterpret_cast<const int *>(head_part) + b * 2 + 1);
      if (bvv > vb || (bvv == vb && bii < ib)) { vb = bvv; ib = bii; }
    }
    block_argmax(vb, ib, bv, bi);
    if (tid != 0) return;
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

size_t mega_attn_tile_floats(int hd, int) {
  return (size_t)2 * ATILE * ((hd * 2 + 16) + hd * 2) / sizeof(float);  // the 2-slot K/V ring
}
int mega_warps() { return MW; }

}  // namespace rv
