// Single-row (batch 1) decode kernels of the River-LLM token-level early exit:
// one kernel per GEMV of the decode step, launched as a chain.
//
//   qkv  : exit decision of the layer before (s(l-1) = cos of its input and
//          output, from the same registers as) RMSNorm(h) -> [q;k;v] = W_qkv x
//          -> RoPE -> K/V into slot (l, 0, p)
//   attn : split-KV GQA decode attention (attention.cu)
//   o    : h_mid = h + W_o o
//   gu   : RMSNorm(h_mid) -> a = silu(W_g x) * (W_u x)
//   down : h_out = h_mid + W_d a
// and a final LM-head GEMV with a fused greedy argmax.  Every GEMV reads the
// row's route flag on the device and streams either the 16-bit backbone
// matrix or its int4 river copy (same kernel, same grid).  The GEMV itself is
// the shared core in gemv_core.cuh; here each kernel is one grid over it (the
// LM head's blocks combine their argmax candidates in the last block to
// finish).  In the programmatic-dependent-launch chain every kernel starts
// its weight stream before waiting on its predecessor; QKV streams the route
// it reads then and re-streams in the one layer per token where its decision
// flips the route.
//
// Method: "River-LLM: Large Language Model Seamless Exit Based on KV Share",
// paperlayer.ai summary section 4 (KV-Shared Exit Layer; Inference with
// Seamless Exit) and aitrends.kr (s(l) = cos(h(l-1), h(l)) > tau; W4A16 exit
// layers copied from the backbone blocks).
#include "gemv_core.cuh"

namespace rv {

constexpr int NW = 16;  // warps per block: one block per SM (the SM frees at once for the next kernel)

template <int ACT, int PRO, int EPI>
__global__ void __launch_bounds__(NW * 32, 1) k_gemv_b1(GemvArgs a) {
  extern __shared__ __align__(16) float smem[];
  const Geo g = geo_of(a.m);
  const int tid = threadIdx.x, warp = tid >> 5;
  float *scratch = smem + x_floats(g);
  char *ring = reinterpret_cast<char *>(scratch + 256) + (size_t)warp * NST * STAGE;

  // The route a GEMV streams is final before the kernel starts, except for
  // the QKV kernel, which itself makes the exit decision of the layer before
  // (from h_prev and h, available only after the wait).  QKV starts streaming
  // the matrices of the current route and re-streams in the one layer per
  // token where the decision flips it.  Every block reaches the same
  // decision (same sums in the same order); block 0 records it.  Another
  // block may already see block 0's update when it reads the route: the
  // update only ever says "river", which that block then decides as well.
  float *bsum = scratch + 128;
  int river = (EPI == EPI_LOGITS) ? 0 : ld_relaxed_i32(a.st.route);
  ItemStream is = gemv_begin<NW, EPI>(a, river, ring, blockIdx.x, gridDim.x);
  DecideScalars dsc{};
  if ((EPI == EPI_QKV || EPI == EPI_LOGITS) && a.decide_layer1 > 0) dsc = load_decide_scalars(a.st, 0);
  pdl_wait();
  pdl_trigger();
  float ss = -1.f;  // sum of h^2, shared by the decision and the RMSNorm prologue
  NormRegs nr;
  bool have_nr = false;
  if ((EPI == EPI_QKV || EPI == EPI_LOGITS) && a.decide_layer1 > 0) {
    float dot = 0.f, n1 = 0.f, n2 = 0.f;
    if (norm_fits(g)) {  // h and h_prev read once, kept for the RMSNorm prologue
      norm_load<true>(a, g, a.h_prev, nr);
      dot = nr.dot;
      n1 = nr.n1;
      n2 = nr.ss;
      have_nr = true;
    } else {
      for (int i = tid * 4; i < a.m.K; i += blockDim.x * 4) {
        const float4 x = __ldcg(reinterpret_cast<const float4 *>(a.h_prev + i));
        const float4 y = __ldcg(reinterpret_cast<const float4 *>(a.h + i));
        dot = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, dot))));
        n1 = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, n1))));
        n2 = fmaf(y.x, y.x, fmaf(y.y, y.y, fmaf(y.z, y.z, fmaf(y.w, y.w, n2))));
      }
    }
    const float3 t = block_sum3(dot, n1, n2, bsum);
    dot = t.x;
    n1 = t.y;
    n2 = t.z;
    ss = n2;
    const int route_now = (EPI == EPI_LOGITS) ? a.st.route[0] : river;
    const Decision dc = decide(dsc, route_now, a.decide_layer1, a.L, dot, n1, n2);
    if (blockIdx.x == 0 && tid == 0) commit_decision(a.st, 0, a.decide_layer1, dc, a.dbg_s);
    if (EPI == EPI_QKV && dc.route != river) {
      cp_wait<0>();  // drop the speculative items, then stream the river copy
      river = dc.route;
      is = gemv_begin<NW, EPI>(a, river, ring, blockIdx.x, gridDim.x);
    }
  }
  PhaseOut o = gemv_run<NW, ACT, PRO, EPI>(a, river, smem, scratch, ring, is, blockIdx.x, gridDim.x, ss,
                                           have_nr ? &nr : nullptr);

  if (EPI == EPI_DOWN) {
    (void)o;  // the next QKV (or the LM head) makes this layer's exit decision
  } else if (EPI == EPI_LOGITS) {
    // block argmax (lowest index on ties), then the last block to finish
    // reduces the blocks' candidates: both by shuffles, no serial loops
    __shared__ float bv[NW];
    __shared__ int bi[NW];
    float vb = o.best;
    int ib = o.best_i;
    block_argmax(vb, ib, bv, bi);
    if (tid == 0) {
      a.partials[blockIdx.x * 2] = vb;
      reinterpret_cast<int *>(a.partials)[blockIdx.x * 2 + 1] = ib;
    }
    if (!last_block(a.counter)) return;
    vb = -INFINITY;
    ib = 0x7fffffff;
    for (int b = tid; b < (int)gridDim.x; b += blockDim.x) {
      const float bvv = __ldcg(a.partials + b * 2);
      const int bii = __ldcg(reinterpret_cast<const int *>(a.partials) + b * 2 + 1);
      if (bvv > vb || (bvv == vb && bii < ib)) { vb = bvv; ib = bii; }
    }
    block_argmax(vb, ib, bv, bi);
    if (tid == 0) {
      a.st.next_ids[0] = ib == 0x7fffffff ? 0 : ib;
      a.st.len[0] += 1;
    }
  }
}

// ------------------------------------------------------------------ launch

// K splits per row quad (S warps of a block share a quad's chunks; 1, 2, 4
// or 8): the choice that gives the busiest warp of the launch the fewest work
// items, with at most grid_cap blocks; ties go to fewer splits (fewer
// cross-warp reductions).
static int best_splits(int nq, int nk, int grid_cap) {
  int best = 1;
  long best_cost = -1;
  for (int S = 1; S <= 8 && S <= nk; S *= 2) {
    const long iters = (nq + NW / S - 1) / (NW / S);  // block iterations of RG = NW / S quads
    const long grid = iters < grid_cap ? iters : grid_cap;
    const long cost = (iters + grid - 1) / grid * ((nk + S - 1) / S);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

template <int ACT, int PRO, int EPI>
static cudaError_t launch_t(const GemvArgs &a_in, int max_grid, cudaStream_t s, int pdl) {
  GemvArgs a = a_in;
  const Geo g = geo_of(a.m);
  const int nq = a.m.N / 4;
  const size_t smem = smem_bytes(g, NW);
  auto fn = k_gemv_b1<ACT, PRO, EPI>;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int per_sm = 0, dev = 0, n_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, NW * 32, smem);
  if (e != cudaSuccess) return e;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (per_sm < 1) per_sm = 1;
  // never beyond one resident wave; the grid-stride loop covers the rest
  int cap = per_sm * n_sm;
  if (cap > max_grid) cap = max_grid;
  a.s4 = best_splits(nq, g.nk4, cap);
  a.s16 = best_splits(nq, g.nk16, cap);
  // enough blocks for the path with more block iterations
  const int s_max = a.s4 > a.s16 ? a.s4 : a.s16;
  const int RG = NW / s_max;
  int grid = (nq + RG - 1) / RG;
  if (grid > cap) grid = cap;
  return launch_k(fn, dim3(grid), dim3(NW * 32), smem, s, pdl, a);
}

cudaError_t launch_gemv_b1(int act, int pro, int epi, const GemvArgs &a, int max_grid, cudaStream_t s, int pdl) {
  if (a.m.N % 4 || a.m.K % 8) return cudaErrorInvalidValue;
#define RV_DISPATCH(PRO_, EPI_)                                                                          \
  if (pro == PRO_ && epi == EPI_)                                                                        \
    return act ? launch_t<1, PRO_, EPI_>(a, max_grid, s, pdl) : launch_t<0, PRO_, EPI_>(a, max_grid, s, pdl);
  RV_DISPATCH(PRO_NORM, EPI_QKV)
  RV_DISPATCH(PRO_VEC, EPI_RESID)
  RV_DISPATCH(PRO_NORM, EPI_SWIGLU)
  RV_DISPATCH(PRO_VEC, EPI_DOWN)
  RV_DISPATCH(PRO_NORM, EPI_LOGITS)
#undef RV_DISPATCH
  return cudaErrorInvalidValue;
}

}  // namespace rv
