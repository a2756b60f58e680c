// Persistent, warp-specialized batch-1 decode step: the whole token
// (embedding, every layer on its backbone or river path, the exit decision,
// the LM head and the greedy pick) in one cooperative launch with one block
// per SM.
//
// Each block has one producer warp and CW compute warps.
//
// Producer: one thread walks the block's share of every weight matrix of the
// step in consumption order (layer by layer: QKV, O, gate/up, down; then the
// LM head) and copies it into a ring of shared-memory stages with tensor
// copies (TMA, completion counted in bytes on the stage's mbarrier; the
// copies bypass the load/store path that the compute warps' shared-memory
// reads use).  A stage is one item: 16 rows x one 512-byte chunk of each row (1024 int4
// codes plus their (scale, zero) pairs, or 256 16-bit weights).  The
// producer never waits on activations, only on free stages and, while the
// token is still in the backbone, on the route of the next layer (published
// by the compute warps when they take the exit decision), so the weight
// stream keeps running through grid barriers, activation loads, the
// attention phase and epilogues.
//
// Compute warps: for each phase, load the phase's activation vector (after a
// grid barrier), stage it in shared memory as 16-bit values, and consume
// their items: a row group of 16 rows is one mma.sync m16n8k16 row block,
// with the activation chunk as column 0 of B (the other columns zero).
//   16-bit path: A fragments straight from the stage (ldmatrix).
//   int4 path: a LOP3 turns two codes of a word into two fp16 values that
//   carry them in their mantissa, 1024 + q (nibbles at bits 0..3 of each
//   half: codes 8W, 8W+4 of word W) or 1024 + 16 q (bits 4..7: codes 8W+1,
//   8W+5); one shift by 8 exposes the other four codes, so a word costs one
//   shift and four LOP3s.  Lane (g, t) takes words t*w .. t*w + w - 1 of a
//   block of 4w words (one quantization group, w = group / 32) of rows g
//   and g + 8; the MMA's k order follows the nibbles, and the activations
//   are staged in the same order as fp16 pairs (x[8W+p], x[8W+p+4]) (the
//   model's 16-bit activations, exact in fp16 for |x| in [2^-14, 65504]).
//   The even-k codes (1024 + q) and the odd-k codes (1024 + 16 q) go to two
//   accumulators D0, D1; per group,
//     sum (q - z) x = D0 + D1 / 16 - (1024 + z) X0 - (64 + z) X1
//   with X0, X1 the group's activation sums over even and odd k, times the
//   group's scale, into fp32 row sums.
// Products of 16-bit values are exact; sums are fp32.  Row groups are split
// over teams of warps; partial sums meet in shared memory in a fixed order;
// the team's first warp runs the epilogue (RoPE + K/V append, residual,
// SwiGLU, argmax).
//
// Phases of layer l, separated by grid barriers:
//   QKV  : exit decision of layer l (1-based l, from h(l-1) and h(l); every
//          block reaches the same decision), RMSNorm(h) -> W_qkv -> RoPE ->
//          K/V into slot (l, 0, p)
//   ATTN : split-KV GQA attention over positions 0..p, one task per block;
//          the last split of a kv head to finish merges its heads' states
//   O    : h_mid = h + W_o o
//   GU   : RMSNorm(h_mid) -> a = silu(W_g x) * (W_u x)
//   DOWN : h_out = h_mid + W_d a
// then RMSNorm(h(L)) -> LM head -> greedy argmax.
//
// Every wait is bounded (grid barrier, stage and route waits): on a timeout a
// block sets an error bit (8: grid barrier, 32: stage ring) and an abort
// flag; all warps then run the rest of their control flow without waiting
// (named barriers stay matched), the producer drains its copies, and the
// kernel returns.
//
// Method: "River-LLM: Large Language Model Seamless Exit Based on KV Share",
// paperlayer.ai summary section 4 (KV-Shared Exit Layer; Inference with
// Seamless Exit) and aitrends.kr (s(l) = cos(h(l-1), h(l)) > tau; W4A16 exit
// layers copied from the backbone blocks).
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.cuh"
#include "stream.cuh"

namespace rv {
namespace sk {

// ---------------------------------------------------------------- primitives

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *m, uint64_t *bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          su32(dst)),
      "l"(m), "r"(su32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *m, uint64_t *bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          su32(dst)),
      "l"(m), "r"(su32(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t ph) {
  uint32_t ok;
  asm volatile("{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
               : "=r"(ok)
               : "r"(su32(b)), "r"(ph)
               : "memory");
  return ok != 0;
}
// Named barrier of the compute warps (id 1) and of a team (id 2 + team).
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory"); }
__device__ __forceinline__ void team_bar(int t, int S) {
  asm volatile("bar.sync %0, %1;" ::"r"(2 + t), "r"(S * 32) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int ACT>
__device__ __forceinline__ void mma16816(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  if (ACT == 1)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t *r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
  return d;
}

// int4 code extraction (fp16 for both activation types): from word w,
//   p0 = codes (8W, 8W+4)   as 1024 + q      (bits 0..3 of each half)
//   p1 = codes (8W+1, 8W+5) as 1024 + 16 q   (bits 4..7)
//   p2, p3 the same for (8W+2, 8W+6), (8W+3, 8W+7) from w >> 8.
constexpr uint32_t kNibLo = 0x000F000Fu, kNibHi = 0x00F000F0u, kF16_1024 = 0x64006400u;
__device__ __forceinline__ void code_pairs(uint32_t w, uint32_t mlo, uint32_t mhi, uint32_t o, uint32_t *p) {
  const uint32_t u = w >> 8;
  p[0] = lop3_and_or(w, mlo, o);
  p[1] = lop3_and_or(w, mhi, o);
  p[2] = lop3_and_or(u, mlo, o);
  p[3] = lop3_and_or(u, mhi, o);
}

// ---------------------------------------------------------------- shared state

struct Shared {
  uint64_t *full, *empty;       // [nstages] each
  unsigned char *ring;          // nstages x STAGE_BYTES
  unsigned char *xr;            // activation / attention-tile region
  float *red;                   // team partials [T][2][S][16] (at most 2 * CW * 16 floats)
  float *scr;                   // 128 floats of reduction scratch
  int *routes;                  // [L]
  volatile int *known;          // routes known for layers < *known
  volatile int *abort_flag;
  volatile int *issued;         // [nstages]: the last item issued into each stage
  int *misc;                    // [0] am-last flag
  unsigned long long wait_ns;   // limit of a bounded wait
};

__device__ __forceinline__ bool aborted(const Shared &sh) { return *sh.abort_flag != 0; }

__device__ __forceinline__ void set_abort(const Shared &sh, int32_t *err, int bit) {
  *sh.abort_flag = 1;
  atomicOr(err, bit);
}

__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s: far beyond any healthy step (the drain's limit)

// Bounded wait on a stage barrier; false on timeout (after sh.wait_ns) or abort.
// try_wait itself suspends the thread for a while, so the loop spins
// without sleeping (a sleep would add its wake-up latency to every item).
__device__ __forceinline__ bool wait_stage(const Shared &sh, uint64_t *b, uint32_t ph, int32_t *err) {
  if (mbar_try(b, ph)) return true;
  const unsigned long long t0 = gtime();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(b, ph)) return true;
    if (aborted(sh)) return false;
    if ((i & 63) == 0 && gtime() - t0 > sh.wait_ns) break;
  }
  set_abort(sh, err, 32);
  return false;
}

// A consumer's wait for item n.  Several warps consume one ring, so a warp
// can reach item n while its stage still holds an older item that has not
// landed; a parity test alone would then match the older item's phase.
// Once item n has been issued (the stage's marker says n), the stage's
// previous item has been consumed (its producer waited for that), so the
// parity test is exact.
__device__ __forceinline__ bool wait_item(const Shared &sh, int n, int NS, int32_t *err) {
  const unsigned q = (unsigned)n / (unsigned)NS;
  const int slot = n - (int)q * NS;
  if (sh.issued[slot] != n) {
    const unsigned long long t0 = gtime();
    for (uint32_t i = 1; sh.issued[slot] != n; ++i) {
      if (aborted(sh)) return false;
      if ((i & 255) == 0 && gtime() - t0 > sh.wait_ns) {
        set_abort(sh, err, 32);
        return false;
      }
    }
  }
  return wait_stage(sh, &sh.full[slot], q & 1u, err);
}

// Grid barrier of the compute warps: a counter that only grows within a
// launch; thread 0 adds 1 (release) and polls (acquire) until epoch x blocks
// have arrived.  Bounded: gives up (error bit 8, abort) after sh.wait_ns.
__device__ __forceinline__ void grid_barrier(const Shared &sh, unsigned *bar, unsigned &epoch, int32_t *err) {
  cbar();  // the block's writes are ordered before thread 0's release (cumulative)
  if (threadIdx.x == 0) {
    epoch += 1;
    const unsigned target = epoch * gridDim.x;
    red_release_add(bar, 1u);
    if (!aborted(sh)) {
      const unsigned long long t0 = gtime();
      while ((int)(ld_acquire(bar) - target) < 0) {
        if (gtime() - t0 > sh.wait_ns) {
          set_abort(sh, err, 8);
          break;
        }
        if (aborted(sh)) break;
      }
    }
  }
  cbar();  // the acquire above orders every later read of the block
}

// Sum over the compute warps (every compute thread gets the totals).
__device__ __forceinline__ float3 csum3(const Shared &sh, float a, float b, float c) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  c = warp_sum(c);
  cbar();
  if (lane == 0) {
    sh.scr[w] = a;
    sh.scr[32 + w] = b;
    sh.scr[64 + w] = c;
  }
  cbar();
  float3 t = make_float3(0.f, 0.f, 0.f);
  for (int i = 0; i < CW; ++i) {  // fixed order: deterministic
    t.x += sh.scr[i];
    t.y += sh.scr[32 + i];
    t.z += sh.scr[64 + i];
  }
  return t;
}

// ---------------------------------------------------------------- producer
// Item order of a phase (the consumers use the same): row groups in rounds of
// T (one per team); inside a round, chunk-major: (c = 0, teams 0..T-1),
// (c = 1, ...), so every team's next chunk is close in the stream.

// The producer: one thread walks every item of the step in consumption order
// and copies each into its stage with tensor copies (TMA): two boxes of 8
// rows x 512 bytes (rows 0..7 and 8..15 of the row group; the rows of a half
// are consecutive matrix rows for every epilogue's row order), and for an
// int4 item two boxes of the rows' (scale, zero) pairs.  The copies complete
// on the stage's mbarrier in bytes; rows past the matrix arrive as zeros.
__device__ void producer(const StreamArgs &A, const Shared &sh, int bid, int nb) {
  if ((threadIdx.x & 31) != 0) return;
  const int NS = A.nstages;
  int n = 0, slot = 0;  // items issued; stage of the next item
  uint32_t ph = 0;      // parity of the next item's stage use
  bool stop = false;
  auto put = [&](const PhasePlan &p) {
    const int Rb = p.j1 - p.j0, N = p.m.N, hd = A.hd;
    const int gpc = p.river ? CK4 / p.m.r.g : 0;
    const uint32_t bytes = 2 * HALF_BYTES + (p.river ? (uint32_t)(2 * 8 * p.szw * 4) : 0u);
    for (int r0 = 0; r0 < Rb && !stop; r0 += p.T) {
      const int tr = min(p.T, Rb - r0);
      for (int c = 0; c < p.nk && !stop; ++c)
        for (int t = 0; t < tr; ++t) {
          if (n >= NS && !wait_stage(sh, &sh.empty[slot], ph ^ 1u, A.st.err)) {
            stop = true;
            break;
          }
          const int j = p.j0 + r0 + t;
          const int row0 = rg_row(p.epi, j, 0, N, hd), row8 = rg_row(p.epi, j, 8, N, hd);
          unsigned char *stage = sh.ring + (size_t)slot * STAGE_BYTES;
          mbar_expect_tx(&sh.full[slot], bytes);
          tma3d(stage, p.tm, &sh.full[slot], 0, row0, 4 * c);
          tma3d(stage + HALF_BYTES, p.tm, &sh.full[slot], 0, row8, 4 * c);
          if (p.river) {
            tma2d(stage + SZ_OFF, p.tsz, &sh.full[slot], c * gpc, row0);
            tma2d(stage + SZ_OFF + 8 * p.szw * 4, p.tsz, &sh.full[slot], c * gpc, row8);
          }
          sh.issued[slot] = n;
          ++n;
          if (++slot == NS) {
            slot = 0;
            ph ^= 1u;
          }
        }
    }
  };
  for (int l = 0; l < A.L && !stop; ++l) {
    // the route of layer l: known from the start (forced exits), after the
    // exit (the river to the end), or once the compute warps have decided
    {
      const unsigned long long t0 = gtime();
      while (*sh.known <= l) {
        if (aborted(sh) || gtime() - t0 > sh.wait_ns) {
          if (!aborted(sh)) set_abort(sh, A.st.err, 32);
          stop = true;
          break;
        }
      }
      if (stop) break;
      __threadfence_block();
    }
    const int river = ((volatile int *)sh.routes)[l];
    const LayerDesc &ly = A.layers[l];
    put(make_plan(ly.m[0], river, PH_QKV, bid, nb, ly.tw[0], ly.tq[0], ly.ts[0]));
    put(make_plan(ly.m[1], river, PH_O, bid, nb, ly.tw[1], ly.tq[1], ly.ts[1]));
    put(make_plan(ly.m[2], river, PH_GU, bid, nb, ly.tw[2], ly.tq[2], ly.ts[2]));
    put(make_plan(ly.m[3], river, PH_DOWN, bid, nb, ly.tw[3], ly.tq[3], ly.ts[3]));
  }
  if (!stop) {
    Mat lm{};
    lm.w = A.lm_head;
    lm.N = A.V;
    lm.K = A.d;
    put(make_plan(lm, 0, PH_HEAD, bid, nb, A.t_head));
  }
  // drain: no copy may still be in flight when the block exits
  for (int m = n - NS < 0 ? 0 : n - NS; m < n; ++m) {
    const unsigned q = (unsigned)m / (unsigned)NS;
    const int sl = m - (int)q * NS;
    const unsigned long long t0 = gtime();
    while (!mbar_try(&sh.full[sl], q & 1u) && gtime() - t0 < kWaitNs) {
    }
  }
}

// ---------------------------------------------------------------- activation staging

// x (16-bit) of a phase into shared memory in the layout of its path.
// src: fp32 vector [K]; norm: multiply by r * gamma first (RMSNorm).
//   16-bit path: x16[k] natural order.
//   int4 path:   pair word W = (x[8W+p], x[8W+p+4]) for p = 0..3 as one uint4,
//                zero beyond K up to a whole number of groups; then the
//                groups' sums X[G] as floats.
template <int ACT>
__device__ __forceinline__ void stage_word(int river, int t, int wpg, const float *x, unsigned char *xr, float *xs) {
  uint4 *xw = reinterpret_cast<uint4 *>(xr);
  if (river) {
    // fp16 pairs (the values are already rounded to the model's 16-bit type;
    // clamped to the fp16 range)
    uint32_t pr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      pr[q] = (uint32_t)__half_as_ushort(__float2half_rn(fminf(fmaxf(x[q], -65504.f), 65504.f))) |
              ((uint32_t)__half_as_ushort(__float2half_rn(fminf(fmaxf(x[q + 4], -65504.f), 65504.f))) << 16);
    xw[t] = make_uint4(pr[0], pr[1], pr[2], pr[3]);
    float X0 = (x[0] + x[2]) + (x[4] + x[6]), X1 = (x[1] + x[3]) + (x[5] + x[7]);
    for (int o = 1; o < wpg; o <<= 1) {
      X0 += __shfl_xor_sync(0xffffffffu, X0, o);
      X1 += __shfl_xor_sync(0xffffffffu, X1, o);
    }
    if ((t & (wpg - 1)) == 0) reinterpret_cast<float2 *>(xs)[t / wpg] = make_float2(X0, X1);
  } else {
    xw[t] = make_uint4((uint32_t)f_to_act(x[0], ACT) | ((uint32_t)f_to_act(x[1], ACT) << 16),
                       (uint32_t)f_to_act(x[2], ACT) | ((uint32_t)f_to_act(x[3], ACT) << 16),
                       (uint32_t)f_to_act(x[4], ACT) | ((uint32_t)f_to_act(x[5], ACT) << 16),
                       (uint32_t)f_to_act(x[6], ACT) | ((uint32_t)f_to_act(x[7], ACT) << 16));
  }
}

// Plain vector (O: attention output, DOWN: SwiGLU output).
template <int ACT>
__device__ void stage_vec(const Mat &m, int river, const float *src, unsigned char *xr) {
  const XGeom xg = x_geom(m, river);
  const int nw = xg.nw_valid, nwr = xg.nw, wpg = xg.wpg;
  float *xs = reinterpret_cast<float *>(xr + xg.xs_off);
  const int ctid = threadIdx.x, lane = ctid & 31;
  for (int t0 = ctid; t0 < nwr; t0 += 4 * CW * 32) {
    float4 u[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = t0 + i * CW * 32;
      u[i][0] = u[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < nw && t * 8 < m.K) {
        const float4 *sp = reinterpret_cast<const float4 *>(src + t * 8);
        u[i][0] = __ldcg(sp);
        u[i][1] = __ldcg(sp + 1);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = t0 + i * CW * 32;
      if (t - lane >= nwr) break;
      const float x[8] = {u[i][0].x, u[i][0].y, u[i][0].z, u[i][0].w, u[i][1].x, u[i][1].y, u[i][1].z, u[i][1].w};
      if (t < nwr) stage_word<ACT>(river, t, wpg, x, xr, xs);
    }
  }
}

// RMSNorm of h with gain gamma; optionally also the exit decision's sums
// with h_prev.  ss / dot / n1 come back block-wide.
constexpr int NRW = 4;  // words per thread held in registers (d <= NRW * 8 * CW * 32 = 8192)
struct NormIn {
  float4 h[NRW][2];
  uint4 g[NRW];
};

template <int ACT>
__device__ void stage_norm(const Shared &sh, const Mat &m, int river, const float *h, const uint16_t *gamma, float eps,
                           const float *hprev, float3 *dec_sums, unsigned char *xr) {
  const XGeom xg = x_geom(m, river);
  const int nwr = xg.nw, wpg = xg.wpg;
  float *xs = reinterpret_cast<float *>(xr + xg.xs_off);
  const int ctid = threadIdx.x, lane = ctid & 31, K = m.K;
  float ss = 0.f, dot = 0.f, n1 = 0.f;
  if ((K + 7) / 8 <= NRW * CW * 32) {
    NormIn in;
#pragma unroll
    for (int i = 0; i < NRW; ++i) {
      const int t = ctid + i * CW * 32;
      in.h[i][0] = in.h[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      in.g[i] = make_uint4(0u, 0u, 0u, 0u);
      float4 p0 = make_float4(0.f, 0.f, 0.f, 0.f), p1 = p0;
      if (t * 8 < K) {
        const float4 *sp = reinterpret_cast<const float4 *>(h + t * 8);
        in.h[i][0] = __ldcg(sp);
        in.h[i][1] = __ldcg(sp + 1);
        in.g[i] = *reinterpret_cast<const uint4 *>(gamma + t * 8);
        if (hprev) {
          const float4 *pp = reinterpret_cast<const float4 *>(hprev + t * 8);
          p0 = __ldcg(pp);
          p1 = __ldcg(pp + 1);
        }
      }
      const float4 y0 = in.h[i][0], y1 = in.h[i][1];
      ss = fmaf(y0.x, y0.x, fmaf(y0.y, y0.y, fmaf(y0.z, y0.z, fmaf(y0.w, y0.w, ss))));
      ss = fmaf(y1.x, y1.x, fmaf(y1.y, y1.y, fmaf(y1.z, y1.z, fmaf(y1.w, y1.w, ss))));
      if (hprev) {
        dot = fmaf(p0.x, y0.x, fmaf(p0.y, y0.y, fmaf(p0.z, y0.z, fmaf(p0.w, y0.w, dot))));
        dot = fmaf(p1.x, y1.x, fmaf(p1.y, y1.y, fmaf(p1.z, y1.z, fmaf(p1.w, y1.w, dot))));
        n1 = fmaf(p0.x, p0.x, fmaf(p0.y, p0.y, fmaf(p0.z, p0.z, fmaf(p0.w, p0.w, n1))));
        n1 = fmaf(p1.x, p1.x, fmaf(p1.y, p1.y, fmaf(p1.z, p1.z, fmaf(p1.w, p1.w, n1))));
      }
    }
    const float3 t3 = csum3(sh, ss, dot, n1);
    if (dec_sums) *dec_sums = make_float3(t3.y, t3.z, t3.x);  // (dot, |h_prev|^2, |h|^2)
    const float r = 1.0f / sqrtf(t3.x / (float)K + eps);
    // the decision may have changed the route: the caller re-derives river
    // before this point, so the layout below is final
#pragma unroll
    for (int i = 0; i < NRW; ++i) {
      const int t = ctid + i * CW * 32;
      if (t - lane >= nwr) break;
      float x[8] = {in.h[i][0].x, in.h[i][0].y, in.h[i][0].z, in.h[i][0].w,
                    in.h[i][1].x, in.h[i][1].y, in.h[i][1].z, in.h[i][1].w};
      const uint16_t *gp = reinterpret_cast<const uint16_t *>(&in.g[i]);
#pragma unroll
      for (int q = 0; q < 8; ++q) x[q] = round_act(x[q] * r * act_to_f(gp[q], ACT), ACT);
      if (t < nwr) stage_word<ACT>(river, t, wpg, x, xr, xs);
    }
    // words beyond the register cache (none for d <= 8192) are staged below
  } else {
    for (int i = ctid * 4; i < K; i += CW * 32 * 4) {
      const float4 y = __ldcg(reinterpret_cast<const float4 *>(h + i));
      ss = fmaf(y.x, y.x, fmaf(y.y, y.y, fmaf(y.z, y.z, fmaf(y.w, y.w, ss))));
      if (hprev) {
        const float4 x = __ldcg(reinterpret_cast<const float4 *>(hprev + i));
        dot = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, dot))));
        n1 = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, n1))));
      }
    }
    const float3 t3 = csum3(sh, ss, dot, n1);
    if (dec_sums) *dec_sums = make_float3(t3.y, t3.z, t3.x);
    const float r = 1.0f / sqrtf(t3.x / (float)K + eps);
    for (int t = ctid; t < nwr; t += CW * 32) {
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (t * 8 < K) {
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(h + t * 8));
        const float4 b = __ldcg(reinterpret_cast<const float4 *>(h + t * 8) + 1);
        const uint4 gw = *reinterpret_cast<const uint4 *>(gamma + t * 8);
        const uint16_t *gp = reinterpret_cast<const uint16_t *>(&gw);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = round_act(v[q] * r * act_to_f(gp[q], ACT), ACT);
      }
      stage_word<ACT>(river, t, wpg, x, xr, xs);
    }
  }
}

// ---------------------------------------------------------------- GEMV consumer

// One group of an int4 item: the lane's w words of rows g and g + 8 against
// the activation pairs; even-k codes into d, odd-k codes into e (fp16 MMAs).
// Byte offset of word w (0..127) of a row within its half of a stage (the
// 128-byte swizzle: 16-byte unit u of row r sits at unit u ^ r).
__device__ __forceinline__ int sw_word(int w, int r) {
  return ((w >> 5) << 10) + (r << 7) + ((((w & 31) >> 2) ^ r) << 4) + ((w & 3) << 2);
}

template <int W>
__device__ __forceinline__ void group_mma(const unsigned char *h0, const unsigned char *h1, int r, const uint4 *xp,
                                          int w0, bool col0, uint32_t mlo, uint32_t mhi, uint32_t o, float *d,
                                          float *e) {
  uint32_t wa[W], wb[W];
  if (W == 2) {
    const int off = sw_word(w0, r);
    const uint2 a = *reinterpret_cast<const uint2 *>(h0 + off), b = *reinterpret_cast<const uint2 *>(h1 + off);
    wa[0] = a.x; wa[1 % W] = a.y; wb[0] = b.x; wb[1 % W] = b.y;
  } else {
#pragma unroll
    for (int i = 0; i < W; i += 4) {
      const int off = sw_word(w0 + i, r);
      const uint4 a = *reinterpret_cast<const uint4 *>(h0 + off), b = *reinterpret_cast<const uint4 *>(h1 + off);
      wa[i] = a.x; wa[(i + 1) % W] = a.y; wa[(i + 2) % W] = a.z; wa[(i + 3) % W] = a.w;
      wb[i] = b.x; wb[(i + 1) % W] = b.y; wb[(i + 2) % W] = b.z; wb[(i + 3) % W] = b.w;
    }
  }
#pragma unroll
  for (int i = 0; i < W; ++i) {
    uint4 xv = make_uint4(0u, 0u, 0u, 0u);
    if (col0) xv = xp[w0 + i];
    uint32_t pa[4], pb[4];
    code_pairs(wa[i], mlo, mhi, o, pa);
    code_pairs(wb[i], mlo, mhi, o, pb);
    mma16816<0>(d, pa[0], pb[0], pa[2], pb[2], xv.x, xv.z);  // codes 8W+{0,4}, 8W+{2,6}
    mma16816<0>(e, pa[1], pb[1], pa[3], pb[3], xv.y, xv.w);  // codes 8W+{1,5}, 8W+{3,7}
  }
}

// One int4 item (16 rows x one chunk) into the lane's row sums v0 (row g),
// v1 (row g + 8); lanes with t == 0 hold the meaningful values.  Two groups
// at a time, each on its own accumulators.
__device__ __forceinline__ void item_int4_fold(const __half2 *szs, const float2 *xs2, int c, int gpc, int szw,
                                               int blk, int gq, const float *d, const float *e, float &v0, float &v1) {
  const float2 X = xs2[c * gpc + blk];
  const float2 s0 = __half22float2(szs[gq * szw + blk]);
  const float2 s1 = __half22float2(szs[(gq + 8) * szw + blk]);
  const float b0 = fmaf(-(1024.f + s0.y), X.x, -(64.f + s0.y) * X.y);
  const float b1 = fmaf(-(1024.f + s1.y), X.x, -(64.f + s1.y) * X.y);
  v0 = fmaf(s0.x, fmaf(e[0], 0.0625f, d[0] + b0), v0);
  v1 = fmaf(s1.x, fmaf(e[2], 0.0625f, d[2] + b1), v1);
}

template <int W>
__device__ __forceinline__ void item_int4(const unsigned char *stage, const unsigned char *xr, const float *xs,
                                          int c, int nwc, int gpc, int szw, float &v0, float &v1, int lane) {
  const int gq = lane >> 2, tq = lane & 3;
  uint32_t mlo, mhi, o;
  asm("mov.b32 %0, %1;" : "=r"(mlo) : "n"(kNibLo));
  asm("mov.b32 %0, %1;" : "=r"(mhi) : "n"(kNibHi));
  asm("mov.b32 %0, %1;" : "=r"(o) : "n"(kF16_1024));
  const unsigned char *h0 = stage, *h1 = stage + HALF_BYTES;  // rows gq and gq + 8 (row gq of each half)
  const uint4 *xp = reinterpret_cast<const uint4 *>(xr) + c * (CK4 / 8);
  const __half2 *szs = reinterpret_cast<const __half2 *>(stage + SZ_OFF);
  const float2 *xs2 = reinterpret_cast<const float2 *>(xs);
  const int nblk = (nwc + 4 * W - 1) / (4 * W);
  const bool col0 = gq == 0;
  int blk = 0;
  for (; blk + 1 < nblk; blk += 2) {
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, e0[4] = {0.f, 0.f, 0.f, 0.f};
    float d1[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
    group_mma<W>(h0, h1, gq, xp, blk * 4 * W + tq * W, col0, mlo, mhi, o, d0, e0);
    group_mma<W>(h0, h1, gq, xp, (blk + 1) * 4 * W + tq * W, col0, mlo, mhi, o, d1, e1);
    if (tq == 0) {
      item_int4_fold(szs, xs2, c, gpc, szw, blk, gq, d0, e0, v0, v1);
      item_int4_fold(szs, xs2, c, gpc, szw, blk + 1, gq, d1, e1, v0, v1);
    }
  }
  if (blk < nblk) {
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, e0[4] = {0.f, 0.f, 0.f, 0.f};
    group_mma<W>(h0, h1, gq, xp, blk * 4 * W + tq * W, col0, mlo, mhi, o, d0, e0);
    if (tq == 0) item_int4_fold(szs, xs2, c, gpc, szw, blk, gq, d0, e0, v0, v1);
  }
}

// One 16-bit item into the MMA accumulators d (even k-steps) and e (odd);
// column 0 (lanes t == 0) holds the row sums.
template <int ACT>
__device__ __forceinline__ void item_16(const unsigned char *stage, const unsigned char *xr, int c, int nsteps,
                                        float *d, float *e, int lane) {
  const int gq = lane >> 2, tq = lane & 3;
  // ldmatrix: lane L gives row L & 15 (half (L & 15) >> 3, row r = L & 7 of
  // it) at k offset 8 * (L >> 4) of the k-step; k-step s is 128-byte piece
  // s >> 2, 16-byte unit 2 (s & 3) + (L >> 4), swizzled by r
  const int r = lane & 7, hi = lane >> 4;
  const uint32_t a_base = su32(stage) + ((lane & 15) >> 3) * HALF_BYTES + (r << 7);
  auto a_addr = [&](int s) { return a_base + ((s >> 2) << 10) + (((((s & 3) << 1) | hi) ^ r) << 4); };
  const uint32_t *x32 = reinterpret_cast<const uint32_t *>(xr) + c * (CK16 / 2);
  int s = 0;
#pragma unroll 2
  for (; s + 1 < nsteps; s += 2) {
    uint32_t a[4], b[4];
    ldsm_x4(a, a_addr(s));
    ldsm_x4(b, a_addr(s + 1));
    uint32_t x0 = 0u, x1 = 0u, x2 = 0u, x3 = 0u;
    if (gq == 0) {
      x0 = x32[s * 8 + tq];
      x1 = x32[s * 8 + 4 + tq];
      x2 = x32[s * 8 + 8 + tq];
      x3 = x32[s * 8 + 12 + tq];
    }
    mma16816<ACT>(d, a[0], a[1], a[2], a[3], x0, x1);
    mma16816<ACT>(e, b[0], b[1], b[2], b[3], x2, x3);
  }
  if (s < nsteps) {
    uint32_t a[4];
    ldsm_x4(a, a_addr(s));
    uint32_t x0 = 0u, x1 = 0u;
    if (gq == 0) {
      x0 = x32[s * 8 + tq];
      x1 = x32[s * 8 + 4 + tq];
    }
    mma16816<ACT>(d, a[0], a[1], a[2], a[3], x0, x1);
  }
}

// Epilogue context of a GEMV phase.
struct Epi {
  int l, pos;
  const float *h_base;  // O / DOWN: residual added to
  float *h_out;
  float *dbg_h;
  float best;  // LM head: this lane's candidate
  int best_i;
};

template <int ACT>
__device__ __forceinline__ void epilogue(const StreamArgs &A, const PhasePlan &p, Epi &e, int j, int gq, float y0,
                                         float y1) {
  const int N = p.m.N;
  const int row0 = rg_row(p.epi, j, gq, N, A.hd);
  if (p.epi == PH_QKV) {
    if (row0 >= N) return;
    const int hd = A.hd, half = hd >> 1, slot = row0 / hd, i = row0 - slot * hd;  // y1: row i + hd/2
    if (slot < A.H + A.Hkv) {
      const float2 cs = A.rope_cs[(size_t)e.pos * half + i];
      const float o0 = y0 * cs.x - y1 * cs.y, o1 = y0 * cs.y + y1 * cs.x;
      if (slot < A.H) {
        A.q[slot * hd + i] = round_act(o0, ACT);
        A.q[slot * hd + i + half] = round_act(o1, ACT);
      } else {
        uint16_t *kp = A.kv.base + A.kv.idx(e.l, 0, 0, slot - A.H, e.pos);
        kp[i] = f_to_act(o0, ACT);
        kp[i + half] = f_to_act(o1, ACT);
      }
    } else {
      uint16_t *vp = A.kv.base + A.kv.idx(e.l, 1, 0, slot - A.H - A.Hkv, e.pos);
      vp[i] = f_to_act(y0, ACT);
      vp[i + half] = f_to_act(y1, ACT);
    }
  } else if (p.epi == PH_GU) {
    const float sg = y0 / (1.0f + expf(-y0));
    A.a[row0] = round_act(sg * y1, ACT);
  } else if (p.epi == PH_HEAD) {
    const int r1 = row0 + 8;
    if (row0 < N) {
      if (A.dbg_logits) A.dbg_logits[row0] = y0;
      if (y0 > e.best || (y0 == e.best && row0 < e.best_i)) { e.best = y0; e.best_i = row0; }
    }
    if (r1 < N) {
      if (A.dbg_logits) A.dbg_logits[r1] = y1;
      if (y1 > e.best || (y1 == e.best && r1 < e.best_i)) { e.best = y1; e.best_i = r1; }
    }
  } else {  // residual (O, DOWN)
    const int r1 = row0 + 8;
    if (row0 < N) {
      const float v = __ldcg(e.h_base + row0) + y0;
      e.h_out[row0] = v;
      if (e.dbg_h) e.dbg_h[row0] = v;
    }
    if (r1 < N) {
      const float v = __ldcg(e.h_base + r1) + y1;
      e.h_out[r1] = v;
      if (e.dbg_h) e.dbg_h[r1] = v;
    }
  }
}

// Consume the block's items of one phase; returns the items consumed.
template <int ACT>
__device__ int consume(const StreamArgs &A, const Shared &sh, const PhasePlan &p, int nbase, Epi &e) {
  const int NS = A.nstages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  const int S = p.S, T = p.T, t = warp / S, s = warp % S;
  const int Rb = p.j1 - p.j0;
  const float *xs = reinterpret_cast<const float *>(sh.xr + x_geom(p.m, p.river).xs_off);
  const int gpc = p.river ? CK4 / p.m.r.g : 0, W = p.river ? p.m.r.g / 32 : 0;
  int par = 0;
  for (int r = t; r < Rb; r += T, par ^= 1) {
    float y0 = 0.f, y1 = 0.f, d[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
    // item order (shared with the producer): row groups in rounds of T (one
    // per team), chunk-major inside a round, so the teams advance together
    const int r0 = r - t, tr = min(T, Rb - r0);
    for (int c = s; c < p.nk; c += S) {
      const int n = nbase + r0 * p.nk + c * tr + t;
      const int slot = n - (int)((unsigned)n / (unsigned)NS) * NS;
      // every lane waits; the warp computes only if all lanes saw the data
      const bool ok = __all_sync(0xffffffffu, wait_item(sh, n, NS, A.st.err));
      if (ok) {
        const unsigned char *stg = sh.ring + (size_t)slot * STAGE_BYTES;
        if (p.river) {
          const int nwc = min(CK4, p.m.r.Kp - c * CK4) / 8;
          if (W == 4) item_int4<4>(stg, sh.xr, xs, c, nwc, gpc, p.szw, y0, y1, lane);
          else if (W == 2) item_int4<2>(stg, sh.xr, xs, c, nwc, gpc, p.szw, y0, y1, lane);
          else item_int4<8>(stg, sh.xr, xs, c, nwc, gpc, p.szw, y0, y1, lane);
        } else {
          item_16<ACT>(stg, sh.xr, c, min(CK16, p.m.K - c * CK16) / 16, d, d2, lane);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[slot]);
    }
    if (!p.river) {
      y0 = d[0] + d2[0];
      y1 = d[2] + d2[2];
    }
    if (S > 1) {
      float *rb = sh.red + ((t * 2 + par) * S) * 16;
      if (tq == 0) {
        rb[s * 16 + gq] = y0;
        rb[s * 16 + gq + 8] = y1;
      }
      team_bar(t, S);
      if (s == 0 && tq == 0) {
        y0 = 0.f;
        y1 = 0.f;
        for (int k = 0; k < S; ++k) {  // fixed order: deterministic
          y0 += rb[k * 16 + gq];
          y1 += rb[k * 16 + gq + 8];
        }
      }
    }
    if (s == 0 && tq == 0) epilogue<ACT>(A, p, e, p.j0 + r, gq, y0, y1);
  }
  return Rb * p.nk;
}

// ---------------------------------------------------------------- attention

template <int HD>
struct ATile {
  static constexpr int KROW = HD * 2 + 16;
  static constexpr int VROW = HD * 2;
  static constexpr int BYTES = ATILE * (KROW + VROW);
};

__device__ __forceinline__ void split_tiles(int p, int S, int sp, int &tb, int &te) {
  const int ntile = (p + ATILE - 1) / ATILE, per = (ntile + S - 1) / S;
  tb = min(ntile, sp * per);
  te = min(ntile, tb + per);
}

template <int HD>
__device__ __forceinline__ void attn_issue(const StreamArgs &A, int l, int g, int tile, int te, int p, int slot,
                                           unsigned char *ring_a) {
  using TL = ATile<HD>;
  if (tile < te) {
    const int t0 = tile * ATILE, n = min(ATILE, p - t0);
    const uint16_t *Kb = A.kv.base + A.kv.idx(l, 0, 0, g, 0), *Vb = A.kv.base + A.kv.idx(l, 1, 0, g, 0);
    const unsigned st = su32(ring_a) + slot * TL::BYTES;
    constexpr int PR = HD / 8;
    for (int v = threadIdx.x; v < 2 * ATILE * PR; v += CW * 32) {
      const int kv = v >= ATILE * PR, rem = v - kv * ATILE * PR, t = rem / PR, c = rem - t * PR;
      if (t < n)
        cp16s(st + (kv ? ATILE * TL::KROW + t * TL::VROW : t * TL::KROW) + c * 16,
              (kv ? Vb : Kb) + (size_t)(t0 + t) * HD + c * 8);
    }
  }
  cp_commit();
}

// Split sp of kv head g: positions of tiles [tb, te) of 0..p-1 and, for the
// last split, position p; warps 0..GRP-1 take the GRP query heads.  The
// last split of the head to finish merges the splits' states into o.
template <int ACT, int HD, int GRP>
__device__ void attn_task(const StreamArgs &A, const Shared &sh, int l, int task, int p, bool first_issued) {
  using TL = ATile<HD>;
  constexpr int PER = HD / 32, PR = HD / 8;
  const int S = A.att_splits;
  const int g = task / S, sp = task - g * S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char *ring_a = sh.xr;
  uint32_t *qs = reinterpret_cast<uint32_t *>(sh.xr + 2 * TL::BYTES);  // GRP * HD / 2 words
  int tb, te;
  split_tiles(p, S, sp, tb, te);
  if (!first_issued) attn_issue<HD>(A, l, g, tb, te, p, 0, ring_a);
  for (int i = threadIdx.x; i < GRP * HD / 2; i += CW * 32) {
    const float2 v = __ldcg(reinterpret_cast<const float2 *>(A.q + (size_t)g * GRP * HD) + i);
    qs[i] = (uint32_t)f_to_act(v.x, ACT) | ((uint32_t)f_to_act(v.y, ACT) << 16);
  }
  const int hw = warp < GRP ? warp : 0;
  const int h = g * GRP + hw;
  const uint4 *q4 = reinterpret_cast<const uint4 *>(qs + hw * (HD / 2));
  const float scale = 1.0f / sqrtf((float)HD);
  float mrun = -INFINITY, lrun = 0.f, o[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) o[r] = 0.f;
  for (int tile = tb, it = 0; tile < te; ++tile, ++it) {
    cbar();  // every warp is done with the slot refilled next (and qs is written)
    attn_issue<HD>(A, l, g, tile + 1, te, p, (it + 1) & 1, ring_a);
    cp_wait<1>();
    cbar();
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
      for (int t2 = 0; t2 < n; ++t2) {
        const float pt = __shfl_sync(0xffffffffu, pe, t2);
        const uint16_t *vr = reinterpret_cast<const uint16_t *>(tv + t2 * TL::VROW) + lane * PER;
#pragma unroll
        for (int r = 0; r < PER; ++r) o[r] = fmaf(pt, act_to_f(vr[r], ACT), o[r]);
      }
      mrun = mnew;
    }
  }
  cp_wait<0>();
  if (te <= tb) cbar();  // qs written before use
  if (warp < GRP) {
    if (sp == S - 1) {  // position p, written in the QKV phase
      const float *qp = A.q + (size_t)h * HD;
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
  // the last split of kv head g to finish merges (no waiting)
  __threadfence();
  cbar();
  if (threadIdx.x == 0) {
    const unsigned t = atomicAdd(A.attn_counter + g, 1u);
    sh.misc[0] = t == (unsigned)S - 1;
    if (t == (unsigned)S - 1) A.attn_counter[g] = 0u;
  }
  cbar();
  if (!sh.misc[0]) return;
  __threadfence();
  if (warp < GRP) {
    const float *base = A.attn_part + (size_t)h * S * (HD + 2);
    float M = -INFINITY;
    for (int s2 = 0; s2 < S; ++s2) M = fmaxf(M, __ldcg(base + s2 * (HD + 2) + HD));
    float Ls = 0.f, acc[PER];
#pragma unroll
    for (int r = 0; r < PER; ++r) acc[r] = 0.f;
    for (int s2 = 0; s2 < S; ++s2) {
      const float ms = __ldcg(base + s2 * (HD + 2) + HD);
      const float w = ms == -INFINITY ? 0.f : expf(ms - M);
      Ls = fmaf(w, __ldcg(base + s2 * (HD + 2) + HD + 1), Ls);
#pragma unroll
      for (int r = 0; r < PER; ++r) acc[r] = fmaf(w, __ldcg(base + s2 * (HD + 2) + lane * PER + r), acc[r]);
    }
    const float inv = 1.0f / Ls;
#pragma unroll
    for (int r = 0; r < PER; ++r) A.o[(size_t)h * HD + lane * PER + r] = round_act(acc[r] * inv, ACT);
  }
}

// ---------------------------------------------------------------- the kernel

template <int ACT, int HD, int GRP>
__global__ void __launch_bounds__(NTHREADS, 1) k_decode_stream(StreamArgs A) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // the swizzled tensor boxes need 1024-byte aligned stages
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int NS = A.nstages;
  Shared sh;
  sh.ring = smem;
  sh.xr = smem + (size_t)NS * STAGE_BYTES;
  unsigned char *tail = sh.xr + A.xbytes;
  sh.red = reinterpret_cast<float *>(tail);
  sh.scr = sh.red + 2 * CW * 16;
  sh.full = reinterpret_cast<uint64_t *>(sh.scr + 128);
  sh.empty = sh.full + NS;
  int *ip = reinterpret_cast<int *>(sh.empty + NS);
  sh.known = ip;
  sh.abort_flag = ip + 1;
  sh.misc = ip + 2;
  sh.issued = ip + 4;
  sh.routes = ip + 4 + NS;
  sh.wait_ns = A.wait_ns ? A.wait_ns : kWaitNs;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, bid = blockIdx.x, nb = gridDim.x;
  const int L = A.L;
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sh.full[i], 1);   // the producer's arrive (with the item's byte count)
      mbar_init(&sh.empty[i], 1);  // the consuming warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *sh.abort_flag = 0;
    for (int i = 0; i < NS; ++i) sh.issued[i] = -1;
    // routes known at the start: forced exits give every layer's route; the
    // tau rule starts in the backbone (the first decision follows layer 1)
    int known = 1;
    if (*A.st.mode == 1) {
      int f = A.st.forced[0];
      if (f < 0 || f > L) {
        if (bid == 0) atomicOr(A.st.err, 2);
        f = L;
      }
      const int cap = *A.st.cap;
      for (int i = 0; i < L; ++i) sh.routes[i] = (i >= f || i >= cap) ? 1 : 0;
      known = L;
    } else {
      sh.routes[0] = 0;
      for (int i = 1; i < L; ++i) sh.routes[i] = 0;
    }
    __threadfence_block();
    *sh.known = known;
  }
  __syncthreads();

  if (warp == CW) {  // ------------------------------------------------ producer
    producer(A, sh, bid, nb);
    return;
  }

  // ------------------------------------------------------------------ compute warps
  unsigned epoch = 0;
  const int pos = A.st.len[0];
  const DecideScalars dsc = load_decide_scalars(A.st, 0);  // read once: the decisions wait on no memory
  // the route and exit layer as the decisions below update them (forced
  // exit 0: every layer in the river)
  int route = 0, exit_l = L;
  if (*A.st.mode == 1) {
    int f = A.st.forced[0];
    if (f < 0 || f > L) f = L;
    if (f == 0) {
      route = 1;
      exit_l = 0;
    }
  }
  {
    int tok = A.st.tokens[0];
    if (tok < 0 || tok >= A.V) {
      if (bid == 0 && tid == 0) atomicOr(A.st.err, 1);
      tok = 0;
    }
    for (int i = bid * CW * 32 + tid; i < A.d; i += nb * CW * 32) {
      const float v = act_to_f(A.embed[(size_t)tok * A.d + i], ACT);
      A.h[0][i] = v;
      if (A.dbg_h) A.dbg_h[i] = v;
    }
  }
  grid_barrier(sh, A.bar, epoch, A.st.err);

  int nbase = 0;
  const int S_att = A.att_splits;
  for (int l = 0; l < L; ++l) {
    const LayerDesc &ly = A.layers[l];
    float *hin = A.h[l & 1], *hout = A.h[(l + 1) & 1];
    // ---- QKV (+ the exit decision of layer l, 1-based)
    {
      float3 ds = make_float3(0.f, 0.f, 0.f);
      const bool decide_now = l > 0 && route == 0;
      // stage for the route before the decision; re-stage if it flips
      PhasePlan p = make_plan(ly.m[0], route, PH_QKV, bid, nb, ly.tw[0], ly.tq[0], ly.ts[0]);
      stage_norm<ACT>(sh, p.m, p.river, hin, ly.attn_norm, A.eps, decide_now ? A.h[(l - 1) & 1] : nullptr,
                      decide_now ? &ds : nullptr, sh.xr);
      if (l > 0) {
        if (decide_now) {
          const Decision dc = decide(dsc, 0, l, L, ds.x, ds.y, ds.z);
          if (bid == 0 && tid == 0 && A.dbg_s) A.dbg_s[(size_t)(l - 1) * A.Bmax] = dc.s;
          if (dc.exited) {
            route = 1;
            exit_l = l;
          }
        } else if (bid == 0 && tid == 0 && A.dbg_s) {
          A.dbg_s[(size_t)(l - 1) * A.Bmax] = __int_as_float(0x7fc00000);
        }
        if (tid == 0 && *sh.known <= l) {  // publish for the producer
          for (int i = l; i < L; ++i) sh.routes[i] = route;
          __threadfence_block();
          *sh.known = route ? L : l + 1;
        }
      }
      cbar();
      if (p.river != (route || !ly.m[0].w ? 1 : 0)) {
        p = make_plan(ly.m[0], route, PH_QKV, bid, nb, ly.tw[0], ly.tq[0], ly.ts[0]);
        stage_norm<ACT>(sh, p.m, p.river, hin, ly.attn_norm, A.eps, nullptr, nullptr, sh.xr);
        cbar();
      }
      Epi e{l, pos, nullptr, nullptr, nullptr, 0.f, 0};
      nbase += consume<ACT>(A, sh, p, nbase, e);
    }
    // this block's first K/V tile of the attention (positions < p are final)
    cbar();
    const int task = bid;
    if (task < A.Hkv * S_att) {
      int tb, te;
      split_tiles(pos, S_att, task % S_att, tb, te);
      attn_issue<HD>(A, l, task / S_att, tb, te, pos, 0, sh.xr);
    }
    grid_barrier(sh, A.bar, epoch, A.st.err);
    // ---- attention (one task per block; more tasks than blocks loop)
    for (int tk = bid; tk < A.Hkv * S_att; tk += nb) {
      cbar();
      attn_task<ACT, HD, GRP>(A, sh, l, tk, pos, tk == bid);
    }
    cp_wait<0>();
    grid_barrier(sh, A.bar, epoch, A.st.err);
    // ---- O + residual
    {
      PhasePlan p = make_plan(ly.m[1], route, PH_O, bid, nb, ly.tw[1], ly.tq[1], ly.ts[1]);
      stage_vec<ACT>(p.m, p.river, A.o, sh.xr);
      cbar();
      Epi e{l, pos, hin, A.hmid, nullptr, 0.f, 0};
      nbase += consume<ACT>(A, sh, p, nbase, e);
    }
    grid_barrier(sh, A.bar, epoch, A.st.err);
    // ---- gate/up + SwiGLU
    {
      PhasePlan p = make_plan(ly.m[2], route, PH_GU, bid, nb, ly.tw[2], ly.tq[2], ly.ts[2]);
      stage_norm<ACT>(sh, p.m, p.river, A.hmid, ly.mlp_norm, A.eps, nullptr, nullptr, sh.xr);
      cbar();
      Epi e{l, pos, nullptr, nullptr, nullptr, 0.f, 0};
      nbase += consume<ACT>(A, sh, p, nbase, e);
    }
    grid_barrier(sh, A.bar, epoch, A.st.err);
    // ---- down + residual
    {
      PhasePlan p = make_plan(ly.m[3], route, PH_DOWN, bid, nb, ly.tw[3], ly.tq[3], ly.ts[3]);
      stage_vec<ACT>(p.m, p.river, A.a, sh.xr);
      cbar();
      Epi e{l, pos, A.hmid, hout, A.dbg_h ? A.dbg_h + (size_t)(l + 1) * A.Bmax * A.d : nullptr, 0.f, 0};
      nbase += consume<ACT>(A, sh, p, nbase, e);
    }
    grid_barrier(sh, A.bar, epoch, A.st.err);
  }

  // s(L) for the debug dump (no exit after the last layer)
  if (A.dbg_s && bid == 0) {
    const float *hp = A.h[(L - 1) & 1], *hc = A.h[L & 1];
    float dot = 0.f, n1 = 0.f, n2 = 0.f;
    for (int i = tid; i < A.d; i += CW * 32) {
      const float x = __ldcg(hp + i), y = __ldcg(hc + i);
      dot = fmaf(x, y, dot);
      n1 = fmaf(x, x, n1);
      n2 = fmaf(y, y, n2);
    }
    const float3 t3 = csum3(sh, dot, n1, n2);
    const Decision dc = decide(dsc, route, L, L, t3.x, t3.y, t3.z);
    if (tid == 0) A.dbg_s[(size_t)(L - 1) * A.Bmax] = dc.s;
  }

  // ---- final norm + LM head + greedy pick
  Mat lm{};
  lm.w = A.lm_head;
  lm.N = A.V;
  lm.K = A.d;
  PhasePlan ph = make_plan(lm, 0, PH_HEAD, bid, nb, A.t_head);
  stage_norm<ACT>(sh, ph.m, 0, A.h[L & 1], A.final_norm, A.eps, nullptr, nullptr, sh.xr);
  cbar();
  Epi e{L, pos, nullptr, nullptr, nullptr, -INFINITY, 0x7fffffff};
  nbase += consume<ACT>(A, sh, ph, nbase, e);
  // block argmax (lowest index on ties), then the last block to finish
  // reduces the blocks' candidates
  float vb = e.best;
  int ib = e.best_i;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, vb, o);
    const int oi = __shfl_xor_sync(0xffffffffu, ib, o);
    if (ov > vb || (ov == vb && oi < ib)) { vb = ov; ib = oi; }
  }
  cbar();
  if (lane == 0) {
    sh.scr[warp] = vb;
    reinterpret_cast<int *>(sh.scr)[32 + warp] = ib;
  }
  cbar();
  if (tid == 0) {
    for (int w2 = 0; w2 < CW; ++w2) {
      const float v = sh.scr[w2];
      const int i = reinterpret_cast<int *>(sh.scr)[32 + w2];
      if (v > vb || (v == vb && i < ib)) { vb = v; ib = i; }
    }
    A.partials[bid * 2] = vb;
    reinterpret_cast<int *>(A.partials)[bid * 2 + 1] = ib;
    __threadfence();
    const unsigned t = atomicAdd(A.bar + 1, 1u);
    sh.misc[0] = t == (unsigned)nb - 1;
  }
  cbar();
  if (!sh.misc[0]) return;
  __threadfence();
  vb = -INFINITY;
  ib = 0x7fffffff;
  for (int b = tid; b < nb; b += CW * 32) {
    const float v = __ldcg(A.partials + b * 2);
    const int i = __ldcg(reinterpret_cast<const int *>(A.partials) + b * 2 + 1);
    if (v > vb || (v == vb && i < ib)) { vb = v; ib = i; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, vb, o);
    const int oi = __shfl_xor_sync(0xffffffffu, ib, o);
    if (ov > vb || (ov == vb && oi < ib)) { vb = ov; ib = oi; }
  }
  cbar();
  if (lane == 0) {
    sh.scr[warp] = vb;
    reinterpret_cast<int *>(sh.scr)[32 + warp] = ib;
  }
  cbar();
  if (tid == 0) {
    for (int w2 = 0; w2 < CW; ++w2) {
      const float v = sh.scr[w2];
      const int i = reinterpret_cast<int *>(sh.scr)[32 + w2];
      if (v > vb || (v == vb && i < ib)) { vb = v; ib = i; }
    }
    A.st.next_ids[0] = ib == 0x7fffffff ? 0 : ib;
    A.st.route[0] = route;
    A.st.exit_layer[0] = exit_l;
    // a step whose waits ran out did not happen: the position stays (its
    // K/V slot is rewritten by the next step)
    if ((*(volatile int32_t *)A.st.err & (8 | 32)) == 0) A.st.len[0] = pos + 1;
    A.bar[1] = 0u;
  }
}

}  // namespace sk

// ------------------------------------------------------------------ host side

namespace {

size_t stream_smem(const StreamArgs &A) {
  return 1024 + (size_t)A.nstages * sk::STAGE_BYTES + A.xbytes + sizeof(float) * (2 * sk::CW * 16 + 128) +
         2 * sizeof(uint64_t) * A.nstages + sizeof(int) * (4 + A.nstages + A.L);
}

template <int ACT, int HD, int GRP>
cudaError_t prepare_t(StreamArgs &A, int n_sm, int *grid) {
  auto fn = sk::k_decode_stream<ACT, HD, GRP>;
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  // as many stages (each with its two mbarriers) as fit next to the activation region
  A.nstages = 0;
  const size_t fixed = stream_smem(A), per = sk::STAGE_BYTES + 2 * sizeof(uint64_t) + sizeof(int);
  if ((size_t)optin < fixed + 4 * per) return cudaErrorInvalidValue;
  int ns = (int)(((size_t)optin - fixed) / per);
  A.nstages = ns > sk::MAX_STAGES ? sk::MAX_STAGES : ns;
  const size_t smem = stream_smem(A);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, sk::NTHREADS, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  *grid = n_sm;  // one resident block per SM
  return cudaSuccess;
}

template <int ACT, int HD, int GRP>
cudaError_t launch_t(const StreamArgs &A, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(sk::NTHREADS);
  cfg.dynamicSmemBytes = stream_smem(A);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, sk::k_decode_stream<ACT, HD, GRP>, A);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool stream_map_w16(CUtensorMap *t, const void *w, int N, int K, int act) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!enc || !w || N < 1 || K < 8) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)N, (cuuint64_t)((K + 63) / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128};
  cuuint32_t box[3] = {64, 8, 4}, es[3] = {1, 1, 1};
  return enc(t, act == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(w),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool stream_map_q(CUtensorMap *t, const void *q, int N, int Kp) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!enc || !q || N < 1 || Kp < 32) return false;
  cuuint64_t dims[3] = {32, (cuuint64_t)N, (cuuint64_t)((Kp / 8 + 31) / 32)};
  cuuint64_t strides[2] = {(cuuint64_t)Kp / 2, 128};
  cuuint32_t box[3] = {32, 8, 4}, es[3] = {1, 1, 1};
  return enc(t, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(q), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool stream_map_sz(CUtensorMap *t, const void *sz, int N, int Gs, int g) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!enc || !sz || N < 1 || Gs < 4 || g < 64) return false;
  const int gpc = sk::CK4 / g, w = gpc < Gs ? gpc : Gs;
  cuuint64_t dims[2] = {(cuuint64_t)Gs, (cuuint64_t)N};
  cuuint64_t strides[1] = {(cuuint64_t)Gs * 4};
  cuuint32_t box[2] = {(cuuint32_t)w, 8}, es[2] = {1, 1};
  return enc(t, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(sz), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#define RV_STREAM_DISPATCH(CALL)                                      \
  const int grp = A.H / A.Hkv;                                        \
  if (A.act == 1 && A.hd == 128 && grp == 4) return CALL(1, 128, 4);  \
  if (A.act == 1 && A.hd == 64 && grp == 4) return CALL(1, 64, 4);    \
  if (A.act == 0 && A.hd == 64 && grp == 2) return CALL(0, 64, 2);    \
  if (A.act == 1 && A.hd == 64 && grp == 2) return CALL(1, 64, 2);    \
  if (A.act == 0 && A.hd == 128 && grp == 4) return CALL(0, 128, 4);  \
  if (A.act == 0 && A.hd == 64 && grp == 4) return CALL(0, 64, 4);    \
  return cudaErrorNotSupported;

bool stream_supported(int hd, int grp, int act, int group) {
  const bool shape = (hd == 128 && grp == 4) || (hd == 64 && (grp == 4 || grp == 2));
  (void)act;
  return shape && (group == 0 || group == 64 || group == 128 || group == 256);
}

cudaError_t stream_prepare(StreamArgs &A, int n_sm, int *grid) {
#define RV_P(ACT_, HD_, G_) prepare_t<ACT_, HD_, G_>(A, n_sm, grid)
  RV_STREAM_DISPATCH(RV_P)
#undef RV_P
}

cudaError_t stream_launch(const StreamArgs &A, int grid, cudaStream_t s) {
#define RV_L(ACT_, HD_, G_) launch_t<ACT_, HD_, G_>(A, grid, s)
  RV_STREAM_DISPATCH(RV_L)
#undef RV_L
}

}  // namespace rv
