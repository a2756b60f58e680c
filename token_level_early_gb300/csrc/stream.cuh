// Persistent, warp-specialized batch-1 decode step (stream.cu): argument
// block, the per-phase work plan shared by the producer and the consumers,
// and the host entry points.  Internal header.
#pragma once

#include "kernels.cuh"

namespace rv {
namespace sk {

constexpr int CW = 8;              // compute warps per block
constexpr int PW = 8;              // producer warps per block (item n goes to producer n % PW)
constexpr int NTHREADS = (CW + PW) * 32;
constexpr int RGR = 16;            // rows per row group (the MMA's M)
constexpr int CK4 = 1024;          // int4 codes per chunk (512 bytes of a row)
constexpr int CK16 = 256;          // 16-bit weights per chunk (512 bytes of a row)
constexpr int ROW4 = 576;          // shared-memory row stride of an int4 stage (512 + 64 bytes)
constexpr int ROW16 = 528;         // shared-memory row stride of a 16-bit stage (512 + 16 bytes)
constexpr int SZ_OFF = RGR * ROW4;           // (scale, zero) rows of an int4 stage
constexpr int STAGE_BYTES = SZ_OFF + RGR * 64;  // room for 16 groups per row and chunk (g >= 64)
constexpr int MAX_STAGES = 24;
constexpr int ATILE = 32;          // attention positions per K/V tile

enum { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_DOWN = 3, PH_HEAD = 4 };

}  // namespace sk

// One decoder layer as the persistent kernel sees it (device array [L]).
struct LayerDesc {
  Mat m[4];  // fused QKV, O, fused gate/up, down (16-bit + river copy)
  const uint16_t *attn_norm, *mlp_norm;
};

struct StreamArgs {
  const LayerDesc *layers;  // [L]
  const uint16_t *embed, *final_norm, *lm_head;
  int L, d, H, Hkv, hd, F, V, act, Bmax;
  float eps;
  KVGeom kv;
  const float2 *rope_cs;
  StepState st;
  float *h[2], *hmid, *q, *o, *a;  // residual stream, q after RoPE, attention output, SwiGLU output
  float *attn_part;                // [H][att_splits][hd + 2]
  unsigned *attn_counter;          // [Hkv]: splits of a kv head done (the last one merges)
  int att_splits;
  float *partials;    // [2 * blocks]: the LM head's (value, index) per block
  unsigned *bar;      // [0] grid-barrier arrival counter (zeroed by the host before a step), [1] head counter
  float *dbg_h, *dbg_s, *dbg_logits;
  int nstages;        // ring stages
  int xbytes;         // activation / attention-tile region of shared memory
};

// Work of one GEMV phase for one block: row groups [j0, j1) of the matrix,
// each nk chunks (items) long, consumed by T teams of S warps (team t takes
// local row groups t, t + T, ...; member s of a team takes chunks s, s + S, ...).
struct PhasePlan {
  Mat m;
  int river;   // 1: int4 river copy, 0: 16-bit backbone matrix
  int epi;     // sk::PH_*
  int R, nk, j0, j1, S, T;
};

// Matrix row of row r (0..15) of row group j.  QKV: 8 consecutive rotary
// indices i of one head slot and their partners i + hd/2; gate/up: 8 gate
// rows and the matching up rows; otherwise 16 consecutive rows.  >= N: none.
__host__ __device__ __forceinline__ int rg_row(int epi, int j, int r, int N, int hd) {
  if (epi == sk::PH_QKV) {
    const int per = hd / 16, slot = j / per, i0 = (j - slot * per) * 8;
    return slot * hd + (r < 8 ? i0 + r : hd / 2 + i0 + r - 8);
  }
  if (epi == sk::PH_GU) {
    const int F = N / 2;
    return r < 8 ? j * 8 + r : F + j * 8 + r - 8;
  }
  return j * sk::RGR + r;
}

__host__ __device__ __forceinline__ int row_groups(int epi, int N) {
  if (epi == sk::PH_GU) return N / 16;  // N = 2F, F a multiple of 8
  return (N + sk::RGR - 1) / sk::RGR;   // QKV: N = slots * hd, hd a multiple of 16
}

// K splits per row group: the S (1, 2, 4 or 8) that gives the busiest warp
// the fewest items; ties go to fewer splits.
__host__ __device__ __forceinline__ void pick_team(int rmax, int nk, int &S, int &T) {
  int best = -1;
  S = 1;
  for (int s = 1; s <= sk::CW; s *= 2) {
    const int t = sk::CW / s, rounds = (rmax + t - 1) / t, per = (nk + s - 1) / s;
    const int cost = rounds * per;
    if (best < 0 || cost < best) {
      best = cost;
      S = s;
    }
  }
  T = sk::CW / S;
}

__host__ __device__ __forceinline__ PhasePlan make_plan(const Mat &m, int river, int epi, int bid, int nb) {
  PhasePlan p;
  p.m = m;
  p.river = (river || !m.w) ? 1 : 0;  // an offloaded backbone layer exists only in the river
  p.epi = epi;
  p.R = row_groups(epi, m.N);
  p.nk = p.river ? (m.r.Kp + sk::CK4 - 1) / sk::CK4 : (m.K + sk::CK16 - 1) / sk::CK16;
  p.j0 = (int)(((long)bid * p.R) / nb);
  p.j1 = (int)(((long)(bid + 1) * p.R) / nb);
  pick_team((p.R + nb - 1) / nb, p.nk, p.S, p.T);
  return p;
}

// Activations of a phase staged in shared memory: words of 8 values (16 bytes
// as 16-bit), a whole number of warps of them.  16-bit path: the vector in
// natural order; int4 path: pair words (x[8W+p], x[8W+p+4]), p = 0..3, zero
// beyond K up to whole groups, then the groups' activation sums (floats).
struct XGeom {
  int nw_valid;  // words holding activations
  int nw;        // words staged (a multiple of 32)
  int wpg;       // words per quantization group (int4 path; 1 otherwise)
  int xs_off;    // byte offset of the group sums (int4 path)
  int bytes;     // bytes of the region
};
__host__ __device__ __forceinline__ XGeom x_geom(const Mat &m, int river) {
  XGeom x;
  x.nw_valid = (m.K + 7) / 8;
  if (river) {
    const int g = m.r.g, kg = ((m.r.Kp + g - 1) / g) * g;
    x.nw = ((kg / 8) + 31) & ~31;
    x.wpg = g / 8;
    x.xs_off = x.nw * 16;
    x.bytes = x.xs_off + 4 * (((x.nw / x.wpg) + 3) & ~3);
  } else {
    x.nw = (x.nw_valid + 31) & ~31;
    x.wpg = 1;
    x.xs_off = 0;
    x.bytes = x.nw * 16;
  }
  return x;
}

cudaError_t stream_prepare(StreamArgs &A, int n_sm, int *grid);
cudaError_t stream_launch(const StreamArgs &A, int grid, cudaStream_t s);
// Whether the stream engine supports these shapes (river group, dims).
bool stream_supported(int hd, int grp, int act, int group);

}  // namespace rv
