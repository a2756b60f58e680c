// Persistent, warp-specialized batch-1 decode step (stream.cu): argument
// block, the per-phase work plan shared by the producer and the consumers,
// and the host entry points.  Internal header.
#pragma once

#include <cuda.h>

#include "kernels.cuh"

namespace rv {
namespace sk {

constexpr int CW = 8;              // compute warps per block
constexpr int NTHREADS = (CW + 1) * 32;  // + one producer warp (one thread issues the tensor copies)
constexpr int RGR = 16;            // rows per row group (the MMA's M)
constexpr int CK4 = 1024;          // int4 codes per chunk (512 bytes of a row)
constexpr int CK16 = 256;          // 16-bit weights per chunk (512 bytes of a row)
// A stage holds one item as two tensor boxes of 8 rows x 4 x 128 bytes
// (rows 0..7 then 8..15 of the row group), each laid out [128-byte piece q]
// [row r][128 bytes] with the 128-byte swizzle (16-byte unit u of row r at
// unit u ^ r); for int4 the rows' (scale, zero) pairs follow.
constexpr int HALF_BYTES = 4096;
constexpr int SZ_OFF = 2 * HALF_BYTES;
constexpr int STAGE_BYTES = SZ_OFF + RGR * 64;  // room for 16 groups per row and chunk (g >= 64)
constexpr int MAX_STAGES = 24;
constexpr int ATILE = 32;          // attention positions per K/V tile

enum { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_DOWN = 3, PH_HEAD = 4 };

}  // namespace sk

// One decoder layer as the persistent kernel sees it (device array [L]).
struct LayerDesc {
  Mat m[4];  // fused QKV, O, fused gate/up, down (16-bit + river copy)
  // tensor maps (device memory) of each matrix: 16-bit weights, int4 codes,
  // (scale, zero) pairs; NULL where the matrix does not exist
  const CUtensorMap *tw[4], *tq[4], *ts[4];
  const uint16_t *attn_norm, *mlp_norm;
};

struct StreamArgs {
  const LayerDesc *layers;  // [L]
  const uint16_t *embed, *final_norm, *lm_head;
  const CUtensorMap *t_head;  // the LM head's tensor map
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
  unsigned long long wait_ns;  // limit of every bounded wait (the final drain excepted)
};

// Work of one GEMV phase for one block: row groups [j0, j1) of the matrix,
// each nk chunks (items) long, consumed by T teams of S warps (team t takes
// local row groups t, t + T, ...; member s of a team takes chunks s, s + S, ...).
struct PhasePlan {
  Mat m;
  int river;   // 1: int4 river copy, 0: 16-bit backbone matrix
  int epi;     // sk::PH_*
  int R, nk, j0, j1, S, T;
  const CUtensorMap *tm, *tsz;  // weights (16-bit or int4 codes), (scale, zero) pairs
  int szw;                      // (scale, zero) pairs per row in a stage (int4)
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

__host__ __device__ __forceinline__ PhasePlan make_plan(const Mat &m, int river, int epi, int bid, int nb,
                                                      const CUtensorMap *tw = nullptr, const CUtensorMap *tq = nullptr,
                                                      const CUtensorMap *ts = nullptr) {
  PhasePlan p;
  p.m = m;
  p.river = (river || !m.w) ? 1 : 0;  // an offloaded backbone layer exists only in the river
  p.tm = p.river ? tq : tw;
  p.tsz = ts;
  p.szw = p.river ? (sk::CK4 / m.r.g < m.r.Gs ? sk::CK4 / m.r.g : m.r.Gs) : 0;
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
// natural order, in the model's 16-bit type; int4 path: pair words
// (x[8W+p], x[8W+p+4]), p = 0..3, as fp16, zero beyond K up to whole groups,
// then per group the activation sums over even and odd k (two floats).
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
    x.bytes = x.xs_off + 8 * (((x.nw / x.wpg) + 3) & ~3);
  } else {
    x.nw = (x.nw_valid + 31) & ~31;
    x.wpg = 1;
    x.xs_off = 0;
    x.bytes = x.nw * 16;
  }
  return x;
}

// Tensor maps of the persistent engine (false if the driver refuses one):
// 16-bit weights [N][K] and int4 codes [N][Kp/8] as 3-D tensors (128-byte
// piece, row, piece index) with 8 x 4 x 128-byte boxes and the 128-byte
// swizzle; (scale, zero) pairs [N][Gs] as 2-D with min(1024 / g, Gs) x 8 boxes.
bool stream_map_w16(CUtensorMap *t, const void *w, int N, int K, int act);
bool stream_map_q(CUtensorMap *t, const void *q, int N, int Kp);
bool stream_map_sz(CUtensorMap *t, const void *sz, int N, int Gs, int g);

cudaError_t stream_prepare(StreamArgs &A, int n_sm, int *grid);
cudaError_t stream_launch(const StreamArgs &A, int grid, cudaStream_t s);
// Whether the stream engine supports these shapes (river group, dims).
bool stream_supported(int hd, int grp, int act, int group);

}  // namespace rv
