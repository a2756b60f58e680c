// Persistent batch-1 decode-step kernel (mega.cu): argument block and host
// entry points.  Internal header.
#pragma once

#include "kernels.cuh"

namespace rv {

// One decoder layer as the persistent kernel sees it (device array [L]).
struct LayerDesc {
  Mat m[4];  // fused QKV, O, fused gate/up, down (16-bit + river copy)
  const uint16_t *attn_norm, *mlp_norm;
};

struct MegaArgs {
  const LayerDesc *layers;  // [L]
  const uint16_t *embed, *final_norm, *lm_head;
  int L, d, H, Hkv, hd, F, V, act, Bmax;
  float eps;
  KVGeom kv;
  const float2 *rope_cs;
  StepState st;
  float *h[2], *hmid, *q, *o, *a;  // residual stream, q after RoPE, attention output, SwiGLU output
  float *attn_part;                // [H][splits][hd + 2]
  int splits;
  float *partials;   // [2 * nblocks][3]: s(l) sums, then the head's (value, index)
  unsigned *bar;     // [0] arrival counter, [1] epoch
  float *dbg_h, *dbg_s, *dbg_logits;
  size_t xs_floats;  // activation / attention-tile region of dynamic shared memory
};

cudaError_t mega_prepare(MegaArgs &A, int n_sm, int *grid);
cudaError_t mega_launch(const MegaArgs &A, int grid, cudaStream_t s);
size_t mega_smem_bytes(const MegaArgs &A);
size_t mega_attn_tile_floats(int hd, int grp);
int mega_warps();

}  // namespace rv
