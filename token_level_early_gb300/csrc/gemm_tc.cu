// Rows GEMM on the 5th-generation tensor cores (tcgen05) for the general
// path (prefill and batched decode): Y[m][n] = sum_k W[n][k] X[m][k] for the
// listed rows m, W a 16-bit backbone matrix [N][K].
//
// The listed rows of X (fp32 values already rounded to the model's 16-bit
// type, so the conversion is exact) are gathered into a compact 16-bit
// staging buffer; then one CTA per 128 x 128 tile of (rows, outputs):
// TMA copies 128 x 64 tiles of both operands (128-byte swizzle, K-major)
// into a 4-stage shared-memory ring, one thread issues tcgen05.mma
// (M = 128, N = 128, K = 16 per instruction, fp32 accumulator in tensor
// memory) and commits each stage back to the ring, and the four warps read
// the accumulator out of tensor memory (tcgen05.ld, one warp per 32 rows)
// and store the listed rows.  Products of 16-bit values are exact; the sums
// are fp32.  Every mbarrier wait is bounded: on timeout the kernel sets
// error bit 16, frees its tensor memory and returns.
//
// Method context: prefill runs the backbone layers 1..e over all prompt
// tokens (paperlayer.ai section 4, sequence-level exit in prefill).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace rv {

namespace {

constexpr int TBM = 128, TBN = 128, TBK = 64, TST = 4;
constexpr int TA_BYTES = TBM * TBK * 2, TB_BYTES = TBN * TBK * 2;
constexpr int TSMEM = 1024 + TST * (TA_BYTES + TB_BYTES) + 256;
constexpr uint32_t kWaitLimit = 1u << 20;

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t ph) {
  uint32_t ok;
  asm volatile("{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
               : "=r"(ok)
               : "r"(su32(b)), "r"(ph)
               : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t ph) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try(b, ph)) return true;
  return false;
}
__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *m, uint64_t *b, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          su32(dst)),
      "l"(m), "r"(su32(b)), "r"(x), "r"(y)
      : "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
  d |= (uint64_t)1 << 16;                   // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset
  d |= (uint64_t)1 << 46;                   // descriptor version
  d |= (uint64_t)2 << 61;                   // 128-byte swizzle
  return d;
}
__device__ __forceinline__ void umma(uint32_t dt, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
  asm volatile("{.reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;}" ::"r"(dt),
               "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
               : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t ta, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Gather the listed rows of X into the 16-bit staging buffer Xb [rows][K].
__global__ void k_pack_rows(const float *X, int K, int act, const int32_t *list, const int32_t *count, uint16_t *Xb,
                            int max_rows) {
  const int cnt = min(*count, max_rows), per = K / 8;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < (long)cnt * per; i += (long)gridDim.x * blockDim.x) {
    const int r = (int)(i / per), c = (int)(i - (long)r * per) * 8;
    const int m = list ? list[r] : r;
    const float4 a = *reinterpret_cast<const float4 *>(X + (size_t)m * K + c);
    const float4 b = *reinterpret_cast<const float4 *>(X + (size_t)m * K + c + 4);
    uint4 o;
    o.x = (uint32_t)f_to_act(a.x, act) | ((uint32_t)f_to_act(a.y, act) << 16);
    o.y = (uint32_t)f_to_act(a.z, act) | ((uint32_t)f_to_act(a.w, act) << 16);
    o.z = (uint32_t)f_to_act(b.x, act) | ((uint32_t)f_to_act(b.y, act) << 16);
    o.w = (uint32_t)f_to_act(b.z, act) | ((uint32_t)f_to_act(b.w, act) << 16);
    *reinterpret_cast<uint4 *>(Xb + (size_t)r * K + c) = o;
  }
}

template <int ACT>
__global__ void __launch_bounds__(128, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, float *Y, int N, int K,
              const int32_t *list, const int32_t *count, int32_t *err, int accumulate, int mtiles, int gm) {
  const int cnt = *count;
  // Grouped raster over a 1-D grid: groups of gm row tiles, and within a
  // group the row tiles vary fastest.  The CTAs resident at a time then share
  // weight tiles, and a group's gm row tiles of X stay in L2 while the group
  // walks every weight tile: X is read from DRAM once and W once per group.
  const int ntiles = (N + TBN - 1) / TBN;
  const int per_group = gm * ntiles, grp = blockIdx.x / per_group, in = blockIdx.x - grp * per_group;
  const int first = grp * gm, rows_here = min(gm, mtiles - first);
  const int m0 = (first + in % rows_here) * TBM, n0 = (in / rows_here) * TBN;
  if (m0 >= cnt) return;  // no listed row in this tile (before any allocation)
  extern __shared__ uint8_t smraw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  uint8_t *sA = base, *sB = base + TST * TA_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(sB + TST * TB_BYTES), *empty = full + TST, *done = empty + TST;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nk = (K + TBK - 1) / TBK;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tslot)), "r"(TBN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < TST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tacc = *tslot;
  // instruction descriptor: fp32 accumulator, A and B of the 16-bit type
  // (1 = bf16, 0 = fp16), both K-major, N / 8, M / 16
  const uint32_t ab = ACT == 1 ? 1u : 0u;
  const uint32_t idesc = (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(TBN >> 3) << 17) | ((uint32_t)(TBM >> 4) << 24);
  if (tid == 0) {
    bool ok = true;
    for (int s = 0; s < TST && s < nk; ++s) {
      mbar_expect_tx(&full[s], TA_BYTES + TB_BYTES);
      tma2d(sA + s * TA_BYTES, &ta, &full[s], s * TBK, m0);
      tma2d(sB + s * TB_BYTES, &tb, &full[s], s * TBK, n0);
    }
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % TST;
      if (!mbar_wait(&full[s], (kb / TST) & 1)) {
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint64_t ad = desc_sw128(su32(sA + s * TA_BYTES)), bd = desc_sw128(su32(sB + s * TB_BYTES));
#pragma unroll
      for (int j = 0; j < TBK / 16; ++j) umma(tacc, ad + 2 * j, bd + 2 * j, idesc, (kb | j) != 0);
      umma_commit(&empty[s]);
      // refill the stage the previous k-block used once its MMAs are done
      if (kb >= 1) {
        const int kp = kb - 1, sp = kp % TST;
        if (kp + TST < nk) {
          if (!mbar_wait(&empty[sp], (kp / TST) & 1)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[sp], TA_BYTES + TB_BYTES);
          tma2d(sA + sp * TA_BYTES, &ta, &full[sp], (kp + TST) * TBK, m0);
          tma2d(sB + sp * TB_BYTES, &tb, &full[sp], (kp + TST) * TBK, n0);
        }
      }
    }
    umma_commit(done);
    if (!ok) atomicOr(err, 16);
  }
  __syncwarp();
  const bool fin = mbar_wait(done, 0);
  if (!fin && lane == 0) atomicOr(err, 16);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (fin) {
    const int r = m0 + warp * 32 + lane;
    const int m = r < cnt ? (list ? list[r] : r) : -1;
    for (int c = 0; c < TBN / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tacc + ((uint32_t)(warp * 32) << 16) + c * 32, v);
      const int nb = n0 + c * 32;
      if (m >= 0) {
        float *dst = Y + (size_t)m * N + nb;
        if (nb + 32 <= N && (N & 3) == 0) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float4 o = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                                   __uint_as_float(v[i + 3]));
            if (accumulate) {
              const float4 y = *reinterpret_cast<const float4 *>(dst + i);
              o.x += y.x; o.y += y.y; o.z += y.z; o.w += y.w;
            }
            *reinterpret_cast<float4 *>(dst + i) = o;
          }
        } else {
          for (int i = 0; i < 32; ++i)
            if (nb + i < N) dst[i] = accumulate ? dst[i] + __uint_as_float(v[i]) : __uint_as_float(v[i]);
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tacc), "r"(TBN) : "memory");
}

// River matrix -> two 16-bit matrices hi + lo with hi = round16(w), lo =
// round16(w - hi), w = (q - z) * s exact in fp32.  w has at most 16
// significant bits (a 5-bit integer times an 11-bit fp16 scale), so hi + lo
// is w exactly for both 16-bit types.
__global__ void k_river_split(RiverMat r, int N, int K, int act, uint16_t *hi, uint16_t *lo) {
  const int words = r.Kp >> 3;
  const long total = (long)N * (K / 8);
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int n = (int)(i / (K / 8)), k0 = (int)(i - (long)n * (K / 8)) * 8;
    const uint32_t word = r.q[(size_t)n * words + (k0 >> 3)];
    const float2 sz = __half22float2(r.sz[(size_t)n * r.Gs + k0 / r.g]);
    uint16_t h[8], l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float w = ((float)((word >> (4 * j)) & 0xFu) - sz.y) * sz.x;
      h[j] = f_to_act(w, act);
      l[j] = f_to_act(w - act_to_f(h[j], act), act);
    }
    *reinterpret_cast<uint4 *>(hi + (size_t)n * K + k0) =
        make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
    *reinterpret_cast<uint4 *>(lo + (size_t)n * K + k0) =
        make_uint4(l[0] | (l[1] << 16), l[2] | (l[3] << 16), l[4] | (l[5] << 16), l[6] | (l[7] << 16));
  }
}

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_looked = false;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_looked) {
    g_looked = true;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaGetLastError();
  }
  return g_encode;
}

bool make_map(CUtensorMap *m, const void *p, int rows, int K, int act) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {TBK, 128};
  cuuint32_t es[2] = {1, 1};
  return encoder()(m, act == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                   const_cast<void *>(p), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

void *tensor_map_encoder() { return reinterpret_cast<void *>(encoder()); }

bool gemm_tc_available() {
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  return major >= 10 && encoder() != nullptr;
}

namespace {

cudaError_t gemm_tc_run(const void *W, int N, int K, int act, float *Y, const int32_t *list, const int32_t *count,
                        int max_rows, const uint16_t *xb, int32_t *err, int accumulate, cudaStream_t s) {
  CUtensorMap ta, tb;
  if (!make_map(&ta, xb, max_rows, K, act) || !make_map(&tb, W, N, K, act)) return cudaErrorInvalidValue;
  const long mtiles = (max_rows + TBM - 1) / TBM, ntiles = (N + TBN - 1) / TBN;
  if (mtiles * ntiles > 0x7FFFFFFFL) return cudaErrorInvalidValue;
  // row tiles per group: their X tiles (TBM x K 16-bit each) within ~32 MB
  // of L2 (the L2 is split between the two dies; on the 16K-token prefill
  // QKV GEMM, groups of 64 MB of X read 1.49 GB from DRAM, of 32 MB 0.34 GB,
  // of 16 MB 0.53 GB, for 0.18 GB of operands)
  const long tile_bytes = (long)TBM * K * 2;
  long gm = (32L << 20) / (tile_bytes > 0 ? tile_bytes : 1);
  if (gm < 1) gm = 1;
  if (gm > mtiles) gm = mtiles;
  const dim3 grid((unsigned)(mtiles * ntiles));
  cudaError_t e;
  if (act == 1) {
    e = cudaFuncSetAttribute(k_gemm_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, TSMEM);
    if (e == cudaSuccess)
      k_gemm_tc<1><<<grid, 128, TSMEM, s>>>(ta, tb, Y, N, K, list, count, err, accumulate, (int)mtiles, (int)gm);
  } else {
    e = cudaFuncSetAttribute(k_gemm_tc<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, TSMEM);
    if (e == cudaSuccess)
      k_gemm_tc<0><<<grid, 128, TSMEM, s>>>(ta, tb, Y, N, K, list, count, err, accumulate, (int)mtiles, (int)gm);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t pack_rows(const float *X, int K, int act, const int32_t *list, const int32_t *count, int max_rows,
                      uint16_t *xb, cudaStream_t s) {
  const long work = (long)max_rows * (K / 8);
  const int pg = (int)((work + 255) / 256 < 4096 ? (work + 255) / 256 : 4096);
  k_pack_rows<<<pg, 256, 0, s>>>(X, K, act, list, count, xb, max_rows);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_tc(const Mat &m, int act, const float *X, float *Y, const int32_t *list, const int32_t *count,
                           int max_rows, uint16_t *xb, int32_t *err, cudaStream_t s) {
  if (max_rows <= 0) return cudaSuccess;
  if (m.K % 8 || !xb || !encoder()) return cudaErrorInvalidValue;
  cudaError_t e = pack_rows(X, m.K, act, list, count, max_rows, xb, s);
  if (e != cudaSuccess) return e;
  return gemm_tc_run(m.w, m.N, m.K, act, Y, list, count, max_rows, xb, err, 0, s);
}

cudaError_t launch_gemm_tc_river(const Mat &m, int act, const float *X, float *Y, const int32_t *list,
                                 const int32_t *count, int max_rows, uint16_t *xb, uint16_t *whi, uint16_t *wlo,
                                 int32_t *err, cudaStream_t s) {
  if (max_rows <= 0) return cudaSuccess;
  const int N = m.N, K = m.K;
  if (K % 8 || !xb || !whi || !wlo || !encoder()) return cudaErrorInvalidValue;
  const long work = (long)N * (K / 8);
  const int sg = (int)((work + 255) / 256 < 8192 ? (work + 255) / 256 : 8192);
  k_river_split<<<sg, 256, 0, s>>>(m.r, N, K, act, whi, wlo);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = pack_rows(X, K, act, list, count, max_rows, xb, s);
  if (e != cudaSuccess) return e;
  e = gemm_tc_run(whi, N, K, act, Y, list, count, max_rows, xb, err, 0, s);
  if (e != cudaSuccess) return e;
  return gemm_tc_run(wlo, N, K, act, Y, list, count, max_rows, xb, err, 1, s);
}

}  // namespace rv
