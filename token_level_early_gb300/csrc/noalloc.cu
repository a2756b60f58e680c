// Greedy LM head (final RMSNorm + LM-head GEMV + argmax) for callers that
// cannot allocate device memory.
//
// The decode step's LM-head kernel combines per-block results in scratch
// memory (one (value, index) pair per block and a completion counter).
// rv_greedy_head_noalloc runs the same kernel with that scratch in a fixed
// array compiled into the library instead of memory from cudaMalloc, so a
// caller that must not allocate (a serving runtime that owns the whole device
// memory budget, or code that must not trigger the implicit synchronization
// of cudaMalloc / cudaFree) can still run the head.  It launches the existing
// kernel unchanged.
#include <mutex>

#include "../../include/rv.h"
#include "common.cuh"
#include "kernels.cuh"

namespace {

// Scratch: one (float, int) pair per block, then the completion counter and
// a position word the kernel advances (unused by this entry point).
constexpr int kMaxBlocks = 1024;
constexpr size_t kPartialBytes = 8 * (size_t)kMaxBlocks;
constexpr size_t kScratchBytes = kPartialBytes + 256;

static __device__ __align__(256) unsigned char g_head_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char *g_addr[kMaxDevices] = {nullptr};

int fail(int code, const char *msg) {
  rv::set_error_message(msg);  // read back with rv_last_error()
  return code;
}

}  // namespace

extern "C" int rv_greedy_head_noalloc(const void *d_lm_head, const void *d_final_norm, const float *d_h, int vocab,
                                      int d_model, int act_dtype, float rms_eps, int32_t *d_next_id, float *d_logits,
                                      void *stream) {
  rv::set_error_message("");
  if (!d_lm_head || !d_final_norm || !d_h || !d_next_id) return fail(RV_EINVAL, "null pointer");
  if (act_dtype != 0 && act_dtype != 1) return fail(RV_EINVAL, "act_dtype must be 0 (fp16) or 1 (bf16)");
  if (vocab < 4 || vocab % 4) return fail(RV_EINVAL, "vocab must be a positive multiple of 4");
  if (d_model < 8 || d_model % 8) return fail(RV_EINVAL, "d_model must be a positive multiple of 8");
  if (d_model > 16384) return fail(RV_EINVAL, "d_model above the maximum of 16384 (shared-memory staging)");
  // the GEMV keeps element offsets of the matrix in 32 bits
  if ((uint64_t)vocab * (uint64_t)d_model > 0xFFFFFFFFull)
    return fail(RV_EINVAL, "vocab x d_model above 2^32 - 1 elements");
  // the kernel reads these with 16-byte loads and copies
  if ((reinterpret_cast<uintptr_t>(d_lm_head) | reinterpret_cast<uintptr_t>(d_final_norm) |
       reinterpret_cast<uintptr_t>(d_h)) & 15u)
    return fail(RV_EINVAL, "d_lm_head, d_final_norm and d_h must be 16-byte aligned");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail(RV_ECUDA, "no usable device");
  unsigned char *base;
  {
    // First call on this device: look up the array's device address (a
    // host-side name is not a device pointer).
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
      void *p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_head_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return fail(RV_ECUDA, "cudaGetSymbolAddress failed for the head scratch");
      }
      g_addr[dev] = static_cast<unsigned char *>(p);
    }
    base = g_addr[dev];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned *counter = reinterpret_cast<unsigned *>(base + kPartialBytes);
  int32_t *pos_word = reinterpret_cast<int32_t *>(base + kPartialBytes + 16);
  // the counter must start at zero (a previous call may have been cut short)
  if (cudaMemsetAsync(counter, 0, 32, s) != cudaSuccess) {
    cudaGetLastError();
    return fail(RV_ECUDA, "cudaMemsetAsync of the head scratch failed");
  }
  rv::GemvArgs a{};
  a.m.w = static_cast<const uint16_t *>(d_lm_head);
  a.m.N = vocab;
  a.m.K = d_model;
  a.h = d_h;
  a.gamma = static_cast<const uint16_t *>(d_final_norm);
  a.eps = rms_eps;
  a.partials = reinterpret_cast<float *>(base);
  a.counter = counter;
  a.dbg_logits = d_logits;
  a.st.next_ids = d_next_id;
  a.st.len = pos_word;
  cudaError_t e = rv::launch_gemv_b1(act_dtype, rv::PRO_NORM, rv::EPI_LOGITS, a, kMaxBlocks, s, 0);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RV_ECUDA, cudaGetErrorString(e));
  }
  return RV_OK;
}
