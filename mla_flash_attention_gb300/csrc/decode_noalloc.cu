// mla_decode_noalloc: the decode entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point where they
// run decode -- for example an inference engine that hands out all device memory itself at
// start-up and forbids allocation afterwards, or a plugin whose execute hook may not
// allocate -- and so cannot supply mla_decode's workspace.  This entry point uses a fixed
// scratch array compiled into the library instead: a file-scope __device__ array of
// kNoAllocScratchBytes (48 MiB) that every GPU which loads the library holds until the
// process exits.  The caller still passes every input and output buffer.
//
// Set-up: the first call on a device looks up the array's device address with
// cudaGetSymbolAddress (with that device current) and caches it; that first call should
// come before any stream capture.  In host code the array's name is only a host-side
// stand-in, so nothing here ever passes the name itself to a kernel.
//
// Sharing: every call on a device uses the same array and it keeps the previous call's
// contents.  Decode never reads a scratch entry it has not written in the same call, so
// nothing has to be cleared, but calls that overlap on the GPU (different streams, or
// different host threads without ordering) race on the array and must be serialised by
// the caller.
#include <cuda_runtime.h>

#include "../../include/mla.h"

namespace mla {
mla_status set_last_error(mla_status st, const char* fmt, ...);
}  // namespace mla

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;

__device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device, or nullptr.
void* scratch_address(cudaError_t* err) {
  static void* cache[64] = {nullptr};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  if (!cache[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (*err != cudaSuccess) return nullptr;
    cache[dev] = p;
  }
  return cache[dev];
}

}  // namespace

extern "C" {

size_t mla_decode_noalloc_max_workspace(void) { return kNoAllocScratchBytes; }

mla_status mla_decode_noalloc(const void* q_latent, const void* q_rope, const void* kv_cache,
                              const float* kv_scale, const int* page_table, const int* cache_lens,
                              void* out, float* lse, int B, int H, int q_len, int d_latent,
                              int d_rope, int page_size, int max_pages_per_seq, int num_pages,
                              float softmax_scale, int causal, mla_dtype kv_dtype, void* stream) {
  const size_t need = mla_decode_workspace_size(B, H, q_len, d_latent);
  if (need > kNoAllocScratchBytes)
    return mla::set_last_error(MLA_ERR_WORKSPACE,
                               "mla_decode_noalloc: this batch needs %zu bytes of scratch but the "
                               "built-in array holds %zu; split the batch or use mla_decode",
                               need, kNoAllocScratchBytes);
  cudaError_t e = cudaSuccess;
  void* scratch = scratch_address(&e);
  if (!scratch)
    return mla::set_last_error(MLA_ERR_CUDA, "mla_decode_noalloc: scratch address lookup failed: %s",
                               cudaGetErrorString(e));
  return mla_decode(q_latent, q_rope, kv_cache, kv_scale, page_table, cache_lens, out, lse, B, H,
                    q_len, d_latent, d_rope, page_size, max_pages_per_seq, num_pages,
                    softmax_scale, causal, kv_dtype, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
