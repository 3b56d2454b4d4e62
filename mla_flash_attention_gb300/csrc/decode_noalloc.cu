// mla_decode_noalloc: the decode entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point where they
// run decode -- for example an inference engine that hands out all device memory itself at
// start-up and forbids allocation afterwards, or a plugin whose execute hook may not
// allocate -- and so cannot supply mla_decode's workspace.  This entry point uses a fixed
// scratch array compiled into the library instead: a file-scope __device__ array of
// kNoAllocScratchBytes (48 MiB).  The caller still passes every input and output buffer.
//
// When the array exists on a device: this file is its own module, and under CUDA's lazy
// module loading (the default) the driver loads that module -- allocating the 48 MiB on the
// device -- the first time the array's address is looked up there, not when the library is
// loaded.  It then stays allocated until the process exits.  A call with B = 0 does only
// this set-up on the current device: it looks up the array's address (cudaGetSymbolAddress,
// with that device current), loads the decode kernels and the device error word, and
// returns without launching anything.  A caller that reserves device memory at start-up
// makes that call first, before its reservation and before any stream capture; later calls
// on the device then allocate nothing.  Without it, the first ordinary call does the same
// set-up (and may then fail if the device has no free memory left).
//
// In host code the array's name is only a host-side stand-in, so nothing here ever passes
// the name itself to a kernel: kernels get the address looked up above.
//
// Sharing: every call on a device uses the same array and it keeps the previous call's
// contents.  The split partials are always written before they are read in the same call;
// the merge counters (also in the array) must start each call at zero, which the decode
// launch guarantees by zeroing them with a kernel queued ahead of the split kernel on every
// call -- this entry point relies on that.  Calls that overlap on the GPU (different
// streams, or different host threads without ordering) race on the array and must be
// serialised by the caller.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/mla.h"

namespace mla {
mla_status set_last_error(mla_status st, const char* fmt, ...);
unsigned int* error_word_address();
cudaError_t load_decode_kernels();
}  // namespace mla

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;

__device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device, or nullptr.  Cache entries are
// atomics: host threads may make their first calls on a device at the same time (both then
// look up and store the same address).
void* scratch_address(cudaError_t* err) {
  static std::atomic<void*> cache[64];
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  void* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    *err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (*err != cudaSuccess) return nullptr;
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace

extern "C" {

size_t mla_decode_noalloc_max_workspace(void) { return kNoAllocScratchBytes; }

mla_status mla_decode_noalloc(const void* q_latent, const void* q_rope, const void* kv_cache,
                              const float* kv_scale, const int* page_table, const int* cache_lens,
                              void* out, float* lse, int B, int H, int q_len, int d_latent,
                              int d_rope, int page_size, int max_pages_per_seq, int num_pages,
                              float softmax_scale, int causal, mla_dtype kv_dtype, void* stream) {
  if (B > 0) {
    const size_t need = mla_decode_workspace_size(B, H, q_len, d_latent);
    if (need > kNoAllocScratchBytes)
      return mla::set_last_error(MLA_ERR_WORKSPACE,
                                 "mla_decode_noalloc: this batch needs %zu bytes of scratch but the "
                                 "built-in array holds %zu; split the batch or use mla_decode",
                                 need, kNoAllocScratchBytes);
  }
  cudaError_t e = cudaSuccess;
  void* scratch = scratch_address(&e);
  if (!scratch)
    return mla::set_last_error(MLA_ERR_CUDA, "mla_decode_noalloc: scratch address lookup failed: %s",
                               cudaGetErrorString(e));
  if (B == 0) {
    // set-up only: the kernels' modules and the error word, so later calls load nothing
    if ((e = mla::load_decode_kernels()) != cudaSuccess)
      return mla::set_last_error(MLA_ERR_CUDA, "mla_decode_noalloc: loading the decode kernels failed: %s",
                                 cudaGetErrorString(e));
    if (!mla::error_word_address())
      return mla::set_last_error(MLA_ERR_CUDA, "mla_decode_noalloc: device error word not reachable");
    return MLA_OK;
  }
  return mla_decode(q_latent, q_rope, kv_cache, kv_scale, page_table, cache_lens, out, lse, B, H,
                    q_len, d_latent, d_rope, page_size, max_pages_per_seq, num_pages,
                    softmax_scale, causal, kv_dtype, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
