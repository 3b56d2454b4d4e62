// Shared device helpers of the GB300 MLA library (CUDA path only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

// Device error word bits (latched with atomicOr, read and cleared by the host).
enum : unsigned int {
  kErrTimeout = 1u,     // a bounded mbarrier / flag wait ran out
  kErrBadPage = 2u,     // a page-table entry outside [0, num_pages)
  kErrBounds = 4u,      // a store fell outside its buffer (bounds-checked build only)
};

__device__ __forceinline__ void latch_error(unsigned int* err, unsigned int bits) {
  if (err) atomicOr(err, bits);
}

// Store bounds checks of the bounds-checked build (compiled with -DMLA_DEBUG): every store of
// an output, LSE or workspace element goes through MLA_STORE_OK(ptr, base, bytes, err), true
// when the element at ptr lies inside [base, base + bytes); otherwise the check latches
// kErrBounds and the caller skips the store, so an indexing mistake shows up as an error
// status rather than as a write outside the buffer.  In the normal build it is `true`.
#ifdef MLA_DEBUG
__device__ __forceinline__ bool store_ok(const void* ptr, size_t n, const void* base, size_t bytes,
                                         unsigned int* err) {
  const char* c = static_cast<const char*>(ptr);
  const char* b = static_cast<const char*>(base);
  const bool ok = c >= b && c + n <= b + bytes;
  if (!ok) latch_error(err, kErrBounds);
  return ok;
}
#define MLA_STORE_OK(ptr, base, bytes, err) ::mla::store_ok((ptr), sizeof(*(ptr)), (base), (bytes), (err))
#else
#define MLA_STORE_OK(ptr, base, bytes, err) true
#endif

// Bytes by which launches under-report the output buffer's size to the store checks (a test
// hook: with a positive value the bounds-checked build must catch the last rows' stores).
size_t testing_out_shrink();

// Number of cache pages of a sequence of length L.
__device__ __forceinline__ int pages_of(int L, int page_size) {
  return L > 0 ? (L + page_size - 1) / page_size : 0;
}

// Split plan of the decode key axis (computed from cache_lens alone, identically by every
// CTA of the split kernel): the pages of all (sequence, query tile) work items are numbered
// in order (item v owns flat pages [P_v, P_v + n_v)), and work unit c of G takes flat pages
// [c*chunk, (c+1)*chunk) with chunk = ceil(total / G).  The partial result of unit c for
// item v goes to slot c + v, which is unique because consecutive units never move backwards
// through the items; there are at most G + (number of items) - 1 slots.

// Opt `kernel` into `bytes` of dynamic shared memory on the current device.  The attribute
// belongs to the device, so it is set once per device ordinal: `done` holds one bit per
// ordinal below 64 (higher ordinals set it on every call).
template <typename Kernel>
inline cudaError_t smem_attr_once(Kernel kernel, int bytes, unsigned long long* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (__atomic_load_n(done, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) __atomic_fetch_or(done, bit, __ATOMIC_ACQ_REL);
  return e;
}

}  // namespace mla
