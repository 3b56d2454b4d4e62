// Host helper: TMA tensor-map encoding through the driver entry point (no libcuda link).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}
}  // namespace

// Tiled tensor map: `dims` innermost first, `strides` in bytes for dims 1..rank-1, box of
// `box` elements per dim, the given swizzle, zero fill outside the tensor.
cudaError_t encode_tensor_map_swizzle(CUtensorMap* map, CUtensorMapDataType dt, int rank,
                                      const void* ptr, const uint64_t* dims,
                                      const uint64_t* strides, const uint32_t* box,
                                      CUtensorMapSwizzle swizzle) {
  auto fn = encoder();
  if (!fn) return cudaErrorNotSupported;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, dt, rank, const_cast<void*>(ptr), reinterpret_cast<const cuuint64_t*>(dims),
                  reinterpret_cast<const cuuint64_t*>(strides),
                  reinterpret_cast<const cuuint32_t*>(box), es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The same with a 128-byte swizzle (or none).
cudaError_t encode_tensor_map_swz(CUtensorMap* map, CUtensorMapDataType dt, int rank,
                                  const void* ptr, const uint64_t* dims, const uint64_t* strides,
                                  const uint32_t* box, bool swizzle128) {
  return encode_tensor_map_swizzle(map, dt, rank, ptr, dims, strides, box,
                                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* ptr,
                              const uint64_t* dims, const uint64_t* strides, const uint32_t* box) {
  return encode_tensor_map_swz(map, dt, rank, ptr, dims, strides, box, true);
}

}  // namespace mla
