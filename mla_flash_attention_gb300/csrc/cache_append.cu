// Append the new tokens' latent + rope rows to the paged latent cache (the step before
// absorbed decode), with per-token e4m3 quantisation for an fp8 cache.
//
// Token t of sequence b goes to position L_b - T + t (cache_lens count the new tokens, as
// decode reads them): page page_table[b, pos / 64], row pos % 64.  fp8: the 576 values of
// the row (bf16, widened exactly to fp32) get scale = amax / 448 (1 when amax = 0) and codes
// e4m3(clamp(x / scale, +-448)), round to nearest even; the scale goes to kv_scale.
// One warp per row: lane l owns the bf16 pairs at columns 2l + 64k (k = 0..8), so every
// load and store of the warp covers one contiguous segment of the row.
#include "common.cuh"

namespace mla {

constexpr int kAppendD = 576, kAppendPage = 64;
constexpr int kAppendPairs = kAppendD / 64;  // bf16 pairs per lane
constexpr int kAppendWarps = 4;

__global__ void __launch_bounds__(kAppendWarps * 32) cache_append_kernel(
    const uint32_t* __restrict__ c_new, void* __restrict__ cache, float* __restrict__ kv_scale,
    const int* __restrict__ page_table, const int* __restrict__ cache_lens, int B, int T,
    int max_pages, int num_pages, int fp8, unsigned int* err) {
  const int lane = threadIdx.x & 31;
  const int row_id = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  if (row_id >= B * T) return;
  const int b = row_id / T, t = row_id % T;
  const int pos = __ldg(cache_lens + b) - T + t;
  if (pos < 0) return;  // fewer cached tokens than new ones: nothing to write for this t
  const int pg = pos / kAppendPage, r = pos % kAppendPage;
  const int page = pg < max_pages ? __ldg(page_table + (size_t)b * max_pages + pg) : -1;
  if (page < 0 || page >= num_pages) {
    if (lane == 0) latch_error(err, kErrBadPage);
    return;
  }
  const uint32_t* src = c_new + (size_t)row_id * (kAppendD / 2);
  const size_t dst_row = (size_t)page * kAppendPage + r;
  uint32_t w[kAppendPairs];
#pragma unroll
  for (int k = 0; k < kAppendPairs; ++k) w[k] = __ldg(src + lane + 32 * k);
  if (!fp8) {
    uint32_t* dst = static_cast<uint32_t*>(cache) + dst_row * (kAppendD / 2);
#pragma unroll
    for (int k = 0; k < kAppendPairs; ++k) dst[lane + 32 * k] = w[k];
    return;
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < kAppendPairs; ++k)
    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[k] << 16)), fabsf(__uint_as_float(w[k] & 0xffff0000u))));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint16_t* dst = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(cache) + dst_row * kAppendD);
#pragma unroll
  for (int k = 0; k < kAppendPairs; ++k) {
    const float lo = fminf(fmaxf(__fdiv_rn(__uint_as_float(w[k] << 16), scale), -448.f), 448.f);
    const float hi = fminf(fmaxf(__fdiv_rn(__uint_as_float(w[k] & 0xffff0000u), scale), -448.f), 448.f);
    uint16_t codes;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(codes) : "f"(hi), "f"(lo));
    dst[lane + 32 * k] = codes;
  }
  if (lane == 0) kv_scale[dst_row] = scale;
}

cudaError_t launch_cache_append(const void* c_new, void* cache, float* kv_scale,
                                const int* page_table, const int* cache_lens, int B, int T,
                                int max_pages, int num_pages, bool fp8, unsigned int* err,
                                cudaStream_t stream) {
  const int rows = B * T;
  if (rows <= 0) return cudaSuccess;
  const int grid = (rows + kAppendWarps - 1) / kAppendWarps;
  cache_append_kernel<<<grid, kAppendWarps * 32, 0, stream>>>(
      static_cast<const uint32_t*>(c_new), cache, kv_scale, page_table, cache_lens, B, T,
      max_pages, num_pages, fp8 ? 1 : 0, err);
  return cudaGetLastError();
}

}  // namespace mla
