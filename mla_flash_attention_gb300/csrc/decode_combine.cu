// Log-sum-exp merge of the decode split partials.
//
// For sequence b, the work units c_first..c_last that covered its pages wrote
// (O_s / l_s, m_s + ln l_s) into slots c + b (see the split plan in common.cuh).  The
// merged output is O = sum_s exp(lse_s - lse) O_s with lse = ln sum_s exp(lse_s);
// 128-bit loads of the fp32 partials, bf16 output.
#include "common.cuh"

namespace mla {

constexpr int kCombDl = 512, kCombPage = 64;

__device__ __forceinline__ int comb_clamp_len(int L, int max_pages) {
  return min(max(L, 0), max_pages * kCombPage);
}

// Combine: one CTA per (sequence, group of 8 rows); 64 threads per row, 8 columns each.
__global__ void __launch_bounds__(512) decode_combine_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_lse,
    const int* __restrict__ cache_lens, uint16_t* __restrict__ out, float* __restrict__ lse,
    int B, int H, int T, int max_pages, int G) {
  const int b = blockIdx.x;
  const int TH = T * H;
  const int row = blockIdx.y * 8 + (threadIdx.x >> 6);
  const int lane64 = threadIdx.x & 63;
  __shared__ int s_pb, s_n, s_chunk;
  if (threadIdx.x == 0) {
    int total = 0, pb = 0;
    for (int bb = 0; bb < B; ++bb) {
      int n = pages_of(comb_clamp_len(__ldg(cache_lens + bb), max_pages), kCombPage);
      if (bb == b) pb = total;
      total += n;
    }
    s_pb = pb;
    s_n = pages_of(comb_clamp_len(__ldg(cache_lens + b), max_pages), kCombPage);
    s_chunk = total > 0 ? (total + G - 1) / G : 1;
  }
  __syncthreads();
  if (row >= TH) return;
  const int t = row / H, h = row % H;
  float* o_dst_lse = lse + ((size_t)b * H + h) * T + t;
  uint16_t* o_dst = out + ((size_t)b * TH + row) * kCombDl + lane64 * 8;
  if (s_n == 0) {
    for (int c = 0; c < 8; ++c) o_dst[c] = 0;
    if (lane64 == 0) *o_dst_lse = -INFINITY;
    return;
  }
  const int c_first = s_pb / s_chunk, c_last = (s_pb + s_n - 1) / s_chunk;
  float mx = -INFINITY;
  for (int c = c_first; c <= c_last; ++c) mx = fmaxf(mx, part_lse[((size_t)c + b) * TH + row]);
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int c = c_first; c <= c_last; ++c) {
      const size_t slot = (size_t)c + b;
      const float ls = part_lse[slot * TH + row];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - mx);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(part_o + (slot * TH + row) * kCombDl + lane64 * 8);
      float4 a = src[0], bq = src[1];
      acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
      acc[4] += w * bq.x; acc[5] += w * bq.y; acc[6] += w * bq.z; acc[7] += w * bq.w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint32_t packed[4];
  for (int c = 0; c < 4; ++c)
    packed[c] = (uint32_t)f32_to_bf16_rne(acc[2 * c] * inv) |
                ((uint32_t)f32_to_bf16_rne(acc[2 * c + 1] * inv) << 16);
  *reinterpret_cast<uint4*>(o_dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  if (lane64 == 0) *o_dst_lse = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

cudaError_t launch_decode_combine(const float* part_o, const float* part_lse,
                                  const int* cache_lens, void* out, float* lse, int B, int H,
                                  int T, int max_pages, int G, cudaStream_t stream) {
  const int TH = T * H;
  dim3 grid(B, (TH + 7) / 8);
  decode_combine_kernel<<<grid, 512, 0, stream>>>(part_o, part_lse, cache_lens,
                                                  static_cast<uint16_t*>(out), lse, B, H, T,
                                                  max_pages, G);
  return cudaGetLastError();
}

}  // namespace mla
