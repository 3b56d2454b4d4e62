// Log-sum-exp merge of the decode split partials.
//
// For sequence b, the work units c_first..c_last that covered its pages wrote
// (O_s / l_s, m_s + ln l_s) into slots c + b (see the split plan in common.cuh).  The
// merged output is O = sum_s exp(lse_s - lse) O_s with lse = ln sum_s exp(lse_s);
// 128-bit loads of the fp32 partials, bf16 output.
#include "common.cuh"

namespace mla {

constexpr int kCombDl = 512, kCombPage = 64;
constexpr int kCombRows = 8;  // query rows per CTA (64 threads per row, 8 columns each)

__device__ __forceinline__ int comb_clamp_len(int L, int max_pages) {
  return min(max(L, 0), max_pages * kCombPage);
}

__global__ void __launch_bounds__(512) decode_combine_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_lse,
    const int* __restrict__ cache_lens, uint16_t* __restrict__ out, float* __restrict__ lse,
    int B, int H, int T, int max_pages, int G) {
  const int b = blockIdx.x;
  const int TH = T * H;
  __shared__ int s_pb, s_n, s_chunk;
  if (threadIdx.x < 32) {
    // pages of sequences before b and in total, 32 lengths at a time
    int before = 0, total = 0;
    for (int base = 0; base < B; base += 32) {
      const int bb = base + threadIdx.x;
      const int n = bb < B ? pages_of(comb_clamp_len(__ldg(cache_lens + bb), max_pages), kCombPage) : 0;
      int nb = bb < b ? n : 0;
      int nt = n;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        nb += __shfl_xor_sync(0xffffffffu, nb, off);
        nt += __shfl_xor_sync(0xffffffffu, nt, off);
      }
      before += nb;
      total += nt;
    }
    if (threadIdx.x == 0) {
      s_pb = before;
      s_n = pages_of(comb_clamp_len(__ldg(cache_lens + b), max_pages), kCombPage);
      s_chunk = total > 0 ? (total + G - 1) / G : 1;
    }
  }
  __syncthreads();
  const int row = blockIdx.y * kCombRows + (threadIdx.x >> 6);
  const int lane64 = threadIdx.x & 63;
  if (row >= TH) return;
  const int t = row / H, h = row % H;
  float* o_lse = lse + ((size_t)b * H + h) * T + t;
  uint16_t* o_dst = out + ((size_t)b * TH + row) * kCombDl + lane64 * 8;
  if (s_n == 0) {
    *reinterpret_cast<uint4*>(o_dst) = make_uint4(0, 0, 0, 0);
    if (lane64 == 0) *o_lse = -INFINITY;
    return;
  }
  const int c_first = s_pb / s_chunk, c_last = (s_pb + s_n - 1) / s_chunk;
  // pass 1: the largest partial LSE (independent loads)
  float mx = -INFINITY;
  for (int c = c_first; c <= c_last; ++c) mx = fmaxf(mx, __ldg(part_lse + ((size_t)c + b) * TH + row));
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  float wsum = 0.f;
  if (mx != -INFINITY) {
    // pass 2: weights and 128-bit loads, four splits in flight
    for (int c0 = c_first; c0 <= c_last; c0 += 4) {
      float w[4];
      float4 a[4], bq[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = c0 + k;
        w[k] = 0.f;
        a[k] = bq[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c <= c_last) {
          const size_t slot = (size_t)c + b;
          const float ls = __ldg(part_lse + slot * TH + row);
          if (ls != -INFINITY) {
            w[k] = __expf(ls - mx);
            const float4* src = reinterpret_cast<const float4*>(part_o + (slot * TH + row) * kCombDl + lane64 * 8);
            a[k] = __ldg(src);
            bq[k] = __ldg(src + 1);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        wsum += w[k];
        acc[0] += w[k] * a[k].x; acc[1] += w[k] * a[k].y; acc[2] += w[k] * a[k].z; acc[3] += w[k] * a[k].w;
        acc[4] += w[k] * bq[k].x; acc[5] += w[k] * bq[k].y; acc[6] += w[k] * bq[k].z; acc[7] += w[k] * bq[k].w;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint32_t packed[4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
    packed[c] = (uint32_t)f32_to_bf16_rne(acc[2 * c] * inv) |
                ((uint32_t)f32_to_bf16_rne(acc[2 * c + 1] * inv) << 16);
  *reinterpret_cast<uint4*>(o_dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  if (lane64 == 0) *o_lse = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

cudaError_t launch_decode_combine(const float* part_o, const float* part_lse,
                                  const int* cache_lens, void* out, float* lse, int B, int H,
                                  int T, int max_pages, int G, cudaStream_t stream) {
  const int TH = T * H;
  dim3 grid(B, (TH + kCombRows - 1) / kCombRows);
  decode_combine_kernel<<<grid, 512, 0, stream>>>(part_o, part_lse, cache_lens,
                                                  static_cast<uint16_t*>(out), lse, B, H, T,
                                                  max_pages, G);
  return cudaGetLastError();
}

}  // namespace mla
