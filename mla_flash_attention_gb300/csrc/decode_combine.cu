// Log-sum-exp merge of the decode split partials.
//
// For sequence b, the work units c_first..c_last that covered its pages wrote
// (O_s / l_s, m_s + ln l_s) into slots c + b (see the split plan in common.cuh).  The
// merged output is O = sum_s exp(lse_s - lse) O_s with lse = ln sum_s exp(lse_s);
// 128-bit loads of the fp32 partials, bf16 output.
#include "common.cuh"

namespace mla {

constexpr int kCombDl = 512, kCombPage = 64;
constexpr int kCombRows = 32;    // query rows per CTA: one per lane
constexpr int kCombWarps = 8;    // each warp merges every 8th column quad of those rows
constexpr int kCombMaxSplits = 80;   // split weights of one sequence kept in shared memory

__device__ __forceinline__ int comb_clamp_len(int L, int max_pages) {
  return min(max(L, 0), max_pages * kCombPage);
}

// Partials are laid out [slot][column quad q (128)][row (T*H)][4 floats]; lane = row, so
// every load of a warp is 512 contiguous bytes.  The bf16 rows are assembled in shared
// memory and written out row by row.
__global__ void __launch_bounds__(kCombWarps * 32) decode_combine_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_lse,
    const int* __restrict__ cache_lens, uint16_t* __restrict__ out, float* __restrict__ lse,
    int B, int H, int T, int max_pages, int G) {
  const int b = blockIdx.x;
  const int TH = T * H;
  const int row0 = blockIdx.y * kCombRows;
  const int nrows = min(kCombRows, TH - row0);
  __shared__ int s_pb, s_n, s_chunk;
  __shared__ float s_w[kCombMaxSplits][kCombRows];  // exp(lse_s - max) / sum
  __shared__ float s_mx[kCombRows], s_inv[kCombRows];
  __shared__ __align__(16) uint16_t s_out[kCombRows][kCombDl];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    // pages of sequences before b and in total, 32 lengths at a time
    int before = 0, total = 0;
    for (int base = 0; base < B; base += 32) {
      const int bb = base + lane;
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
    if (lane == 0) {
      s_pb = before;
      s_n = pages_of(comb_clamp_len(__ldg(cache_lens + b), max_pages), kCombPage);
      s_chunk = total > 0 ? (total + G - 1) / G : 1;
    }
  }
  __syncthreads();
  const int n = s_n;
  const int c_first = n > 0 ? s_pb / s_chunk : 0, c_last = n > 0 ? (s_pb + n - 1) / s_chunk : -1;
  const int nsplit = c_last - c_first + 1;
  const int row = row0 + lane;
  const bool live = lane < nrows;
  // weights of the splits, per row: w_s = exp(lse_s - max) / sum
  float mx = -INFINITY, wsum = 0.f;
  if (warp == 0 && live) {
    for (int c = c_first; c <= c_last; ++c) mx = fmaxf(mx, __ldg(part_lse + ((size_t)c + b) * TH + row));
    for (int c = c_first; c <= c_last; ++c) {
      const float ls = __ldg(part_lse + ((size_t)c + b) * TH + row);
      const float w = (mx == -INFINITY || ls == -INFINITY) ? 0.f : __expf(ls - mx);
      wsum += w;
      if (c - c_first < kCombMaxSplits) s_w[c - c_first][lane] = w;
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    for (int k = 0; k < min(nsplit, kCombMaxSplits); ++k) s_w[k][lane] *= inv;
    s_mx[lane] = mx;
    s_inv[lane] = inv;
    lse[((size_t)b * H + row % H) * T + row / H] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
  }
  __syncthreads();
  // weight of split k of this lane's row (beyond the shared-memory table: from its LSE)
  auto weight = [&](int k) -> float {
    if (k < kCombMaxSplits) return s_w[k][lane];
    const float ls = __ldg(part_lse + ((size_t)(c_first + k) + b) * TH + row);
    return (s_mx[lane] == -INFINITY || ls == -INFINITY) ? 0.f : __expf(ls - s_mx[lane]) * s_inv[lane];
  };
  for (int q = warp; q < kCombDl / 4; q += kCombWarps) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
      const float4* src = reinterpret_cast<const float4*>(part_o) + ((size_t)(c_first + b) * 128 + q) * TH + row;
      const size_t slot_stride = (size_t)128 * TH;
      int k = 0;
      for (; k + 4 <= nsplit; k += 4) {  // four splits in flight
        float4 a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) a[u] = __ldg(src + (size_t)(k + u) * slot_stride);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float w = weight(k + u);
          if (w != 0.f) {
            acc.x += w * a[u].x; acc.y += w * a[u].y; acc.z += w * a[u].z; acc.w += w * a[u].w;
          }
        }
      }
      for (; k < nsplit; ++k) {
        const float4 a = __ldg(src + (size_t)k * slot_stride);
        const float w = weight(k);
        if (w != 0.f) {
          acc.x += w * a.x; acc.y += w * a.y; acc.z += w * a.z; acc.w += w * a.w;
        }
      }
    }
    const uint32_t lo = (uint32_t)f32_to_bf16_rne(acc.x) | ((uint32_t)f32_to_bf16_rne(acc.y) << 16);
    const uint32_t hi = (uint32_t)f32_to_bf16_rne(acc.z) | ((uint32_t)f32_to_bf16_rne(acc.w) << 16);
    *reinterpret_cast<uint2*>(&s_out[lane][q * 4]) = make_uint2(lo, hi);
  }
  __syncthreads();
  // rows out: 64 x 16 bytes each
  for (int i = threadIdx.x; i < nrows * (kCombDl / 8); i += kCombWarps * 32) {
    const int rr = i / (kCombDl / 8), cc = i % (kCombDl / 8);
    reinterpret_cast<uint4*>(out + ((size_t)b * TH + row0 + rr) * kCombDl)[cc] =
        reinterpret_cast<const uint4*>(&s_out[rr][0])[cc];
  }
}

cudaError_t launch_decode_combine(const float* part_o, const float* part_lse,
                                  const int* cache_lens, void* out, float* lse, int B, int H,
                                  int T, int max_pages, int G, cudaStream_t stream) {
  const int TH = T * H;
  dim3 grid(B, (TH + kCombRows - 1) / kCombRows);
  decode_combine_kernel<<<grid, kCombWarps * 32, 0, stream>>>(part_o, part_lse, cache_lens,
                                                  static_cast<uint16_t*>(out), lse, B, H, T,
                                                  max_pages, G);
  return cudaGetLastError();
}

}  // namespace mla
