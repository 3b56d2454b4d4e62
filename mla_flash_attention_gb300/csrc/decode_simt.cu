// First decode path: plain CUDA-core split-KV attention over the paged latent cache,
// followed by the log-sum-exp combine of the per-split partial results.
//
// Split plan (identical in both kernels, see SplitPlan in common.cuh): work CTA c
// handles flat pages [c*chunk, (c+1)*chunk) of the concatenated page lists; its
// partial result for sequence b is (O_s / l_s, m_s + ln l_s) in workspace slot c + b.
#include "common.cuh"

namespace mla {

constexpr int kDl = 512, kDrr = 64, kDc = kDl + kDrr, kPage = 64;
constexpr int kRowsPerCta = 16;

struct DecodeSimtSmem {
  float q[kRowsPerCta][kDc];
  float c[kPage][kDc + 1];
  float p[kRowsPerCta][kPage + 1];
  int first_b;
  int first_pb;
};

// Sequence length as the kernels use it: negative lengths count as 0, lengths past the
// page table are clamped (and latched as a bounds error by the split kernel).
__device__ __forceinline__ int clamp_len(int L, int max_pages, int page_size) {
  return min(max(L, 0), max_pages * page_size);
}

template <bool kFp8>
__global__ void __launch_bounds__(256) decode_split_simt_kernel(
    const uint16_t* __restrict__ q_latent, const uint16_t* __restrict__ q_rope,
    const void* __restrict__ kv_cache, const float* __restrict__ kv_scale,
    const int* __restrict__ page_table, const int* __restrict__ cache_lens,
    float* __restrict__ part_o, float* __restrict__ part_lse, int B, int H, int T,
    int max_pages, int num_pages, float softmax_scale, int causal, unsigned int* err) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  DecodeSimtSmem& sm = *reinterpret_cast<DecodeSimtSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int G = gridDim.x;
  const int cta = blockIdx.x;
  const int TH = T * H;
  const int row0 = blockIdx.y * kRowsPerCta;

  // split plan
  int total = 0;
  for (int b = 0; b < B; ++b) total += pages_of(clamp_len(__ldg(cache_lens + b), max_pages, kPage), kPage);
  const int chunk = total > 0 ? (total + G - 1) / G : 1;
  const int start = cta * chunk, end = min(total, start + chunk);
  if (start >= end) return;
  if (tid == 0) {
    int acc = 0, b = 0;
    for (; b < B; ++b) {
      int L = __ldg(cache_lens + b);
      if (L > max_pages * kPage) latch_error(err, kErrBadPage);
      int n = pages_of(clamp_len(L, max_pages, kPage), kPage);
      if (acc + n > start) break;
      acc += n;
    }
    sm.first_b = b;
    sm.first_pb = acc;
  }
  __syncthreads();

  const int r = tid >> 4;   // row within the CTA's 16 rows
  const int sub = tid & 15; // 16 threads per row
  const int row = row0 + r; // flattened (t, h)
  const int t_row = row / H;

  int b = sm.first_b, pb = sm.first_pb;
  while (b < B && pb < end) {
    const int L = clamp_len(__ldg(cache_lens + b), max_pages, kPage);
    const int n = pages_of(L, kPage);
    const int p_lo = max(start, pb) - pb, p_hi = min(end, pb + n) - pb;
    if (p_lo < p_hi) {
      __syncthreads();
      for (int e = tid; e < kRowsPerCta * kDc; e += blockDim.x) {
        int rr = e / kDc, c = e % kDc, rw = row0 + rr;
        float x = 0.f;
        if (rw < TH) {
          size_t base = (size_t)b * TH + rw;  // [B, T, H] flattened
          x = c < kDl ? bf16_to_f32(q_latent[base * kDl + c])
                      : bf16_to_f32(q_rope[base * kDrr + (c - kDl)]);
        }
        sm.q[rr][c] = x;
      }
      float m = -INFINITY, l = 0.f, o[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) o[c] = 0.f;
      const int last_visible = causal ? (L - T + t_row) : (L - 1);

      for (int p = p_lo; p < p_hi; ++p) {
        int page = __ldg(page_table + (size_t)b * max_pages + p);
        const bool bad = page < 0 || page >= num_pages;
        if (bad && tid == 0) latch_error(err, kErrBadPage);
        __syncthreads();
        for (int e = tid; e < kPage * kDc; e += blockDim.x) {
          int kk = e / kDc, c = e % kDc, j = p * kPage + kk;
          float x = 0.f;
          if (!bad && j < L) {
            size_t idx = ((size_t)page * kPage + kk) * kDc + c;
            if constexpr (kFp8)
              x = e4m3_to_f32(static_cast<const uint8_t*>(kv_cache)[idx]) *
                  kv_scale[(size_t)page * kPage + kk];
            else
              x = bf16_to_f32(static_cast<const uint16_t*>(kv_cache)[idx]);
          }
          sm.c[kk][c] = x;
        }
        __syncthreads();
        float s[4], tmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int kk = sub * 4 + jj, j = p * kPage + kk;
          float acc = 0.f;
#pragma unroll 8
          for (int c = 0; c < kDc; ++c) acc = fmaf(sm.q[r][c], sm.c[kk][c], acc);
          const bool vis = !bad && row < TH && j < L && j <= last_visible;
          s[jj] = vis ? acc * softmax_scale : -INFINITY;
          tmax = fmaxf(tmax, s[jj]);
        }
#pragma unroll
        for (int off = 1; off < 16; off <<= 1)
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        const float m_new = fmaxf(m, tmax);
        const float alpha = (m_new == -INFINITY) ? 1.f : expf(m - m_new);
        float psum = 0.f;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float pv = (s[jj] == -INFINITY) ? 0.f : expf(s[jj] - m_new);
          psum += pv;
          sm.p[r][sub * 4 + jj] = pv;
        }
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l = l * alpha + psum;
        m = m_new;
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] *= alpha;
#pragma unroll 1
        for (int kk = 0; kk < kPage; ++kk) {
          const float pv = sm.p[r][kk];
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = fmaf(pv, sm.c[kk][sub * 32 + c], o[c]);
        }
      }
      if (row < TH) {
        const size_t slot = (size_t)cta + b;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float* dst = part_o + (slot * TH + row) * kDl + sub * 32;
#pragma unroll
        for (int c = 0; c < 32; c += 4)
          *reinterpret_cast<float4*>(dst + c) =
              make_float4(o[c] * inv, o[c + 1] * inv, o[c + 2] * inv, o[c + 3] * inv);
        if (sub == 0) part_lse[slot * TH + row] = l > 0.f ? m + logf(l) : -INFINITY;
      }
    }
    pb += n;
    ++b;
  }
}

cudaError_t launch_decode_simt(const void* q_latent, const void* q_rope, const void* kv_cache,
                               const float* kv_scale, const int* page_table,
                               const int* cache_lens, void* out, float* lse, int B, int H,
                               int T, int max_pages, int num_pages, float softmax_scale,
                               int causal, bool fp8, float* part_o, float* part_lse, int G,
                               unsigned int* err, cudaStream_t stream) {
  const int TH = T * H;
  dim3 grid(G, (TH + kRowsPerCta - 1) / kRowsPerCta);
  size_t smem = sizeof(DecodeSimtSmem);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 256, smem, stream>>>((const uint16_t*)q_latent, (const uint16_t*)q_rope,
                                      kv_cache, kv_scale, page_table, cache_lens, part_o,
                                      part_lse, B, H, T, max_pages, num_pages, softmax_scale,
                                      causal, err);
    return cudaGetLastError();
  };
  cudaError_t e = fp8 ? go(decode_split_simt_kernel<true>) : go(decode_split_simt_kernel<false>);
  return e;
}

}  // namespace mla
