// First prefill kernel: plain CUDA-core flash attention over split nope+rope depths.
//
// One CTA per (64-query tile, head, batch); keys in tiles of 64 with an online
// softmax (running max m, running sum l, rescale of O by exp(m_old - m_new)).
// fp32 arithmetic throughout.  Layouts as in include/mla.h.
#include "common.cuh"

namespace mla {

constexpr int kSimtBM = 64;
constexpr int kSimtBN = 64;
constexpr int kDn = 128, kDr = 64, kDv = 128, kDqk = kDn + kDr;

struct PrefillSimtSmem {
  float q[kSimtBM][kDqk];
  float k[kSimtBN][kDqk + 1];
  float v[kSimtBN][kDv];
  float p[kSimtBM][kSimtBN + 1];
};

template <bool kFp8, bool kOutF32>
__global__ void __launch_bounds__(256) prefill_simt_kernel(
    const void* __restrict__ q_nope, const uint16_t* __restrict__ q_rope,
    const void* __restrict__ k_nope, const uint16_t* __restrict__ k_rope,
    const void* __restrict__ v, const float* __restrict__ q_scale,
    const float* __restrict__ k_scale, void* __restrict__ out, float* __restrict__ lse, int B,
    int H, int S, float softmax_scale, int causal) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PrefillSimtSmem& sm = *reinterpret_cast<PrefillSimtSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int i0 = blockIdx.x * kSimtBM;
  const int h = blockIdx.y;
  const int b = blockIdx.z;

  auto load_nope = [&](const void* base, size_t idx) -> float {
    if constexpr (kFp8) return e4m3_to_f32(static_cast<const uint8_t*>(base)[idx]);
    else return bf16_to_f32(static_cast<const uint16_t*>(base)[idx]);
  };

  // Q tile
  for (int e = tid; e < kSimtBM * kDqk; e += blockDim.x) {
    int r = e / kDqk, c = e % kDqk, i = i0 + r;
    float x = 0.f;
    if (i < S) {
      size_t tok = (size_t)b * S + i;
      if (c < kDn) {
        x = load_nope(q_nope, (tok * H + h) * kDn + c);
        if constexpr (kFp8) x *= q_scale[tok];
      } else {
        x = bf16_to_f32(q_rope[(tok * H + h) * kDr + (c - kDn)]);
      }
    }
    sm.q[r][c] = x;
  }

  const int r = tid >> 2;          // query row owned by this thread (4 threads per row)
  const int sub = tid & 3;         // quarter of the key tile / of d_v
  const int i = i0 + r;
  float m = -INFINITY, l = 0.f;
  float o[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) o[c] = 0.f;

  const int kv_end = causal ? min(S, i0 + kSimtBM) : S;
  for (int j0 = 0; j0 < kv_end; j0 += kSimtBN) {
    __syncthreads();
    for (int e = tid; e < kSimtBN * kDqk; e += blockDim.x) {
      int rr = e / kDqk, c = e % kDqk, j = j0 + rr;
      float x = 0.f;
      if (j < S) {
        size_t tok = (size_t)b * S + j;
        if (c < kDn) {
          x = load_nope(k_nope, (tok * H + h) * kDn + c);
          if constexpr (kFp8) x *= k_scale[tok];
        } else {
          x = bf16_to_f32(k_rope[tok * kDr + (c - kDn)]);
        }
      }
      sm.k[rr][c] = x;
    }
    for (int e = tid; e < kSimtBN * kDv; e += blockDim.x) {
      int rr = e / kDv, c = e % kDv, j = j0 + rr;
      float x = 0.f;
      if (j < S) {
        size_t tok = (size_t)b * S + j;
        x = load_nope(v, (tok * H + h) * kDv + c);
        if constexpr (kFp8) x *= k_scale[tok];
      }
      sm.v[rr][c] = x;
    }
    __syncthreads();

    float tmax = -INFINITY;
#pragma unroll 1
    for (int jj = 0; jj < 16; ++jj) {
      const int kk = sub * 16 + jj, j = j0 + kk;
      float acc = 0.f;
#pragma unroll 8
      for (int c = 0; c < kDqk; ++c) acc = fmaf(sm.q[r][c], sm.k[kk][c], acc);
      bool vis = (j < S) && (!causal || j <= i);
      const float sv = vis ? acc * softmax_scale : -INFINITY;
      sm.p[r][kk] = sv;
      tmax = fmaxf(tmax, sv);
    }
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const float m_new = fmaxf(m, tmax);
    const float alpha = (m_new == -INFINITY) ? 1.f : expf(m - m_new);
    float psum = 0.f;
#pragma unroll 1
    for (int jj = 0; jj < 16; ++jj) {
      const float sv = sm.p[r][sub * 16 + jj];
      const float p = (sv == -INFINITY) ? 0.f : expf(sv - m_new);
      psum += p;
      sm.p[r][sub * 16 + jj] = p;
    }
    psum += __shfl_xor_sync(0xffffffffu, psum, 1);
    psum += __shfl_xor_sync(0xffffffffu, psum, 2);
    l = l * alpha + psum;
    m = m_new;
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 32; ++c) o[c] *= alpha;
#pragma unroll 1
    for (int kk = 0; kk < kSimtBN; ++kk) {
      const float p = sm.p[r][kk];
#pragma unroll
      for (int c = 0; c < 32; ++c) o[c] = fmaf(p, sm.v[kk][sub * 32 + c], o[c]);
    }
  }

  if (i < S) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    size_t obase = (((size_t)b * S + i) * H + h) * kDv + sub * 32;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      float x = o[c] * inv;
      if constexpr (kOutF32) static_cast<float*>(out)[obase + c] = x;
      else static_cast<uint16_t*>(out)[obase + c] = f32_to_bf16_rne(x);
    }
    if (sub == 0) lse[((size_t)b * H + h) * S + i] = l > 0.f ? m + logf(l) : -INFINITY;
  }
}

cudaError_t launch_prefill_simt(const void* q_nope, const void* q_rope, const void* k_nope,
                                const void* k_rope, const void* v, const float* q_scale,
                                const float* k_scale, void* out, float* lse, int B, int H,
                                int S, float softmax_scale, int causal, bool fp8, bool out_f32,
                                cudaStream_t stream) {
  dim3 grid((S + kSimtBM - 1) / kSimtBM, H, B);
  size_t smem = sizeof(PrefillSimtSmem);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 256, smem, stream>>>(q_nope, (const uint16_t*)q_rope, k_nope,
                                      (const uint16_t*)k_rope, v, q_scale, k_scale, out, lse,
                                      B, H, S, softmax_scale, causal);
    return cudaGetLastError();
  };
  if (fp8) return out_f32 ? go(prefill_simt_kernel<true, true>) : go(prefill_simt_kernel<true, false>);
  return out_f32 ? go(prefill_simt_kernel<false, true>) : go(prefill_simt_kernel<false, false>);
}

}  // namespace mla
