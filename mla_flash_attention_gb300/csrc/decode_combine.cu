// Log-sum-exp merge of the decode split partials.
//
// For sequence b, the work units c_first..c_last that covered its pages wrote
// (O_s / l_s, m_s + ln l_s) into slots c + b (see the split plan in common.cuh).  The
// merged output is O = sum_s exp(lse_s - lse) O_s with lse = ln sum_s exp(lse_s);
// 128-bit loads of the fp32 partials, bf16 output.
#include "common.cuh"

namespace mla {

constexpr int kCombDl = 512, kCombPage = 64;
constexpr int kCombRows = 32;        // query rows per CTA: one per lane
constexpr int kCombWarps = 8;
constexpr int kCombParts = 4;        // CTAs per row group, each merging 128 of the 512 columns
constexpr int kCombQuads = kCombDl / 4 / kCombParts;  // 32 column quads per CTA, 4 per warp

__device__ __forceinline__ int comb_clamp_len(int L, int max_pages) {
  return min(max(L, 0), max_pages * kCombPage);
}

// Partials are laid out [slot][column quad q (128)][row (T*H)][4 floats]; lane = row, so
// every load of a warp is 512 contiguous bytes.  CTA (b, row group, part) merges quads
// [32 part, 32 part + 32) of 32 rows; each warp keeps 4 quads x 2 splits of loads in
// flight, and each thread weighs the splits of its own row from their LSEs.  The bf16
// rows are assembled in shared memory and written out row by row.
__global__ void __launch_bounds__(kCombWarps * 32) decode_combine_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_lse,
    const int* __restrict__ cache_lens, uint16_t* __restrict__ out, float* __restrict__ lse,
    int B, int H, int T, int max_pages, int G) {
  const int b = blockIdx.x;
  const int TH = T * H;
  const int row0 = blockIdx.y * kCombRows;
  const int nrows = min(kCombRows, TH - row0);
  // the rows are planned in query tiles of 128 (TQ = min(TH, 128) rows each): this CTA's 32
  // rows lie in tile qt, whose work item is the virtual sequence b * NQT + qt
  const int NQT = (TH + 127) / 128, TQ = TH < 128 ? TH : 128;
  const int qt = row0 / 128, r0 = row0 % 128, v = b * NQT + qt;
  const int q_base = blockIdx.z * kCombQuads;
  __shared__ int s_pb, s_n, s_chunk;
  __shared__ __align__(16) uint16_t s_out[kCombRows][kCombQuads * 4];
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
    if (lane == 0) {  // every sequence is planned NQT times (once per query tile)
      s_n = pages_of(comb_clamp_len(__ldg(cache_lens + b), max_pages), kCombPage);
      s_pb = before * NQT + qt * s_n;
      total *= NQT;
      s_chunk = total > 0 ? (total + G - 1) / G : 1;
    }
  }
  __syncthreads();
  // launched as a programmatic dependent of the split kernel: everything above only read
  // the lengths; the partials are read after the split grid has completed and flushed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n = s_n;
  const int c_first = n > 0 ? s_pb / s_chunk : 0, c_last = n > 0 ? (s_pb + n - 1) / s_chunk : -1;
  const int nsplit = c_last - c_first + 1;
  const int row = row0 + lane;
  const bool live = lane < nrows;
  constexpr int kQ = kCombQuads / kCombWarps;  // quads per warp
  float4 acc[kQ];
#pragma unroll
  for (int j = 0; j < kQ; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  float mx = -INFINITY, wsum = 0.f;
  if (live && nsplit > 0) {
    // every thread weighs the splits of its own row: w_s = exp(lse_s - max) / sum; the
    // partial loads of the first two splits are issued before the weights are known
    const size_t slot_stride = (size_t)128 * TQ;
    const float4* src = reinterpret_cast<const float4*>(part_o) +
                        ((size_t)(c_first + v) * 128 + q_base + warp) * TQ + r0 + lane;
    const float* lsp = part_lse + ((size_t)c_first + v) * TQ + r0 + lane;
    float4 a[2][kQ];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int j = 0; j < kQ; ++j)
        a[u][j] = u < nsplit ? __ldg(src + (size_t)u * slot_stride + (size_t)j * kCombWarps * TQ)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < nsplit; ++k) mx = fmaxf(mx, __ldg(lsp + (size_t)k * TQ));
    for (int k = 0; k < nsplit; ++k) {
      const float ls = __ldg(lsp + (size_t)k * TQ);
      wsum += (mx == -INFINITY || ls == -INFINITY) ? 0.f : __expf(ls - mx);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    auto weight = [&](int k) -> float {
      const float ls = __ldg(lsp + (size_t)k * TQ);
      return (mx == -INFINITY || ls == -INFINITY) ? 0.f : __expf(ls - mx) * inv;
    };
    for (int k = 0; k < nsplit; k += 2) {
      if (k > 0) {
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int j = 0; j < kQ; ++j)
            a[u][j] = k + u < nsplit ? __ldg(src + (size_t)(k + u) * slot_stride + (size_t)j * kCombWarps * TQ)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float w = k + u < nsplit ? weight(k + u) : 0.f;
#pragma unroll
        for (int j = 0; j < kQ; ++j) {
          acc[j].x += w * a[u][j].x; acc[j].y += w * a[u][j].y;
          acc[j].z += w * a[u][j].z; acc[j].w += w * a[u][j].w;
        }
      }
    }
  }
  if (live && warp == 0 && blockIdx.z == 0)
    lse[((size_t)b * H + row % H) * T + row / H] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
#pragma unroll
  for (int j = 0; j < kQ; ++j) {
    const int ql = warp + j * kCombWarps;  // quad within this CTA's 32
    const uint32_t lo = (uint32_t)f32_to_bf16_rne(acc[j].x) | ((uint32_t)f32_to_bf16_rne(acc[j].y) << 16);
    const uint32_t hi = (uint32_t)f32_to_bf16_rne(acc[j].z) | ((uint32_t)f32_to_bf16_rne(acc[j].w) << 16);
    *reinterpret_cast<uint2*>(&s_out[lane][ql * 4]) = make_uint2(lo, hi);
  }
  __syncthreads();
  // rows out: this CTA's 128 columns of each row are 16 x 16 bytes
  for (int i = threadIdx.x; i < nrows * 16; i += kCombWarps * 32) {
    const int rr = i >> 4, cc = i & 15;
    reinterpret_cast<uint4*>(out + ((size_t)b * TH + row0 + rr) * kCombDl + q_base * 4)[cc] =
        reinterpret_cast<const uint4*>(&s_out[rr][0])[cc];
  }
}

cudaError_t launch_decode_combine(const float* part_o, const float* part_lse,
                                  const int* cache_lens, void* out, float* lse, int B, int H,
                                  int T, int max_pages, int G, cudaStream_t stream) {
  const int TH = T * H;
  // programmatic dependent launch: the CTAs may start (and scan the lengths) while the split
  // kernel drains; they wait for its completion before reading the partials
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B, (TH + kCombRows - 1) / kCombRows, kCombParts);
  cfg.blockDim = dim3(kCombWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel, part_o, part_lse, cache_lens,
                            static_cast<uint16_t*>(out), lse, B, H, T, max_pages, G);
}

}  // namespace mla
