// Per-head absorption products either side of absorbed decode, on tcgen05 / TMEM / TMA:
//
//   y[r, h, :] = x[r, h, :] @ w[h]      x [R, H, K] bf16, w [H, K, N] bf16, y [R, H, N] bf16
//
// (q_latent = q_nope W_UK[h] before decode: K = 128, N = 512; o = O_latent W_UV[h] after
// it: K = 512, N = 128.)  One CTA per (128-row tile of r, 128 columns of n, head h), 4 warps:
// warp 0 (one lane) streams K in 64-deep chunks by TMA through a ring of min(K / 64, 6)
// stages, so a deep contraction keeps most of its chunks in flight at once (x chunk
// 128 rows x 64 K-major, w chunk 64 K-rows x 128 columns N-major, both 128B-swizzled);
// warp 1 (one lane) issues the bf16 MMAs (M = N = 128, K = 16) into a 128-column fp32 TMEM
// accumulator; then every thread takes one row of it to bf16 and stores 256 bytes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace sm103_absorb {

constexpr int BM = 128, BN = 128, BK = 64, kMaxStages = 6;
constexpr int kAChunk = BM * 128;               // 128 rows x 64 bf16
constexpr int kBHalf = BK * 128;                // 64 K-rows x 64 bf16 (one 64-column half)
constexpr int kStageBytes = kAChunk + 2 * kBHalf;  // 32 KB
constexpr int kSmemMax = kMaxStages * kStageBytes + 1024;  // 193 KB
constexpr int kThreads = 128;

struct Params {
  uint16_t* y;
  unsigned int* err;
  int R, H, K, N;
  int stages;  // ring depth, min(K / BK, kMaxStages)
};

__global__ void __launch_bounds__(kThreads) absorb_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                         const __grid_constant__ CUtensorMap tm_w,
                                                         const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN, h = blockIdx.z;
  const int nk = p.K / BK;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(&done, 1);
    ptx::fence_barrier_init();
  }
  if (warp == 0) ptx::tmem_alloc(&tmem_base, BN);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort_ptr = &abort_flag;

  if (warp == 0) {
    if (ptx::elect_one()) {  // TMA producer
      ptx::prefetch_tensormap(&tm_x);
      ptx::prefetch_tensormap(&tm_w);
      for (int kc = 0; kc < nk; ++kc) {
        const int s = kc % p.stages;
        if (!ptx::mbar_wait(&empty[s], ((kc / p.stages) & 1) ^ 1, abort_ptr, p.err)) break;
        unsigned char* st = sm + s * kStageBytes;
        ptx::mbar_arrive_expect_tx(&full[s], kStageBytes);
        ptx::tma_load_3d(st, &tm_x, &full[s], kc * BK, h, m0);
        ptx::tma_load_3d(st + kAChunk, &tm_w, &full[s], n0, kc * BK, h);
        ptx::tma_load_3d(st + kAChunk + kBHalf, &tm_w, &full[s], n0 + 64, kc * BK, h);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (ptx::elect_one()) {  // MMA issuer
      constexpr uint32_t kId = ptx::make_idesc(1, BM, BN, 0, 1);  // bf16, B N-major
      const uint32_t s0 = ptx::smem_u32(sm);
      bool ok = true;
      for (int kc = 0; kc < nk && ok; ++kc) {
        const int s = kc % p.stages;
        if (!(ok = ptx::mbar_wait(&full[s], (kc / p.stages) & 1, abort_ptr, p.err))) break;
        ptx::tc_fence_after();
        const uint32_t a = s0 + s * kStageBytes, b = a + kAChunk;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t da = ptx::sw128_desc(a + kk * 32, 16, 1024);
          const uint64_t db = ptx::sw128_desc(b + kk * 2048, kBHalf, 1024);
          ptx::mma_bf16_ss(tmem, da, db, kId, (kc > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(&empty[s]);
      }
      if (ok) ptx::mma_commit(&done);
    }
    __syncwarp();
  }

  // epilogue: thread = row of the tile (TMEM lane), 128 fp32 columns -> bf16
  const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(&done, 0, abort_ptr, p.err));
  if (ok) {
    ptx::tc_fence_after();
    const int r = m0 + warp * 32 + lane;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    uint4* dst = reinterpret_cast<uint4*>(p.y + ((size_t)r * p.H + h) * p.N + n0);
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t v[32];
      ptx::tmem_ld32(taddr + c * 32, v);
      ptx::tmem_ld_wait();
      if (r < p.R) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 o;
          o.x = ptx::pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
          o.y = ptx::pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
          o.z = ptx::pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
          o.w = ptx::pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
          dst[c * 4 + q] = o;
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, BN);
  }
}

}  // namespace sm103_absorb

cudaError_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* ptr,
                              const uint64_t* dims, const uint64_t* strides, const uint32_t* box);

cudaError_t launch_absorb_sm103(const void* x, const void* w, void* y, int R, int H, int K, int N,
                                unsigned int* err, cudaStream_t stream) {
  using namespace sm103_absorb;
  CUtensorMap tx, tw;
  // x [R, H, K]: boxes of 64 K x 1 head x 128 rows; w [H, K, N]: boxes of 64 N x 64 K x 1 head
  uint64_t xd[3] = {(uint64_t)K, (uint64_t)H, (uint64_t)R};
  uint64_t xs[2] = {(uint64_t)K * 2, (uint64_t)H * K * 2};
  uint32_t xb[3] = {BK, 1, BM};
  uint64_t wd[3] = {(uint64_t)N, (uint64_t)K, (uint64_t)H};
  uint64_t ws[2] = {(uint64_t)N * 2, (uint64_t)K * N * 2};
  uint32_t wb[3] = {64, BK, 1};
  cudaError_t e;
  if ((e = encode_tensor_map(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, xd, xs, xb)) != cudaSuccess ||
      (e = encode_tensor_map(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w, wd, ws, wb)) != cudaSuccess)
    return e;
  static unsigned long long smem_set = 0;
  if ((e = smem_attr_once(absorb_kernel, kSmemMax, &smem_set)) != cudaSuccess) return e;
  Params p;
  p.y = static_cast<uint16_t*>(y);
  p.err = err;
  p.R = R;
  p.H = H;
  p.K = K;
  p.N = N;
  p.stages = K / BK < kMaxStages ? K / BK : kMaxStages;
  if (p.stages < 1) return cudaErrorInvalidValue;
  dim3 grid((R + BM - 1) / BM, N / BN, H);
  absorb_kernel<<<grid, kThreads, p.stages * kStageBytes + 1024, stream>>>(tx, tw, p);
  return cudaGetLastError();
}

}  // namespace mla
