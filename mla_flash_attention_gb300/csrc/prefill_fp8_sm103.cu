// Fused MLA prefill with fp8 e4m3 Q_nope / K_nope / V and one fp32 scale per query and per
// key token (tcgen05 + TMEM + TMA).
//
// Score: s_ij = qs_i ks_j Sn_ij + Sr_ij with Sn = Qn8 Kn8' on the 8-bit MMA (kind::f8f6f4)
// and Sr = Qr Kr' on the bf16 MMA, accumulated in two separate fp32 TMEM buffers (the
// scales are applied per element in the softmax, so nothing is rounded before the fp32
// sum).  V_j = ks_j V8_j, so the value product takes P''_ij = p_ij ks_j against V8 widened
// to f16 (exact), with p_ij = 2^(c s_ij - m_i), c = softmax scale x log2(e).  The row's
// reference m_i is the running maximum of u_ij = c s_ij + log2 ks_j (the key scale folded
// into the exponent, log2 ks floored at -16), raised lazily only when some u exceeds it by
// more than 2^8: then P'' <= 2^8 fits f16 (11 significant bits) whatever the key scales, and
// p itself stays below 2^24.  The row sum for the LSE and the normalisation is the fp32 sum
// of p (exact up to fp32 rounding); O is accumulated in fp32 and written in fp32 by default.
//
// One CTA = (batch, head, 256 query rows) as two 128-row Q tiles; keys in tiles of 64.  Each
// Q tile has its own score buffers (Sn, Sr: 64 + 64 TMEM columns, P'' written over Sr) and
// O (128 columns): 2 x 256 = 512 TMEM columns.  The MMA warp interleaves the tiles
// (Sn_0(j+1), PV_0(j), Sr_0(j+1), then the same for tile 1), each tile's next nope scores
// going out as soon as its softmax has read S(j), so one softmax warpgroup works while the
// tensor core serves the other.  Warps: 0 TMA producer (3-stage rings), 1 MMA issuer, 2-3
// converters (V8 -> f16 N-major tile, key scales into shared memory; warp 2 also owns the
// TMEM allocation), 4-7 softmax of Q tile 0, 8-11 softmax of Q tile 1 (one thread per row).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>

#include "common.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace sm103_prefill_fp8 {

constexpr int BM = 128, BN = 64, NQ = 2;   // two 128-row Q tiles, 64-key tiles
constexpr int kQChunk = BM * 128;          // 128 rows x 128 bytes
constexpr int kKChunk = BN * 128;          // 64 rows x 128 bytes
constexpr int kStages = 3;
constexpr int kOffQn = 0;                                  // NQ x 16 KB (fp8 nope)
constexpr int kOffQr = kOffQn + NQ * kQChunk;              // NQ x 16 KB (bf16 rope)
constexpr int kOffKn = kOffQr + NQ * kQChunk;              // stages x 8 KB
constexpr int kOffKr = kOffKn + kStages * kKChunk;         // stages x 8 KB
constexpr int kOffV8 = kOffKr + kStages * kKChunk;         // stages x 8 KB
constexpr int kOffVh = kOffV8 + kStages * kKChunk;         // stages x 16 KB (2 chunks, f16)
constexpr int kSmemBytes = kOffVh + kStages * 2 * kKChunk; // 64 + 3 x 40 = 184 KB
constexpr int kSmemAlloc = kSmemBytes + 1024;
constexpr int kThreads = 384;
constexpr int kConvThreads = 64;
// registers per thread after the run-time hand-off (setmaxnreg): warpgroup 0 (producer, MMA,
// converters) drops to kRegsLow, the two softmax warpgroups rise to kRegsHigh; the launch
// must provide their average (rounded up to the allocation granule of 8)
constexpr int kRegsLow = 80, kRegsHigh = 208;
constexpr int kRegsAtLaunch = ((128 * kRegsLow + 256 * kRegsHigh + kThreads - 1) / kThreads + 7) / 8 * 8;
static_assert(kRegsAtLaunch * kThreads <= 65536, "register hand-off exceeds the SM's file");
constexpr float kLog2KsFloor = -16.f;       // log2 ks below this counts as this (see above)

struct Params {
  int B, H, S, causal, nrb, out_f32;
  float scale_log2;
  const float* q_scale;
  const float* k_scale;
  void* out;
  float* lse;
  unsigned int* err;
  size_t out_bytes, lse_bytes;  // for the store checks of the bounds-checked build
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v8_full[kStages], v8_empty[kStages], vh_full[kStages], vh_empty[kStages];
  uint64_t ks_full[kStages];
  uint64_t s_full[NQ], s_read[NQ], p_full[NQ], o_done[NQ];
  uint32_t tmem_base;
  int abort_flag;
  // read 16 bytes at a time by the softmax warps (one shared-memory wavefront per four keys)
  alignas(16) float ks[kStages][BN];    // the key tile's dequantisation scales
  alignas(16) float lks[kStages][BN];   // max(log2 ks, kLog2KsFloor)
};
static_assert(offsetof(Bars, ks) % 16 == 0 && offsetof(Bars, lks) % 16 == 0 && (BN * 4) % 16 == 0,
              "the key-scale rows are read 16 bytes at a time");

__device__ __forceinline__ int n_kv_tiles(const Params& p, int rows_end) {
  const int all = (p.S + BN - 1) / BN;
  return p.causal ? min(all, (rows_end + BN - 1) / BN) : all;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_fp8_kernel(const __grid_constant__ CUtensorMap tm_qn,
                       const __grid_constant__ CUtensorMap tm_qr,
                       const __grid_constant__ CUtensorMap tm_kn,
                       const __grid_constant__ CUtensorMap tm_kr,
                       const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ Bars bars;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int bid = blockIdx.x;
  const int bh = bid / p.nrb;
  const int rb = p.nrb - 1 - (bid % p.nrb);  // longest row blocks of a (b, h) first
  const int b = bh / p.H, h = bh % p.H;
  const int q_row0 = rb * NQ * BM;
  const int n_kv = n_kv_tiles(p, q_row0 + NQ * BM);  // key tiles Q tile 1 sees
  const int n_kv0 = n_kv_tiles(p, q_row0 + BM);      // Q tile 0 (one row tile less)

  if (threadIdx.x == 0) {
    ptx::prefetch_tensormap(&tm_qn);
    ptx::prefetch_tensormap(&tm_qr);
    ptx::prefetch_tensormap(&tm_kn);
    ptx::prefetch_tensormap(&tm_kr);
    ptx::prefetch_tensormap(&tm_v);
    bars.abort_flag = 0;
    ptx::mbar_init(&bars.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(&bars.k_full[i], 1);
      ptx::mbar_init(&bars.k_empty[i], 1);
      ptx::mbar_init(&bars.v8_full[i], 1);
      ptx::mbar_init(&bars.v8_empty[i], kConvThreads / 32);
      ptx::mbar_init(&bars.vh_full[i], kConvThreads / 32);
      ptx::mbar_init(&bars.vh_empty[i], 1);
      ptx::mbar_init(&bars.ks_full[i], kConvThreads / 32);
    }
    for (int t = 0; t < NQ; ++t) {
      ptx::mbar_init(&bars.s_full[t], 1);
      ptx::mbar_init(&bars.p_full[t], 4);  // one arrival per softmax warp of the tile
      ptx::mbar_init(&bars.s_read[t], 4);
      ptx::mbar_init(&bars.o_done[t], 1);
    }
    ptx::fence_barrier_init();
  }
  if (warp == 2) ptx::tmem_alloc(&bars.tmem_base, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort_flag = &bars.abort_flag;

  if (warp < 4) {
    ptx::regs_dec<kRegsLow>();
    if (warp == 0 && ptx::elect_one()) {
      // ------------------------------------------------------------ producer
      ptx::mbar_arrive_expect_tx(&bars.q_full, NQ * 2 * kQChunk);
      for (int t = 0; t < NQ; ++t) {
        const int row = q_row0 + t * BM;
        ptx::tma_load_4d(sm + kOffQn + t * kQChunk, &tm_qn, &bars.q_full, 0, h, row, b);
        ptx::tma_load_4d(sm + kOffQr + t * kQChunk, &tm_qr, &bars.q_full, 0, h, row, b);
      }
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % kStages, ph = ((j / kStages) & 1) ^ 1, key0 = j * BN;
        if (!ptx::mbar_wait(&bars.k_empty[s], ph, abort_flag, p.err)) break;
        ptx::mbar_arrive_expect_tx(&bars.k_full[s], 2 * kKChunk);
        ptx::tma_load_4d(sm + kOffKn + s * kKChunk, &tm_kn, &bars.k_full[s], 0, h, key0, b);
        ptx::tma_load_3d(sm + kOffKr + s * kKChunk, &tm_kr, &bars.k_full[s], 0, key0, b);
        if (!ptx::mbar_wait(&bars.v8_empty[s], ph, abort_flag, p.err)) break;
        ptx::mbar_arrive_expect_tx(&bars.v8_full[s], kKChunk);
        ptx::tma_load_4d(sm + kOffV8 + s * kKChunk, &tm_v, &bars.v8_full[s], 0, h, key0, b);
      }
    } else if (warp == 1 && ptx::elect_one()) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdSn = ptx::make_idesc(0, BM, BN, 0, 0);   // e4m3 x e4m3
      constexpr uint32_t kIdSr = ptx::make_idesc(1, BM, BN, 0, 0);   // bf16 rope
      constexpr uint32_t kIdPV = ptx::make_idesc(0, BM, 128, 0, 1);  // f16 P'' x f16 V (N-major)
      const uint32_t qn = ptx::smem_u32(sm + kOffQn), qr = ptx::smem_u32(sm + kOffQr);
      const uint32_t kn = ptx::smem_u32(sm + kOffKn), kr = ptx::smem_u32(sm + kOffKr);
      const uint32_t vh = ptx::smem_u32(sm + kOffVh);
      const uint64_t dqn = ptx::sw128_desc(qn, 16, 1024), dqr = ptx::sw128_desc(qr, 16, 1024);
      const uint64_t dkn = ptx::sw128_desc(kn, 16, 1024), dkr = ptx::sw128_desc(kr, 16, 1024);
      const uint64_t dvh = ptx::sw128_desc(vh, kKChunk, 1024);
      // operand descriptors built once; a tile at a byte offset from its base differs only in
      // the start-address field (address / 16, no carry below 256 KB)
      auto at = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
      bool ok = ptx::mbar_wait(&bars.q_full, 0, abort_flag, p.err);
      // S_t(j): Sn_t over the nope depth (K = 128 fp8 = 4 x 32), Sr_t over the rope depth
      // (K = 64 bf16 = 4 x 16); TMEM columns of tile t: [256t, 256t+64) Sn,
      // [256t+64, 256t+128) Sr (P'' in its first 32), [256t+128, 256t+256) O
      auto issue_sn = [&](int t, int j) {
        const int s = j % kStages;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ptx::mma_f8_ss(tmem + t * 256, at(dqn, t * kQChunk + k * 32), at(dkn, s * kKChunk + k * 32), kIdSn, k > 0);
        }
      };
      auto issue_sr = [&](int t, int j) {
        const int s = j % kStages;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ptx::mma_bf16_ss(tmem + t * 256 + 64, at(dqr, t * kQChunk + k * 32), at(dkr, s * kKChunk + k * 32), kIdSr, k > 0);
        }
      };
      auto wait_k = [&](int j) -> bool {
        return ptx::mbar_wait(&bars.k_full[j % kStages], (j / kStages) & 1, abort_flag, p.err);
      };
      // O_t (+)= P''_t(j) V(j): P'' (f16 pairs, 32 TMEM columns over Sr_t), 4 k-steps of 16
      // keys; B = the f16 V tile, N-major (two 64-column chunks 8 KB apart)
      auto issue_pv = [&](int t, int j) -> bool {
        if (!ptx::mbar_wait(&bars.p_full[t], j & 1, abort_flag, p.err)) return false;
        ptx::tc_fence_after();
        const uint32_t v = (j % kStages) * 2 * kKChunk;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          ptx::mma_bf16_ts(tmem + t * 256 + 128, tmem + t * 256 + 64 + k * 8, at(dvh, v + k * 2048), kIdPV,
                           (j > 0 || k > 0) ? 1u : 0u);
        return true;
      };
      // Per key tile j and Q tile t: the nope scores of tile j + 1 go out as soon as the
      // softmax has read S_t(j) (their columns are then free), the PV product on P''_t(j)
      // (written over Sr_t), then the rope scores of j + 1 over it; the two Q tiles interleave.
      if (ok && n_kv > 0 && (ok = wait_k(0))) {
        ptx::tc_fence_after();
        for (int t = 0; t < NQ; ++t) {
          issue_sn(t, 0);
          issue_sr(t, 0);
          ptx::mma_commit(&bars.s_full[t]);
        }
        ptx::mma_commit(&bars.k_empty[0]);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % kStages;
        if (!(ok = ptx::mbar_wait(&bars.vh_full[s], (j / kStages) & 1, abort_flag, p.err))) break;
        const bool more = j + 1 < n_kv;
        bool k_ready = false;
        if (j < n_kv0) {
          const bool next0 = j + 1 < n_kv0;
          if (next0) {
            if (!(ok = wait_k(j + 1))) break;
            k_ready = true;
            if (!(ok = ptx::mbar_wait(&bars.s_read[0], j & 1, abort_flag, p.err))) break;
            ptx::tc_fence_after();
            issue_sn(0, j + 1);
          }
          if (!(ok = issue_pv(0, j))) break;
          ptx::mma_commit(&bars.o_done[0]);
          if (next0) {
            issue_sr(0, j + 1);
            ptx::mma_commit(&bars.s_full[0]);
          }
        }
        if (more) {
          if (!k_ready && !(ok = wait_k(j + 1))) break;
          if (!(ok = ptx::mbar_wait(&bars.s_read[1], j & 1, abort_flag, p.err))) break;
          ptx::tc_fence_after();
          issue_sn(1, j + 1);
        }
        if (!(ok = issue_pv(1, j))) break;
        ptx::mma_commit(&bars.o_done[1]);
        ptx::mma_commit(&bars.vh_empty[s]);
        if (more) {
          issue_sr(1, j + 1);
          ptx::mma_commit(&bars.s_full[1]);
          ptx::mma_commit(&bars.k_empty[(j + 1) % kStages]);
        }
      }
    } else if (warp >= 2) {
      // ------------------------------------------------------------ converters (64 threads)
      const int ct = threadIdx.x - 64;         // 0..63: key row of the tile
      bool ok = true;
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % kStages, ph = (j / kStages) & 1, key = j * BN + ct;
        // slot s is free once PV_1(j - kStages) is done
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.vh_empty[s], ph ^ 1, abort_flag, p.err));
        if (!ok) break;
        {
          const float ksv = key < p.S ? __ldg(p.k_scale + (size_t)b * p.S + key) : 0.f;
          bars.ks[s][ct] = ksv;
          bars.lks[s][ct] = ksv > 0.f ? fmaxf(__log2f(ksv), kLog2KsFloor) : kLog2KsFloor;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars.ks_full[s]);
        // V8 (64 keys x 128 fp8, one 128B-swizzled row per key) -> f16 N-major tile: row
        // `ct`, all eight 16-byte groups of 16 codes
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.v8_full[s], ph, abort_flag, p.err));
        if (!ok) break;
        const unsigned char* src = sm + kOffV8 + s * kKChunk + ct * 128;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 raw = *reinterpret_cast<const uint4*>(src + ((g ^ (ct & 7)) << 4));  // 128B swizzle
          const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t w[8];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            ptx::e4m3x4_to_f16x2x2(rw[x], w[2 * x], w[2 * x + 1]);
          }
          // columns 16g .. 16g+15 -> chunk g / 4, 16-byte groups 2(g%4), 2(g%4)+1 (swizzled)
          unsigned char* dst = sm + kOffVh + s * 2 * kKChunk + (g >> 2) * kKChunk + ct * 128;
          const int g0 = 2 * (g & 3);
          *reinterpret_cast<uint4*>(dst + ((g0 ^ (ct & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(dst + (((g0 + 1) ^ (ct & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        ptx::fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&bars.v8_empty[s]);
          ptx::mbar_arrive(&bars.vh_full[s]);
        }
      }
    }
  } else {
    // -------------------------------------------------------------- softmax warpgroups
    ptx::regs_inc<kRegsHigh>();
    const int t = (warp >> 2) - 1;          // Q tile of this warpgroup
    const int r = (warp & 3) * 32 + lane;   // row within the tile == TMEM lane
    const int i = q_row0 + t * BM + r;      // query index
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t sn_addr = tmem + lane_off + t * 256;  // Sn; Sr (then P'') at + 64
    const uint32_t o_addr = sn_addr + 128;
    const float qs = i < p.S ? __ldg(p.q_scale + (size_t)b * p.S + i) : 0.f;
    const uint64_t qs2 = ptx::f2(qs, qs), c2 = ptx::f2(p.scale_log2, p.scale_log2);
    float m = -INFINITY;             // reference of u = c s + log2 ks (exponent domain)
    uint64_t l2 = ptx::f2(0.f, 0.f); // row sum of p = 2^(c s - m), two lanes
    bool ok = true;
    const int n_t = t == 0 ? n_kv0 : n_kv;  // key tiles this Q tile sees
    for (int j = 0; j < n_t; ++j) {
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.s_full[t], j & 1, abort_flag, p.err));
      if (!ok) break;
      ptx::tc_fence_after();
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.ks_full[j % kStages], (j / kStages) & 1, abort_flag, p.err));
      if (!ok) break;
      const float4* ks4 = reinterpret_cast<const float4*>(bars.ks[j % kStages]);
      const float4* lks4 = reinterpret_cast<const float4*>(bars.lks[j % kStages]);
      // scores s = qs ks Sn + Sr and the running maxima of u = c s + log2 ks (four chains),
      // two keys per packed instruction, 32 keys per half
      uint64_t s2[32];
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      const int key0 = j * BN;
      const bool need_mask = (key0 + BN > p.S) || (p.causal && key0 + BN - 1 > q_row0 + t * BM);
      const int lim = p.causal ? min(i + 1, p.S) : p.S;  // keys < lim are visible
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t vn[32], vr[32];
        ptx::tmem_ld32(sn_addr + hf * 32, vn);
        ptx::tmem_ld32(sn_addr + 64 + hf * 32, vr);
        ptx::tmem_ld_wait();
        if (need_mask) {  // masked keys: Sn = 0, Sr = -inf, so s = u = -inf
#pragma unroll
          for (int y = 0; y < 32; ++y)
            if (key0 + hf * 32 + y >= lim) {
              vn[y] = 0u;
              vr[y] = __float_as_uint(-INFINITY);
            }
        }
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 kq = ks4[hf * 8 + q4], lq = lks4[hf * 8 + q4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int x = 2 * q4 + e;  // key pair within the half
            const uint64_t ks2 = e == 0 ? ptx::f2(kq.x, kq.y) : ptx::f2(kq.z, kq.w);
            const uint64_t lks2 = e == 0 ? ptx::f2(lq.x, lq.y) : ptx::f2(lq.z, lq.w);
            s2[hf * 16 + x] = ptx::fma2(ptx::f2(__uint_as_float(vn[2 * x]), __uint_as_float(vn[2 * x + 1])),
                                        ptx::mul2(qs2, ks2),
                                        ptx::f2(__uint_as_float(vr[2 * x]), __uint_as_float(vr[2 * x + 1])));
            const uint64_t u = ptx::fma2(s2[hf * 16 + x], c2, lks2);
            mx4[x & 3] = ptx::fmax3(mx4[x & 3], ptx::f2_lo(u), ptx::f2_hi(u));
          }
        }
      }
      // S_t(j) is in registers: the MMA warp may write the next tile's nope scores
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars.s_read[t]);
      const float mx = ptx::fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
      float m_use = m;
      if (j == 0) {
        m_use = mx;
      } else {
        const bool grow = mx > m + 8.0f;
        if (__any_sync(0xffffffffu, grow)) {
          // O of PV_t(j-1) must be complete before it is rescaled
          ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.o_done[t], (j - 1) & 1, abort_flag, p.err));
          if (!ok) break;
          ptx::tc_fence_after();
          const float alpha = grow ? ptx::ex2(m - mx) : 1.f;
          if (grow) m_use = mx;
          uint32_t v[2][32];
#pragma unroll
          for (int c = 0; c < 4; c += 2) {
            ptx::tmem_ld32(o_addr + c * 32, v[0]);
            ptx::tmem_ld32(o_addr + (c + 1) * 32, v[1]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32; ++x) {
              v[0][x] = __float_as_uint(__uint_as_float(v[0][x]) * alpha);
              v[1][x] = __float_as_uint(__uint_as_float(v[1][x]) * alpha);
            }
            ptx::tmem_st32(o_addr + c * 32, v[0]);
            ptx::tmem_st32(o_addr + (c + 1) * 32, v[1]);
          }
          l2 = ptx::mul2(l2, ptx::f2(alpha, alpha));
        }
      }
      m = m_use;
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      const uint64_t nm2 = ptx::f2(neg_m, neg_m);
      // p = 2^(c s - m) (fp32; the row sum), P'' = p ks in f16 over Sr (the PV weight)
      uint32_t pk[32];
#pragma unroll
      for (int q4 = 0; q4 < 16; ++q4) {
        const float4 kq = ks4[q4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int x = 2 * q4 + e;
          const uint64_t a2 = ptx::fma2(s2[x], c2, nm2);
          const uint64_t pp = ptx::f2(ptx::ex2(ptx::f2_lo(a2)), ptx::ex2(ptx::f2_hi(a2)));
          l2 = ptx::add2(l2, pp);
          const uint64_t w2 = ptx::mul2(pp, e == 0 ? ptx::f2(kq.x, kq.y) : ptx::f2(kq.z, kq.w));
          pk[x] = ptx::pack_f16x2(ptx::f2_lo(w2), ptx::f2_hi(w2));
        }
      }
      ptx::tmem_st32(sn_addr + 64, pk);  // over Sr_t
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars.p_full[t]);
    }
    // epilogue: O / l -> out, LSE
    if (ok && n_t > 0 &&
        __all_sync(0xffffffffu, ptx::mbar_wait(&bars.o_done[t], (n_t - 1) & 1, abort_flag, p.err))) {
      ptx::tc_fence_after();
      const float l = ptx::f2_lo(l2) + ptx::f2_hi(l2);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool store = i < p.S;
      const size_t row_off = ((static_cast<size_t>(b) * p.S + i) * p.H + h) * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::tmem_ld32(o_addr + c * 32, v);
        ptx::tmem_ld_wait();
        if (store) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + row_off + c * 32);
#pragma unroll
            for (int x = 0; x < 8; ++x)
              if (MLA_STORE_OK(dst + x, p.out, p.out_bytes, p.err))
                dst[x] = make_float4(__uint_as_float(v[4 * x]) * inv, __uint_as_float(v[4 * x + 1]) * inv,
                                   __uint_as_float(v[4 * x + 2]) * inv, __uint_as_float(v[4 * x + 3]) * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row_off + c * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              uint4 wv;
              wv.x = ptx::pack_bf16x2(__uint_as_float(v[8 * x + 0]) * inv, __uint_as_float(v[8 * x + 1]) * inv);
              wv.y = ptx::pack_bf16x2(__uint_as_float(v[8 * x + 2]) * inv, __uint_as_float(v[8 * x + 3]) * inv);
              wv.z = ptx::pack_bf16x2(__uint_as_float(v[8 * x + 4]) * inv, __uint_as_float(v[8 * x + 5]) * inv);
              wv.w = ptx::pack_bf16x2(__uint_as_float(v[8 * x + 6]) * inv, __uint_as_float(v[8 * x + 7]) * inv);
              if (MLA_STORE_OK(dst + x, p.out, p.out_bytes, p.err)) dst[x] = wv;
            }
          }
        }
      }
      if (store)
        if (MLA_STORE_OK(p.lse + (static_cast<size_t>(b) * p.H + h) * p.S + i, p.lse, p.lse_bytes, p.err))
          p.lse[(static_cast<size_t>(b) * p.H + h) * p.S + i] =
            l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace sm103_prefill_fp8

cudaError_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* ptr,
                              const uint64_t* dims, const uint64_t* strides, const uint32_t* box);

cudaError_t launch_prefill_sm103_fp8(const void* q_nope, const void* q_rope, const void* k_nope,
                                     const void* k_rope, const void* v, const float* q_scale,
                                     const float* k_scale, void* out, float* lse, int B, int H,
                                     int S, float softmax_scale, int causal, bool out_f32,
                                     unsigned int* err, cudaStream_t stream) {
  using namespace sm103_prefill_fp8;
  CUtensorMap tqn, tqr, tkn, tkr, tv;
  // fp8 [B,S,H,128]: one 128-byte box row per token (Q: 128 tokens per box, K/V: 64)
  uint64_t n_dims[4] = {128, (uint64_t)H, (uint64_t)S, (uint64_t)B};
  uint64_t n_str[3] = {128, (uint64_t)H * 128, (uint64_t)S * H * 128};
  uint32_t q_box[4] = {128, 1, BM, 1};
  uint32_t k_box[4] = {128, 1, BN, 1};
  // bf16 q_rope [B,S,H,64]
  uint64_t r_dims[4] = {64, (uint64_t)H, (uint64_t)S, (uint64_t)B};
  uint64_t r_str[3] = {128, (uint64_t)H * 128, (uint64_t)S * H * 128};
  uint32_t r_box[4] = {64, 1, BM, 1};
  // bf16 k_rope [B,S,64]
  uint64_t kr_dims[3] = {64, (uint64_t)S, (uint64_t)B};
  uint64_t kr_str[2] = {128, (uint64_t)S * 128};
  uint32_t kr_box[3] = {64, BN, 1};
  cudaError_t e;
  if ((e = encode_tensor_map(&tqn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, q_nope, n_dims, n_str, q_box)) != cudaSuccess ||
      (e = encode_tensor_map(&tkn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, k_nope, n_dims, n_str, k_box)) != cudaSuccess ||
      (e = encode_tensor_map(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, v, n_dims, n_str, k_box)) != cudaSuccess ||
      (e = encode_tensor_map(&tqr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, q_rope, r_dims, r_str, r_box)) != cudaSuccess ||
      (e = encode_tensor_map(&tkr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_rope, kr_dims, kr_str, kr_box)) != cudaSuccess)
    return e;
  Params p;
  p.B = B;
  p.H = H;
  p.S = S;
  p.causal = causal;
  p.nrb = (S + NQ * BM - 1) / (NQ * BM);
  p.out_f32 = out_f32 ? 1 : 0;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.out = out;
  p.lse = lse;
  {
    const size_t out_full = (size_t)B * S * H * 128 * (out_f32 ? 4 : 2);
    p.out_bytes = out_full - (testing_out_shrink() < out_full ? testing_out_shrink() : out_full);
    p.lse_bytes = (size_t)B * H * S * sizeof(float);
  }
  p.err = err;
  // The warpgroups trade registers at run time (setmaxnreg); the raised counts are drawn
  // from the registers the CTA was launched with, so refuse to launch with fewer than their
  // average (the raise would wait forever).
  static int regs_ok = 0;  // 0 unknown, 1 checked
  if (!__atomic_load_n(&regs_ok, __ATOMIC_ACQUIRE)) {
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, prefill_fp8_kernel)) != cudaSuccess) return e;
    if (fa.numRegs < kRegsAtLaunch) return cudaErrorInvalidDeviceFunction;
    __atomic_store_n(&regs_ok, 1, __ATOMIC_RELEASE);
  }
  static unsigned long long smem_set = 0;
  if ((e = smem_attr_once(prefill_fp8_kernel, kSmemAlloc, &smem_set)) != cudaSuccess) return e;
  const long long grid = (long long)B * H * p.nrb;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prefill_fp8_kernel<<<(unsigned)grid, kThreads, kSmemAlloc, stream>>>(tqn, tqr, tkn, tkr, tv, p);
  return cudaGetLastError();
}

}  // namespace mla
