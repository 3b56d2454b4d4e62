// Fused MLA prefill with fp8 e4m3 Q_nope / K_nope / V and one fp32 scale per query and per
// key token (tcgen05 + TMEM + TMA).
//
// Score: s_ij = scale * (qs_i ks_j Sn_ij + Sr_ij) with Sn = Qn8 Kn8' on the 8-bit MMA
// (kind::f8f6f4) and Sr = Qr Kr' on the bf16 MMA, accumulated in two separate fp32 TMEM
// buffers (the scales are applied per element in the softmax, so nothing is rounded
// before the fp32 sum).  V_j = ks_j V8_j, so the PV product uses P'_ij = p_ij ks_j against
// V8 widened to bf16 (exact); P' is split into a bf16 high part and a bf16 low part (two
// MMAs), keeping ~16 significant bits -- O reaches |O| ~ 40 on the fp8 workload and is
// accumulated and (by default) written in fp32.
//
// One CTA = (batch, head, 128 query rows), keys in tiles of 64.  The score buffers are
// double-buffered so that S(j+1) runs on the tensor cores while the softmax of tile j runs.
// TMEM: Sn buffers [0,64) [64,128) (later P' of the tile), Sr buffers [128,192) [192,256),
// O [256,384).  Roles (14 warps): warp 0 TMA producer (4-stage rings); warp 1 MMA issuer;
// warps 2-3 and 12-13 converters (V8 -> bf16 into a 128B-swizzled N-major tile, key scales
// into smem); softmax warpgroups 4-7 and 8-11 take keys 0..31 and 32..63 of every tile for
// the same 128 rows, and agree on the running row maximum through shared memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace sm103_prefill_fp8 {

constexpr int BM = 128, BN = 64, KH = 32;   // KH: keys of a tile per softmax warpgroup
constexpr int kQChunk = BM * 128;          // 128 rows x 128 bytes
constexpr int kKChunk = BN * 128;          // 64 rows x 128 bytes
constexpr int kStages = 4;
constexpr int kOffQn = 0;                                  // 16 KB (fp8 nope)
constexpr int kOffQr = kOffQn + kQChunk;                   // 16 KB (bf16 rope)
constexpr int kOffKn = kOffQr + kQChunk;                   // stages x 8 KB
constexpr int kOffKr = kOffKn + kStages * kKChunk;         // stages x 8 KB
constexpr int kOffV8 = kOffKr + kStages * kKChunk;         // stages x 8 KB
constexpr int kOffVb = kOffV8 + kStages * kKChunk;         // stages x 16 KB (2 chunks)
constexpr int kSmemBytes = kOffVb + kStages * 2 * kKChunk; // 32 + 160 = 192 KB
constexpr int kSmemAlloc = kSmemBytes + 1024;
constexpr int kThreads = 448;
constexpr int kConvThreads = 128;
constexpr int kSoftWarps = 8;

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
  uint64_t v8_full[kStages], v8_empty[kStages], vb_full[kStages], vb_empty[kStages];
  uint64_t ks_full[kStages];
  uint64_t s_full[2], p_full[2], o_done;
  uint64_t mx_bar[2], l_bar;  // the two warpgroups' partial row maxima / row sums are in
  uint32_t tmem_base;
  int abort_flag;
  float ks[kStages][BN];
  float mx_part[2][2][BM];    // [tile parity][warpgroup][row]
  float l_part[2][BM];
};

__device__ __forceinline__ int n_kv_tiles(const Params& p, int q_row0) {
  const int all = (p.S + BN - 1) / BN;
  return p.causal ? min(all, (q_row0 + BM + BN - 1) / BN) : all;
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
  const int rb = p.nrb - 1 - (bid % p.nrb);  // longest row blocks first
  const int b = bh / p.H, h = bh % p.H;
  const int q_row0 = rb * BM;
  const int n_kv = n_kv_tiles(p, q_row0);

  if (threadIdx.x == 0) {
    bars.abort_flag = 0;
    ptx::mbar_init(&bars.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(&bars.k_full[i], 1);
      ptx::mbar_init(&bars.k_empty[i], 1);
      ptx::mbar_init(&bars.v8_full[i], 1);
      ptx::mbar_init(&bars.v8_empty[i], kConvThreads);
      ptx::mbar_init(&bars.vb_full[i], kConvThreads);
      ptx::mbar_init(&bars.vb_empty[i], 1);
      ptx::mbar_init(&bars.ks_full[i], kConvThreads);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(&bars.s_full[t], 1);
      ptx::mbar_init(&bars.p_full[t], kSoftWarps);
      ptx::mbar_init(&bars.mx_bar[t], kSoftWarps);
    }
    ptx::mbar_init(&bars.o_done, 1);
    ptx::mbar_init(&bars.l_bar, kSoftWarps);
    ptx::fence_barrier_init();
  }
  if (warp == 2) ptx::tmem_alloc(&bars.tmem_base, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort_flag = &bars.abort_flag;

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (ptx::elect_one()) {
      ptx::mbar_arrive_expect_tx(&bars.q_full, 2 * kQChunk);
      ptx::tma_load_4d(sm + kOffQn, &tm_qn, &bars.q_full, 0, h, q_row0, b);
      ptx::tma_load_4d(sm + kOffQr, &tm_qr, &bars.q_full, 0, h, q_row0, b);
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
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (ptx::elect_one()) {
      constexpr uint32_t kIdS8 = ptx::make_idesc(0, BM, BN, 0, 0);   // e4m3 x e4m3
      constexpr uint32_t kIdS16 = ptx::make_idesc(1, BM, BN, 0, 0);  // bf16 rope
      constexpr uint32_t kIdPV = ptx::make_idesc(1, BM, 128, 0, 1);
      const uint32_t qn = ptx::smem_u32(sm + kOffQn), qr = ptx::smem_u32(sm + kOffQr);
      const uint32_t kn = ptx::smem_u32(sm + kOffKn), kr = ptx::smem_u32(sm + kOffKr);
      const uint32_t vb = ptx::smem_u32(sm + kOffVb);
      bool ok = ptx::mbar_wait(&bars.q_full, 0, abort_flag, p.err);
      // S(j): both score buffers of tile parity j & 1, then the K slot is free
      auto s_tile = [&](int j) -> bool {
        const int s = j % kStages;
        if (!ptx::mbar_wait(&bars.k_full[s], (j / kStages) & 1, abort_flag, p.err)) return false;
        ptx::tc_fence_after();
        const uint32_t dn = tmem + (j & 1) * 64, dr = tmem + 128 + (j & 1) * 64;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // nope: K = 128 fp8 = 4 x 32
          const uint64_t da = ptx::sw128_desc(qn + k * 32, 16, 1024);
          const uint64_t db = ptx::sw128_desc(kn + s * kKChunk + k * 32, 16, 1024);
          ptx::mma_f8_ss(dn, da, db, kIdS8, k > 0);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // rope: K = 64 bf16 = 4 x 16
          const uint64_t da = ptx::sw128_desc(qr + k * 32, 16, 1024);
          const uint64_t db = ptx::sw128_desc(kr + s * kKChunk + k * 32, 16, 1024);
          ptx::mma_bf16_ss(dr, da, db, kIdS16, k > 0);
        }
        ptx::mma_commit(&bars.s_full[j & 1]);
        ptx::mma_commit(&bars.k_empty[s]);
        return true;
      };
      // O += P'(j) V(j): key block k (16 keys) belongs to warpgroup k / 2, whose P' high
      // and low halves sit at columns (k / 2) * 32 + (k & 1) * 8 and 16 further on
      auto pv_tile = [&](int j) {
        const uint32_t v = vb + (j % kStages) * 2 * kKChunk;
        const uint32_t pa = tmem + (j & 1) * 64;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t db = ptx::sw128_desc(v + k * 2048, kKChunk, 1024);
          const uint32_t hi = pa + (k >> 1) * 32 + (k & 1) * 8;
          ptx::mma_bf16_ts(tmem + 256, hi, db, kIdPV, (j > 0 || k > 0) ? 1u : 0u);
          ptx::mma_bf16_ts(tmem + 256, hi + 16, db, kIdPV, 1u);
        }
      };
      if (ok && n_kv > 0) ok = s_tile(0);
      if (ok && n_kv > 1) ok = s_tile(1);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % kStages;
        if (!(ok = ptx::mbar_wait(&bars.vb_full[s], (j / kStages) & 1, abort_flag, p.err))) break;
        if (!(ok = ptx::mbar_wait(&bars.p_full[j & 1], (j >> 1) & 1, abort_flag, p.err))) break;
        ptx::tc_fence_after();
        pv_tile(j);
        ptx::mma_commit(&bars.o_done);
        ptx::mma_commit(&bars.vb_empty[s]);
        // the score buffers of parity j & 1 are free once PV(j) has read P'(j) (in order)
        if (j + 2 < n_kv) ok = s_tile(j + 2);
      }
    }
  } else if (warp < 4 || warp >= 12) {
    // -------------------------------------------------------------- converters (128 threads)
    const int ct = warp < 4 ? threadIdx.x - 64 : threadIdx.x - 320;  // 0..127
    const int row = ct & (BN - 1), g_first = (ct >> 6) * 4;  // key row, first of 4 groups
    bool ok = true;
    for (int j = 0; ok && j < n_kv; ++j) {
      const int s = j % kStages, ph = (j / kStages) & 1, key = j * BN + ct;
      // slot s is free once PV(j - kStages) is done (which needed that tile's softmax)
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.vb_empty[s], ph ^ 1, abort_flag, p.err));
      if (!ok) break;
      if (ct < BN) bars.ks[s][ct] = key < p.S ? __ldg(p.k_scale + (size_t)b * p.S + key) : 0.f;
      ptx::mbar_arrive(&bars.ks_full[s]);
      // V8 (64 keys x 128 fp8, one swizzled 128-byte row per key) -> bf16 N-major tile
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.v8_full[s], ph, abort_flag, p.err));
      if (!ok) break;
      const unsigned char* src = sm + kOffV8 + s * kKChunk + row * 128;
#pragma unroll
      for (int g = g_first; g < g_first + 4; ++g) {  // 16 fp8 values = 16-byte group g of the row
        const uint4 raw = *reinterpret_cast<const uint4*>(src + ((g ^ (row & 7)) << 4));
        const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t w[8];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          w[2 * x] = ptx::e4m3x2_to_bf16x2(rw[x]);
          w[2 * x + 1] = ptx::e4m3x2_to_bf16x2(rw[x] >> 16);
        }
        // columns 16g .. 16g+15 -> chunk (g / 4), logical groups 2(g%4) and 2(g%4)+1
        unsigned char* dst = sm + kOffVb + s * 2 * kKChunk + (g >> 2) * kKChunk + row * 128;
        const int g0 = 2 * (g & 3);
        *reinterpret_cast<uint4*>(dst + ((g0 ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(dst + (((g0 + 1) ^ (row & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      ptx::fence_proxy_async();
      ptx::mbar_arrive(&bars.v8_empty[s]);
      ptx::mbar_arrive(&bars.vb_full[s]);
    }
  } else {
    // -------------------------------------------------------------- softmax warpgroups
    const int w = (warp >> 2) - 1;          // 0: keys 0..31 of a tile, 1: keys 32..63
    const int r = (warp & 3) * 32 + lane;   // query row == TMEM lane
    const int i = q_row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t o_addr = tmem + lane_off + 256 + w * 64;  // this warpgroup's half of O
    const float qs = i < p.S ? __ldg(p.q_scale + (size_t)b * p.S + i) : 1.f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int buf = j & 1;
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.s_full[buf], (j >> 1) & 1, abort_flag, p.err));
      if (!ok) break;
      ptx::tc_fence_after();
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.ks_full[j % kStages], (j / kStages) & 1, abort_flag, p.err));
      if (!ok) break;
      const float* ks = bars.ks[j % kStages] + w * KH;
      const uint32_t sn_addr = tmem + lane_off + buf * 64 + w * KH;
      // unscaled scores qs ks_x Sn + Sr, two keys per packed fp32x2 instruction (the softmax
      // scale is applied inside the exponent argument)
      uint64_t s2[KH / 2];
      {
        uint32_t vn[32], vr[32];
        ptx::tmem_ld32(sn_addr, vn);
        ptx::tmem_ld32(sn_addr + 128, vr);
        ptx::tmem_ld_wait();
        const uint64_t qs2 = ptx::f2(qs, qs);
#pragma unroll
        for (int x = 0; x < KH / 2; ++x)
          s2[x] = ptx::fma2(ptx::f2(__uint_as_float(vn[2 * x]), __uint_as_float(vn[2 * x + 1])),
                            ptx::mul2(qs2, ptx::f2(ks[2 * x], ks[2 * x + 1])),
                            ptx::f2(__uint_as_float(vr[2 * x]), __uint_as_float(vr[2 * x + 1])));
      }
      const int key0 = j * BN + w * KH;
      if ((key0 + KH > p.S) || (p.causal && key0 + KH - 1 > q_row0)) {
        const int lim = p.causal ? min(i + 1, p.S) : p.S;
#pragma unroll
        for (int x = 0; x < KH / 2; ++x)
          s2[x] = ptx::f2(key0 + 2 * x >= lim ? -INFINITY : ptx::f2_lo(s2[x]),
                          key0 + 2 * x + 1 >= lim ? -INFINITY : ptx::f2_hi(s2[x]));
      }
      float mx4[4] = {ptx::f2_lo(s2[0]), ptx::f2_hi(s2[0]), ptx::f2_lo(s2[1]), ptx::f2_hi(s2[1])};
#pragma unroll
      for (int x = 2; x < KH / 2; ++x) mx4[x & 3] = ptx::fmax3(mx4[x & 3], ptx::f2_lo(s2[x]), ptx::f2_hi(s2[x]));
      // both warpgroups' partial maxima of the row -> the same tile maximum in each (scaled
      // to the exponent domain; the scale is positive, -inf stays -inf)
      bars.mx_part[buf][w][r] = ptx::fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]) * p.scale_log2;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars.mx_bar[buf]);
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.mx_bar[buf], (j >> 1) & 1, abort_flag, p.err));
      if (!ok) break;
      const float mx = fmaxf(bars.mx_part[buf][0][r], bars.mx_part[buf][1][r]);
      float m_use = m;
      if (j == 0) {
        m_use = mx;
      } else {
        const bool grow = mx > m + 8.0f;
        if (__any_sync(0xffffffffu, grow)) {
          ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.o_done, (j - 1) & 1, abort_flag, p.err));
          if (!ok) break;
          ptx::tc_fence_after();
          const float alpha = grow ? ptx::ex2(m - mx) : 1.f;
          if (grow) m_use = mx;
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            ptx::tmem_ld32(o_addr + c * 32, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32; ++x) v[x] = __float_as_uint(__uint_as_float(v[x]) * alpha);
            ptx::tmem_st32(o_addr + c * 32, v);
          }
          l *= alpha;
        }
      }
      m = m_use;
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      const uint64_t sc2 = ptx::f2(p.scale_log2, p.scale_log2), nm2 = ptx::f2(neg_m, neg_m);
      uint64_t ps2[2] = {ptx::f2(0.f, 0.f), ptx::f2(0.f, 0.f)};
      uint32_t pk[32];  // P' high part (columns 0..15), low part (16..31)
#pragma unroll
      for (int x = 0; x < KH / 2; ++x) {
        const uint64_t a2 = ptx::fma2(s2[x], sc2, nm2);
        const float p0 = ptx::ex2(ptx::f2_lo(a2));
        const float p1 = ptx::ex2(ptx::f2_hi(a2));
        const uint64_t pp = ptx::f2(p0, p1);
        ps2[x & 1] = ptx::add2(ps2[x & 1], pp);
        const uint64_t ab = ptx::mul2(pp, ptx::f2(ks[2 * x], ks[2 * x + 1]));  // P' = p ks
        const uint32_t hw = ptx::pack_bf16x2(ptx::f2_lo(ab), ptx::f2_hi(ab));
        pk[x] = hw;
        const uint64_t lo2 = ptx::sub2(ab, ptx::f2(__uint_as_float(hw << 16), __uint_as_float(hw & 0xffff0000u)));
        pk[16 + x] = ptx::pack_bf16x2(ptx::f2_lo(lo2), ptx::f2_hi(lo2));
      }
      ptx::tmem_st32(sn_addr, pk);
      const uint64_t ps_all = ptx::add2(ps2[0], ps2[1]);
      l += ptx::f2_lo(ps_all) + ptx::f2_hi(ps_all);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars.p_full[buf]);
    }
    if (ok && n_kv > 0) {
      // the row sum is the sum of both warpgroups' partial sums (in the same order in both)
      bars.l_part[w][r] = l;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars.l_bar);
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.l_bar, 0, abort_flag, p.err)) &&
           __all_sync(0xffffffffu, ptx::mbar_wait(&bars.o_done, (n_kv - 1) & 1, abort_flag, p.err));
    }
    if (ok && n_kv > 0) {
      ptx::tc_fence_after();
      const float lt = bars.l_part[0][r] + bars.l_part[1][r];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const bool store = i < p.S;
      const size_t row_off = ((static_cast<size_t>(b) * p.S + i) * p.H + h) * 128 + w * 64;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
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
      if (store && w == 0)
        if (MLA_STORE_OK(p.lse + (static_cast<size_t>(b) * p.H + h) * p.S + i, p.lse, p.lse_bytes, p.err))
          p.lse[(static_cast<size_t>(b) * p.H + h) * p.S + i] =
            lt > 0.f ? (m + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
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
  p.nrb = (S + BM - 1) / BM;
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
  static unsigned long long smem_set = 0;
  if ((e = smem_attr_once(prefill_fp8_kernel, kSmemAlloc, &smem_set)) != cudaSuccess) return e;
  const long long grid = (long long)B * H * p.nrb;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prefill_fp8_kernel<<<(unsigned)grid, kThreads, kSmemAlloc, stream>>>(tqn, tqr, tkn, tkr, tv, p);
  return cudaGetLastError();
}

}  // namespace mla
