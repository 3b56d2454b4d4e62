// Fused MLA prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), bf16.
//
// One CTA = one (batch, head) and 256 query rows held as two 128-row Q tiles; keys in
// tiles of BN = 128.  Warp roles (12 warps):
//   warp 0      TMA producer: the two Q tiles once, then a ring of K_nope / V slots
//               (32 KB each) and K_rope slots (16 KB) through mbarrier full/empty pairs
//   warp 1      MMA issuer (one elected thread): S_t = Q_t K' over the nope and rope
//               depths into TMEM, then O_t += P_t V with P_t read from TMEM
//   warp 2      TMEM allocation / release (512 columns: S_0, S_1, O_0, O_1)
//   warps 4-7   softmax of Q tile 0, warps 8-11 softmax of Q tile 1: one thread per
//               row; row max, exp2, row sum, P (bf16) written over S in TMEM, and the
//               conditional rescale of O when the running max grows by more than 2^8
// The MMA warp interleaves the two tiles (PV_0(j), S_0(j+1), PV_1(j), S_1(j+1)) so one
// softmax warpgroup works while the tensor core serves the other.
//
// Structure after the pages' KVPipelineGeneric (ring of K/V stages released by the
// consumer's commit) and MLASmemStorage (Q nope+rope, KV nope sharing one column budget
// with V plus a rope slice per stage); tile sizes and roles are this kernel's own.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace sm103_prefill {

constexpr int BM = 128, BN = 128, NQ = 2;
constexpr int kChunk = 128 * 128;                     // one 128-row x 128-byte swizzled chunk
constexpr int kQTile = 3 * kChunk;                    // nope (2 chunks) + rope (1 chunk)
constexpr int kRingSlots = 3, kRopeSlots = 2;
constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + NQ * kQTile;         // 96 KB
constexpr int kOffRope = kOffRing + kRingSlots * 2 * kChunk;
constexpr int kSmemBytes = kOffRope + kRopeSlots * kChunk;  // 224 KB
constexpr int kSmemAlloc = kSmemBytes + 1024;
constexpr int kThreads = 384;
// registers per thread after the run-time hand-off (setmaxnreg): 128 producer/MMA threads
// drop to kRegsLow, 256 softmax threads rise to kRegsHigh; the launch must provide their
// average (rounded up to the allocation granule of 8)
constexpr int kRegsLow = 56, kRegsHigh = 224;
constexpr int kRegsAtLaunch = ((128 * kRegsLow + 256 * kRegsHigh + kThreads - 1) / kThreads + 7) / 8 * 8;
static_assert(kRegsAtLaunch * kThreads <= 65536, "register hand-off exceeds the SM's file");

struct Params {
  int B, H, S, causal, nrb, out_f32;
  float scale_log2;
  void* out;
  float* lse;
  unsigned int* err;
  size_t out_bytes, lse_bytes;  // for the store checks of the bounds-checked build
};

struct Bars {
  uint64_t q_full;
  uint64_t ring_full[kRingSlots], ring_empty[kRingSlots];
  uint64_t rope_full[kRopeSlots], rope_empty[kRopeSlots];
  uint64_t s_full[NQ], p_full[NQ][2], o_done[NQ];  // p_full[t][h]: keys 64h..64h+63 of P_t
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ int n_kv_tiles(const Params& p, int q_row0) {
  const int all = (p.S + BN - 1) / BN;
  return p.causal ? min(all, (q_row0 + NQ * BM + BN - 1) / BN) : all;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tm_qn,
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
  const int n_kv = n_kv_tiles(p, q_row0);
  // causal: Q tile 0 never sees the last key tile of its row block (all of it is above the
  // diagonal), so its S / softmax / PV stop one tile earlier
  const int n_kv0 = p.causal ? min(n_kv, (q_row0 + BM + BN - 1) / BN) : n_kv;

  if (threadIdx.x == 0) {
    bars.abort_flag = 0;
    ptx::mbar_init(&bars.q_full, 1);
    for (int i = 0; i < kRingSlots; ++i) {
      ptx::mbar_init(&bars.ring_full[i], 1);
      ptx::mbar_init(&bars.ring_empty[i], 1);
    }
    for (int i = 0; i < kRopeSlots; ++i) {
      ptx::mbar_init(&bars.rope_full[i], 1);
      ptx::mbar_init(&bars.rope_empty[i], 1);
    }
    for (int t = 0; t < NQ; ++t) {
      ptx::mbar_init(&bars.s_full[t], 1);
      ptx::mbar_init(&bars.p_full[t][0], BM / 32);  // one arrival per softmax warp
      ptx::mbar_init(&bars.p_full[t][1], BM / 32);
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
      ptx::prefetch_tensormap(&tm_qn);
      ptx::prefetch_tensormap(&tm_kn);
      ptx::mbar_arrive_expect_tx(&bars.q_full, NQ * kQTile);
      for (int t = 0; t < NQ; ++t) {
        unsigned char* q = sm + kOffQ + t * kQTile;
        const int row = q_row0 + t * BM;
        ptx::tma_load_4d(q, &tm_qn, &bars.q_full, 0, h, row, b);
        ptx::tma_load_4d(q + kChunk, &tm_qn, &bars.q_full, 64, h, row, b);
        ptx::tma_load_4d(q + 2 * kChunk, &tm_qr, &bars.q_full, 0, h, row, b);
      }
      for (int j = 0; j < n_kv; ++j) {
        const int key0 = j * BN;
        // K_nope -> ring slot (sequence number 2j), K_rope -> rope slot j
        {
          const int seq = 2 * j, s = seq % kRingSlots;
          if (!ptx::mbar_wait(&bars.ring_empty[s], ((seq / kRingSlots) & 1) ^ 1, abort_flag, p.err)) break;
          unsigned char* dst = sm + kOffRing + s * 2 * kChunk;
          ptx::mbar_arrive_expect_tx(&bars.ring_full[s], 2 * kChunk);
          ptx::tma_load_4d(dst, &tm_kn, &bars.ring_full[s], 0, h, key0, b);
          ptx::tma_load_4d(dst + kChunk, &tm_kn, &bars.ring_full[s], 64, h, key0, b);
        }
        {
          const int s = j % kRopeSlots;
          if (!ptx::mbar_wait(&bars.rope_empty[s], ((j / kRopeSlots) & 1) ^ 1, abort_flag, p.err)) break;
          ptx::mbar_arrive_expect_tx(&bars.rope_full[s], kChunk);
          ptx::tma_load_3d(sm + kOffRope + s * kChunk, &tm_kr, &bars.rope_full[s], 0, key0, b);
        }
        // V -> ring slot (sequence number 2j + 1)
        {
          const int seq = 2 * j + 1, s = seq % kRingSlots;
          if (!ptx::mbar_wait(&bars.ring_empty[s], ((seq / kRingSlots) & 1) ^ 1, abort_flag, p.err)) break;
          unsigned char* dst = sm + kOffRing + s * 2 * kChunk;
          ptx::mbar_arrive_expect_tx(&bars.ring_full[s], 2 * kChunk);
          ptx::tma_load_4d(dst, &tm_v, &bars.ring_full[s], 0, h, key0, b);
          ptx::tma_load_4d(dst + kChunk, &tm_v, &bars.ring_full[s], 64, h, key0, b);
        }
        // warm L2 with the key tile two ahead: its ring slot frees only once this tile's PV is
        // done, and the load then pays the full latency unless the bytes are already in L2
        if (j + 2 < n_kv) {
          const int key2 = key0 + 2 * BN;
          ptx::tma_prefetch_4d(&tm_kn, 0, h, key2, b);
          ptx::tma_prefetch_4d(&tm_kn, 64, h, key2, b);
          ptx::tma_prefetch_3d(&tm_kr, 0, key2, b);
          ptx::tma_prefetch_4d(&tm_v, 0, h, key2, b);
          ptx::tma_prefetch_4d(&tm_v, 64, h, key2, b);
        }
      }
    } else if (warp == 1 && ptx::elect_one()) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdS = ptx::make_idesc(1, BM, BN, 0, 0);    // Q K', both K-major
      constexpr uint32_t kIdPV = ptx::make_idesc(1, BM, 128, 0, 1);  // P V, V is N-major
      const uint32_t q_base = ptx::smem_u32(sm + kOffQ);
      const uint32_t ring_base = ptx::smem_u32(sm + kOffRing);
      const uint32_t rope_base = ptx::smem_u32(sm + kOffRope);
      // operand descriptors built once; a tile at a byte offset from its base differs only in
      // the start-address field (address / 16, no carry below 256 KB)
      const uint64_t d_q = ptx::sw128_desc(q_base, 16, 1024);
      const uint64_t d_ring = ptx::sw128_desc(ring_base, 16, 1024);
      const uint64_t d_rope = ptx::sw128_desc(rope_base, 16, 1024);
      const uint64_t d_v = ptx::sw128_desc(ring_base, kChunk, 1024);
      // (an opaque add, so the compiler forms each descriptor where it is used instead of
      // keeping all of them live)
      auto at = [](uint64_t d, uint32_t bytes) {
        uint64_t r;
        asm volatile("add.u64 %0, %1, %2;" : "=l"(r) : "l"(d), "l"(static_cast<uint64_t>(bytes >> 4)));
        return r;
      };
      bool ok = ptx::mbar_wait(&bars.q_full, 0, abort_flag, p.err);

      // S_t(j) = Q_t K(j)': 8 k-steps over the nope chunks + 4 over the rope chunk
      auto issue_s = [&](int t, int j) {
        const int ks = (2 * j) % kRingSlots, rs = j % kRopeSlots;
        const uint64_t qa = at(d_q, t * kQTile);
        const uint64_t kb = at(d_ring, ks * 2 * kChunk);
        const uint64_t rb_ = at(d_rope, rs * kChunk);
        const uint32_t d = tmem + t * BN;
#pragma unroll
        for (int k = 0; k < 12; ++k) {
          const int c = k >> 2, kk = k & 3;
          const uint64_t da = at(qa, c * kChunk + kk * 32);
          const uint64_t db = c < 2 ? at(kb, c * kChunk + kk * 32) : at(rb_, kk * 32);
          ptx::mma_bf16_ss(d, da, db, kIdS, k > 0);
        }
      };
      auto wait_k = [&](int j) -> bool {
        const int seq = 2 * j;
        return ptx::mbar_wait(&bars.ring_full[seq % kRingSlots], (seq / kRingSlots) & 1, abort_flag, p.err) &&
               ptx::mbar_wait(&bars.rope_full[j % kRopeSlots], (j / kRopeSlots) & 1, abort_flag, p.err);
      };
      // O_t (+)= P_t V(j): P_t (bf16, 64 TMEM columns over S_t), 8 k-steps of 16 keys
      // PV in two halves of 64 keys, each issued as soon as that half of P is in TMEM
      auto issue_pv = [&](int t, int j) -> bool {
        const int vs = (2 * j + 1) % kRingSlots;
        const uint64_t vb = at(d_v, vs * 2 * kChunk);
        const uint32_t d = tmem + 2 * BN + t * 128;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (!ptx::mbar_wait(&bars.p_full[t][hf], j & 1, abort_flag, p.err)) return false;
          ptx::tc_fence_after();
#pragma unroll
          for (int k = 4 * hf; k < 4 * hf + 4; ++k) {
            ptx::mma_bf16_ts(d, tmem + t * BN + k * 8, at(vb, k * 2048), kIdPV, (j > 0 || k > 0) ? 1u : 0u);
          }
        }
        return true;
      };
      if (ok && n_kv > 0 && (ok = wait_k(0))) {
        issue_s(0, 0);
        ptx::mma_commit(&bars.s_full[0]);
        issue_s(1, 0);
        ptx::mma_commit(&bars.s_full[1]);
        ptx::mma_commit(&bars.ring_empty[0]);
        ptx::mma_commit(&bars.rope_empty[0]);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int vseq = 2 * j + 1;
        if (!(ok = ptx::mbar_wait(&bars.ring_full[vseq % kRingSlots], (vseq / kRingSlots) & 1, abort_flag, p.err))) break;
        const bool more = j + 1 < n_kv;
        bool k_ready = false;
        if (j < n_kv0) {
          if (!(ok = issue_pv(0, j))) break;
          ptx::mma_commit(&bars.o_done[0]);
          if (j + 1 < n_kv0) {
            if (!(ok = wait_k(j + 1))) break;
            k_ready = true;
            issue_s(0, j + 1);
            ptx::mma_commit(&bars.s_full[0]);
          }
        }
        if (!(ok = issue_pv(1, j))) break;
        ptx::mma_commit(&bars.o_done[1]);
        ptx::mma_commit(&bars.ring_empty[vseq % kRingSlots]);
        if (more) {
          if (!k_ready && !(ok = wait_k(j + 1))) break;
          issue_s(1, j + 1);
          ptx::mma_commit(&bars.s_full[1]);
          ptx::mma_commit(&bars.ring_empty[(2 * j + 2) % kRingSlots]);
          ptx::mma_commit(&bars.rope_empty[(j + 1) % kRopeSlots]);
        }
      }
    }
  } else {
    // -------------------------------------------------------------- softmax warpgroups
    ptx::regs_inc<kRegsHigh>();
    const int t = (warp >> 2) - 1;      // Q tile of this warpgroup
    const int r = (warp & 3) * 32 + lane;  // row within the tile == TMEM lane
    const int i = q_row0 + t * BM + r;     // query index
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + t * BN;
    const uint32_t o_addr = tmem + lane_off + 2 * BN + t * 128;
    float m = -INFINITY, l = 0.f, lr = 0.f;  // exact row sum (LSE), bf16-rounded sum (O)
    bool ok = true;
    const int n_t = t == 0 ? n_kv0 : n_kv;  // key tiles this Q tile sees
    for (int j = 0; j < n_t; ++j) {
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.s_full[t], j & 1, abort_flag, p.err));
      if (!ok) break;
      ptx::tc_fence_after();
      float s[128];
      {
        // all four 32-column loads in flight before one wait
        uint32_t* su = reinterpret_cast<uint32_t*>(s);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          ptx::tmem_ld32(s_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(su + c * 32));
        ptx::tmem_ld_wait();
      }
      const int key0 = j * BN;
      const bool need_mask = (key0 + BN > p.S) || (p.causal && key0 + BN - 1 > q_row0 + t * BM);
      if (need_mask) {
        const int lim = p.causal ? min(i + 1, p.S) : p.S;  // keys < lim are visible
#pragma unroll
        for (int x = 0; x < 128; ++x)
          if (key0 + x >= lim) s[x] = -INFINITY;
      }
      // row max: four independent chains of three-input maxima
      float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int x = 4; x < 128; x += 2) mx4[(x >> 1) & 3] = ptx::fmax3(mx4[(x >> 1) & 3], s[x], s[x + 1]);
      const float mx = ptx::fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
      const float m_tile = mx * p.scale_log2;  // -inf stays -inf
      float m_use = m;
      if (j == 0) {
        m_use = m_tile;
      } else {
        const bool grow = m_tile > m + 8.0f;
        if (__any_sync(0xffffffffu, grow)) {
          // O of PV(j-1) must be complete before it is rescaled
          ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.o_done[t], (j - 1) & 1, abort_flag, p.err));
          if (!ok) break;
          ptx::tc_fence_after();
          const float alpha = grow ? ptx::ex2(m - m_tile) : 1.f;
          if (grow) m_use = m_tile;
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
          l *= alpha;
          lr *= alpha;
        }
      }
      m = m_use;
      const float neg_m = -m;
      // two keys per packed fp32x2 instruction: exponent argument, exact row sum and the
      // sum of the bf16-rounded values the PV product uses (O is normalised by the latter,
      // so a dominant key is normalised exactly; the LSE uses the exact sum)
      const uint64_t sc2 = ptx::f2(p.scale_log2, p.scale_log2), nm2 = ptx::f2(neg_m, neg_m);
      uint64_t ps2[2] = {ptx::f2(0.f, 0.f), ptx::f2(0.f, 0.f)};
      float pr[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const uint64_t a2 = ptx::fma2(ptx::f2(s[c * 64 + 2 * x], s[c * 64 + 2 * x + 1]), sc2, nm2);
          const float p0 = ptx::ex2(ptx::f2_lo(a2));
          const float p1 = ptx::ex2(ptx::f2_hi(a2));
          const uint32_t w = ptx::pack_bf16x2(p0, p1);
          pk[x] = w;
          ps2[x & 1] = ptx::add2(ps2[x & 1], ptx::f2(p0, p1));
          ptx::add_bf16x2(pr[2 * (x & 1)], pr[2 * (x & 1) + 1], w);
        }
        ptx::tmem_st32(s_addr + c * 32, pk);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars.p_full[t][c]);
      }
      const uint64_t ps_all = ptx::add2(ps2[0], ps2[1]);
      l += ptx::f2_lo(ps_all) + ptx::f2_hi(ps_all);
      lr += (pr[0] + pr[1]) + (pr[2] + pr[3]);
    }
    // epilogue: O / l -> out, LSE
    if (ok && n_t > 0 &&
        __all_sync(0xffffffffu, ptx::mbar_wait(&bars.o_done[t], (n_t - 1) & 1, abort_flag, p.err))) {
      ptx::tc_fence_after();
      const float inv = lr > 0.f ? 1.f / lr : 0.f;
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
              uint4 w;
              w.x = ptx::pack_bf16x2(__uint_as_float(v[8 * x + 0]) * inv, __uint_as_float(v[8 * x + 1]) * inv);
              w.y = ptx::pack_bf16x2(__uint_as_float(v[8 * x + 2]) * inv, __uint_as_float(v[8 * x + 3]) * inv);
              w.z = ptx::pack_bf16x2(__uint_as_float(v[8 * x + 4]) * inv, __uint_as_float(v[8 * x + 5]) * inv);
              w.w = ptx::pack_bf16x2(__uint_as_float(v[8 * x + 6]) * inv, __uint_as_float(v[8 * x + 7]) * inv);
              if (MLA_STORE_OK(dst + x, p.out, p.out_bytes, p.err)) dst[x] = w;
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

}  // namespace sm103_prefill

// ---------------------------------------------------------------- host side

cudaError_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* ptr,
                              const uint64_t* dims, const uint64_t* strides, const uint32_t* box);

static bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* p,
                   const uint64_t* dims, const uint64_t* strides, const uint32_t* box) {
  return encode_tensor_map(m, dt, rank, p, dims, strides, box) == cudaSuccess;
}

// [B, S, H, d] tensor of 2-byte elements, box = 64 columns x 1 head x `rows` tokens
static bool map_bshd(CUtensorMap* m, const void* p, int B, int S, int H, int d, int rows) {
  uint64_t dims[4] = {(uint64_t)d, (uint64_t)H, (uint64_t)S, (uint64_t)B};
  uint64_t strides[3] = {(uint64_t)d * 2, (uint64_t)H * d * 2, (uint64_t)S * H * d * 2};
  uint32_t box[4] = {64, 1, (uint32_t)rows, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p, dims, strides, box);
}

cudaError_t launch_prefill_sm103_bf16(const void* q_nope, const void* q_rope, const void* k_nope,
                                      const void* k_rope, const void* v, void* out, float* lse,
                                      int B, int H, int S, float softmax_scale, int causal,
                                      bool out_f32, unsigned int* err, cudaStream_t stream) {
  using namespace sm103_prefill;
  CUtensorMap tqn, tqr, tkn, tkr, tv;
  uint64_t kr_dims[3] = {64, (uint64_t)S, (uint64_t)B};
  uint64_t kr_strides[2] = {64 * 2, (uint64_t)S * 64 * 2};
  uint32_t kr_box[3] = {64, BN, 1};
  if (!map_bshd(&tqn, q_nope, B, S, H, 128, BM) || !map_bshd(&tqr, q_rope, B, S, H, 64, BM) ||
      !map_bshd(&tkn, k_nope, B, S, H, 128, BN) || !map_bshd(&tv, v, B, S, H, 128, BN) ||
      !encode(&tkr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_rope, kr_dims, kr_strides, kr_box))
    return cudaErrorInvalidValue;
  Params p;
  p.B = B;
  p.H = H;
  p.S = S;
  p.causal = causal;
  p.nrb = (S + NQ * BM - 1) / (NQ * BM);
  p.out_f32 = out_f32 ? 1 : 0;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = out;
  p.lse = lse;
  {
    const size_t out_full = (size_t)B * S * H * 128 * (out_f32 ? 4 : 2);
    p.out_bytes = out_full - (testing_out_shrink() < out_full ? testing_out_shrink() : out_full);
    p.lse_bytes = (size_t)B * H * S * sizeof(float);
  }
  p.err = err;
  // The warpgroups trade registers at run time (setmaxnreg): the producer/MMA warpgroup drops
  // to kRegsLow and the two softmax warpgroups rise to kRegsHigh.  The raised counts are drawn
  // from the registers the CTA was launched with, so the launch must give every thread at
  // least their average; with fewer the raise would wait forever.  Refuse to launch then.
  static int regs_ok = 0;  // 0 unknown, 1 checked
  if (!__atomic_load_n(&regs_ok, __ATOMIC_ACQUIRE)) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, prefill_bf16_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kRegsAtLaunch) return cudaErrorInvalidDeviceFunction;
    __atomic_store_n(&regs_ok, 1, __ATOMIC_RELEASE);
  }
  static unsigned long long smem_set = 0;
  {
    cudaError_t e = smem_attr_once(prefill_bf16_kernel, kSmemAlloc, &smem_set);
    if (e != cudaSuccess) return e;
  }
  const long long grid = (long long)B * H * p.nrb;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prefill_bf16_kernel<<<(unsigned)grid, kThreads, kSmemAlloc, stream>>>(tqn, tqr, tkn, tkr, tv, p);
  return cudaGetLastError();
}

}  // namespace mla
