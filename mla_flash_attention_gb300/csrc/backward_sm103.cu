// MLA prefill backward on tcgen05 / TMEM / TMA, bf16 operands.
//
// For one (batch, head), with s = scale * [Qn|Qr][Kn|Kr]' and P = exp(s - LSE) (the forward's
// log-sum-exp reused, so no row statistics are recomputed):
//   dV = P' dO,  dP = dO V',  D_i = sum_d dO_id O_id,  dS = P * (dP - D),
//   dQ = scale dS K,  dK = scale dS' Q   (the rope key is shared by every head: its gradient
//   is the sum over heads, accumulated by fp32 atomics).
//
// Two CTA roles share one launch, one kernel body and one shared-memory plan:
//   key-tile CTAs (b, h, 128 keys): K and V stay in shared memory; query tiles stream by.
//     TMEM: X [0,128) S' = K Q' (keys on lanes), then dP' = V dO'; dV [128,256);
//           dK [256,448) (nope 128 + rope 64); Y [448,512) P', then dS' (bf16 pairs)
//     MMAs per query tile n: dP'(n), dV += P' dO (TS: A = Y), S'(n+1), dK += dS' Q (TS: A = Y)
//   query-tile CTAs (b, h, 128 queries): Q and dO stay; key tiles stream by.
//     TMEM: X [0,128) S = Q K'; [128,256) dP = dO V'; dQ [256,448); Y [448,512) dS (bf16)
//     MMAs per key tile n: S(n+1), dQ += dS K (TS: A = Y), dP(n+1)
//   Scores of the next tile are issued as soon as the elementwise warps have read the
//   current ones out of X, so the tensor pipe works while the exponentials are computed.
// Shared memory (both roles): fixed 3-chunk tile (K | Q) + fixed 2-chunk tile (V | dO), a
// 2-stage ring of streamed 3-chunk tiles (Q | K), one streamed 2-chunk tile (dO | V), and
// the streamed query tiles' -LSE*log2(e) and D vectors (key-tile role).
// Warps: 0 TMA producer, 1 MMA issuer, 2-9 elementwise (TMEM lane quarter = warp % 4,
// column half = (warp - 2) / 4; each half owns 64 score columns and 32 packed columns of Y).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace sm103_bwd {

constexpr int BT = 128;                        // rows of every tile (queries or keys)
constexpr int kChunk = BT * 128;               // 128 rows x 64 bf16, 128B-swizzled (16 KB)
constexpr int kOffFix3 = 0;                    // K (key role) | Q (query role): 3 chunks
constexpr int kOffFix2 = kOffFix3 + 3 * kChunk;  // V | dO: 2 chunks
constexpr int kOffRing = kOffFix2 + 2 * kChunk;  // 2 stages x 3 chunks: Q | K
constexpr int kOffOne = kOffRing + 2 * 3 * kChunk;  // dO | V: 2 chunks
constexpr int kOffVec = kOffOne + 2 * kChunk;    // per ring stage: -LSE*log2e [128], D [128]
constexpr int kSmemBytes = kOffVec + 2 * 2 * BT * 4;  // 210 KB
constexpr int kSmemAlloc = kSmemBytes + 1024;
constexpr int kThreads = 320;
constexpr uint32_t kColX = 0, kColDP = 128, kColDV = 128, kColAcc = 256, kColY = 448;

struct Params {
  const float* nlse2;  // [B*H, S_pad]: -LSE * log2(e); +padding rows hold -inf
  const float* dvec;   // [B*H, S_pad]: D = rowsum(dO * O); padding rows hold 0
  uint16_t* dq_nope;   // [B, S, H, 128]
  uint16_t* dq_rope;   // [B, S, H, 64]
  uint16_t* dk_nope;   // [B, S, H, 128]
  float* dk_rope;      // [B, S, 64], accumulated (zeroed before the launch)
  uint16_t* dv;        // [B, S, H, 128]
  unsigned int* err;
  int B, H, S, S_pad, nt, causal, n_key_ctas;
  float scale, scale_log2;
};

struct Bars {
  // one full barrier per 16 KB chunk of a streamed tile, so the MMAs over its first chunk can
  // start while the later ones are still arriving
  uint64_t fix_full, ring_full[2][3], ring_empty[2], one_full[2], one_empty;
  uint64_t s_full, x_read, dp_full, dp_read, p_ready, dv_done, ds_ready, acc_step, acc_done;
  uint32_t tmem_base;
  int abort_flag;
};

// D = rowsum(dO * O) and -LSE*log2(e) per (b, h, query) into padded [B*H, S_pad] vectors.
// One warp per (b, h, 32 consecutive queries): each 256-byte row of dO and O is read by the
// whole warp (8 bytes a lane), the 32 per-lane partial sums are reduced across lanes by a
// transposing butterfly (16 + 8 + 4 + 2 + 1 exchanges) that leaves row i0 + lane's sum in
// lane `lane`, so the D and LSE accesses are 128-byte coalesced.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t* __restrict__ out,
                                                       const uint16_t* __restrict__ d_out,
                                                       const float* __restrict__ lse,
                                                       float* __restrict__ nlse2,
                                                       float* __restrict__ dvec, int B, int H,
                                                       int S, int S_pad) {
  const long long task = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int groups = S_pad / 32;
  if (task >= (long long)B * H * groups) return;
  const int g = static_cast<int>(task % groups);
  const int bh = static_cast<int>(task / groups);
  const int b = bh / H, h = bh % H;
  const int i0 = g * 32;
  auto lo = [](uint32_t w) { return __uint_as_float(w << 16); };
  auto hi = [](uint32_t w) { return __uint_as_float(w & 0xffff0000u); };
  float part[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    part[r] = 0.f;
    if (i0 + r < S) {
      const size_t ro = (((size_t)b * S + i0 + r) * H + h) * 128 + lane * 4;
      const uint2 a = __ldg(reinterpret_cast<const uint2*>(d_out + ro));
      const uint2 o = __ldg(reinterpret_cast<const uint2*>(out + ro));
      float acc = lo(a.x) * lo(o.x);
      acc = fmaf(hi(a.x), hi(o.x), acc);
      acc = fmaf(lo(a.y), lo(o.y), acc);
      part[r] = fmaf(hi(a.y), hi(o.y), acc);
    }
  }
  // Each exchange with offset w halves the rows a lane keeps: lanes with bit w set keep the
  // upper half of their remaining rows, the others the lower half, and each adds its
  // partner's partial sums of the rows it keeps.  After w = 16, 8, 4, 2, 1, part[0] of lane
  // l holds row l summed over all 32 lanes.
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int r = 0; r < w; ++r) {
      const float send = upper ? part[r] : part[r + w];
      const float keep = upper ? part[r + w] : part[r];
      part[r] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  const int i = i0 + lane;
  const size_t vo = (size_t)bh * S_pad + i;
  if (i < S) {
    dvec[vo] = part[0];
    nlse2[vo] = -lse[(size_t)bh * S + i] * 1.4426950408889634f;
  } else {
    dvec[vo] = 0.f;
    nlse2[vo] = -INFINITY;
  }
}

// Zero the rope-key gradient accumulator (n4 float4 stores).
__global__ void __launch_bounds__(256) bwd_zero_kernel(float4* __restrict__ p, long long n4) {
  for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < n4;
       k += (long long)gridDim.x * blockDim.x)
    p[k] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// 32 fp32 accumulator columns (times `mul`) -> 32 bf16 at dst (64 bytes, 16-byte aligned)
__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const uint32_t (&u)[32], float mul) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    uint4 w;
    w.x = ptx::pack_bf16x2(__uint_as_float(u[8 * x + 0]) * mul, __uint_as_float(u[8 * x + 1]) * mul);
    w.y = ptx::pack_bf16x2(__uint_as_float(u[8 * x + 2]) * mul, __uint_as_float(u[8 * x + 3]) * mul);
    w.z = ptx::pack_bf16x2(__uint_as_float(u[8 * x + 4]) * mul, __uint_as_float(u[8 * x + 5]) * mul);
    w.w = ptx::pack_bf16x2(__uint_as_float(u[8 * x + 6]) * mul, __uint_as_float(u[8 * x + 7]) * mul);
    d[x] = w;
  }
}

struct Maps {
  const CUtensorMap *qn, *qr, *kn, *kr, *v, *dout;
};

// kKeyRole: this CTA owns key tile `tile` and streams query tiles (dK, dV); otherwise it
// owns query tile `tile` and streams key tiles (dQ).
template <bool kKeyRole>
__device__ __forceinline__ void bwd_body(const Maps& m, const Params& p, unsigned char* sm,
                                         Bars& bars, int b, int h, int tile) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t_begin = kKeyRole ? (p.causal ? tile : 0) : 0;
  const int t_end = kKeyRole ? p.nt : (p.causal ? tile + 1 : p.nt);
  const int nsteps = t_end - t_begin;
  const int bh = b * p.H + h;
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort_flag = &bars.abort_flag;

  if (warp == 0) {
    if (ptx::elect_one()) {
      // ------------------------------------------------------------ TMA producer
      ptx::prefetch_tensormap(m.qn);
      ptx::prefetch_tensormap(m.kn);
      const int row0 = tile * BT;
      ptx::mbar_arrive_expect_tx(&bars.fix_full, 5 * kChunk);
      unsigned char* f3 = sm + kOffFix3;
      unsigned char* f2_ = sm + kOffFix2;
      if (kKeyRole) {
        ptx::tma_load_4d(f3, m.kn, &bars.fix_full, 0, h, row0, b);
        ptx::tma_load_4d(f3 + kChunk, m.kn, &bars.fix_full, 64, h, row0, b);
        ptx::tma_load_3d(f3 + 2 * kChunk, m.kr, &bars.fix_full, 0, row0, b);
        ptx::tma_load_4d(f2_, m.v, &bars.fix_full, 0, h, row0, b);
        ptx::tma_load_4d(f2_ + kChunk, m.v, &bars.fix_full, 64, h, row0, b);
      } else {
        ptx::tma_load_4d(f3, m.qn, &bars.fix_full, 0, h, row0, b);
        ptx::tma_load_4d(f3 + kChunk, m.qn, &bars.fix_full, 64, h, row0, b);
        ptx::tma_load_4d(f3 + 2 * kChunk, m.qr, &bars.fix_full, 0, h, row0, b);
        ptx::tma_load_4d(f2_, m.dout, &bars.fix_full, 0, h, row0, b);
        ptx::tma_load_4d(f2_ + kChunk, m.dout, &bars.fix_full, 64, h, row0, b);
      }
      constexpr int kAhead = 2;  // tiles warmed in L2 ahead of their load
      auto warm = [&](int n) {
        const int r0 = (t_begin + n) * BT;
        if (kKeyRole) {
          ptx::tma_prefetch_4d(m.qn, 0, h, r0, b);
          ptx::tma_prefetch_4d(m.qn, 64, h, r0, b);
          ptx::tma_prefetch_4d(m.qr, 0, h, r0, b);
          ptx::tma_prefetch_4d(m.dout, 0, h, r0, b);
          ptx::tma_prefetch_4d(m.dout, 64, h, r0, b);
          const size_t vo = (size_t)bh * p.S_pad + r0;
          ptx::bulk_prefetch(p.nlse2 + vo, BT * 4);
          ptx::bulk_prefetch(p.dvec + vo, BT * 4);
        } else {
          ptx::tma_prefetch_4d(m.kn, 0, h, r0, b);
          ptx::tma_prefetch_4d(m.kn, 64, h, r0, b);
          ptx::tma_prefetch_3d(m.kr, 0, r0, b);
          ptx::tma_prefetch_4d(m.v, 0, h, r0, b);
          ptx::tma_prefetch_4d(m.v, 64, h, r0, b);
        }
      };
      for (int n = 0; n < kAhead && n < nsteps; ++n) warm(n);
      for (int n = 0; n < nsteps; ++n) {
        if (n + kAhead < nsteps) warm(n + kAhead);
        const int r0 = (t_begin + n) * BT, s = n & 1;
        if (!ptx::mbar_wait(&bars.ring_empty[s], ((n >> 1) & 1) ^ 1, abort_flag, p.err)) break;
        unsigned char* dst = sm + kOffRing + s * 3 * kChunk;
        if (kKeyRole) {
          ptx::mbar_arrive_expect_tx(&bars.ring_full[s][0], kChunk + 2 * BT * 4);
          ptx::mbar_arrive_expect_tx(&bars.ring_full[s][1], kChunk);
          ptx::mbar_arrive_expect_tx(&bars.ring_full[s][2], kChunk);
          ptx::tma_load_4d(dst, m.qn, &bars.ring_full[s][0], 0, h, r0, b);
          ptx::tma_load_4d(dst + kChunk, m.qn, &bars.ring_full[s][1], 64, h, r0, b);
          ptx::tma_load_4d(dst + 2 * kChunk, m.qr, &bars.ring_full[s][2], 0, h, r0, b);
          const size_t vo = (size_t)bh * p.S_pad + r0;
          unsigned char* vec = sm + kOffVec + s * 2 * BT * 4;
          ptx::bulk_load(vec, p.nlse2 + vo, BT * 4, &bars.ring_full[s][0]);
          ptx::bulk_load(vec + BT * 4, p.dvec + vo, BT * 4, &bars.ring_full[s][0]);
        } else {
          for (int c = 0; c < 3; ++c) ptx::mbar_arrive_expect_tx(&bars.ring_full[s][c], kChunk);
          ptx::tma_load_4d(dst, m.kn, &bars.ring_full[s][0], 0, h, r0, b);
          ptx::tma_load_4d(dst + kChunk, m.kn, &bars.ring_full[s][1], 64, h, r0, b);
          ptx::tma_load_3d(dst + 2 * kChunk, m.kr, &bars.ring_full[s][2], 0, r0, b);
        }
        if (!ptx::mbar_wait(&bars.one_empty, (n & 1) ^ 1, abort_flag, p.err)) break;
        unsigned char* one = sm + kOffOne;
        const CUtensorMap* tm = kKeyRole ? m.dout : m.v;
        ptx::mbar_arrive_expect_tx(&bars.one_full[0], kChunk);
        ptx::mbar_arrive_expect_tx(&bars.one_full[1], kChunk);
        ptx::tma_load_4d(one, tm, &bars.one_full[0], 0, h, r0, b);
        ptx::tma_load_4d(one + kChunk, tm, &bars.one_full[1], 64, h, r0, b);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (ptx::elect_one()) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdS = ptx::make_idesc(1, BT, BT, 0, 0);     // both K-major
      constexpr uint32_t kIdDV = ptx::make_idesc(1, BT, 128, 0, 1);   // B N-major, N = 128
      constexpr uint32_t kIdAcc = ptx::make_idesc(1, BT, 192, 0, 1);  // B N-major, N = 192
      const uint32_t base = ptx::smem_u32(sm);
      const uint32_t one = base + kOffOne;
      auto ring_of = [&](int n) { return base + kOffRing + (n & 1) * 3 * kChunk; };
      // scores over the 192-deep nope+rope contraction (key role: transposed, keys on lanes)
      auto issue_s = [&](int n) -> bool {
        const uint32_t ring = ring_of(n);
#pragma unroll
        for (int k = 0; k < 12; ++k) {
          if ((k & 3) == 0) {  // each 64-deep chunk as soon as it has landed
            if (!ptx::mbar_wait(&bars.ring_full[n & 1][k >> 2], (n >> 1) & 1, abort_flag, p.err)) return false;
            ptx::tc_fence_after();
          }
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          ptx::mma_bf16_ss(tmem + kColX, ptx::sw128_desc(base + kOffFix3 + off, 16, 1024),
                           ptx::sw128_desc(ring + off, 16, 1024), kIdS, k > 0);
        }
        ptx::mma_commit(&bars.s_full);
        return true;
      };
      // dP = dO V' over d_v = 128 (key role: dP' = V dO' into X; query role: own columns)
      auto issue_dp = [&](int n) -> bool {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if ((k & 3) == 0) {
            if (!ptx::mbar_wait(&bars.one_full[k >> 2], n & 1, abort_flag, p.err)) return false;
            ptx::tc_fence_after();
          }
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          ptx::mma_bf16_ss(tmem + (kKeyRole ? kColX : kColDP),
                           ptx::sw128_desc(base + kOffFix2 + off, 16, 1024),
                           ptx::sw128_desc(one + off, 16, 1024), kIdS, k > 0);
        }
        ptx::mma_commit(&bars.dp_full);
        return true;
      };
      // dK += dS' Q (key role) or dQ += dS K: A = dS (bf16 pairs in Y), B = the streamed
      // 192-wide tile, N-major
      auto issue_acc = [&](int n) {
        const uint32_t ring = ring_of(n);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          ptx::mma_bf16_ts(tmem + kColAcc, tmem + kColY + k * 8,
                           ptx::sw128_desc(ring + k * 2048, kChunk, 1024), kIdAcc,
                           (n > 0 || k > 0) ? 1u : 0u);
        ptx::mma_commit(&bars.ring_empty[n & 1]);
        ptx::mma_commit(&bars.acc_step);
      };
      auto wait = [&](uint64_t* bar, int n) -> bool {
        if (!ptx::mbar_wait(bar, n & 1, abort_flag, p.err)) return false;
        ptx::tc_fence_after();
        return true;
      };
      bool ok = ptx::mbar_wait(&bars.fix_full, 0, abort_flag, p.err) && issue_s(0);
      if (kKeyRole) {
        // per query tile n: dP'(n) | dV(n) | S'(n+1) | dK(n) -- the next scores run while the
        // elementwise warps turn dP'(n) into dS(n)
        for (int n = 0; ok && n < nsteps; ++n) {
          if (!(ok = wait(&bars.x_read, n) && issue_dp(n))) break;
          if (!(ok = wait(&bars.p_ready, n))) break;
#pragma unroll
          for (int k = 0; k < 8; ++k)  // dV += P' dO: A = P' (bf16 pairs in Y), B = dO N-major
            ptx::mma_bf16_ts(tmem + kColDV, tmem + kColY + k * 8,
                             ptx::sw128_desc(one + k * 2048, kChunk, 1024), kIdDV,
                             (n > 0 || k > 0) ? 1u : 0u);
          ptx::mma_commit(&bars.dv_done);
          ptx::mma_commit(&bars.one_empty);
          if (n + 1 < nsteps && !(ok = wait(&bars.dp_read, n) && issue_s(n + 1))) break;
          if (!(ok = wait(&bars.ds_ready, n))) break;
          issue_acc(n);
        }
      } else {
        // per key tile n: S(n+1) | dQ(n) | dP(n+1), with dP(0) issued up front
        if (ok && (ok = issue_dp(0))) ptx::mma_commit(&bars.one_empty);
        for (int n = 0; ok && n < nsteps; ++n) {
          if (n + 1 < nsteps && !(ok = wait(&bars.x_read, n) && issue_s(n + 1))) break;
          if (!(ok = wait(&bars.ds_ready, n))) break;
          issue_acc(n);
          if (n + 1 < nsteps) {
            if (!(ok = wait(&bars.dp_read, n) && issue_dp(n + 1))) break;
            ptx::mma_commit(&bars.one_empty);
          }
        }
      }
      if (ok) ptx::mma_commit(&bars.acc_done);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- elementwise warps
    const int q4 = warp & 3, hf = (warp - 2) >> 2;
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tX = tmem + lane_off + kColX + hf * 64;
    const uint32_t tDP = tmem + lane_off + (kKeyRole ? kColX : kColDP) + hf * 64;
    const uint32_t tY = tmem + lane_off + kColY + hf * 32;
    const int row_idx = tile * BT + r;  // key (key role) or query
    float nl_row = 0.f, d_row = 0.f;
    if (!kKeyRole) {
      nl_row = p.nlse2[(size_t)bh * p.S_pad + row_idx];
      d_row = p.dvec[(size_t)bh * p.S_pad + row_idx];
    }
    const uint64_t sc2 = ptx::f2(p.scale_log2, p.scale_log2);
    // all lanes wait (bounded); the warp goes on only if every lane saw the phase
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool w = __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort_flag, p.err));
      if (w) ptx::tc_fence_after();
      return w;
    };
    // one arrival per warp once its TMEM reads / writes are complete
    auto arrive = [&](uint64_t* bar) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar);
    };
    bool ok = true;
    for (int n = 0; n < nsteps; ++n) {
      const int t = t_begin + n, s = n & 1;
      const float* vec = reinterpret_cast<const float*>(sm + kOffVec + s * 2 * BT * 4);
      ok = wait(&bars.s_full, n & 1);
      // the query vectors of this stage arrived with its TMA transaction: observe it directly
      if (kKeyRole && ok) ok = wait(&bars.ring_full[s][0], (n >> 1) & 1);
      if (!ok) break;
      uint32_t u[64];
      ptx::tmem_ld32(tX, *reinterpret_cast<uint32_t(*)[32]>(u));
      ptx::tmem_ld32(tX + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
      ptx::tmem_ld_wait();
      arrive(&bars.x_read);
      // P = exp2(s * scale * log2(e) - LSE * log2(e)), two columns per packed instruction
      float pr[64];
      if (kKeyRole) {
        const float2* nl = reinterpret_cast<const float2*>(vec) + hf * 32;  // per query
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const float2 l = nl[x];
          const uint64_t a2 = ptx::fma2(ptx::f2(__uint_as_float(u[2 * x]), __uint_as_float(u[2 * x + 1])),
                                        sc2, ptx::f2(l.x, l.y));
          pr[2 * x] = ptx::ex2(ptx::f2_lo(a2));
          pr[2 * x + 1] = ptx::ex2(ptx::f2_hi(a2));
        }
        if (p.causal && t == tile) {  // diagonal tile: a query before the key sees nothing
#pragma unroll
          for (int x = 0; x < 64; ++x)
            if (hf * 64 + x < r) pr[x] = 0.f;
        }
      } else {
        const uint64_t nl2 = ptx::f2(nl_row, nl_row);
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const uint64_t a2 = ptx::fma2(ptx::f2(__uint_as_float(u[2 * x]), __uint_as_float(u[2 * x + 1])),
                                        sc2, nl2);
          pr[2 * x] = ptx::ex2(ptx::f2_lo(a2));
          pr[2 * x + 1] = ptx::ex2(ptx::f2_hi(a2));
        }
        if (p.causal && t == tile) {  // diagonal tile: keys after the query are masked
#pragma unroll
          for (int x = 0; x < 64; ++x)
            if (hf * 64 + x > r) pr[x] = 0.f;
        } else if (!p.causal && (t + 1) * BT > p.S) {  // keys past the sequence end
          const int lim = p.S - t * BT - hf * 64;
#pragma unroll
          for (int x = 0; x < 64; ++x)
            if (x >= lim) pr[x] = 0.f;
        }
      }
      uint32_t pk[32];
      if (kKeyRole) {
        // P' (bf16) into Y once dK(n-1) has consumed the dS' held there
        if (n > 0 && !(ok = wait(&bars.acc_step, (n - 1) & 1))) break;
#pragma unroll
        for (int x = 0; x < 32; ++x) pk[x] = ptx::pack_bf16x2(pr[2 * x], pr[2 * x + 1]);
        ptx::tmem_st32(tY, pk);
        ptx::tmem_st_wait();
        arrive(&bars.p_ready);
      }
      if (!(ok = wait(&bars.dp_full, n & 1))) break;
      ptx::tmem_ld32(tDP, *reinterpret_cast<uint32_t(*)[32]>(u));
      ptx::tmem_ld32(tDP + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
      ptx::tmem_ld_wait();
      arrive(&bars.dp_read);
      // dS = P * (dP - D) as bf16 pairs
      if (kKeyRole) {
        const float2* dd = reinterpret_cast<const float2*>(vec + BT) + hf * 32;  // per query
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const float2 d = dd[x];
          const uint64_t g = ptx::mul2(ptx::f2(pr[2 * x], pr[2 * x + 1]),
                                       ptx::sub2(ptx::f2(__uint_as_float(u[2 * x]), __uint_as_float(u[2 * x + 1])),
                                                 ptx::f2(d.x, d.y)));
          pk[x] = ptx::pack_bf16x2(ptx::f2_lo(g), ptx::f2_hi(g));
        }
      } else {
        const uint64_t d2 = ptx::f2(d_row, d_row);
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const uint64_t g = ptx::mul2(ptx::f2(pr[2 * x], pr[2 * x + 1]),
                                       ptx::sub2(ptx::f2(__uint_as_float(u[2 * x]), __uint_as_float(u[2 * x + 1])), d2));
          pk[x] = ptx::pack_bf16x2(ptx::f2_lo(g), ptx::f2_hi(g));
        }
      }
      // dS into Y once its previous reader is done: dV(n) (key role: P' lives there) or
      // dQ(n-1)
      if (kKeyRole) {
        if (!(ok = wait(&bars.dv_done, n & 1))) break;
      } else if (n > 0 && !(ok = wait(&bars.acc_step, (n - 1) & 1))) {
        break;
      }
      ptx::tmem_st32(tY, pk);
      ptx::tmem_st_wait();
      arrive(&bars.ds_ready);
    }
    // ---------------------------------------------------------------- epilogue
    if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.acc_done, 0, abort_flag, p.err));
    if (ok) {
      ptx::tc_fence_after();
      const bool store = row_idx < p.S;
      const size_t ro = ((size_t)b * p.S + row_idx) * p.H + h;  // row of a [B, S, H, d] tensor
      if (kKeyRole) {
        // half 0: dV (4 chunks) and rope columns 0..31 of dK; half 1: dK nope (4 chunks) and
        // rope columns 32..63
#pragma unroll
        for (int c = 0; c < 5; ++c) {
          const uint32_t col = hf == 0 ? (c < 4 ? kColDV + 32 * c : kColAcc + 128)
                                       : (c < 4 ? kColAcc + 32 * c : kColAcc + 160);
          uint32_t w[32];
          ptx::tmem_ld32(tmem + lane_off + col, w);
          ptx::tmem_ld_wait();
          if (!store) continue;
          if (c < 4) {
            if (hf == 0)
              store_bf16x32(p.dv + ro * 128 + 32 * c, w, 1.f);
            else
              store_bf16x32(p.dk_nope + ro * 128 + 32 * c, w, p.scale);
          } else {
            float4* dst = reinterpret_cast<float4*>(p.dk_rope + ((size_t)b * p.S + row_idx) * 64 + 32 * hf);
#pragma unroll
            for (int x = 0; x < 8; ++x)
              atomicAdd(dst + x, make_float4(__uint_as_float(w[4 * x]) * p.scale,
                                             __uint_as_float(w[4 * x + 1]) * p.scale,
                                             __uint_as_float(w[4 * x + 2]) * p.scale,
                                             __uint_as_float(w[4 * x + 3]) * p.scale));
          }
        }
      } else {
        // dQ: half 0 takes columns 0..95, half 1 columns 96..191 (nope 0..127, rope 128..191)
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const int cc = hf * 3 + c;
          uint32_t w[32];
          ptx::tmem_ld32(tmem + lane_off + kColAcc + 32 * cc, w);
          ptx::tmem_ld_wait();
          if (!store) continue;
          if (cc < 4)
            store_bf16x32(p.dq_nope + ro * 128 + 32 * cc, w, p.scale);
          else
            store_bf16x32(p.dq_rope + ro * 64 + 32 * (cc - 4), w, p.scale);
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_bwd_kernel(const __grid_constant__ CUtensorMap tm_qn,
                       const __grid_constant__ CUtensorMap tm_qr,
                       const __grid_constant__ CUtensorMap tm_kn,
                       const __grid_constant__ CUtensorMap tm_kr,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do, const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ Bars bars;
  const int warp = threadIdx.x >> 5;
  // key-tile CTAs first, then query-tile CTAs; within a role the tiles of one (b, h) are
  // consecutive (most work first), so CTAs that run together stream the same (b, h)'s tiles
  // and find them in L2
  const bool key_role = static_cast<int>(blockIdx.x) < p.n_key_ctas;
  const int idx = key_role ? blockIdx.x : blockIdx.x - p.n_key_ctas;
  const int bh = idx / p.nt;
  const int tile = key_role ? idx % p.nt : p.nt - 1 - idx % p.nt;
  const int b = bh / p.H, h = bh % p.H;

  if (threadIdx.x == 0) {
    bars.abort_flag = 0;
    ptx::mbar_init(&bars.fix_full, 1);
    for (int s = 0; s < 2; ++s) {
      for (int c = 0; c < 3; ++c) ptx::mbar_init(&bars.ring_full[s][c], 1);
      ptx::mbar_init(&bars.ring_empty[s], 1);
    }
    ptx::mbar_init(&bars.one_full[0], 1);
    ptx::mbar_init(&bars.one_full[1], 1);
    ptx::mbar_init(&bars.one_empty, 1);
    ptx::mbar_init(&bars.s_full, 1);
    ptx::mbar_init(&bars.x_read, 8);    // one arrival per elementwise warp
    ptx::mbar_init(&bars.dp_full, 1);
    ptx::mbar_init(&bars.dp_read, 8);
    ptx::mbar_init(&bars.acc_step, 1);
    ptx::mbar_init(&bars.p_ready, 8);
    ptx::mbar_init(&bars.dv_done, 1);
    ptx::mbar_init(&bars.ds_ready, 8);
    ptx::mbar_init(&bars.acc_done, 1);
    ptx::fence_barrier_init();
  }
  if (warp == 0) ptx::tmem_alloc(&bars.tmem_base, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const Maps m{&tm_qn, &tm_qr, &tm_kn, &tm_kr, &tm_v, &tm_do};
  if (key_role)
    bwd_body<true>(m, p, sm, bars, b, h, tile);
  else
    bwd_body<false>(m, p, sm, bars, b, h, tile);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(bars.tmem_base, 512);
  }
}

}  // namespace sm103_bwd

// ---------------------------------------------------------------- host side

cudaError_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* ptr,
                              const uint64_t* dims, const uint64_t* strides, const uint32_t* box);

namespace {
// [B, S, H, d] tensor of bf16, box = 64 columns x 1 head x 128 tokens
bool bwd_map_bshd(CUtensorMap* m, const void* p, int B, int S, int H, int d) {
  uint64_t dims[4] = {(uint64_t)d, (uint64_t)H, (uint64_t)S, (uint64_t)B};
  uint64_t strides[3] = {(uint64_t)d * 2, (uint64_t)H * d * 2, (uint64_t)S * H * d * 2};
  uint32_t box[4] = {64, 1, sm103_bwd::BT, 1};
  return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p, dims, strides, box) == cudaSuccess;
}
}  // namespace

// Bytes of workspace the backward needs: the padded -LSE*log2(e) and D vectors.
size_t prefill_bwd_workspace_bytes(int B, int H, int S) {
  const size_t s_pad = (size_t)(S + sm103_bwd::BT - 1) / sm103_bwd::BT * sm103_bwd::BT;
  const size_t vec = ((size_t)B * H * s_pad * sizeof(float) + 255) / 256 * 256;
  return 2 * vec;
}

cudaError_t launch_prefill_bwd_sm103(const void* q_nope, const void* q_rope, const void* k_nope,
                                     const void* k_rope, const void* v, const void* out,
                                     const float* lse, const void* d_out, void* dq_nope,
                                     void* dq_rope, void* dk_nope, float* dk_rope, void* dv,
                                     int B, int H, int S, float softmax_scale, int causal,
                                     void* workspace, unsigned int* err, cudaStream_t stream) {
  using namespace sm103_bwd;
  const int nt = (S + BT - 1) / BT, S_pad = nt * BT;
  const size_t vec = prefill_bwd_workspace_bytes(B, H, S) / 2;
  float* nlse2 = static_cast<float*>(workspace);
  float* dvec = reinterpret_cast<float*>(static_cast<char*>(workspace) + vec);

  const long long tasks = (long long)B * H * (S_pad / 32);
  const long long prep_blocks = (tasks + 7) / 8;
  if (prep_blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  bwd_prep_kernel<<<(unsigned)prep_blocks, 256, 0, stream>>>(
      static_cast<const uint16_t*>(out), static_cast<const uint16_t*>(d_out), lse, nlse2, dvec, B,
      H, S, S_pad);
  bwd_zero_kernel<<<1024, 256, 0, stream>>>(reinterpret_cast<float4*>(dk_rope),
                                            (long long)B * S * 64 / 4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap tqn, tqr, tkn, tkr, tv, tdo;
  uint64_t kr_dims[3] = {64, (uint64_t)S, (uint64_t)B};
  uint64_t kr_strides[2] = {64 * 2, (uint64_t)S * 64 * 2};
  uint32_t kr_box[3] = {64, BT, 1};
  if (!bwd_map_bshd(&tqn, q_nope, B, S, H, 128) || !bwd_map_bshd(&tqr, q_rope, B, S, H, 64) ||
      !bwd_map_bshd(&tkn, k_nope, B, S, H, 128) || !bwd_map_bshd(&tv, v, B, S, H, 128) ||
      !bwd_map_bshd(&tdo, d_out, B, S, H, 128) ||
      encode_tensor_map(&tkr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_rope, kr_dims, kr_strides,
                        kr_box) != cudaSuccess)
    return cudaErrorInvalidValue;
  Params p;
  p.nlse2 = nlse2;
  p.dvec = dvec;
  p.dq_nope = static_cast<uint16_t*>(dq_nope);
  p.dq_rope = static_cast<uint16_t*>(dq_rope);
  p.dk_nope = static_cast<uint16_t*>(dk_nope);
  p.dk_rope = dk_rope;
  p.dv = static_cast<uint16_t*>(dv);
  p.err = err;
  p.B = B;
  p.H = H;
  p.S = S;
  p.S_pad = S_pad;
  p.nt = nt;
  p.causal = causal;
  p.scale = softmax_scale;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  const long long per_role = (long long)B * H * nt;
  if (2 * per_role > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  p.n_key_ctas = (int)per_role;
  static unsigned long long smem_set = 0;
  if ((e = smem_attr_once(prefill_bwd_kernel, kSmemAlloc, &smem_set)) != cudaSuccess) return e;
  prefill_bwd_kernel<<<(unsigned)(2 * per_role), kThreads, kSmemAlloc, stream>>>(tqn, tqr, tkn,
                                                                                  tkr, tv, tdo, p);
  return cudaGetLastError();
}

}  // namespace mla
