// Absorbed MLA decode over an fp8 paged latent cache, in transposed form, for sequences with
// few query rows (T*H <= 32): the score MMA puts 128 keys on M and the query rows on N, and
// the value MMA accumulates O' (512 latent rows x the query rows) -- 128 TMEM columns for 32
// rows, so one CTA holds the whole output of its work unit and nothing is computed twice.
// The split over the key axis, the partial slots and the merge by the last split to finish
// follow the shared split plan (decode_plan.cuh).
//
// Operands are f16: each fp8 code widens to f16 exactly (one conversion per pair of codes);
// Q is scaled per row by a power of two so its largest magnitude lands in [2^14, 2^15) (f16's
// range, no rounding of a bf16 value in it), and the factor is folded into that row's score
// scale.  With t = scale * ks * s the log2-domain score of a key whose dequantisation scale
// is ks, the value MMA takes P'' = exp2(u - m), u = t + log2(ks): the probability already
// multiplied by ks, which dequantises the key's value row.  The row sum is kept in fp32 as
// sum P'' / ks = sum exp2(t - m).  The reference m of a query row is the running maximum of
// u, updated lazily: only when some u exceeds it by more than 2^8 (so P'' <= 2^8 stays inside
// f16) are the columns' maxima recomputed and O' and the sums rescaled.
//
// A work unit's keys are walked in blocks of two pages (128 keys).  Each block is consumed
// as 17 units: nine score units (64 cache columns x 128 keys, 8 KB of fp8 -> 16 KB of f16,
// K-major) and, per page, four value units (128 latent columns x 64 keys, MN-major).  The
// producer loads every unit's fp8 bytes from L2 into a ring (the pages are warmed in L2
// ahead), the widening warps turn them into f16 operand tiles in a second ring, and the MMA
// warp consumes them in the order S(0), S(1), PV(0), S(2), PV(1), ... so that the softmax of
// block j runs while the scores of block j+1 are computed.
//
// Per CTA (10 warps):
//   warp 0      TMA producer (raw fp8 units) and L2 warm-up of pages and scales ahead
//   warp 1      MMA issuer: S'(j) = C(j) Q' into one of two S' buffers, O' += C(j)' P''(j)
//   warps 2-5   widening: fp8 units -> f16 operand tiles (zero rows for keys outside the
//               sequence); per sequence, Q -> scaled f16 and the rows' score scales
//   warps 6-9   softmax (one thread per key of the block), P'' into shared memory; at the
//               end of a sequence's segment the epilogue (one thread per latent row of O')
//               and, in the CTA that completes a sequence, the merge of its splits
// TMEM columns: [0, 4 NP) O' (four blocks of 128 latent rows), [4 NP, 6 NP) two S' buffers,
// [6 NP, 7 NP) each softmax thread's part of the row sums (lane = the thread's key slot).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "decode_plan.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace sm103_decode_t {

using decode_plan::Plan;
using decode_plan::Segments;
using decode_plan::clamp_len;
using decode_plan::make_plan;
constexpr int kPage = decode_plan::kPage;
constexpr int kDl = 512, kDc = 576;
constexpr int kKeys = 128;            // keys per block: the M of the score MMA
constexpr int kSUnits = 9;            // score units per block (64 cache columns each)
constexpr int kVUnitsPerPage = 4;     // value units per page (128 latent columns each)
constexpr int kRawUnit = 8192;        // fp8 bytes of a unit
constexpr int kWideUnit = 16384;      // f16 bytes of a unit
constexpr int kRawSlots = 12, kWideSlots = 4;
constexpr int kThreads = 320;
constexpr int kPrefetchBlocks = 4;    // blocks warmed in L2 ahead of their loads
constexpr float kTau = 8.f;           // headroom of the lazy reference (log2 units)

template <int NP>
struct Lay {
  static constexpr int kQChunk = NP * 128;  // NP rows x 64 f16, 128B-swizzled
  static constexpr int kOffQ = 0;
  static constexpr int kOffWide = 9 * kQChunk;
  static constexpr int kOffRaw = kOffWide + kWideSlots * kWideUnit;
  static constexpr int kPRow = 2 * NP;     // bytes of one key's P'' row (NP f16)
  static constexpr int kPBytes = kKeys * kPRow;
  static constexpr int kOffP = kOffRaw + kRawSlots * kRawUnit;
  static constexpr int kSmem = kOffP + 2 * kPBytes;
  static constexpr int kSmemAlloc = kSmem + 1024;
  // TMEM columns: O' (4 blocks of NP), two S' buffers, and the softmax threads' row-sum parts
  static constexpr int kTmemO = 0, kTmemS = 4 * NP, kTmemL = 6 * NP;
  static constexpr int kTmemCols = 7 * NP <= 128 ? 128 : 256;
  static constexpr uint32_t kPSwz = NP == 32 ? ptx::kSwz64 : ptx::kSwz32;
  static_assert(kOffWide % 1024 == 0 && kOffP % 1024 == 0, "operand tiles need 1 KB alignment");
  static_assert(kSmemAlloc <= 227 * 1024, "shared memory");
};

struct Params {
  const uint16_t* q_latent;  // [B, T, H, 512] bf16
  const uint16_t* q_rope;    // [B, T, H, 64] bf16
  const uint8_t* kv_cache;   // [num_pages, 64, 576] e4m3 (L2 warm-up)
  const float* kv_scale;     // [num_pages, 64]
  const int* page_table;     // [B, max_pages]
  const int* cache_lens;     // [B]
  float* part_o;             // [n_slots][TQ][512]
  float* part_lse;           // [n_slots][TQ]
  int* counters;             // [B]: finished splits per sequence, zeroed per call
  uint16_t* out;             // [B, T, H, 512] bf16
  float* lse;                // [B, H, T]
  unsigned int* err;
  int B, H, T, max_pages, num_pages, causal, G;
  int NQT;      // query tiles per sequence: 1 (the rows of a sequence fit one tile)
  int TQ;       // query rows per sequence (T * H)
  int n_slots;  // G + B
  float scale_log2;
  long long wait_limit;  // SM clocks a pipeline wait may last before it gives up
  int skip_unit;         // test hook: >= 0 leaves that raw unit unloaded (a wait then runs out)
  int item_cost;         // flat pages the split plan charges per work item (see decode_plan.cuh)
  // buffer sizes for the store checks of the bounds-checked build
  size_t out_bytes, lse_bytes, part_o_bytes, part_lse_bytes, counters_bytes;
};

struct Bars {
  uint64_t raw_full[kRawSlots], raw_empty[kRawSlots];
  uint64_t raw_issued[kRawSlots];  // the producer has waited for the slot and issued its unit
  uint64_t wide_full[kWideSlots], wide_empty[kWideSlots];
  uint64_t q_free, q_ready;
  uint64_t qsc_full[2], qsc_free[2];
  uint64_t s_full[2], s_free[2], p_full[2], p_free[2];
  uint64_t o_done, seg_done, o_free, drain;
  uint64_t soft_sync;   // group barrier of the four softmax warps (one arrival per warp)
  uint32_t tmem_base;
  int abort_flag;
  int merge_last;
  Plan plan;
  __align__(16) float qsc[2][32];  // per query row: scale * log2(e) * 2^-e of its Q scaling
  float red[4][32];     // column reductions across the four softmax warps
  float colv[32];       // reduced columns
  float mref[32];       // reference of each query row (the same in every softmax thread)
  float alpha[32];      // rescale factors of a change of references
  int vote[2][4];       // per-warp votes, by group-barrier parity
  float mx[32], winv[32];  // merge: per row, the largest split LSE and the inverse weight sum
};

// One block of (up to) two pages of a segment, as every role walks them, with the raw
// page-table entries of its pages (pt[q], -1 for an absent second page).
struct Block {
  int seq, L, pg0, npg, j, seg, flat0, lo, hi;
  int pt[2];
  bool first, last;
};

// Walks the blocks of this CTA's work unit in order.  The page-table entries of the block
// after the one handed out are loaded at once, so their latency is spent while the caller
// works on the current block.
struct BlockIter {
  Segments segs;
  const int* table;
  int max_pages;
  int seq, L, lo, hi, pg, seg, j;
  bool open, has;
  Block nxt;
  __device__ bool advance(Block& b) {
    if (!open || pg >= hi) {
      if (!segs.next(seq, L, lo, hi)) return false;
      open = true;
      pg = lo;
      ++seg;
    }
    b.seq = seq;
    b.L = L;
    b.pg0 = pg;
    b.npg = min(2, hi - pg);
    b.j = j++;
    b.seg = seg;
    b.first = pg == lo;
    pg += b.npg;
    b.last = pg >= hi;
    b.flat0 = segs.flat0;
    b.lo = lo;
    b.hi = hi;
    const int* row = table + (size_t)b.seq * max_pages + b.pg0;
    b.pt[0] = __ldg(row);
    b.pt[1] = b.npg > 1 ? __ldg(row + 1) : -1;
    return true;
  }
  __device__ void init(const Params& p, const Plan& plan) {
    segs.init(p, plan);
    table = p.page_table;
    max_pages = p.max_pages;
    open = false;
    seg = -1;
    j = 0;
    has = advance(nxt);
  }
  __device__ bool next(Block& b) {
    if (!has) return false;
    b = nxt;
    has = advance(nxt);
    return true;
  }
};

// Rows of page q (0/1) of block b that hold keys of the sequence (0 for an absent page or a
// page-table entry outside [0, num_pages)); *phys = the physical page or -1.
__device__ __forceinline__ int valid_rows(const Params& p, const Block& b, int q, int* phys) {
  const int page = q == 0 ? b.pt[0] : b.pt[1];  // (no runtime index: keeps Block in registers)
  if (q >= b.npg || page < 0 || page >= p.num_pages) {
    *phys = -1;
    return 0;
  }
  *phys = page;
  return min(kPage, b.L - (b.pg0 + q) * kPage);
}

// Column sums over the 32 lanes of a warp, in place: on return lane l holds the sum over the
// warp of column l (NP = 32) or of column l & 15 (NP = 16).
template <int NP>
__device__ __forceinline__ float warp_column_sums(float (&v)[NP]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = NP / 2; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = keep + got;
    }
  }
  float r = v[0];
  if (NP == 16) {
    const float o = __shfl_xor_sync(0xffffffffu, r, 16);
    r = r + o;
  }
  return r;
}

template <int NP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_t_kernel(const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_v,
                    const Params p) {
  using L_ = Lay<NP>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ Bars bars;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x;
  const int TH = p.T * p.H, TQ = p.TQ;
  const long long lim = p.wait_limit;

  if (threadIdx.x == 0) {
    // the descriptors are fetched while the barriers are set up and the plan is made
    ptx::prefetch_tensormap(&tm_s);
    ptx::prefetch_tensormap(&tm_v);
    bars.abort_flag = 0;
    for (int i = 0; i < kRawSlots; ++i) {
      ptx::mbar_init(&bars.raw_full[i], 1);
      ptx::mbar_init(&bars.raw_empty[i], 1);
      ptx::mbar_init(&bars.raw_issued[i], 1);
    }
    for (int i = 0; i < kWideSlots; ++i) {
      ptx::mbar_init(&bars.wide_full[i], 1);
      ptx::mbar_init(&bars.wide_empty[i], 1);
    }
    ptx::mbar_init(&bars.q_free, 1);
    ptx::mbar_init(&bars.q_ready, 4);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars.qsc_full[i], 4);
      ptx::mbar_init(&bars.qsc_free[i], 4);
      ptx::mbar_init(&bars.s_full[i], 1);
      ptx::mbar_init(&bars.s_free[i], 4);
      ptx::mbar_init(&bars.p_full[i], 4);
      ptx::mbar_init(&bars.p_free[i], 1);
    }
    ptx::mbar_init(&bars.o_done, 1);
    ptx::mbar_init(&bars.seg_done, 1);
    ptx::mbar_init(&bars.o_free, 4);
    ptx::mbar_init(&bars.drain, 1);
    ptx::mbar_init(&bars.soft_sync, 4);
    ptx::fence_barrier_init();
  }
  // the plan's length loads go out first; the other warps set up meanwhile
  if (warp == 2) make_plan(p, unit, &bars.plan);
  // Q rows TQ..NP-1 are never written: keep the whole Q area zero
  for (int i = threadIdx.x; i < 9 * L_::kQChunk / 16; i += kThreads)
    reinterpret_cast<uint4*>(sm + L_::kOffQ)[i] = make_uint4(0, 0, 0, 0);
  ptx::fence_proxy_async();
  if (warp == 1) ptx::tmem_alloc(&bars.tmem_base, L_::kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort_flag = &bars.abort_flag;
  BlockIter it;
  it.init(p, bars.plan);
  Block cur, prev;
  bool have_prev = false;

  if (warp == 0) {
    // -------------------------------------------------------------- TMA producer
    // The whole warp walks the units; lane 0 arms each raw slot and lanes 0 and 1 issue its
    // (up to) two boxes, so that two tile loads are in issue at once.
    int u = 0, last_unit = -1;  // units handed out / the last one whose copies were issued
    bool ok = true;
    // warm L2 with the pages (and their scales) a few blocks ahead of the loads
    BlockIter ahead;
    ahead.init(p, bars.plan);
    Block a;
    int ahead_n = 0;
    auto warm = [&](const Block& bb) {
      for (int q = 0; q < bb.npg; ++q) {
        int ph;
        valid_rows(p, bb, q, &ph);
        if (ph < 0 || lane != 0) continue;
        ptx::bulk_prefetch(p.kv_cache + (size_t)ph * kPage * kDc, kPage * kDc);
        ptx::bulk_prefetch(p.kv_scale + (size_t)ph * kPage, kPage * 4);
      }
    };
    // one raw unit of 8 KB: score units take two 64 x 64 boxes (page a, then page b, at
    // cache column c); value units one 128 x 64 box (page a, columns c .. c + 127).  A page
    // of -1 is not loaded (its rows are zeroed by the widening).
    // marks a slot's unit as handed out.  A widening warp can reach unit u before unit
    // u - kRawSlots has landed (its own previous unit is u - 4), and a raw_full parity only
    // names unit u once that has happened; it waits on raw_issued first, whose phase can be
    // at most one behind (the producer has handed out u - 4, hence u - kRawSlots).
    auto publish = [&](int slot) {
      if (lane == 0) ptx::mbar_arrive(&bars.raw_issued[slot]);
    };
    auto load = [&](bool score, int pa, int pb, int c) -> bool {
      const int slot = u % kRawSlots;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bars.raw_empty[slot], ((u / kRawSlots) & 1) ^ 1, abort_flag, p.err, lim)))
        return false;
      if (u == p.skip_unit) {  // test hook: this unit's bytes never arrive
        publish(slot);
        ++u;
        return true;
      }
      const int bytes = score ? (pa >= 0 ? 4096 : 0) + (pb >= 0 ? 4096 : 0) : (pa >= 0 ? 8192 : 0);
      if (lane == 0) ptx::mbar_arrive_expect_tx(&bars.raw_full[slot], bytes);
      __syncwarp();
      unsigned char* dst = sm + L_::kOffRaw + slot * kRawUnit;
      if (score) {
        if (lane == 0 && pa >= 0) ptx::tma_load_2d(dst, &tm_s, &bars.raw_full[slot], c, pa * kPage);
        if (lane == 1 && pb >= 0) ptx::tma_load_2d(dst + 4096, &tm_s, &bars.raw_full[slot], c, pb * kPage);
      } else if (lane == 0 && pa >= 0) {
        ptx::tma_load_2d(dst, &tm_v, &bars.raw_full[slot], c, pa * kPage);
      }
      last_unit = u;
      publish(slot);
      ++u;
      return true;
    };
    auto load_s = [&](const Block& bb) -> bool {
      int pa, pb;
      valid_rows(p, bb, 0, &pa);
      valid_rows(p, bb, 1, &pb);
      for (int c = 0; c < kSUnits; ++c)
        if (!load(true, pa, pb, c * 64)) return false;
      return true;
    };
    auto load_v = [&](const Block& bb) -> bool {
      for (int q = 0; q < bb.npg; ++q) {
        int pa;
        valid_rows(p, bb, q, &pa);
        if (pa < 0 && lane == 0) latch_error(p.err, kErrBadPage);
        for (int mb = 0; mb < kVUnitsPerPage; ++mb)
          if (!load(false, pa, -1, 128 * mb)) return false;
      }
      return true;
    };
    while (ok && it.next(cur)) {
      while (ahead_n <= cur.j + kPrefetchBlocks && ahead.next(a)) {
        warm(a);
        ++ahead_n;
      }
      ok = load_s(cur);
      if (ok && have_prev) ok = load_v(prev);
      prev = cur;
      have_prev = true;
    }
    if (ok && have_prev) load_v(prev);
    // let every copy issued into this CTA's shared memory land before leaving: the last
    // kRawSlots units handed out are the only ones that can still be in flight (an earlier
    // unit's slot was reused, i.e. consumed); the skipped unit of the test hook was never
    // issued
    if (lane == 0)
      for (int v = max(0, last_unit - kRawSlots + 1); v <= last_unit; ++v)
        if (v != p.skip_unit) ptx::mbar_wait_drain(&bars.raw_full[v % kRawSlots], (v / kRawSlots) & 1);
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (ptx::elect_one()) {
      constexpr uint32_t kIdS = ptx::make_idesc(0, kKeys, NP, 0, 0);   // f16, A K-major, B K-major
      constexpr uint32_t kIdV = ptx::make_idesc(0, kKeys, NP, 1, 1);   // f16, A MN-major, B MN-major
      const uint32_t q0 = ptx::smem_u32(sm + L_::kOffQ);
      const uint32_t w0 = ptx::smem_u32(sm + L_::kOffWide);
      const uint32_t p0 = ptx::smem_u32(sm + L_::kOffP);
      int u = 0;
      bool ok = true;
      auto take = [&](uint32_t* addr) -> bool {
        const int slot = u % kWideSlots;
        if (!ptx::mbar_wait(&bars.wide_full[slot], (u / kWideSlots) & 1, abort_flag, p.err, lim)) return false;
        ptx::tc_fence_after();
        *addr = w0 + slot * kWideUnit;
        return true;
      };
      auto give = [&]() {
        ptx::mma_commit(&bars.wide_empty[u % kWideSlots]);
        ++u;
      };
      auto issue_s = [&](const Block& bb) -> bool {
        if (bb.first) {
          if (!ptx::mbar_wait(&bars.q_ready, bb.seg & 1, abort_flag, p.err, lim)) return false;
          ptx::tc_fence_after();
        }
        if (!ptx::mbar_wait(&bars.s_free[bb.j & 1], ((bb.j >> 1) & 1) ^ 1, abort_flag, p.err, lim)) return false;
        ptx::tc_fence_after();
        const uint32_t d = tmem + L_::kTmemS + (bb.j & 1) * NP;
        for (int c = 0; c < kSUnits; ++c) {
          uint32_t a;
          if (!take(&a)) return false;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_bf16_ss(d, ptx::sw128_desc(a + kk * 32, 16, 1024),
                             ptx::sw128_desc(q0 + c * L_::kQChunk + kk * 32, 16, 1024), kIdS,
                             (c | kk) != 0);
          give();
        }
        ptx::mma_commit(&bars.s_full[bb.j & 1]);
        if (bb.last) ptx::mma_commit(&bars.q_free);
        return true;
      };
      auto issue_v = [&](const Block& bb) -> bool {
        if (bb.first && bb.seg > 0) {
          // the previous segment's epilogue has read O'
          if (!ptx::mbar_wait(&bars.o_free, (bb.seg - 1) & 1, abort_flag, p.err, lim)) return false;
          ptx::tc_fence_after();
        }
        if (!ptx::mbar_wait(&bars.p_full[bb.j & 1], (bb.j >> 1) & 1, abort_flag, p.err, lim)) return false;
        ptx::tc_fence_after();
        const uint32_t pb = p0 + (bb.j & 1) * L_::kPBytes;
        for (int q = 0; q < bb.npg; ++q) {
          for (int mb = 0; mb < kVUnitsPerPage; ++mb) {
            uint32_t a;
            if (!take(&a)) return false;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_bf16_ss(tmem + L_::kTmemO + mb * NP, ptx::sw128_desc(a + kk * 2048, 8192, 1024),
                               ptx::smem_desc(pb + (64 * q + 16 * kk) * L_::kPRow, 16 * 64, 8 * L_::kPRow, L_::kPSwz),
                               kIdV, !(bb.first && q == 0 && kk == 0));
            give();
          }
        }
        ptx::mma_commit(&bars.p_free[bb.j & 1]);
        ptx::mma_commit(&bars.o_done);
        if (bb.last) ptx::mma_commit(&bars.seg_done);
        return true;
      };
      while (ok && it.next(cur)) {
        ok = issue_s(cur);
        if (ok && have_prev) ok = issue_v(prev);
        prev = cur;
        have_prev = true;
      }
      if (ok && have_prev) issue_v(prev);
      // every MMA issued here completes before the CTA frees its TMEM
      ptx::mma_commit(&bars.drain);
      ptx::mbar_wait_drain(&bars.drain, 0);
    }
  } else if (warp < 6) {
    // -------------------------------------------------------------- widening (and Q)
    const int wl = warp - 2;           // 0..3
    int u = 0;
    bool ok = true;
    // Q of sequence `seq`: per row a power-of-two scale 2^e with the row's largest magnitude
    // in [2^14, 2^15), written as f16 into the 128B-swizzled operand; the row's score scale
    // scale * log2(e) * 2^-e goes to qsc[parity]
    auto prep_q = [&](int seq, int parity) {
      for (int r = wl; r < TQ; r += 4) {
        const uint16_t* ql = p.q_latent + ((size_t)seq * TH + r) * kDl + 16 * lane;
        const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(ql));
        const uint4 a1 = __ldg(reinterpret_cast<const uint4*>(ql) + 1);
        const uint32_t rp = __ldg(reinterpret_cast<const uint32_t*>(p.q_rope + ((size_t)seq * TH + r) * 64) + lane);
        const uint32_t w[9] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w, rp};
        float x[18];
#pragma unroll
        for (int i = 0; i < 9; ++i) {
          x[2 * i] = __uint_as_float(w[i] << 16);
          x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 18; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const int E = (int)((__float_as_uint(amax) >> 23) & 0xFF);
        const int e = amax > 0.f ? max(-100, min(100, 141 - E)) : 0;  // 2^e * amax in [2^14, 2^15)
        const float f1 = __uint_as_float((uint32_t)(127 + e / 2) << 23);
        const float f2 = __uint_as_float((uint32_t)(127 + (e - e / 2)) << 23);
        uint32_t h[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) h[i] = ptx::pack_f16x2(x[2 * i] * f1 * f2, x[2 * i + 1] * f1 * f2);
        unsigned char* row = sm + L_::kOffQ + (lane >> 2) * L_::kQChunk + r * 128;
        const int g0 = (lane & 3) * 2;
        *reinterpret_cast<uint4*>(row + ((g0 ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(row + (((g0 + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
        *reinterpret_cast<uint32_t*>(sm + L_::kOffQ + 8 * L_::kQChunk + r * 128 +
                                     (((lane >> 2) ^ (r & 7)) << 4) + (lane & 3) * 4) = h[8];
        if (lane == 0) bars.qsc[parity][r] = p.scale_log2 * __uint_as_float((uint32_t)(127 - e) << 23);
      }
    };
    // One unit, converted by one warp (unit u by widening warp u mod 4, so four units are in
    // conversion at once): 512 granules of 16 fp8 codes, 16 per lane, each to 16 f16 in two
    // 128B-swizzled 16-byte chunks.  Score units: granule G = row (key) G >> 2, codes
    // 16 (G & 3).. of the unit's 64 columns, raw rows of page (row >> 6) at 4 KB each.  Value
    // units: row G >> 3, codes 16 (G & 7).. of the 128 latent columns; the f16 tile holds
    // latent 0-63 and 64-127 of the unit as two 8 KB halves.  Raw reads are 512 contiguous
    // bytes per warp instruction.
    auto widen = [&](bool score, int v0, int v1) -> bool {
      const int mine = (u & 3) == wl;
      const int rs = u % kRawSlots, ws = u % kWideSlots;
      if (mine) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bars.raw_issued[rs], (u / kRawSlots) & 1, abort_flag, p.err, lim)))
          return false;
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bars.raw_full[rs], (u / kRawSlots) & 1, abort_flag, p.err, lim)))
          return false;
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bars.wide_empty[ws], ((u / kWideSlots) & 1) ^ 1, abort_flag, p.err, lim)))
          return false;
        const unsigned char* raw = sm + L_::kOffRaw + rs * kRawUnit;
        unsigned char* wide = sm + L_::kOffWide + ws * kWideUnit;
#pragma unroll 1
        for (int i0 = 0; i0 < 16; i0 += 4) {
          uint4 g[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int G = lane + 32 * (i0 + i);
            const int row = score ? G >> 2 : G >> 3;
            const bool live = score ? (row & 63) < (row >> 6 ? v1 : v0) : row < v0;
            g[i] = live ? *reinterpret_cast<const uint4*>(raw + 16 * G) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int G = lane + 32 * (i0 + i);
            const int row = score ? G >> 2 : G >> 3;
            const int h = G & 3;
            const int base = score ? row * 128 : ((G >> 2) & 1) * 8192 + row * 128;
            const uint32_t c[4] = {g[i].x, g[i].y, g[i].z, g[i].w};
            uint32_t o[8];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              ptx::e4m3x4_to_f16x2x2(c[x], o[2 * x], o[2 * x + 1]);
            }
            *reinterpret_cast<uint4*>(wide + base + (((2 * h) ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(wide + base + (((2 * h + 1) ^ (row & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars.raw_empty[rs]);
        ptx::fence_proxy_async();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars.wide_full[ws]);
      }
      ++u;
      return true;
    };
    auto widen_s = [&](const Block& bb) -> bool {
      int ph;
      const int v0 = valid_rows(p, bb, 0, &ph), v1 = valid_rows(p, bb, 1, &ph);
      for (int c = 0; c < kSUnits; ++c)
        if (!widen(true, v0, v1)) return false;
      return true;
    };
    auto widen_v = [&](const Block& bb) -> bool {
      for (int q = 0; q < bb.npg; ++q) {
        int ph;
        const int v = valid_rows(p, bb, q, &ph);
        for (int mb = 0; mb < kVUnitsPerPage; ++mb)
          if (!widen(false, v, 0)) return false;
      }
      return true;
    };
    while (ok && it.next(cur)) {
      if (cur.first) {
        // the previous segment's scores are done with Q, and the softmax has taken the
        // score scales written two segments ago
        if (cur.seg > 0 &&
            !(ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.q_free, (cur.seg - 1) & 1, abort_flag, p.err, lim))))
          break;
        if (cur.seg > 1 &&
            !(ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.qsc_free[cur.seg & 1], ((cur.seg >> 1) - 1) & 1,
                                                         abort_flag, p.err, lim))))
          break;
        prep_q(cur.seq, cur.seg & 1);
        ptx::fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&bars.q_ready);
          ptx::mbar_arrive(&bars.qsc_full[cur.seg & 1]);
        }
      }
      ok = widen_s(cur);
      if (ok && have_prev) ok = widen_v(prev);
      prev = cur;
      have_prev = true;
    }
    if (ok && have_prev) widen_v(prev);
  } else {
    // -------------------------------------------------------------- softmax / epilogue / merge
    const int kq = 32 * (warp & 3) + lane;  // key of the block == TMEM lane == latent row in a block of O'
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int st = threadIdx.x - 192;       // 0..127
    bool ok = true;
    // this thread's part of the row sums (over the keys it has seen) lives in TMEM columns
    // [kTmemL, kTmemL + NP) of its lane
    const uint32_t lp_addr = tmem + lane_off + L_::kTmemL;
    auto lp_ld = [&](int c, uint32_t (&v)[16]) { ptx::tmem_ld16(lp_addr + c, v); };
    auto lp_st = [&](int c, const uint32_t (&v)[16]) { ptx::tmem_st16(lp_addr + c, v); };
    // the rows' references, the same in every softmax thread, live in registers; the rows' score
    // scales are read once per block as 16-byte vectors (the shared-memory queue is busy with
    // the widening, so few and independent loads)
    float m[NP];
    // Group barrier of the four softmax warps on an mbarrier (bounded wait, so that a warp that
    // gave up cannot leave the others waiting forever).  Every warp passes the same sequence of
    // barriers, so the phase of barrier number n is n & 1.
    uint32_t n_sync = 0;
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars.soft_sync);
      const bool r = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.soft_sync, n_sync & 1, abort_flag, p.err, lim));
      ++n_sync;
      return r;
    };
    // sequences with no cached key are in no work unit's range: unit u writes O = 0 and
    // LSE = -inf for the empty sequences u, u + G, u + 2G, ...
    for (int b = unit; b < p.B; b += p.G) {
      if (clamp_len(__ldg(p.cache_lens + b), p.max_pages) > 0) continue;
      uint4* o = reinterpret_cast<uint4*>(p.out + (size_t)b * TH * kDl);
      for (int i = st; i < TH * (kDl / 8); i += 128)
        if (MLA_STORE_OK(o + i, p.out, p.out_bytes, p.err)) o[i] = make_uint4(0, 0, 0, 0);
      for (int i = st; i < TH; i += 128) {
        float* lp = p.lse + ((size_t)b * p.H + i % p.H) * p.T + i / p.H;
        if (MLA_STORE_OK(lp, p.lse, p.lse_bytes, p.err)) *lp = -INFINITY;
      }
    }
    // key scales one block ahead (the iterator already holds the next block and its pages)
    auto fetch_ks = [&](const Block& bb) -> float {
      const int q = kq >> 6, r = kq & 63;
      int ph;
      const int v = valid_rows(p, bb, q, &ph);
      return r < v ? __ldg(p.kv_scale + (size_t)ph * kPage + r) : 0.f;
    };
    float ks_next = it.has ? fetch_ks(it.nxt) : 0.f;
    int n_epi = 0;
    while (ok && it.next(cur)) {
      const float ks_raw = ks_next;
      if (it.has) ks_next = fetch_ks(it.nxt);
      if (cur.first) {
        if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.qsc_full[cur.seg & 1], (cur.seg >> 1) & 1,
                                                          abort_flag, p.err, lim))))
          break;
#pragma unroll
        for (int q = 0; q < NP; ++q) m[q] = -INFINITY;
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
        for (int c = 0; c < NP; c += 16) lp_st(c, z);
        ptx::tmem_st_wait();
      }
      // this thread's key; a zero scale is raised to 2^-64 (its key and value are then ~0 but
      // its probability still counts in the row sum)
      const int half = kq >> 6, r64 = kq & 63;
      int ph;
      const bool valid = r64 < valid_rows(p, cur, half, &ph);
      const int key = (cur.pg0 + half) * kPage + r64;
      const float ks = fmaxf(ks_raw, 5.421010862427522e-20f);
      const float lks = __log2f(ks), inv_ks = 1.f / ks;
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.s_full[cur.j & 1], (cur.j >> 1) & 1, abort_flag, p.err, lim))))
        break;
      ptx::tc_fence_after();
      float u[NP];
      {
        uint32_t sv[NP];
        if constexpr (NP == 32)
          ptx::tmem_ld32(tmem + lane_off + L_::kTmemS + (cur.j & 1) * NP, sv);
        else
          ptx::tmem_ld16(tmem + lane_off + L_::kTmemS + (cur.j & 1) * NP, sv);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < NP; ++q) u[q] = __uint_as_float(sv[q]);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars.s_free[cur.j & 1]);
      // u = t + log2(ks) with t = scale * ks * s (the log2-domain score); invisible keys and
      // padding rows -inf
      const int vis_all = p.causal ? cur.L - p.T : cur.L - 1;  // keys <= this are seen by every row
      float qs[NP];
#pragma unroll
      for (int q = 0; q < NP; q += 4) {
        const float4 v = *reinterpret_cast<const float4*>(&bars.qsc[cur.seg & 1][q]);
        qs[q] = v.x;
        qs[q + 1] = v.y;
        qs[q + 2] = v.z;
        qs[q + 3] = v.w;
      }
      // Row q is (token q / H, head q % H) and sees the key iff key <= L - T + q / H (causal),
      // i.e. iff q >= H (key - (L - T)): the rows that see this key are q_lo .. TQ - 1, found
      // with one multiply (no division or branch in the loop below)
      int q_lo = 0;
      if (key > vis_all) q_lo = p.causal ? p.H * (key - (cur.L - p.T)) : NP;
      if (!valid) q_lo = NP;
      // (the first block of a segment always sets the references; the old ones are stale)
      bool grow = cur.first;
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        const bool see = q >= q_lo && q < TQ;
        const float x = see ? fmaf(u[q], qs[q] * ks, lks) : -INFINITY;
        u[q] = x;
        grow |= x > m[q] + kTau;
      }
      // does any key of the block exceed its row's reference by more than 2^kTau?
      const unsigned wv = __ballot_sync(0xffffffffu, grow);
      if (lane == 0) bars.vote[n_sync & 1][warp & 3] = wv != 0;
      if (!(ok = group_sync())) break;
      const int* vt = bars.vote[(n_sync - 1) & 1];
      if (vt[0] | vt[1] | vt[2] | vt[3]) {
        // new references: the column maxima over the block's keys (a warp maximum per column
        // on an integer image of the float that preserves its order)
        float wmax = -INFINITY;
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          const int b = __float_as_int(u[q]);
          const int r = __reduce_max_sync(0xffffffffu, b >= 0 ? b : b ^ 0x7FFFFFFF);
          if (lane == q) wmax = __int_as_float(r >= 0 ? r : r ^ 0x7FFFFFFF);
        }
        if (lane < NP) bars.red[warp & 3][lane] = wmax;
        if (!(ok = group_sync())) break;
        if (st < NP)
          bars.colv[st] = fmaxf(fmaxf(bars.red[0][st], bars.red[1][st]), fmaxf(bars.red[2][st], bars.red[3][st]));
        if (!(ok = group_sync())) break;
        // new references; the rescale factors go to shared memory (read by the O' rescale)
        bool shrink = false;
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          const float mn = fmaxf(m[q], bars.colv[q]);
          const float al = (m[q] == -INFINITY || mn == -INFINITY) ? 1.f : ptx::ex2(m[q] - mn);
          shrink = shrink || al != 1.f;
          if (st == q) bars.alpha[q] = al;
          m[q] = mn;
        }
        const float* alpha = bars.alpha;
        if (!cur.first && shrink) {
          // O' holds the contributions of this segment's earlier blocks (PV(j-1) included):
          // scale its columns, and the row sums, to the new references (16 columns at a time:
          // the scores stay live in registers meanwhile)
          if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.o_done, (cur.j - 1) & 1, abort_flag, p.err, lim))))
            break;
          ptx::tc_fence_after();
#pragma unroll 1
          for (int c1 = 0; c1 < 5 * NP; c1 += 16) {
            uint32_t ov[16];
            const int c0 = c1 < 4 * NP ? c1 : L_::kTmemL + (c1 - 4 * NP);  // O' blocks, then the sums
            const uint32_t oa = tmem + lane_off + L_::kTmemO + c0;
            ptx::tmem_ld16(oa, ov);
            ptx::tmem_ld_wait();
            const float* al = alpha + (c0 % NP);
#pragma unroll
            for (int q = 0; q < 16; ++q) ov[q] = __float_as_uint(__uint_as_float(ov[q]) * al[q]);
            ptx::tmem_st16(oa, ov);
          }
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
        }
      }
      // P'' = exp2(u - m) (f16, <= 2^kTau), and the row sums of P'' / ks = exp2(t - m)
      uint32_t pk[NP / 2];
#pragma unroll
      for (int c = 0; c < NP; c += 16) {
        uint32_t lv[16];
        lp_ld(c, lv);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int q = c; q < c + 16; q += 2) {
          const float a = ptx::ex2(u[q] - (m[q] == -INFINITY ? 0.f : m[q]));
          const float b = ptx::ex2(u[q + 1] - (m[q + 1] == -INFINITY ? 0.f : m[q + 1]));
          lv[q - c] = __float_as_uint(fmaf(a, inv_ks, __uint_as_float(lv[q - c])));
          lv[q + 1 - c] = __float_as_uint(fmaf(b, inv_ks, __uint_as_float(lv[q + 1 - c])));
          pk[q / 2] = ptx::pack_f16x2(a, b);
        }
        lp_st(c, lv);
      }
      ptx::tmem_st_wait();
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.p_free[cur.j & 1], ((cur.j >> 1) & 1) ^ 1, abort_flag, p.err, lim))))
        break;
      {
        unsigned char* prow = sm + L_::kOffP + (cur.j & 1) * L_::kPBytes + kq * L_::kPRow;
#pragma unroll
        for (int g = 0; g < NP / 8; ++g) {
          const int sw = NP == 32 ? (g ^ ((kq >> 1) & 3)) : (g ^ ((kq >> 2) & 1));
          *reinterpret_cast<uint4*>(prow + sw * 16) = make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        }
      }
      ptx::fence_proxy_async();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars.p_full[cur.j & 1]);
      if (!cur.last) continue;
      if (lane == 0) ptx::mbar_arrive(&bars.qsc_free[cur.seg & 1]);  // done with this segment's qsc

      // ---------------- epilogue of the segment: O = O' / l for rows q < TQ
      if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.seg_done, n_epi & 1, abort_flag, p.err, lim)))) break;
      ++n_epi;
      ptx::tc_fence_after();
      {
        float lp[NP];
#pragma unroll
        for (int c = 0; c < NP; c += 16) {
          uint32_t lv[16];
          lp_ld(c, lv);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) lp[c + i] = __uint_as_float(lv[i]);
        }
        const float wsum = warp_column_sums<NP>(lp);
        if (lane < NP) bars.red[warp & 3][lane] = wsum;
      }
      if (!(ok = group_sync())) break;
      if (st < NP) {
        const float l = (bars.red[0][st] + bars.red[1][st]) + (bars.red[2][st] + bars.red[3][st]);
        bars.colv[st] = l;
        bars.winv[st] = l > 0.f ? 1.f / l : 0.f;
      }
      if (!(ok = group_sync())) break;
      const float* inv = bars.winv;
      const int n_pages = pages_of(cur.L, kPage);
      const bool whole = cur.lo == 0 && cur.hi == n_pages;  // no other unit has keys of it
      const size_t slot = (size_t)unit + cur.seq;
#pragma unroll 1
      for (int mb = 0; mb < 4; ++mb) {
        uint32_t ov[NP];
        const uint32_t oa = tmem + lane_off + L_::kTmemO + mb * NP;
        if constexpr (NP == 32) ptx::tmem_ld32(oa, ov); else ptx::tmem_ld16(oa, ov);
        ptx::tmem_ld_wait();
        const int col = 128 * mb + kq;  // latent column
        if (whole) {
          __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)cur.seq * TH * kDl + col;
#pragma unroll
          for (int q = 0; q < NP; ++q)
            if (q < TQ && MLA_STORE_OK(o + (size_t)q * kDl, p.out, p.out_bytes, p.err))
              o[(size_t)q * kDl] = __float2bfloat16_rn(__uint_as_float(ov[q]) * inv[q]);
        } else {
          float* o = p.part_o + slot * TQ * kDl + col;
#pragma unroll
          for (int q = 0; q < NP; ++q)
            if (q < TQ && MLA_STORE_OK(o + (size_t)q * kDl, p.part_o, p.part_o_bytes, p.err))
              o[(size_t)q * kDl] = __uint_as_float(ov[q]) * inv[q];
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars.o_free);  // O' may be overwritten
      if (st < TQ) {
        float mq = 0.f;
#pragma unroll
        for (int q = 0; q < NP; ++q) mq = q == st ? m[q] : mq;
        const float l = bars.colv[st];
        const float ls = l > 0.f ? (mq + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        float* lp = p.lse + ((size_t)cur.seq * p.H + st % p.H) * p.T + st / p.H;
        float* plp = p.part_lse + slot * TQ + st;
        if (whole) {
          if (MLA_STORE_OK(lp, p.lse, p.lse_bytes, p.err)) *lp = ls;
        } else if (MLA_STORE_OK(plp, p.part_lse, p.part_lse_bytes, p.err)) {
          *plp = ls;
        }
      }
      if (whole) continue;
      // Merge by the last split to finish: the units that covered this sequence wrote their
      // partials into slots c + seq, c_first <= c <= c_last; each makes its stores visible and
      // counts itself in, and the one that completes the count merges them.
      __threadfence();
      if (!(ok = group_sync())) break;
      const int c_first = cur.flat0 / bars.plan.chunk;
      const int nsplit = (cur.flat0 + n_pages - 1) / bars.plan.chunk - c_first + 1;
      if (st == 0) {
        asm volatile("griddepcontrol.wait;" ::: "memory");  // counters zeroed by the kernel ahead
        __threadfence();
        int* cnt = p.counters + cur.seq;
        const int done = MLA_STORE_OK(cnt, p.counters, p.counters_bytes, p.err) ? atomicAdd(cnt, 1) + 1 : 0;
        __threadfence();
        bars.merge_last = done == nsplit ? 1 : 0;
      }
      if (!(ok = group_sync())) break;
      if (!*reinterpret_cast<volatile int*>(&bars.merge_last)) continue;
      // row statistics of the splits: maximum LSE and the inverse weight sum, and the merged LSE
      const float* lsp = p.part_lse + ((size_t)c_first + cur.seq) * TQ;
      if (st < TQ) {
        float mx = -INFINITY;
#pragma unroll 4
        for (int k = 0; k < nsplit; ++k) mx = fmaxf(mx, ptx::ld_l2(lsp + (size_t)k * TQ + st));
        float ws = 0.f;
#pragma unroll 4
        for (int k = 0; k < nsplit; ++k) {
          const float ls = ptx::ld_l2(lsp + (size_t)k * TQ + st);
          ws += (mx == -INFINITY || ls == -INFINITY) ? 0.f : __expf(ls - mx);
        }
        bars.mx[st] = mx;
        bars.winv[st] = ws > 0.f ? 1.f / ws : 0.f;
        float* lp = p.lse + ((size_t)cur.seq * p.H + st % p.H) * p.T + st / p.H;
        if (MLA_STORE_OK(lp, p.lse, p.lse_bytes, p.err)) *lp = ws > 0.f ? mx + logf(ws) : -INFINITY;
      }
      if (!(ok = group_sync())) break;
      // thread st: latent quad st (columns 4 st .. 4 st + 3) of every row, four rows and two
      // splits per round: eight independent 16-byte loads in flight
      const float4* src = reinterpret_cast<const float4*>(p.part_o) + ((size_t)c_first + cur.seq) * TQ * (kDl / 4) + st;
      const size_t sstride = (size_t)TQ * (kDl / 4);
#pragma unroll 1
      for (int q0 = 0; q0 < TQ; q0 += 4) {
        float4 acc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int k = 0; k < nsplit; k += 2) {
          const bool two = k + 1 < nsplit;
          float l0[4], l1[4];
          float4 x0[4], x1[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int q = min(q0 + i, TQ - 1);
            l0[i] = ptx::ld_l2(lsp + (size_t)k * TQ + q);
            x0[i] = ptx::ld_l2(src + (size_t)k * sstride + (size_t)q * (kDl / 4));
            l1[i] = two ? ptx::ld_l2(lsp + (size_t)(k + 1) * TQ + q) : -INFINITY;
            x1[i] = two ? ptx::ld_l2(src + (size_t)(k + 1) * sstride + (size_t)q * (kDl / 4))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int q = min(q0 + i, TQ - 1);
            const float mx = bars.mx[q], wi = bars.winv[q];
            const float w0 = (mx == -INFINITY || l0[i] == -INFINITY) ? 0.f : __expf(l0[i] - mx) * wi;
            const float w1 = (mx == -INFINITY || l1[i] == -INFINITY) ? 0.f : __expf(l1[i] - mx) * wi;
            acc[i].x += w0 * x0[i].x + w1 * x1[i].x;
            acc[i].y += w0 * x0[i].y + w1 * x1[i].y;
            acc[i].z += w0 * x0[i].z + w1 * x1[i].z;
            acc[i].w += w0 * x0[i].w + w1 * x1[i].w;
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint2* od = reinterpret_cast<uint2*>(p.out + ((size_t)cur.seq * TH + q0 + i) * kDl + 4 * st);
          if (q0 + i < TQ && MLA_STORE_OK(od, p.out, p.out_bytes, p.err))
            *od = make_uint2(ptx::pack_bf16x2(acc[i].x, acc[i].y), ptx::pack_bf16x2(acc[i].z, acc[i].w));
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L_::kTmemCols);
  }
}

// Zeroes the per-sequence split counters of a call; the decode kernel is launched behind it as
// a programmatic dependent and waits for it only where it first touches a counter.
__global__ void __launch_bounds__(256) zero_counters_t_kernel(int* __restrict__ c, int n) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) c[i] = 0;
}

}  // namespace sm103_decode_t

// ---------------------------------------------------------------- host side

cudaError_t encode_tensor_map_swz(CUtensorMap* map, CUtensorMapDataType dt, int rank,
                                  const void* ptr, const uint64_t* dims, const uint64_t* strides,
                                  const uint32_t* box, bool swizzle128);

// Makes the driver load the transposed decode kernels on the current device.
cudaError_t load_decode_t_kernels() {
  using namespace sm103_decode_t;
  cudaFuncAttributes fa;
  cudaError_t e;
  if ((e = cudaFuncGetAttributes(&fa, decode_t_kernel<16>)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, decode_t_kernel<32>)) != cudaSuccess) return e;
  return cudaFuncGetAttributes(&fa, zero_counters_t_kernel);
}

cudaError_t launch_decode_t_sm103(const void* q_latent, const void* q_rope, const void* kv_cache,
                                  const float* kv_scale, const int* page_table,
                                  const int* cache_lens, int B, int H, int T, int max_pages,
                                  int num_pages, float softmax_scale, int causal, float* part_o,
                                  float* part_lse, int* counters, void* out, float* lse, int G,
                                  unsigned int* err, long long wait_limit, int skip_unit,
                                  cudaStream_t stream) {
  using namespace sm103_decode_t;
  const int TQ = T * H;
  if (TQ < 1 || TQ > 32) return cudaErrorInvalidValue;
  CUtensorMap tm_s, tm_v;
  // the cache as a 2-D byte tensor [num_pages * 64 rows, 576 columns]: boxes of 64 columns x
  // 64 rows for the score units, 128 x 64 for the value units
  uint64_t dims[2] = {(uint64_t)kDc, (uint64_t)num_pages * kPage};
  uint64_t strides[1] = {(uint64_t)kDc};
  uint32_t box[2] = {64, kPage};
  cudaError_t e = encode_tensor_map_swz(&tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, kv_cache, dims,
                                        strides, box, /*swizzle128=*/false);
  if (e != cudaSuccess) return e;
  box[0] = 128;
  e = encode_tensor_map_swz(&tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, kv_cache, dims, strides, box,
                            /*swizzle128=*/false);
  if (e != cudaSuccess) return e;
  Params p;
  p.q_latent = static_cast<const uint16_t*>(q_latent);
  p.q_rope = static_cast<const uint16_t*>(q_rope);
  p.kv_cache = static_cast<const uint8_t*>(kv_cache);
  p.kv_scale = kv_scale;
  p.page_table = page_table;
  p.cache_lens = cache_lens;
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.counters = counters;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.err = err;
  p.B = B;
  p.H = H;
  p.T = T;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.causal = causal;
  p.G = G;
  p.NQT = 1;
  p.TQ = TQ;
  p.n_slots = G + B;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.wait_limit = wait_limit;
  p.skip_unit = skip_unit;
  // an item (its Q preparation, epilogue and merge) costs this kernel about three pages
  p.item_cost = 3;
  const size_t out_full = (size_t)B * T * H * kDl * 2;
  p.out_bytes = out_full - std::min(out_full, testing_out_shrink());
  p.lse_bytes = (size_t)B * H * T * sizeof(float);
  p.part_o_bytes = (size_t)(reinterpret_cast<char*>(part_lse) - reinterpret_cast<char*>(part_o));
  p.part_lse_bytes = (size_t)(reinterpret_cast<char*>(counters) - reinterpret_cast<char*>(part_lse));
  p.counters_bytes = (size_t)B * sizeof(int);
  const int zero_blocks = std::min((B + 2047) / 2048, 1024);
  zero_counters_t_kernel<<<zero_blocks, 256, 0, stream>>>(counters, B);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto go = [&](auto kern, int smem) -> cudaError_t {
    static unsigned long long smem_set[2] = {0, 0};
    const cudaError_t e2 = smem_attr_once(kern, smem, &smem_set[smem == Lay<32>::kSmemAlloc ? 1 : 0]);
    if (e2 != cudaSuccess) return e2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tm_s, tm_v, p);
  };
  return TQ <= 16 ? go(decode_t_kernel<16>, Lay<16>::kSmemAlloc) : go(decode_t_kernel<32>, Lay<32>::kSmemAlloc);
}

}  // namespace mla
