// Absorbed MLA decode over the paged latent cache on tcgen05 / TMEM: split-KV, with the
// log-sum-exp merge of the splits done by the last split of each sequence to finish.
//
// Each work unit (a contiguous range of pages from the split plan) is served by a pair
// of CTAs that differ only in which half of the 512 latent output columns they own:
// O (128 query rows x 512 fp32) is exactly the 512-column TMEM, so one CTA cannot also
// hold the scores.  Both CTAs of a pair compute the full scores S = Q C' (the redundant
// part) and their own half of O += P C[:, half].  Query rows are the (token, head) pairs
// of one sequence, padded to the MMA's M = 128.
//
// Per CTA (8 warps; 12 with the fp8 cache):
//   warp 0      TMA producer: each sequence's Q latent 0..255 (staged in shared memory),
//               then the cache pages (64 keys x 576 columns) -- bf16: in two parts, the
//               five score-only 64-column chunks and the CTA's four value chunks, 128B-
//               swizzled, ready for the MMA; fp8: the whole raw page into the upper half of
//               a stage -- plus L2 prefetch of pages ahead
//   warp 1      MMA issuer: at a sequence change, copies the staged Q latent 0..255 into
//               TMEM (tcgen05.cp) and loads latent 256..511 + rope into shared memory by TMA;
//               then S(g) = Q C(g)' into one of two S buffers (A operand = Q: latent 0..255
//               from TMEM, the rest from shared memory), and O_half += P(g) C(g)[:, half]
//               with P read from TMEM.  S(g+1) and PV(g) are issued in whichever order their
//               inputs arrive.
//   warps 2-3   stage preparation: zero the rows past the sequence end of a partial page;
//   (+ 8-11)    fp8: widen the page to bf16 in place (three lockstep steps of three
//               64-column chunks, 16-byte granules spread over the preparation threads;
//               warps 8-11 exist in the fp8 kernel only, and softmax warps whose 32 rows
//               are all padding of the M = 128 MMA join them) and stage its scales
//   warps 4-7   softmax, one thread per query row; they also write the split's partial
//               (O_half / l, log-sum-exp), column quads of 32 rows per 512-byte store, and,
//               in the CTA that completes a (sequence, column half), merge its splits into
//               the bf16 output and the LSE
// TMEM columns: [0,128) Q latent 0..255 (bf16 pairs), [128,256) two S / P buffers of 64,
// [256,512) O half.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "decode_plan.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace sm103_decode {

using decode_plan::Plan;
using decode_plan::Segments;
using decode_plan::clamp_len;
using decode_plan::make_plan;
constexpr int kPage = decode_plan::kPage;
constexpr int kDl = 512, kDc = 576, kRows = 128;
constexpr int kPageChunk = kPage * 128;       // 64 rows x 64 bf16 (8 KB), 128B-swizzled
constexpr int kStageBytes = 9 * kPageChunk;   // 72 KB
constexpr int kRawChunk = kPage * 64;         // 64 rows x 64 fp8 bytes (4 KB), unswizzled
constexpr int kRawOffset = 9 * kRawChunk;     // fp8 page lands in the upper 36 KB of a stage
constexpr int kStages = 2;
constexpr int kQChunk = kRows * 128;          // 128 rows x 64 bf16 (16 KB)
constexpr int kOffQhi = 0;                    // latent 256..511 (4 chunks) + rope (1 chunk)
constexpr int kOffStage = 5 * kQChunk;        // 80 KB
constexpr int kSmemBytes = kOffStage + kStages * kStageBytes;  // 224 KB
// bf16 pages arrive in two parts: the score-only chunks (the other column half's four latent
// chunks and the rope chunk, 40 KB) into one slot, free again once the score MMAs that read
// them are done, and this CTA's own four latent chunks (32 KB), which the PV product reads
// too, into a ring of three, so that they land two pages ahead of their use.
constexpr int kSPartBytes = 5 * kPageChunk;
constexpr int kVPartBytes = 4 * kPageChunk;
constexpr int kVSlots = 3;
constexpr int kOffSPart = kOffStage;
constexpr int kOffVPart = kOffStage + kSPartBytes;
static_assert(kOffVPart + kVSlots * kVPartBytes <= kSmemBytes, "bf16 page parts fit the stages");
// position of 64-column chunk c (0..8) within its part, for column half `half`: the value
// chunks 4 half .. 4 half + 3 in order; the score-only ones (half 0: 4..8, half 1: 0..3, 8)
__host__ __device__ constexpr int chunk_idx(int c, int half) {
  return ((c >> 2) == half && c < 8) ? c - 4 * half : (half == 0 ? c - 4 : (c < 4 ? c : 4));
}
constexpr int kSmemAlloc = kSmemBytes + 1024;
// bf16: 8 warps; fp8: 12 (four more page-widening warps)
template <bool kFp8> constexpr int kThreadsOf = kFp8 ? 384 : 256;
template <bool kFp8> constexpr int kPrepOf = kFp8 ? 192 : 64;
constexpr int kPrefetchAhead = 4;             // pages warmed in L2 ahead of their load

struct Params {
  const uint16_t* q_latent;  // [B, T, H, 512]
  const uint16_t* q_rope;    // [B, T, H, 64]
  const float* kv_scale;     // [num_pages, 64] (fp8 path)
  const unsigned char* cache_bytes;  // the cache as bytes: page g at g * 64 * 576 * element size
  const int* page_table;
  const int* cache_lens;
  float* part_o;
  float* part_lse;   // [2][n_slots][TQ]: each column half writes its own copy
  int* counters;     // [B * NQT][2]: finished splits per (virtual sequence, half), zeroed per call
  uint16_t* out;     // [B, T, H, 512] bf16
  float* lse;        // [B, H, T]
  unsigned int* err;
  int B, H, T, max_pages, num_pages, causal, G;
  int NQT, TQ;  // query tiles per sequence (T*H rows in tiles of 128) and rows per tile
  int n_slots;  // partial slots: G + B * NQT
  float scale_log2;
  int page_box;  // 1: a page is one box of the 3-D cache map (else nine boxes of the 2-D one)
  int item_cost;  // flat pages the split plan charges per work item (see decode_plan.cuh)
  // buffer sizes for the store checks of the bounds-checked build
  size_t out_bytes, lse_bytes, part_o_bytes, part_lse_bytes, counters_bytes;
};

struct Bars {
  // stage_ready[s][k]: bf16 pages are ready at once (k = 0); fp8 pages in three parts, k = 0..2
  // covering 64-column chunks 3k..3k+2, as the in-place widening completes them
  uint64_t stage_full[kStages], stage_ready[kStages][3], stage_empty[kStages];
  // bf16 page parts: the score-only slot and the ring of this half's value chunks; a page
  // that ends a sequence part-way is handed to the preparation warps (zero_go) and back once
  // the rows past the end are zeroed (zeroed), one phase each per such page
  uint64_t spart_full, spart_empty;
  uint64_t vpart_full[kVSlots], vpart_empty[kVSlots];
  uint64_t zero_go, zeroed;
  uint64_t s_full[2], p_full[2], o_done, seg_done, conv_sync;
  uint64_t q_free, q_lo_full, q_cp_done, q_hi_full;  // per-sequence Q staging
  uint64_t q0_copied;  // the first sequence's staged Q is in TMEM (one phase per launch)
  uint64_t part_done, merge_go;  // partial written by the 4 softmax warps / merge decision
  uint64_t dec_go;               // the segment's merge path decided
  uint64_t merge_full;           // the other split's partial copied into shared memory
  int merge_last, merge_fast, merge_bulk;
  uint32_t tmem_base;
  int abort_flag;
  Plan plan;
  float kscale[kStages][kPage];
};

__device__ __forceinline__ int page_of(const Params& p, int vseq, int pg) {
  return __ldg(p.page_table + (size_t)(vseq / p.NQT) * p.max_pages + pg);
}
__device__ __forceinline__ int row_of_page(const Params& p, int page) {
  // an out-of-range page reads as zeros (coordinates outside the tensor) and is masked
  return (page >= 0 && page < p.num_pages) ? page * kPage : -2 * kPage;
}
__device__ __forceinline__ int page_row(const Params& p, int vseq, int pg) {
  return row_of_page(p, page_of(p, vseq, pg));
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreadsOf<kFp8>, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_cache,
                        const __grid_constant__ CUtensorMap tm_page,
                        const __grid_constant__ CUtensorMap tm_c4,
                        const __grid_constant__ CUtensorMap tm_c5,
                        const __grid_constant__ CUtensorMap tm_qlat,
                        const __grid_constant__ CUtensorMap tm_qrope, const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ Bars bars;
  constexpr int kThreads = kThreadsOf<kFp8>;
  // fp8: with fewer than 128 query rows per tile, softmax warps whose 32 rows are all padding
  // of the M = 128 MMA (never stored) widen pages instead: warps 4 .. 4 + n_soft - 1 run the
  // softmax, warps 4 + n_soft .. 7 join the preparation warps (2-3 and 8-11)
  const int n_soft = kFp8 ? (p.TQ + 31) / 32 : kRows / 32;
  const int n_prep = kPrepOf<kFp8> + (kFp8 ? 32 * (kRows / 32 - n_soft) : 0);
  // readiness parts of a page stage: fp8 three groups of three widened chunks; bf16 the
  // score-only part, then the value part
  constexpr int kParts = kFp8 ? 3 : 2;
  // the first sequence's Q latent 0..255 (four 16 KB chunks) is staged where pages 1 (fp8)
  // or 1 and 2 (bf16: value slots 1 and 2) land
  auto q_stage_off = [&](int c) -> int {
    if constexpr (kFp8) return kOffStage + kStageBytes + c * kQChunk;
    return kOffVPart + (1 + (c >> 1)) * kVPartBytes + (c & 1) * kQChunk;
  };
  const int warp = threadIdx.x >> 5;
  const int unit = blockIdx.x >> 1, half = blockIdx.x & 1;
  const int TH = p.T * p.H, TQ = p.TQ;
  // first Q row of virtual sequence v: its sequence's rows, then 128 per query tile
  auto q_row0 = [&](int v) { return (v / p.NQT) * TH + (v % p.NQT) * kRows; };

  if (threadIdx.x == 0) {
    // the descriptors are fetched while the barriers are set up and the plan is made: a TMA
    // instruction whose map is not cached waits for that fetch
    ptx::prefetch_tensormap(&tm_qlat);
    ptx::prefetch_tensormap(&tm_qrope);
    if (kFp8 || p.page_box) ptx::prefetch_tensormap(&tm_page);
    if (!kFp8 && p.page_box) {
      ptx::prefetch_tensormap(&tm_c4);
      ptx::prefetch_tensormap(&tm_c5);
    }
    ptx::prefetch_tensormap(&tm_cache);
    bars.abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&bars.stage_full[s], 1);
      for (int k = 0; k < 3; ++k) ptx::mbar_init(&bars.stage_ready[s][k], n_prep / 32);
      ptx::mbar_init(&bars.stage_empty[s], 1);
    }
    ptx::mbar_init(&bars.spart_full, 1);
    ptx::mbar_init(&bars.spart_empty, 1);
    for (int v = 0; v < kVSlots; ++v) {
      ptx::mbar_init(&bars.vpart_full[v], 1);
      ptx::mbar_init(&bars.vpart_empty[v], 1);
    }
    ptx::mbar_init(&bars.zero_go, 1);
    ptx::mbar_init(&bars.zeroed, n_prep / 32);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars.s_full[i], 1);
      ptx::mbar_init(&bars.p_full[i], n_soft);  // one arrival per softmax warp
    }
    ptx::mbar_init(&bars.o_done, 1);
    ptx::mbar_init(&bars.seg_done, 1);
    ptx::mbar_init(&bars.q_free, 1);
    ptx::mbar_init(&bars.q_lo_full, 1);
    ptx::mbar_init(&bars.q_cp_done, 1);
    ptx::mbar_init(&bars.q_hi_full, 1);
    ptx::mbar_init(&bars.q0_copied, 1);
    ptx::mbar_init(&bars.conv_sync, n_prep / 32);  // one arrival per preparation warp
    ptx::mbar_init(&bars.part_done, n_soft);
    ptx::mbar_init(&bars.merge_go, 1);
    ptx::mbar_init(&bars.dec_go, 1);
    ptx::mbar_init(&bars.merge_full, 1);
    ptx::fence_barrier_init();
  }
  // the plan's length loads go out first; the other warps set up meanwhile
  if (warp == 3) make_plan(p, unit, &bars.plan);
  // Q rows T*H..127 are never loaded: keep them zero (finite scores in the padded rows)
  for (int i = threadIdx.x; i < 5 * kQChunk / 16; i += kThreads)
    reinterpret_cast<uint4*>(sm + kOffQhi)[i] = make_uint4(0, 0, 0, 0);
  ptx::fence_proxy_async();
  if (warp == 2) ptx::tmem_alloc(&bars.tmem_base, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort_flag = &bars.abort_flag;
  Segments segs;
  segs.init(p, bars.plan);
  int seq, L, lo, hi;

  if (warp == 0) {
    // -------------------------------------------------------------- TMA producer
    // One lane issues Q, the pages in order (fp8: whole pages; bf16: the value part as soon
    // as its ring slot frees, then the score-only part once the previous page's scores are
    // done with that slot) and the L2 warming.  Copies are served in issue order, so the
    // value part, which goes out about a page earlier, never waits behind a score-only part.
    if ((threadIdx.x & 31) == 0) {
      int g = 0, nseg = 0;
      bool ok = true;
      while (ok && segs.next(seq, L, lo, hi)) {
        // the first page's table entry is read before Q is issued, so its latency overlaps
        // the Q copies instead of delaying the page's own
        const int page_first = page_of(p, seq, lo);
        {
          if (nseg == 0) {
            // first sequence: Q latent 0..255 staged in the (still unused) second page
            // stage, the rest of Q straight into the Q area, all at once
            ptx::mbar_arrive_expect_tx(&bars.q_lo_full, 4 * TQ * 128);
            for (int c = 0; c < 4; ++c)
              ptx::tma_load_2d(sm + q_stage_off(c), &tm_qlat, &bars.q_lo_full, c * 64, q_row0(seq));
            ptx::mbar_arrive_expect_tx(&bars.q_hi_full, 5 * TQ * 128);
            for (int c = 0; c < 4; ++c)
              ptx::tma_load_2d(sm + kOffQhi + c * kQChunk, &tm_qlat, &bars.q_hi_full, 256 + c * 64, q_row0(seq));
            ptx::tma_load_2d(sm + kOffQhi + 4 * kQChunk, &tm_qrope, &bars.q_hi_full, 0, q_row0(seq));
          } else {
            // Q latent 0..255 into the Q area once the previous sequence's last S is done
            if (!(ok = ptx::mbar_wait(&bars.q_free, (nseg - 1) & 1, abort_flag, p.err))) break;
            ptx::mbar_arrive_expect_tx(&bars.q_lo_full, 4 * TQ * 128);
            for (int c = 0; c < 4; ++c)
              ptx::tma_load_2d(sm + kOffQhi + c * kQChunk, &tm_qlat, &bars.q_lo_full, c * 64, q_row0(seq));
          }
          ++nseg;
        }
        // warm L2 with the next segment's Q (read when this one's pages are done) once this
        // segment's first page is issued: finding the next segment reads the lengths again
        auto warm_next_q = [&]() {
          Segments nx = segs;
          int s2, L2, lo2, hi2;
          if (nx.next(s2, L2, lo2, hi2)) {
            const int r0 = q_row0(s2), rows = min(TQ, p.B * TH - r0);
            if (rows > 0) {
              ptx::bulk_prefetch(p.q_latent + (size_t)r0 * kDl, rows * kDl * 2);
              ptx::bulk_prefetch(p.q_rope + (size_t)r0 * 64, rows * 128);
            }
          }
        };
        for (int pg = lo; pg < hi; ++pg, ++g) {
          const int s = g % kStages;
          if (kFp8 && !(ok = ptx::mbar_wait(&bars.stage_empty[s], ((g / kStages) & 1) ^ 1, abort_flag, p.err)))
            break;
          // the first sequence's staged Q stays in place until it is copied to TMEM
          if (kFp8 && g == 1 && !(ok = ptx::mbar_wait(&bars.q0_copied, 0, abort_flag, p.err))) break;
          const int y = pg == lo ? row_of_page(p, page_first) : page_row(p, seq, pg);
          if constexpr (kFp8) {
            unsigned char* dst = sm + kOffStage + s * kStageBytes + kRawOffset;
            ptx::mbar_arrive_expect_tx(&bars.stage_full[s], 9 * kRawChunk);
            if (p.page_box) {
              ptx::tma_load_3d(dst, &tm_page, &bars.stage_full[s], 0, y, 0);
            } else {
              for (int c = 0; c < 9; ++c)
                ptx::tma_load_2d(dst + c * kRawChunk, &tm_cache, &bars.stage_full[s], c * 64, y);
            }
          } else {
            // The value part first: its slot (the page three back has had its PV) frees about
            // a page before the score-only slot does, so it goes out then and lands before the
            // score k-steps reach it, instead of queueing behind this page's score-only part.
            // Own latent chunks 4 half .. 4 half + 3 (value slots 1 and 2 first hold the first
            // sequence's staged Q).
            const int v = g % kVSlots;
            if (!(ok = ptx::mbar_wait(&bars.vpart_empty[v], ((g / kVSlots) & 1) ^ 1, abort_flag, p.err))) break;
            if ((g == 1 || g == 2) && !(ok = ptx::mbar_wait(&bars.q0_copied, 0, abort_flag, p.err))) break;
            unsigned char* dst = sm + kOffVPart + v * kVPartBytes;
            ptx::mbar_arrive_expect_tx(&bars.vpart_full[v], kVPartBytes);
            if (p.page_box) {
              ptx::tma_load_3d(dst, &tm_c4, &bars.vpart_full[v], 0, y, 4 * half);
            } else {
              for (int c = 0; c < 4; ++c)
                ptx::tma_load_2d(dst + c * kPageChunk, &tm_cache, &bars.vpart_full[v], (4 * half + c) * 64, y);
            }
            // then the score-only chunks (chunk_idx order: half 0 takes 4..8, half 1 0..3 and
            // 8), once the previous page's score k-steps over them are done
            if (!(ok = ptx::mbar_wait(&bars.spart_empty, (g & 1) ^ 1, abort_flag, p.err))) break;
            dst = sm + kOffSPart;
            ptx::mbar_arrive_expect_tx(&bars.spart_full, kSPartBytes);
            if (p.page_box && half == 0) {
              ptx::tma_load_3d(dst, &tm_c5, &bars.spart_full, 0, y, 4);
            } else if (p.page_box) {
              ptx::tma_load_3d(dst, &tm_c4, &bars.spart_full, 0, y, 0);
              ptx::tma_load_2d(dst + 4 * kPageChunk, &tm_cache, &bars.spart_full, 512, y);
            } else {
              for (int i = 0; i < 5; ++i)
                ptx::tma_load_2d(dst + i * kPageChunk, &tm_cache, &bars.spart_full,
                                 (half == 0 ? 4 + i : (i < 4 ? i : 8)) * 64, y);
            }
          }
          if (pg == lo) warm_next_q();
          // warm L2 with the pages ahead (after this page's own load has been issued)
          for (int a = (pg == lo ? lo + 1 : pg + kPrefetchAhead); a <= min(hi - 1, pg + kPrefetchAhead); ++a) {
            const int ya = page_row(p, seq, a);
            if (ya < 0) continue;
            // the page is 72 KB (bf16; 36 KB fp8) of contiguous bytes: one linear prefetch
            // reads it in address order
            constexpr uint32_t kPageBytes = kPage * kDc * (kFp8 ? 1 : 2);
            ptx::bulk_prefetch(p.cache_bytes + (size_t)ya * (kDc * (kFp8 ? 1 : 2)), kPageBytes);
          }
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (ptx::elect_one()) {
      constexpr uint32_t kIdS = ptx::make_idesc(1, kRows, kPage, 0, 0);
      constexpr uint32_t kIdPV = ptx::make_idesc(1, kRows, 256, 0, 1);
      const uint32_t qhi = ptx::smem_u32(sm + kOffQhi);
      const uint32_t stage0 = ptx::smem_u32(sm + kOffStage);
      const uint32_t o_tm = tmem + 256;
      int g = 0, nseg = 0;
      int n_zeroed = 0;  // bf16: partial pages zeroed so far
      bool ok = true;
      const uint32_t smb = ptx::smem_u32(sm);
      // Operand descriptors, built once (k-step j of a chunk is 32 bytes further, i.e. 2 in
      // the start-address field; a chunk 8 KB, i.e. 512): B = the page chunks (fp8: stage 0 /
      // 1 in chunk order; bf16: the score-only slot, value slot 0 / 1 / 2), A = the shared-
      // memory Q chunks.  This keeps the issue loop at an add or two per MMA: the MMA thread
      // shares its SM sub-partition with a softmax warp.
      const uint64_t b0 = ptx::sw128_desc(smb + (kFp8 ? kOffStage : kOffSPart), 16, 1024);
      const uint64_t b1 = ptx::sw128_desc(smb + (kFp8 ? kOffStage + kStageBytes : kOffVPart), 16, 1024);
      const uint64_t b2 = ptx::sw128_desc(smb + kOffVPart + kVPartBytes, 16, 1024);
      const uint64_t b3 = ptx::sw128_desc(smb + kOffVPart + 2 * kVPartBytes, 16, 1024);
      const uint64_t qd = ptx::sw128_desc(qhi, 16, 1024);
      // k-step k (a compile-time constant at every call) of S into d, B from chunk base bc
      auto mma_k = [&](uint32_t d, uint64_t bc, int k, bool acc) {
        const uint64_t db = bc + 2 * (k & 3);
        if (k < 16)  // latent 0..255: A from TMEM
          ptx::mma_bf16_ts(d, tmem + k * 8, db, kIdS, acc ? 1u : 0u);
        else         // latent 256..511 + rope: A from shared memory (16 KB per Q chunk)
          ptx::mma_bf16_ss(d, qd + 1024 * ((k - 16) >> 2) + 2 * ((k - 16) & 3), db, kIdS, acc ? 1u : 0u);
      };
      // part `part` of S(gg): fp8 k-steps 12 part .. 12 part + 11; bf16 the k-steps of the
      // score-only chunks (part 0), then those of the value chunks (part 1).  The first MMA
      // of S(gg) starts the accumulator.
      auto issue_s = [&](int gg, int part) {
        const uint32_t d = tmem + 128 + (gg & 1) * 64;
        if constexpr (kFp8) {
          const uint64_t st = (gg % kStages) ? b1 : b0;
          if (part == 0) {
#pragma unroll
            for (int k = 0; k < 12; ++k) mma_k(d, st + 512 * (k >> 2), k, k > 0);
          } else if (part == 1) {
#pragma unroll
            for (int k = 12; k < 24; ++k) mma_k(d, st + 512 * (k >> 2), k, true);
          } else {
#pragma unroll
            for (int k = 24; k < 36; ++k) mma_k(d, st + 512 * (k >> 2), k, true);
          }
        } else if (part == 0) {
          if (half == 0) {
#pragma unroll
            for (int k = 16; k < 36; ++k) mma_k(d, b0 + 512 * chunk_idx(k >> 2, 0), k, k > 16);
          } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) mma_k(d, b0 + 512 * chunk_idx(k >> 2, 1), k, k > 0);
#pragma unroll
            for (int k = 32; k < 36; ++k) mma_k(d, b0 + 512 * chunk_idx(k >> 2, 1), k, true);
          }
        } else {
          const int v = gg % kVSlots;
          const uint64_t vb = v == 0 ? b1 : v == 1 ? b2 : b3;
          if (half == 0) {
#pragma unroll
            for (int k = 0; k < 16; ++k) mma_k(d, vb + 512 * (k >> 2), k, true);
          } else {
#pragma unroll
            for (int k = 16; k < 32; ++k) mma_k(d, vb + 512 * ((k >> 2) - 4), k, true);
          }
        }
      };
      // PV: B = this half's 256 latent columns (four chunks 8 KB apart), 16 keys per k-step
      auto issue_pv = [&](int gg, bool first) {
        uint32_t st;
        if constexpr (kFp8) st = kOffStage + (gg % kStages) * kStageBytes + 4 * half * kPageChunk;
        else st = kOffVPart + (gg % kVSlots) * kVPartBytes;
        const uint64_t vd = ptx::sw128_desc(smb + st, kPageChunk, 1024);
        const uint32_t pa = tmem + 128 + (gg & 1) * 64;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          ptx::mma_bf16_ts(o_tm, pa + k * 8, vd + 128 * k, kIdPV, (!first || k > 0) ? 1u : 0u);
      };
      while (ok && segs.next(seq, L, lo, hi)) {
        // Q latent 0..255: staged in the Q area by the producer, copied into TMEM columns
        // 0..127 (lane = query row); then latent 256..511 + rope over the staging copy
        if (!(ok = ptx::mbar_wait(&bars.q_lo_full, nseg & 1, abort_flag, p.err))) break;
        ptx::tc_fence_after();
        // the first sequence's Q latent 0..255 was staged in the second page stage
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint32_t qc = nseg == 0 ? smb + q_stage_off(k >> 2) : qhi + (k >> 2) * kQChunk;
          ptx::tmem_cp_128x256b(tmem + k * 8, ptx::sw128_desc(qc + (k & 3) * 32, 16, 1024));
        }
        ptx::mma_commit(&bars.q_cp_done);
        if (nseg == 0) ptx::mma_commit(&bars.q0_copied);
        if (nseg > 0) {  // the rest of Q over the staging copy (the producer loaded the first)
          if (!(ok = ptx::mbar_wait(&bars.q_cp_done, nseg & 1, abort_flag, p.err))) break;
          ptx::mbar_arrive_expect_tx(&bars.q_hi_full, 5 * TQ * 128);
          for (int c = 0; c < 4; ++c)
            ptx::tma_load_2d(sm + kOffQhi + c * kQChunk, &tm_qlat, &bars.q_hi_full, 256 + c * 64, q_row0(seq));
          ptx::tma_load_2d(sm + kOffQhi + 4 * kQChunk, &tm_qrope, &bars.q_hi_full, 0, q_row0(seq));
        }
        if (!(ok = ptx::mbar_wait(&bars.q_hi_full, nseg & 1, abort_flag, p.err))) break;
        ptx::tc_fence_after();
        const int g_end = g + (hi - lo), g_first = g;
        int gs = g, gp = g;  // next page whose S / whose PV is to be issued
        int sp = 0;          // next part of S(gs)
        bool zero_asked = false;  // bf16: the partial page gs was handed to the preparation warps
        long long t0 = clock64();
        while (gp < g_end) {
          bool progress = false;
          // PV first: it releases the page stage for the next load
          if (gp < gs && ptx::mbar_test_wait(&bars.p_full[gp & 1], (gp >> 1) & 1)) {
            ptx::tc_fence_after();
            issue_pv(gp, gp == g_first);
            ptx::mma_commit(&bars.o_done);
            // fp8: the whole stage; bf16: the value part (the score-only part was released
            // after the scores)
            ptx::mma_commit(kFp8 ? &bars.stage_empty[gp % kStages] : &bars.vpart_empty[gp % kVSlots]);
            ++gp;
            progress = true;
          }
          // S(gs) may run at most one page ahead of the oldest unissued PV (two S buffers).
          // A full bf16 page needs no preparation: its parts are ready when they land.  A page
          // that ends its sequence part-way goes to the preparation warps once both parts have
          // landed and comes back with the rows past the end zeroed.
          bool can = false;
          if (gs < g_end && gs <= gp + 1) {
            if constexpr (kFp8) {
              can = ptx::mbar_test_wait(&bars.stage_ready[gs % kStages][sp], (gs / kStages) & 1);
            } else if ((lo + (gs - g_first) + 1) * kPage <= L) {
              can = sp == 0 ? ptx::mbar_test_wait(&bars.spart_full, gs & 1)
                            : ptx::mbar_test_wait(&bars.vpart_full[gs % kVSlots], (gs / kVSlots) & 1);
            } else if (sp == 1) {
              can = true;  // zeroed before its part 0
            } else if (!zero_asked) {
              if (ptx::mbar_test_wait(&bars.spart_full, gs & 1) &&
                  ptx::mbar_test_wait(&bars.vpart_full[gs % kVSlots], (gs / kVSlots) & 1)) {
                ptx::mbar_arrive(&bars.zero_go);
                zero_asked = true;
                progress = true;
              }
            } else if (ptx::mbar_test_wait(&bars.zeroed, n_zeroed & 1)) {
              can = true;
              zero_asked = false;
              ++n_zeroed;
            }
          }
          if (can) {
            ptx::tc_fence_after();
            issue_s(gs, sp);
            if (!kFp8 && sp == 0) ptx::mma_commit(&bars.spart_empty);
            if (sp + 1 < kParts) {
              ++sp;
            } else {
              sp = 0;
              ptx::mma_commit(&bars.s_full[gs & 1]);
              ++gs;
              if (gs == g_end) ptx::mma_commit(&bars.q_free);  // Q no longer read
            }
            progress = true;
          }
          if (progress) {
            t0 = clock64();
          } else if (*abort_flag) {
            ok = false;
            break;
          } else if (clock64() - t0 > 1000000000LL) {
            latch_error(p.err, kErrTimeout);
            *abort_flag = 1;
            ok = false;
            break;
          }
        }
        if (ok) ptx::mma_commit(&bars.seg_done);  // the segment's last PV product is complete
        g = g_end;
        ++nseg;
      }
    }
  } else if (warp < 4 || warp >= 8 || warp >= 4 + n_soft) {
    // -------------------------------------------------------------- stage preparation
    // 0 .. n_prep - 1: warps 2-3, then 8-11, then the softmax warps that joined
    const int tid = warp < 4 ? threadIdx.x - 64
                  : warp >= 8 ? threadIdx.x - 192
                              : kPrepOf<kFp8> + threadIdx.x - 32 * (4 + n_soft);
    const int row = tid & (kPage - 1);  // the page row whose scale (fp8) this thread stages
    int g = 0, n_zero = 0;
    bool ok = true;
    while (ok && segs.next(seq, L, lo, hi)) {
      for (int pg = lo; pg < hi; ++pg, ++g) {
        const int s = g % kStages;
        unsigned char* st = sm + kOffStage + s * kStageBytes;
        const int valid = min(kPage, L - pg * kPage);  // rows holding tokens of this sequence
        const int page = __ldg(p.page_table + (size_t)(seq / p.NQT) * p.max_pages + pg);
        const bool bad = page < 0 || page >= p.num_pages;
        if (bad && tid == 0 && seq % p.NQT == 0) latch_error(p.err, kErrBadPage);
        const bool live = !bad && row < valid;
        auto live_row = [&](int rr) { return !bad && rr < valid; };
        float ksc = 0.f;
        if constexpr (kFp8) ksc = live && tid < kPage ? __ldg(p.kv_scale + (size_t)page * kPage + row) : 0.f;
        if constexpr (!kFp8) {
          // A page that ends its sequence part-way: once the MMA thread has seen both of its
          // parts land it hands the page over (zero_go); rows valid..63 of its nine chunks
          // are zeroed (16-byte granules; whole rows, so the swizzle is immaterial) and handed
          // back (zeroed).  Full pages go straight from the copy to the MMA.
          if (valid < kPage) {
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.zero_go, n_zero & 1, abort_flag, p.err));
            if (!ok) break;
            const int nrow = kPage - valid;
            for (int part = 0; part < 2; ++part) {
              const int nch = part == 0 ? 5 : 4;
              unsigned char* base = sm + (part == 0 ? kOffSPart : kOffVPart + (g % kVSlots) * kVPartBytes);
              for (int e = tid; e < nrow * nch * 8; e += n_prep) {
                const int rw = valid + e / (nch * 8), rem = e % (nch * 8), c = rem >> 3, gr = rem & 7;
                *reinterpret_cast<uint4*>(base + c * kPageChunk + rw * 128 + gr * 16) = make_uint4(0, 0, 0, 0);
              }
            }
            ptx::fence_proxy_async();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&bars.zeroed);
            ++n_zero;
          }
        } else {
          ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.stage_full[s], (g / kStages) & 1, abort_flag, p.err));
          if (!ok) break;
          if (tid < kPage) bars.kscale[s][row] = ksc;
          // Widen in place, in three lockstep steps of three chunks (four 16-byte granules
          // per thread per step).  bf16 chunk c (bytes [8c, 8c+8) KB) overlaps raw chunks 2c-9
          // and 2c-8 (raw chunk c' sits at [36 + 4c', 40 + 4c') KB), which are at most the
          // step's own chunks 3k..3k+2 or earlier ones: after every thread has read its raw
          // granules of the step (bounded mbarrier), the step's writes only destroy bytes that
          // were already read, and never those of a later step.
#pragma unroll 1
          for (int k = 0; k < 3 && ok; ++k) {
            // the step's 3 chunks are 768 granules of 16 raw bytes (64 rows x 4 per chunk);
            // thread tid takes granules tid + n_prep q (at most four: n_prep >= 192), so a warp
            // reads 512 contiguous bytes
            uint4 raw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int G = tid + n_prep * q, c = 3 * k + (G >> 8), gi = G & 255;
              raw[q] = (G < 768 && live_row(gi >> 2))
                           ? *reinterpret_cast<const uint4*>(st + kRawOffset + c * kRawChunk + gi * 16)
                           : make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&bars.conv_sync);
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.conv_sync, (3 * g + k) & 1, abort_flag, p.err));
            if (!ok) break;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int G = tid + n_prep * q, c = 3 * k + (G >> 8), gi = G & 255;
              if (G >= 768) continue;
              const int rw = gi >> 2, quarter = gi & 3;  // 16 columns 16 quarter .. of row rw
              const uint32_t words[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
              uint32_t w[8];
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                w[2 * x] = ptx::e4m3x2_to_bf16x2(words[x]);
                w[2 * x + 1] = ptx::e4m3x2_to_bf16x2(words[x] >> 16);
              }
              unsigned char* dst = st + c * kPageChunk + rw * 128;
              *reinterpret_cast<uint4*>(dst + (((2 * quarter) ^ (rw & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4*>(dst + (((2 * quarter + 1) ^ (rw & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
            // chunks 3k..3k+2 are ready for the score MMA (the next steps write above them)
            ptx::fence_proxy_async();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&bars.stage_ready[s][k]);
          }
          if (!ok) break;
        }
      }
    }
  } else {
    // -------------------------------------------------------------- softmax / epilogue
    const int r = threadIdx.x - 128;  // query row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int g = 0, n_epi = 0, n_part = 0, n_bulk = 0, n_bulk_issued = 0;
    bool ok = true;
    // a sequence with no cached key is in no work unit's range: unit u writes O = 0 and
    // LSE = -inf for the empty sequences u, u + G, u + 2G, ...
    if (half == 0) {
      for (int b = unit; b < p.B; b += p.G) {
        if (clamp_len(__ldg(p.cache_lens + b), p.max_pages) > 0) continue;
        uint4* o = reinterpret_cast<uint4*>(p.out + (size_t)b * TH * kDl);
        for (int i = r; i < TH * (kDl / 8); i += 32 * n_soft)
          if (MLA_STORE_OK(o + i, p.out, p.out_bytes, p.err)) o[i] = make_uint4(0, 0, 0, 0);
        for (int i = r; i < TH; i += 32 * n_soft) {
          float* lp = p.lse + ((size_t)b * p.H + i % p.H) * p.T + i / p.H;
          if (MLA_STORE_OK(lp, p.lse, p.lse_bytes, p.err)) *lp = -INFINITY;
        }
      }
    }
    while (ok && segs.next(seq, L, lo, hi)) {
      const int gr = (seq % p.NQT) * kRows + r;  // row within the sequence's T*H rows
      const int t_row = gr / p.H;
      const int last_visible = p.causal ? (L - p.T + t_row) : (L - 1);  // keys <= this are visible
      float m = -INFINITY, l = 0.f, lr = 0.f;  // exact row sum (LSE) and bf16-rounded (PV)
      const uint32_t o_addr = tmem + lane_off + 256;
      for (int pg = lo; pg < hi; ++pg, ++g) {
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.s_full[g & 1], (g >> 1) & 1, abort_flag, p.err));
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t s_addr = tmem + lane_off + 128 + (g & 1) * 64;
        float s[64];
        {
          uint32_t* su = reinterpret_cast<uint32_t*>(s);
          ptx::tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(su));
          ptx::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(su + 32));
          ptx::tmem_ld_wait();
        }
        const int page = __ldg(p.page_table + (size_t)(seq / p.NQT) * p.max_pages + pg);
        const bool bad = page < 0 || page >= p.num_pages;
        const int key0 = pg * kPage;
        const int lim = bad ? -1 : min(last_visible, L - 1);  // visible keys: key0+x <= lim
        // unscaled scores (fp8: times the key's scale), two keys per packed instruction; the
        // softmax scale is applied in the exponent argument
        const float* ks = bars.kscale[g % kStages];
        uint64_t s2[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          s2[x] = ptx::f2(s[2 * x], s[2 * x + 1]);
          if constexpr (kFp8) s2[x] = ptx::mul2(s2[x], ptx::f2(ks[2 * x], ks[2 * x + 1]));
        }
        if (key0 + kPage - 1 > lim) {  // a partial page (or a bad one): mask invisible keys
#pragma unroll
          for (int x = 0; x < 32; ++x)
            s2[x] = ptx::f2(key0 + 2 * x <= lim ? ptx::f2_lo(s2[x]) : -INFINITY,
                            key0 + 2 * x + 1 <= lim ? ptx::f2_hi(s2[x]) : -INFINITY);
        }
        float mx4[4] = {ptx::f2_lo(s2[0]), ptx::f2_hi(s2[0]), ptx::f2_lo(s2[1]), ptx::f2_hi(s2[1])};
#pragma unroll
        for (int x = 2; x < 32; ++x) mx4[x & 3] = ptx::fmax3(mx4[x & 3], ptx::f2_lo(s2[x]), ptx::f2_hi(s2[x]));
        // tile maximum in the exponent domain (the scale is positive; -inf stays -inf)
        const float mx = ptx::fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]) * p.scale_log2;
        float m_use = m;
        if (pg == lo) {
          m_use = mx;
        } else {
          const bool grow = mx > m + 8.0f;
          if (__any_sync(0xffffffffu, grow)) {
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.o_done, (g - 1) & 1, abort_flag, p.err));
            if (!ok) break;
            ptx::tc_fence_after();
            const float alpha = grow ? ptx::ex2(m - mx) : 1.f;  // m = -inf gives 0
            if (grow) m_use = mx;
            uint32_t v[2][32];
#pragma unroll 1
            for (int c = 0; c < 8; c += 2) {
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
        const float neg_m = (m == -INFINITY) ? 0.f : -m;
        const uint64_t sc2 = ptx::f2(p.scale_log2, p.scale_log2), nm2 = ptx::f2(neg_m, neg_m);
        uint64_t ps2[2] = {ptx::f2(0.f, 0.f), ptx::f2(0.f, 0.f)};
        float pr[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const uint64_t a2 = ptx::fma2(s2[x], sc2, nm2);
          const uint64_t pp = ptx::f2(ptx::ex2(ptx::f2_lo(a2)), ptx::ex2(ptx::f2_hi(a2)));
          ps2[x & 1] = ptx::add2(ps2[x & 1], pp);
          if constexpr (kFp8) {
            const uint64_t ab = ptx::mul2(pp, ptx::f2(ks[2 * x], ks[2 * x + 1]));  // P' = p ks
            pk[x] = ptx::pack_bf16x2(ptx::f2_lo(ab), ptx::f2_hi(ab));
          } else {
            // O is normalised by the sum of the bf16-rounded values the PV product uses
            // (exact for a dominant key); the LSE uses the exact sum
            const uint32_t w = ptx::pack_bf16x2(ptx::f2_lo(pp), ptx::f2_hi(pp));
            pk[x] = w;
            ptx::add_bf16x2(pr[2 * (x & 1)], pr[2 * (x & 1) + 1], w);
          }
        }
        const uint64_t ps_all = ptx::add2(ps2[0], ps2[1]);
        const float psum = ptx::f2_lo(ps_all) + ptx::f2_hi(ps_all);
        l += psum;
        lr += kFp8 ? psum : (pr[0] + pr[1]) + (pr[2] + pr[3]);
        ptx::tmem_st32(s_addr, pk);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&bars.p_full[g & 1]);
      }
      if (!ok) break;
      // epilogue of the segment: partial (O_half / l, LSE) into slot unit + seq, once the
      // segment's last PV product is complete.  That is signalled once per segment: the
      // per-page o_done cannot be used here, since a warp that ran ahead of a slower one may
      // arrive while PV(g-2) is still pending and one parity bit cannot tell that phase from
      // the one after PV(g-1).  seg_done of the next segment needs this warp's P, so it is
      // never more than one phase ahead.
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.seg_done, n_epi & 1, abort_flag, p.err));
      if (!ok) break;
      ptx::tc_fence_after();
      const size_t slot = (size_t)unit + seq;
      const float inv = lr > 0.f ? 1.f / lr : 0.f;
      const float lse_own = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      const bool row_live = r < TQ && gr < TH;
      // The work units that cover this virtual sequence write their partials of this column
      // half into slots c + seq, c_first <= c <= c_first + nsplit - 1; this one is k_own.
      const int n_pages = pages_of(L, kPage);
      const int c_first = segs.flat0 / bars.plan.chunk;
      const int nsplit = (segs.flat0 + n_pages - 1) / bars.plan.chunk - c_first + 1;
      const int k_own = unit - c_first;
      // Merge path.  A split that finds every other split of this (sequence, column half)
      // counted in (always so for a sequence with one split) merges at once, its own share
      // read from the accumulator.  Otherwise it writes its partial (O_half / l, LSE), makes
      // it visible device-wide and counts itself in; the split that completes the count
      // merges: O = sum_c exp(lse_c - lse) O_c with lse = ln sum_c exp(lse_c).
      // After the unit's last segment nothing more is loaded and every MMA is complete: Q's
      // area takes the staged bf16 output rows, the page stages a bulk copy of the other
      // split's partial when the sequence has exactly two (one TMA transfer instead of
      // rounds of dependent L2 loads per thread).
      bool last_seg;
      {
        Segments nx = segs;
        int s2, L2, lo2, hi2;
        last_seg = !nx.next(s2, L2, lo2, hi2);
      }
      if (r == 0) {
        int fast = 1, bulk = 0;
        if (nsplit > 1) {
          // the counters were zeroed by the kernel this one was launched behind
          asm volatile("griddepcontrol.wait;" ::: "memory");
          fast = ptx::ld_acquire_gpu(p.counters + (size_t)seq * 2 + half) == nsplit - 1;
          if (fast && nsplit == 2 && last_seg) {
            const float4* src = reinterpret_cast<const float4*>(p.part_o) +
                                ((size_t)(c_first + seq + (1 - k_own)) * 128 + half * 64) * TQ;
            ptx::fence_proxy_async_global();
            ptx::mbar_arrive_expect_tx(&bars.merge_full, 1024u * TQ);
            ptx::bulk_load(sm + kOffStage, src, 1024u * TQ, &bars.merge_full);
            bulk = 1;
            ++n_bulk_issued;
          }
        }
        bars.merge_fast = fast;
        bars.merge_bulk = bulk;
        ptx::mbar_arrive(&bars.dec_go);
      }
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.dec_go, n_epi & 1, abort_flag, p.err));
      ++n_epi;
      if (!ok) break;
      // The accumulator is intact until the next segment's first PV product, which waits for
      // this epilogue: a split that merges always takes its own share from it.
      bool own_in_tmem = *reinterpret_cast<volatile int*>(&bars.merge_fast) != 0;
      bool bulk = *reinterpret_cast<volatile int*>(&bars.merge_bulk) != 0;
      bool merge = own_in_tmem;
      if (!own_in_tmem) {
        // partial layout [slot][column quad (128)][row (T*H)][4]: the 32 rows of a warp store
        // one quad as 512 contiguous bytes; kept in L2 ahead of the cache lines streaming past,
        // since the merge reads it back, possibly at the end of the launch
        const uint64_t keep = ptx::l2_policy_evict_last();
        float4* dst = reinterpret_cast<float4*>(p.part_o) + (slot * 128 + half * 64) * TQ + r;
#pragma unroll 1
        for (int c = 0; c < 8; c += 2) {
          uint32_t v[2][32];
          ptx::tmem_ld32(o_addr + c * 32, v[0]);
          ptx::tmem_ld32(o_addr + (c + 1) * 32, v[1]);
          ptx::tmem_ld_wait();
          if (row_live) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
              for (int x = 0; x < 8; ++x) {
                float4* d4 = dst + (size_t)((c + h2) * 8 + x) * TQ;
                if (MLA_STORE_OK(d4, p.part_o, p.part_o_bytes, p.err))
                  ptx::st_l2_hint(d4,
                                  make_float4(__uint_as_float(v[h2][4 * x]) * inv, __uint_as_float(v[h2][4 * x + 1]) * inv,
                                              __uint_as_float(v[h2][4 * x + 2]) * inv,
                                              __uint_as_float(v[h2][4 * x + 3]) * inv),
                                  keep);
              }
          }
        }
        float* plp = p.part_lse + ((size_t)half * p.n_slots + slot) * TQ + r;
        if (row_live && MLA_STORE_OK(plp, p.part_lse, p.part_lse_bytes, p.err)) *plp = lse_own;
        __threadfence();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&bars.part_done);
        if (r == 0) {
          bool go = ptx::mbar_wait(&bars.part_done, n_part & 1, abort_flag, p.err);
          if (go) {
            __threadfence();
            int* cnt = p.counters + (size_t)seq * 2 + half;
            const int done = MLA_STORE_OK(cnt, p.counters, p.counters_bytes, p.err) ? atomicAdd(cnt, 1) + 1 : 0;
            __threadfence();
            bars.merge_last = done == nsplit ? 1 : 0;
            if (done == nsplit && nsplit == 2 && last_seg) {
              const float4* src = reinterpret_cast<const float4*>(p.part_o) +
                                  ((size_t)(c_first + seq + (1 - k_own)) * 128 + half * 64) * TQ;
              ptx::fence_proxy_async_global();
              ptx::mbar_arrive_expect_tx(&bars.merge_full, 1024u * TQ);
              ptx::bulk_load(sm + kOffStage, src, 1024u * TQ, &bars.merge_full);
              bars.merge_bulk = 1;
              ++n_bulk_issued;
            }
          } else {
            bars.merge_last = 0;
          }
          ptx::mbar_arrive(&bars.merge_go);
        }
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.merge_go, n_part & 1, abort_flag, p.err));
        ++n_part;
        if (!ok) break;
        merge = *reinterpret_cast<volatile int*>(&bars.merge_last) != 0;
        bulk = *reinterpret_cast<volatile int*>(&bars.merge_bulk) != 0;
        own_in_tmem = merge;
      }
      if (merge) {
        // Every lane of a warp runs this block (the accumulator loads are warp-collective:
        // a lane that skipped them would stall its warp for good); global memory is touched
        // for the live rows only.  This thread's row: weights of the splits from their LSEs
        // (read through L2: they were written by other SMs during this launch).  The first
        // kLseRegs LSEs are loaded together and kept; any further split's is read again
        // where it is used.
        const float* lsp = p.part_lse + ((size_t)half * p.n_slots + c_first + seq) * TQ + r;
        auto lse_of = [&](int k) -> float {
          if (own_in_tmem && k == k_own) return lse_own;
          return row_live ? ptx::ld_l2(lsp + (size_t)k * TQ) : -INFINITY;
        };
        constexpr int kLseRegs = 4;
        float lse_r[kLseRegs];
#pragma unroll
        for (int k = 0; k < kLseRegs; ++k) lse_r[k] = k < nsplit ? lse_of(k) : -INFINITY;
        float mxl = -INFINITY;
#pragma unroll
        for (int k = 0; k < kLseRegs; ++k) mxl = fmaxf(mxl, lse_r[k]);
        for (int k = kLseRegs; k < nsplit; ++k) mxl = fmaxf(mxl, lse_of(k));
        auto wraw = [&](float ls) { return (mxl == -INFINITY || ls == -INFINITY) ? 0.f : __expf(ls - mxl); };
        float wsum = 0.f;
#pragma unroll
        for (int k = 0; k < kLseRegs; ++k) wsum += wraw(lse_r[k]);
        for (int k = kLseRegs; k < nsplit; ++k) wsum += wraw(lse_of(k));
        const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
        float w_r[kLseRegs];
#pragma unroll
        for (int k = 0; k < kLseRegs; ++k) w_r[k] = wraw(lse_r[k]) * winv;
        const float4* src = reinterpret_cast<const float4*>(p.part_o) +
                            ((size_t)(c_first + seq) * 128 + half * 64) * TQ + r;
        const size_t slot_stride = (size_t)128 * TQ;
        uint4* orow = reinterpret_cast<uint4*>(
            p.out + ((size_t)(seq / p.NQT) * TH + gr) * kDl + half * 256);
        // After the unit's last segment the bf16 rows are staged in Q's area, 512 bytes per
        // row with 16-byte chunk c of row r at chunk c ^ (r mod 32), and each warp then stores
        // its 32 rows as one 512-byte run per instruction.  Earlier segments store straight
        // from the row's thread.
        const bool staged = last_seg;
        unsigned char* stage_out = sm + kOffQhi;
        // the bulk-copied partial of the other split: [quad][row][4] floats from the stages
        const float4* part_sm = reinterpret_cast<const float4*>(sm + kOffStage) + r;
        if (bulk) {
          ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars.merge_full, n_bulk & 1, abort_flag, p.err));
          ++n_bulk;
          if (!ok) break;
        }
        // Sixteen column quads (64 columns) per round: 16 independent 16-byte loads of a
        // split's partial in flight.  The splits are summed in split order, each as weight x
        // (O_c / l_c) in fp32, the own share formed from the accumulator exactly as its stored
        // partial would be: the result does not depend on which split merges.
#pragma unroll 1
        for (int q = 0; q < 64; q += 16) {
          float4 acc[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
          for (int k = 0; k < nsplit; ++k) {
            const float w = k == 0 ? w_r[0] : k == 1 ? w_r[1] : k == 2 ? w_r[2] : k == 3 ? w_r[3]
                                                                                 : wraw(lse_of(k)) * winv;
            float4 x[16];
            if (own_in_tmem && k == k_own) {
              uint32_t v[2][32];
              ptx::tmem_ld32(o_addr + q * 4, v[0]);
              ptx::tmem_ld32(o_addr + q * 4 + 32, v[1]);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; ++j)
                x[j] = make_float4(__uint_as_float(v[j >> 3][4 * (j & 7)]) * inv,
                                   __uint_as_float(v[j >> 3][4 * (j & 7) + 1]) * inv,
                                   __uint_as_float(v[j >> 3][4 * (j & 7) + 2]) * inv,
                                   __uint_as_float(v[j >> 3][4 * (j & 7) + 3]) * inv);
            } else if (bulk) {  // the other split of two, copied into shared memory
#pragma unroll
              for (int j = 0; j < 16; ++j)
                x[j] = row_live ? part_sm[(size_t)(q + j) * TQ] : make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
              const float4* b = src + (size_t)k * slot_stride;
#pragma unroll
              for (int j = 0; j < 16; ++j)
                x[j] = row_live ? ptx::ld_l2(b + (size_t)(q + j) * TQ) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              acc[j].x = fmaf(w, x[j].x, acc[j].x);
              acc[j].y = fmaf(w, x[j].y, acc[j].y);
              acc[j].z = fmaf(w, x[j].z, acc[j].z);
              acc[j].w = fmaf(w, x[j].w, acc[j].w);
            }
          }
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const uint4 w = make_uint4(ptx::pack_bf16x2(acc[j].x, acc[j].y), ptx::pack_bf16x2(acc[j].z, acc[j].w),
                                       ptx::pack_bf16x2(acc[j + 1].x, acc[j + 1].y),
                                       ptx::pack_bf16x2(acc[j + 1].z, acc[j + 1].w));
            const int ch = (q + j) >> 1;  // 16-byte chunk of the row's 512 bytes
            if (staged)
              *reinterpret_cast<uint4*>(stage_out + r * 512 + ((ch ^ (r & 31)) << 4)) = w;
            else if (row_live && MLA_STORE_OK(orow + ch, p.out, p.out_bytes, p.err))
              orow[ch] = w;
          }
        }
        if (staged) {
          __syncwarp();
          const int lane = threadIdx.x & 31;
          const int r_base = r - lane;  // the warp's 32 rows
#pragma unroll 4
          for (int i = 0; i < 32; ++i) {
            const int rr = r_base + i, grr = (seq % p.NQT) * kRows + rr;
            uint4* od = reinterpret_cast<uint4*>(p.out + ((size_t)(seq / p.NQT) * TH + grr) * kDl + half * 256) + lane;
            if (rr < TQ && grr < TH && MLA_STORE_OK(od, p.out, p.out_bytes, p.err))
              *od = *reinterpret_cast<const uint4*>(stage_out + rr * 512 + ((lane ^ (rr & 31)) << 4));
          }
        }
        float* lp = p.lse + ((size_t)(seq / p.NQT) * p.H + gr % p.H) * p.T + gr / p.H;
        if (half == 0 && row_live && MLA_STORE_OK(lp, p.lse, p.lse_bytes, p.err))
          *lp = wsum > 0.f ? mxl + logf(wsum) : -INFINITY;
      }
      // the accumulator was read: the next segment's first PV product may overwrite it
      ptx::tc_fence_before();
    }
    // after an abort: a bulk copy issued but never waited for lands before the CTA exits
    if (r == 0 && n_bulk_issued > n_bulk) ptx::mbar_wait_drain(&bars.merge_full, n_bulk & 1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Zeroes the split counters of a decode call; the split kernel is launched behind it as a
// programmatic dependent and waits for it only where it first touches a counter.
__global__ void __launch_bounds__(256) zero_counters_kernel(int* __restrict__ c, int n) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) c[i] = 0;
}

}  // namespace sm103_decode

// ---------------------------------------------------------------- host side

// Makes the driver load every decode kernel on the current device (under lazy module loading
// a kernel's module is otherwise loaded, and its device memory allocated, at its first launch).
cudaError_t load_decode_t_kernels();
cudaError_t load_decode_kernels() {
  using namespace sm103_decode;
  cudaFuncAttributes fa;
  cudaError_t e = load_decode_t_kernels();
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, decode_split_kernel<false>)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, decode_split_kernel<true>)) != cudaSuccess) return e;
  return cudaFuncGetAttributes(&fa, zero_counters_kernel);
}

cudaError_t encode_tensor_map_swz(CUtensorMap* map, CUtensorMapDataType dt, int rank,
                                  const void* ptr, const uint64_t* dims, const uint64_t* strides,
                                  const uint32_t* box, bool swizzle128);

cudaError_t launch_decode_sm103(const void* q_latent, const void* q_rope, const void* kv_cache,
                                const float* kv_scale, const int* page_table,
                                const int* cache_lens, int B, int H, int T, int max_pages,
                                int num_pages, float softmax_scale, int causal, bool fp8,
                                float* part_o, float* part_lse, int* counters, void* out,
                                float* lse, int G, unsigned int* err, cudaStream_t stream) {
  using namespace sm103_decode;
  CUtensorMap tm;
  // the cache as a 2-D tensor [num_pages * 64 rows, 576 columns]; boxes of 64 x 64
  uint64_t dims[2] = {(uint64_t)kDc, (uint64_t)num_pages * kPage};
  uint64_t strides[1] = {(uint64_t)kDc * (fp8 ? 1 : 2)};
  uint32_t box[2] = {64, kPage};
  cudaError_t e = encode_tensor_map_swz(
      &tm, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_cache,
      dims, strides, box, /*swizzle128=*/!fp8);
  if (e != cudaSuccess) return e;
  // The same bytes as a 3-D tensor (64 columns of a chunk, row, chunk of 64 columns): a box
  // of 64 x 64 x n is n consecutive 64-column chunks of a page, landing chunk-major exactly as
  // n 2-D boxes do (one TMA instruction instead of n): fp8 pages take one box of nine chunks,
  // bf16 page parts boxes of four and five.  The chunk stride is smaller than the row stride
  // (an overlapping view); should the driver refuse that, the 2-D boxes are used.
  CUtensorMap tm_page = tm, tm_c4 = tm, tm_c5 = tm;
  uint64_t pdims[3] = {64, (uint64_t)num_pages * kPage, 9};
  uint64_t pstrides[2] = {(uint64_t)kDc * (fp8 ? 1 : 2), (uint64_t)(fp8 ? 64 : 128)};
  const CUtensorMapDataType pdt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  auto enc3 = [&](CUtensorMap* m, uint32_t nchunks) {
    uint32_t pbox[3] = {64, (uint32_t)kPage, nchunks};
    return encode_tensor_map_swz(m, pdt, 3, kv_cache, pdims, pstrides, pbox, /*swizzle128=*/!fp8) == cudaSuccess;
  };
  const bool page_box = enc3(&tm_page, 9) && (fp8 || (enc3(&tm_c4, 4) && enc3(&tm_c5, 5)));
  if (!page_box) tm_page = tm_c4 = tm_c5 = tm;
  // Q as 2-D tensors [B*T*H rows, 512 | 64 columns]; boxes of 64 columns x T*H rows
  // (one sequence), 128B-swizzled like the operand tiles
  const int TH = T * H;
  CUtensorMap tm_qlat, tm_qrope;
  uint64_t qdims[2] = {(uint64_t)kDl, (uint64_t)B * TH};
  uint64_t qstrides[1] = {(uint64_t)kDl * 2};
  const int TQ = TH < 128 ? TH : 128;
  uint32_t qbox[2] = {64, (uint32_t)TQ};
  e = encode_tensor_map_swz(&tm_qlat, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q_latent, qdims, qstrides, qbox, true);
  if (e != cudaSuccess) return e;
  qdims[0] = 64;
  qstrides[0] = 128;
  e = encode_tensor_map_swz(&tm_qrope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q_rope, qdims, qstrides, qbox, true);
  if (e != cudaSuccess) return e;
  Params p;
  p.q_latent = static_cast<const uint16_t*>(q_latent);
  p.q_rope = static_cast<const uint16_t*>(q_rope);
  p.kv_scale = kv_scale;
  p.cache_bytes = static_cast<const unsigned char*>(kv_cache);
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
  p.NQT = (TH + 127) / 128;
  p.TQ = TQ;
  p.n_slots = G + B * p.NQT;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.causal = causal;
  p.G = G;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.page_box = page_box ? 1 : 0;
  // one flat page charged per work item (its Q load, epilogue and merge; measured against
  // 0, 2 and 4 on uniform and ragged batches: the same time for 64 sequences of 4096 keys,
  // up to 7 % less where sequences split over several units or end mid-unit)
  p.item_cost = 1;
  const size_t out_full = (size_t)B * T * H * kDl * 2;
  p.out_bytes = out_full - std::min(out_full, testing_out_shrink());
  p.lse_bytes = (size_t)B * H * T * sizeof(float);
  p.part_o_bytes = (size_t)(reinterpret_cast<char*>(part_lse) - reinterpret_cast<char*>(part_o));
  p.part_lse_bytes = (size_t)(reinterpret_cast<char*>(counters) - reinterpret_cast<char*>(part_lse));
  p.counters_bytes = (size_t)2 * B * p.NQT * sizeof(int);
  // the split counters of the merge start at zero on every call
  const long long n_cnt = 2LL * B * p.NQT;
  if (n_cnt > 0x7fffffffLL) return cudaErrorInvalidValue;
  // same shared-memory carveout as the split kernel, so the SMs are not reconfigured between
  // the two launches
  static int carveout_set = 0;
  if (!__atomic_load_n(&carveout_set, __ATOMIC_ACQUIRE)) {
    if ((e = cudaFuncSetAttribute(zero_counters_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
    __atomic_store_n(&carveout_set, 1, __ATOMIC_RELEASE);
  }
  const int zero_blocks = (int)std::min<long long>((n_cnt + 2047) / 2048, 1024);
  zero_counters_kernel<<<zero_blocks, 256, 0, stream>>>(counters, (int)n_cnt);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto go = [&](auto kern) -> cudaError_t {
    static unsigned long long smem_set[2] = {0, 0};
    const cudaError_t e2 = smem_attr_once(kern, kSmemAlloc, &smem_set[fp8 ? 1 : 0]);
    if (e2 != cudaSuccess) return e2;
    // programmatic dependent of the zeroing kernel: the prologue (barriers, TMEM, plan, first
    // loads) overlaps it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * G);
    cfg.blockDim = dim3(fp8 ? kThreadsOf<true> : kThreadsOf<false>);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tm, tm_page, tm_c4, tm_c5, tm_qlat, tm_qrope, p);
  };
  return fp8 ? go(decode_split_kernel<true>) : go(decode_split_kernel<false>);
}

}  // namespace mla
