// Split plan of the decode key axis, shared by the decode kernels.
//
// The pages of all (sequence, query tile) work items are numbered in order (item v owns flat
// pages [P_v, P_v + n_v + item_cost)), and work unit c of G takes flat pages
// [c*chunk, (c+1)*chunk) with chunk = ceil(total / G).  The item_cost flat pages after a
// non-empty item's n_v pages hold no keys: a unit pays for every item it touches (loading the
// item's queries, its epilogue and partial, the merge), so units that touch more items get
// fewer real pages.  Every CTA computes its unit's plan from cache_lens alone.  The
// partial result of unit c for item v goes to slot c + v, which is unique because consecutive
// units never move backwards through the items; there are at most G + (items) - 1 slots.
// A parameter struct passed to make_plan / Segments::init provides cache_lens, B, NQT
// (query tiles per sequence), max_pages, G and item_cost (flat pages charged per item).
#pragma once

#include "common.cuh"

namespace mla {
namespace decode_plan {

constexpr int kPage = 64;

// The work unit's page range [start, end) of the flat page numbering and the first
// sequence that reaches into it (b0, whose pages start at flat page pb0).
struct Plan {
  int start, end, b0, pb0, chunk;
  // the unit's first segment, as Segments::next finds it (valid if seg_ok): sequence b0 of
  // length seg_L, pages [seg_lo, seg_hi); lets the roles start without reloading lengths
  int seg_L, seg_lo, seg_hi, seg_ok;
};

__device__ __forceinline__ int clamp_len(int L, int max_pages) {
  return min(max(L, 0), max_pages * kPage);
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// The Plan of work unit `unit`, computed by one warp with coalesced loads of the lengths
// (256 at a time) and warp scans.
template <typename Prm>
__device__ void make_plan(const Prm& prm, int unit, Plan* out) {
  const int lane = threadIdx.x & 31;
  const int B = prm.B * prm.NQT;  // work is planned per (sequence, query tile)
  auto len_at = [&](int bb) {
    return bb < B ? clamp_len(__ldg(prm.cache_lens + bb / prm.NQT), prm.max_pages) : 0;
  };
  auto flat_of = [&](int Lb) {
    const int n = pages_of(Lb, kPage);
    return n > 0 ? n + prm.item_cost : 0;
  };
  int total = 0;
  int l0s[8];  // the first 256 items' lengths, kept for the second pass
  for (int base = 0; base < B; base += 256) {
    int l[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) l[i] = len_at(base + i * 32 + lane);
    if (base == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) l0s[i] = l[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += flat_of(l[i]);
    total += warp_sum(sum);
  }
  const int chunk = total > 0 ? (total + prm.G - 1) / prm.G : 1;
  const int start = min(total, unit * chunk), end = min(total, start + chunk);
  int pb = 0, b0 = B, pb0 = total, L0 = 0;
  bool found = false;
  for (int base = 0; base < B && !found; base += 256) {
    int l[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) l[i] = base == 0 ? l0s[i] : len_at(base + i * 32 + lane);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (found) break;
      const int n_i = flat_of(l[i]);
      int incl = n_i;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      // the first sequence whose pages end past `start`; every earlier one ends at or before it
      const int bb = base + i * 32 + lane;
      const unsigned hit = __ballot_sync(0xffffffffu, bb < B && pb + incl > start);
      if (hit) {
        const int first = __ffs(hit) - 1;
        b0 = base + i * 32 + first;
        pb0 = pb + __shfl_sync(0xffffffffu, incl - n_i, first);
        L0 = __shfl_sync(0xffffffffu, l[i], first);
        found = true;
      } else {
        pb += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
  }
  // the first segment: what Segments::next computes for item b0 at flat page pb0
  int seg_lo = 0, seg_hi = 0, seg_ok = 0;
  if (found && pb0 < end) {
    const int n = pages_of(L0, kPage), nv = flat_of(L0);
    seg_lo = max(start, pb0) - pb0;
    seg_hi = min(min(end, pb0 + nv) - pb0, n);
    seg_ok = seg_lo < seg_hi ? 1 : 0;
  }
  if (lane == 0) *out = Plan{start, end, b0, pb0, chunk, L0, seg_lo, seg_hi, seg_ok};
}

// Walks the (sequence, page range) segments of this CTA's work unit in order; every
// role runs its own copy and sees the same sequence.
struct Segments {
  const int* lens;
  int B, NQT, max_pages, item_cost, start, end, b, pb;
  template <typename Prm>
  __device__ void init(const Prm& prm, const Plan& plan) {
    lens = prm.cache_lens;
    NQT = prm.NQT;
    B = prm.B * prm.NQT;
    max_pages = prm.max_pages;
    item_cost = prm.item_cost;
    start = plan.start;
    end = plan.end;
    b = plan.b0;
    pb = plan.pb0;
    seg_ok = plan.seg_ok;
    seg_L = plan.seg_L;
    seg_lo = plan.seg_lo;
    seg_hi = plan.seg_hi;
  }
  // Next non-empty segment: sets seq (the virtual sequence: sequence * NQT + query tile),
  // L, lo, hi (page indices within the sequence); flat0 = the sequence's first flat page.
  // A unit whose range reaches only into an item's key-less flat pages gets no segment of it.
  // Lengths are fetched eight at a time so that skipping to this unit's first sequence
  // costs one load latency per eight sequences rather than one per sequence.
  int flat0 = 0;
  int seg_ok, seg_L, seg_lo, seg_hi;  // the first segment, from the plan
  __device__ bool next(int& seq, int& L, int& lo, int& hi) {
    if (seg_ok) {
      seg_ok = 0;
      flat0 = pb;
      seq = b;
      L = seg_L;
      lo = seg_lo;
      hi = seg_hi;
      const int n = pages_of(seg_L, kPage);
      pb += n > 0 ? n + item_cost : 0;
      ++b;
      return true;
    }
    while (b < B && pb < end) {
      int Ls[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) Ls[i] = b + i < B ? __ldg(lens + (b + i) / NQT) : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (b >= B || pb >= end) return false;
        const int Lb = clamp_len(Ls[i], max_pages);
        const int n = pages_of(Lb, kPage);
        const int nv = n > 0 ? n + item_cost : 0;  // flat pages of the item
        const int l0 = max(start, pb) - pb, h0 = min(min(end, pb + nv) - pb, n);
        const int cur = b, cur_pb = pb;
        pb += nv;
        ++b;
        if (l0 < h0) {
          flat0 = cur_pb;
          seq = cur;
          L = Lb;
          lo = l0;
          hi = h0;
          return true;
        }
      }
    }
    return false;
  }
};


}  // namespace decode_plan
}  // namespace mla
