// topk_cand.cuh -- per-query selection from a candidate list, and the sampled
// threshold that decides which pools become candidates; device routines run
// by one 128-thread group (4 warps, one named barrier) per query row.
//
// [SkyRL-1M §1 DSA 真稀疏] each query keeps its highest-scoring pools as int32
// indices; ties go to the lower pool index.  Pools are ordered by the
// composite key (score desc, index asc), so every pool has a distinct rank.
//
// A row's candidates are the pools whose composite key is at or above a
// threshold (t, p_t): score key > t, or score key == t and index <= p_t.  If
// at least topk pools are candidates, the row's top-k lies among them, so
// selecting from the candidates alone is exact.
//
// sample_threshold  the rsel-th largest composite key among a row's sampled
//                   pools (every sigma-th pool), so that about rsel * sigma
//                   pools of the row lie above it;
// select            the exact top-k of a candidate list: digit rounds find the
//                   k-th largest score key T and how many keys equal to T are
//                   kept; when more candidates tie at T than are kept, a second
//                   select on the indices keeps the lowest; the kept indices
//                   are sorted ascending (bitonic network in shared memory).
// Candidate and sample loads go through L2 only (__ldcg): other CTAs wrote
// them during this kernel.
#pragma once

#include "topk_row.cuh"

namespace dsa {
namespace cand {

using topk::Group;
using topk::kBins;
using topk::kGT;
using topk::kGW;
using topk::kSmall;

constexpr int kMaxOut = 2048;  // largest topk

struct alignas(16) Smem {
  uint32_t hist[kBins];
  uint32_t small[kSmall];
  uint32_t wsum[2][kGW];
  uint32_t red[2 * kGW];
  uint32_t sel[4];
  uint32_t nsmall;
  uint32_t pad[3];
  uint32_t out[kMaxOut];
};

// A candidate: x = order-preserving score key, y = pool index.
__device__ __forceinline__ uint2 load_cand(const uint2* c, int j) {
  const unsigned long long v = __ldcg(reinterpret_cast<const unsigned long long*>(c) + j);
  return make_uint2(static_cast<uint32_t>(v), static_cast<uint32_t>(v >> 32));
}

__device__ __forceinline__ uint32_t group_sum(const Group& g, uint32_t v, Smem& sm) {
  uint32_t tot;
  topk::group_excl_scan(g, v, sm.wsum[0], &tot);
  g.sync();  // wsum[0] is reused by the next scan
  return tot;
}

// The rsel-th largest composite key (score key, -index) among the G sampled
// scores samp[0 .. G) of one row (sample j is pool j * sigma).  Returns
// (t, p_t): t the score key, p_t the pool index of that sample.  rsel is
// clamped to G.  All threads of the group call it; it ends with a barrier.
__device__ __noinline__ uint2 sample_threshold(const Group& g, Smem& sm, const float* samp, int G, int rsel,
                                               int sigma) {
  const int tid = g.tid;
  int parity = 0;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int j = tid; j < G; j += kGT) {
    const uint32_t k = topk::score_key(__ldcg(samp + j));
    lo = min(lo, k);
    hi = max(hi, k);
  }
  topk::group_minmax(g, lo, hi, sm);
  const uint32_t need = static_cast<uint32_t>(min(rsel, G));
  uint32_t take_eq;
  const uint32_t T = topk::digit_select(
      g, sm, lo, hi, need, G,
      [&](int j, uint32_t& k) {
        k = topk::score_key(__ldcg(samp + j));
        return true;
      },
      &take_eq, parity);
  // among the samples whose key is T, the take_eq-th smallest index: the
  // take_eq-th largest of (G - 1 - j)
  uint32_t vlo = 0xFFFFFFFFu, vhi = 0u;
  for (int j = tid; j < G; j += kGT)
    if (topk::score_key(__ldcg(samp + j)) == T) {
      const uint32_t v = static_cast<uint32_t>(G - 1 - j);
      vlo = min(vlo, v);
      vhi = max(vhi, v);
    }
  topk::group_minmax(g, vlo, vhi, sm);
  uint32_t dummy;
  const uint32_t v = topk::digit_select(
      g, sm, vlo, vhi, take_eq, G,
      [&](int j, uint32_t& k) {
        if (topk::score_key(__ldcg(samp + j)) != T) return false;
        k = static_cast<uint32_t>(G - 1 - j);
        return true;
      },
      &dummy, parity);
  g.sync();
  return make_uint2(T, static_cast<uint32_t>(G - 1 - static_cast<int>(v)) * static_cast<uint32_t>(sigma));
}

// Sorts out[0 .. n) ascending (n <= kMaxOut) in place, padding to a power of
// two with 0xFFFFFFFF.  Ends with a barrier.
__device__ __forceinline__ void bitonic_sort(const Group& g, uint32_t* out, int n) {
  int N = 1;
  while (N < n) N <<= 1;
  for (int j = n + g.tid; j < N; j += kGT) out[j] = 0xFFFFFFFFu;
  g.sync();
  for (int k = 2; k <= N; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = g.tid; i < N / 2; i += kGT) {
        const int a = ((i & ~(j - 1)) << 1) | (i & (j - 1));
        const int b = a + j;
        const bool up = (a & k) == 0;
        const uint32_t x = out[a], y = out[b];
        if ((x > y) == up) {
          out[a] = y;
          out[b] = x;
        }
      }
      g.sync();
    }
  }
}

// Exact top-k of the candidate list c[0 .. count) (count >= topk, every pool
// of the row at or above the threshold is in it); writes orow[0 .. topk) with
// the kept pool indices ascending.  Returns false (nothing written) if the
// kept count does not come out at topk, which a complete list rules out.
__device__ __noinline__ bool select(const Group& g, Smem& sm, const uint2* c, int count, int topk, int32_t* orow) {
  const int tid = g.tid;
  int parity = 0;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int j = tid; j < count; j += kGT) {
    const uint32_t k = load_cand(c, j).x;
    lo = min(lo, k);
    hi = max(hi, k);
  }
  topk::group_minmax(g, lo, hi, sm);
  uint32_t take_eq;
  const uint32_t T = topk::digit_select(
      g, sm, lo, hi, static_cast<uint32_t>(topk), count,
      [&](int j, uint32_t& k) {
        k = load_cand(c, j).x;
        return true;
      },
      &take_eq, parity);
  // how many candidates tie at T, and the span of their indices
  uint32_t eq = 0, ilo = 0xFFFFFFFFu, ihi = 0u;
  for (int j = tid; j < count; j += kGT) {
    const uint2 x = load_cand(c, j);
    if (x.x == T) {
      ++eq;
      ilo = min(ilo, x.y);
      ihi = max(ihi, x.y);
    }
  }
  const uint32_t eq_total = group_sum(g, eq, sm);
  uint32_t idx_cut = 0xFFFFFFFFu;
  if (eq_total > take_eq) {
    // keep the take_eq lowest indices among the ties: the take_eq-th largest of ~idx
    topk::group_minmax(g, ilo, ihi, sm);
    uint32_t dummy;
    const uint32_t v = topk::digit_select(
        g, sm, ~ihi, ~ilo, take_eq, count,
        [&](int j, uint32_t& k) {
          const uint2 x = load_cand(c, j);
          if (x.x != T) return false;
          k = ~x.y;
          return true;
        },
        &dummy, parity);
    idx_cut = ~v;
  }
  // compaction: each thread takes a contiguous stretch of the list
  const int seg = (count + kGT - 1) / kGT;
  const int j0 = min(count, tid * seg), j1 = min(count, j0 + seg);
  uint32_t mine = 0;
  for (int j = j0; j < j1; ++j) {
    const uint2 x = load_cand(c, j);
    mine += x.x > T || (x.x == T && x.y <= idx_cut);
  }
  uint32_t tot;
  uint32_t pos = topk::group_excl_scan(g, mine, sm.wsum[1], &tot);
  if (tot != static_cast<uint32_t>(topk)) {
    g.sync();
    return false;
  }
  for (int j = j0; j < j1; ++j) {
    const uint2 x = load_cand(c, j);
    if (x.x > T || (x.x == T && x.y <= idx_cut)) sm.out[pos++] = x.y;
  }
  g.sync();
  bitonic_sort(g, sm.out, topk);
  for (int j = tid; j < topk; j += kGT) orow[j] = static_cast<int32_t>(sm.out[j]);
  g.sync();
  return true;
}

}  // namespace cand
}  // namespace dsa
