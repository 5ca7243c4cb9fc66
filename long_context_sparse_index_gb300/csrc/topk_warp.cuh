// topk_warp.cuh -- one warp per query row: the row's threshold from its
// sampled scores, and its exact top-k from its candidate list, with no block
// or group barriers (warp shuffles, ballots and a small per-warp shared
// buffer), so the 16 epilogue warps of the indexer select 16 rows at once.
//
// [SkyRL-1M §1 DSA 真稀疏] each query keeps its highest-scoring pools as int32
// indices, ties to the lower pool index: pools are ordered by the composite
// key (score desc, index asc).  Keys are the order-preserving 32-bit images of
// the fp32 scores (topk_row.cuh: score_key).
//
// Selections run as passes over data that other CTAs wrote to global memory
// (candidate lists, sampled scores), read through L2 with kU loads in flight
// per lane.  A selection of the need-th largest key takes a min/max pass, then
// rounds that histogram the remaining span into 256 bins and keep the bin
// holding the need-th largest; a bin of at most 32 keys is ranked directly in
// the next pass.  Two selections can share their passes (select2).
//
// threshold   the rsel-th largest composite key among a row's sampled pools;
// topk        the exact top-k (topk <= 512) of a candidate list {key, pool}:
//             T = the topk-th largest key, then one pass files the pools
//             above T and the ties at T; the lowest-index ties complete the
//             row (ranked in shared memory), which is sorted by pool index
//             with a bitonic network held in registers.
#pragma once

#include "topk_row.cuh"

namespace dsa {
namespace wsel {

constexpr int kBins = 256;
constexpr int kMaxK = 512;     // largest topk of the warp path
constexpr int kPer = kMaxK / 32;
constexpr int kMaxTies = 2 * kBins;  // ties at the k-th key ranked in shared memory
constexpr int kU = 16;         // loads in flight per lane in a pass (8 B or less each)

struct alignas(16) Smem {
  union {
    uint32_t hist[2][kBins];  // the selections' histograms
    uint32_t ties[kMaxTies];  // then: the pools tied at the k-th key
  } r1;
  uint32_t out[kMaxK];
  uint32_t small[2][32];
};

__device__ __forceinline__ uint32_t warp_min(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ uint32_t warp_max(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// exclusive prefix over lanes
__device__ __forceinline__ uint32_t warp_excl(uint32_t v, int lane) {
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x - v;
}
__device__ __forceinline__ uint32_t lanes_below(int lane) { return (1u << lane) - 1u; }

// One pass over src[0 .. n): f(j, value, valid) for each element, called by
// all lanes together (warp-uniform), U loads in flight per lane.
template <int U = kU, typename T, typename F>
__device__ __forceinline__ void scan(const T* src, int n, int lane, F&& f) {
  for (int j0 = 0; j0 < n; j0 += 32 * U) {
    T x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + 32 * u + lane;
      x[u] = j < n ? __ldcg(src + j) : T{};
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (j0 + 32 * u >= n) break;
      const int j = j0 + 32 * u + lane;
      f(j, x[u], j < n);
    }
  }
}

// A selection: the need-th largest key in [lo, hi] (at least need keys lie
// there).  On completion val = that key and take = how many keys equal to it
// are among the need largest.
enum : int { kSelHist = 0, kSelSmall = 1, kSelDone = 2 };
struct Sel {
  uint32_t lo, hi, need;
  uint32_t val, take;
  uint32_t n;  // keys collected by a small pass
  int sh;      // digit shift of a histogram pass
  int st;
};

__device__ __forceinline__ Sel sel_make(uint32_t lo, uint32_t hi, uint32_t need) {
  return Sel{lo, hi, need, 0u, 0u, 0u, 0, kSelHist};
}
__device__ __forceinline__ Sel sel_none(uint32_t val) { return Sel{0u, 0u, 0u, val, 0u, 0u, 0, kSelDone}; }

__device__ __forceinline__ void sel_prepare(Sel& s, uint32_t* hist, int lane) {
  if (s.st == kSelHist) {
    if (s.lo == s.hi) {
      s.val = s.lo;
      s.take = s.need;
      s.st = kSelDone;
      return;
    }
    const int bits = 32 - __clz(s.hi - s.lo);
    s.sh = bits > 8 ? bits - 8 : 0;
#pragma unroll
    for (int q = 0; q < kBins / 32; ++q) hist[lane + 32 * q] = 0u;
  } else if (s.st == kSelSmall) {
    s.n = 0u;
  }
}

__device__ __forceinline__ void sel_feed(Sel& s, uint32_t* hist, uint32_t* small, int lane, uint32_t k, bool has) {
  const bool in = has && k >= s.lo && k <= s.hi;
  if (s.st == kSelHist) {
    if (in) atomicAdd(&hist[(k - s.lo) >> s.sh], 1u);
  } else if (s.st == kSelSmall) {
    const uint32_t bal = __ballot_sync(0xffffffffu, in);
    const uint32_t pos = s.n + __popc(bal & lanes_below(lane));
    if (in && pos < 32u) small[pos] = k;
    s.n += __popc(bal);
  }
}

// After a pass; false when the pass's counts contradict the selection (the
// data changed), which the callers treat as a failed row.
__device__ __forceinline__ bool sel_resolve(Sel& s, const uint32_t* hist, const uint32_t* small, int lane) {
  if (s.st == kSelHist) {
    const uint32_t nb = ((s.hi - s.lo) >> s.sh) + 1u;
    // lane L holds bins nb-1-8L .. nb-8-8L, in descending order
    uint32_t c[8], sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int b = static_cast<int>(nb) - 1 - 8 * lane - q;
      c[q] = b >= 0 ? hist[b] : 0u;
      sum += c[q];
    }
    const uint32_t excl = warp_excl(sum, lane);
    const bool mine = excl < s.need && excl + sum >= s.need;
    const uint32_t who = __ballot_sync(0xffffffffu, mine);
    if (who == 0u) return false;
    const int owner = __ffs(who) - 1;
    uint32_t b_sel = 0, above = 0, inbin = 0;
    if (mine) {
      uint32_t cum = excl;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (cum + c[q] >= s.need) {
          b_sel = nb - 1 - 8 * lane - q;
          above = cum;
          inbin = c[q];
          break;
        }
        cum += c[q];
      }
    }
    b_sel = __shfl_sync(0xffffffffu, b_sel, owner);
    above = __shfl_sync(0xffffffffu, above, owner);
    inbin = __shfl_sync(0xffffffffu, inbin, owner);
    s.need -= above;
    const uint32_t nlo = s.lo + (b_sel << s.sh);
    const uint64_t nhi = static_cast<uint64_t>(nlo) + ((1ull << s.sh) - 1ull);
    s.lo = nlo;
    s.hi = nhi < s.hi ? static_cast<uint32_t>(nhi) : s.hi;
    if (s.sh == 0) {
      s.val = s.lo;
      s.take = s.need;
      s.st = kSelDone;
    } else if (inbin <= 32u) {
      s.st = kSelSmall;
    }
  } else if (s.st == kSelSmall) {
    // at most 32 keys in [lo, hi]: one per lane, ranked directly
    const uint32_t n = min(s.n, 32u);
    const uint32_t kj = lane < static_cast<int>(n) ? small[lane] : 0u;
    uint32_t gt = 0, eq = 0;
    for (uint32_t q = 0; q < n; ++q) {
      const uint32_t kq = small[q];
      gt += kq > kj;
      eq += kq == kj;
    }
    const bool hit = lane < static_cast<int>(n) && gt < s.need && s.need <= gt + eq;
    const uint32_t who = __ballot_sync(0xffffffffu, hit);
    if (who == 0u || s.n > 32u) return false;
    const int w = __ffs(who) - 1;
    s.val = __shfl_sync(0xffffffffu, kj, w);
    s.take = s.need - __shfl_sync(0xffffffffu, gt, w);
    s.st = kSelDone;
  }
  return true;
}

// Runs selections s0 and s1 to completion over shared passes: pass(f) makes
// one pass calling f(k0, has0, k1, has1) warp-uniformly per element.
template <typename Pass>
__device__ __forceinline__ bool select2(Smem& sm, int lane, Sel& s0, Sel& s1, Pass&& pass) {
  // each histogram pass narrows the span by 8 bits; a small pass ends it
  for (int round = 0; round < 6; ++round) {
    __syncwarp();
    sel_prepare(s0, sm.r1.hist[0], lane);
    sel_prepare(s1, sm.r1.hist[1], lane);
    if (s0.st == kSelDone && s1.st == kSelDone) return true;
    __syncwarp();
    pass([&](uint32_t k0, bool h0, uint32_t k1, bool h1) {
      sel_feed(s0, sm.r1.hist[0], sm.small[0], lane, k0, h0);
      sel_feed(s1, sm.r1.hist[1], sm.small[1], lane, k1, h1);
    });
    __syncwarp();
    if (!sel_resolve(s0, sm.r1.hist[0], sm.small[0], lane) || !sel_resolve(s1, sm.r1.hist[1], sm.small[1], lane))
      return false;
  }
  return s0.st == kSelDone && s1.st == kSelDone;
}

// The rsel-th largest composite key (score key, -index) among the G sampled
// scores samp[0 .. G) of one row, sample j being pool j * sigma: (t, p_t).
// Should the passes disagree, the threshold lets every pool through, which
// overflows the candidate list and sends the row to the fallback kernel.
__device__ __noinline__ uint2 threshold(Smem& sm, int lane, const float* samp, int G, int rsel, int sigma) {
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  scan(samp, G, lane, [&](int, float v, bool ok) {
    if (ok) {
      const uint32_t k = topk::score_key(v);
      lo = min(lo, k);
      hi = max(hi, k);
    }
  });
  lo = warp_min(lo);
  hi = warp_max(hi);
  const uint2 all = make_uint2(0u, 0x7FFFFFFFu);
  Sel s = sel_make(lo, hi, static_cast<uint32_t>(min(rsel, G))), none = sel_none(0u);
  if (!select2(sm, lane, s, none, [&](auto&& f) {
        scan(samp, G, lane, [&](int, float v, bool ok) { f(topk::score_key(v), ok, 0u, false); });
      }))
    return all;
  const uint32_t T = s.val;
  // among the samples whose key is T, the take-th smallest index: the take-th
  // largest of (G - 1 - j)
  uint32_t vlo = 0xFFFFFFFFu, vhi = 0u;
  scan(samp, G, lane, [&](int j, float v, bool ok) {
    if (ok && topk::score_key(v) == T) {
      vlo = min(vlo, static_cast<uint32_t>(G - 1 - j));
      vhi = max(vhi, static_cast<uint32_t>(G - 1 - j));
    }
  });
  vlo = warp_min(vlo);
  vhi = warp_max(vhi);
  Sel t = sel_make(vlo, vhi, s.take);
  none = sel_none(0u);
  if (!select2(sm, lane, t, none, [&](auto&& f) {
        scan(samp, G, lane, [&](int j, float v, bool ok) {
          f(static_cast<uint32_t>(G - 1 - j), ok && topk::score_key(v) == T, 0u, false);
        });
      }))
    return all;
  return make_uint2(T, static_cast<uint32_t>(G - 1 - static_cast<int>(t.val)) * static_cast<uint32_t>(sigma));
}

// Sorts the kMaxK values x (element r * 32 + lane in x[r]) ascending across
// the warp: bitonic network, partners within a lane's registers (distance >=
// 32) or across lanes (shuffles).
__device__ __forceinline__ void sort_warp(uint32_t (&x)[kPer], int lane) {
#pragma unroll
  for (int k = 2; k <= kMaxK; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        const int rj = j >> 5;
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
          if (r & rj) continue;
          const int e = r * 32 + lane;
          const bool asc = (e & k) == 0;
          const uint32_t a = x[r], b = x[r | rj];
          const bool sw = (a > b) == asc;
          x[r] = sw ? b : a;
          x[r | rj] = sw ? a : b;
        }
      } else {
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
          const int e = r * 32 + lane;
          const bool asc = (e & k) == 0;
          const bool lower = (lane & j) == 0;
          const uint32_t y = __shfl_xor_sync(0xffffffffu, x[r], j);
          x[r] = (asc == lower) ? min(x[r], y) : max(x[r], y);
        }
      }
    }
  }
}

// Exact top-k (topk <= kMaxK) of the candidate list c[0 .. count) ({score
// key, pool}), count >= topk, every pool of the row at or above the threshold
// being in it; writes orow[0 .. topk) ascending.  Returns false (nothing
// written) if the counts do not come out at topk, which a complete list rules
// out.
__device__ __noinline__ bool topk(Smem& sm, int lane, const uint2* c, int count, int topk, int32_t* orow) {
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  scan(c, count, lane, [&](int, const uint2& x, bool v) {
    if (v) {
      lo = min(lo, x.x);
      hi = max(hi, x.x);
    }
  });
  Sel s = sel_make(warp_min(lo), warp_max(hi), static_cast<uint32_t>(topk)), none = sel_none(0u);
  if (!select2(sm, lane, s, none, [&](auto&& f) {
        scan(c, count, lane, [&](int, const uint2& x, bool v) { f(x.x, v, 0u, false); });
      }))
    return false;
  const uint32_t T = s.val, take = s.take, n_gt = static_cast<uint32_t>(topk) - take;
  // one pass: the pools above T, in list order, and the ties at T
  __syncwarp();
  uint32_t ngt = 0, neq = 0;
  scan(c, count, lane, [&](int, const uint2& x, bool v) {
    const bool gt = v && x.x > T, eq = v && x.x == T;
    const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    const uint32_t pg = ngt + __popc(bg & lanes_below(lane)), pe = neq + __popc(be & lanes_below(lane));
    if (gt && pg < static_cast<uint32_t>(kMaxK)) sm.out[pg] = x.y;
    if (eq && pe < static_cast<uint32_t>(kMaxTies)) sm.r1.ties[pe] = x.y;
    ngt += __popc(bg);
    neq += __popc(be);
  });
  if (ngt != n_gt || neq < take) return false;
  __syncwarp();
  uint32_t nk = 0;
  if (neq <= static_cast<uint32_t>(kMaxTies)) {
    // the take lowest pools among the ties (distinct pools: distinct ranks)
    for (uint32_t e0 = 0; e0 < neq; e0 += 32) {
      const uint32_t e = e0 + lane;
      bool keep = false;
      uint32_t p = 0;
      if (e < neq) {
        p = sm.r1.ties[e];
        uint32_t rank = 0;
        for (uint32_t f = 0; f < neq; ++f) rank += sm.r1.ties[f] < p;
        keep = rank < take;
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, keep);
      const uint32_t pos = n_gt + nk + __popc(bal & lanes_below(lane));
      if (keep && pos < static_cast<uint32_t>(kMaxK)) sm.out[pos] = p;
      nk += __popc(bal);
    }
  } else {
    // more ties than the list holds: the take-th smallest pool among them is
    // the take-th largest of ~pool, then a pass keeps the ties up to it
    Sel t = sel_make(0u, 0xFFFFFFFFu, take);
    none = sel_none(0u);
    if (!select2(sm, lane, t, none, [&](auto&& f) {
          scan(c, count, lane, [&](int, const uint2& x, bool v) { f(~x.y, v && x.x == T, 0u, false); });
        }))
      return false;
    const uint32_t cut = ~t.val;
    __syncwarp();
    scan(c, count, lane, [&](int, const uint2& x, bool v) {
      const bool keep = v && x.x == T && x.y <= cut;
      const uint32_t bal = __ballot_sync(0xffffffffu, keep);
      const uint32_t pos = n_gt + nk + __popc(bal & lanes_below(lane));
      if (keep && pos < static_cast<uint32_t>(kMaxK)) sm.out[pos] = x.y;
      nk += __popc(bal);
    });
  }
  if (nk != take) return false;
  __syncwarp();
  uint32_t x[kPer];
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int e = r * 32 + lane;
    x[r] = e < topk ? sm.out[e] : 0xFFFFFFFFu;
  }
  sort_warp(x, lane);
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int e = r * 32 + lane;
    if (e < topk) orow[e] = static_cast<int32_t>(x[r]);
  }
  __syncwarp();
  return true;
}

}  // namespace wsel
}  // namespace dsa
