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
// select_value  the need-th largest of N keys given by a getter: a min/max
//               pass, then rounds that histogram the remaining span into 256
//               bins and keep the bin holding the need-th largest; a bin of
//               at most 32 keys is ranked directly.
// threshold     the rsel-th largest composite key among a row's sampled pools.
// topk          the exact top-k of a candidate list (topk <= 512), sorted by
//               pool index with a bitonic network held in registers.
// Global loads go through L2 only (__ldcg): other CTAs wrote the data during
// this kernel.
#pragma once

#include "topk_row.cuh"

namespace dsa {
namespace wsel {

constexpr int kBins = 256;
constexpr int kMaxK = 512;  // largest topk of the warp path
constexpr int kPer = kMaxK / 32;

struct alignas(16) Smem {
  uint32_t hist[kBins];
  uint32_t small[32];
  uint32_t out[kMaxK];
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

// The need-th largest of the keys get(j, &k) yields for j < N (false: no key
// at j).  Every key lies in [lo, hi] and at least `need` keys do.  Returns
// it; *take_eq = how many keys equal to it are among the need largest.
template <typename Get>
__device__ __forceinline__ uint32_t select_value(Smem& sm, int lane, int N, uint32_t lo, uint32_t hi, uint32_t need,
                                                 Get&& get, uint32_t* take_eq) {
  while (true) {
    if (lo == hi) {
      *take_eq = need;
      return lo;
    }
    const uint32_t span = hi - lo;
    const int bits = 32 - __clz(span);
    const int sh = bits > 8 ? bits - 8 : 0;
    const uint32_t nb = (span >> sh) + 1u;
#pragma unroll
    for (int q = 0; q < kBins / 32; ++q) sm.hist[lane + 32 * q] = 0u;
    __syncwarp();
    for (int j = lane; j < N; j += 32) {
      uint32_t k;
      if (get(j, k) && k >= lo && k <= hi) atomicAdd(&sm.hist[(k - lo) >> sh], 1u);
    }
    __syncwarp();
    // lane L holds bins nb-1-8L .. nb-8-8L, in descending order
    uint32_t c[8], s = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int b = static_cast<int>(nb) - 1 - 8 * lane - q;
      c[q] = b >= 0 ? sm.hist[b] : 0u;
      s += c[q];
    }
    const uint32_t excl = warp_excl(s, lane);
    const bool mine = excl < need && excl + s >= need;
    const int owner = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    uint32_t b_sel = 0, above = 0, inbin = 0;
    if (mine) {
      uint32_t cum = excl;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (cum + c[q] >= need) {
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
    need -= above;
    const uint32_t nlo = lo + (b_sel << sh);
    const uint64_t nhi = static_cast<uint64_t>(nlo) + ((1ull << sh) - 1ull);
    lo = nlo;
    hi = nhi < hi ? static_cast<uint32_t>(nhi) : hi;
    __syncwarp();
    if (sh == 0) {
      *take_eq = need;
      return lo;
    }
    if (inbin > 32u) continue;
    // at most 32 keys left in [lo, hi]: one per lane, ranked directly
    uint32_t n = 0;
    for (int j0 = 0; j0 < N; j0 += 32) {
      const int j = j0 + lane;
      uint32_t k = 0;
      const bool in = j < N && get(j, k) && k >= lo && k <= hi;
      const uint32_t bal = __ballot_sync(0xffffffffu, in);
      if (in) sm.small[n + __popc(bal & ((1u << lane) - 1u))] = k;
      n += __popc(bal);
    }
    __syncwarp();
    const uint32_t kj = lane < static_cast<int>(n) ? sm.small[lane] : 0u;
    uint32_t gt = 0, eq = 0;
    for (uint32_t q = 0; q < n; ++q) {
      const uint32_t kq = sm.small[q];
      gt += kq > kj;
      eq += kq == kj;
    }
    const bool hit = lane < static_cast<int>(n) && gt < need && need <= gt + eq;
    const int who = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
    const uint32_t T = __shfl_sync(0xffffffffu, kj, who);
    *take_eq = need - __shfl_sync(0xffffffffu, gt, who);
    __syncwarp();
    return T;
  }
}

// The rsel-th largest composite key (score key, -index) among the G sampled
// scores samp[0 .. G) of one row, sample j being pool j * sigma: (t, p_t).
__device__ __noinline__ uint2 threshold(Smem& sm, int lane, const float* samp, int G, int rsel, int sigma) {
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int j = lane; j < G; j += 32) {
    const uint32_t k = topk::score_key(__ldcg(samp + j));
    lo = min(lo, k);
    hi = max(hi, k);
  }
  lo = warp_min(lo);
  hi = warp_max(hi);
  uint32_t take_eq;
  const uint32_t T = select_value(sm, lane, G, lo, hi, static_cast<uint32_t>(min(rsel, G)),
                                  [&](int j, uint32_t& k) {
                                    k = topk::score_key(__ldcg(samp + j));
                                    return true;
                                  },
                                  &take_eq);
  // among the samples whose key is T, the take_eq-th smallest index: the
  // take_eq-th largest of (G - 1 - j)
  uint32_t vlo = 0xFFFFFFFFu, vhi = 0u;
  for (int j = lane; j < G; j += 32)
    if (topk::score_key(__ldcg(samp + j)) == T) {
      vlo = min(vlo, static_cast<uint32_t>(G - 1 - j));
      vhi = max(vhi, static_cast<uint32_t>(G - 1 - j));
    }
  vlo = warp_min(vlo);
  vhi = warp_max(vhi);
  uint32_t dummy;
  const uint32_t v = select_value(sm, lane, G, vlo, vhi, take_eq,
                                  [&](int j, uint32_t& k) {
                                    if (topk::score_key(__ldcg(samp + j)) != T) return false;
                                    k = static_cast<uint32_t>(G - 1 - j);
                                    return true;
                                  },
                                  &dummy);
  return make_uint2(T, static_cast<uint32_t>(G - 1 - static_cast<int>(v)) * static_cast<uint32_t>(sigma));
}

__device__ __forceinline__ uint2 load_cand(const uint2* c, int j) {
  const unsigned long long v = __ldcg(reinterpret_cast<const unsigned long long*>(c) + j);
  return make_uint2(static_cast<uint32_t>(v), static_cast<uint32_t>(v >> 32));
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

// Exact top-k (topk <= kMaxK) of the candidate list c[0 .. count), count >=
// topk, every pool of the row at or above the threshold being in it; writes
// orow[0 .. topk) ascending.  Returns false (nothing written) if the kept
// count does not come out at topk, which a complete list rules out.
__device__ __noinline__ bool topk(Smem& sm, int lane, const uint2* c, int count, int topk, int32_t* orow) {
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int j = lane; j < count; j += 32) {
    const uint32_t k = load_cand(c, j).x;
    lo = min(lo, k);
    hi = max(hi, k);
  }
  lo = warp_min(lo);
  hi = warp_max(hi);
  uint32_t take_eq;
  const uint32_t T = select_value(sm, lane, count, lo, hi, static_cast<uint32_t>(topk),
                                  [&](int j, uint32_t& k) {
                                    k = load_cand(c, j).x;
                                    return true;
                                  },
                                  &take_eq);
  uint32_t eq = 0, ilo = 0xFFFFFFFFu, ihi = 0u;
  for (int j = lane; j < count; j += 32) {
    const uint2 x = load_cand(c, j);
    if (x.x == T) {
      ++eq;
      ilo = min(ilo, x.y);
      ihi = max(ihi, x.y);
    }
  }
  eq = warp_sum(eq);
  uint32_t idx_cut = 0xFFFFFFFFu;
  if (eq > take_eq) {
    // keep the take_eq lowest indices among the ties: the take_eq-th largest of ~idx
    ilo = warp_min(ilo);
    ihi = warp_max(ihi);
    uint32_t dummy;
    idx_cut = ~select_value(sm, lane, count, ~ihi, ~ilo, take_eq,
                            [&](int j, uint32_t& k) {
                              const uint2 x = load_cand(c, j);
                              if (x.x != T) return false;
                              k = ~x.y;
                              return true;
                            },
                            &dummy);
  }
  // compaction in list order (ballots), then a sort by pool index
  uint32_t n = 0;
  for (int j0 = 0; j0 < count; j0 += 32) {
    const int j = j0 + lane;
    bool keep = false;
    uint32_t p = 0;
    if (j < count) {
      const uint2 x = load_cand(c, j);
      keep = x.x > T || (x.x == T && x.y <= idx_cut);
      p = x.y;
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, keep);
    const uint32_t pos = n + __popc(bal & ((1u << lane) - 1u));
    if (keep && pos < static_cast<uint32_t>(kMaxK)) sm.out[pos] = p;
    n += __popc(bal);
  }
  __syncwarp();
  if (n != static_cast<uint32_t>(topk)) return false;
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
