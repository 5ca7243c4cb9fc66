// topk.cu -- per-query top-k of indexer scores.
//
// [SkyRL-1M §1 DSA 真稀疏] each query keeps its highest-scoring pools and the
// selection travels as int32 pool indices.  For query i with n = floor(i/4)
// eligible pools the kernel keeps min(topk, n) of them: every pool whose
// score is larger than the k-th largest score T, plus the lowest-indexed
// pools whose score equals T.  Kept pools are written in ascending order,
// then -1.
//
// Method (one CTA per query row).  Scores map to order-preserving 32-bit
// keys.  The search keeps a key interval [lo, hi] known to contain T and the
// number `need` of keys still to take inside it:
//   1. lo, hi = min, max key of the row.
//   2. A 2048-bin histogram of the keys in [lo, hi], bins linear in key
//      value, locates the bin holding the need-th largest key; keys in higher
//      bins are kept, the interval shrinks to that bin.  Repeat until the bin
//      holds at most kCap keys (or the interval is a single key).
//   3. The bin's keys are compacted into shared memory and an exact radix
//      select on them yields T and the number of ties at T to keep.
//   4. A stable compaction pass writes the kept indices in index order.
// Rows of up to kThreads * kEpt scores keep their keys in registers (one
// read of the row); longer rows re-read the scores (L2) in each pass.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kEpt = 64;                       // keys per thread in the register-resident variant
constexpr int kRegMax = kThreads * kEpt;       // 32768
constexpr int kBins = 2048;
constexpr int kCap = 4096;                     // candidate buffer (keys + indices)

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Smem {
  uint32_t hist[kBins];
  uint32_t cand_key[kCap];
  uint32_t warp_tmp[kWarps + 1];
  uint32_t red[2 * kWarps];
  uint32_t sel[4];
  uint32_t ncand;
};

// Exclusive scan of one value per thread over the block; *total gets the sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* s_warp, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = lane < kWarps ? s_warp[lane] : 0u;
    uint32_t incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < kWarps) s_warp[lane] = incl - w;
    if (lane == kWarps - 1) s_warp[kWarps] = incl;
  }
  __syncthreads();
  const uint32_t r = s_warp[warp] + x - v;
  *total = s_warp[kWarps];
  __syncthreads();
  return r;
}

__device__ __forceinline__ void block_minmax(uint32_t& mn, uint32_t& mx, Smem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    sm.red[warp] = mn;
    sm.red[kWarps + warp] = mx;
  }
  __syncthreads();
  mn = sm.red[0];
  mx = sm.red[kWarps];
  for (int w = 1; w < kWarps; ++w) {
    mn = min(mn, sm.red[w]);
    mx = max(mx, sm.red[kWarps + w]);
  }
  __syncthreads();
}

// bin of key k in [lo, lo + range): floor((k - lo) * nb / range)
__device__ __forceinline__ uint32_t bin_of(uint32_t k, uint32_t lo, uint64_t range, uint32_t nb) {
  return static_cast<uint32_t>((static_cast<uint64_t>(k - lo) * nb) / range);
}

// After a histogram of `nb` bins is in sm.hist, finds the bin b holding the
// need-th largest key.  Writes b, the count above b and the count in b to sm.sel.
__device__ __forceinline__ void find_bin(Smem& sm, uint32_t nb, uint32_t need) {
  // thread t owns bins nb-1-4t .. nb-4-4t (descending)
  const int t = threadIdx.x;
  uint32_t c[4], s = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int b = static_cast<int>(nb) - 1 - 4 * t - q;
    c[q] = b >= 0 ? sm.hist[b] : 0u;
    s += c[q];
  }
  uint32_t tot;
  const uint32_t excl = block_excl_scan(s, sm.warp_tmp, &tot);
  if (excl < need && excl + s >= need) {
    uint32_t cum = excl;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (cum + c[q] >= need) {
        sm.sel[0] = nb - 1 - 4 * t - q;
        sm.sel[1] = cum;
        sm.sel[2] = c[q];
        break;
      }
      cum += c[q];
    }
  }
  __syncthreads();
}

// Exact select among the sm.ncand candidate keys: the need-th largest key T
// and how many candidates equal to T are to be kept.  Radix over (key - lo).
__device__ __forceinline__ void select_candidates(Smem& sm, uint32_t lo, uint32_t hi, uint32_t need, uint32_t* T_out,
                                                  uint32_t* take_eq) {
  const uint32_t nc = sm.ncand;
  uint32_t prefix = 0, pmask = 0;
  const uint32_t span = hi - lo;
  int bits = span == 0 ? 0 : 32 - __clz(span);
  while (bits > 0) {
    const int nb = min(8, bits);
    const int shift = bits - nb;
    for (int b = threadIdx.x; b < 256; b += kThreads) sm.hist[b] = 0u;
    __syncthreads();
    for (uint32_t j = threadIdx.x; j < nc; j += kThreads) {
      const uint32_t x = sm.cand_key[j] - lo;
      if ((x & pmask) == prefix) atomicAdd(&sm.hist[(x >> shift) & ((1u << nb) - 1u)], 1u);
    }
    __syncthreads();
    find_bin(sm, 256, need);
    const uint32_t b = sm.sel[0], above = sm.sel[1];
    need -= above;
    prefix |= b << shift;
    pmask |= ((1u << nb) - 1u) << shift;
    bits -= nb;
    __syncthreads();
  }
  *T_out = lo + prefix;
  *take_eq = need;
}

template <bool kRegs>
__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const float* __restrict__ scores, int64_t ld,
                                                           int64_t row0, int topk, int32_t* __restrict__ out) {
  __shared__ Smem sm;
  const int tid = threadIdx.x;
  const int64_t i = row0 + blockIdx.x;
  const int n = static_cast<int>(i / 4);
  int32_t* orow = out + static_cast<int64_t>(blockIdx.x) * topk;
  if (n <= topk) {
    for (int j = tid; j < topk; j += kThreads) orow[j] = j < n ? j : -1;
    return;
  }
  const float* srow = scores + static_cast<int64_t>(blockIdx.x) * ld;
  // thread tid owns the contiguous segment [beg, end) of the row
  const int seg = kRegs ? kEpt : (n + kThreads - 1) / kThreads;
  const int beg = min(n, tid * seg), end = min(n, beg + seg);
  uint32_t keys[kRegs ? kEpt : 1];
  auto key_at = [&](int e) -> uint32_t {  // e-th element of this thread's segment
    if constexpr (kRegs) {
      return keys[e];
    } else {
      return score_key(__ldg(srow + beg + e));
    }
  };
  const int cnt = end - beg;

  // ---- 1. load (register variant) and min / max
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  if constexpr (kRegs) {
#pragma unroll
    for (int e4 = 0; e4 < kEpt / 4; ++e4) {
      const int e = 4 * e4;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e + 3 < cnt) {
        f = __ldg(reinterpret_cast<const float4*>(srow + beg + e));
      } else {
        if (e < cnt) f.x = __ldg(srow + beg + e);
        if (e + 1 < cnt) f.y = __ldg(srow + beg + e + 1);
        if (e + 2 < cnt) f.z = __ldg(srow + beg + e + 2);
      }
      keys[e] = score_key(f.x);
      keys[e + 1] = score_key(f.y);
      keys[e + 2] = score_key(f.z);
      keys[e + 3] = score_key(f.w);
    }
#pragma unroll
    for (int e = 0; e < kEpt; ++e)
      if (e < cnt) {
        lo = min(lo, keys[e]);
        hi = max(hi, keys[e]);
      }
  } else {
    for (int e = 0; e < cnt; ++e) {
      const uint32_t k = key_at(e);
      lo = min(lo, k);
      hi = max(hi, k);
    }
  }
  block_minmax(lo, hi, sm);

  // ---- 2. narrow [lo, hi] with value histograms
  uint32_t need = static_cast<uint32_t>(topk);
  uint32_t T = lo, take_eq = need;
  bool done = false;
  while (!done) {
    if (lo == hi) {
      T = lo;
      take_eq = need;
      break;
    }
    const uint64_t range = static_cast<uint64_t>(hi - lo) + 1u;
    for (int b = tid; b < kBins; b += kThreads) sm.hist[b] = 0u;
    __syncthreads();
    if constexpr (kRegs) {
#pragma unroll
      for (int e = 0; e < kEpt; ++e)
        if (e < cnt && keys[e] >= lo && keys[e] <= hi) atomicAdd(&sm.hist[bin_of(keys[e], lo, range, kBins)], 1u);
    } else {
      for (int e = 0; e < cnt; ++e) {
        const uint32_t k = key_at(e);
        if (k >= lo && k <= hi) atomicAdd(&sm.hist[bin_of(k, lo, range, kBins)], 1u);
      }
    }
    __syncthreads();
    find_bin(sm, kBins, need);
    const uint32_t b = sm.sel[0], above = sm.sel[1], inbin = sm.sel[2];
    need -= above;
    // keys with bin == b: (k - lo) in [ceil(b*range/nb), ceil((b+1)*range/nb) - 1]
    const uint32_t nlo = lo + static_cast<uint32_t>((static_cast<uint64_t>(b) * range + kBins - 1) / kBins);
    const uint32_t nhi = lo + static_cast<uint32_t>((static_cast<uint64_t>(b + 1) * range + kBins - 1) / kBins) - 1u;
    lo = nlo;
    hi = nhi;
    if (inbin <= kCap) {
      // ---- 3. compact the bin's keys and select exactly among them
      if (tid == 0) sm.ncand = 0;
      __syncthreads();
      if constexpr (kRegs) {
#pragma unroll
        for (int e = 0; e < kEpt; ++e)
          if (e < cnt && keys[e] >= lo && keys[e] <= hi) {
            const uint32_t pos = atomicAdd(&sm.ncand, 1u);
            sm.cand_key[pos] = keys[e];
          }
      } else {
        for (int e = 0; e < cnt; ++e) {
          const uint32_t k = key_at(e);
          if (k >= lo && k <= hi) {
            const uint32_t pos = atomicAdd(&sm.ncand, 1u);
            sm.cand_key[pos] = k;
          }
        }
      }
      __syncthreads();
      select_candidates(sm, lo, hi, need, &T, &take_eq);
      done = true;
    }
    __syncthreads();
  }

  // ---- 4. keys > T, plus the first take_eq keys == T in index order
  uint32_t n_gt = 0, n_eq = 0;
  if constexpr (kRegs) {
#pragma unroll
    for (int e = 0; e < kEpt; ++e)
      if (e < cnt) {
        n_gt += keys[e] > T;
        n_eq += keys[e] == T;
      }
  } else {
    for (int e = 0; e < cnt; ++e) {
      const uint32_t k = key_at(e);
      n_gt += k > T;
      n_eq += k == T;
    }
  }
  uint32_t tot;
  const uint32_t eq_before = block_excl_scan(n_eq, sm.warp_tmp, &tot);
  const uint32_t my_eq = eq_before >= take_eq ? 0u : min(n_eq, take_eq - eq_before);
  uint32_t off = block_excl_scan(n_gt + my_eq, sm.warp_tmp, &tot);
  uint32_t eq_seen = 0;
  if constexpr (kRegs) {
#pragma unroll
    for (int e = 0; e < kEpt; ++e)
      if (e < cnt) {
        const uint32_t k = keys[e];
        if (k > T || (k == T && eq_seen < my_eq)) orow[off++] = beg + e;
        eq_seen += k == T;
      }
  } else {
    for (int e = 0; e < cnt; ++e) {
      const uint32_t k = key_at(e);
      if (k > T || (k == T && eq_seen < my_eq)) orow[off++] = beg + e;
      eq_seen += k == T;
    }
  }
  if (tid == 0)
    for (uint32_t j = tot; j < static_cast<uint32_t>(topk); ++j) orow[j] = -1;  // unreachable for finite scores
}

}  // namespace

cudaError_t launch_topk(const float* scores, int64_t ld, int64_t row0, int nrows, int topk, int32_t* out,
                        const LaunchCtx& ctx) {
  if (nrows <= 0) return cudaSuccess;
  const int64_t n_max = (row0 + nrows - 1) / 4;
  if (n_max <= kRegMax) {
    topk_kernel<true><<<nrows, kThreads, 0, ctx.stream>>>(scores, ld, row0, topk, out);
  } else {
    topk_kernel<false><<<nrows, kThreads, 0, ctx.stream>>>(scores, ld, row0, topk, out);
  }
  return cudaGetLastError();
}

}  // namespace dsa
