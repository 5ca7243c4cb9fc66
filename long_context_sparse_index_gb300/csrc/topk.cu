// topk.cu -- per-query top-k of indexer scores.
//
// [SkyRL-1M §1 DSA 真稀疏] each query keeps its highest-scoring pools and the
// selection travels as int32 pool indices.  For query i with n = floor(i/4)
// eligible pools the kernel keeps min(topk, n) of them: every pool whose
// score is larger than the k-th largest score T, plus the lowest-indexed
// pools whose score equals T.  Kept pools are written in ascending order,
// then -1.
//
// Method (one CTA of 512 threads per query row).  Scores map to
// order-preserving 32-bit keys, staged once in shared memory when the row
// fits (n <= kCacheMax), otherwise re-read from the scores in every pass.
//   1. lo, hi = min, max key of the row.
//   2. A 2048-bin histogram of the keys in [lo, hi], bins linear in key
//      value, locates the bin holding the need-th largest key; keys in higher
//      bins are kept and the interval shrinks to that bin.  Repeat until the
//      bin holds at most kCap keys (or the interval is a single key).
//   3. That bin's keys are compacted into shared memory; an exact radix select
//      on them gives T and the number of keys equal to T to keep.
//   4. Round by round over stretches of 2048 keys (4 consecutive keys per
//      thread), one block scan of the packed counts (keys > T, keys == T)
//      gives every thread its output offset: keys > T before it plus
//      min(ties before it, ties to keep).
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPerRound = 4 * kThreads;  // 2048 keys per round
constexpr int kBins = 2048;
constexpr int kCap = 2048;
constexpr int kCacheMax = 49152;        // rows up to 192 KB of keys live in shared memory

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Smem {
  uint32_t hist[kBins];
  uint32_t cand[kCap];
  uint32_t wsum[2][kWarps];
  uint32_t red[2 * kWarps];
  uint32_t sel[4];
  uint32_t ncand;
};

// Exclusive prefix over the block of one value per thread (thread order),
// with one __syncthreads; callers alternate `buf`.  *total gets the sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* buf, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) buf[warp] = x;
  __syncthreads();
  const uint32_t wt = lane < kWarps ? buf[lane] : 0u;
  uint32_t incl = wt;
#pragma unroll
  for (int o = 1; o < kWarps; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t warp_base = __shfl_sync(0xffffffffu, incl - wt, warp);
  *total = __shfl_sync(0xffffffffu, incl, kWarps - 1);
  return warp_base + x - v;
}

// floor((k - lo) * nb / range)
__device__ __forceinline__ uint32_t bin_of(uint32_t k, uint32_t lo, uint64_t range, uint32_t nb) {
  return static_cast<uint32_t>((static_cast<uint64_t>(k - lo) * nb) / range);
}

// With a histogram of nb (<= 2048) bins in sm.hist, finds the bin b holding
// the need-th largest key: sm.sel = {b, count above b, count in b}.
__device__ __forceinline__ void find_bin(Smem& sm, uint32_t nb, uint32_t need, int parity) {
  const int t = threadIdx.x;
  uint32_t c[4], s = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int b = static_cast<int>(nb) - 1 - 4 * t - q;  // descending bins
    c[q] = b >= 0 ? sm.hist[b] : 0u;
    s += c[q];
  }
  uint32_t tot;
  const uint32_t excl = block_excl_scan(s, sm.wsum[parity], &tot);
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

// Keys of elements j .. j+3 (j a multiple of 4); elements >= n read as 0.
template <bool kCached>
__device__ __forceinline__ uint4 keys4(const uint32_t* cache, const float* srow, int j, int n) {
  if constexpr (kCached) {
    return *reinterpret_cast<const uint4*>(cache + j);  // staged with the same padding
  } else {
    if (j + 3 < n) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(srow + j));
      return make_uint4(score_key(f.x), score_key(f.y), score_key(f.z), score_key(f.w));
    }
    uint4 k;
    k.x = j < n ? score_key(__ldg(srow + j)) : 0u;
    k.y = j + 1 < n ? score_key(__ldg(srow + j + 1)) : 0u;
    k.z = j + 2 < n ? score_key(__ldg(srow + j + 2)) : 0u;
    k.w = j + 3 < n ? score_key(__ldg(srow + j + 3)) : 0u;
    return k;
  }
}

template <bool kCached>
__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const float* __restrict__ scores, int64_t ld,
                                                           int64_t row0, int topk, int32_t* __restrict__ out) {
  __shared__ Smem sm;
  extern __shared__ uint4 cache4[];
  uint32_t* cache = reinterpret_cast<uint32_t*>(cache4);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t i = row0 + blockIdx.x;
  const int n = static_cast<int>(i / 4);
  int32_t* orow = out + static_cast<int64_t>(blockIdx.x) * topk;
  if (n <= topk) {
    for (int j = tid; j < topk; j += kThreads) orow[j] = j < n ? j : -1;
    return;
  }
  const float* srow = scores + static_cast<int64_t>(blockIdx.x) * ld;
  const int rounds = (n + kPerRound - 1) / kPerRound;

  // ---- 1. stage keys (cached variant), min and max
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int j = 4 * tid; j < n; j += kPerRound) {
    const uint4 k = keys4<false>(nullptr, srow, j, n);
    if constexpr (kCached) *reinterpret_cast<uint4*>(cache + j) = k;
    const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (j + q < n) {
        lo = min(lo, kk[q]);
        hi = max(hi, kk[q]);
      }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    sm.red[warp] = lo;
    sm.red[kWarps + warp] = hi;
  }
  __syncthreads();
  lo = lane < kWarps ? sm.red[lane] : 0xFFFFFFFFu;
  hi = lane < kWarps ? sm.red[kWarps + lane] : 0u;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  lo = __shfl_sync(0xffffffffu, lo, 0);
  hi = __shfl_sync(0xffffffffu, hi, 0);

  // ---- 2./3. narrow [lo, hi] to the k-th largest key T
  uint32_t need = static_cast<uint32_t>(topk);
  uint32_t T = lo, take_eq = need;
  int parity = 0;
  while (true) {
    if (lo == hi) {
      T = lo;
      take_eq = need;
      break;
    }
    const uint64_t range = static_cast<uint64_t>(hi - lo) + 1u;
    for (int b = tid; b < kBins; b += kThreads) sm.hist[b] = 0u;
    __syncthreads();
    for (int j = 4 * tid; j < n; j += kPerRound) {
      const uint4 k = keys4<kCached>(cache, srow, j, n);
      const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (j + q < n && kk[q] >= lo && kk[q] <= hi) atomicAdd(&sm.hist[bin_of(kk[q], lo, range, kBins)], 1u);
    }
    __syncthreads();
    find_bin(sm, kBins, need, parity);
    parity ^= 1;
    const uint32_t b = sm.sel[0], above = sm.sel[1], inbin = sm.sel[2];
    need -= above;
    // keys in bin b: (k - lo) in [ceil(b*range/nb), ceil((b+1)*range/nb) - 1]
    const uint32_t nlo = lo + static_cast<uint32_t>((static_cast<uint64_t>(b) * range + kBins - 1) / kBins);
    const uint32_t nhi = lo + static_cast<uint32_t>((static_cast<uint64_t>(b + 1) * range + kBins - 1) / kBins) - 1u;
    lo = nlo;
    hi = nhi;
    if (inbin > kCap) continue;
    if (tid == 0) sm.ncand = 0;
    __syncthreads();
    for (int j = 4 * tid; j < n; j += kPerRound) {
      const uint4 k = keys4<kCached>(cache, srow, j, n);
      const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (j + q < n && kk[q] >= lo && kk[q] <= hi) sm.cand[atomicAdd(&sm.ncand, 1u)] = kk[q];
    }
    __syncthreads();
    const uint32_t nc = sm.ncand;
    uint32_t prefix = 0, pmask = 0;
    const uint32_t span = hi - lo;
    int bits = span == 0 ? 0 : 32 - __clz(span);
    while (bits > 0) {
      const int nb = min(8, bits);
      const int shift = bits - nb;
      if (tid < 256) sm.hist[tid] = 0u;
      __syncthreads();
      for (uint32_t j = tid; j < nc; j += kThreads) {
        const uint32_t x = sm.cand[j] - lo;
        if ((x & pmask) == prefix) atomicAdd(&sm.hist[(x >> shift) & ((1u << nb) - 1u)], 1u);
      }
      __syncthreads();
      find_bin(sm, 256, need, parity);
      parity ^= 1;
      need -= sm.sel[1];
      prefix |= sm.sel[0] << shift;
      pmask |= ((1u << nb) - 1u) << shift;
      bits -= nb;
      __syncthreads();
    }
    T = lo + prefix;
    take_eq = need;
    break;
  }
  __syncthreads();

  // ---- 4. stable compaction, one packed block scan per round
  uint32_t gt_base = 0, eq_base = 0;
  for (int m = 0; m < rounds; ++m) {
    const int j = m * kPerRound + 4 * tid;
    const uint4 k = j < n ? keys4<kCached>(cache, srow, j, n) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
    uint32_t gt[4], eq[4], c_gt = 0, c_eq = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bool v = j + q < n;
      gt[q] = v && kk[q] > T;
      eq[q] = v && kk[q] == T;
      c_gt += gt[q];
      c_eq += eq[q];
    }
    uint32_t tot;
    const uint32_t pre = block_excl_scan((c_gt << 16) | c_eq, sm.wsum[parity], &tot);
    parity ^= 1;
    uint32_t gt_before = gt_base + (pre >> 16), eq_before = eq_base + (pre & 0xFFFFu);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (gt[q] || (eq[q] && eq_before < take_eq)) orow[gt_before + min(eq_before, take_eq)] = j + q;
      gt_before += gt[q];
      eq_before += eq[q];
    }
    gt_base += tot >> 16;
    eq_base += tot & 0xFFFFu;
  }
}

}  // namespace

cudaError_t launch_topk(const float* scores, int64_t ld, int64_t row0, int nrows, int topk, int32_t* out,
                        const LaunchCtx& ctx) {
  if (nrows <= 0) return cudaSuccess;
  const int64_t n_max = (row0 + nrows - 1) / 4;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (n_max <= kCacheMax) {
    if (dev < 64 && !attr_done[dev]) {
      cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kCacheMax * sizeof(uint32_t)));
      if (e != cudaSuccess) return e;
      attr_done[dev] = 1;
    }
    // the cache holds the row rounded up to a multiple of 4 keys
    const size_t smem = static_cast<size_t>((n_max + 3) / 4 * 4) * sizeof(uint32_t);
    topk_kernel<true><<<nrows, kThreads, smem, ctx.stream>>>(scores, ld, row0, topk, out);
  } else {
    topk_kernel<false><<<nrows, kThreads, 0, ctx.stream>>>(scores, ld, row0, topk, out);
  }
  return cudaGetLastError();
}

}  // namespace dsa
