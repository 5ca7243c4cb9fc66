// topk.cu -- per-query top-k of indexer scores.
//
// [SkyRL-1M §1 DSA 真稀疏] each query keeps its highest-scoring pools and the
// selection travels as int32 pool indices.  For query i with n = floor(i/4)
// eligible pools the kernel keeps min(topk, n) of them: every pool whose
// score is larger than the k-th largest, plus the lowest-indexed pools tied
// with it.  The kept pools are written in ascending pool order, then -1.
//
// Method: radix select on order-preserving 32-bit keys of the fp32 scores.
// A min/max pass skips the bits all keys share; each further pass builds an
// 8-bit digit histogram of the keys that still match the selected prefix
// (per-warp histograms fed by warp-aggregated increments), and picks the
// digit bin holding the k-th largest key.  A final pass compacts the kept
// indices in index order with two block-wide scans.  One CTA per query row;
// rows of up to kCacheMax scores are staged in shared memory once.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCacheMax = 49152;
constexpr size_t kHistBytes = kWarps * 256 * sizeof(uint32_t);

// Larger float -> larger key; -0 and +0 map to the same key.
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one value per thread; returns the block total in *total.
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
    uint32_t w = lane < kWarps ? s_warp[lane] : 0u;
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

template <bool kCached>
__global__ void __launch_bounds__(kThreads) topk_kernel(const float* __restrict__ scores, int64_t ld, int64_t row0,
                                                        int topk, int32_t* __restrict__ out) {
  extern __shared__ uint32_t smem[];
  uint32_t* hist = smem;                         // [kWarps][256]
  uint32_t* keys = smem + kWarps * 256;          // [n] (kCached)
  __shared__ uint32_t s_warp[kWarps + 1];
  __shared__ uint32_t s_minmax[2 * kWarps];
  __shared__ uint32_t s_sel[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t i = row0 + blockIdx.x;
  const int n = static_cast<int>(i / 4);
  int32_t* orow = out + static_cast<int64_t>(blockIdx.x) * topk;
  if (n <= topk) {
    for (int j = tid; j < topk; j += kThreads) orow[j] = j < n ? j : -1;
    return;
  }
  const float* srow = scores + static_cast<int64_t>(blockIdx.x) * ld;
  auto key_at = [&](int j) -> uint32_t { return kCached ? keys[j] : score_key(__ldg(srow + j)); };

  // ---- pass 0: stage keys, min and max
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  const int n4 = n >> 2;
  for (int j = tid; j < n4; j += kThreads) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(srow) + j);
    const uint32_t k0 = score_key(f.x), k1 = score_key(f.y), k2 = score_key(f.z), k3 = score_key(f.w);
    if (kCached) *reinterpret_cast<uint4*>(keys + 4 * j) = make_uint4(k0, k1, k2, k3);
    kmin = min(kmin, min(min(k0, k1), min(k2, k3)));
    kmax = max(kmax, max(max(k0, k1), max(k2, k3)));
  }
  for (int j = 4 * n4 + tid; j < n; j += kThreads) {
    const uint32_t k = score_key(__ldg(srow + j));
    if (kCached) keys[j] = k;
    kmin = min(kmin, k);
    kmax = max(kmax, k);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    s_minmax[warp] = kmin;
    s_minmax[kWarps + warp] = kmax;
  }
  __syncthreads();
  kmin = s_minmax[0];
  kmax = s_minmax[kWarps];
  for (int w = 1; w < kWarps; ++w) {
    kmin = min(kmin, s_minmax[w]);
    kmax = max(kmax, s_minmax[kWarps + w]);
  }

  // ---- radix passes over the bits below the shared prefix
  uint32_t prefix = kmin, pmask = 0xFFFFFFFFu;
  uint32_t remaining = static_cast<uint32_t>(topk);  // keys still to take among those matching prefix
  if (kmin != kmax) {
    int L = __clz(kmin ^ kmax);
    pmask = L ? (0xFFFFFFFFu << (32 - L)) : 0u;
    prefix = kmin & pmask;
    while (L < 32) {
      const int nb = min(8, 32 - L);
      const int shift = 32 - L - nb;
      const uint32_t dmask = (1u << nb) - 1u;
      for (int b = tid; b < kWarps * 256; b += kThreads) hist[b] = 0u;
      __syncthreads();
      for (int j0 = 0; j0 < n; j0 += kThreads) {
        const int j = j0 + tid;
        const uint32_t k = j < n ? key_at(j) : 0u;
        const bool cand = j < n && (k & pmask) == prefix;
        const uint32_t d = cand ? ((k >> shift) & dmask) : 0xFFFFFFFFu;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        if (cand && lane == __ffs(peers) - 1) hist[warp * 256 + d] += __popc(peers);
      }
      __syncthreads();
      if (tid < 256) {
        uint32_t s = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += hist[w * 256 + tid];
        hist[tid] = s;  // column tid of row 0 is read only by this thread
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t c[8], s = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          c[q] = hist[255 - 8 * lane - q];
          s += c[q];
        }
        uint32_t incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - s;
        const unsigned hit = __ballot_sync(0xffffffffu, excl < remaining && incl >= remaining);
        if (lane == __ffs(hit) - 1) {
          uint32_t cum = excl;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (cum + c[q] >= remaining) {
              s_sel[0] = static_cast<uint32_t>(255 - 8 * lane - q);
              s_sel[1] = cum;
              break;
            }
            cum += c[q];
          }
        }
      }
      __syncthreads();
      const uint32_t bin = s_sel[0], above = s_sel[1];
      remaining -= above;
      prefix |= bin << shift;
      pmask |= dmask << shift;
      L += nb;
      __syncthreads();
    }
  }
  const uint32_t T = prefix;  // key of the k-th largest score

  // ---- final pass: keys > T, plus the first `remaining` keys == T in index order
  int seg = (n + kThreads - 1) / kThreads;
  seg |= 1;  // odd stride: consecutive threads start in different shared-memory banks
  const int beg = min(n, tid * seg), end = min(n, beg + seg);
  uint32_t n_gt = 0, n_eq = 0;
  for (int j = beg; j < end; ++j) {
    const uint32_t k = key_at(j);
    n_gt += k > T;
    n_eq += k == T;
  }
  uint32_t tot;
  const uint32_t eq_before = block_excl_scan(n_eq, s_warp, &tot);
  const uint32_t take_eq = eq_before >= remaining ? 0u : min(n_eq, remaining - eq_before);
  const uint32_t off0 = block_excl_scan(n_gt + take_eq, s_warp, &tot);
  uint32_t off = off0, eq_seen = 0;
  for (int j = beg; j < end; ++j) {
    const uint32_t k = key_at(j);
    if (k > T || (k == T && eq_seen < take_eq)) orow[off++] = j;
    eq_seen += k == T;
  }
  if (tid == 0 && tot != static_cast<uint32_t>(topk)) {
    // cannot happen for finite scores; keep the row well-formed regardless
    for (uint32_t j = tot; j < static_cast<uint32_t>(topk); ++j) orow[j] = -1;
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
    const size_t smem = kHistBytes + static_cast<size_t>(n_max) * sizeof(uint32_t);
    if (dev < 64 && !attr_done[dev]) {
      cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kHistBytes + kCacheMax * sizeof(uint32_t)));
      if (e != cudaSuccess) return e;
      attr_done[dev] = 1;
    }
    topk_kernel<true><<<nrows, kThreads, smem, ctx.stream>>>(scores, ld, row0, topk, out);
  } else {
    topk_kernel<false><<<nrows, kThreads, kHistBytes, ctx.stream>>>(scores, ld, row0, topk, out);
  }
  return cudaGetLastError();
}

}  // namespace dsa
