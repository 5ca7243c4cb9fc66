// indexer.cu -- pooled indexer keys and the causal pooled indexer contraction.
//
// [SkyRL-1M §模型与瓶颈] the indexer scores every query against every earlier
// 4-token key pool; [§1 DSA 真稀疏; Anyscale "稀疏注意力会导致二次成本"] it
// does so one query chunk at a time so the score matrix is never whole.
//
//   Khat_p     = ((k[4p] + k[4p+1]) + (k[4p+2] + k[4p+3])) * 0.25    (fp32)
//   score(i,p) = sum_h w[i,h] * ReLU(q_idx[i,h,:] . Khat_p)
//
// The contraction runs on the tcgen05 tensor cores: per (128-query x
// 256-pool) tile and per head h, one 128x256x128 bf16 MMA chain accumulates
// q_h . [Khat_hi ; Khat_lo] in TMEM (Khat split into a bf16 hi/lo pair so
// the product carries ~16 more mantissa bits than one bf16 rounding), and
// the epilogue warps fold ReLU, the head weight and the sum over heads into
// registers while the next head's MMA runs in the other TMEM buffer.
//
// A chunk with few tiles (early in the sequence, where queries see few pools)
// would leave most SMs idle, so its heads may be split into nsplit equal
// ranges, each tile of each range its own work unit: range s writes its
// partial head-sum to its own slice of the score buffer, and the top-k adds
// the slices in a fixed order.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace {

constexpr int kBM = 128;           // queries per tile (TMEM lanes)
constexpr int kBN = 256;           // pools per tile (TMEM columns per buffer)
constexpr int kDi = 64;            // indexer head dim
constexpr int kAStages = 4;
constexpr int kBStages = 2;
constexpr uint32_t kABytes = kBM * kDi * 2;        // 16 KB: q_idx tile of one head
constexpr uint32_t kBHalf = kBN * kDi * 2;         // 32 KB: Khat hi (or lo) tile
constexpr uint32_t kBBytes = 2 * kBHalf;           // 64 KB
constexpr int kEpiWarps = 16;                      // 4 TMEM lane quarters x 4 column quarters
constexpr int kEpiCols = kBN / 4;                  // 64 columns per epilogue thread
constexpr int kThreads = 32 * (2 + kEpiWarps);     // TMA warp, MMA warp, 16 epilogue warps
constexpr uint32_t kTmemCols = 512;                // 2 accumulators x 256 columns
constexpr uint32_t kBarOff = kBStages * kBBytes + kAStages * kABytes;
constexpr size_t kSmemBytes = 1024 + kBarOff + 256;

struct IndexerArgs {
  const float* w;
  float* scores;
  int64_t ld;
  int64_t split_stride;  // floats between the partial-sum slices
  int64_t row0;
  int nrows;
  int Hi;
  int nsplit;            // head ranges (1, 2 or 4)
  int nqb;
  int npb_max;
  unsigned* status;
  uint64_t limit_ns;
  int inject;
};

__device__ __forceinline__ int pool_tiles_of(const IndexerArgs& a, int qb) {
  const int64_t end = min(a.row0 + static_cast<int64_t>(qb + 1) * kBM, a.row0 + a.nrows);
  const int64_t n = (end - 1) / 4;  // pools eligible for the last query of the block
  return static_cast<int>((n + kBN - 1) / kBN);
}

__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                   const IndexerArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-B swizzle atoms need 1024-B alignment
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sB = base;
  const uint32_t sA = base + kBStages * kBBytes;
  const uint32_t sBar = base + kBarOff;
  const uint32_t bar_a_full = sBar, bar_a_empty = sBar + 32, bar_b_full = sBar + 64, bar_b_empty = sBar + 80;
  const uint32_t bar_acc_full = sBar + 96, bar_acc_empty = sBar + 112, bar_drain = sBar + 128;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kBarOff + 136);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kBarOff + 140);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(bar_a_full + 8 * s, 1);
      mbar_init(bar_a_empty + 8 * s, 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(bar_b_full + 8 * s, 1);
      mbar_init(bar_b_empty + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_acc_full + 8 * s, 1);
      mbar_init(bar_acc_empty + 8 * s, kEpiWarps);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&q_map);
    tma_prefetch_map(&k_map);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = a.nqb * a.npb_max * a.nsplit;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int as = 0, bs = 0;
      uint32_t aph = 0, bph = 0;
      uint32_t a_armed = 0, b_armed = 0, a_par = 0, b_par = 0;  // bit s: stage armed / parity armed
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int hs = t % a.nsplit, qb = (t / a.nsplit) % a.nqb, pb = t / a.nsplit / a.nqb;
        if (pb >= pool_tiles_of(a, qb)) continue;
        if (!mbar_wait(bar_b_empty + 8 * bs, bph ^ 1, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        if (!a.inject) {
          mbar_arrive_expect_tx(bar_b_full + 8 * bs, kBBytes);
          tma_load_2d(sB + bs * kBBytes, &k_map, bar_b_full + 8 * bs, 0, pb * kBN);
          tma_load_2d(sB + bs * kBBytes + kBHalf, &k_map, bar_b_full + 8 * bs, kDi, pb * kBN);
          b_armed |= 1u << bs;
          b_par = (b_par & ~(1u << bs)) | (bph << bs);
        }
        if (++bs == kBStages) {
          bs = 0;
          bph ^= 1;
        }
        const int qrow = static_cast<int>(a.row0) + qb * kBM;
        for (int h = hs * a.Hi / a.nsplit; h < (hs + 1) * a.Hi / a.nsplit; ++h) {
          if (!mbar_wait(bar_a_empty + 8 * as, aph ^ 1, a.limit_ns, abort_flag)) {
            ok = false;
            break;
          }
          if (!a.inject) {
            mbar_arrive_expect_tx(bar_a_full + 8 * as, kABytes);
            tma_load_3d(sA + as * kABytes, &q_map, bar_a_full + 8 * as, 0, h, qrow);
            a_armed |= 1u << as;
            a_par = (a_par & ~(1u << as)) | (aph << as);
          }
          if (++as == kAStages) {
            as = 0;
            aph ^= 1;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, kStatusTimeout);
      }
      // every copy this thread issued lands before the CTA may exit
      for (int s = 0; s < kAStages; ++s)
        if (a_armed & (1u << s)) mbar_wait(bar_a_full + 8 * s, (a_par >> s) & 1u, a.limit_ns, nullptr);
      for (int s = 0; s < kBStages; ++s)
        if (b_armed & (1u << s)) mbar_wait(bar_b_full + 8 * s, (b_par >> s) & 1u, a.limit_ns, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16_f32(kBM, kBN);
      int as = 0, bs = 0, cs = 0;
      uint32_t aph = 0, bph = 0, cph = 0;
      bool ok = true, issued = false;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int hs = t % a.nsplit, qb = (t / a.nsplit) % a.nqb, pb = t / a.nsplit / a.nqb;
        if (pb >= pool_tiles_of(a, qb)) continue;
        if (!mbar_wait(bar_b_full + 8 * bs, bph, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t b_hi = sB + bs * kBBytes, b_lo = b_hi + kBHalf;
        for (int h = hs * a.Hi / a.nsplit; h < (hs + 1) * a.Hi / a.nsplit; ++h) {
          if (!mbar_wait(bar_a_full + 8 * as, aph, a.limit_ns, abort_flag) ||
              !mbar_wait(bar_acc_empty + 8 * cs, cph ^ 1, a.limit_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + cs * kBN;
          const uint32_t aa = sA + as * kABytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = umma_desc_sw128(aa + (kk & 3) * 32);
            const uint64_t bd = umma_desc_sw128((kk < 4 ? b_hi : b_lo) + (kk & 3) * 32);
            umma_bf16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
          }
          issued = true;
          umma_commit(bar_a_empty + 8 * as);
          umma_commit(bar_acc_full + 8 * cs);
          if (++as == kAStages) {
            as = 0;
            aph ^= 1;
          }
          if (++cs == 2) {
            cs = 0;
            cph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(bar_b_empty + 8 * bs);
        if (++bs == kBStages) {
          bs = 0;
          bph ^= 1;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, kStatusTimeout);
      }
      if (issued) {  // all MMAs done before TMEM and shared memory are released
        umma_commit(bar_drain);
        mbar_wait(bar_drain, 0, a.limit_ns, nullptr);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    // Warp w (2..17) reads TMEM lanes 32*(w%4).. (its hardware lane quarter)
    // and columns 64*((w-2)/4).. of each accumulator: one query row and 64
    // pools per thread.  16 warps keep several TMEM loads in flight per SM
    // sub-partition while others compute.
    const int ew = warp - 2;
    const int lq = warp & 3;
    const int cq = ew >> 2;
    int cs = 0;
    uint32_t cph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const int hs = t % a.nsplit, qb = (t / a.nsplit) % a.nqb, pb = t / a.nsplit / a.nqb;
      if (pb >= pool_tiles_of(a, qb)) continue;
      const int h0 = hs * a.Hi / a.nsplit, h1 = (hs + 1) * a.Hi / a.nsplit;
      const int64_t row = a.row0 + static_cast<int64_t>(qb) * kBM + lq * 32 + lane;
      const bool valid = row < a.row0 + a.nrows;
      const float* wrow = a.w + (valid ? row : a.row0) * a.Hi;
      float2 acc[kEpiCols / 2];
#pragma unroll
      for (int j = 0; j < kEpiCols / 2; ++j) acc[j] = make_float2(0.f, 0.f);
      // the head weight is fetched one head ahead so its load latency hides
      // behind the previous head's epilogue
      float w_next = valid && h0 < h1 ? __ldg(wrow + h0) : 0.f;
      for (int h = h0; h < h1; ++h) {
        const float wv = w_next;
        if (h + 1 < h1) w_next = valid ? __ldg(wrow + h + 1) : 0.f;
        if (!mbar_wait(bar_acc_full + 8 * cs, cph, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float2 w2 = make_float2(wv, wv);
        const uint32_t taddr = tmem + (static_cast<uint32_t>(lq * 32) << 16) + cs * kBN + cq * kEpiCols;
#pragma unroll
        for (int c = 0; c < kEpiCols / 16; ++c) {
          uint32_t r[16];
          tmem_ld16(taddr + c * 16, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 x = make_float2(fmaxf(__uint_as_float(r[2 * j]), 0.f), fmaxf(__uint_as_float(r[2 * j + 1]), 0.f));
            acc[c * 8 + j] = __ffma2_rn(w2, x, acc[c * 8 + j]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acc_empty + 8 * cs);
        if (++cs == 2) {
          cs = 0;
          cph ^= 1;
        }
      }
      if (!ok) break;
      // the preceding top-k may still be reading the score buffer
      pdl_wait();
      if (valid) {
        float4* dst = reinterpret_cast<float4*>(a.scores + hs * a.split_stride + (row - a.row0) * a.ld +
                                                static_cast<int64_t>(pb) * kBN + cq * kEpiCols);
#pragma unroll
        for (int c = 0; c < kEpiCols / 4; ++c)
          dst[c] = make_float4(acc[2 * c].x, acc[2 * c].y, acc[2 * c + 1].x, acc[2 * c + 1].y);
      }
    }
    if (!ok) {
      *abort_flag = 1;
      record_status(a.status, kStatusTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();  // all scores of this CTA are written
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Khat in fp32 with the fixed summation order, then split into bf16 hi + lo.
// One thread per (pool, 8-dim group); Di = 64.
__global__ void pool_keys_kernel(const __nv_bfloat16* __restrict__ k_idx, int64_t P,
                                 __nv_bfloat16* __restrict__ khat2) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t p = t >> 3;
  const int g = static_cast<int>(t & 7);
  if (p >= P) return;
  const uint4* src = reinterpret_cast<const uint4*>(k_idx + 4 * p * kDi) + g;
  uint4 rows[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) rows[r] = src[r * (kDi / 8)];
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float v[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t word = (&rows[r].x)[e];
      v[r][0] = __uint_as_float(word << 16);
      v[r][1] = __uint_as_float(word & 0xFFFF0000u);
    }
    float kh[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float s01 = __fadd_rn(v[0][c], v[1][c]);
      const float s23 = __fadd_rn(v[2][c], v[3][c]);
      kh[c] = __fmul_rn(__fadd_rn(s01, s23), 0.25f);
    }
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(kh[0], kh[1]);
    const float2 hf = __bfloat1622float2(h2);
    const __nv_bfloat162 l2 = __floats2bfloat162_rn(__fsub_rn(kh[0], hf.x), __fsub_rn(kh[1], hf.y));
    hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
    lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
  }
  uint4* dst = reinterpret_cast<uint4*>(khat2 + p * (2 * kDi));
  dst[g] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  dst[8 + g] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

}  // namespace

size_t indexer_smem_bytes() { return kSmemBytes; }

cudaError_t launch_pool_keys(const void* k_idx, int64_t P, void* khat2, const LaunchCtx& ctx) {
  if (P <= 0) return cudaSuccess;
  const int64_t threads = P * 8;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  pool_keys_kernel<<<static_cast<unsigned>(grid), block, 0, ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(k_idx), P, static_cast<__nv_bfloat16*>(khat2));
  return cudaGetLastError();
}

cudaError_t launch_indexer(const CUtensorMap& q_map, const CUtensorMap& khat_map, const float* w, float* scores,
                           int64_t ld, int nsplit, int64_t split_stride, int64_t row0, int nrows, int Hi,
                           const LaunchCtx& ctx) {
  IndexerArgs a;
  a.w = w;
  a.scores = scores;
  a.ld = ld;
  a.split_stride = split_stride;
  a.row0 = row0;
  a.nrows = nrows;
  a.Hi = Hi;
  a.nsplit = nsplit;
  a.nqb = (nrows + kBM - 1) / kBM;
  a.npb_max = static_cast<int>(((row0 + nrows - 1) / 4 + kBN - 1) / kBN);
  a.status = ctx.status;
  a.limit_ns = ctx.wait_limit_ns;
  a.inject = ctx.inject_timeout;
  if (a.npb_max <= 0) return cudaSuccess;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(indexer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done[dev] = 1;
  }
  const int ntiles = a.nqb * a.npb_max * a.nsplit;
  const int grid = ntiles < ctx.num_sms ? ntiles : ctx.num_sms;
  return launch_ex(ctx, indexer_kernel, dim3(grid), dim3(kThreads), kSmemBytes, q_map, khat_map, a);
}

}  // namespace dsa
