// probes.cu -- measurement kernels for the ceilings the attention kernels
// meet when their working set sits in L2 (no part of the layer's arithmetic).
//
// The sparse attention gathers 1 KB key pools (four 256-byte K or V rows)
// chosen by the selection, and the backward adds each (query, key) pair's
// dK/dV rows into fp32 accumulators with 16-byte vector reductions, one
// pool's four rows x 128 bytes per warp instruction.  At S = 131072 both K/V
// (64 MiB) and the accumulators (128 MiB) are L2-sized, so HBM bandwidth does
// not bound those kernels; these probes measure the L2 rates of the same
// access shapes on the caller's buffer:
//   kind 0  streaming 16-byte loads over the whole buffer, repeated
//   kind 1  random 1 KB blocks, each read by one warp (two 16-byte loads a lane)
//   kind 2  red.global.add.v4.f32 on random 2 KB blocks (4 rows x 512 B):
//           each warp instruction adds 128 bytes to each of the 4 rows
//   kind 3  bulk reductions (cp.reduce.async.bulk .add.f32) from shared
//           memory: one 2 KB block per operation, random blocks, up to 8
//           operations in flight per warp
//   kind 4  the same with 512-byte operations (one row each)
//   kind 5  red.v4 with 2 rows x 256 B per warp instruction (two rows of a block)
//   kind 6  red.v4 with 8 rows x 64 B (four rows of each of two blocks)
//   kind 7  red.v4 with 16 rows x 32 B (four blocks; the shape of reductions
//           issued straight from mma.sync accumulator fragments)
//   kind 8  kind 2 from half of each CTA's warps and kind 3 from the other
//           half at the same time (do the two issue paths add up?)
// All report bytes moved (read, or added) per second.
//
// dsa_measure_fold times the indexer's accumulator handoff in isolation: the
// same 19-warp layout (one MMA issuer, two idle control warps, 16 epilogue
// warps, so the same 96-register cap), a chain of 8 tcgen05.mma (M 128,
// N 256, K 16: one head of the hi/lo contraction) into one of two tensor-
// memory accumulators per head, and each epilogue warp loading its lane
// quarter's 64 columns 16 at a time and folding them (ReLU, then a packed
// FMA into 64 fp32 sums) before the accumulator is released.
//
// dsa_measure_umma times the tensor core on the attention's product shape:
// one thread per CTA issues back-to-back groups of 8 chained tcgen05.mma
// (kind::f16, bf16 operands from 128-byte swizzled shared memory, M = 128,
// K = 16 each, N given) into a tensor-memory accumulator, and reports the
// issuing thread's clock cycles per instruction, with `issuers` CTAs (each
// its own issuer) resident on every SM.
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "../../include/dsa.h"
#include "dsa_device.cuh"

namespace dsa {
void set_last_error(const std::string& msg);
}

namespace {

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  // a 32-bit integer hash (xorshift-multiply rounds) picking pseudo-random blocks
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

__global__ void probe_stream_kernel(const float4* __restrict__ buf, int64_t n4, int iters, float* sink) {
  float acc = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int it = 0; it < iters; ++it)
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n4; j += stride) {
      const float4 v = __ldcg(buf + j);
      acc += v.x + v.y + v.z + v.w;
    }
  if (acc == 1.2345f) sink[0] = acc;  // a data-dependent store (practically never taken) keeps the loads
}

__global__ void probe_gather_kernel(const uint4* __restrict__ buf, uint32_t nblocks, int per_warp, float* sink) {
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  uint32_t acc = 0;
  for (int it = 0; it < per_warp; it += 4) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {  // four blocks in flight per warp
      const uint32_t b = mix32(warp * 0x9E3779B9u + static_cast<uint32_t>(it + u)) % nblocks;
      const uint4* src = buf + static_cast<int64_t>(b) * 64 + lane;
      v[2 * u] = __ldcg(src);
      v[2 * u + 1] = __ldcg(src + 32);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  if (acc == 0x12345678u) sink[0] = 1.f;
}

__global__ void probe_red_kernel(float* __restrict__ buf, uint32_t nblocks, int per_warp) {
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (int it = 0; it < per_warp; ++it) {
    const uint32_t h = mix32(warp * 0x9E3779B9u + static_cast<uint32_t>(it));
    const uint32_t b = h % nblocks;
    const int jj = static_cast<int>((h >> 28) & 3u);  // 32-dim block of the rows
    float* dst = buf + static_cast<int64_t>(b) * 512 + (lane >> 3) * 128 + 32 * jj + 4 * (lane & 7);
    dsa::red_add_v4(dst, 1.f, 1.f, 1.f, 1.f);
  }
}

// red.v4 with R rows per warp instruction, 512 / R bytes of each: the rows
// are rows of R / 4 random 2 KB blocks (R >= 4), or R consecutive rows of one
// random block (R = 2).
template <int R>
__global__ void probe_red_shape_kernel(float* __restrict__ buf, uint32_t nblocks, int per_warp) {
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int kTpr = 32 / R;        // lanes per row
  constexpr int kChunks = 128 / (4 * kTpr);  // chunks of 4 * kTpr floats in a 128-float row
  const int row = lane / kTpr, c = lane % kTpr;
  for (int it = 0; it < per_warp; ++it) {
    const uint32_t h = mix32(warp * 0x9E3779B9u + static_cast<uint32_t>(it));
    const int jj = static_cast<int>((h >> 24) % kChunks);
    uint32_t b;
    int r;
    if (R >= 4) {
      b = mix32(h + static_cast<uint32_t>(row >> 2) * 0x85EBCA6Bu) % nblocks;
      r = row & 3;
    } else {
      b = h % nblocks;
      r = static_cast<int>((h >> 20) & 2u) + row;  // rows 0-1 or 2-3
    }
    float* dst = buf + static_cast<int64_t>(b) * 512 + r * 128 + jj * 4 * kTpr + 4 * c;
    dsa::red_add_v4(dst, 1.f, 1.f, 1.f, 1.f);
  }
}

// Warp w's lane 0 adds its 2 KB shared-memory block of ones into random
// 2 KB blocks of buf (op_bytes per bulk operation), keeping at most 8 bulk
// groups in flight; all complete before the CTA exits.
__global__ void probe_bulk_red_kernel(float* __restrict__ buf, uint32_t nblocks, int per_warp, int op_bytes) {
  __shared__ __align__(128) float src[8][512];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = lane; e < 512; e += 32) src[wib][e] = 1.f;
  __syncwarp();
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  if (lane == 0) {
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t s = dsa::smem_u32(src[wib]);
    const int nops = 2048 / op_bytes;
    for (int it = 0; it < per_warp; ++it) {
      const uint32_t b = mix32(warp * 0x9E3779B9u + static_cast<uint32_t>(it)) % nblocks;
      float* dst = buf + static_cast<int64_t>(b) * 512;
      for (int o = 0; o < nops; ++o)
        asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                         dst + o * (op_bytes / 4)),
                     "r"(s + o * op_bytes), "r"(op_bytes)
                     : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 8;" ::: "memory");
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
}

// Warps 0-3 of each 8-warp CTA issue kind 2's reductions (red_iters each),
// warps 4-7 kind 3's bulk 2 KB reductions (bulk_iters each, lane 0, at most
// 8 in flight), all at once.
__global__ void probe_red_mix_kernel(float* __restrict__ buf, uint32_t nblocks, int red_iters, int bulk_iters) {
  __shared__ __align__(128) float src[4][512];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (wib < 4) {
    for (int it = 0; it < red_iters; ++it) {
      const uint32_t h = mix32(warp * 0x9E3779B9u + static_cast<uint32_t>(it));
      const uint32_t b = h % nblocks;
      const int jj = static_cast<int>((h >> 28) & 3u);
      float* dst = buf + static_cast<int64_t>(b) * 512 + (lane >> 3) * 128 + 32 * jj + 4 * (lane & 7);
      dsa::red_add_v4(dst, 1.f, 1.f, 1.f, 1.f);
    }
    return;
  }
  float* mine = src[wib - 4];
  for (int e = lane; e < 512; e += 32) mine[e] = 1.f;
  __syncwarp();
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  if (lane == 0) {
    const uint32_t s = dsa::smem_u32(mine);
    for (int it = 0; it < bulk_iters; ++it) {
      const uint32_t b = mix32(warp * 0x85EBCA6Bu + static_cast<uint32_t>(it)) % nblocks;
      asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                       buf + static_cast<int64_t>(b) * 512),
                   "r"(s), "r"(2048)
                   : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 8;" ::: "memory");
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  __syncwarp();
}

// ---------------------------------------------------------------- tensor-core issue probe
constexpr int kUmmaGroup = 8;  // chained MMAs per group (accumulate after the first)

template <int N>
__global__ void __launch_bounds__(128, 3) probe_umma_kernel(int groups, uint64_t limit_ns, unsigned long long* cycles,
                                                          int* failed) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dsa::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* g = smem_raw + (base - raw);
  const uint32_t sA = base, sB = base + 16384;  // A: 128 rows x 128 B; B: N rows x 128 B
  const uint32_t bar = sB + N * 128;
  uint32_t* slot = reinterpret_cast<uint32_t*>(g + 16384 + N * 128 + 64);
  // small nonzero operands (bf16 1/64 .. 8/64, exact), in place before the first product
  for (int i = threadIdx.x; i < (16384 + N * 128) / 4; i += blockDim.x) {
    const uint32_t h = 0x3C80u + ((i * 7u) & 7u);
    reinterpret_cast<uint32_t*>(g)[i] = h | (h << 16);
  }
  dsa::fence_proxy_async_smem();
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    dsa::mbar_init(bar, 1);
    dsa::mbar_fence_init();
  }
  constexpr uint32_t kCols = N < 32 ? 32 : N;
  if (warp == 0) dsa::tmem_alloc(dsa::smem_u32(slot), kCols);
  dsa::tc_fence_before();
  __syncthreads();
  dsa::tc_fence_after();
  const uint32_t tmem = *slot;
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = dsa::umma_idesc_bf16_f32(128, N);
    const uint64_t dA = dsa::umma_desc_sw128(sA), dB = dsa::umma_desc_sw128(sB);
    const long long t0 = clock64();
    for (int i = 0; i < groups; ++i) {
#pragma unroll
      for (int kk = 0; kk < kUmmaGroup; ++kk)
        dsa::umma_bf16(tmem, dA + (((kk & 3) * 32) >> 4), dB + (((kk & 3) * 32) >> 4), idesc, kk > 0 ? 1u : 0u);
    }
    dsa::umma_commit(bar);
    if (!dsa::mbar_wait(bar, 0, limit_ns, nullptr)) atomicExch(failed, 1);
    atomicAdd(cycles, static_cast<unsigned long long>(clock64() - t0));
  }
  dsa::tc_fence_before();
  __syncthreads();
  dsa::tc_fence_after();
  if (warp == 0) dsa::tmem_dealloc(tmem, kCols);
}

template <int N>
static cudaError_t launch_probe_umma(int grid, int groups, unsigned long long* cycles, int* failed, cudaStream_t st) {
  const int smem = 1024 + 16384 + N * 128 + 128;
  cudaError_t e = cudaFuncSetAttribute(probe_umma_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  probe_umma_kernel<N><<<grid, 128, smem, st>>>(groups, 2000000000ull, cycles, failed);
  return cudaGetLastError();
}


// ---------------------------------------------------------------- accumulator handoff probe
constexpr int kFoldThreads = 608;  // warp 0 issues, warps 1-2 idle, warps 3..18 fold
constexpr int kFoldHeadMmas = 8;
constexpr uint32_t kFoldA = 32768, kFoldB = 65536;  // [2][128 rows][128 B], [2][256 rows][128 B]

template <int kMode>
__global__ void __launch_bounds__(kFoldThreads, 1) probe_fold_kernel(int heads, uint64_t limit_ns,
                                                                   unsigned long long* cycles, int* failed,
                                                                   float* sink) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dsa::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* g = smem_raw + (base - raw);
  const uint32_t sA = base, sB = base + kFoldA;
  const uint32_t full = sB + kFoldB, empty = full + 16;
  uint32_t* slot = reinterpret_cast<uint32_t*>(g + kFoldA + kFoldB + 64);
  for (int i = threadIdx.x; i < static_cast<int>((kFoldA + kFoldB) / 4); i += blockDim.x) {
    const uint32_t h = 0x3C80u + ((i * 7u) & 7u);  // small bf16 operands
    reinterpret_cast<uint32_t*>(g)[i] = h | (h << 16);
  }
  dsa::fence_proxy_async_smem();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      dsa::mbar_init(full + 8 * x, 1);
      dsa::mbar_init(empty + 8 * x, 16);
    }
    dsa::mbar_fence_init();
  }
  if (warp == 0) dsa::tmem_alloc(dsa::smem_u32(slot), 512);
  dsa::tc_fence_before();
  __syncthreads();
  dsa::tc_fence_after();
  const uint32_t tmem = *slot;
  bool ok = true;
  if (kMode == 2) {
    // one warp: a 32-column load of its own lane quarter and its wait, back to back
    if (warp == 3) {
      uint32_t acc = 0;
      const long long t0 = clock64();
      for (int i = 0; i < heads; ++i) {
        uint32_t r[32];
        dsa::tmem_ld32(tmem + (static_cast<uint32_t>(3 * 32) << 16) + static_cast<uint32_t>(i & 7) * 32, r);
        dsa::tmem_ld_wait();
        acc += r[0] ^ r[31];
      }
      if (lane == 0) atomicAdd(cycles, static_cast<unsigned long long>((clock64() - t0) / heads));
      if (acc == 0x9E3779B9u) sink[threadIdx.x] = 1.f;
    }
  } else if (warp == 0) {
    if (lane == 0) {
      constexpr uint32_t idesc = dsa::umma_idesc_bf16_f32(128, 256);
      const uint64_t dA = dsa::umma_desc_sw128(sA), dB = dsa::umma_desc_sw128(sB);
      const long long t0 = clock64();
      for (int h = 0; h < heads && ok; ++h) {
        const int cs = h & 1;
        if (h >= 2) ok = dsa::mbar_wait(empty + 8 * cs, ((h >> 1) - 1) & 1, limit_ns, nullptr);
        dsa::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kFoldHeadMmas; ++kk)
          dsa::umma_bf16(tmem + cs * 256, dA + (((kk >> 2) * (kFoldA / 2) + (kk & 3) * 32) >> 4),
                         dB + (((kk >> 2) * (kFoldB / 2) + (kk & 3) * 32) >> 4), idesc, kk > 0 ? 1u : 0u);
        dsa::umma_commit(full + 8 * cs);
      }
      if (ok) ok = dsa::mbar_wait(empty + 8 * ((heads - 1) & 1), ((heads - 1) >> 1) & 1, limit_ns, nullptr);
      atomicAdd(cycles, static_cast<unsigned long long>((clock64() - t0) / heads));
    }
    __syncwarp();
  } else if (warp >= 3) {
    const int ew = warp - 3, lq = warp & 3, cq = ew >> 2;
    float2 acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = make_float2(0.f, 0.f);
    const float2 w2 = make_float2(0.5f, 0.5f);
    for (int h = 0; h < heads && ok; ++h) {
      const int cs = h & 1;
      ok = dsa::mbar_wait(full + 8 * cs, (h >> 1) & 1, limit_ns, nullptr);
      dsa::tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(lq * 32) << 16) + cs * 256 + cq * 64;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t r[16];
        dsa::tmem_ld16(taddr + cc * 16, r);
        dsa::tmem_ld_wait();
        if (cc == 3) {
          dsa::tc_fence_before();
          __syncwarp();
          if (lane == 0) dsa::mbar_arrive(empty + 8 * cs);
        }
        if (kMode == 1) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 x =
                make_float2(fmaxf(__uint_as_float(r[2 * j]), 0.f), fmaxf(__uint_as_float(r[2 * j + 1]), 0.f));
            acc[cc * 8 + j] = __ffma2_rn(w2, x, acc[cc * 8 + j]);
          }
        } else {
          acc[cc] = make_float2(acc[cc].x + __uint_as_float(r[0]), acc[cc].y);
        }
      }
    }
    float t = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) t += acc[j].x + acc[j].y;
    if (t == 1.2345f) sink[threadIdx.x] = t;
  }
  if (!ok) atomicExch(failed, 1);
  dsa::tc_fence_before();
  __syncthreads();
  dsa::tc_fence_after();
  if (warp == 0) dsa::tmem_dealloc(tmem, 512);
}

}  // namespace


extern "C" {

double dsa_measure_l2(int kind, void* buf, size_t bytes, int iters, void* stream) {
  if (!buf || bytes < 4096 || iters < 1 || kind < 0 || kind > 8 || (reinterpret_cast<uintptr_t>(buf) & 15u)) {
    dsa::set_last_error("dsa_measure_l2: kind must be 0..8, buf 16-byte aligned, bytes >= 4096, iters >= 1");
    return -1.0;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    dsa::set_last_error("dsa_measure_l2: no device");
    return -1.0;
  }
  const int block = 256;
  const int grid = sms * 8;
  const int warps = grid * block / 32;
  float* sink = static_cast<float*>(buf);
  double moved = 0.0;
  auto launch = [&](int reps) {
    if (kind == 0) {
      const int64_t n4 = static_cast<int64_t>(bytes / 16);
      probe_stream_kernel<<<grid, block, 0, st>>>(static_cast<const float4*>(buf), n4, reps, sink);
      moved = static_cast<double>(n4) * 16.0 * reps;
    } else if (kind == 1) {
      const uint32_t nb = static_cast<uint32_t>(bytes / 1024);
      const int per_warp = 64 * reps;
      probe_gather_kernel<<<grid, block, 0, st>>>(static_cast<const uint4*>(buf), nb, per_warp, sink);
      moved = static_cast<double>(warps) * per_warp * 1024.0;
    } else if (kind == 2) {
      const uint32_t nb = static_cast<uint32_t>(bytes / 2048);
      const int per_warp = 64 * reps;
      probe_red_kernel<<<grid, block, 0, st>>>(static_cast<float*>(buf), nb, per_warp);
      moved = static_cast<double>(warps) * per_warp * 512.0;
    } else if (kind == 3 || kind == 4) {
      const uint32_t nb = static_cast<uint32_t>(bytes / 2048);
      const int per_warp = 16 * reps;
      probe_bulk_red_kernel<<<grid, block, 0, st>>>(static_cast<float*>(buf), nb, per_warp, kind == 3 ? 2048 : 512);
      moved = static_cast<double>(warps) * per_warp * 2048.0;
    } else if (kind <= 7) {
      const uint32_t nb = static_cast<uint32_t>(bytes / 2048);
      const int per_warp = 64 * reps;
      float* fb = static_cast<float*>(buf);
      if (kind == 5) probe_red_shape_kernel<2><<<grid, block, 0, st>>>(fb, nb, per_warp);
      else if (kind == 6) probe_red_shape_kernel<8><<<grid, block, 0, st>>>(fb, nb, per_warp);
      else probe_red_shape_kernel<16><<<grid, block, 0, st>>>(fb, nb, per_warp);
      moved = static_cast<double>(warps) * per_warp * 512.0;
    } else {
      // equal bytes per warp on both paths: a red.v4 instruction adds 512 B, a bulk operation 2 KB
      const uint32_t nb = static_cast<uint32_t>(bytes / 2048);
      const int red_iters = 64 * reps, bulk_iters = 16 * reps;
      probe_red_mix_kernel<<<grid, block, 0, st>>>(static_cast<float*>(buf), nb, red_iters, bulk_iters);
      moved = static_cast<double>(grid) * 4.0 * (red_iters * 512.0 + bulk_iters * 2048.0);
    }
  };
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  launch(1);  // warm-up: brings the buffer into L2
  cudaEventRecord(a, st);
  launch(iters);
  cudaEventRecord(b, st);
  cudaError_t e = cudaEventSynchronize(b);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  if (e != cudaSuccess || ms <= 0.f) {
    dsa::set_last_error(std::string("dsa_measure_l2: ") + cudaGetErrorString(e));
    return -1.0;
  }
  return moved / (ms * 1e-3) / 1e9;
}

double dsa_measure_umma(int n, int issuers, int groups, void* stream) {
  if ((n != 16 && n != 32 && n != 64 && n != 128 && n != 256) || issuers < 1 || issuers > 3 || groups < 1 ||
      issuers * (n < 32 ? 32 : n) > 512) {
    dsa::set_last_error("dsa_measure_umma: n in {16, 32, 64, 128, 256}, issuers 1..3 with issuers * max(n, 32) <= "
                        "512 tensor-memory columns, groups >= 1");
    return -1.0;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    dsa::set_last_error("dsa_measure_umma: no device");
    return -1.0;
  }
  unsigned long long* cycles = nullptr;
  int* failed = nullptr;
  cudaError_t e = cudaMalloc(&cycles, sizeof(unsigned long long) + sizeof(int));
  if (e != cudaSuccess) {
    dsa::set_last_error(std::string("dsa_measure_umma: ") + cudaGetErrorString(e));
    return -1.0;
  }
  failed = reinterpret_cast<int*>(cycles + 1);
  const int grid = sms * issuers;
  for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {  // the first pass warms up
    e = cudaMemsetAsync(cycles, 0, sizeof(unsigned long long) + sizeof(int), st);
    if (e != cudaSuccess) break;
    switch (n) {
      case 16: e = launch_probe_umma<16>(grid, groups, cycles, failed, st); break;
      case 32: e = launch_probe_umma<32>(grid, groups, cycles, failed, st); break;
      case 64: e = launch_probe_umma<64>(grid, groups, cycles, failed, st); break;
      case 128: e = launch_probe_umma<128>(grid, groups, cycles, failed, st); break;
      default: e = launch_probe_umma<256>(grid, groups, cycles, failed, st); break;
    }
  }
  unsigned long long total = 0;
  int bad = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&total, cycles, sizeof(total), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&bad, failed, sizeof(bad), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(cycles);
  if (e != cudaSuccess || bad) {
    dsa::set_last_error(std::string("dsa_measure_umma: ") + (bad ? "a completion wait ran out" : cudaGetErrorString(e)));
    return -1.0;
  }
  return static_cast<double>(total) / grid / (static_cast<double>(groups) * kUmmaGroup);
}

double dsa_measure_fold(int mode, int heads, void* stream) {
  if (mode < 0 || mode > 2 || heads < 2) {
    dsa::set_last_error("dsa_measure_fold: mode 0 (no arithmetic), 1 (the fold) or 2 (TMEM load), heads >= 2");
    return -1.0;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned long long* cycles = nullptr;
  cudaError_t e = cudaMalloc(&cycles, sizeof(unsigned long long) + sizeof(int) + kFoldThreads * sizeof(float));
  if (e != cudaSuccess) {
    dsa::set_last_error(std::string("dsa_measure_fold: ") + cudaGetErrorString(e));
    return -1.0;
  }
  int* failed = reinterpret_cast<int*>(cycles + 1);
  float* sink = reinterpret_cast<float*>(failed + 1);
  const int smem = 1024 + static_cast<int>(kFoldA + kFoldB) + 128;
  e = cudaFuncSetAttribute(probe_fold_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(probe_fold_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(probe_fold_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {  // the first pass warms up
    e = cudaMemsetAsync(cycles, 0, sizeof(unsigned long long) + sizeof(int), st);
    if (e == cudaSuccess) {
      if (mode == 0) probe_fold_kernel<0><<<1, kFoldThreads, smem, st>>>(heads, 2000000000ull, cycles, failed, sink);
      else if (mode == 1) probe_fold_kernel<1><<<1, kFoldThreads, smem, st>>>(heads, 2000000000ull, cycles, failed, sink);
      else probe_fold_kernel<2><<<1, kFoldThreads, smem, st>>>(heads, 2000000000ull, cycles, failed, sink);
      e = cudaGetLastError();
    }
  }
  unsigned long long c = 0;
  int bad = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&c, cycles, sizeof(c), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&bad, failed, sizeof(bad), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(cycles);
  if (e != cudaSuccess || bad) {
    dsa::set_last_error(std::string("dsa_measure_fold: ") + (bad ? "a completion wait ran out" : cudaGetErrorString(e)));
    return -1.0;
  }
  return static_cast<double>(c);
}

}  // extern "C"
