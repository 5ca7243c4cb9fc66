// attn_bwd.cu -- sparse attention backward over the selected key pools.
//
// [SkyRL-1M §模型与瓶颈] the selected-key attention is trained, so its
// gradient flows to q, k and v.  For query i, head h and key j of its key set
// (selected pools plus its own partial pool):
//   P_hj  = exp(s_hj - lse_h)              s_hj = scale * q_h . k_j
//   dS_hj = P_hj (dO_h . v_j - Delta_h)    Delta_h = dO_h . O_h
//   dq_h  = scale * sum_j dS_hj k_j
//   dk_j += scale * sum_h dS_hj q_h ;  dv_j += sum_h P_hj dO_h
// The forward's lse lets P be recomputed instead of stored.
//
// One CTA (4 warps) per query gathers K and V blocks exactly as the forward
// does.  Per warp and 16-key slice: S and dP on mma.sync (the Q and dO
// A fragments are read from shared memory once per query and stay in
// registers), dQ accumulated in registers, and the slice's dK/dV rows (16 keys x 128 dims, already summed
// over the 16 heads by the MMA) added into fp32 accumulators with 16-byte
// reductions.  The reductions are L2-bound, and L2 serves them best when one
// warp instruction covers whole 128-byte lines: each reduction instruction
// adds one pool's four key rows, 128 bytes of each.  The dK/dV products read
// Q and dO from copies whose dims are interleaved within each 16-dim group,
// so that every lane's accumulator fragment holds four consecutive dims of a
// key row; one lane exchange across the warp's halves then gives each
// instruction its pool's four rows, with no shared-memory staging.  A final
// kernel rounds the accumulators to bf16.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace {

constexpr int kHq = 16;
constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kBlkPools = 16;
constexpr int kBlkKeys = 4 * kBlkPools;
constexpr int kStages = 2;
constexpr int kWarpKeys = kBlkKeys / kWarps;           // 16 keys of each block per warp
constexpr uint32_t kWarpTile = kWarpKeys * kD * 2;     // 4 KB: K (or V) rows of a warp's keys
constexpr uint32_t kWarpStage = 2 * kWarpTile;         // K then V
constexpr uint32_t kStageBytes = kWarps * kWarpStage;  // 32 KB: one block
constexpr uint32_t kQBytes = kHq * kD * 2;
constexpr int kMaxTopk = 2048;
// Q, dO, then their dim-interleaved copies, the gather ring
constexpr size_t kSmemFixed = 128 + 4 * kQBytes + kStages * kStageBytes;
// row table: one int32 per key of every block (topk pools + the own pool, in blocks of 16 slots)
constexpr size_t smem_bytes(int topk) {
  return kSmemFixed + static_cast<size_t>((topk + 1 + kBlkPools - 1) / kBlkPools) * kBlkKeys * sizeof(int32_t);
}

// Position in a block's row table of key kr (0..63): warp w's keys 16w..16w+15
// fill slots 16w..16w+15, its even keys first, so the lane that gathers keys
// p, p + 2, ..., p + 14 of the warp (p = 0 or 1) reads their rows with two
// 16-byte loads.
__device__ __forceinline__ int row_slot(int kr) { return (kr & ~15) + (kr & 1) * 8 + ((kr & 15) >> 1); }

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * 256 + ((c ^ (r & 7)) << 4));
}

// Transposes an 8x8 bf16 matrix held one 32-bit word per lane in the mma
// fragment order (lane 4r + c holds row r, columns 2c and 2c + 1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Gathers the K and V rows of warp `w`'s 16 keys of block `blk` into the
// warp's part `st` of a stage (rows as in the forward: -1 = zero-filled and
// masked).  Lane l copies 16-byte chunk l % 16 of the warp's keys
// l / 16 + 2u, u = 0..7.  Only the warp reads them, so a warp-level wait
// and __syncwarp() order them: the warps of a CTA do not wait for each other.
__device__ __forceinline__ void gather_warp(uint32_t st, const __nv_bfloat16* __restrict__ k,
                                            const __nv_bfloat16* __restrict__ v, const int32_t* rows, int blk,
                                            int w, int lane) {
  const int p = lane >> 4, cc = lane & 15;
  const int4 ra = *reinterpret_cast<const int4*>(rows + blk * kBlkKeys + w * kWarpKeys + p * 8);
  const int4 rb = *reinterpret_cast<const int4*>(rows + blk * kBlkKeys + w * kWarpKeys + p * 8 + 4);
  const int32_t r8[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int kl = p + 2 * u;
    const bool ok = r8[u] >= 0;
    const int64_t src = static_cast<int64_t>(ok ? r8[u] : 0) * kD + cc * 8;
    cp_async16(st + swz(kl, cc), k + src, ok);
    cp_async16(st + kWarpTile + swz(kl, cc), v + src, ok);
  }
}

__global__ void __launch_bounds__(kThreads, 2)
    attn_bwd_kernel(const __nv_bfloat16* __restrict__ dO, const __nv_bfloat16* __restrict__ q,
                    const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                    const float* __restrict__ lse, const float* __restrict__ delta,
                    const int32_t* __restrict__ pool_idx, int64_t q0, int topk, float scale, float scale_log2,
                    __nv_bfloat16* __restrict__ dq, float* __restrict__ dk_acc, float* __restrict__ dv_acc,
                    unsigned* status, const __grid_constant__ SeqTable tab) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sdO = base + kQBytes;
  const uint32_t sQi = base + 2 * kQBytes;   // Q with dims interleaved (below)
  const uint32_t sdOi = base + 3 * kQBytes;  // dO likewise
  const uint32_t sKV = base + 4 * kQBytes;
  int32_t* rows = reinterpret_cast<int32_t*>(gbase + 4 * kQBytes + kStages * kStageBytes);
  __shared__ int s_nsel;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  // query i (global position) is local row r of q, dO, lse, Delta, pool_idx and dq
  const int64_t r = blockIdx.x;
  int64_t i, kv0;
  seq_locate(tab, q0, r, &i, &kv0);  // i: position in its sequence; its keys start at packed row kv0
  k += kv0 * kD;
  v += kv0 * kD;
  if (dk_acc != nullptr) {
    dk_acc += kv0 * kD;
    dv_acc += kv0 * kD;
  }
  const int64_t n_elig = i >> 2;

  if (tid == 0) s_nsel = topk;
  __syncthreads();
  const int32_t* prow = pool_idx + r * topk;
  for (int j = tid; j < topk; j += kThreads)
    if (prow[j] < 0) atomicMin(&s_nsel, j);
  __syncthreads();
  const int nsel = s_nsel;
  const int nblk = (nsel + 1 + kBlkPools - 1) / kBlkPools;
  // row table of every block, built and checked as in the forward
  bool bad = false;
  for (int e = tid; e < nblk * kBlkKeys; e += kThreads) {
    const int blk = e / kBlkKeys, pos = e % kBlkKeys;
    const int kr = (pos & ~15) + 2 * (pos & 7) + ((pos >> 3) & 1);  // inverse of row_slot
    const int slot = blk * kBlkPools + (kr >> 2);
    int32_t row = -1;
    if (slot < nsel) {
      const int32_t p = prow[slot];
      if (p < n_elig) row = 4 * p + (kr & 3);
      else bad = true;
      if ((kr & 3) == 0 && slot > 0 && p <= prow[slot - 1]) bad = true;
    } else if (slot == nsel) {
      const int64_t r = 4 * n_elig + (kr & 3);
      if (r <= i) row = static_cast<int32_t>(r);
    }
    DSA_CHECK(status, row >= -1 && row <= i);
    rows[e] = row;
  }
  if (bad) record_status(status, kStatusInternal);

  {
    const __nv_bfloat16* qrow = q + r * (kHq * kD);
    const __nv_bfloat16* drow = dO + r * (kHq * kD);
#pragma unroll
    for (int u = 0; u < (kHq * 16) / kThreads; ++u) {
      const int c = tid + u * kThreads;
      cp_async16(sQ + swz(c >> 4, c & 15), qrow + c * 8, true);
      cp_async16(sdO + swz(c >> 4, c & 15), drow + c * 8, true);
    }
  }
  // the row table is visible to the gather; with no hole anywhere, only the
  // last block (the own pool and the empty slots after it) needs a mask
  const bool any_hole = __syncthreads_or(bad) != 0;
  gather_warp(sKV + warp * kWarpStage, k, v, rows, 0, warp, lane);  // nblk >= 1
  cp_async_commit();

  // per-row constants (rows g and g+8 of this thread's fragments = heads)
  const float lse2_0 = lse[r * kHq + g] * kLog2e, lse2_1 = lse[r * kHq + g + 8] * kLog2e;
  const float dl0 = delta[r * kHq + g], dl1 = delta[r * kHq + g + 8];

  float dq_acc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) dq_acc[j][0] = dq_acc[j][1] = dq_acc[j][2] = dq_acc[j][3] = 0.f;
  uint32_t qa[8][4], dga[8][4];  // Q and dO A fragments, read once per query

  for (int b = 0; b < nblk; ++b) {
    cp_async_wait<0>();  // this lane's copies of block b (and, at b = 0, its part of Q and dO)
    if (b == 0) {
      __syncthreads();  // every thread's part of Q and dO
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int mat = lane >> 3;
        const int r = (lane & 7) + ((mat & 1) << 3);
        const int c = 2 * kk + (mat >> 1);
        ldsm_x4(sQ + swz(r, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
        ldsm_x4(sdO + swz(r, c), dga[kk][0], dga[kk][1], dga[kk][2], dga[kk][3]);
      }
      // Interleaved copies: in each 16-dim group (chunks 2j, 2j+1 of a head's
      // row), chunk 2j holds dims {0,1,4,5,8,9,12,13} and chunk 2j+1 dims
      // {2,3,6,7,10,11,14,15}.  Read as the B operand of an n8 product, the
      // two chunks put dims 4t..4t+1 and 4t+2..4t+3 in the columns of lane
      // group t, so each lane's dK/dV fragment holds four consecutive dims.
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int h = tid >> 3, j = tid & 7;
        const uint32_t src = u == 0 ? sQ : sdO, dst = u == 0 ? sQi : sdOi;
        const uint4 a = *reinterpret_cast<const uint4*>(gbase + (src - base) + swz(h, 2 * j));
        const uint4 c = *reinterpret_cast<const uint4*>(gbase + (src - base) + swz(h, 2 * j + 1));
        *reinterpret_cast<uint4*>(gbase + (dst - base) + swz(h, 2 * j)) = make_uint4(a.x, a.z, c.x, c.z);
        *reinterpret_cast<uint4*>(gbase + (dst - base) + swz(h, 2 * j + 1)) = make_uint4(a.y, a.w, c.y, c.w);
      }
      __syncthreads();
    } else {
      __syncwarp();  // the warp's copies of block b are visible to its lanes, and block b - 1 is read
    }
    if (b + 1 < nblk) gather_warp(sKV + ((b + 1) & 1) * kStageBytes + warp * kWarpStage, k, v, rows, b + 1, warp, lane);
    cp_async_commit();
    const uint32_t sK = sKV + (b & 1) * kStageBytes + warp * kWarpStage;
    const uint32_t sV = sK + kWarpTile;
    const int key0 = warp * 16;

    // S = Q K^T and dP = dO V^T for this warp's 16 keys
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int mat = lane >> 3;
      const int r = ((mat >> 1) << 3) + (lane & 7);
      const int c = 2 * kk + (mat & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(sK + swz(r, c), b0, b1, b2, b3);
      mma_bf16_16816(s0, qa[kk], b0, b1);
      mma_bf16_16816(s1, qa[kk], b2, b3);
      ldsm_x4(sV + swz(r, c), b0, b1, b2, b3);
      mma_bf16_16816(p0, dga[kk], b0, b1);
      mma_bf16_16816(p1, dga[kk], b2, b3);
    }

    // key validity of this thread's columns (2t, 2t+1, 8+2t, 9+2t)
    bool valid[4] = {true, true, true, true};
    if (b + 1 == nblk || any_hole) {
      const int kc[4] = {key0 + 2 * t4, key0 + 2 * t4 + 1, key0 + 8 + 2 * t4, key0 + 9 + 2 * t4};
#pragma unroll
      for (int e = 0; e < 4; ++e) valid[e] = rows[b * kBlkKeys + row_slot(kc[e])] >= 0;
    }
    // P and dS (fragment order: e=0..3 row g / g+8 for n-tile 0, then n-tile 1)
    float P[8], dS[8];
    {
      const float sc[8] = {s0[0], s0[1], s0[2], s0[3], s1[0], s1[1], s1[2], s1[3]};
      const float dp[8] = {p0[0], p0[1], p0[2], p0[3], p1[0], p1[1], p1[2], p1[3]};
      const bool vm[8] = {valid[0], valid[1], valid[0], valid[1], valid[2], valid[3], valid[2], valid[3]};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const bool hi = (e & 2) != 0;  // row g+8
        P[e] = vm[e] ? ex2_ftz(fmaf(sc[e], scale_log2, -(hi ? lse2_1 : lse2_0))) : 0.f;
        dS[e] = P[e] * (dp[e] - (hi ? dl1 : dl0));
      }
    }
    uint32_t dsa[4];
    dsa[0] = pack_bf16(dS[0], dS[1]);
    dsa[1] = pack_bf16(dS[2], dS[3]);
    dsa[2] = pack_bf16(dS[4], dS[5]);
    dsa[3] = pack_bf16(dS[6], dS[7]);
    // dQ += dS K (K rows are the k dimension: ldmatrix .trans)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int mat = lane >> 3;
      const int r = ((mat & 1) << 3) + (lane & 7);
      const int c = 2 * j + (mat >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(sK + swz(r, c), b0, b1, b2, b3);
      mma_bf16_16816(dq_acc[2 * j], dsa, b0, b1);
      mma_bf16_16816(dq_acc[2 * j + 1], dsa, b2, b3);
    }

    if (dk_acc == nullptr) continue;  // dq only: the deterministic backward adds dK/dV key by key

    // P^T and (scale dS)^T as A fragments [16 keys][16 heads], each split
    // into bf16 hi + lo (x = hi + lo to ~2^-17): the dK/dV sums run over
    // thousands of queries for popular keys, where a single bf16 rounding of
    // P or dS accumulates beyond the gradient tolerance.  The S fragment's
    // 8x8 quadrant (head block a, key block b) transposes in registers into
    // the A fragment's quadrant (key block b, head block a).
    uint32_t pth[4], ptl[4], dth[4], dtl[4];
    {
      constexpr int kSrc[4] = {0, 2, 1, 3};  // A word w <- S quadrant pair kSrc[w] (x[2q], x[2q+1])
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const float* x = m == 0 ? P : dS;
        const float mul = m == 0 ? 1.f : scale;  // the dK fragments carry scale * dS
        uint32_t* th = m == 0 ? pth : dth;
        uint32_t* tl = m == 0 ? ptl : dtl;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int q = kSrc[w];
          const float x0 = mul * x[2 * q], x1 = mul * x[2 * q + 1];
          const uint32_t hi = pack_bf16(x0, x1);
          const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xFFFF0000u);
          th[w] = movmatrix_t(hi);
          tl[w] = movmatrix_t(pack_bf16(x0 - h0, x1 - h1));
        }
      }
    }
    // Reductions: instruction kq adds slot (key0/4 + kq)'s pool: key
    // (lane & 15) / 4 of it, dims 32 jj + 16 (lane / 16) + 4 (lane & 3) .. + 3.
    const int kin = (lane & 15) >> 2;
    const bool upper = lane >= 16;
    const int dim0 = ((lane >> 4) << 4) + 4 * t4;
    int64_t rrow[4];
    bool rok[4];
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
      const int32_t r = rows[b * kBlkKeys + row_slot(key0 + 4 * kq + kin)];
      rrow[kq] = r;
      rok[kq] = r >= 0;
    }
    // dV rows += P^T dO ; dK rows += (scale dS)^T Q   (16 keys x 128 dims, in 32-dim blocks)
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {  // m = 0: dV from P and dO; m = 1: dK from scale dS and Q
        const uint32_t(&th)[4] = m == 0 ? pth : dth;
        const uint32_t(&tl)[4] = m == 0 ? ptl : dtl;
        const uint32_t sB = m == 0 ? sdOi : sQi;
        float* acc = m == 0 ? dv_acc : dk_acc;
        // x[hh][e]: dims 16 (2 jj + hh) + 4 t4 + e of key g (lo) and of key g + 8 (hi)
        float lo[2][4], hi[2][4];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int j = 2 * jj + hh;
          const int mat = lane >> 3;
          const int r = (lane & 7) + ((mat & 1) << 3);
          const int c = 2 * j + (mat >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sB + swz(r, c), b0, b1, b2, b3);
          float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16_16816(c0, th, b0, b1);
          mma_bf16_16816(c0, tl, b0, b1);
          mma_bf16_16816(c1, th, b2, b3);
          mma_bf16_16816(c1, tl, b2, b3);
          lo[hh][0] = c0[0];
          lo[hh][1] = c0[1];
          lo[hh][2] = c1[0];
          lo[hh][3] = c1[1];
          hi[hh][0] = c0[2];
          hi[hh][1] = c0[3];
          hi[hh][2] = c1[2];
          hi[hh][3] = c1[3];
        }
        // Lanes 0-15 hold keys 0-3 (lo) / 8-11 (hi) of the slice, lanes 16-31
        // keys 4-7 / 12-15.  Each lane sends the 16-dim half its partner
        // lane (lane ^ 16) needs: then lanes 0-15 carry the first half and
        // lanes 16-31 the second half of the same four keys.
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float(*x)[4] = half == 0 ? lo : hi;
          float first[4], second[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float y = __shfl_xor_sync(0xffffffffu, upper ? x[0][e] : x[1][e], 16);
            first[e] = upper ? y : x[0][e];
            second[e] = upper ? x[1][e] : y;
          }
          const int kq0 = 2 * half;
          if (rok[kq0])
            red_add_v4(acc + rrow[kq0] * kD + 32 * jj + dim0, first[0], first[1], first[2], first[3]);
          if (rok[kq0 + 1])
            red_add_v4(acc + rrow[kq0 + 1] * kD + 32 * jj + dim0, second[0], second[1], second[2], second[3]);
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- dq = scale * sum over the four warps' partial dq (rows padded to
  // 132 floats so the fragment stores spread over the banks)
  constexpr int kRedLd = kD + 4;
  float* red = reinterpret_cast<float*>(gbase + 4 * kQBytes);  // reuses the gather ring
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int col = 8 * j + 2 * t4;
    *reinterpret_cast<float2*>(red + (warp * kHq + g) * kRedLd + col) = make_float2(dq_acc[j][0], dq_acc[j][1]);
    *reinterpret_cast<float2*>(red + (warp * kHq + g + 8) * kRedLd + col) = make_float2(dq_acc[j][2], dq_acc[j][3]);
  }
  __syncthreads();
  // thread tid owns element pairs e = 2 * (tid + 128 m), m = 0..7 (consecutive across threads)
  __nv_bfloat16* dqrow = dq + r * (kHq * kD);
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int e = 2 * (tid + kThreads * m);
    const int r = e / kD, c = e % kD;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float2 x = *reinterpret_cast<const float2*>(red + (w * kHq + r) * kRedLd + c);
      a0 += x.x;
      a1 += x.y;
    }
    *reinterpret_cast<uint32_t*>(dqrow + e) = pack_bf16(scale * a0, scale * a1);
  }
}

// Delta[r] = dO[r,:] . O[r,:] for every (query, head) row r; zeroes the dK/dV
// accumulators.  Half a warp per row, 8 dims per lane.
__global__ void bwd_pre_kernel(const __nv_bfloat16* __restrict__ dO, const __nv_bfloat16* __restrict__ o,
                               int64_t rows, float* __restrict__ delta, float4* __restrict__ zero, int64_t nzero4) {
  const int64_t gt = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gt >> 4;
  const int part = threadIdx.x & 15;
  float acc = 0.f;
  if (row < rows) {
    const uint4 a = reinterpret_cast<const uint4*>(dO + row * kD)[part];
    const uint4 b = reinterpret_cast<const uint4*>(o + row * kD)[part];
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(aw[e] << 16), __uint_as_float(bw[e] << 16), acc);
      acc = fmaf(__uint_as_float(aw[e] & 0xFFFF0000u), __uint_as_float(bw[e] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) delta[row] = acc;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t z = gt; z < nzero4; z += nthreads) zero[z] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void cast_kernel(const float* __restrict__ a, const float* __restrict__ b, int64_t n8,
                            __nv_bfloat16* __restrict__ ao, __nv_bfloat16* __restrict__ bo) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= 2 * n8) return;
  const bool second = t >= n8;
  const int64_t e = second ? t - n8 : t;
  const float4* src = reinterpret_cast<const float4*>(second ? b : a) + 2 * e;
  const float4 x = src[0], y = src[1];
  uint4 out = make_uint4(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w), pack_bf16(y.x, y.y), pack_bf16(y.z, y.w));
  reinterpret_cast<uint4*>(second ? bo : ao)[e] = out;
}

}  // namespace

cudaError_t launch_attn_bwd_pre(const void* dO, const void* o, int64_t nq, int64_t S, float* delta, float* dk_acc,
                                float* dv_acc, const LaunchCtx& ctx) {
  // Delta for the nq local query rows; dk_acc and dv_acc are adjacent in the
  // workspace: zero 2 * S * D floats from dk_acc (nothing when dk_acc is null)
  (void)dv_acc;
  const int64_t rows = nq * kHq;
  const int block = 256;
  const int64_t nzero4 = dk_acc != nullptr ? 2 * S * kD / 4 : 0;
  const int64_t threads = rows * 16 > nzero4 / 4 ? rows * 16 : nzero4 / 4;  // each zeroes ~4 float4
  const int64_t grid = (threads + block - 1) / block;
  bwd_pre_kernel<<<static_cast<unsigned>(grid), block, 0, ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(o), rows, delta,
      reinterpret_cast<float4*>(dk_acc), nzero4);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const void* dO, const void* q, const void* k, const void* v, const float* lse,
                            const float* delta, const int32_t* pool_idx, int64_t q_begin, int64_t q_end, int topk,
                            float scale, void* dq, float* dk_acc, float* dv_acc, const LaunchCtx& ctx,
                            const SeqTable* tab) {
  if (q_end <= q_begin) return cudaSuccess;
  static const SeqTable kNoTable = {};
  static std::atomic<bool> attr_done[kAttrDevices];
  const cudaError_t e = set_smem_limit_once(attn_bwd_kernel, static_cast<int>(smem_bytes(kMaxTopk)), attr_done);
  if (e != cudaSuccess) return e;
  attn_bwd_kernel<<<static_cast<unsigned>(q_end - q_begin), kThreads, smem_bytes(topk), ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(q),
      static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), lse, delta, pool_idx, q_begin, topk,
      scale, scale * kLog2e, static_cast<__nv_bfloat16*>(dq), dk_acc, dv_acc, ctx.status, tab ? *tab : kNoTable);
  return cudaGetLastError();
}

cudaError_t launch_cast_dkdv(const float* dk_acc, const float* dv_acc, int64_t n, void* dk, void* dv,
                             const LaunchCtx& ctx) {
  const int64_t n8 = n / 8;  // n = S * D, a multiple of 8
  const int block = 256;
  const int64_t grid = (2 * n8 + block - 1) / block;
  if (grid == 0) return cudaSuccess;
  cast_kernel<<<static_cast<unsigned>(grid), block, 0, ctx.stream>>>(dk_acc, dv_acc, n8,
                                                                        static_cast<__nv_bfloat16*>(dk),
                                                                        static_cast<__nv_bfloat16*>(dv));
  return cudaGetLastError();
}

}  // namespace dsa
