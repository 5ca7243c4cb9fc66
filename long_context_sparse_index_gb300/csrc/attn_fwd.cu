// attn_fwd.cu -- sparse attention forward over the selected key pools.
//
// [SkyRL-1M §模型与瓶颈] each query attends to ~2048 selected keys (the 4
// tokens of each selected pool) rather than to the whole prefix; here query i
// also attends to its own partial pool {4*floor(i/4), ..., i}.  The 16 query
// heads share one KV head, so one gathered K/V row serves all 16 heads.
// [CP-lesson §改进二, evidence ②] the softmax is computed online over blocks
// of keys, which reproduces the one-shot softmax exactly in real arithmetic.
//
// Layout of the work: one CTA (4 warps) per query.  The key list is walked in
// blocks of 16 pool slots (64 keys); each warp gathers the K and V rows of its
// own 16 keys of a block with 16-byte cp.async copies into its quarter of a
// 2-stage ring in shared memory (rows XOR-swizzled in 16-B chunks so ldmatrix
// reads are conflict-free), and waits only for its own copies.
// The Q tile sits in the ring's second stage until it is read into
// registers, so a CTA takes 74 KB and three run per SM (12 warps), which
// hides more of the MMA and gather latency than a deeper ring at two per SM.
// Warp w owns keys 16w..16w+15 of every block: S = Q K^T and O += P V run on
// bf16 mma.sync (m16n8k16, M = the 16 heads), with a lagging per-row softmax
// reference, the normaliser and O in fp32 registers.  The four warps' partial softmax
// states are merged through shared memory at the end.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace {

constexpr int kHq = 16;
constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kBlkPools = 16;
constexpr int kBlkKeys = 4 * kBlkPools;       // 64
constexpr int kStages = 2;
constexpr int kWarpKeys = kBlkKeys / kWarps;           // 16 keys of each block per warp
constexpr uint32_t kWarpTile = kWarpKeys * kD * 2;     // 4 KB: K (or V) rows of a warp's keys
constexpr uint32_t kWarpStage = 2 * kWarpTile;         // K then V
constexpr uint32_t kStageBytes = kWarps * kWarpStage;  // 32 KB: one block
constexpr uint32_t kQBytes = kHq * kD * 2;           // 4 KB
constexpr int kMaxTopk = 2048;
// Q lives inside stage 1 of the ring until it is read into registers (before
// block 1 is gathered), so a CTA needs 74 KB at topk = 512 and three fit per SM
constexpr size_t kSmemFixed = 128 + kStages * kStageBytes;
static_assert(kQBytes <= kStageBytes, "Q fits in a stage");
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
constexpr float kLn2 = 0.6931471805599453f;
// A row's softmax reference moves up only when a score exceeds it by more
// than this (log2 units): P stays below 2^8, and the accumulators are
// rescaled only then, not whenever the maximum rises a little.
constexpr float kLag = 8.f;

// byte offset of 16-B chunk c (0..15) of row r in a swizzled [rows][256 B] tile
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * 256 + ((c ^ (r & 7)) << 4));
}

// Gathers the K and V rows of warp `w`'s 16 keys of block `blk` into the
// warp's part `st` of a stage.  `rows` holds the block's 64 key rows (-1:
// empty slot, hole or a row past the query, zero-filled and masked by the
// caller).  Lane l copies 16-byte chunk l % 16 of the warp's keys l / 16 + 2u,
// u = 0..7.  Only the warp reads them, so a warp-level wait and __syncwarp()
// order them: the warps of a CTA do not wait for each other.
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

__global__ void __launch_bounds__(kThreads, 3)
    attn_fwd_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v, const int32_t* __restrict__ pool_idx, int64_t q0, int topk,
                    float scale_log2, __nv_bfloat16* __restrict__ o, float* __restrict__ lse, unsigned* status,
                    const __grid_constant__ SeqTable tab) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sKV = base;
  const uint32_t sQ = base + kStageBytes;  // inside stage 1: read before block 1 is gathered
  int32_t* rows = reinterpret_cast<int32_t*>(gbase + kStages * kStageBytes);
  __shared__ int s_nsel;
  __shared__ float s_m[kWarps][kHq], s_l[kWarps][kHq];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  // query i (position in its sequence) is local row r of q, pool_idx, o and
  // lse; its sequence's keys start at packed row kv0 of k and v
  const int64_t r = blockIdx.x;
  int64_t i, kv0;
  seq_locate(tab, q0, r, &i, &kv0);
  k += kv0 * kD;
  v += kv0 * kD;
  const int64_t n_elig = i >> 2;

  // ---- selected pools of this query (leading non-negative entries)
  if (tid == 0) s_nsel = topk;
  __syncthreads();
  const int32_t* prow = pool_idx + r * topk;
  for (int j = tid; j < topk; j += kThreads)
    if (prow[j] < 0) atomicMin(&s_nsel, j);
  __syncthreads();
  const int nsel = s_nsel;
  const int nblk = (nsel + 1 + kBlkPools - 1) / kBlkPools;
  // Row table of every block.  Slot s < nsel holds pool prow[s]; slot nsel is
  // the query's own pool m (rows 4m .. i); slots beyond are empty.  An entry
  // that is not an eligible pool, or breaks ascending order, is recorded as a
  // device-side check failure; ineligible entries become holes (-1: never
  // read, always masked) so no access leaves the K/V rows.
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

  // ---- Q tile (swizzled) and the gather pipeline prologue
  {
    const __nv_bfloat16* qrow = q + r * (kHq * kD);
#pragma unroll
    for (int u = 0; u < (kHq * 16) / kThreads; ++u) {
      const int c = tid + u * kThreads;
      cp_async16(sQ + swz(c >> 4, c & 15), qrow + c * 8, true);
    }
  }
  // the row table is visible to the gather; with no hole anywhere, only the
  // last block (the own pool and the empty slots after it) needs a mask
  const bool any_hole = __syncthreads_or(bad) != 0;
  gather_warp(sKV + warp * kWarpStage, k, v, rows, 0, warp, lane);  // nblk >= 1
  cp_async_commit();

  float o_acc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o_acc[j][0] = o_acc[j][1] = o_acc[j][2] = o_acc[j][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  uint32_t qa[8][4];

  for (int b = 0; b < nblk; ++b) {
    cp_async_wait<0>();  // this lane's copies of block b (and, at b = 0, its part of Q)
    if (b == 0) {
      __syncthreads();  // every thread's part of Q
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int mat = lane >> 3;
        const int r = (lane & 7) + ((mat & 1) << 3);
        const int c = 2 * kk + (mat >> 1);
        ldsm_x4(sQ + swz(r, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
      __syncthreads();  // every warp has Q: block 1 may overwrite it
    } else {
      __syncwarp();  // the warp's copies of block b are visible to its lanes, and block b - 1 is read
    }
    if (b + 1 < nblk) gather_warp(sKV + ((b + 1) & 1) * kStageBytes + warp * kWarpStage, k, v, rows, b + 1, warp, lane);
    cp_async_commit();
    const uint32_t sK = sKV + (b & 1) * kStageBytes + warp * kWarpStage;
    const uint32_t sV = sK + kWarpTile;
    const int key0 = warp * 16;

    // S = Q K^T for this warp's 16 keys (two n-tiles of 8)
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int mat = lane >> 3;
      const int r = ((mat >> 1) << 3) + (lane & 7);
      const int c = 2 * kk + (mat & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(sK + swz(r, c), b0, b1, b2, b3);
      mma_bf16_16816(s0, qa[kk], b0, b1);
      mma_bf16_16816(s1, qa[kk], b2, b3);
    }

    // mask: slot of each of this thread's 4 key columns (raw scores; the
    // scale is positive, so the maxima can be taken before scaling)
    float x[8] = {s0[0], s0[1], s0[2], s0[3], s1[0], s1[1], s1[2], s1[3]};
    if (b + 1 == nblk || any_hole) {
      const int kc[4] = {key0 + 2 * t4, key0 + 2 * t4 + 1, key0 + 8 + 2 * t4, key0 + 9 + 2 * t4};
      bool valid[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) valid[e] = rows[b * kBlkKeys + row_slot(kc[e])] >= 0;
      const bool vm[8] = {valid[0], valid[1], valid[0], valid[1], valid[2], valid[3], valid[2], valid[3]};
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = vm[e] ? x[e] : -INFINITY;
    }
    // online softmax: row g holds x[0,1,4,5]; row g+8 holds x[2,3,6,7]
    float mx0 = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[4], x[5]));
    float mx1 = fmaxf(fmaxf(x[2], x[3]), fmaxf(x[6], x[7]));
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    mx0 *= scale_log2;
    mx1 *= scale_log2;
    // lagging reference: unchanged while the block's maximum stays within kLag of it
    const float mn0 = mx0 > m_run[0] + kLag ? mx0 : m_run[0];
    const float mn1 = mx1 > m_run[1] + kLag ? mx1 : m_run[1];
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = ex2_ftz(m_run[0] - mu0), al1 = ex2_ftz(m_run[1] - mu1);
    float p[8];
    p[0] = ex2_ftz(fmaf(x[0], scale_log2, -mu0));
    p[1] = ex2_ftz(fmaf(x[1], scale_log2, -mu0));
    p[4] = ex2_ftz(fmaf(x[4], scale_log2, -mu0));
    p[5] = ex2_ftz(fmaf(x[5], scale_log2, -mu0));
    p[2] = ex2_ftz(fmaf(x[2], scale_log2, -mu1));
    p[3] = ex2_ftz(fmaf(x[3], scale_log2, -mu1));
    p[6] = ex2_ftz(fmaf(x[6], scale_log2, -mu1));
    p[7] = ex2_ftz(fmaf(x[7], scale_log2, -mu1));
    l_run[0] = l_run[0] * al0 + (p[0] + p[1] + p[4] + p[5]);
    l_run[1] = l_run[1] * al1 + (p[2] + p[3] + p[6] + p[7]);
    m_run[0] = mn0;
    m_run[1] = mn1;
    // the accumulators are rescaled only when some row of the warp moved its
    // reference (a factor of exactly 1 leaves them unchanged)
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o_acc[j][0] *= al0;
        o_acc[j][1] *= al0;
        o_acc[j][2] *= al1;
        o_acc[j][3] *= al1;
      }
    }
    uint32_t pa[4];
    pa[0] = pack_bf16(p[0], p[1]);
    pa[1] = pack_bf16(p[2], p[3]);
    pa[2] = pack_bf16(p[4], p[5]);
    pa[3] = pack_bf16(p[6], p[7]);
    // O += P V: V rows are the k dimension (ldmatrix .trans)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int mat = lane >> 3;
      const int r = ((mat & 1) << 3) + (lane & 7);
      const int c = 2 * j + (mat >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(sV + swz(r, c), b0, b1, b2, b3);
      mma_bf16_16816(o_acc[2 * j], pa, b0, b1);
      mma_bf16_16816(o_acc[2 * j + 1], pa, b2, b3);
    }
  }
  cp_async_wait<0>();

  // ---- merge the four warps' partial states
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
    l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
  }
  if (t4 == 0) {
    s_m[warp][g] = m_run[0];
    s_m[warp][g + 8] = m_run[1];
    s_l[warp][g] = l_run[0];
    s_l[warp][g + 8] = l_run[1];
  }
  __syncthreads();
  float fac[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = g + 8 * hh;
    float M = s_m[0][h];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_m[w][h]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) L += s_l[w][h] * exp2f(s_m[w][h] - M);
    const float mine = m_run[hh] == -INFINITY ? 0.f : exp2f(m_run[hh] - M);
    fac[hh] = mine / L;
    if (warp == 0 && t4 == 0) lse[r * kHq + h] = (M + log2f(L)) * kLn2;
  }
  // partial O (already normalised) into shared memory, one [16][132] fp32 slab
  // per warp (padded rows spread the fragment stores over the banks)
  constexpr int kRedLd = kD + 4;
  float* red = reinterpret_cast<float*>(gbase);  // reuses the gather ring
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int col = 8 * j + 2 * t4;
    *reinterpret_cast<float2*>(red + (warp * kHq + g) * kRedLd + col) =
        make_float2(o_acc[j][0] * fac[0], o_acc[j][1] * fac[0]);
    *reinterpret_cast<float2*>(red + (warp * kHq + g + 8) * kRedLd + col) =
        make_float2(o_acc[j][2] * fac[1], o_acc[j][3] * fac[1]);
  }
  __syncthreads();
  // thread tid owns element pairs e = 2 * (tid + 128 m), m = 0..7 (consecutive across threads)
  __nv_bfloat16* orow = o + r * (kHq * kD);
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
    *reinterpret_cast<uint32_t*>(orow + e) = pack_bf16(a0, a1);
  }
}

}  // namespace

cudaError_t launch_attn_fwd(const void* q, const void* k, const void* v, const int32_t* pool_idx, int64_t q_begin,
                            int64_t q_end, int topk, float scale, void* o, float* lse, const LaunchCtx& ctx,
                            const SeqTable* tab) {
  if (q_end <= q_begin) return cudaSuccess;
  static const SeqTable kNoTable = {};
  static std::atomic<bool> attr_done[kAttrDevices];
  const cudaError_t e = set_smem_limit_once(attn_fwd_kernel, static_cast<int>(smem_bytes(kMaxTopk)), attr_done);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<<<static_cast<unsigned>(q_end - q_begin), kThreads, smem_bytes(topk), ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), pool_idx, q_begin, topk, scale * kLog2e, static_cast<__nv_bfloat16*>(o), lse,
      ctx.status, tab ? *tab : kNoTable);
  return cudaGetLastError();
}

}  // namespace dsa
