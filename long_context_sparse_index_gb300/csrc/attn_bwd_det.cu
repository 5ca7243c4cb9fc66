// attn_bwd_det.cu -- deterministic dK/dV for the sparse attention backward.
//
// [SkyRL-1M §模型与瓶颈] the selected-key attention is trained end to end; for
// key j of pool p the gradient sums over every query i whose key set holds it:
//   dv_j = sum_i sum_h P_ihj dO_ih        dk_j = scale * sum_i sum_h dS_ihj q_ih
// The default backward adds each query's contribution with fp32 atomics, so
// the summation order (and the last bits) vary from run to run.  Here the
// sums run key-major in a fixed order, so the gradients are reproducible bit
// for bit:
//   1. transpose: for every pool, the queries that selected it, ascending
//      (a counting sort that is stable by construction: per-(pool, query
//      block) counts, one exclusive scan, then each query block fills its
//      cells in query order);
//   2. one launch per span of 4096 queries (span order fixes the order of
//      the sums): a CTA takes a pool, and each of its four warps keeps the
//      pool's 4 keys' K/V in registers and runs over a fixed quarter of the
//      pool's queries in the span (its own partial-pool queries first, then
//      its selecting queries, ascending) with bf16 mma.sync (P and scale*dS
//      split into bf16 hi + lo, both halves in one MMA's columns); the four
//      sums are added in warp order into the pool's fp32 dK/dV rows, which
//      no other CTA of the launch touches.  A span's q and dO (32 MB) stay
//      in L2 while every pool's CTA reads them;
//   3. the fp32 rows are rounded to bf16.
// dq comes from the default backward kernel with its dK/dV part switched off.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
namespace {

constexpr int kHq = 16;
constexpr int kD = 128;
constexpr int kSpan = 4096;            // queries per span (one launch each)
constexpr int kSegWarps = 4;           // warps per CTA of the span kernel
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ transpose
// One warp per query row: the row's valid entries are its leading
// non-negative ones (the first -1 ends the selection) that are eligible pools;
// ineligible or non-ascending entries are reported, and ineligible ones are
// left out, exactly as the attention kernels treat them.
__global__ void det_count_kernel(const int32_t* __restrict__ pool_idx, int64_t S, int topk, int qb_size, int nb,
                                 uint32_t* __restrict__ cnt, int32_t* __restrict__ nsel_out, unsigned* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
  if (i >= S) return;
  const int32_t* row = pool_idx + i * topk;
  const int64_t n_elig = i >> 2;
  const int b = static_cast<int>(i / qb_size);
  int nsel = topk;
  for (int j0 = 0; j0 < topk; j0 += 32) {
    const int j = j0 + lane;
    const unsigned neg = __ballot_sync(0xffffffffu, j < topk && row[j < topk ? j : 0] < 0);
    if (neg) {
      nsel = j0 + __ffs(neg) - 1;
      break;
    }
  }
  bool bad = false;
  for (int j = lane; j < nsel; j += 32) {
    const int32_t p = row[j];
    if (p >= n_elig) bad = true;
    else atomicAdd(&cnt[static_cast<int64_t>(p) * nb + b], 1u);
    if (j > 0 && p <= row[j - 1]) bad = true;
  }
  if (lane == 0) nsel_out[i] = nsel;
  if (__any_sync(0xffffffffu, bad) && lane == 0) record_status(status, kStatusInternal);
}

// One CTA per query block: queries in order, a barrier between them, so each
// (pool, block) cell receives its queries ascending.
__global__ void det_fill_kernel(const int32_t* __restrict__ pool_idx, const int32_t* __restrict__ nsel_in, int64_t S,
                                int topk, int qb_size, int nb, uint32_t* __restrict__ cur, int32_t* __restrict__ qlist) {
  const int b = blockIdx.x;
  const int64_t i0 = static_cast<int64_t>(b) * qb_size;
  const int64_t i1 = min(S, i0 + qb_size);
  for (int64_t i = i0; i < i1; ++i) {
    const int32_t* row = pool_idx + i * topk;
    const int nsel = nsel_in[i];
    const int64_t n_elig = i >> 2;
    for (int j = threadIdx.x; j < nsel; j += blockDim.x) {
      const int32_t p = row[j];
      if (p < n_elig) {
        // distinct pools within a row touch distinct cells; the atomic only
        // keeps a malformed row with a repeated pool from losing an entry
        const uint32_t pos = atomicAdd(&cur[static_cast<int64_t>(p) * nb + b], 1u);
        qlist[pos] = static_cast<int32_t>(i);
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ exclusive scan (uint32, in place)
constexpr int kScanThreads = 1024;
constexpr int kScanPer = 4;
constexpr int kScanTile = kScanThreads * kScanPer;

__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = warp_tot[lane];
    uint32_t u = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, u, o);
      if (lane >= o) u += y;
    }
    warp_tot[lane] = u - t;
    if (lane == 31) warp_tot[32] = u;
  }
  __syncthreads();
  const uint32_t r = warp_tot[warp] + x - v;
  *total = warp_tot[32];
  __syncthreads();
  return r;
}

// each CTA scans kScanTile elements; tile totals go to bsum
__global__ void scan_tiles_kernel(uint32_t* __restrict__ a, int64_t n, uint32_t* __restrict__ bsum) {
  __shared__ uint32_t wt[33];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile + threadIdx.x * kScanPer;
  uint32_t v[kScanPer], s = 0;
#pragma unroll
  for (int q = 0; q < kScanPer; ++q) {
    v[q] = base + q < n ? a[base + q] : 0u;
    s += v[q];
  }
  uint32_t tot;
  uint32_t run = block_excl_scan(s, wt, &tot);
#pragma unroll
  for (int q = 0; q < kScanPer; ++q) {
    if (base + q < n) a[base + q] = run;
    run += v[q];
  }
  if (threadIdx.x == 0) bsum[blockIdx.x] = tot;
}

// one CTA: exclusive scan of the tile totals (nt <= kScanThreads * 16); the
// grand total goes to *total_out
__global__ void scan_top_kernel(uint32_t* __restrict__ bsum, int64_t nt, uint32_t* __restrict__ total_out) {
  __shared__ uint32_t wt[33];
  constexpr int kPer = 16;
  const int64_t base = static_cast<int64_t>(threadIdx.x) * kPer;
  uint32_t v[kPer], s = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    v[q] = base + q < nt ? bsum[base + q] : 0u;
    s += v[q];
  }
  uint32_t tot;
  uint32_t run = block_excl_scan(s, wt, &tot);
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    if (base + q < nt) bsum[base + q] = run;
    run += v[q];
  }
  if (threadIdx.x == 0 && total_out) *total_out = tot;
}

__global__ void scan_add_kernel(uint32_t* __restrict__ a, int64_t n, const uint32_t* __restrict__ bsum) {
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile + threadIdx.x * kScanPer;
  const uint32_t add = bsum[blockIdx.x];
#pragma unroll
  for (int q = 0; q < kScanPer; ++q)
    if (base + q < n) a[base + q] += add;
}

// ------------------------------------------------------------------ pool items
// After the fill, cur[c] is the end of cell c = p * nb + b (and the start of
// cell c + 1).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * 256 + ((c ^ (r & 7)) << 4));
}

struct ItemArgs {
  const __nv_bfloat16* dO;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* lse;
  const float* delta;
  const int32_t* qlist;
  const uint32_t* cur;   // cell ends (after the fill)
  int64_t S, P;
  int nb;                // counting blocks of qb queries
  int G;                 // counting blocks per span
  int64_t span;          // queries per span: G * qb
  float scale, scale_log2;
  float* dk_acc;         // [S][128] fp32
  float* dv_acc;
  uint32_t* tickets;     // one counter per span, zero before the span's launch
};

constexpr uint32_t kStageTile = kHq * kD * 2;  // 4 KB: one query's q (or dO)
struct ItemSmem {
  union {
    uint8_t stage[kSegWarps][2][2][kStageTile];  // [warp][buffer][q, dO]
    float4 comb[kSegWarps][8][2][32];            // [warp][m-tile][dK, dV][lane]: the warps' sums
  };
  uint32_t t[kSegWarps][2][8 * 8];               // [warp][P, dS][column][head pair]
  uint32_t ticket;
};
constexpr size_t kItemSmem = sizeof(ItemSmem) + 128;

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  return __ldcs(reinterpret_cast<const unsigned int*>(p));
}

// Span `sp`: pools p with 4p <= its last query.  A pool's queries in the
// span are its own partial-pool queries 4p .. 4p+3 (when they fall in the
// span, keys causal) and then the queries of cells (p, G*sp .. G*sp+G-1),
// ascending.  A CTA takes one pool at a time; warp w sums the w-th quarter
// of those queries in order, and the four sums are added in warp order.
// Everything but the span's q and dO is read or written once per pool, with
// evict-first hints, so the span's q and dO keep the L2.
__global__ void __launch_bounds__(32 * kSegWarps) det_item_kernel(const ItemArgs a, int sp) {
  extern __shared__ uint8_t item_raw[];
  ItemSmem& sm = *reinterpret_cast<ItemSmem*>(item_raw + ((128u - (smem_u32(item_raw) & 127u)) & 127u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int64_t q_lo = static_cast<int64_t>(sp) * a.span;
  const int64_t q_hi = min(a.S, q_lo + a.span);
  const int64_t pmax = (q_hi - 1) / 4 + 1;
  const int b0 = sp * a.G, b1 = min(a.nb, b0 + a.G) - 1;
  const uint32_t sq[2] = {smem_u32(sm.stage[warp][0][0]), smem_u32(sm.stage[warp][1][0])};
  const uint32_t sd[2] = {smem_u32(sm.stage[warp][0][1]), smem_u32(sm.stage[warp][1][1])};
  uint16_t* tw = reinterpret_cast<uint16_t*>(sm.t[warp]);
  for (;;) {
    __syncthreads();  // the previous pool's sums are read; the ticket may be rewritten
    if (threadIdx.x == 0) sm.ticket = atomicAdd(&a.tickets[sp], 1u);
    __syncthreads();
    const int64_t p = sm.ticket;
    if (p >= pmax) break;
    uint32_t ls = 0, le = 0;
    if (p < a.P) {
      const int64_t c0 = p * a.nb + b0;
      ls = c0 > 0 ? ld_stream_u32(a.cur + c0 - 1) : 0u;
      le = ld_stream_u32(a.cur + p * a.nb + b1);
    }
    const int64_t key0 = 4 * p;
    const int n_own = key0 >= q_lo ? static_cast<int>(a.S - key0 < 4 ? a.S - key0 : 4) : 0;
    const uint32_t n = static_cast<uint32_t>(n_own) + (le - ls);
    if (n == 0) continue;
    // this warp's quarter of the pool's entries
    const uint32_t w0 = static_cast<uint32_t>((static_cast<uint64_t>(n) * warp) / kSegWarps);
    const uint32_t w1 = static_cast<uint32_t>((static_cast<uint64_t>(n) * (warp + 1)) / kSegWarps);

    // K and V of the pool as B fragments (column n = key g; keys 4..7 are zero)
    uint32_t kb[8][2], vb[8][2];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const bool kv = g < 4 && key0 + g < a.S;
      const int64_t off = (key0 + (kv ? g : 0)) * kD + kk * 16 + 2 * t4;
      kb[kk][0] = kv ? ld_stream_u32(a.k + off) : 0u;
      kb[kk][1] = kv ? ld_stream_u32(a.k + off + 8) : 0u;
      vb[kk][0] = kv ? ld_stream_u32(a.v + off) : 0u;
      vb[kk][1] = kv ? ld_stream_u32(a.v + off + 8) : 0u;
    }
    // dK^T / dV^T per m-tile of 16 dims: C columns 0..3 = keys (hi halves), 4..7 = keys (lo halves)
    float dk[8][4], dv[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) dk[mt][e] = dv[mt][e] = 0.f;

    auto query_of = [&](uint32_t e) -> int64_t {
      return static_cast<int>(e) < n_own ? key0 + e : static_cast<int64_t>(ld_stream_u32(a.qlist + ls + e - n_own));
    };
    auto stage = [&](int buf, int64_t i) {
      const __nv_bfloat16* qr = a.q + i * (kHq * kD);
      const __nv_bfloat16* dr = a.dO + i * (kHq * kD);
#pragma unroll
      for (int u = 0; u < (kHq * 16) / 32; ++u) {
        const int c = lane + 32 * u;
        cp_async16(sq[buf] + swz(c >> 4, c & 15), qr + c * 8, true);
        cp_async16(sd[buf] + swz(c >> 4, c & 15), dr + c * 8, true);
      }
      cp_async_commit();
    };
    if (w0 < w1) stage(0, query_of(w0));
    int buf = 0;
    for (uint32_t e = w0; e < w1; ++e, buf ^= 1) {
      const int64_t i = query_of(e);
      if (e + 1 < w1) {
        stage(buf ^ 1, query_of(e + 1));
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncwarp();
      // S = q K^T and dP = dO V^T  (16 heads x 8 columns)
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int mat = lane >> 3;
        const int r = (lane & 7) + ((mat & 1) << 3);
        const int c = 2 * kk + (mat >> 1);
        uint32_t qa[4], da[4];
        ldsm_x4(sq[buf] + swz(r, c), qa[0], qa[1], qa[2], qa[3]);
        ldsm_x4(sd[buf] + swz(r, c), da[0], da[1], da[2], da[3]);
        mma_bf16_16816(sc, qa, kb[kk][0], kb[kk][1]);
        mma_bf16_16816(dp, da, vb[kk][0], vb[kk][1]);
      }
      // P and scale * dS for heads g, g+8 and keys 2t4, 2t4+1 (lanes t4 < 2
      // hold the four real keys), split into bf16 hi (column key) and lo
      // (column key + 4) of the transposed [column][head] tiles
      if (t4 < 2) {
        const float l0 = a.lse[i * kHq + g] * kLog2e, l1 = a.lse[i * kHq + g + 8] * kLog2e;
        const float d0 = a.delta[i * kHq + g], d1 = a.delta[i * kHq + g + 8];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int key = 2 * t4 + (e2 & 1), head = g + (e2 >= 2 ? 8 : 0);
          const bool hi_row = e2 >= 2;
          const bool valid = key0 + key <= i;  // selected pools lie wholly before the query
          const float P = valid ? exp2f(sc[e2] * a.scale_log2 - (hi_row ? l1 : l0)) : 0.f;
          const float xs[2] = {P, a.scale * P * (dp[e2] - (hi_row ? d1 : d0))};
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const __nv_bfloat16 h = __float2bfloat16_rn(xs[m]);
            const __nv_bfloat16 l = __float2bfloat16_rn(xs[m] - __bfloat162float(h));
            tw[m * 128 + key * 16 + head] = *reinterpret_cast<const uint16_t*>(&h);
            tw[m * 128 + (key + 4) * 16 + head] = *reinterpret_cast<const uint16_t*>(&l);
          }
        }
      }
      __syncwarp();
      uint32_t pb[2][2];  // [P, dS]: B fragment (k = heads 2t4.., n = column g)
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        pb[m][0] = sm.t[warp][m][g * 8 + t4];
        pb[m][1] = sm.t[warp][m][g * 8 + 4 + t4];
      }
      // dV^T += dO^T P ;  dK^T += q^T (scale dS)   (m-tiles of 16 dims; A from ldmatrix.trans)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int mat = lane >> 3;
        const int r = (lane & 7) + ((mat >> 1) << 3);  // head row of the staged [16 heads][128 dims] tile
        const int c = 2 * mt + (mat & 1);              // 16-byte chunk: dims 8c .. 8c+7
        uint32_t ad[4], aq[4];
        ldsm_x4_t(sd[buf] + swz(r, c), ad[0], ad[1], ad[2], ad[3]);
        mma_bf16_16816(dv[mt], ad, pb[0][0], pb[0][1]);
        ldsm_x4_t(sq[buf] + swz(r, c), aq[0], aq[1], aq[2], aq[3]);
        mma_bf16_16816(dk[mt], aq, pb[1][0], pb[1][1]);
      }
      __syncwarp();  // the stage buffer and the transpose tiles are rewritten next
    }
    // hi + lo (lanes t4 < 2 take the lo columns from lane + 2), to shared memory
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      float xk[4], xv[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        xk[e2] = dk[mt][e2] + __shfl_down_sync(0xffffffffu, dk[mt][e2], 2);
        xv[e2] = dv[mt][e2] + __shfl_down_sync(0xffffffffu, dv[mt][e2], 2);
      }
      dk[mt][0] = xk[0], dk[mt][1] = xk[1], dk[mt][2] = xk[2], dk[mt][3] = xk[3];
      dv[mt][0] = xv[0], dv[mt][1] = xv[1], dv[mt][2] = xv[2], dv[mt][3] = xv[3];
    }
    __syncthreads();  // every warp is done with its stage buffers
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      sm.comb[warp][mt][0][lane] = make_float4(dk[mt][0], dk[mt][1], dk[mt][2], dk[mt][3]);
      sm.comb[warp][mt][1][lane] = make_float4(dv[mt][0], dv[mt][1], dv[mt][2], dv[mt][3]);
    }
    __syncthreads();
    // warp w adds m-tiles 2w, 2w+1 of the four warps' sums, in warp order, into
    // the pool's fp32 rows: keys 2t4 + (e2 & 1), dims mt*16 + g (+8)
    if (t4 < 2) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int mt = 2 * warp + h;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          float4 acc4 = sm.comb[0][mt][x][lane];
#pragma unroll
          for (int w = 1; w < kSegWarps; ++w) {
            const float4 y = sm.comb[w][mt][x][lane];
            acc4.x += y.x, acc4.y += y.y, acc4.z += y.z, acc4.w += y.w;
          }
          const float vals[4] = {acc4.x, acc4.y, acc4.z, acc4.w};
          float* dst = x == 0 ? a.dk_acc : a.dv_acc;
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int key = 2 * t4 + (e2 & 1), dim = mt * 16 + g + (e2 >= 2 ? 8 : 0);
            if (key0 + key < a.S) {
              float* o = dst + (key0 + key) * kD + dim;
              __stcs(o, __ldcs(o) + vals[e2]);
            }
          }
        }
      }
    }
  }
}

int64_t scan_tiles(int64_t n) { return (n + kScanTile - 1) / kScanTile; }

cudaError_t scan_inplace(uint32_t* a, int64_t n, uint32_t* bsum, uint32_t* total, cudaStream_t st) {
  const int64_t nt = scan_tiles(n);
  if (nt == 0) return cudaSuccess;
  scan_tiles_kernel<<<static_cast<unsigned>(nt), kScanThreads, 0, st>>>(a, n, bsum);
  scan_top_kernel<<<1, kScanThreads, 0, st>>>(bsum, nt, total);
  scan_add_kernel<<<static_cast<unsigned>(nt), kScanThreads, 0, st>>>(a, n, bsum);
  return cudaGetLastError();
}

}  // namespace

int64_t det_scan_max_elems() { return static_cast<int64_t>(kScanThreads) * 16 * kScanTile; }

DetPlan det_plan(int64_t S, int topk) {
  DetPlan d;
  d.P = S / 4;
  d.nP = (S + 3) / 4;
  // counting blocks of 1024 queries, coarser where P * blocks would outgrow
  // the scan (finer blocks, tried at 256, only add counters); one block at
  // most (then P itself may exceed the scan: the caller rejects that shape)
  int64_t qb = 1024;
  while (qb < S && d.P * ((S + qb - 1) / qb) > det_scan_max_elems()) qb *= 2;
  d.qb = static_cast<int>(qb < S ? qb : (S > 0 ? S : 1));
  d.nb = static_cast<int>((S + d.qb - 1) / d.qb);
  d.G = d.qb < kSpan ? kSpan / d.qb : 1;  // spans of 4096 queries (or one counting block)
  d.nspan = (d.nb + d.G - 1) / d.G;
  d.cnt_n = d.P * d.nb;
  d.bsum_n = scan_tiles(d.cnt_n) + 1;
  (void)topk;
  return d;
}

int det_lists_kernels(const DetPlan& d) { return 1 + (d.cnt_n > 0 ? 4 : 0); }

cudaError_t launch_det_lists(const int32_t* pool_idx, int64_t S, int topk, const DetPlan& d, const DetBuffers& w,
                             const LaunchCtx& ctx) {
  cudaStream_t st = ctx.stream;
  cudaError_t e = cudaMemsetAsync(w.tickets, 0, static_cast<size_t>(d.nspan) * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  if (d.cnt_n > 0) {
    e = cudaMemsetAsync(w.cnt, 0, static_cast<size_t>(d.cnt_n) * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
  }
  det_count_kernel<<<static_cast<unsigned>((S + 7) / 8), 256, 0, st>>>(pool_idx, S, topk, d.qb, d.nb, w.cnt, w.nsel,
                                                                       ctx.status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (d.cnt_n > 0) {
    if ((e = scan_inplace(w.cnt, d.cnt_n, w.bsum, nullptr, st)) != cudaSuccess) return e;
    det_fill_kernel<<<static_cast<unsigned>(d.nb), 512, 0, st>>>(pool_idx, w.nsel, S, topk, d.qb, d.nb, w.cnt, w.qlist);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_det_span(const void* dO, const void* q, const void* k, const void* v, const float* lse,
                            const float* delta, int64_t S, float scale, const DetPlan& d, const DetBuffers& w, int sp,
                            const LaunchCtx& ctx) {
  ItemArgs a;
  a.dO = static_cast<const __nv_bfloat16*>(dO);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.lse = lse;
  a.delta = delta;
  a.qlist = w.qlist;
  a.cur = w.cnt;
  a.S = S;
  a.P = d.P;
  a.nb = d.nb;
  a.G = d.G;
  a.span = static_cast<int64_t>(d.G) * d.qb;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.dk_acc = w.dk_acc;
  a.dv_acc = w.dv_acc;
  a.tickets = w.tickets;
  static std::atomic<bool> attr_done[kAttrDevices];
  const cudaError_t e = set_smem_limit_once(det_item_kernel, static_cast<int>(kItemSmem), attr_done);
  if (e != cudaSuccess) return e;
  det_item_kernel<<<static_cast<unsigned>(ctx.num_sms * 3), 32 * kSegWarps, kItemSmem, ctx.stream>>>(a, sp);
  return cudaGetLastError();
}

}  // namespace dsa
