// index_topk.cu -- pooled indexer keys, and the causal pooled indexer with
// its per-query top-k as one persistent kernel that never stores the score
// matrix: each tile's scores are compared in the epilogue against the row's
// threshold, and only the pools at or above it are kept, as candidates.
//
// [SkyRL-1M §模型与瓶颈] the indexer scores every query against every earlier
// 4-token key pool; [§1 DSA 真稀疏; Anyscale, second lesson (the indexer)] it
// does so one query chunk at a time so the score matrix is never whole, and
// keeps each query's best pools as int32 indices.
//
//   Khat_p     = ((k[4p] + k[4p+1]) + (k[4p+2] + k[4p+3])) * 0.25    (fp32)
//   score(i,p) = sum_h w[i,h] * ReLU(q_idx[i,h,:] . Khat_p)
//
// Pools are ranked by the composite key (score desc, index asc).  For query i
// with n = floor(i/4) eligible pools (n > topk; shorter rows keep all pools):
//   * n <= cap: every eligible pool is a candidate;
//   * n > cap: the threshold is the rsel-th largest composite key among the
//     row's sampled pools (every sigma-th pool); about rsel * sigma pools of
//     the row lie above it, which is more than topk and fewer than cap.
// The row's candidates are the pools at or above its threshold.  When there
// are at least topk of them (and no more than cap), the row's top-k is among
// them, and selecting from the candidates is exact; otherwise the row is
// listed for the fallback kernel, which recomputes all its scores.
//
// Work items, for each query chunk c (rows row0 .. row0+nrows-1):
//   sample  (128-query block, 256 sampled pools): the block's scores against
//           every sigma-th pool, stored in the chunk's sample buffer;
//   thresh  four rows: each row's threshold from its samples; zeroes its
//           candidate count;
//   tile    (128-query block, 256-pool tile): the indexer scores; the
//           epilogue appends the row's pools at or above its threshold to
//           its candidate list (slots from one atomic add per thread);
//   rows    four rows: each row's top-k from its candidate list.
// A sample or tile item: TMA brings the 64 KB Khat hi/lo tile and, per head
// h, the q_idx tile of head h; one 128x256x128 bf16 tcgen05 MMA chain per head
// accumulates q_h . [Khat_hi ; Khat_lo] in TMEM (Khat as a bf16 hi/lo pair:
// the product keeps ~16 more mantissa bits than one bf16 rounding); 16
// epilogue warps fold ReLU, the head weight and the sum over heads into
// registers while the next head's MMA fills the other TMEM buffer.  For
// thresh and rows items the 16 warps form four 128-thread groups, one row
// each (topk_cand.cuh).
//
// Items come from one global ticket counter, step by step; step s holds
//     sample(s), thresh(s-1-L), tile(s-2-L), rows(s-2-2L)
// with L = min(3, (nbuf-1)/2), and chunk c uses slot c % nbuf of a ring of
// per-chunk buffers (samples, thresholds, candidate counts and lists).  Every
// wait is on an earlier step (L < nbuf-1), or on an earlier item of the same
// step: a sample item (step c) waits, before storing, for the thresh items
// of chunk c-nbuf (step c-nbuf+1+L) to be done reading the slot's samples;
// thresh(c) (step c+1+L) waits for the samples of c and for the rows of
// c-nbuf (step c-nbuf+2+2L), done with the slot's candidates; a tile waits,
// before appending, for thresh(c); rows(c) wait for the tiles of c.  L steps
// between samples and thresholds and between tiles and rows give the items
// waited for time to finish when a step holds fewer items than CTAs.  With one CTA
// per SM (cooperative launch: all resident), the lowest unfinished ticket can
// always proceed.  There is no barrier per chunk, and the chunk size only
// bounds the per-chunk buffers.
#include "dsa_device.cuh"
#include "dsa_kernels.h"
#include "topk_cand.cuh"
#include "topk_row.cuh"
#include "topk_warp.cuh"

namespace dsa {
namespace {

constexpr int kBM = 128;           // queries per tile (TMEM lanes)
constexpr int kBN = 256;           // pools per tile (TMEM columns per buffer)
constexpr int kDi = 64;            // indexer head dim
constexpr int kAStages = 4;
constexpr int kItems = 2;          // work-item ring between the roles (the item in work + one prefetched)
constexpr int kRowsPerGroupItem = 4;   // topk > 512: one row per 128-thread group
constexpr int kRowsPerWarpItem = 16;   // topk <= 512: one row per epilogue warp
constexpr int kMaxLead = 3;        // thresholds of chunk c come in step c + 1 + lead, rows in c + 2 + 2 lead
constexpr uint32_t kABytes = kBM * kDi * 2;        // 16 KB: q_idx tile of one head
constexpr uint32_t kBHalf = kBN * kDi * 2;         // 32 KB: Khat hi (or lo) tile
constexpr uint32_t kBBytes = 2 * kBHalf;           // 64 KB, one stage
constexpr int kEpiWarps = 16;                      // 4 TMEM lane quarters x 4 column quarters
constexpr int kEpiCols = kBN / 4;                  // 64 columns per epilogue thread
constexpr int kEpiWarp0 = 3;                       // first epilogue warp
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);  // TMA warp, MMA warp, scheduler warp, 16 epilogue warps
constexpr uint32_t kTmemCols = 512;                // 2 accumulators x 256 columns
constexpr uint32_t kCtlOff = kBBytes + kAStages * kABytes;
constexpr uint32_t kCtlBytes = 512;
constexpr uint32_t kThrOff = kCtlOff + kCtlBytes;   // thresholds of a tile's rows, per ring slot
constexpr uint32_t kThrBytes = kItems * kBM * 8;
constexpr uint32_t kGrpOff = kThrOff + kThrBytes;
// Sample stores go through a per-warp staging tile (32 rows x 32 columns,
// rows padded to 36 floats), so that each warp store covers four rows x 128
// contiguous bytes; it shares space with the groups' selection buffers.
constexpr int kStgLd = 36;
constexpr uint32_t kStgBytes = 32 * kStgLd * 4;
constexpr size_t cmax(size_t x, size_t y) { return x > y ? x : y; }
constexpr size_t kGrpBytes =
    cmax(cmax(kRowsPerGroupItem * sizeof(cand::Smem), kEpiWarps * kStgBytes), kEpiWarps * sizeof(wsel::Smem));
constexpr size_t kSmemBytes = 1024 + kGrpOff + kGrpBytes;
static_assert(kRowsPerGroupItem * topk::kGT == 32 * kEpiWarps, "the epilogue warps form the top-k groups");
static_assert(kRowsPerWarpItem == kEpiWarps, "one row per epilogue warp");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(sizeof(cand::Smem) % 16 == 0, "group buffers stay 16-byte aligned");

constexpr int kEpiBar = 1;  // named barrier of the 512 epilogue threads; the groups use 2..5

// control block offsets (bytes from kCtlOff)
constexpr uint32_t kBarAFull = 0, kBarAEmpty = 32, kBarBFull = 64, kBarBEmpty = 72, kBarAccFull = 80,
                   kBarAccEmpty = 96, kBarDrain = 112, kBarItemFull = 120, kBarItemEmpty = 136, kBarDeps = 152,
                   kBarDone = 168;
constexpr uint32_t kTmemSlot = 184, kAbort = 188, kGroupOk = 192, kWaitOk = 196, kItemData = 256;  // kItems x 16 B
static_assert(kItems == 2 && kItemData + kItems * 16 <= kCtlBytes, "control block");

enum : int { kItemSample = 0, kItemThresh = 1, kItemTile = 2, kItemRows = 3, kItemEnd = 4 };
struct Item {
  int kind;
  int chunk;
  int a;  // sample, tile: qb        thresh, rows: first row within the chunk
  int b;  // sample: sample tile     tile: pb      thresh, rows: number of rows (1..4)
};

// global 64-bit words, zeroed by pool_keys_kernel before each launch; the
// done counters are per slot (chunk c uses slot c % nbuf) and cumulative
enum : int {
  kTicket = 0,
  kSampDone = 1,                 // kMaxBufs words: sample tiles stored
  kThrDone = 1 + kMaxBufs,       // rows whose threshold is set
  kTilesDone = 1 + 2 * kMaxBufs, // tiles appended
  kRowsDone = 1 + 3 * kMaxBufs,  // rows selected
  kGAbort = 1 + 4 * kMaxBufs
};
static_assert(kGAbort < kIndexFallbackRowsWord && kIndexFallbackRowsWord < kIndexSyncWords, "global words");

struct Args {
  const float* w;
  float* samples;       // per slot: slot_rows rows x samp_ld sampled scores
  int64_t samp_ld, samp_slot;
  uint2* cands;         // per slot: slot_rows rows x cap candidates (score key, pool)
  int64_t cand_slot;
  uint2* thr;           // per slot: thr_ld thresholds (score key, pool), one per row
  unsigned* cnt;        // per slot: thr_ld candidate counts
  int64_t thr_ld;       // slot rows rounded up to 128 (a tile's 128 thresholds are 16-byte aligned)
  int cap;
  int sigma;            // sample stride in pools
  int rsel;             // the threshold is the rsel-th largest sample
  int rpi;              // rows per thresh / rows item: 16 (one per warp, topk <= 512) or 4 (one per group)
  int nbuf;             // slots, 1 .. kMaxBufs
  int lead;             // min(kMaxLead, (nbuf - 1) / 2)
  int lag;              // = lead
  int64_t q_begin, q_end;
  int chunk;
  int nchunks;
  int Hi;
  int topk;
  int32_t* pool_idx;
  int32_t* fb_rows;     // rows listed for the fallback kernel
  IndexTraceRec* trace;  // item-trace build only (DSA_ITEM_TRACE)
  unsigned long long* trace_count;
  int64_t trace_cap;
  unsigned long long* sync;
  unsigned* status;
  uint64_t limit_ns;
  int inject;
};

struct Chunk {
  int64_t row0;
  int nrows;
  int nqb;
  int npb_max;
  int ntiles;  // nqb * npb_max (tiles past the causal edge included); 0 when no row has more than topk pools
};

__device__ __forceinline__ Chunk chunk_of(const Args& a, int c) {
  Chunk ch;
  ch.row0 = a.q_begin + static_cast<int64_t>(c) * a.chunk;
  ch.nrows = static_cast<int>(min(static_cast<int64_t>(a.chunk), a.q_end - ch.row0));
  ch.nqb = (ch.nrows + kBM - 1) / kBM;
  const int64_t n_last = (ch.row0 + ch.nrows - 1) / 4;  // pools eligible for the chunk's last query
  ch.npb_max = static_cast<int>((n_last + kBN - 1) / kBN);
  ch.ntiles = n_last > a.topk ? ch.nqb * ch.npb_max : 0;
  return ch;
}

// pools eligible for the last query of block qb
__device__ __forceinline__ int64_t block_pools(const Chunk& ch, int qb) {
  const int64_t end = min(ch.row0 + static_cast<int64_t>(qb + 1) * kBM, ch.row0 + ch.nrows);
  return (end - 1) / 4;
}

__device__ __forceinline__ int pool_tiles_of(const Chunk& ch, int qb) {
  return static_cast<int>((block_pools(ch, qb) + kBN - 1) / kBN);
}

// sample tiles of block qb: only blocks with a row past cap pools need samples
__device__ __forceinline__ int sample_tiles_of(const Args& a, const Chunk& ch, int qb) {
  const int64_t n = block_pools(ch, qb);
  if (ch.ntiles == 0 || n <= a.cap) return 0;
  const int64_t G = (n + a.sigma - 1) / a.sigma;
  return static_cast<int>((G + kBN - 1) / kBN);
}

__device__ __forceinline__ int sample_tiles(const Args& a, const Chunk& ch) {
  int n = 0;
  for (int qb = 0; qb < ch.nqb; ++qb) n += sample_tiles_of(a, ch, qb);
  return n;
}

// Tiles of the chunk that hold eligible pairs (the ones that are computed).
// Only these count toward the chunk's completion: a count raised when a
// ticket is taken could run ahead of a store that is still waiting.
__device__ __forceinline__ unsigned long long valid_tiles(const Chunk& ch) {
  if (ch.ntiles == 0) return 0ull;
  unsigned long long n = 0;
  for (int qb = 0; qb < ch.nqb; ++qb) n += static_cast<unsigned long long>(pool_tiles_of(ch, qb));
  return n;
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Bounded spin of one thread until *ctr >= target.  False when the time limit
// runs out or some CTA has raised the global abort word.
__device__ bool wait_counter(const Args& a, const unsigned long long* ctr, unsigned long long target) {
  if (ld_acquire(ctr) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (ld_acquire(ctr) >= target) return true;
    if (*reinterpret_cast<const volatile unsigned long long*>(a.sync + kGAbort) != 0ull) return false;
    if (globaltimer_ns() - t0 > a.limit_ns) return false;
    __nanosleep(128);
  }
}

__device__ __forceinline__ void raise_abort(const Args& a, volatile int* local_abort) {
  *local_abort = 1;
  atomicExch(a.sync + kGAbort, 1ull);
  record_status(a.status, kStatusTimeout);
}

// Item-trace build: epilogue thread 0 records each item (see IndexTraceRec).
__device__ __forceinline__ void trace_item(const Args& a, int kind, int chunk, uint64_t t0, uint64_t t1, uint64_t t2) {
#ifdef DSA_ITEM_TRACE
  if (a.trace == nullptr) return;
  const uint64_t t3 = globaltimer_ns();
  const unsigned long long slot = atomicAdd(a.trace_count, 1ull);
  if (static_cast<int64_t>(slot) >= a.trace_cap) return;
  uint32_t sm;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
  IndexTraceRec r;
  r.kind_sm = static_cast<uint32_t>(kind) | (sm << 8);
  r.chunk = static_cast<uint32_t>(chunk);
  r.t0 = t0;
  r.t1 = t1;
  r.t2 = t2;
  r.t3 = t3;
  a.trace[slot] = r;
#else
  (void)a, (void)kind, (void)chunk, (void)t0, (void)t1, (void)t2;
#endif
}

#ifdef DSA_ITEM_TRACE
#define DSA_STAMP(v) v = globaltimer_ns()
#else
#define DSA_STAMP(v) (void)0
#endif

// Item-trace build: SM-cycle sums of the fold's and the MMA issuer's waits,
// in the kernel words after the fallback count (zero cost otherwise).
enum : int {
  kCycFoldWait = kIndexFallbackRowsWord + 1,  // epilogue thread 0: waiting for a head's accumulator
  kCycFold,                                   // ... folding tiles and samples, waits included
  kCycMmaA,                                   // MMA issuer: waiting for a head's query tile
  kCycMmaAcc,                                 // ... for a free accumulator
  kCycMmaB,                                   // ... for a pooled-key tile
  kCycMmaHeads,                               // heads issued (a count)
  kCycFoldHeads,                              // heads folded by epilogue thread 0 (a count)
  kCycAppendCmp,                              // epilogue thread 0: a tile's threshold compares
  kCycAppendAtomic,                           // ... its row-count atomic (issue to result)
  kCycAppendWrite,                            // ... its candidate writes
  kCycAppends                                 // tiles appended by epilogue thread 0 (a count)
};
static_assert(kCycAppends < kIndexSyncWords, "trace words");

// (not in the stamps-only trace build, DSA_TRACE_STAMPS_ONLY, whose clock
// reads inside the fold would change the kernel it measures)
struct CycleSum {
#if defined(DSA_ITEM_TRACE) && !defined(DSA_TRACE_STAMPS_ONLY)
  long long sum = 0, t = 0;
  __device__ __forceinline__ void start() { t = clock64(); }
  __device__ __forceinline__ void stop() { sum += clock64() - t; }
  __device__ __forceinline__ void add(long long n) { sum += n; }
#else
  __device__ __forceinline__ void start() {}
  __device__ __forceinline__ void stop() {}
  __device__ __forceinline__ void add(long long) {}
#endif
};

__device__ __forceinline__ void cycles_publish(const Args& a, int word, const CycleSum& c) {
#if defined(DSA_ITEM_TRACE) && !defined(DSA_TRACE_STAMPS_ONLY)
  if (a.trace != nullptr && c.sum != 0) atomicAdd(a.sync + word, static_cast<unsigned long long>(c.sum));
#else
  (void)a, (void)word, (void)c;
#endif
}

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kEpiBar), "n"(32 * kEpiWarps) : "memory");
}

// Rows of chunks c' <= c that use slot c % nbuf, every such chunk before the
// last of the call being full (thresh and rows items count rows).
__device__ __forceinline__ unsigned long long rows_through(const Args& a, int c) {
  return static_cast<unsigned long long>(c / a.nbuf) * a.chunk + chunk_of(a, c).nrows;
}

// The ticket taker's view of the sequence: step s holds the sample items of
// chunk s, the thresh items of chunk s-1-lead, the tiles of chunk s-2-lead
// and the row items of chunk s-2-lead-lag.
struct Cursor {
  int s;
  int64_t base;        // first ticket of step s
  int ns, nh, nt, nr;  // sample, thresh, tile and row items in step s
};

__device__ __forceinline__ int steps(const Args& a) { return a.nchunks + 2 + a.lead + a.lag; }

__device__ __forceinline__ void cursor_load(const Args& a, Cursor& cur) {
  const int cs = cur.s, ch_ = cur.s - 1 - a.lead, ct = ch_ - 1, cr = ct - a.lag;
  cur.ns = cs < a.nchunks ? sample_tiles(a, chunk_of(a, cs)) : 0;
  cur.nh = ch_ >= 0 && ch_ < a.nchunks ? (chunk_of(a, ch_).nrows + a.rpi - 1) / a.rpi : 0;
  cur.nt = ct >= 0 && ct < a.nchunks ? chunk_of(a, ct).ntiles : 0;
  cur.nr = cr >= 0 && cr < a.nchunks ? (chunk_of(a, cr).nrows + a.rpi - 1) / a.rpi : 0;
}

__device__ __forceinline__ int cursor_items(const Cursor& cur) { return cur.ns + cur.nh + cur.nt + cur.nr; }

__global__ void __launch_bounds__(kThreads, 1)
    index_topk_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                      const __grid_constant__ CUtensorMap s_map, const Args a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-B swizzle atoms need 1024-B alignment
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sB = base;
  const uint32_t sA = base + kBBytes;
  const uint32_t sCtl = base + kCtlOff;
  uint8_t* gctl = gbase + kCtlOff;
  const uint32_t bar_a_full = sCtl + kBarAFull, bar_a_empty = sCtl + kBarAEmpty;
  const uint32_t bar_b_full = sCtl + kBarBFull, bar_b_empty = sCtl + kBarBEmpty;
  const uint32_t bar_acc_full = sCtl + kBarAccFull, bar_acc_empty = sCtl + kBarAccEmpty;
  const uint32_t bar_drain = sCtl + kBarDrain;
  const uint32_t bar_item_full = sCtl + kBarItemFull, bar_item_empty = sCtl + kBarItemEmpty;
  const uint32_t bar_deps = sCtl + kBarDeps, bar_done = sCtl + kBarDone;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gctl + kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gctl + kAbort);
  volatile int* group_ok = reinterpret_cast<volatile int*>(gctl + kGroupOk);
  volatile int* wait_ok = reinterpret_cast<volatile int*>(gctl + kWaitOk);
  volatile Item* items = reinterpret_cast<volatile Item*>(gctl + kItemData);
  uint2* thr_s = reinterpret_cast<uint2*>(gbase + kThrOff);  // [kItems][kBM] thresholds of a tile's rows
  cand::Smem* csm = reinterpret_cast<cand::Smem*>(gbase + kGrpOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(bar_a_full + 8 * s, 1);
      mbar_init(bar_a_empty + 8 * s, 1);
    }
    mbar_init(bar_b_full, 1);
    mbar_init(bar_b_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_acc_full + 8 * s, 1);
      mbar_init(bar_acc_empty + 8 * s, kEpiWarps);
    }
    for (int s = 0; s < kItems; ++s) {
      mbar_init(bar_item_full + 8 * s, 1);   // the scheduler wrote the item
      mbar_init(bar_item_empty + 8 * s, 3);  // the TMA and MMA threads read it; the publisher published it
      mbar_init(bar_deps + 8 * s, 1);        // the scheduler found its dependencies met
      mbar_init(bar_done + 8 * s, kEpiWarps);  // every epilogue warp finished it
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    *group_ok = 1;
    *wait_ok = 1;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int as = 0, is = 0;
      uint32_t aph = 0, bph = 0, iph = 0;
      uint32_t a_armed = 0, a_par = 0;  // bit s: stage armed / parity armed
      bool b_armed = false;
      uint32_t b_par = 0;
      bool ok = true, maps_ready = false;
      while (ok) {
        if (!mbar_wait(bar_item_full + 8 * is, iph, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        const Item it{items[is].kind, items[is].chunk, items[is].a, items[is].b};
        mbar_arrive(bar_item_empty + 8 * is);
        if (++is == kItems) {
          is = 0;
          iph ^= 1;
        }
        if (it.kind == kItemEnd) break;
        if (it.kind != kItemSample && it.kind != kItemTile) continue;
        if (!maps_ready) {
          tma_prefetch_map(&q_map);
          tma_prefetch_map(&k_map);
          tma_prefetch_map(&s_map);
          maps_ready = true;
        }
        if (!mbar_wait(bar_b_empty, bph ^ 1, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        if (!a.inject) {
          // tile: pools pb*256 ..; sample: sampled pools (st*256 + j) * sigma
          const CUtensorMap* bm = it.kind == kItemTile ? &k_map : &s_map;
          mbar_arrive_expect_tx(bar_b_full, kBBytes);
          tma_load_2d(sB, bm, bar_b_full, 0, it.b * kBN);
          tma_load_2d(sB + kBHalf, bm, bar_b_full, kDi, it.b * kBN);
          b_armed = true;
          b_par = bph;
        }
        bph ^= 1;
        const int qrow = static_cast<int>(a.q_begin + static_cast<int64_t>(it.chunk) * a.chunk) + it.a * kBM;
        for (int h = 0; h < a.Hi; ++h) {
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
      if (!ok) raise_abort(a, abort_flag);
      // every copy this thread issued lands before the CTA may exit
      for (int s = 0; s < kAStages; ++s)
        if (a_armed & (1u << s)) mbar_wait(bar_a_full + 8 * s, (a_par >> s) & 1u, a.limit_ns, nullptr);
      if (b_armed) mbar_wait(bar_b_full, b_par, a.limit_ns, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16_f32(kBM, kBN);
      int as = 0, cs = 0, is = 0;
      uint32_t aph = 0, bph = 0, cph = 0, iph = 0;
      bool ok = true, issued = false;
      CycleSum cyc_a, cyc_acc, cyc_b, cyc_heads;
      while (ok) {
        if (!mbar_wait(bar_item_full + 8 * is, iph, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        const int kind = items[is].kind;
        mbar_arrive(bar_item_empty + 8 * is);
        if (++is == kItems) {
          is = 0;
          iph ^= 1;
        }
        if (kind == kItemEnd) break;
        if (kind != kItemTile && kind != kItemSample) continue;
        cyc_b.start();
        if (!mbar_wait(bar_b_full, bph, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        cyc_b.stop();
        tc_fence_after();
        const uint32_t b_hi = sB, b_lo = sB + kBHalf;
        for (int h = 0; h < a.Hi; ++h) {
          cyc_a.start();
          const bool got_a = mbar_wait(bar_a_full + 8 * as, aph, a.limit_ns, abort_flag);
          cyc_a.stop();
          cyc_acc.start();
          if (!got_a || !mbar_wait(bar_acc_empty + 8 * cs, cph ^ 1, a.limit_ns, abort_flag)) {
            ok = false;
            break;
          }
          cyc_acc.stop();
          cyc_heads.add(1);
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
        umma_commit(bar_b_empty);
        bph ^= 1;
      }
      if (!ok) raise_abort(a, abort_flag);
      cycles_publish(a, kCycMmaA, cyc_a);
      cycles_publish(a, kCycMmaAcc, cyc_acc);
      cycles_publish(a, kCycMmaB, cyc_b);
      cycles_publish(a, kCycMmaHeads, cyc_heads);
      if (issued) {  // all MMAs done before TMEM and shared memory are released
        umma_commit(bar_drain);
        mbar_wait(bar_drain, 0, a.limit_ns, nullptr);
      }
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // -------------------------------------------------------------- scheduler: tickets and dependencies
      // Takes the next ticket once the ring has a free slot (a CTA never
      // holds work it cannot start soon, so tickets are served close to their
      // order), then waits until the item's dependencies -- earlier tickets,
      // published by other CTAs -- are met, and for a tile brings the
      // thresholds of its 128 rows into shared memory.  The epilogue then
      // waits only on shared-memory barriers.
      int is = 0;
      uint32_t iph = 0;
      bool ok = true;
      Cursor cur{0, 0, 0, 0, 0, 0};
      cursor_load(a, cur);
      const int nsteps = steps(a);
      unsigned long long tiles_cum[kMaxBufs], samp_cum[kMaxBufs];
#pragma unroll
      for (int q = 0; q < kMaxBufs; ++q) tiles_cum[q] = samp_cum[q] = 0ull;
      int tiles_upto = -1, samp_upto = -1;
      while (ok) {
        if (!mbar_wait(bar_item_empty + 8 * is, iph ^ 1, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        Item it{kItemEnd, 0, 0, 0};
        while (true) {
          const int64_t t = static_cast<int64_t>(atomicAdd(a.sync + kTicket, 1ull));
          while (t >= cur.base + cursor_items(cur) && cur.s < nsteps) {
            cur.base += cursor_items(cur);
            ++cur.s;
            cursor_load(a, cur);
          }
          if (cur.s >= nsteps) break;  // no work left: the end item
          int off = static_cast<int>(t - cur.base);
          if (off < cur.ns) {
            const Chunk ch = chunk_of(a, cur.s);
            int qb = 0;
            while (qb + 1 < ch.nqb) {
              const int n = sample_tiles_of(a, ch, qb);
              if (off < n) break;
              off -= n;
              ++qb;
            }
            it = Item{kItemSample, cur.s, qb, off};
            break;
          }
          off -= cur.ns;
          if (off < cur.nh) {
            const Chunk ch = chunk_of(a, cur.s - 1 - a.lead);
            const int r0 = off * a.rpi;
            it = Item{kItemThresh, cur.s - 1 - a.lead, r0, min(a.rpi, ch.nrows - r0)};
            break;
          }
          off -= cur.nh;
          if (off < cur.nt) {
            const Chunk ch = chunk_of(a, cur.s - 2 - a.lead);
            const int qb = off % ch.nqb, pb = off / ch.nqb;
            if (pb >= pool_tiles_of(ch, qb)) continue;  // past the causal edge: nothing to compute
            it = Item{kItemTile, cur.s - 2 - a.lead, qb, pb};
            break;
          }
          off -= cur.nt;
          const Chunk ch = chunk_of(a, cur.s - 2 - a.lead - a.lag);
          const int r0 = off * a.rpi;
          it = Item{kItemRows, cur.s - 2 - a.lead - a.lag, r0, min(a.rpi, ch.nrows - r0)};
          break;
        }
        items[is].kind = it.kind;
        items[is].chunk = it.chunk;
        items[is].a = it.a;
        items[is].b = it.b;
        mbar_arrive(bar_item_full + 8 * is);  // release: the item's fields are visible to the waiters
        if (it.kind != kItemEnd) {
          const int bi = it.chunk % a.nbuf;
          const Chunk ch = chunk_of(a, it.chunk);
          bool go = true;
          if (it.kind == kItemSample) {
            // the thresh items of chunks c-nbuf, ... are done reading the slot's samples
            if (it.chunk >= a.nbuf) go = wait_counter(a, a.sync + kThrDone + bi, rows_through(a, it.chunk - a.nbuf));
          } else if (it.kind == kItemThresh) {
            if (ch.row0 + it.a + it.b - 1 > 4ll * a.cap + 3) {  // some row has more than cap pools: its samples
              while (samp_upto < it.chunk) {
                const int c = ++samp_upto;
                samp_cum[c % a.nbuf] += static_cast<unsigned long long>(sample_tiles(a, chunk_of(a, c)));
              }
              go = wait_counter(a, a.sync + kSampDone + bi, samp_cum[bi]);
            }
            // the rows of chunks c-nbuf, ... are done with the slot's candidates
            if (go && it.chunk >= a.nbuf) go = wait_counter(a, a.sync + kRowsDone + bi, rows_through(a, it.chunk - a.nbuf));
          } else if (it.kind == kItemTile) {
            // the thresholds of chunk c are set (and its candidate counts zeroed)
            go = wait_counter(a, a.sync + kThrDone + bi, rows_through(a, it.chunk));
            if (go) {
              // thresholds of the tile's 128 rows (rows past the chunk read padding)
              const uint2* src = a.thr + static_cast<int64_t>(bi) * a.thr_ld + static_cast<int64_t>(it.a) * kBM;
              const uint32_t dst = smem_u32(thr_s + is * kBM);
#pragma unroll 8
              for (int j = 0; j < kBM / 2; ++j) cp_async16(dst + 16 * j, src + 2 * j, true);
              cp_async_commit();
              cp_async_wait<0>();
            }
          } else if (ch.row0 + it.a + it.b - 1 > 4ll * a.topk + 3) {
            // rows: some row reads candidates, so its chunk's tiles must be appended
            while (tiles_upto < it.chunk) {
              const int c = ++tiles_upto;
              tiles_cum[c % a.nbuf] += valid_tiles(chunk_of(a, c));
            }
            go = wait_counter(a, a.sync + kTilesDone + bi, tiles_cum[bi]);
          }
          if (!go) {
            ok = false;
            raise_abort(a, abort_flag);
          }
        }
        mbar_arrive(bar_deps + 8 * is);  // release: the thresholds are visible to the epilogue
        if (++is == kItems) {
          is = 0;
          iph ^= 1;
        }
        if (it.kind == kItemEnd) break;
      }
      if (!ok) raise_abort(a, abort_flag);
    } else if (lane == 1) {
      // -------------------------------------------------------------- publisher
      // Once every epilogue warp has finished an item (their arrivals order
      // its writes before this thread's fence, whose effect is cumulative),
      // adds it to the chunk slot's done counter and frees its ring slot.
      int is = 0;
      uint32_t iph = 0;
      bool ok = true;
      while (ok) {
        if (!mbar_wait(bar_item_full + 8 * is, iph, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        const Item it{items[is].kind, items[is].chunk, items[is].a, items[is].b};
        if (it.kind == kItemEnd) break;
        if (!mbar_wait(bar_done + 8 * is, iph, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        __threadfence();
        const int bi = it.chunk % a.nbuf;
        if (it.kind == kItemSample) atomicAdd(a.sync + kSampDone + bi, 1ull);
        else if (it.kind == kItemTile) atomicAdd(a.sync + kTilesDone + bi, 1ull);
        else if (it.kind == kItemThresh) atomicAdd(a.sync + kThrDone + bi, static_cast<unsigned long long>(it.b));
        else atomicAdd(a.sync + kRowsDone + bi, static_cast<unsigned long long>(it.b));
        mbar_arrive(bar_item_empty + 8 * is);
        if (++is == kItems) {
          is = 0;
          iph ^= 1;
        }
      }
      if (!ok) raise_abort(a, abort_flag);
    }
  } else {
    // ---------------------------------------------------------------- epilogue + thresholds + top-k
    // Warp w (3..18) reads TMEM lanes 32*(w%4).. (its hardware lane quarter)
    // and columns 64*((w-3)/4).. of each accumulator: one query row and 64
    // pools per thread.  For thresh and rows items, warps 3+4g .. 6+4g form
    // group g.  Decisions that steer the 512-thread barrier are taken by
    // epilogue thread 0 and read by all from shared memory, so every epilogue
    // thread takes the same branch.
    const int etid = static_cast<int>(threadIdx.x) - 32 * kEpiWarp0;
    const int ew = warp - kEpiWarp0;
    const int lq = warp & 3;
    const int cq = ew >> 2;
    const int gid = ew >> 2;
    int cs = 0, is = 0;
    uint32_t cph = 0, iph = 0;
    CycleSum cyc_fw, cyc_fold, cyc_fheads, cyc_cmp, cyc_atom, cyc_wr, cyc_app;
    while (true) {
      bool ok = mbar_wait(bar_item_full + 8 * is, iph, a.limit_ns, abort_flag);
      Item it{kItemEnd, 0, 0, 0};
      if (ok) {
        it.kind = items[is].kind;
        it.chunk = items[is].chunk;
        it.a = items[is].a;
        it.b = items[is].b;
      }
      if (!ok) raise_abort(a, abort_flag);
      // every warp saw the same item (or an abort): agree before branching
      epi_sync();
      if (etid == 0) *group_ok = !*abort_flag;
      epi_sync();
      if (!*group_ok || it.kind == kItemEnd) break;

      Chunk ch = chunk_of(a, it.chunk);
      int bi = it.chunk % a.nbuf;
      uint64_t ts0 = 0, ts1 = 0, ts2 = 0;
      DSA_STAMP(ts0);
      ts1 = ts0;
      if (it.kind == kItemTile || it.kind == kItemSample) {
        int qb = it.a;
        int64_t row = ch.row0 + static_cast<int64_t>(qb) * kBM + lq * 32 + lane;
        const bool valid = row < ch.row0 + ch.nrows;
        const float* wrow = a.w + (valid ? row : ch.row0) * a.Hi;
        float2 acc[kEpiCols / 2];
#pragma unroll
        for (int j = 0; j < kEpiCols / 2; ++j) acc[j] = make_float2(0.f, 0.f);
        // the head weight is fetched one head ahead so its load latency hides
        // behind the previous head's epilogue
        float w_next = valid ? __ldg(wrow) : 0.f;
        cyc_fold.start();
        for (int h = 0; h < a.Hi; ++h) {
          const float wv = w_next;
          if (h + 1 < a.Hi) w_next = valid ? __ldg(wrow + h + 1) : 0.f;
          cyc_fw.start();
          if (!mbar_wait(bar_acc_full + 8 * cs, cph, a.limit_ns, abort_flag)) {
            ok = false;
            break;
          }
          cyc_fw.stop();
          cyc_fheads.add(1);
          tc_fence_after();
          const float2 w2 = make_float2(wv, wv);
          const uint32_t taddr = tmem + (static_cast<uint32_t>(lq * 32) << 16) + cs * kBN + cq * kEpiCols;
          // 16 columns at a time (64 accumulator registers leave room for no
          // more); the accumulator is released as soon as the last load has
          // landed, before its columns are folded
#pragma unroll
          for (int cc = 0; cc < kEpiCols / 16; ++cc) {
            uint32_t r[16];
            tmem_ld16(taddr + cc * 16, r);
            tmem_ld_wait();
            if (cc == kEpiCols / 16 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_acc_empty + 8 * cs);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float2 x =
                  make_float2(fmaxf(__uint_as_float(r[2 * j]), 0.f), fmaxf(__uint_as_float(r[2 * j + 1]), 0.f));
              acc[cc * 8 + j] = __ffma2_rn(w2, x, acc[cc * 8 + j]);
            }
          }
          if (++cs == 2) {
            cs = 0;
            cph ^= 1;
          }
        }
        cyc_fold.stop();
        // the item, its chunk and this thread's row are read again here
        // rather than held in registers through the fold (the item's ring
        // slot stays as it is until every epilogue warp is done with it)
        it.kind = items[is].kind;
        it.chunk = items[is].chunk;
        it.a = items[is].a;
        it.b = items[is].b;
        ch = chunk_of(a, it.chunk);
        bi = it.chunk % a.nbuf;
        qb = it.a;
        row = ch.row0 + static_cast<int64_t>(qb) * kBM + lq * 32 + lane;
        DSA_STAMP(ts1);
        // the item's dependencies (met long ago, as a rule)
        if (ok) ok = mbar_wait(bar_deps + 8 * is, iph, a.limit_ns, abort_flag);
        if (!ok) raise_abort(a, abort_flag);
        DSA_STAMP(ts2);
        const int64_t rloc = row - ch.row0;
        DSA_CHECK(a.status, !valid || (rloc >= 0 && rloc < a.thr_ld));
        if (!ok) {
          // nothing is written; the publisher times out and the call reports it
        } else if (it.kind == kItemSample) {
          float* stg = reinterpret_cast<float*>(gbase + kGrpOff + ew * kStgBytes);
          float* buf = a.samples + static_cast<int64_t>(bi) * a.samp_slot;
          const int64_t rbase = static_cast<int64_t>(qb) * kBM + lq * 32;  // this warp's first row in the chunk
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            // lane holds row rbase + lane: columns 32*half .. +31 of its 64
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float2 u = acc[16 * half + 2 * j], v = acc[16 * half + 2 * j + 1];
              *reinterpret_cast<float4*>(stg + lane * kStgLd + 4 * j) = make_float4(u.x, u.y, v.x, v.y);
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int r = 4 * k + (lane >> 3), c = 4 * (lane & 7);
              const float4 x = *reinterpret_cast<const float4*>(stg + r * kStgLd + c);
              if (rbase + r < ch.nrows)
                *reinterpret_cast<float4*>(buf + (rbase + r) * a.samp_ld + static_cast<int64_t>(it.b) * kBN +
                                           cq * kEpiCols + 32 * half + c) = x;
            }
            __syncwarp();
          }
        } else {
          // append this row's pools at or above its threshold
          const int64_t n_r = row / 4;
          if (valid && n_r > a.topk) {
            const uint2 th = thr_s[is * kBM + lq * 32 + lane];
            const uint32_t pbase = static_cast<uint32_t>(it.b) * kBN + cq * kEpiCols;
            // pool pbase + j is a candidate when j < jn (eligible) and its
            // score is above the threshold's, or equal with j <= jt; the key
            // order is the float order (-0 and +0 being one key), so the
            // scores are compared as floats
            const float tf = topk::key_score(th.x);
            const int jn = static_cast<int>(min(n_r - static_cast<int64_t>(pbase), static_cast<int64_t>(kEpiCols)));
            const int jt = static_cast<int>(
                min(static_cast<int64_t>(th.y) - static_cast<int64_t>(pbase), static_cast<int64_t>(kEpiCols)));
            // bit j of `hit`: pool pbase + j is a candidate
            cyc_app.add(1);
            cyc_cmp.start();
            unsigned long long hit = 0ull;
            if (jn == kEpiCols && (jt < 0 || jt >= kEpiCols - 1)) {
              // every pool eligible, and the threshold's pool before (jt < 0)
              // or at or after (jt >= 63) all of them: one compare per pool,
              // v >= tf (ties count) or v > tf, the latter as v >= the next
              // float above tf (+0 and -0 compare equal, so above both zeros
              // comes the smallest positive subnormal)
              float tq = tf;
              if (jt < 0) {
                const uint32_t b = __float_as_uint(tf);
                tq = (b & 0x7FFFFFFFu) == 0u ? __uint_as_float(1u)
                                             : __uint_as_float((b & 0x80000000u) ? b - 1u : b + 1u);
              }
              uint32_t lo = 0u, hi = 0u;
#pragma unroll
              for (int j = 0; j < kEpiCols; ++j) {
                const float v = (j & 1) ? acc[j >> 1].y : acc[j >> 1].x;
                if (v >= tq) {
                  if (j < 32) lo |= 1u << j;
                  else hi |= 1u << (j - 32);
                }
              }
              hit = (static_cast<unsigned long long>(hi) << 32) | lo;
            } else {
#pragma unroll
              for (int j = 0; j < kEpiCols; ++j) {
                const float v = (j & 1) ? acc[j >> 1].y : acc[j >> 1].x;
                if (j < jn && (v > tf || (v == tf && j <= jt))) hit |= 1ull << j;
              }
            }
            cyc_cmp.stop();
            if (hit != 0ull) {
              cyc_atom.start();
              unsigned pos = atomicAdd(a.cnt + static_cast<int64_t>(bi) * a.thr_ld + rloc,
                                       static_cast<unsigned>(__popcll(hit)));
#ifdef DSA_ITEM_TRACE
              asm volatile("" ::"r"(pos));  // the timer below waits for the atomic's result
#endif
              cyc_atom.stop();
              cyc_wr.start();
              uint2* dst = a.cands + static_cast<int64_t>(bi) * a.cand_slot + rloc * a.cap;
              const unsigned cap = static_cast<unsigned>(a.cap);
              // each half of the thread's 64 scores goes through the warp's
              // staging tile, so that every lane walks only its own hits
              // (a register array cannot be indexed by a hit's position);
              // the rows of a warp have different hits, and a loop over all
              // 64 positions would issue a store step for each of them
              float* stg = reinterpret_cast<float*>(gbase + kGrpOff + ew * kStgBytes) + lane * kStgLd;
#pragma unroll
              for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const float2 u = acc[16 * half + 2 * q], w = acc[16 * half + 2 * q + 1];
                  *reinterpret_cast<float4*>(stg + 4 * q) = make_float4(u.x, u.y, w.x, w.y);
                }
                // (a lane reads only its own staged row: no warp barrier, and
                // lanes without hits never come here)
                uint32_t h = static_cast<uint32_t>(hit >> (32 * half));
                while (h != 0u) {
                  const int j = __ffs(h) - 1;
                  h &= h - 1u;
                  if (pos < cap) dst[pos] = make_uint2(topk::score_key(stg[j]), pbase + 32 * half + j);
                  ++pos;
                }
              }
              cyc_wr.stop();
            }
          }
        }
      } else {
        // ---- thresh or rows: up to four rows, one per group, once the
        // item's dependencies are met (all warps agree before the groups'
        // barriers)
        bool dep = mbar_wait(bar_deps + 8 * is, iph, a.limit_ns, abort_flag);
        if (!dep) raise_abort(a, abort_flag);
        epi_sync();
        if (etid == 0) *wait_ok = !*abort_flag;
        epi_sync();
        if (!*wait_ok) break;
        DSA_STAMP(ts2);
        const int r0 = it.a, nr = it.b;
        const topk::Group grp{etid - gid * topk::kGT, 2 + gid};
        if (a.rpi == kRowsPerWarpItem) {
          // one row per warp (topk <= 512)
          if (ew < nr) {
            wsel::Smem& wsm = reinterpret_cast<wsel::Smem*>(gbase + kGrpOff)[ew];
            const int64_t rloc = r0 + ew;
            const int64_t i = ch.row0 + rloc;
            const int64_t n = i / 4;
            if (it.kind == kItemThresh) {
              if (n > a.topk) {
                uint2 th = make_uint2(0u, 0x7FFFFFFFu);  // every eligible pool
                if (n > a.cap) {
                  const int G = static_cast<int>((n + a.sigma - 1) / a.sigma);
                  th = wsel::threshold(wsm, lane, a.samples + static_cast<int64_t>(bi) * a.samp_slot + rloc * a.samp_ld,
                                       G, a.rsel, a.sigma);
                }
                if (lane == 0) {
                  a.thr[static_cast<int64_t>(bi) * a.thr_ld + rloc] = th;
                  a.cnt[static_cast<int64_t>(bi) * a.thr_ld + rloc] = 0u;
                }
              }
            } else {
              int32_t* orow = a.pool_idx + (i - a.q_begin) * a.topk;
              if (n <= a.topk) {
                for (int j = lane; j < a.topk; j += 32) orow[j] = j < n ? j : -1;
              } else {
                const unsigned count = __ldcg(a.cnt + static_cast<int64_t>(bi) * a.thr_ld + rloc);
                bool done = false;
                if (count >= static_cast<unsigned>(a.topk) && count <= static_cast<unsigned>(a.cap))
                  done = wsel::topk(wsm, lane, a.cands + static_cast<int64_t>(bi) * a.cand_slot + rloc * a.cap,
                                    static_cast<int>(count), a.topk, orow);
                if (!done && lane == 0) {
                  const unsigned long long f = atomicAdd(a.sync + kIndexFallbackRowsWord, 1ull);
                  a.fb_rows[f] = static_cast<int32_t>(i);
                }
              }
            }
          }
        } else if (gid < nr) {
          // one row per 128-thread group (topk > 512)
          const int64_t rloc = r0 + gid;
          const int64_t i = ch.row0 + rloc;
          const int64_t n = i / 4;
          if (it.kind == kItemThresh) {
            if (n > a.topk) {
              uint2 th = make_uint2(0u, 0x7FFFFFFFu);  // every eligible pool
              if (n > a.cap) {
                const int G = static_cast<int>((n + a.sigma - 1) / a.sigma);
                th = cand::sample_threshold(grp, csm[gid],
                                            a.samples + static_cast<int64_t>(bi) * a.samp_slot + rloc * a.samp_ld, G,
                                            a.rsel, a.sigma);
              }
              if (grp.tid == 0) {
                a.thr[static_cast<int64_t>(bi) * a.thr_ld + rloc] = th;
                a.cnt[static_cast<int64_t>(bi) * a.thr_ld + rloc] = 0u;
              }
            }
          } else {
            int32_t* orow = a.pool_idx + (i - a.q_begin) * a.topk;
            if (n <= a.topk) {
              for (int j = grp.tid; j < a.topk; j += topk::kGT) orow[j] = j < n ? j : -1;
            } else {
              const unsigned count = __ldcg(a.cnt + static_cast<int64_t>(bi) * a.thr_ld + rloc);
              bool done = false;
              if (count >= static_cast<unsigned>(a.topk) && count <= static_cast<unsigned>(a.cap))
                done = cand::select(grp, csm[gid], a.cands + static_cast<int64_t>(bi) * a.cand_slot + rloc * a.cap,
                                    static_cast<int>(count), a.topk, orow);
              if (!done && grp.tid == 0) {
                const unsigned long long f = atomicAdd(a.sync + kIndexFallbackRowsWord, 1ull);
                a.fb_rows[f] = static_cast<int32_t>(i);
              }
            }
          }
        }
      }
      // this warp is done with the item: the publisher counts it once all are
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_done + 8 * is);
      if (etid == 0) trace_item(a, it.kind, it.chunk, ts0, ts1, ts2 == 0 ? ts1 : ts2);
      if (++is == kItems) {
        is = 0;
        iph ^= 1;
      }
    }
    if (etid == 0) {
      cycles_publish(a, kCycFoldWait, cyc_fw);
      cycles_publish(a, kCycFold, cyc_fold);
      cycles_publish(a, kCycFoldHeads, cyc_fheads);
      cycles_publish(a, kCycAppendCmp, cyc_cmp);
      cycles_publish(a, kCycAppendAtomic, cyc_atom);
      cycles_publish(a, kCycAppendWrite, cyc_wr);
      cycles_publish(a, kCycAppends, cyc_app);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Rows the main kernel could not certify (fewer than topk candidates, or
// more than cap): all n = floor(i/4) scores of the row are recomputed on the
// CUDA cores -- fp32 dot products of q_idx with the fp32 pooled keys, ReLU,
// head weight, sum over heads in head order -- into this CTA's scratch row,
// and the row's top-k is taken from them (topk_row.cuh).  CTAs take the
// listed rows in turn.
constexpr int kFbThreads = 256;
constexpr int kMaxHi = 64;

__global__ void __launch_bounds__(kFbThreads)
    index_fallback_kernel(const __nv_bfloat16* __restrict__ q_idx, const float* __restrict__ khat32,
                          const float* __restrict__ w, int Hi, int topk, int64_t q_begin, int32_t* __restrict__ pool_idx,
                          const int32_t* __restrict__ fb_rows, const unsigned long long* __restrict__ sync,
                          float* __restrict__ scratch, int64_t scratch_ld) {
  __shared__ topk::Smem tsm;
  __shared__ float qs[kMaxHi * kDi];
  __shared__ float ws[kMaxHi];
  __shared__ unsigned long long general_rows;
  const unsigned long long nfb = sync[kIndexFallbackRowsWord];
  float* srow = scratch + static_cast<int64_t>(blockIdx.x) * scratch_ld;
  for (unsigned long long f = blockIdx.x; f < nfb; f += gridDim.x) {
    const int64_t i = fb_rows[f];
    const int n = static_cast<int>(i / 4);
    for (int e = threadIdx.x; e < Hi * kDi; e += kFbThreads)
      qs[e] = __bfloat162float(q_idx[i * Hi * kDi + e]);
    for (int h = threadIdx.x; h < Hi; h += kFbThreads) ws[h] = w[i * Hi + h];
    __syncthreads();
    for (int p = threadIdx.x; p < n; p += kFbThreads) {
      float kh[kDi];
      const float4* src = reinterpret_cast<const float4*>(khat32 + static_cast<int64_t>(p) * kDi);
#pragma unroll
      for (int d4 = 0; d4 < kDi / 4; ++d4) {
        const float4 v = src[d4];
        kh[4 * d4] = v.x;
        kh[4 * d4 + 1] = v.y;
        kh[4 * d4 + 2] = v.z;
        kh[4 * d4 + 3] = v.w;
      }
      float acc = 0.f;
      for (int h = 0; h < Hi; ++h) {
        float x = 0.f;
#pragma unroll
        for (int d = 0; d < kDi; ++d) x = fmaf(qs[h * kDi + d], kh[d], x);
        acc = fmaf(ws[h], fmaxf(x, 0.f), acc);
      }
      srow[p] = acc;
    }
    __syncthreads();
    if (threadIdx.x < topk::kGT) {
      const topk::Group grp{static_cast<int>(threadIdx.x), 1};
      topk::row(grp, tsm, srow, n, topk, pool_idx + (i - q_begin) * topk, &general_rows);
    }
    __syncthreads();
  }
}

// Khat in fp32 with the fixed summation order, stored as fp32 and split into
// bf16 hi + lo.  One thread per (pool, 8-dim group); Di = 64.  The first
// threads also zero index_topk_kernel's global words.
__global__ void pool_keys_kernel(const __nv_bfloat16* __restrict__ k_idx, int64_t P,
                                 __nv_bfloat16* __restrict__ khat2, float* __restrict__ khat32,
                                 unsigned long long* sync_words) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t < kIndexSyncWords) sync_words[t] = 0ull;
  const int64_t p = t >> 3;
  const int g = static_cast<int>(t & 7);
  if (p >= P) return;
  const uint4* src = reinterpret_cast<const uint4*>(k_idx + 4 * p * kDi) + g;
  uint4 rows[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) rows[r] = src[r * (kDi / 8)];
  uint32_t hi[4], lo[4];
  float kf[8];
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
    kf[2 * e] = kh[0];
    kf[2 * e + 1] = kh[1];
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(kh[0], kh[1]);
    const float2 hf = __bfloat1622float2(h2);
    const __nv_bfloat162 l2 = __floats2bfloat162_rn(__fsub_rn(kh[0], hf.x), __fsub_rn(kh[1], hf.y));
    hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
    lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
  }
  uint4* dst = reinterpret_cast<uint4*>(khat2 + p * (2 * kDi));
  dst[g] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  dst[8 + g] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  float4* d32 = reinterpret_cast<float4*>(khat32 + p * kDi + 8 * g);
  d32[0] = make_float4(kf[0], kf[1], kf[2], kf[3]);
  d32[1] = make_float4(kf[4], kf[5], kf[6], kf[7]);
}

// A short sequence's rows all keep every eligible pool (see launch_short_rows).
__global__ void __launch_bounds__(256) short_rows_kernel(int32_t* __restrict__ pool_idx, int topk,
                                                         const __grid_constant__ ShortSeqs seqs) {
  const int64_t start = seqs.start[blockIdx.x], len = seqs.len[blockIdx.x];
  int32_t* out = pool_idx + start * topk;
  const int64_t total = len * topk;
  for (int64_t e = threadIdx.x; e < total; e += blockDim.x) {
    const int64_t i = e / topk;
    const int j = static_cast<int>(e - i * topk);
    out[e] = j < (i >> 2) ? j : -1;
  }
}

}  // namespace

size_t index_topk_smem_bytes() { return kSmemBytes; }

cudaError_t launch_short_rows(int32_t* pool_idx, int topk, const ShortSeqs& seqs, const LaunchCtx& ctx) {
  if (seqs.n < 1) return cudaSuccess;
  short_rows_kernel<<<static_cast<unsigned>(seqs.n), 256, 0, ctx.stream>>>(pool_idx, topk, seqs);
  return cudaGetLastError();
}

cudaError_t launch_pool_keys(const void* k_idx, int64_t P, void* khat2, float* khat32, unsigned long long* sync_words,
                             const LaunchCtx& ctx) {
  const int64_t threads = P * 8 > kIndexSyncWords ? P * 8 : kIndexSyncWords;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  pool_keys_kernel<<<static_cast<unsigned>(grid), block, 0, ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(k_idx), P, static_cast<__nv_bfloat16*>(khat2), khat32, sync_words);
  return cudaGetLastError();
}

cudaError_t launch_index_topk(const CUtensorMap& q_map, const CUtensorMap& khat_map, const CUtensorMap& samp_map,
                              const IndexPlan& pl, const IndexBuffers& b, const float* w, int64_t q_begin,
                              int64_t q_end, int chunk, int Hi, int topk, int32_t* pool_idx, const LaunchCtx& ctx) {
  Args a;
  a.w = w;
  a.samples = b.samples;
  a.samp_ld = pl.samp_ld;
  a.samp_slot = pl.samp_slot;
  a.cands = b.cands;
  a.cand_slot = pl.cand_slot;
  a.thr = b.thr;
  a.cnt = b.cnt;
  a.thr_ld = pl.thr_ld;
  a.cap = pl.cap;
  a.sigma = pl.sigma;
  a.rsel = pl.rsel;
  a.rpi = topk <= wsel::kMaxK ? kRowsPerWarpItem : kRowsPerGroupItem;
  a.nbuf = b.nbuf;
  // lead = lag = (nbuf-1)/2 (at most kMaxLead) leaves each of the four
  // distances between an item and what it waits for at least one step
  const int half = (b.nbuf - 1) / 2;
  a.lead = half < kMaxLead ? half : kMaxLead;
  a.lag = a.lead;
  a.q_begin = q_begin;
  a.q_end = q_end;
  a.chunk = chunk;
  a.nchunks = static_cast<int>((q_end - q_begin + chunk - 1) / chunk);
  a.Hi = Hi;
  a.topk = topk;
  a.pool_idx = pool_idx;
  a.fb_rows = b.fb_rows;
  a.trace = b.trace;
  a.trace_count = b.trace_count;
  a.trace_cap = b.trace_cap;
  a.sync = b.sync;
  a.status = ctx.status;
  a.limit_ns = ctx.wait_limit_ns;
  a.inject = ctx.inject_timeout;
  static std::atomic<bool> attr_done[kAttrDevices];
  {
    const cudaError_t e = set_smem_limit_once(index_topk_kernel, static_cast<int>(kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
  }
  // One CTA per SM, launched cooperatively so that all are resident at once.
  // The items' waits do not depend on that: an item waits only for items of
  // earlier tickets, and a CTA takes a ticket only while it runs, so the
  // earliest unfinished item can always proceed.  A smaller grid
  // (ctx.persistent_ctas) is therefore launched as a plain launch, which lets
  // several short calls share the GPU from different streams.
  const bool part = ctx.persistent_ctas > 0 && ctx.persistent_ctas < ctx.num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(part ? ctx.persistent_ctas : ctx.num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = part ? 0 : 1;
  return cudaLaunchKernelEx(&cfg, index_topk_kernel, q_map, khat_map, samp_map, a);
}

cudaError_t launch_index_fallback(const void* q_idx, const IndexPlan& pl, const IndexBuffers& b, const float* w,
                                  int64_t q_begin, int Hi, int topk, int32_t* pool_idx, const LaunchCtx& ctx) {
  index_fallback_kernel<<<pl.fb_ctas, kFbThreads, 0, ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(q_idx), b.khat32, w, Hi, topk, q_begin, pool_idx, b.fb_rows, b.sync,
      b.fb_scratch, pl.fb_ld);
  return cudaGetLastError();
}

}  // namespace dsa
