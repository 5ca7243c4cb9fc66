// index_topk.cu -- pooled indexer keys, and the causal pooled indexer with
// its per-query top-k as one persistent kernel.
//
// [SkyRL-1M §模型与瓶颈] the indexer scores every query against every earlier
// 4-token key pool; [§1 DSA 真稀疏; Anyscale, second lesson (the indexer)] it
// does so one query chunk at a time so the score matrix is never whole, and
// keeps each query's best pools as int32 indices.
//
//   Khat_p     = ((k[4p] + k[4p+1]) + (k[4p+2] + k[4p+3])) * 0.25    (fp32)
//   score(i,p) = sum_h w[i,h] * ReLU(q_idx[i,h,:] . Khat_p)
//
// Work items.  A chunk's indexer work is its (128-query x 256-pool) tiles; its
// top-k work is its query rows, four to an item.  Items are handed out in the
// order
//     tiles(0), tiles(1), tiles(2), tiles(3), rows(0), tiles(4), rows(1), ...
// (a chunk's rows `lag` chunks after its tiles, so that its tiles are done;
// lag = 3 here, less when there are fewer than four score buffers)
// from one global ticket counter to one CTA per SM (cooperative launch, so
// every CTA is resident).  A CTA processes its items in ticket order:
//   tile    TMA brings the 64 KB Khat hi/lo tile and, per head h, the q_idx
//           tile of head h; one 128x256x128 bf16 tcgen05 MMA chain per head
//           accumulates q_h . [Khat_hi ; Khat_lo] in TMEM (Khat kept as a bf16
//           hi/lo pair, so the product keeps ~16 more mantissa bits than one
//           bf16 rounding); 16 epilogue warps fold ReLU, the head weight and
//           the sum over heads into registers while the next head's MMA fills
//           the other TMEM buffer; the tile's scores go to the chunk's score
//           buffer (a ring of up to eight chunk buffers);
//   rows    the same 16 warps split into four groups of four; each group
//           selects one row's top-k (topk_row.cuh), once every tile of its
//           chunk has been stored.  Handing out a row item brings the scores
//           of the row item two tickets later into L2.
// Dependencies run only from later tickets to earlier ones -- rows wait for
// their chunk's tiles, and a tile of chunk c waits, before it stores, for the
// rows of chunk c-nbuf that read the same buffer -- so the lowest unfinished
// ticket can always proceed (rows of chunk c-nbuf are handed out in step
// c-nbuf+lag < c).  With two buffers, tiles waited on rows handed out just
// before them (84 us per tile on average at S = 131072); more buffers put
// chunks of work between a buffer's readers and its next writers.
// There is no barrier per chunk: a CTA that has finished its part of one
// chunk takes the next chunk's work, so SMs do not idle on a chunk whose tile
// count is not a multiple of the SM count, and the chunk size only bounds the
// score scratch.
#include "dsa_device.cuh"
#include "dsa_kernels.h"
#include "topk_row.cuh"

namespace dsa {
namespace {

constexpr int kBM = 128;           // queries per tile (TMEM lanes)
constexpr int kBN = 256;           // pools per tile (TMEM columns per buffer)
constexpr int kDi = 64;            // indexer head dim
constexpr int kAStages = 4;
constexpr int kItems = 2;          // work-item ring between the roles (the item in work + one prefetched)
constexpr int kRowsPerItem = 4;    // one per top-k group
constexpr int kPrefetchItems = 2;  // row items whose scores are brought into L2 ahead of their turn
constexpr int kMaxRowLag = 3;      // a chunk's rows are handed out after the tiles of the chunk this far ahead
constexpr uint32_t kABytes = kBM * kDi * 2;        // 16 KB: q_idx tile of one head
constexpr uint32_t kBHalf = kBN * kDi * 2;         // 32 KB: Khat hi (or lo) tile
constexpr uint32_t kBBytes = 2 * kBHalf;           // 64 KB, one stage
constexpr int kEpiWarps = 16;                      // 4 TMEM lane quarters x 4 column quarters
constexpr int kEpiCols = kBN / 4;                  // 64 columns per epilogue thread
constexpr int kThreads = 32 * (2 + kEpiWarps);     // TMA warp, MMA warp, 16 epilogue warps
constexpr uint32_t kTmemCols = 512;                // 2 accumulators x 256 columns
constexpr uint32_t kCtlOff = kBBytes + kAStages * kABytes;
constexpr uint32_t kCtlBytes = 512;
constexpr uint32_t kTopkOff = kCtlOff + kCtlBytes;
constexpr size_t kSmemBytes = 1024 + kTopkOff + kRowsPerItem * sizeof(topk::Smem);
static_assert(kRowsPerItem * topk::kGT == 32 * kEpiWarps, "the epilogue warps form the top-k groups");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(sizeof(topk::Smem) % 16 == 0, "top-k group buffers stay 16-byte aligned");

constexpr int kEpiBar = 1;   // named barrier of the 512 epilogue threads; the groups use 2..5
// Tile stores go through a per-warp staging tile (32 rows x 32 columns, rows
// padded to 36 floats) in the top-k buffers, which tiles do not otherwise use,
// so that each warp store covers four rows x 128 contiguous bytes.
constexpr int kStgLd = 36;
constexpr uint32_t kStgBytes = 32 * kStgLd * 4;
static_assert(kEpiWarps * kStgBytes <= kRowsPerItem * sizeof(topk::Smem), "staging fits the top-k buffers");

// control block offsets (bytes from kCtlOff)
constexpr uint32_t kBarAFull = 0, kBarAEmpty = 32, kBarBFull = 64, kBarBEmpty = 72, kBarAccFull = 80,
                   kBarAccEmpty = 96, kBarDrain = 112, kBarItemFull = 120, kBarItemEmpty = 152;
constexpr uint32_t kTmemSlot = 184, kAbort = 188, kGroupOk = 192, kWaitOk = 196, kItemData = 256;  // 4 x 16 B

enum : int { kItemTile = 0, kItemRows = 1, kItemEnd = 2 };
struct Item {
  int kind;
  int chunk;
  int a;  // tile: qb   rows: first row within the chunk
  int b;  // tile: pb   rows: number of rows (1..4)
};

// global 64-bit words, zeroed by pool_keys_kernel before each launch; the
// done counters are per buffer (chunk c uses buffer c % nbuf) and cumulative
enum : int { kTicket = 0, kTilesDone = 1 /* kMaxBufs words */, kRowsDone = 1 + kMaxBufs, kGAbort = 1 + 2 * kMaxBufs };
static_assert(kGAbort < kIndexSyncWords && kIndexGeneralRowsWord > kGAbort, "global words");

struct Args {
  const float* w;
  float* scores;        // nbuf buffers of `chunk` rows x ld floats
  int64_t ld;
  int64_t buf_stride;   // floats between consecutive buffers
  int nbuf;             // 1 .. kMaxBufs
  int lag;              // min(kMaxRowLag, nbuf - 1): rows of chunk c come in step c + lag
  int64_t q_begin, q_end;
  int chunk;
  int nchunks;
  int Hi;
  int topk;
  int32_t* pool_idx;
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

__device__ __forceinline__ int pool_tiles_of(const Chunk& ch, int qb) {
  const int64_t end = min(ch.row0 + static_cast<int64_t>(qb + 1) * kBM, ch.row0 + ch.nrows);
  const int64_t n = (end - 1) / 4;  // pools eligible for the last query of the block
  return static_cast<int>((n + kBN - 1) / kBN);
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

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kEpiBar), "n"(32 * kEpiWarps) : "memory");
}

// The ticket taker's view of the sequence: step s holds the tiles of chunk s
// (s < nchunks) followed by the row items of chunk s - lag.
struct Cursor {
  int s;
  int64_t base;  // first ticket of step s
  int nt, nr;    // tile and row items in step s
};

__device__ __forceinline__ void cursor_load(const Args& a, Cursor& cur) {
  cur.nt = cur.s < a.nchunks ? chunk_of(a, cur.s).ntiles : 0;
  const int rc = cur.s - a.lag;
  cur.nr = rc >= 0 && rc < a.nchunks ? (chunk_of(a, rc).nrows + kRowsPerItem - 1) / kRowsPerItem : 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    index_topk_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                      const Args a) {
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
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gctl + kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gctl + kAbort);
  volatile int* group_ok = reinterpret_cast<volatile int*>(gctl + kGroupOk);
  volatile int* wait_ok = reinterpret_cast<volatile int*>(gctl + kWaitOk);
  volatile Item* items = reinterpret_cast<volatile Item*>(gctl + kItemData);
  topk::Smem* tsm = reinterpret_cast<topk::Smem*>(gbase + kTopkOff);

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
      mbar_init(bar_item_full + 8 * s, 1);
      mbar_init(bar_item_empty + 8 * s, 1 + kEpiWarps);  // the MMA thread and one lane per epilogue warp
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
    // ---------------------------------------------------------------- ticket taker + TMA producer
    if (lane == 0) {
      int as = 0, is = 0;
      uint32_t aph = 0, bph = 0, iph = 0;
      uint32_t a_armed = 0, a_par = 0;  // bit s: stage armed / parity armed
      bool b_armed = false;
      uint32_t b_par = 0;
      bool ok = true, maps_ready = false;
      Cursor cur{0, 0, 0, 0};
      cursor_load(a, cur);
      while (ok) {
        // A ticket is taken only once the ring has room for its item: a CTA
        // never holds work it cannot start soon, so tickets are served close
        // to their order and the items that wait on earlier ones find them done.
        if (!mbar_wait(bar_item_empty + 8 * is, iph ^ 1, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        Item it{kItemEnd, 0, 0, 0};
        while (true) {
          const int64_t t = static_cast<int64_t>(atomicAdd(a.sync + kTicket, 1ull));
          while (t >= cur.base + cur.nt + cur.nr && cur.s < a.nchunks + a.lag) {
            cur.base += cur.nt + cur.nr;
            ++cur.s;
            cursor_load(a, cur);
          }
          if (cur.s >= a.nchunks + a.lag) break;  // no work left: the end item
          if (t - cur.base < cur.nt) {
            const Chunk ch = chunk_of(a, cur.s);
            const int tt = static_cast<int>(t - cur.base);
            const int qb = tt % ch.nqb, pb = tt / ch.nqb;
            if (pb >= pool_tiles_of(ch, qb)) continue;  // past the causal edge: nothing to compute
            it = Item{kItemTile, cur.s, qb, pb};
          } else {
            const Chunk ch = chunk_of(a, cur.s - a.lag);
            const int r0 = static_cast<int>(t - cur.base - cur.nt) * kRowsPerItem;
            it = Item{kItemRows, cur.s - a.lag, r0, min(kRowsPerItem, ch.nrows - r0)};
          }
          break;
        }
        items[is].kind = it.kind;
        items[is].chunk = it.chunk;
        items[is].a = it.a;
        items[is].b = it.b;
        mbar_arrive(bar_item_full + 8 * is);  // release: the item's fields are visible to the waiters
        if (++is == kItems) {
          is = 0;
          iph ^= 1;
        }
        if (it.kind == kItemEnd) break;
        if (it.kind == kItemRows) {
          // The rows' scores may have left L2 (the ring is larger than L2):
          // bring back those of the chunk's row item kPrefetchItems tickets
          // ahead, whichever CTA will take it (the first items of a chunk
          // also fetch their own rows).  (Their tiles may not all be stored
          // yet; L2 keeps them coherent.)
          const Chunk ch = chunk_of(a, it.chunk);
          const float* buf = a.scores + static_cast<int64_t>(it.chunk % a.nbuf) * a.buf_stride;
          const int ahead = kPrefetchItems * kRowsPerItem;
          const int f0 = it.a < ahead ? it.a : it.a + ahead;
          const int f1 = min(ch.nrows, it.a + ahead + kRowsPerItem);
          for (int r = f0; r < f1; ++r) {
            const int64_t n = (ch.row0 + r) / 4;
            if (n > a.topk) bulk_prefetch_l2(buf + static_cast<int64_t>(r) * a.ld, static_cast<uint32_t>((n * 4 + 15) & ~15ll));
          }
          continue;
        }
        if (!maps_ready) {
          tma_prefetch_map(&q_map);
          tma_prefetch_map(&k_map);
          maps_ready = true;
        }
        if (!mbar_wait(bar_b_empty, bph ^ 1, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        if (!a.inject) {
          mbar_arrive_expect_tx(bar_b_full, kBBytes);
          tma_load_2d(sB, &k_map, bar_b_full, 0, it.b * kBN);
          tma_load_2d(sB + kBHalf, &k_map, bar_b_full, kDi, it.b * kBN);
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
        if (kind != kItemTile) continue;
        if (!mbar_wait(bar_b_full, bph, a.limit_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t b_hi = sB, b_lo = sB + kBHalf;
        for (int h = 0; h < a.Hi; ++h) {
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
        umma_commit(bar_b_empty);
        bph ^= 1;
      }
      if (!ok) raise_abort(a, abort_flag);
      if (issued) {  // all MMAs done before TMEM and shared memory are released
        umma_commit(bar_drain);
        mbar_wait(bar_drain, 0, a.limit_ns, nullptr);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue + top-k
    // Warp w (2..17) reads TMEM lanes 32*(w%4).. (its hardware lane quarter)
    // and columns 64*((w-2)/4).. of each accumulator: one query row and 64
    // pools per thread.  For row items, warps 2+4g .. 5+4g form top-k group g.
    // Decisions that steer the 512-thread barrier are taken by epilogue
    // thread 0 and read by all from shared memory, so every epilogue thread
    // takes the same branch; the two decision words alternate so that a
    // write never overtakes a reader of the previous value.
    const int etid = static_cast<int>(threadIdx.x) - 64;
    const int ew = warp - 2;
    const int lq = warp & 3;
    const int cq = ew >> 2;
    const int gid = ew >> 2;
    const topk::Group grp{etid - gid * topk::kGT, 2 + gid};
    int cs = 0, is = 0;
    uint32_t cph = 0, iph = 0;
    // cumulative valid-tile counts of chunks 0..tc_upto by buffer (epilogue thread 0 only)
    unsigned long long tiles_cum[kMaxBufs];
#pragma unroll
    for (int q = 0; q < kMaxBufs; ++q) tiles_cum[q] = 0ull;
    int tc_upto = -1;
    while (true) {
      bool ok = mbar_wait(bar_item_full + 8 * is, iph, a.limit_ns, abort_flag);
      Item it{kItemEnd, 0, 0, 0};
      if (ok) {
        it.kind = items[is].kind;
        it.chunk = items[is].chunk;
        it.a = items[is].a;
        it.b = items[is].b;
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(bar_item_empty + 8 * is);
      if (++is == kItems) {
        is = 0;
        iph ^= 1;
      }
      if (!ok) raise_abort(a, abort_flag);
      // every warp saw the same item (or an abort): agree before branching
      epi_sync();
      if (etid == 0) *group_ok = !*abort_flag;
      epi_sync();
      if (!*group_ok || it.kind == kItemEnd) break;

      const Chunk ch = chunk_of(a, it.chunk);
      const int bi = it.chunk % a.nbuf;
      float* buf = a.scores + static_cast<int64_t>(bi) * a.buf_stride;
      if (it.kind == kItemTile) {
        const int qb = it.a, pb = it.b;
        const int64_t row = ch.row0 + static_cast<int64_t>(qb) * kBM + lq * 32 + lane;
        const bool valid = row < ch.row0 + ch.nrows;
        const float* wrow = a.w + (valid ? row : ch.row0) * a.Hi;
        float2 acc[kEpiCols / 2];
#pragma unroll
        for (int j = 0; j < kEpiCols / 2; ++j) acc[j] = make_float2(0.f, 0.f);
        // the head weight is fetched one head ahead so its load latency hides
        // behind the previous head's epilogue
        float w_next = valid ? __ldg(wrow) : 0.f;
        for (int h = 0; h < a.Hi; ++h) {
          const float wv = w_next;
          if (h + 1 < a.Hi) w_next = valid ? __ldg(wrow + h + 1) : 0.f;
          if (!mbar_wait(bar_acc_full + 8 * cs, cph, a.limit_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float2 w2 = make_float2(wv, wv);
          const uint32_t taddr = tmem + (static_cast<uint32_t>(lq * 32) << 16) + cs * kBN + cq * kEpiCols;
#pragma unroll
          for (int cc = 0; cc < kEpiCols / 16; ++cc) {
            uint32_t r[16];
            tmem_ld16(taddr + cc * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float2 x =
                  make_float2(fmaxf(__uint_as_float(r[2 * j]), 0.f), fmaxf(__uint_as_float(r[2 * j + 1]), 0.f));
              acc[cc * 8 + j] = __ffma2_rn(w2, x, acc[cc * 8 + j]);
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
        if (!ok) raise_abort(a, abort_flag);
        epi_sync();
        if (etid == 0) {
          // the rows of chunks c-nbuf, c-2*nbuf, ... (same buffer) must be done reading it
          bool go = !*abort_flag;
          if (go && it.chunk >= a.nbuf)
            go = wait_counter(a, a.sync + kRowsDone + bi,
                              static_cast<unsigned long long>(it.chunk / a.nbuf) * a.chunk);
          if (!go) raise_abort(a, abort_flag);
          *wait_ok = go;
        }
        epi_sync();
        if (!*wait_ok) break;
        {
          float* stg = reinterpret_cast<float*>(gbase + kTopkOff + ew * kStgBytes);
          const int64_t rbase = ch.row0 + static_cast<int64_t>(qb) * kBM + lq * 32;  // this warp's first row
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
              if (rbase + r < ch.row0 + ch.nrows)
                *reinterpret_cast<float4*>(buf + (rbase + r - ch.row0) * a.ld + static_cast<int64_t>(pb) * kBN +
                                           cq * kEpiCols + 32 * half + c) = x;
            }
            __syncwarp();
          }
        }
        // publish: the barrier orders every thread's stores before thread 0's
        // fence, whose effect is cumulative, then the count (only thread 0 waits)
        epi_sync();
        if (etid == 0) {
          __threadfence();
          atomicAdd(a.sync + kTilesDone + bi, 1ull);
        }
      } else {
        // ---- up to four top-k rows, one per group
        const int r0 = it.a, nr = it.b;
        const int64_t i_last = ch.row0 + r0 + nr - 1;
        if (i_last / 4 > a.topk) {  // some row reads scores: its chunk's tiles must be stored
          if (etid == 0) {
            while (tc_upto < it.chunk) {
              ++tc_upto;
              tiles_cum[tc_upto % a.nbuf] += valid_tiles(chunk_of(a, tc_upto));
            }
            const bool go = wait_counter(a, a.sync + kTilesDone + bi, tiles_cum[bi]);
            if (!go) raise_abort(a, abort_flag);
            *wait_ok = go;
            __threadfence();
          }
          epi_sync();
          if (!*wait_ok) break;
        }
        if (gid < nr) {
          const int64_t i = ch.row0 + r0 + gid;
          topk::row(grp, tsm[gid], buf + static_cast<int64_t>(r0 + gid) * a.ld, static_cast<int>(i / 4), a.topk,
                    a.pool_idx + (i - a.q_begin) * a.topk, a.sync + kIndexGeneralRowsWord);
        }
        epi_sync();
        if (etid == 0) atomicAdd(a.sync + kRowsDone + bi, static_cast<unsigned long long>(nr));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Khat in fp32 with the fixed summation order, then split into bf16 hi + lo.
// One thread per (pool, 8-dim group); Di = 64.  The first threads also zero
// index_topk_kernel's global words.
__global__ void pool_keys_kernel(const __nv_bfloat16* __restrict__ k_idx, int64_t P,
                                 __nv_bfloat16* __restrict__ khat2, unsigned long long* sync_words) {
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

size_t index_topk_smem_bytes() { return kSmemBytes; }

cudaError_t launch_pool_keys(const void* k_idx, int64_t P, void* khat2, unsigned long long* sync_words,
                             const LaunchCtx& ctx) {
  const int64_t threads = P * 8 > kIndexSyncWords ? P * 8 : kIndexSyncWords;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  pool_keys_kernel<<<static_cast<unsigned>(grid), block, 0, ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(k_idx), P, static_cast<__nv_bfloat16*>(khat2), sync_words);
  return cudaGetLastError();
}

cudaError_t launch_index_topk(const CUtensorMap& q_map, const CUtensorMap& khat_map, const float* w, float* scores,
                              int64_t ld, int64_t buf_stride, int nbuf, int64_t q_begin, int64_t q_end, int chunk,
                              int Hi, int topk, int32_t* pool_idx, unsigned long long* sync_words,
                              const LaunchCtx& ctx) {
  Args a;
  a.w = w;
  a.scores = scores;
  a.ld = ld;
  a.buf_stride = buf_stride;
  a.nbuf = nbuf;
  a.lag = nbuf - 1 < kMaxRowLag ? nbuf - 1 : kMaxRowLag;
  a.q_begin = q_begin;
  a.q_end = q_end;
  a.chunk = chunk;
  a.nchunks = static_cast<int>((q_end - q_begin + chunk - 1) / chunk);
  a.Hi = Hi;
  a.topk = topk;
  a.pool_idx = pool_idx;
  a.sync = sync_words;
  a.status = ctx.status;
  a.limit_ns = ctx.wait_limit_ns;
  a.inject = ctx.inject_timeout;
  static std::atomic<bool> attr_done[kAttrDevices];
  {
    const cudaError_t e = set_smem_limit_once(index_topk_kernel, static_cast<int>(kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctx.num_sms);  // one CTA per SM, all resident: the items' waits need it
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, index_topk_kernel, q_map, khat_map, a);
}

}  // namespace dsa
