// attn_fwd_tc.cu -- sparse attention forward with both contractions on
// tcgen05 (dsa_sparse_attn_fwd_tc): the same result as attn_fwd.cu within
// rounding, by a persistent warp-specialised kernel.  On GB300 it is slower
// than attn_fwd.cu's mma.sync kernel: with only 16 query heads every MMA has
// N = 16, so each one spends its time fetching its 4 KB A tile (K or V) from
// shared memory rather than multiplying, and that fetch competes with the
// gather's shared-memory writes.  It is kept as the measured tensor-core
// alternative.
//
// [SkyRL-1M §模型与瓶颈] each query attends to ~2048 selected keys (the 4
// tokens of each selected pool) rather than to the whole prefix; here query i
// also attends to its own partial pool {4*floor(i/4), ..., i}.  The 16 query
// heads share one KV head, so one gathered K/V row serves all 16 heads.
// [CP-lesson §改进二, evidence ②] the softmax is computed online over blocks
// of keys, which reproduces the one-shot softmax exactly in real arithmetic.
//
// One persistent CTA per SM walks its queries (launch rows blockIdx.x,
// blockIdx.x + gridDim.x, ...) as one stream of key blocks of 32 pool slots
// (128 keys); a query's last block holds what is left of its slots.  Three
// warp roles run that stream as a pipeline, linked by mbarriers:
//
//   producers (warps 0-7) gather each block's K and V rows with 16-byte
//     cp.async copies straight into the tensor core's 128-byte swizzled
//     layout, into a 3-stage ring (64 KB a stage), with the query's Q tile
//     at its first block.  A per-stage record carries the block's pools.
//   MMA issuer (warp 8, one thread) runs both contractions on tcgen05 with
//     fp32 accumulators in tensor memory:
//       S^T (128 keys x 16 heads)   = K_blk (K-major) . Q^T      (M = 128, N = 16)
//       O^T (128 dims x 16 heads)  += V_blk^T (MN-major) . P^T (MN-major)  (M = 128, N = 16)
//     issuing S of block b before O^T of block b - 1, so the softmax of
//     block b overlaps the second product of block b - 1.
//   softmax (warps 9-12) take one key per thread from S^T, write P^T (bf16)
//     for the issuer, and at a query's last block normalise O^T and store
//     o and lse.
//
// Online softmax with a lagging maximum: a block's probabilities are taken
// against m_h, a per-head maximum shared by the softmax threads, as long as no
// score of the block exceeds m_h + kLagLog2 (so each p <= 2^kLagLog2 and
// nothing overflows).  When one does (always at a query's first block), they
// take the block's exact maxima, set m_h to them and rescale O^T in tensor
// memory and the running normalisers by 2^(m_old - m_new).  The normalised
// result does not depend on which m_h was used, so this is the same softmax;
// it only avoids a cross-thread maximum and an accumulator rescale per block.
//
// Every mbarrier wait is bounded; a wait that runs out records
// kStatusTimeout and raises the CTA's abort word, and every role then leaves
// its loop at its next check (the roles' group barriers decide that
// uniformly).  Before the tensor memory is freed, the issuer waits (bounded)
// for every product it issued.
#include "dsa_device.cuh"
#include "dsa_kernels.h"

// Measurement build (DSA_FWD_PROFILE=1, off by default): each role adds the
// clock64 cycles of its pipeline segments into per-thread counters, and one
// thread of each role stores them per CTA in g_fwd_prof[cta][32] (producer
// segments at 0.., issuer at 8.., softmax at 16..; the role's block count in
// its last slot), read back by dsa_fwd_tc_profile.
#if DSA_FWD_PROFILE
__device__ unsigned long long g_fwd_prof[1024 * 32];
#define FWD_PROF_BEGIN long long prof_[8] = {0, 0, 0, 0, 0, 0, 0, 0}, prof_t_ = clock64()
#define FWD_PROF(i) (prof_[i] += clock64() - prof_t_, prof_t_ = clock64())
#define FWD_PROF_STORE(off, blocks)                                                         \
  do {                                                                                      \
    for (int x_ = 0; x_ < 7; ++x_) g_fwd_prof[blockIdx.x * 32 + (off) + x_] = prof_[x_];  \
    g_fwd_prof[blockIdx.x * 32 + (off) + 7] = (blocks);                                   \
  } while (0)
#else
#define FWD_PROF_BEGIN
#define FWD_PROF(i)
#define FWD_PROF_STORE(off, blocks)
#endif

namespace dsa {
namespace {

constexpr int kHq = 16;
constexpr int kD = 128;
constexpr int kSlots = 32;                     // pool slots per block
constexpr int kBlkKeys = 4 * kSlots;           // 128
constexpr int kStages = 3;
constexpr uint32_t kHalf = kBlkKeys * 128;     // 16 KB: 64 dims of the block's 128 keys
constexpr uint32_t kTile = 2 * kHalf;          // 32 KB: K (or V) of a block
constexpr uint32_t kStage = 2 * kTile;         // 64 KB: K then V
constexpr uint32_t kQHalf = kHq * 128;         // 2 KB: 64 dims of the 16 heads
constexpr uint32_t kQBytes = 2 * kQHalf;       // 4 KB
constexpr uint32_t kPHeads8 = kBlkKeys * 16;   // 2 KB: P^T of 8 heads (rows of 8 bf16, one per key)
constexpr uint32_t kPBytes = 2 * kPHeads8;     // 4 KB
constexpr uint32_t kOutBytes = kHq * kD * 2;   // 4 KB: one query's o, staged
constexpr int kProducerWarps = 8;
constexpr int kProducerThreads = 32 * kProducerWarps;  // warps 0..7
constexpr int kKeysPerProducer = kBlkKeys * 16 / kProducerThreads;  // 16-B chunks of K (and of V) per thread: 8
constexpr int kMmaWarp = kProducerWarps;               // warp 8
constexpr int kSoftmaxWarp0 = kProducerWarps + 1;      // warps 9..12
constexpr int kSoftmaxThreads = 128;
constexpr int kThreads = (kProducerWarps + 5) * 32;
constexpr uint32_t kBarProducers = 1, kBarSoftmax = 2;  // named barrier ids
constexpr uint32_t kTmemCols = 64;             // S^T buffers at columns 0, 16; O^T buffers at 32, 48
constexpr uint32_t kColO = 32;
constexpr float kLagLog2 = 8.f;                // p <= 2^8 between maximum updates

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Per-stage record of the block in it, written by the producers before they
// arrive on the stage's full barrier.
struct BlockInfo {
  int32_t pools[kSlots];  // pool of each slot (-1: empty or a hole)
  int64_t i;              // the query's position in its sequence
  int64_t r;              // the query's launch row
  int32_t flags;          // kFirst | kLast, or kEnd (no block: end of work)
  int32_t qpar;           // parity of the CTA's query count: Q and O^T buffer
  int32_t pad[2];
};
constexpr int32_t kFirst = 1, kLast = 2, kEnd = 4;

// shared memory map (offsets from the 1024-B aligned base)
constexpr uint32_t kOffQ = kStages * kStage;                 // 196608
constexpr uint32_t kOffP = kOffQ + 2 * kQBytes;              // 204800
constexpr uint32_t kOffOut = kOffP + 2 * kPBytes;            // 212992
constexpr uint32_t kOffInfo = kOffOut + kOutBytes;           // 217088
constexpr uint32_t kOffBars = kOffInfo + 512;                // 217600
constexpr uint32_t kOffMisc = kOffBars + 256;                // 217856
constexpr uint32_t kOffProw = kOffMisc + 512;                // 218368: pool_idx rows, 1 or 2 buffers
constexpr uint32_t kSmemFixed = 1024 + kOffProw;             // 219392 (with the alignment slack)
constexpr uint32_t kSmemMax = 227 * 1024;                    // opt-in shared memory of one CTA
static_assert(kStages * sizeof(BlockInfo) <= 512, "block records fit");

// barrier slots (8 B each) from kOffBars
constexpr uint32_t kBarFull = 0;      // [3] a stage's copies landed and its record is written
constexpr uint32_t kBarKvEmpty = 3;   // [3] the stage's O^T product completed (commit)
constexpr uint32_t kBarSFull = 6;     // [2] S^T buffer written (commit)
constexpr uint32_t kBarSEmpty = 8;    // [2] S^T buffer read (128 softmax arrivals)
constexpr uint32_t kBarPFull = 10;    // [2] P^T buffer written (128 softmax arrivals)
constexpr uint32_t kBarPEmpty = 12;   // [2] O^T product that read the P^T buffer completed (commit)
constexpr uint32_t kBarQEmpty = 14;   // [2] last S^T product of the Q buffer's query completed (commit)
constexpr uint32_t kBarOFull = 16;    // [2] O^T buffer complete for its query (commit)
constexpr uint32_t kBarOEmpty = 18;   // [2] O^T buffer read (128 softmax arrivals)
constexpr uint32_t kBarDrain = 20;    // every product issued has completed (commit)
constexpr uint32_t kBarProw = 21;     // [2] a pool_idx row landed (a copy-completion arrival per producer)
constexpr int kNumBars = 23;
static_assert(kNumBars * 8 <= 256, "barriers fit");
static_assert(kProducerThreads % 16 == 0 && kKeysPerProducer * kProducerThreads == kBlkKeys * 16, "gather map");
// kBarFull: one copy-completion arrival per producer thread, plus one
// ordinary arrival from producer 0 once the block's record is written
constexpr uint32_t kFullArrivals = kProducerThreads + 1;

// bytes of one pool_idx row buffer (whole 16-B units)
__host__ __device__ constexpr uint32_t prow_bytes(int topk) { return static_cast<uint32_t>((topk + 3) / 4) * 16; }

// Byte offset of the 16-B chunk holding dims 8c..8c+7 (c = 0..15) of row r
// in a tile of 128-byte swizzled rows split in two 64-dim halves `half`
// bytes apart.
__device__ __forceinline__ uint32_t sw_off(int r, int c, uint32_t half) {
  return (c >> 3) * half + r * 128 + ((((c & 7) ^ r) & 7) << 4);
}

// Issues block pb's O^T product (all 8 key steps: absent keys have p = 0 and
// zero-filled V rows) once its P^T is written and, at the first block of a
// query, once the O^T buffer's previous query has been read out; then
// commits the stage, the P^T buffer and (at a query's last block) the O^T
// buffer.  False when a wait runs out.
__device__ __forceinline__ bool issue_pv(uint32_t bars, uint32_t tmem, uint64_t dV0, uint64_t dP0, int64_t pb, int st,
                                         int flags, int qpar, int64_t qn, uint64_t limit_ns,
                                         const volatile int* abort_flag) {
  constexpr uint32_t idesc_pv = umma_idesc_bf16_f32(128, 16) | kUmmaAMnMajor | kUmmaBMnMajor;
  if (!mbar_wait(bars + 8 * (kBarPFull + (pb & 1)), (pb >> 1) & 1, limit_ns, abort_flag)) return false;
  if ((flags & kFirst) && qn >= 2 &&
      !mbar_wait(bars + 8 * (kBarOEmpty + qpar), ((qn - 2) >> 1) & 1, limit_ns, abort_flag))
    return false;
  tc_fence_after();
  const uint64_t dv = dV0 + ((st * kStage) >> 4);
  const uint64_t dp = dP0 + ((static_cast<uint32_t>(pb & 1) * kPBytes) >> 4);
  const uint32_t d = tmem + kColO + static_cast<uint32_t>(qpar) * 16;
  const uint32_t acc0 = (flags & kFirst) ? 0u : 1u;
#pragma unroll
  for (int kk = 0; kk < kBlkKeys / 16; ++kk)
    umma_bf16(d, dv + ((kk * 2048) >> 4), dp + ((kk * 256) >> 4), idesc_pv, kk == 0 ? acc0 : 1u);
  umma_commit(bars + 8 * (kBarKvEmpty + st));
  umma_commit(bars + 8 * (kBarPEmpty + (pb & 1)));
  if (flags & kLast) umma_commit(bars + 8 * (kBarOFull + qpar));
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                       const __nv_bfloat16* __restrict__ v, const int32_t* __restrict__ pool_idx, int64_t q0,
                       int64_t rows, int topk, float scale_log2, __nv_bfloat16* __restrict__ o,
                       float* __restrict__ lse, unsigned* status, uint64_t limit_ns, int prow_bufs,
                       const __grid_constant__ SeqTable tab) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-B swizzle atoms need 1024-B alignment
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sRing = base, sQ = base + kOffQ, sP = base + kOffP;
  BlockInfo* info = reinterpret_cast<BlockInfo*>(gbase + kOffInfo);
  const uint32_t bars = base + kOffBars;
  uint8_t* misc = gbase + kOffMisc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  int* s_nsel = reinterpret_cast<int*>(misc + 8);
  float* s_red = reinterpret_cast<float*>(misc + 64);  // [4][kHq]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](uint32_t slot) { return bars + 8 * slot; };

  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), kFullArrivals);
      mbar_init(bar(kBarKvEmpty + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(kBarSFull + x), 1);
      mbar_init(bar(kBarSEmpty + x), kSoftmaxThreads);
      mbar_init(bar(kBarPFull + x), kSoftmaxThreads);
      mbar_init(bar(kBarPEmpty + x), 1);
      mbar_init(bar(kBarQEmpty + x), 1);
      mbar_init(bar(kBarOFull + x), 1);
      mbar_init(bar(kBarOEmpty + x), kSoftmaxThreads);
    }
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarProw), kProducerThreads);
    mbar_init(bar(kBarProw + 1), kProducerThreads);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kMmaWarp) {
    // ================================================================ producers
    const int pt = tid;                      // 0..255
    constexpr int kKeyStep = kProducerThreads / 16;  // 16
    const int kr0 = pt >> 4, cc = pt & 15;   // keys kr0 + 16u (u = 0..7), 16-B chunk cc
    const int jj = kr0 & 3;                  // key offset within its pool
    const uint32_t dst_off = sw_off(kr0, cc, kHalf);
    const uint32_t prow_ld = prow_bytes(topk);
    // Query n's pool_idx row is copied into buffer n % prow_bufs ahead of
    // use; every producer arrives on the buffer's barrier once per fill.
    auto prefetch_prow = [&](int64_t n) {
      const int64_t r = blockIdx.x + n * gridDim.x;
      const uint32_t dst = base + kOffProw + static_cast<uint32_t>(n % prow_bufs) * prow_ld;
      if (r < rows) {
        const int32_t* prow = pool_idx + r * topk;
        for (int j = pt; j < topk; j += kProducerThreads) cp_async4(dst + 4 * j, prow + j);
      }
      cp_async_mbar_arrive_noinc(bar(kBarProw + static_cast<int>(n % prow_bufs)));
    };
    bool fail = false, bad = false;
    int64_t b = 0;  // blocks issued by this CTA
    FWD_PROF_BEGIN;
    prefetch_prow(0);
    for (int64_t n = 0;; ++n) {
      const int64_t r = blockIdx.x + n * gridDim.x;
      if (r >= rows) break;
      if (!mbar_wait(bar(kBarProw + static_cast<int>(n % prow_bufs)), (n / prow_bufs) & 1, limit_ns, abort_flag))
        fail = true;
      if (named_bar_or(kBarProducers, kProducerThreads, fail)) {
        fail = true;
        break;
      }
      FWD_PROF(0);
      if (prow_bufs == 2) prefetch_prow(n + 1);
      const int32_t* prow =
          reinterpret_cast<const int32_t*>(gbase + kOffProw + static_cast<uint32_t>(n % prow_bufs) * prow_ld);
      int64_t i, kv0;
      seq_locate(tab, q0, r, &i, &kv0);
      const int64_t n_elig = i >> 2;
      const __nv_bfloat16* kq = k + kv0 * kD;
      const __nv_bfloat16* vq = v + kv0 * kD;
      // selected pools: the leading non-negative entries
      if (pt == 0) *s_nsel = topk;
      named_bar_sync(kBarProducers, kProducerThreads);
      for (int j = pt; j < topk; j += kProducerThreads)
        if (prow[j] < 0) atomicMin(s_nsel, j);
      named_bar_sync(kBarProducers, kProducerThreads);
      const int nsel = *s_nsel;
      const int nblk = (nsel + 1 + kSlots - 1) / kSlots;
      FWD_PROF(1);
      for (int bq = 0; bq < nblk; ++bq, ++b) {
        const int st = static_cast<int>(b % kStages);
        // the stage's previous block has been consumed by its O^T product
        if (b >= kStages && !mbar_wait(bar(kBarKvEmpty + st), ((b / kStages) - 1) & 1, limit_ns, abort_flag))
          fail = true;
        // the Q buffer's previous query has had its last S^T product
        if (bq == 0 && n >= 2 && !mbar_wait(bar(kBarQEmpty + (n & 1)), ((n - 2) >> 1) & 1, limit_ns, abort_flag))
          fail = true;
        if (named_bar_or(kBarProducers, kProducerThreads, fail)) {
          fail = true;
          break;
        }
        FWD_PROF(2);
        // Slot s < nsel holds pool prow[s]; slot nsel is the query's own
        // pool n_elig (rows 4 n_elig .. i); slots beyond are empty.  An
        // entry that is not an eligible pool, or breaks ascending order, is
        // recorded as a device-side check failure and becomes a hole (never
        // read, always masked), so no access leaves the K/V rows.
        BlockInfo* inf = info + st;
        if (pt < kSlots) {
          const int s = kSlots * bq + pt;
          int32_t p = -1;
          if (s < nsel) {
            const int32_t x = prow[s];
            if (x < n_elig) p = x;
            else bad = true;
            if (s > 0 && x <= prow[s - 1]) bad = true;
          } else if (s == nsel) {
            p = static_cast<int32_t>(n_elig);
          }
          inf->pools[pt] = p;
        }
        if (pt == 0) {
          inf->i = i;
          inf->r = r;
          inf->flags = (bq == 0 ? kFirst : 0) | (bq == nblk - 1 ? kLast : 0);
          inf->qpar = static_cast<int32_t>(n & 1);
        }
        named_bar_sync(kBarProducers, kProducerThreads);
        FWD_PROF(3);
        if (bq == 0) {
          const __nv_bfloat16* qrow = q + r * (kHq * kD);
          const uint32_t qb = sQ + static_cast<uint32_t>(n & 1) * kQBytes;
#pragma unroll
          for (int u = 0; u < (kHq * 16) / kProducerThreads; ++u) {
            const int c = pt + kProducerThreads * u;  // head c / 16, dims 8 (c % 16) ..
            cp_async16(qb + sw_off(c >> 4, c & 15, kQHalf), qrow + c * 8, true);
          }
        }
        // K rows of absent keys are left as they are (their scores are
        // masked); V rows of absent keys are zero-filled (their p is 0)
        const uint32_t sb = sRing + st * kStage + dst_off;
        const int32_t* bp = inf->pools + (kr0 >> 2);
#pragma unroll
        for (int u = 0; u < kKeysPerProducer; ++u) {
          const int32_t p = bp[(kKeyStep / 4) * u];
          const int64_t row = 4 * static_cast<int64_t>(p) + jj;
          const bool ok = p >= 0 && row <= i;
          DSA_CHECK(status, p <= n_elig && dst_off + u * (kKeyStep * 128) + 16 <= kTile);
          const int64_t src = (ok ? row : 0) * kD + cc * 8;
          if (ok) cp_async16(sb + u * (kKeyStep * 128), kq + src, true);
          cp_async16(sb + kTile + u * (kKeyStep * 128), vq + src, ok);
        }
        // the stage is full once these copies land; the issuer makes them
        // visible to the tensor core with a proxy fence after its wait
        cp_async_mbar_arrive_noinc(bar(kBarFull + st));
        if (pt == 0) mbar_arrive(bar(kBarFull + st));
        FWD_PROF(4);
      }
      if (fail) break;
      if (prow_bufs == 1) prefetch_prow(n + 1);  // the row buffer is no longer read
    }
    if (bad) record_status(status, kStatusInternal);
    if (!fail) {
      // end-of-work record in the next stage
      const int st = static_cast<int>(b % kStages);
      if (b >= kStages && !mbar_wait(bar(kBarKvEmpty + st), ((b / kStages) - 1) & 1, limit_ns, abort_flag))
        fail = true;
      if (!named_bar_or(kBarProducers, kProducerThreads, fail)) {
        if (pt == 0) info[st].flags = kEnd;
        cp_async_mbar_arrive_noinc(bar(kBarFull + st));
        if (pt == 0) mbar_arrive(bar(kBarFull + st));
      } else {
        fail = true;
      }
    }
    cp_async_wait<0>();
    FWD_PROF(5);
    if (pt == 0) FWD_PROF_STORE(0, b);
    if (fail) {
      *abort_flag = 1;
      record_status(status, kStatusTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16_f32(128, 16);
      // descriptors of stage 0's K and V tiles, Q buffer 0 and P^T buffer 0;
      // the others differ by whole 16-B units of the start address field
      const uint64_t dK0 = umma_desc_sw128(sRing);
      const uint64_t dV0 = umma_desc_sw128_mn(sRing + kTile, kHalf, 1024);
      const uint64_t dQ0 = umma_desc_sw128(sQ);
      const uint64_t dP0 = umma_desc_mn_noswizzle(sP, 128, kPHeads8);
      bool fail = false;
      int64_t b = 0;
      int64_t qn = -1;  // the CTA's query count of the current block
      // the block whose O^T product is still to be issued
      bool have_prev = false;
      FWD_PROF_BEGIN;
      int prev_st = 0, prev_flags = 0, prev_qpar = 0;
      int64_t prev_qn = 0;
      while (true) {
        const int st = static_cast<int>(b % kStages);
        if (!mbar_wait(bar(kBarFull + st), (b / kStages) & 1, limit_ns, abort_flag)) {
          fail = true;
          break;
        }
        FWD_PROF(0);
        // the producers' cp.async writes (generic proxy) become visible to
        // the tensor core's operand reads (async proxy)
        fence_proxy_async_smem();
        const BlockInfo* inf = info + st;
        const int flags = inf->flags;
        if (flags & kEnd) break;
        const int qpar = inf->qpar;
        if (flags & kFirst) ++qn;
        // S^T of block b into S buffer b & 1 (read by the softmax of block b - 2)
        if (b >= 2 && !mbar_wait(bar(kBarSEmpty + (b & 1)), ((b - 2) >> 1) & 1, limit_ns, abort_flag)) {
          fail = true;
          break;
        }
        FWD_PROF(1);
        tc_fence_after();
        {
          const uint64_t dk = dK0 + ((st * kStage) >> 4);
          const uint64_t dq = dQ0 + ((static_cast<uint32_t>(qpar) * kQBytes) >> 4);
          const uint32_t d = tmem + static_cast<uint32_t>(b & 1) * 16;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            umma_bf16(d, dk + (((kk >> 2) * kHalf + (kk & 3) * 32) >> 4),
                      dq + (((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4), idesc_s, kk > 0 ? 1u : 0u);
          umma_commit(bar(kBarSFull + (b & 1)));
          if (flags & kLast) umma_commit(bar(kBarQEmpty + qpar));
        }
        FWD_PROF(2);
        // O^T product of block b - 1
        if (have_prev && !issue_pv(bars, tmem, dV0, dP0, b - 1, prev_st, prev_flags, prev_qpar, prev_qn, limit_ns,
                                   abort_flag)) {
          fail = true;
          break;
        }
        FWD_PROF(3);
        have_prev = true;
        prev_st = st;
        prev_flags = flags;
        prev_qpar = qpar;
        prev_qn = qn;
        ++b;
      }
      if (!fail && have_prev &&
          !issue_pv(bars, tmem, dV0, dP0, b - 1, prev_st, prev_flags, prev_qpar, prev_qn, limit_ns, abort_flag))
        fail = true;
      // every product issued has completed before the tensor memory is read
      // for the last time or freed
      umma_commit(bar(kBarDrain));
      if (!mbar_wait(bar(kBarDrain), 0, limit_ns, nullptr)) fail = true;
      FWD_PROF(4);
      FWD_PROF_STORE(8, b);
      if (fail) {
        *abort_flag = 1;
        record_status(status, kStatusTimeout);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ softmax + epilogue
    const int sth = tid - kSoftmaxWarp0 * 32;  // 0..127
    const int quarter = warp & 3;              // tensor-memory lane quarter this warp may access
    const int key = quarter * 32 + lane;       // this thread's key of every block (S^T row)
    const int dim = key;                       // and its dim of O^T
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    float m_h[kHq], l_part[kHq];
#pragma unroll
    for (int h = 0; h < kHq; ++h) {
      m_h[h] = -INFINITY;
      l_part[h] = 0.f;
    }
    bool fail = false;
    int64_t b = 0, qn = 0;
    FWD_PROF_BEGIN;
    while (true) {
      const int st = static_cast<int>(b % kStages);
      if (!mbar_wait(bar(kBarFull + st), (b / kStages) & 1, limit_ns, abort_flag)) fail = true;
      if (named_bar_or(kBarSoftmax, kSoftmaxThreads, fail)) break;
      FWD_PROF(0);
      // everything the block's record holds is read here: once this
      // thread's P^T is handed over, the producers may reuse the stage
      const BlockInfo* inf = info + st;
      const int flags = inf->flags;
      if (flags & kEnd) break;
      const int qpar = inf->qpar;
      const int64_t r = inf->r;
      if (flags & kFirst) {
#pragma unroll
        for (int h = 0; h < kHq; ++h) {
          m_h[h] = -INFINITY;
          l_part[h] = 0.f;
        }
      }
      bool valid;
      {
        const int32_t p = inf->pools[key >> 2];
        valid = p >= 0 && 4 * static_cast<int64_t>(p) + (key & 3) <= inf->i;
      }
      float x[kHq];
      {
        if (!mbar_wait(bar(kBarSFull + (b & 1)), (b >> 1) & 1, limit_ns, abort_flag)) fail = true;
        tc_fence_after();
        uint32_t sr[16];
        tmem_ld16(tmem + t_lane + static_cast<uint32_t>(b & 1) * 16, sr);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarSEmpty + (b & 1)));
#pragma unroll
        for (int h = 0; h < kHq; ++h) x[h] = valid ? __uint_as_float(sr[h]) * scale_log2 : -INFINITY;
      }
      FWD_PROF(1);
      bool above = false;
#pragma unroll
      for (int h = 0; h < kHq; ++h) above |= x[h] > m_h[h] + kLagLog2;
      if (named_bar_or(kBarSoftmax, kSoftmaxThreads, above)) {
        // exact maxima of the block
        float mx[kHq];
#pragma unroll
        for (int h = 0; h < kHq; ++h) {
          mx[h] = x[h];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], off));
        }
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < kHq; ++h) s_red[quarter * kHq + h] = mx[h];
        }
        named_bar_sync(kBarSoftmax, kSoftmaxThreads);
        float alpha[kHq];
#pragma unroll
        for (int h = 0; h < kHq; ++h) {
          const float bm = fmaxf(fmaxf(s_red[h], s_red[kHq + h]), fmaxf(s_red[2 * kHq + h], s_red[3 * kHq + h]));
          const float mn = fmaxf(m_h[h], bm);
          // nothing has been accumulated against an undefined maximum (every
          // earlier key of the head was masked): its sums are zero either way
          const float mu_new = mn == -INFINITY ? 0.f : mn;
          alpha[h] = m_h[h] == -INFINITY ? 0.f : exp2f(m_h[h] - mu_new);
          m_h[h] = mn;
          l_part[h] *= alpha[h];
        }
        if (!(flags & kFirst)) {
          // O^T holds the query's earlier blocks once block b - 1's product completed
          if (!mbar_wait(bar(kBarPEmpty + ((b - 1) & 1)), ((b - 1) >> 1) & 1, limit_ns, abort_flag)) fail = true;
          tc_fence_after();
          uint32_t ov[16];
          const uint32_t ta = tmem + t_lane + kColO + static_cast<uint32_t>(qpar) * 16;
          tmem_ld16(ta, ov);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < kHq; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
          tmem_st16(ta, ov);
          tmem_st_wait();
        }
        named_bar_sync(kBarSoftmax, kSoftmaxThreads);  // s_red is read before it is reused
      }
      // probabilities against the lagging maximum, into P^T buffer b & 1
      // (bf16, MN-major without swizzle: for each group of 8 heads, one
      // 16-B row per key); its previous reader is block b - 2's product
      FWD_PROF(2);
      if (b >= 2 && !mbar_wait(bar(kBarPEmpty + (b & 1)), ((b - 2) >> 1) & 1, limit_ns, abort_flag)) fail = true;
      FWD_PROF(3);
      {
        uint32_t pk[kHq / 2];
#pragma unroll
        for (int h = 0; h < kHq; h += 2) {
          const float mu0 = m_h[h] == -INFINITY ? 0.f : m_h[h];
          const float mu1 = m_h[h + 1] == -INFINITY ? 0.f : m_h[h + 1];
          const float p0 = exp2f(x[h] - mu0), p1 = exp2f(x[h + 1] - mu1);
          l_part[h] += p0;
          l_part[h + 1] += p1;
          pk[h / 2] = pack_bf16(p0, p1);
        }
        DSA_CHECK(status, key >= 0 && key < kBlkKeys);
        const uint32_t pa = sP + static_cast<uint32_t>(b & 1) * kPBytes + key * 16;
        st_shared_v4(pa, pk[0], pk[1], pk[2], pk[3]);
        st_shared_v4(pa + kPHeads8, pk[4], pk[5], pk[6], pk[7]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + (b & 1)));
      FWD_PROF(4);

      if (flags & kLast) {
        // ---- the query's epilogue: normalisers, lse, o
#pragma unroll
        for (int h = 0; h < kHq; ++h) {
          float t = l_part[h];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
          if (lane == 0) s_red[quarter * kHq + h] = t;
        }
        named_bar_sync(kBarSoftmax, kSoftmaxThreads);
        float inv[kHq];
#pragma unroll
        for (int h = 0; h < kHq; ++h) {
          const float L = (s_red[h] + s_red[kHq + h]) + (s_red[2 * kHq + h] + s_red[3 * kHq + h]);
          inv[h] = __frcp_rn(L);
          if (sth == h) {
            const float mu = m_h[h] == -INFINITY ? 0.f : m_h[h];
            lse[r * kHq + h] = (mu + log2f(L)) * kLn2;
          }
        }
        if (!mbar_wait(bar(kBarOFull + qpar), (qn >> 1) & 1, limit_ns, abort_flag)) fail = true;
        tc_fence_after();
        uint32_t ov[16];
        tmem_ld16(tmem + t_lane + kColO + static_cast<uint32_t>(qpar) * 16, ov);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarOEmpty + qpar));
        __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(gbase + kOffOut);
#pragma unroll
        for (int h = 0; h < kHq; ++h) stage[h * kD + dim] = __float2bfloat16_rn(__uint_as_float(ov[h]) * inv[h]);
        named_bar_sync(kBarSoftmax, kSoftmaxThreads);
        const int4* src = reinterpret_cast<const int4*>(stage);
        int4* dst = reinterpret_cast<int4*>(o + r * (kHq * kD));
#pragma unroll
        for (int u = 0; u < static_cast<int>(kOutBytes / 16) / kSoftmaxThreads; ++u)
          dst[sth + u * kSoftmaxThreads] = src[sth + u * kSoftmaxThreads];
        named_bar_sync(kBarSoftmax, kSoftmaxThreads);  // staging and s_red free for the next query
        ++qn;
        FWD_PROF(5);
      }
      ++b;
    }
    if (sth == 0) FWD_PROF_STORE(16, b);
    if (fail) {
      *abort_flag = 1;
      record_status(status, kStatusTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_attn_fwd_tc(const void* q, const void* k, const void* v, const int32_t* pool_idx, int64_t q_begin,
                            int64_t q_end, int topk, float scale, void* o, float* lse, const LaunchCtx& ctx,
                            const SeqTable* tab) {
  if (q_end <= q_begin) return cudaSuccess;
  static const SeqTable kNoTable = {};
  static std::atomic<bool> attr_done[kAttrDevices];
  const cudaError_t e = set_smem_limit_once(attn_fwd_tc_kernel, static_cast<int>(kSmemMax), attr_done);
  if (e != cudaSuccess) return e;
  // two pool_idx row buffers (the next query's row is fetched a whole query
  // ahead) when they fit, else one (fetched after the query's last block)
  const int prow_bufs = kSmemFixed + 2 * prow_bytes(topk) <= kSmemMax ? 2 : 1;
  const size_t smem = kSmemFixed + static_cast<size_t>(prow_bufs) * prow_bytes(topk);
  const int64_t rows = q_end - q_begin;
  const int64_t grid = rows < ctx.num_sms ? rows : ctx.num_sms;
  attn_fwd_tc_kernel<<<static_cast<unsigned>(grid), kThreads, smem, ctx.stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), pool_idx, q_begin, rows, topk, scale * kLog2e,
      static_cast<__nv_bfloat16*>(o), lse, ctx.status, ctx.wait_limit_ns, prow_bufs, tab ? *tab : kNoTable);
  return cudaGetLastError();
}

// Role counters of the last profiled launch (profile build): ctas x 32
// words, see g_fwd_prof.  Returns the words copied, or -1 without the build.
int fwd_tc_profile_read(unsigned long long* out, int ctas) {
#if DSA_FWD_PROFILE
  if (ctas < 0 || ctas > 1024) return -1;
  if (cudaMemcpyFromSymbol(out, g_fwd_prof, sizeof(unsigned long long) * 32 * ctas) != cudaSuccess) return -1;
  return 32 * ctas;
#else
  (void)out, (void)ctas;
  return -1;
#endif
}

}  // namespace dsa
