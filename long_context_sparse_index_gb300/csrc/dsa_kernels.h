// dsa_kernels.h -- host-side launchers of the libdsa kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>
#include <utility>

namespace dsa {

// Raises `kernel`'s dynamic shared memory limit to `bytes` on the current
// device, once per device and call site: `done` holds one flag per device
// ordinal (atomic, so host threads racing here at worst repeat the
// idempotent call; ordinals past the array are set on every call).
constexpr int kAttrDevices = 64;
template <typename Kernel>
inline cudaError_t set_smem_limit_once(Kernel kernel, int bytes, std::atomic<bool> (&done)[kAttrDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kAttrDevices;
  if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) done[dev].store(true, std::memory_order_release);
  return e;
}

// Host side of every public entry point: an NVTX range named for it, and (for
// the outermost entry a host thread is in) a fresh record of the kernels it
// launches and the plan they ran with, read back by dsa_last_kernel_config.
void call_begin(const char* fn);
void call_end();
void call_param(const char* key, long long value);
void call_variant(const char* variant);
struct CallScope {
  explicit CallScope(const char* fn) { call_begin(fn); }
  ~CallScope() { call_end(); }
  CallScope(const CallScope&) = delete;
  CallScope& operator=(const CallScope&) = delete;
};

// sequences per launch of the varlen calls (their table rides in the kernel
// parameters)
constexpr int kSeqBatch = 256;

struct LaunchCtx {
  cudaStream_t stream;
  unsigned* status;        // device status word (kStatus* bits)
  uint64_t wait_limit_ns;  // bound on every device-side spin-wait
  int inject_timeout;      // fault injection: producers issue no copies, so waits run out
  int num_sms;
  int pdl;                 // launch may start early (programmatic stream serialization)
  int persistent_ctas;     // the persistent indexer's CTAs: 0 = one per SM, cooperative; else that many
};

// Launches `kernel` on ctx.stream, allowing early start when ctx.pdl is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(const LaunchCtx& ctx, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ctx.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Global words of the fused indexer + top-k kernel (64-bit each), at the start
// of its workspace, and its most per-chunk buffer slots.
constexpr int kIndexSyncWords = 48;
constexpr int kMaxBufs = 8;
// word counting the rows listed for the fallback kernel (their candidates
// could not certify the top-k); it survives the call (the next call's key
// pooling zeroes it)
constexpr int kIndexFallbackRowsWord = 36;

// Sizes of the indexer's per-chunk buffers and scratch, from S, chunk and topk.
struct IndexPlan {
  int64_t P;          // selectable pools, floor(S/4)
  int64_t Ppad;       // P rounded up to 256 (at least 256)
  int sigma;          // sample stride in pools (power of two)
  int rsel;           // the row threshold is the rsel-th largest sample
  int cap;            // candidate slots per row
  int64_t samp_ld;    // sampled scores per row: ceil(P / sigma) rounded up to 256
  int64_t slot_rows;  // rows per slot: min(chunk, S)
  int64_t thr_ld;     // thresholds and counts per slot: slot_rows rounded up to 128
  int64_t samp_slot;  // floats of samples per slot
  int64_t cand_slot;  // candidates per slot
  int fb_ctas;        // CTAs of the fallback kernel
  int64_t fb_ld;      // floats per fallback scratch row (Ppad)
};
// One work item of the persistent indexer, recorded by the item-trace build
// (DSA_ITEM_TRACE): globaltimer stamps when its epilogue took it (t0), when
// the fold over heads ended (t1; = t0 for row items), when its dependency wait
// ended (t2) and when it was published (t3).
struct IndexTraceRec {
  uint32_t kind_sm;   // item kind in bits 0..7, SM id in bits 8..
  uint32_t chunk;
  uint64_t t0, t1, t2, t3;
};
struct IndexBuffers {
  unsigned long long* sync;
  IndexTraceRec* trace;            // item-trace build only: records, and
  unsigned long long* trace_count; // their count (caller zeroes it); null: none
  int64_t trace_cap;
  void* khat2;        // [P, 128] bf16: hi in columns 0..63, lo in 64..127
  float* khat32;      // [P, 64] fp32
  float* samples;     // [nbuf][slot_rows][samp_ld]
  uint2* thr;         // [nbuf][thr_ld]
  unsigned* cnt;      // [nbuf][thr_ld]
  uint2* cands;       // [nbuf][slot_rows][cap]
  int nbuf;
  int32_t* fb_rows;   // [rows of the call]
  float* fb_scratch;  // [fb_ctas][fb_ld]
};

// Pooled indexer keys: khat2 [P, 128] bf16 (hi, lo) and khat32 [P, 64] fp32.
// Also zeroes the kIndexSyncWords words at sync_words (always launch it, even
// with P == 0, before launch_index_topk).
cudaError_t launch_pool_keys(const void* k_idx, int64_t P, void* khat2, float* khat32, unsigned long long* sync_words,
                             const LaunchCtx& ctx);

// Indexer scores and per-row top-k for query rows [q_begin, q_end), in query
// chunks of `chunk` rows, as one persistent cooperative kernel (one CTA per
// SM); chunk c uses slot c % b.nbuf of the per-chunk buffers; pool_idx row r
// is query q_begin + r.  Rows it cannot certify are listed in b.fb_rows for
// launch_index_fallback, which must follow it on the same stream.
cudaError_t launch_index_topk(const CUtensorMap& q_map, const CUtensorMap& khat_map, const CUtensorMap& samp_map,
                              const IndexPlan& pl, const IndexBuffers& b, const float* w, int64_t q_begin,
                              int64_t q_end, int chunk, int Hi, int topk, int32_t* pool_idx, const LaunchCtx& ctx);
cudaError_t launch_index_fallback(const void* q_idx, const IndexPlan& pl, const IndexBuffers& b, const float* w,
                                  int64_t q_begin, int Hi, int topk, int32_t* pool_idx, const LaunchCtx& ctx);
size_t index_topk_smem_bytes();

// Rows whose query keeps every eligible pool (n = floor(i/4) <= topk), for
// whole short sequences of a packed batch: row i of sequence s (packed row
// start[s] + i) gets pools 0 .. n-1, then -1.  One CTA per sequence.
struct ShortSeqs {
  int n;
  int64_t start[kSeqBatch];
  int64_t len[kSeqBatch];
};
cudaError_t launch_short_rows(int32_t* pool_idx, int topk, const ShortSeqs& seqs, const LaunchCtx& ctx);

// Packed sequences of one attention launch (the varlen calls): the launch's
// rows are packed rows row0 .. row0 + rows - 1, and sequence s of the table
// holds packed rows cu[s] .. cu[s+1] - 1 (its keys and values are packed rows
// too), s < n.  n == 0: one sequence, and the launch's row r is its query
// q_begin + r.  Passed by value as a kernel parameter.
struct SeqTable {
  int n;
  int64_t row0;
  int64_t cu[kSeqBatch + 1];
};

// Query i and the packed row of its sequence's first key, for launch row r.
__device__ __forceinline__ void seq_locate(const SeqTable& t, int64_t q0, int64_t r, int64_t* i, int64_t* kv0) {
  if (t.n == 0) {
    *i = q0 + r;
    *kv0 = 0;
    return;
  }
  const int64_t g = t.row0 + r;
  int lo = 0, hi = t.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t.cu[mid] <= g) lo = mid;
    else hi = mid - 1;
  }
  *kv0 = t.cu[lo];
  *i = g - t.cu[lo];
}

// Queries [q_begin, q_end) (global positions); q, pool_idx, o and lse hold
// their rows locally (row r = query q_begin + r); k and v are the whole
// sequence.  With a table (tab->n > 0), the launch covers its packed rows
// instead (q_begin is unused, q_end - q_begin = rows) and k and v are the
// whole packed batch.
cudaError_t launch_attn_fwd(const void* q, const void* k, const void* v, const int32_t* pool_idx, int64_t q_begin,
                            int64_t q_end, int topk, float scale, void* o, float* lse, const LaunchCtx& ctx,
                            const SeqTable* tab = nullptr);

// The same forward on tcgen05 (attn_fwd_tc.cu): one persistent CTA per SM
// (at most ctx.num_sms CTAs), same arguments and results within rounding.
cudaError_t launch_attn_fwd_tc(const void* q, const void* k, const void* v, const int32_t* pool_idx, int64_t q_begin,
                               int64_t q_end, int topk, float scale, void* o, float* lse, const LaunchCtx& ctx,
                               const SeqTable* tab = nullptr);

// Its profile build's per-CTA role counters (-1 in the default build).
int fwd_tc_profile_read(unsigned long long* out, int ctas);

// Delta for nq query rows, and zeroing of the two fp32 accumulators (skipped when dk_acc is null).
cudaError_t launch_attn_bwd_pre(const void* dO, const void* o, int64_t nq, int64_t S, float* delta, float* dk_acc,
                                float* dv_acc, const LaunchCtx& ctx);
// dq for queries [q_begin, q_end); dK/dV added into dk_acc/dv_acc unless they
// are null (dq only).  A table works as for launch_attn_fwd (dk_acc and dv_acc
// then span the packed batch).
cudaError_t launch_attn_bwd(const void* dO, const void* q, const void* k, const void* v, const float* lse,
                            const float* delta, const int32_t* pool_idx, int64_t q_begin, int64_t q_end, int topk,
                            float scale, void* dq, float* dk_acc, float* dv_acc, const LaunchCtx& ctx,
                            const SeqTable* tab = nullptr);
// Deterministic dK/dV (attn_bwd_det.cu): sizes of the pieces of its workspace.
struct DetPlan {
  int64_t P;         // pools that can be selected: floor(S/4)
  int64_t nP;        // pools with keys: ceil(S/4)
  int qb;            // queries per counting block
  int nb;            // counting blocks
  int G;             // counting blocks per span (one launch each)
  int nspan;         // spans
  int64_t cnt_n;     // P * nb counters
  int64_t bsum_n;    // scan tile totals
};
struct DetBuffers {
  int32_t* nsel;     // [S]
  uint32_t* cnt;     // [cnt_n] counts, then offsets, then cell ends
  uint32_t* bsum;    // [bsum_n]
  int32_t* qlist;    // [S * topk]
  uint32_t* tickets; // [nspan]
  float* dk_acc;     // [S][128] fp32, zero before the first span
  float* dv_acc;     // [S][128]
};
DetPlan det_plan(int64_t S, int topk);
// largest array the two-level scan handles
int64_t det_scan_max_elems();
// 1. per-(pool, counting block) lists of selecting queries, ascending
cudaError_t launch_det_lists(const int32_t* pool_idx, int64_t S, int topk, const DetPlan& d, const DetBuffers& w,
                             const LaunchCtx& ctx);
int det_lists_kernels(const DetPlan& d);  // kernels launch_det_lists launches
// 2. span sp (spans in ascending order): every pool's dK/dV rows += the span's queries' contributions
cudaError_t launch_det_span(const void* dO, const void* q, const void* k, const void* v, const float* lse,
                            const float* delta, int64_t S, float scale, const DetPlan& d, const DetBuffers& w, int sp,
                            const LaunchCtx& ctx);

cudaError_t launch_cast_dkdv(const float* dk_acc, const float* dv_acc, int64_t n, void* dk, void* dv,
                             const LaunchCtx& ctx);

}  // namespace dsa
