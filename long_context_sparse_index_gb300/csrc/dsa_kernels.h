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

struct LaunchCtx {
  cudaStream_t stream;
  unsigned* status;        // device status word (kStatus* bits)
  uint64_t wait_limit_ns;  // bound on every device-side spin-wait
  int inject_timeout;      // fault injection: producers issue no copies, so waits run out
  int num_sms;
  int pdl;                 // launch may start early (programmatic stream serialization)
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
// of its workspace, and its most score buffers.
constexpr int kIndexSyncWords = 24;
constexpr int kMaxBufs = 8;
// word counting the rows whose top-k took the general (full-row) path; it
// survives the call (the next call's key pooling zeroes it)
constexpr int kIndexGeneralRowsWord = 20;

// Pooled indexer keys: khat2 [P, 128] bf16, hi in columns 0..63, lo in 64..127.
// Also zeroes the kIndexSyncWords words at sync_words (always launch it, even
// with P == 0, before launch_index_topk).
cudaError_t launch_pool_keys(const void* k_idx, int64_t P, void* khat2, unsigned long long* sync_words,
                             const LaunchCtx& ctx);

// Indexer scores and per-row top-k for query rows [q_begin, q_end), in query
// chunks of `chunk` rows, as one persistent cooperative kernel (one CTA per
// SM).  scores holds nbuf chunk buffers (`chunk` rows x ld floats each,
// buf_stride floats apart; chunk c uses buffer c % nbuf); pool_idx row r is
// query q_begin + r.
cudaError_t launch_index_topk(const CUtensorMap& q_map, const CUtensorMap& khat_map, const float* w, float* scores,
                              int64_t ld, int64_t buf_stride, int nbuf, int64_t q_begin, int64_t q_end, int chunk,
                              int Hi, int topk, int32_t* pool_idx, unsigned long long* sync_words,
                              const LaunchCtx& ctx);
size_t index_topk_smem_bytes();

// Queries [q_begin, q_end) (global positions); q, pool_idx, o and lse hold
// their rows locally (row r = query q_begin + r); k and v are the whole sequence.
cudaError_t launch_attn_fwd(const void* q, const void* k, const void* v, const int32_t* pool_idx, int64_t q_begin,
                            int64_t q_end, int topk, float scale, void* o, float* lse, const LaunchCtx& ctx);

// Delta for nq query rows, and zeroing of the two fp32 accumulators (skipped when dk_acc is null).
cudaError_t launch_attn_bwd_pre(const void* dO, const void* o, int64_t nq, int64_t S, float* delta, float* dk_acc,
                                float* dv_acc, const LaunchCtx& ctx);
// dq for queries [q_begin, q_end); dK/dV added into dk_acc/dv_acc unless they are null (dq only).
cudaError_t launch_attn_bwd(const void* dO, const void* q, const void* k, const void* v, const float* lse,
                            const float* delta, const int32_t* pool_idx, int64_t q_begin, int64_t q_end, int topk,
                            float scale, void* dq, float* dk_acc, float* dv_acc, const LaunchCtx& ctx);
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
