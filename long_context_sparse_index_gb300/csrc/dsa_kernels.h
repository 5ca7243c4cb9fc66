// dsa_kernels.h -- host-side launchers of the libdsa kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

namespace dsa {

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

cudaError_t launch_attn_bwd_pre(const void* dO, const void* o, int64_t nq, int64_t S, float* delta, float* dk_acc,
                                float* dv_acc, const LaunchCtx& ctx);
cudaError_t launch_attn_bwd(const void* dO, const void* q, const void* k, const void* v, const float* lse,
                            const float* delta, const int32_t* pool_idx, int64_t q_begin, int64_t q_end, int topk,
                            float scale, void* dq, float* dk_acc, float* dv_acc, const LaunchCtx& ctx);
cudaError_t launch_cast_dkdv(const float* dk_acc, const float* dv_acc, int64_t n, void* dk, void* dv,
                             const LaunchCtx& ctx);

}  // namespace dsa
