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

// Pooled indexer keys: khat2 [P, 128] bf16, hi in columns 0..63, lo in 64..127.
cudaError_t launch_pool_keys(const void* k_idx, int64_t P, void* khat2, const LaunchCtx& ctx);

// Scores of query rows [row0, row0 + nrows) against pools [0, floor((row0+nrows-1)/4)),
// as nsplit partial sums over equal head ranges: slice s holds
// scores[s * split_stride + (i - row0) * ld + p]; entries p >= floor(i/4) are
// not meaningful.
cudaError_t launch_indexer(const CUtensorMap& q_map, const CUtensorMap& khat_map, const float* w, float* scores,
                           int64_t ld, int nsplit, int64_t split_stride, int64_t row0, int nrows, int Hi,
                           const LaunchCtx& ctx);
size_t indexer_smem_bytes();

// Per-row top-k of the scores written by launch_indexer (the nsplit slices
// added in slice order); out rows are pool_idx rows for queries row0 .. row0 + nrows - 1.
cudaError_t launch_topk(const float* scores, int64_t ld, int nsplit, int64_t split_stride, int64_t row0, int nrows,
                        int topk, int32_t* out, const LaunchCtx& ctx);

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
