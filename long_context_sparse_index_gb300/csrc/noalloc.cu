// noalloc.cu -- dsa_index_topk_noalloc: the indexer + top-k entry point for
// callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocating
// routine) at the point where they need the indexer: for example a host
// runtime that owns a fixed device-memory budget and must not let a library
// grow it, or a latency-critical path that must not block on the device
// allocator.  For them this file keeps the scratch the call needs in a
// file-scope static device array of fixed size, kNoAllocScratchBytes.  The
// caller still passes its own inputs and outputs.
//
// When the array is reserved: this file is its own CUDA module, and under
// the runtime's default lazy module loading a device reserves the array when
// the module is first loaded on it -- during the first call on that device
// (the address lookup below loads it).  From then on the device holds the
// array until the process exits.  So the first call on each device belongs
// outside any region that must not allocate, and before any stream capture.
//
// Set-up: that first call on each device looks up the device's address of
// the array with cudaGetSymbolAddress (with that device current) and caches
// it under the current context's id; a later call in a new context (after a
// device reset, say) looks it up again.  In host code the array's name is
// only a stand-in, never a device address, so kernels are always given the
// looked-up address.
//
// Every call on a device shares the same array, and the array keeps whatever
// the previous call left in it.  Nothing in it needs to start at zero: each
// call rebuilds the pooled keys and rewrites every score it reads before
// reading it, and the kernel's global words are zeroed by the call's first
// kernel.  Two calls whose work overlaps on the GPU (different streams
// without ordering between them) race on the array and must not be issued.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/dsa.h"
#include "dsa_kernels.h"

namespace dsa {
void set_last_error(const std::string& msg);  // dsa_api.cu: the message dsa_last_error() returns
size_t index_topk_min_workspace(int64_t S, int chunk, int topk);  // dsa_api.cu: the least workspace dsa_index_topk accepts
unsigned long long current_context_id();  // dsa_api.cu: id of the current CUDA context (0: none)
}

namespace {

// 32 MiB.  The call runs the sizes whose least workspace (the one
// dsa_index_topk accepts at the minimum, two chunk slots) fits: every
// S <= 32768 with chunk <= 256 and topk <= 512, for example (at most ~30.2
// MiB: kernel words, pooled keys as bf16 hi/lo and fp32, the fallback rows'
// list and scratch, and two slots of sampled scores, thresholds and candidate
// lists).  It always hands dsa_index_topk the whole array, so at the largest
// sizes only two chunks are in flight (slower than dsa_index_topk with its
// recommended workspace; the result is the same).
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};  // context each address was looked up in

}  // namespace

extern "C" {

dsa_status_t dsa_index_topk_noalloc(const void* q_idx, const void* k_idx, const float* w, int64_t S, int Hi, int Di,
                                    int chunk, int topk, int64_t q_begin, int64_t q_end, int32_t* pool_idx,
                                    void* stream) {
  const dsa::CallScope scope("dsa_index_topk_noalloc");
  const size_t need = dsa_index_topk_workspace(S, Hi, Di, chunk, topk) == 0 ? 0 : dsa::index_topk_min_workspace(S, chunk, topk);
  if (need == 0) {
    // invalid sizes: let the regular entry point report the precise reason
    return dsa_index_topk(q_idx, k_idx, w, S, Hi, Di, chunk, topk, q_begin, q_end, pool_idx, nullptr, 0, stream);
  }
  if (need > kNoAllocScratchBytes) {
    dsa::set_last_error("dsa_index_topk_noalloc: these sizes need " + std::to_string(need) +
                        " bytes of scratch but the built-in buffer holds " + std::to_string(kNoAllocScratchBytes) +
                        " (enough for S <= 32768 with chunk <= 256 and topk <= 512, for example); use "
                        "dsa_index_topk with a caller workspace");
    return DSA_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    dsa::set_last_error(std::string("dsa_index_topk_noalloc: no usable current device: ") + cudaGetErrorString(e));
    return DSA_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const unsigned long long ctx = dsa::current_context_id();
    if (g_scratch_ptr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        dsa::set_last_error(std::string("dsa_index_topk_noalloc: cudaGetSymbolAddress failed: ") +
                            cudaGetErrorString(e));
        return DSA_ERR_CUDA;
      }
      g_scratch_ptr[dev] = p;
      g_scratch_ctx[dev] = dsa::current_context_id();  // the lookup made a context current if none was
    }
    scratch = g_scratch_ptr[dev];
  }
  return dsa_index_topk(q_idx, k_idx, w, S, Hi, Di, chunk, topk, q_begin, q_end, pool_idx, scratch,
                        kNoAllocScratchBytes, stream);
}

}  // extern "C"
