// dsa_api.cu -- the C ABI of libdsa (declared in include/dsa.h): argument
// checks, workspace carving, TMA descriptors and the query-chunk loop.
//
// [SkyRL-1M §1 DSA 真稀疏; Anyscale, second lesson (the indexer)] the indexer
// scores one chunk of queries at a time, so its scratch is a ring of at most
// eight chunks of scores (chunk x pools x 4 B each; two at the least) rather
// than the whole S x S/4 matrix.
// [Anyscale, the lesson on checking that every layer runs the kernel one
// expects] a shape the kernels do not implement is an error, never a silent
// fallback; dsa_last_kernel_config reports what each call launched.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/dsa.h"
#include "dsa_device.cuh"
#include "dsa_kernels.h"

namespace dsa {
// Unique id of the calling thread's current CUDA context, or 0 when there is
// none (or the driver cannot say).  Device addresses looked up in a context
// are cached under its id.
unsigned long long current_context_id();
}  // namespace dsa

namespace {

__device__ unsigned int g_dsa_status;

thread_local std::string g_last_error;

// The record of the outermost entry point in progress (or last finished) on
// this host thread: its name, the kernels it launched (consecutive launches of
// one kernel counted together), its plan parameters and its variant.
struct KernelRecord {
  std::string entry;
  std::string variant;
  std::vector<std::pair<std::string, long long>> kernels;
  std::vector<std::pair<std::string, long long>> params;
};
thread_local KernelRecord g_record;
thread_local int g_call_depth = 0;

constexpr int kMaxDevices = 64;
constexpr int kDi = 64;
constexpr int kHq = 16;
constexpr int kD = 128;
constexpr int kMaxTopk = 2048;
constexpr int kMaxHi = 64;
constexpr int64_t kPoolTile = 256;
constexpr size_t kSyncBytes = 512;  // the fused kernel's global words, first in the index workspace
static_assert(dsa::kIndexSyncWords * 8 <= kSyncBytes, "sync words");

dsa_status_t fail(dsa_status_t st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
dsa_status_t fail(dsa_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

dsa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// fp32 / int32 tensors the kernels only access element by element
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// packed batches: up to this many of the shorter long sequences are indexed
// at once, each on a helper stream of its own
constexpr int kVarlenStreams = 4;

struct DeviceInfo {
  int num_sms = 0;
  unsigned* status = nullptr;
  unsigned long long ctx = 0;  // context the status address was looked up in
  cudaStream_t helpers[kVarlenStreams] = {};
  unsigned long long helpers_ctx = 0;  // context the helper streams were created in (0: none yet)
};

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

dsa_status_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  // a device reset replaces the context, and with it the module that holds
  // the status word: look its address up again in the new context
  const unsigned long long ctx = dsa::current_context_id();
  if (d.num_sms != 0 && (ctx == 0 || ctx != d.ctx)) d.num_sms = 0;
  if (d.num_sms == 0) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
      return fail(DSA_ERR_UNSUPPORTED, "libdsa is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dsa_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    d.status = static_cast<unsigned*>(p);
    d.num_sms = sms;
    d.ctx = dsa::current_context_id();  // the lookup made the context current if it was not
  }
  *out = d;
  return DSA_OK;
}

// The current device's helper streams for packed batches, created on first
// use in the current context (non-blocking: ordered only by the events the
// caller records).
static dsa_status_t varlen_streams(cudaStream_t (&out)[kVarlenStreams]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  const unsigned long long ctx = dsa::current_context_id();
  if (d.helpers_ctx == 0 || ctx != d.helpers_ctx) {
    for (int k = 0; k < kVarlenStreams; ++k) {
      e = cudaStreamCreateWithFlags(&d.helpers[k], cudaStreamNonBlocking);
      if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithFlags");
    }
    d.helpers_ctx = ctx;
  }
  for (int k = 0; k < kVarlenStreams; ++k) out[k] = d.helpers[k];
  return DSA_OK;
}

dsa_status_t make_ctx(void* stream, dsa::LaunchCtx* ctx) {
  DeviceInfo d;
  dsa_status_t st = device_info(&d);
  if (st != DSA_OK) return st;
  ctx->stream = static_cast<cudaStream_t>(stream);
  ctx->status = d.status;
  ctx->num_sms = d.num_sms;
  // every device-side spin-wait gives up after this long (default 2 s)
  double ms = 2000.0;
  if (const char* s = getenv("DSA_WAIT_LIMIT_MS")) ms = atof(s);
  ctx->inject_timeout = 0;
  if (const char* s = getenv("DSA_FAULT_INJECT")) {
    if (strcmp(s, "timeout") == 0) {
      ctx->inject_timeout = 1;
      ms = 1.0;
    }
  }
  ctx->wait_limit_ns = static_cast<uint64_t>(ms * 1e6);
  ctx->pdl = 0;
  ctx->persistent_ctas = 0;
  return DSA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// ---------------------------------------------------------------- item trace (measurement build)
#ifdef DSA_ITEM_TRACE
std::mutex g_trace_mu;
void* g_trace_buf = nullptr;
size_t g_trace_bytes = 0;
#endif

// ---------------------------------------------------------------- launch accounting
std::atomic<int64_t> g_launches{0};
std::atomic<int> g_profiling{0};
std::mutex g_prof_mu;
struct ProfRec {
  const char* name;
  cudaEvent_t start, stop;
};
std::vector<ProfRec> g_prof;

// Runs one launcher, counting its kernels (one unless the caller says how
// many it launched) and, when profiling is on, bracketing it with events on
// the launch stream.
template <typename F>
cudaError_t timed_launch(const char* name, cudaStream_t stream, F&& launch, int kernels = 1) {
  const bool prof = g_profiling.load(std::memory_order_relaxed) != 0;
  ProfRec rec{name, nullptr, nullptr};
  if (prof) {
    cudaEventCreate(&rec.start);
    cudaEventCreate(&rec.stop);
    cudaEventRecord(rec.start, stream);
  }
  cudaError_t e = launch();
  if (e == cudaSuccess) {
    g_launches.fetch_add(kernels, std::memory_order_relaxed);
    auto& ks = g_record.kernels;
    if (!ks.empty() && ks.back().first == name) ks.back().second += kernels;
    else ks.emplace_back(name, kernels);
  }
  if (prof) {
    cudaEventRecord(rec.stop, stream);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.push_back(rec);
  }
  return e;
}

// The index workspace: kernel words, pooled keys (bf16 hi/lo and fp32), the
// fallback kernel's row list and scratch rows, then a ring of per-chunk slots
// (sampled scores, thresholds, candidate counts and candidate lists), at least
// min(2, chunks) and at most dsa::kMaxBufs.  The slot count only changes how
// many chunks are in flight, never the result.
int index_max_bufs(int64_t S, int chunk) {
  const int64_t nchunks = (S + chunk - 1) / chunk;
  return static_cast<int>(nchunks < dsa::kMaxBufs ? nchunks : dsa::kMaxBufs);
}
int index_min_bufs(int64_t S, int chunk) { return index_max_bufs(S, chunk) < 2 ? index_max_bufs(S, chunk) : 2; }

int64_t pow2_ceil(int64_t x) {
  int64_t p = 1;
  while (p < x) p <<= 1;
  return p;
}
int64_t pow2_floor(int64_t x) {
  int64_t p = 1;
  while (2 * p <= x) p <<= 1;
  return p;
}

constexpr int kCandBase = 4096;  // rows with at most this many pools keep every pool as a candidate
constexpr int kFallbackCtas = 64;

// Sampling and candidate sizes.  sigma: every sigma-th pool is sampled, with
// at least 16 samples expected above a row's k-th largest score (sigma <=
// topk/16) and at most kCandBase samples per row.  A threshold at the rsel-th
// largest sample leaves about c = rsel * sigma pools at or above it; c is
// chosen so that c - 4 sqrt(sigma c) = topk (fewer than topk candidates is a
// four-sigma event of the sampling), and cap holds c + 4 sqrt(sigma c).
dsa::IndexPlan index_plan(int64_t S, int chunk, int topk) {
  dsa::IndexPlan pl;
  pl.P = S / 4;
  pl.Ppad = ((pl.P + kPoolTile - 1) / kPoolTile) * kPoolTile + (pl.P == 0 ? kPoolTile : 0);
  const int64_t sig_min = pow2_floor(topk / 16 > 1 ? topk / 16 : 1);
  const int64_t sig_p = pow2_ceil((pl.P + kCandBase - 1) / kCandBase);
  pl.sigma = static_cast<int>(sig_min > sig_p ? sig_min : sig_p);
  const double sg = pl.sigma;
  const double rc = 2.0 * std::sqrt(sg) + std::sqrt(4.0 * sg + topk);
  const double c = rc * rc;
  pl.rsel = static_cast<int>(std::ceil(c / sg));
  const int64_t hold = pow2_ceil(static_cast<int64_t>(std::ceil(c + 4.0 * std::sqrt(sg * c))));
  pl.cap = static_cast<int>(hold > kCandBase ? hold : kCandBase);
  const int64_t G = (pl.P + pl.sigma - 1) / pl.sigma;
  pl.samp_ld = ((G + kPoolTile - 1) / kPoolTile) * kPoolTile + (G == 0 ? kPoolTile : 0);
  pl.slot_rows = chunk < S ? chunk : S;
  pl.thr_ld = (pl.slot_rows + 127) / 128 * 128;
  pl.samp_slot = pl.slot_rows * pl.samp_ld;
  pl.cand_slot = pl.slot_rows * pl.cap;
  pl.fb_ctas = kFallbackCtas;
  pl.fb_ld = pl.Ppad;
  return pl;
}

struct IndexLayout {
  size_t khat2, khat32, fb_rows, fb_scratch, samples, thr, cnt, cands, total;
};

IndexLayout index_layout(int64_t S, const dsa::IndexPlan& pl, int nbuf) {
  IndexLayout L;
  const size_t P1 = static_cast<size_t>(pl.P > 0 ? pl.P : 1);
  size_t off = kSyncBytes;
  L.khat2 = off;
  off += round_up(P1 * 2 * kDi * 2, 256);
  L.khat32 = off;
  off += round_up(P1 * kDi * 4, 256);
  L.fb_rows = off;
  off += round_up(static_cast<size_t>(S) * 4, 256);
  L.fb_scratch = off;
  off += round_up(static_cast<size_t>(pl.fb_ctas) * pl.fb_ld * 4, 256);
  L.samples = off;
  off += round_up(static_cast<size_t>(nbuf) * pl.samp_slot * 4, 256);
  L.thr = off;
  off += round_up(static_cast<size_t>(nbuf) * pl.thr_ld * 8, 256);
  L.cnt = off;
  off += round_up(static_cast<size_t>(nbuf) * pl.thr_ld * 4, 256);
  L.cands = off;
  off += round_up(static_cast<size_t>(nbuf) * pl.cand_slot * 8, 256);
  L.total = off;
  return L;
}

size_t index_ws_bytes(int64_t S, int chunk, int topk, int nbuf) {
  return index_layout(S, index_plan(S, chunk, topk), nbuf).total;
}

}  // namespace

namespace dsa {
void set_last_error(const std::string& msg) { g_last_error = msg; }

void call_begin(const char* fn) {
  nvtxRangePushA(fn);
  if (g_call_depth++ == 0) {
    g_record = KernelRecord{};
    g_record.entry = fn;
  }
}
void call_end() {
  --g_call_depth;
  nvtxRangePop();
}
void call_param(const char* key, long long value) {
  for (auto& kv : g_record.params)
    if (kv.first == key) {
      kv.second = value;
      return;
    }
  g_record.params.emplace_back(key, value);
}
void call_variant(const char* variant) { g_record.variant = variant; }

unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}
size_t index_topk_min_workspace(int64_t S, int chunk, int topk) {
  if (S < 1 || chunk < 1 || topk < 1) return 0;
  return index_ws_bytes(S, chunk, topk, index_min_bufs(S, chunk));
}
}  // namespace dsa

extern "C" {

const char* dsa_last_error(void) { return g_last_error.c_str(); }

int dsa_last_kernel_config(char* buf, size_t len) {
  std::string s = "{\"entry\": \"" + g_record.entry + "\", \"variant\": \"" + g_record.variant + "\", \"kernels\": [";
  for (size_t j = 0; j < g_record.kernels.size(); ++j)
    s += (j ? ", [\"" : "[\"") + g_record.kernels[j].first + "\", " + std::to_string(g_record.kernels[j].second) + "]";
  s += "], \"params\": {";
  for (size_t j = 0; j < g_record.params.size(); ++j)
    s += (j ? ", \"" : "\"") + g_record.params[j].first + "\": " + std::to_string(g_record.params[j].second);
  s += "}}";
  if (buf && len > 0) {
    const size_t n = s.size() < len - 1 ? s.size() : len - 1;
    std::memcpy(buf, s.data(), n);
    buf[n] = '\0';
  }
  return static_cast<int>(s.size());
}

const char* dsa_version(void) { return "libdsa 0.1.0 (sm_103a)"; }

size_t dsa_index_topk_workspace(int64_t S, int Hi, int Di, int chunk, int topk) {
  if (S < 1 || Hi < 1 || Di < 1 || chunk < 1 || topk < 1) return 0;
  return index_ws_bytes(S, chunk, topk, index_max_bufs(S, chunk));
}

size_t dsa_index_topk_workspace_slots(int64_t S, int Hi, int Di, int chunk, int topk, int slots) {
  if (S < 1 || Hi < 1 || Di < 1 || chunk < 1 || topk < 1 || slots < 1 || slots > index_max_bufs(S, chunk)) return 0;
  return index_ws_bytes(S, chunk, topk, slots);
}

// The indexer call once its arguments are checked: plan, workspace carving,
// tensor maps and the launches, on ctx.stream (the packed-batch path calls it
// for each long sequence, on its own streams and grids).
static dsa_status_t index_topk_run(const void* q_idx, const void* k_idx, const float* w, int64_t S, int Hi,
                                   int chunk, int topk, int64_t q_begin, int64_t q_end, int32_t* pool_idx,
                                   void* workspace, size_t ws_bytes, const dsa::LaunchCtx& ctx) {
  const dsa::IndexPlan pl = index_plan(S, chunk, topk);
  const int64_t P = pl.P;
  int nbuf = index_min_bufs(S, chunk);  // as many chunk slots as the workspace holds
  while (nbuf < index_max_bufs(S, chunk) && index_layout(S, pl, nbuf + 1).total <= ws_bytes) ++nbuf;
  const IndexLayout L = index_layout(S, pl, nbuf);
  dsa::call_param("S", S);
  dsa::call_param("q_begin", q_begin);
  dsa::call_param("q_end", q_end);
  dsa::call_param("Hi", Hi);
  dsa::call_param("topk", topk);
  dsa::call_param("chunk", chunk);
  dsa::call_param("chunk_slots", nbuf);
  dsa::call_param("sample_stride", pl.sigma);
  dsa::call_param("threshold_rank", pl.rsel);
  dsa::call_param("candidates_per_row", pl.cap);
  dsa::call_variant("persistent indexer + top-k (bf16 hi/lo pooled keys), fallback rows recomputed");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  dsa::IndexBuffers b;
  b.sync = reinterpret_cast<unsigned long long*>(ws);
  b.khat2 = ws + L.khat2;
  b.khat32 = reinterpret_cast<float*>(ws + L.khat32);
  b.fb_rows = reinterpret_cast<int32_t*>(ws + L.fb_rows);
  b.fb_scratch = reinterpret_cast<float*>(ws + L.fb_scratch);
  b.samples = reinterpret_cast<float*>(ws + L.samples);
  b.thr = reinterpret_cast<uint2*>(ws + L.thr);
  b.cnt = reinterpret_cast<unsigned*>(ws + L.cnt);
  b.cands = reinterpret_cast<uint2*>(ws + L.cands);
  b.nbuf = nbuf;
  b.trace = nullptr;
  b.trace_count = nullptr;
  b.trace_cap = 0;
#ifdef DSA_ITEM_TRACE
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (g_trace_buf != nullptr) {
      b.trace_count = static_cast<unsigned long long*>(g_trace_buf);
      b.trace = reinterpret_cast<dsa::IndexTraceRec*>(static_cast<uint8_t*>(g_trace_buf) + 64);
      b.trace_cap = static_cast<int64_t>((g_trace_bytes - 64) / sizeof(dsa::IndexTraceRec));
    }
  }
#endif

  CUtensorMap q_map, k_map, s_map;
  memset(&q_map, 0, sizeof(q_map));
  memset(&k_map, 0, sizeof(k_map));
  memset(&s_map, 0, sizeof(s_map));
  const bool need_indexer = (q_end - 1) / 4 > topk;  // some row has more eligible pools than topk
  if (need_indexer) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return fail(DSA_ERR_CUDA, "dsa_index_topk: cuTensorMapEncodeTiled unavailable from the driver");
    {
      cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDi), static_cast<cuuint64_t>(Hi), static_cast<cuuint64_t>(S)};
      cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDi) * 2, static_cast<cuuint64_t>(Hi) * kDi * 2};
      cuuint32_t box[3] = {static_cast<cuuint32_t>(kDi), 1u, 128u};
      cuuint32_t estr[3] = {1u, 1u, 1u};
      CUresult r = enc(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q_idx), dims, strides, box,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "dsa_index_topk: q_idx tensor map (CUresult %d)", (int)r);
    }
    {
      cuuint64_t dims[2] = {static_cast<cuuint64_t>(2 * kDi), static_cast<cuuint64_t>(P)};
      cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * kDi) * 2};
      cuuint32_t box[2] = {static_cast<cuuint32_t>(kDi), static_cast<cuuint32_t>(kPoolTile)};
      cuuint32_t estr[2] = {1u, 1u};
      CUresult r = enc(&k_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, b.khat2, dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "dsa_index_topk: pooled-key tensor map (CUresult %d)", (int)r);
    }
    {
      // every sigma-th pooled key: row g of this map is pool g * sigma
      const int64_t G = (P + pl.sigma - 1) / pl.sigma;
      cuuint64_t dims[2] = {static_cast<cuuint64_t>(2 * kDi), static_cast<cuuint64_t>(G)};
      cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * kDi) * 2 * static_cast<cuuint64_t>(pl.sigma)};
      cuuint32_t box[2] = {static_cast<cuuint32_t>(kDi), static_cast<cuuint32_t>(kPoolTile)};
      cuuint32_t estr[2] = {1u, 1u};
      CUresult r = enc(&s_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, b.khat2, dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "dsa_index_topk: sampled-key tensor map (CUresult %d)", (int)r);
    }
  }
  // pool_keys also zeroes the fused kernel's global words, so it always runs
  cudaError_t e = timed_launch("pool_keys", ctx.stream, [&] {
    return dsa::launch_pool_keys(k_idx, P, b.khat2, b.khat32, b.sync, ctx);
  });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_index_topk: pool_keys launch");
  // one persistent kernel walks every chunk: samples, thresholds, indexer
  // tiles and top-k rows (when no row has more than topk pools there are only
  // rows, and no tensor map is read); then the rows it could not certify
  e = timed_launch("index_topk", ctx.stream, [&] {
    return dsa::launch_index_topk(q_map, k_map, s_map, pl, b, w, q_begin, q_end, chunk, Hi, topk, pool_idx, ctx);
  });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_index_topk: index_topk launch");
  if (need_indexer) {
    e = timed_launch("index_fallback", ctx.stream, [&] {
      return dsa::launch_index_fallback(q_idx, pl, b, w, q_begin, Hi, topk, pool_idx, ctx);
    });
    if (e != cudaSuccess) return cuda_fail(e, "dsa_index_topk: index_fallback launch");
  }
  return DSA_OK;
}

dsa_status_t dsa_index_topk(const void* q_idx, const void* k_idx, const float* w, int64_t S, int Hi, int Di,
                            int chunk, int topk, int64_t q_begin, int64_t q_end, int32_t* pool_idx,
                            void* workspace, size_t ws_bytes, void* stream) {
  const dsa::CallScope scope("dsa_index_topk");
  if (!q_idx || !k_idx || !w || !pool_idx) return fail(DSA_ERR_INVALID_ARG, "dsa_index_topk: null tensor pointer");
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned4(w) || !aligned4(pool_idx))
    return fail(DSA_ERR_INVALID_ARG,
                "dsa_index_topk: q_idx and k_idx must be 16-byte aligned, w and pool_idx 4-byte aligned");
  if (S < 1 || S > 0x7FFFFFFFLL) return fail(DSA_ERR_INVALID_ARG, "dsa_index_topk: S=%lld out of range", (long long)S);
  if (chunk < 1) return fail(DSA_ERR_INVALID_ARG, "dsa_index_topk: chunk=%d must be >= 1", chunk);
  if (topk < 1) return fail(DSA_ERR_INVALID_ARG, "dsa_index_topk: topk=%d must be >= 1", topk);
  if (Hi < 1) return fail(DSA_ERR_INVALID_ARG, "dsa_index_topk: Hi=%d must be >= 1", Hi);
  if (q_begin < 0 || q_end > S || q_begin >= q_end)
    return fail(DSA_ERR_INVALID_ARG, "dsa_index_topk: query range [%lld, %lld) not inside [0, %lld)",
                (long long)q_begin, (long long)q_end, (long long)S);
  if (Di != kDi) return fail(DSA_ERR_UNSUPPORTED, "dsa_index_topk: Di=%d unsupported (kernels implement Di=64)", Di);
  if (Hi > kMaxHi) return fail(DSA_ERR_UNSUPPORTED, "dsa_index_topk: Hi=%d unsupported (max %d)", Hi, kMaxHi);
  if (topk > kMaxTopk) return fail(DSA_ERR_UNSUPPORTED, "dsa_index_topk: topk=%d unsupported (max %d)", topk, kMaxTopk);
  const size_t need = index_ws_bytes(S, chunk, topk, index_min_bufs(S, chunk));
  if (!workspace || ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "dsa_index_topk: workspace of at least %zu bytes needed (%zu recommended), %zu given",
                need, dsa_index_topk_workspace(S, Hi, Di, chunk, topk), workspace ? ws_bytes : (size_t)0);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DSA_ERR_INVALID_ARG, "dsa_index_topk: workspace must be 256-byte aligned");

  dsa::LaunchCtx ctx;
  dsa_status_t st = make_ctx(stream, &ctx);
  if (st != DSA_OK) return st;

  return index_topk_run(q_idx, k_idx, w, S, Hi, chunk, topk, q_begin, q_end, pool_idx, workspace, ws_bytes, ctx);
}

static dsa_status_t check_attn_args(const char* fn, int64_t S, int Hq, int D, int topk) {
  if (S < 1 || S > 0x7FFFFFFFLL) return fail(DSA_ERR_INVALID_ARG, "%s: S=%lld out of range", fn, (long long)S);
  if (topk < 1) return fail(DSA_ERR_INVALID_ARG, "%s: topk=%d must be >= 1", fn, topk);
  if (Hq != kHq || D != kD)
    return fail(DSA_ERR_UNSUPPORTED, "%s: Hq=%d, D=%d unsupported (kernels implement Hq=16, D=128)", fn, Hq, D);
  if (topk > kMaxTopk) return fail(DSA_ERR_UNSUPPORTED, "%s: topk=%d unsupported (max %d)", fn, topk, kMaxTopk);
  return DSA_OK;
}

static dsa_status_t check_range(const char* fn, int64_t S, int64_t q_begin, int64_t q_end) {
  if (q_begin < 0 || q_end > S || q_begin >= q_end)
    return fail(DSA_ERR_INVALID_ARG, "%s: query range [%lld, %lld) not inside [0, %lld)", fn, (long long)q_begin,
                (long long)q_end, (long long)S);
  return DSA_OK;
}

dsa_status_t dsa_sparse_attn_fwd_range(const void* q, const void* k, const void* v, const int32_t* pool_idx,
                                       int64_t S, int64_t q_begin, int64_t q_end, int Hq, int D, int topk,
                                       float scale, void* o, float* lse, void* stream) {
  const dsa::CallScope scope("dsa_sparse_attn_fwd_range");
  if (!q || !k || !v || !pool_idx || !o || !lse)
    return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_attn_fwd: null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(pool_idx) || !aligned16(o) || !aligned4(lse))
    return fail(DSA_ERR_INVALID_ARG,
                "dsa_sparse_attn_fwd: bf16 tensors must be 16-byte aligned, pool_idx and lse 4-byte aligned");
  dsa_status_t st = check_attn_args("dsa_sparse_attn_fwd", S, Hq, D, topk);
  if (st != DSA_OK) return st;
  st = check_range("dsa_sparse_attn_fwd", S, q_begin, q_end);
  if (st != DSA_OK) return st;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(D));
  dsa::LaunchCtx ctx;
  st = make_ctx(stream, &ctx);
  if (st != DSA_OK) return st;
  dsa::call_param("S", S);
  dsa::call_param("q_begin", q_begin);
  dsa::call_param("q_end", q_end);
  dsa::call_param("topk", topk);
  dsa::call_variant("gather-bound forward: one CTA per query, cp.async key-pool gather, mma.sync, online softmax");
  cudaError_t e = timed_launch("attn_fwd", ctx.stream, [&] {
    return dsa::launch_attn_fwd(q, k, v, pool_idx, q_begin, q_end, topk, scale, o, lse, ctx);
  });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_fwd: launch");
  return DSA_OK;
}

dsa_status_t dsa_sparse_attn_fwd(const void* q, const void* k, const void* v, const int32_t* pool_idx, int64_t S,
                                 int Hq, int D, int topk, float scale, void* o, float* lse, void* stream) {
  const dsa::CallScope scope("dsa_sparse_attn_fwd");
  return dsa_sparse_attn_fwd_range(q, k, v, pool_idx, S, 0, S, Hq, D, topk, scale, o, lse, stream);
}

dsa_status_t dsa_sparse_attn_fwd_tc(const void* q, const void* k, const void* v, const int32_t* pool_idx, int64_t S,
                                    int Hq, int D, int topk, float scale, void* o, float* lse, void* stream) {
  const dsa::CallScope scope("dsa_sparse_attn_fwd_tc");
  const char* fn = "dsa_sparse_attn_fwd_tc";
  if (!q || !k || !v || !pool_idx || !o || !lse) return fail(DSA_ERR_INVALID_ARG, "%s: null tensor pointer", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(pool_idx) || !aligned16(o) || !aligned4(lse))
    return fail(DSA_ERR_INVALID_ARG, "%s: bf16 tensors must be 16-byte aligned, pool_idx and lse 4-byte aligned", fn);
  dsa_status_t st = check_attn_args(fn, S, Hq, D, topk);
  if (st != DSA_OK) return st;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(D));
  dsa::LaunchCtx ctx;
  st = make_ctx(stream, &ctx);
  if (st != DSA_OK) return st;
  dsa::call_param("S", S);
  dsa::call_param("topk", topk);
  dsa::call_variant("tcgen05 forward: persistent CTA per SM; cp.async producers, one MMA issuer, softmax warps");
  cudaError_t e = timed_launch("attn_fwd_tc", ctx.stream, [&] {
    return dsa::launch_attn_fwd_tc(q, k, v, pool_idx, 0, S, topk, scale, o, lse, ctx);
  });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_fwd_tc: launch");
  return DSA_OK;
}

size_t dsa_sparse_attn_bwd_workspace(int64_t S, int Hq, int D) {
  if (S < 1 || Hq < 1 || D < 1) return 0;
  return round_up(static_cast<size_t>(S) * D * sizeof(float), 256) * 2 +
         round_up(static_cast<size_t>(S) * Hq * sizeof(float), 256);
}

dsa_status_t dsa_sparse_attn_bwd_range(const void* dO, const void* q, const void* k, const void* v, const void* o,
                                       const float* lse, const int32_t* pool_idx, int64_t S, int64_t q_begin,
                                       int64_t q_end, int Hq, int D, int topk, float scale, void* dq, void* dk,
                                       void* dv, void* workspace, size_t ws_bytes, void* stream) {
  const dsa::CallScope scope("dsa_sparse_attn_bwd_range");
  if (!dO || !q || !k || !v || !o || !lse || !pool_idx || !dq || !dk || !dv)
    return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_attn_bwd: null tensor pointer");
  if (!aligned16(dO) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
      !aligned4(pool_idx) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(DSA_ERR_INVALID_ARG,
                "dsa_sparse_attn_bwd: bf16 tensors must be 16-byte aligned, pool_idx and lse 4-byte aligned");
  dsa_status_t st = check_attn_args("dsa_sparse_attn_bwd", S, Hq, D, topk);
  if (st != DSA_OK) return st;
  st = check_range("dsa_sparse_attn_bwd", S, q_begin, q_end);
  if (st != DSA_OK) return st;
  const size_t need = dsa_sparse_attn_bwd_workspace(S, Hq, D);
  if (!workspace || ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "dsa_sparse_attn_bwd: workspace of %zu bytes needed, %zu given", need,
                workspace ? ws_bytes : (size_t)0);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DSA_ERR_INVALID_ARG, "dsa_sparse_attn_bwd: workspace must be 256-byte aligned");
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(D));
  dsa::LaunchCtx ctx;
  st = make_ctx(stream, &ctx);
  if (st != DSA_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t acc_bytes = round_up(static_cast<size_t>(S) * D * sizeof(float), 256);
  float* dk_acc = reinterpret_cast<float*>(ws);
  float* dv_acc = reinterpret_cast<float*>(ws + acc_bytes);
  float* delta = reinterpret_cast<float*>(ws + 2 * acc_bytes);
  const int64_t nq = q_end - q_begin;
  dsa::call_param("S", S);
  dsa::call_param("q_begin", q_begin);
  dsa::call_param("q_end", q_end);
  dsa::call_param("topk", topk);
  dsa::call_variant("atomic: dq query-major, dK/dV fp32 red.v4 per (query, key), bf16 cast");
  // S * D floats is a multiple of 64, so acc_bytes == S * D * 4 and the accumulators are adjacent
  cudaError_t e = timed_launch("attn_bwd_pre", ctx.stream,
                               [&] { return dsa::launch_attn_bwd_pre(dO, o, nq, S, delta, dk_acc, dv_acc, ctx); });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd: preprocess launch");
  e = timed_launch("attn_bwd", ctx.stream, [&] {
    return dsa::launch_attn_bwd(dO, q, k, v, lse, delta, pool_idx, q_begin, q_end, topk, scale, dq, dk_acc, dv_acc,
                                ctx);
  });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd: launch");
  e = timed_launch("attn_bwd_cast", ctx.stream,
                   [&] { return dsa::launch_cast_dkdv(dk_acc, dv_acc, S * D, dk, dv, ctx); });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd: cast launch");
  return DSA_OK;
}

dsa_status_t dsa_sparse_attn_bwd(const void* dO, const void* q, const void* k, const void* v, const void* o,
                                 const float* lse, const int32_t* pool_idx, int64_t S, int Hq, int D, int topk,
                                 float scale, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                                 void* stream) {
  const dsa::CallScope scope("dsa_sparse_attn_bwd");
  return dsa_sparse_attn_bwd_range(dO, q, k, v, o, lse, pool_idx, S, 0, S, Hq, D, topk, scale, dq, dk, dv,
                                   workspace, ws_bytes, stream);
}

namespace {
// pieces of the deterministic backward's workspace, each 256-byte aligned;
// the two fp32 accumulators first and adjacent (the preprocess kernel zeroes
// them as one range)
struct DetLayout {
  size_t dk_acc, dv_acc, delta, nsel, cnt, bsum, qlist, tickets, total;
};
DetLayout det_layout(int64_t S, int Hq, int topk, const dsa::DetPlan& d) {
  DetLayout l;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += round_up(bytes, 256);
    return at;
  };
  l.dk_acc = take(static_cast<size_t>(S) * kD * sizeof(float));
  l.dv_acc = take(static_cast<size_t>(S) * kD * sizeof(float));
  l.delta = take(static_cast<size_t>(S) * Hq * sizeof(float));
  l.nsel = take(static_cast<size_t>(S) * sizeof(int32_t));
  l.cnt = take(static_cast<size_t>(d.cnt_n) * sizeof(uint32_t));
  l.bsum = take(static_cast<size_t>(d.bsum_n) * sizeof(uint32_t));
  l.qlist = take(static_cast<size_t>(S) * topk * sizeof(int32_t));
  l.tickets = take(static_cast<size_t>(d.nspan) * sizeof(uint32_t));
  l.total = off;
  return l;
}
// list positions are 32-bit
constexpr int64_t kDetMaxEntries = (int64_t{1} << 31) - 1;
}  // namespace

size_t dsa_sparse_attn_bwd_deterministic_workspace(int64_t S, int Hq, int D, int topk) {
  if (S < 1 || Hq != kHq || D != kD || topk < 1 || topk > kMaxTopk) return 0;
  if (S > kDetMaxEntries / topk) return 0;
  const dsa::DetPlan d = dsa::det_plan(S, topk);
  if (d.cnt_n > dsa::det_scan_max_elems()) return 0;
  return det_layout(S, Hq, topk, d).total;
}

dsa_status_t dsa_sparse_attn_bwd_deterministic(const void* dO, const void* q, const void* k, const void* v,
                                               const void* o, const float* lse, const int32_t* pool_idx, int64_t S,
                                               int Hq, int D, int topk, float scale, void* dq, void* dk, void* dv,
                                               void* workspace, size_t ws_bytes, void* stream) {
  const dsa::CallScope scope("dsa_sparse_attn_bwd_deterministic");
  const char* fn = "dsa_sparse_attn_bwd_deterministic";
  if (!dO || !q || !k || !v || !o || !lse || !pool_idx || !dq || !dk || !dv)
    return fail(DSA_ERR_INVALID_ARG, "%s: null tensor pointer", fn);
  if (!aligned16(dO) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
      !aligned4(pool_idx) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(DSA_ERR_INVALID_ARG, "%s: bf16 tensors must be 16-byte aligned, pool_idx and lse 4-byte aligned", fn);
  dsa_status_t st = check_attn_args(fn, S, Hq, D, topk);
  if (st != DSA_OK) return st;
  const size_t need = dsa_sparse_attn_bwd_deterministic_workspace(S, Hq, D, topk);
  if (need == 0)
    return fail(DSA_ERR_UNSUPPORTED,
                "%s: S = %lld with topk = %d is beyond its limits (S x topk < 2^31 list entries, S / 4 <= 2^26 "
                "pools)", fn, static_cast<long long>(S), topk);
  if (!workspace || ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                workspace ? ws_bytes : (size_t)0);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DSA_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", fn);
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(D));
  dsa::LaunchCtx ctx;
  st = make_ctx(stream, &ctx);
  if (st != DSA_OK) return st;
  const dsa::DetPlan d = dsa::det_plan(S, topk);
  const DetLayout l = det_layout(S, Hq, topk, d);
  dsa::call_param("S", S);
  dsa::call_param("topk", topk);
  dsa::call_param("spans", d.nspan);
  dsa::call_variant("deterministic: dq query-major, dK/dV key-major in fixed order");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* delta = reinterpret_cast<float*>(ws + l.delta);
  dsa::DetBuffers b;
  b.nsel = reinterpret_cast<int32_t*>(ws + l.nsel);
  b.cnt = reinterpret_cast<uint32_t*>(ws + l.cnt);
  b.bsum = reinterpret_cast<uint32_t*>(ws + l.bsum);
  b.qlist = reinterpret_cast<int32_t*>(ws + l.qlist);
  b.tickets = reinterpret_cast<uint32_t*>(ws + l.tickets);
  b.dk_acc = reinterpret_cast<float*>(ws + l.dk_acc);
  b.dv_acc = reinterpret_cast<float*>(ws + l.dv_acc);
  // Delta, and the accumulators zeroed (S * D floats is a multiple of 64, so they are adjacent)
  cudaError_t e = timed_launch("attn_bwd_pre", ctx.stream, [&] {
    return dsa::launch_attn_bwd_pre(dO, o, S, S, delta, b.dk_acc, b.dv_acc, ctx);
  });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd_deterministic: preprocess launch");
  e = timed_launch("attn_bwd", ctx.stream, [&] {
    return dsa::launch_attn_bwd(dO, q, k, v, lse, delta, pool_idx, 0, S, topk, scale, dq, nullptr, nullptr, ctx);
  });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd_deterministic: dq launch");
  e = timed_launch("det_lists", ctx.stream, [&] { return dsa::launch_det_lists(pool_idx, S, topk, d, b, ctx); },
                   dsa::det_lists_kernels(d));
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd_deterministic: list launch");
  for (int sp = 0; sp < d.nspan; ++sp) {
    e = timed_launch("det_span", ctx.stream,
                     [&] { return dsa::launch_det_span(dO, q, k, v, lse, delta, S, scale, d, b, sp, ctx); });
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd_deterministic: span launch");
  }
  e = timed_launch("attn_bwd_cast", ctx.stream,
                   [&] { return dsa::launch_cast_dkdv(b.dk_acc, b.dv_acc, S * D, dk, dv, ctx); });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd_deterministic: cast launch");
  return DSA_OK;
}

dsa_status_t dsa_zigzag_ranges(int64_t S, int world, int rank, int64_t* ranges) {
  if (!ranges) return fail(DSA_ERR_INVALID_ARG, "dsa_zigzag_ranges: null output");
  if (S < 1 || world < 1 || rank < 0 || rank >= world)
    return fail(DSA_ERR_INVALID_ARG, "dsa_zigzag_ranges: S=%lld, world=%d, rank=%d", (long long)S, world, rank);
  const int64_t nseg = 2 * static_cast<int64_t>(world);
  // segment j = [j*S/nseg, (j+1)*S/nseg): equal lengths when nseg divides S
  auto bound = [&](int64_t j) { return static_cast<int64_t>((static_cast<__int128>(j) * S) / nseg); };
  ranges[0] = bound(rank);
  ranges[1] = bound(rank + 1);
  ranges[2] = bound(nseg - 1 - rank);
  ranges[3] = bound(nseg - rank);
  return DSA_OK;
}

// ---------------------------------------------------------------- packed variable-length batches
// Each sequence of the batch is its own causal layer.  The attention calls
// cover the whole batch with one launch per kernel and per 256 sequences (a
// table of sequence starts rides in the launch's parameters); the indexer
// fills the rows of short sequences (every row keeps all its pools) in one
// launch per 256 of them and runs the persistent indexer once per longer
// sequence.

static dsa_status_t check_cu_seqlens(const char* fn, const int64_t* cu, int nseq) {
  if (!cu || nseq < 1) return fail(DSA_ERR_INVALID_ARG, "%s: need cu_seqlens and nseq >= 1", fn);
  if (cu[0] != 0) return fail(DSA_ERR_INVALID_ARG, "%s: cu_seqlens[0] must be 0", fn);
  for (int s = 0; s < nseq; ++s)
    if (cu[s + 1] <= cu[s])
      return fail(DSA_ERR_INVALID_ARG, "%s: cu_seqlens must be strictly increasing (sequence %d is empty)", fn, s);
  if (cu[nseq] > 0x7FFFFFFFLL)
    return fail(DSA_ERR_INVALID_ARG, "%s: packed length %lld out of range", fn, (long long)cu[nseq]);
  return DSA_OK;
}

static int64_t max_len(const int64_t* cu, int nseq) {
  int64_t m = 0;
  for (int s = 0; s < nseq; ++s) m = cu[s + 1] - cu[s] > m ? cu[s + 1] - cu[s] : m;
  return m;
}

// the table of sequences s0 .. s0+n-1
static dsa::SeqTable seq_table(const int64_t* cu, int s0, int n) {
  dsa::SeqTable t;
  t.n = n;
  t.row0 = cu[s0];
  for (int j = 0; j <= n; ++j) t.cu[j] = cu[s0 + j];
  return t;
}

// The indexer tiles (128 queries x 256 pools) of one sequence of L tokens.
static int64_t index_tiles(int64_t L) {
  int64_t t = 0;
  for (int64_t r0 = 0; r0 < L; r0 += 128) {
    const int64_t last = r0 + 127 < L - 1 ? r0 + 127 : L - 1;
    t += (last / 4 + 255) / 256;
  }
  return t;
}
// A long sequence with fewer tiles than this (two per SM of a GB300) leaves
// most SMs idle in its own launch: such sequences are indexed several at once.
constexpr int64_t kSmallSeqTiles = 304;

// The long sequences (more than 4 * topk + 4 tokens, so the indexer runs)
// with fewer than kSmallSeqTiles tiles.
static int small_long_seqs(const int64_t* cu, int nseq, int topk) {
  int n = 0;
  for (int s = 0; s < nseq; ++s) {
    const int64_t L = cu[s + 1] - cu[s];
    if (L > 4 * static_cast<int64_t>(topk) + 4 && index_tiles(L) < kSmallSeqTiles) ++n;
  }
  return n;
}

size_t dsa_index_topk_varlen_workspace(const int64_t* cu_seqlens, int nseq, int Hi, int Di, int chunk, int topk) {
  if (check_cu_seqlens("dsa_index_topk_varlen_workspace", cu_seqlens, nseq) != DSA_OK) return 0;
  const size_t one = dsa_index_topk_workspace(max_len(cu_seqlens, nseq), Hi, Di, chunk, topk);
  if (one == 0) return 0;
  // one slice per sequence indexed at once (the minimum accepted is one)
  const int n = small_long_seqs(cu_seqlens, nseq, topk);
  const int k = n < 2 ? 1 : (n < kVarlenStreams ? n : kVarlenStreams);
  return one * static_cast<size_t>(k);
}

dsa_status_t dsa_index_topk_varlen(const void* q_idx, const void* k_idx, const float* w, const int64_t* cu_seqlens,
                                   int nseq, int Hi, int Di, int chunk, int topk, int32_t* pool_idx, void* workspace,
                                   size_t ws_bytes, void* stream) {
  const dsa::CallScope scope("dsa_index_topk_varlen");
  const char* fn = "dsa_index_topk_varlen";
  dsa_status_t st = check_cu_seqlens(fn, cu_seqlens, nseq);
  if (st != DSA_OK) return st;
  // every check up front, so that an error leaves every sequence untouched
  if (!q_idx || !k_idx || !w || !pool_idx) return fail(DSA_ERR_INVALID_ARG, "%s: null tensor pointer", fn);
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned4(w) || !aligned4(pool_idx))
    return fail(DSA_ERR_INVALID_ARG, "%s: q_idx and k_idx must be 16-byte aligned, w and pool_idx 4-byte aligned", fn);
  if (chunk < 1 || topk < 1 || Hi < 1)
    return fail(DSA_ERR_INVALID_ARG, "%s: chunk=%d, topk=%d and Hi=%d must be >= 1", fn, chunk, topk, Hi);
  if (Di != kDi) return fail(DSA_ERR_UNSUPPORTED, "%s: Di=%d unsupported (kernels implement Di=64)", fn, Di);
  if (Hi > kMaxHi) return fail(DSA_ERR_UNSUPPORTED, "%s: Hi=%d unsupported (max %d)", fn, Hi, kMaxHi);
  if (topk > kMaxTopk) return fail(DSA_ERR_UNSUPPORTED, "%s: topk=%d unsupported (max %d)", fn, topk, kMaxTopk);
  // one slice (the longest sequence's recommended indexer workspace) is the
  // minimum; the recommended size holds one per sequence indexed at once
  const size_t one = dsa_index_topk_workspace(max_len(cu_seqlens, nseq), Hi, Di, chunk, topk);
  const size_t need = one;
  if (!workspace || ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed (%zu recommended), %zu given", fn, need,
                dsa_index_topk_varlen_workspace(cu_seqlens, nseq, Hi, Di, chunk, topk),
                workspace ? ws_bytes : (size_t)0);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DSA_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", fn);
  dsa::LaunchCtx ctx;
  st = make_ctx(stream, &ctx);
  if (st != DSA_OK) return st;
  // a sequence of at most 4 * topk + 4 tokens: no row has more than topk pools
  const int64_t short_max = 4 * static_cast<int64_t>(topk) + 4;
  dsa::ShortSeqs sh;
  sh.n = 0;
  int n_short = 0, n_long = 0;
  auto flush = [&]() -> dsa_status_t {
    if (sh.n == 0) return DSA_OK;
    const cudaError_t e = timed_launch("short_rows", ctx.stream, [&] {
      return dsa::launch_short_rows(pool_idx, topk, sh, ctx);
    });
    sh.n = 0;
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "dsa_index_topk_varlen: short-row launch");
  };
  for (int s = 0; s < nseq; ++s) {
    const int64_t L = cu_seqlens[s + 1] - cu_seqlens[s];
    if (L > short_max) continue;
    sh.start[sh.n] = cu_seqlens[s];
    sh.len[sh.n] = L;
    ++n_short;
    if (++sh.n == dsa::kSeqBatch && (st = flush()) != DSA_OK) return st;
  }
  if ((st = flush()) != DSA_OK) return st;
  const uint8_t* qb = static_cast<const uint8_t*>(q_idx);
  const uint8_t* kb = static_cast<const uint8_t*>(k_idx);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto run_seq = [&](int s, const dsa::LaunchCtx& c, uint8_t* slice) {
    const int64_t o = cu_seqlens[s], L = cu_seqlens[s + 1] - o;
    return index_topk_run(qb + o * Hi * Di * 2, kb + o * Di * 2, w + o * Hi, L, Hi, chunk, topk, 0, L,
                          pool_idx + o * topk, slice, one, c);
  };
  // the shorter long sequences, several at once when the workspace holds a
  // slice for each: helper streams forked from and joined back into the
  // caller's stream, each launch on a share of the SMs
  const int n_small = small_long_seqs(cu_seqlens, nseq, topk);
  int k_par = static_cast<int>(ws_bytes / one);
  k_par = k_par < n_small ? k_par : n_small;
  k_par = k_par < kVarlenStreams ? k_par : kVarlenStreams;
  int n_par = 0;
  if (k_par >= 2) {
    cudaStream_t hs[kVarlenStreams];
    if ((st = varlen_streams(hs)) != DSA_OK) return st;
    cudaEvent_t fork = nullptr, join[kVarlenStreams] = {};
    cudaError_t e = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
    for (int k = 0; k < k_par && e == cudaSuccess; ++k) e = cudaEventCreateWithFlags(&join[k], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(fork, ctx.stream);
    for (int k = 0; k < k_par && e == cudaSuccess; ++k) e = cudaStreamWaitEvent(hs[k], fork, 0);
    if (e != cudaSuccess) st = cuda_fail(e, "dsa_index_topk_varlen: stream fork");
    // the next sequence goes to the stream with the fewest tiles so far
    int64_t load[kVarlenStreams] = {};
    for (int s = 0; s < nseq && st == DSA_OK; ++s) {
      const int64_t L = cu_seqlens[s + 1] - cu_seqlens[s];
      if (L <= short_max) continue;
      const int64_t t = index_tiles(L);
      if (t >= kSmallSeqTiles) continue;
      int k = 0;
      for (int j = 1; j < k_par; ++j) k = load[j] < load[k] ? j : k;
      load[k] += t;
      dsa::LaunchCtx c = ctx;
      c.stream = hs[k];
      const int share = ctx.num_sms / k_par;
      c.persistent_ctas = static_cast<int>(t < 8 ? 8 : (t < share ? t : share));
      st = run_seq(s, c, ws + static_cast<size_t>(k) * one);
      ++n_long;
      ++n_par;
    }
    // join even after an error, so that nothing on the helpers outlives the call's stream order
    for (int k = 0; k < k_par; ++k) {
      if (join[k] == nullptr) continue;
      cudaError_t je = cudaEventRecord(join[k], hs[k]);
      if (je == cudaSuccess) je = cudaStreamWaitEvent(ctx.stream, join[k], 0);
      if (je != cudaSuccess && st == DSA_OK) st = cuda_fail(je, "dsa_index_topk_varlen: stream join");
    }
    if (fork != nullptr) cudaEventDestroy(fork);
    for (int k = 0; k < k_par; ++k)
      if (join[k] != nullptr) cudaEventDestroy(join[k]);
    if (st != DSA_OK) return st;
  }
  // the rest one at a time on the caller's stream, each on every SM
  for (int s = 0; s < nseq; ++s) {
    const int64_t L = cu_seqlens[s + 1] - cu_seqlens[s];
    if (L <= short_max) continue;
    if (k_par >= 2 && index_tiles(L) < kSmallSeqTiles) continue;  // already indexed
    ++n_long;
    st = run_seq(s, ctx, ws);
    if (st != DSA_OK) return st;
  }
  dsa::call_param("sequences", nseq);
  dsa::call_param("short_sequences", n_short);
  dsa::call_param("indexed_sequences", n_long);
  dsa::call_param("indexed_at_once", n_par);
  dsa::call_param("helper_streams", k_par >= 2 ? k_par : 0);
  dsa::call_variant("short sequences filled in one launch per 256; the persistent indexer once per longer sequence, "
                    "the shorter of them several at once on helper streams");
  return DSA_OK;
}

dsa_status_t dsa_sparse_attn_fwd_varlen(const void* q, const void* k, const void* v, const int32_t* pool_idx,
                                        const int64_t* cu_seqlens, int nseq, int Hq, int D, int topk, float scale,
                                        void* o, float* lse, void* stream) {
  const dsa::CallScope scope("dsa_sparse_attn_fwd_varlen");
  const char* fn = "dsa_sparse_attn_fwd_varlen";
  dsa_status_t st = check_cu_seqlens(fn, cu_seqlens, nseq);
  if (st != DSA_OK) return st;
  if (!q || !k || !v || !pool_idx || !o || !lse) return fail(DSA_ERR_INVALID_ARG, "%s: null tensor pointer", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(pool_idx) || !aligned16(o) || !aligned4(lse))
    return fail(DSA_ERR_INVALID_ARG, "%s: bf16 tensors must be 16-byte aligned, pool_idx and lse 4-byte aligned", fn);
  const int64_t T = cu_seqlens[nseq];
  st = check_attn_args(fn, T, Hq, D, topk);
  if (st != DSA_OK) return st;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(D));
  dsa::LaunchCtx ctx;
  st = make_ctx(stream, &ctx);
  if (st != DSA_OK) return st;
  const int64_t qrow = static_cast<int64_t>(Hq) * D * 2;
  for (int s0 = 0; s0 < nseq; s0 += dsa::kSeqBatch) {
    const int n = nseq - s0 < dsa::kSeqBatch ? nseq - s0 : dsa::kSeqBatch;
    const dsa::SeqTable tab = seq_table(cu_seqlens, s0, n);
    const int64_t r0 = tab.cu[0], rows = tab.cu[n] - r0;
    const cudaError_t e = timed_launch("attn_fwd", ctx.stream, [&] {
      return dsa::launch_attn_fwd(static_cast<const uint8_t*>(q) + r0 * qrow, k, v, pool_idx + r0 * topk, 0, rows,
                                  topk, scale, static_cast<uint8_t*>(o) + r0 * qrow, lse + r0 * Hq, ctx, &tab);
    });
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_fwd_varlen: launch");
  }
  dsa::call_param("sequences", nseq);
  dsa::call_param("T", T);
  dsa::call_param("topk", topk);
  dsa::call_variant("gather-bound forward over the packed batch, one launch per 256 sequences");
  return DSA_OK;
}

size_t dsa_sparse_attn_bwd_varlen_workspace(const int64_t* cu_seqlens, int nseq, int Hq, int D) {
  if (check_cu_seqlens("dsa_sparse_attn_bwd_varlen_workspace", cu_seqlens, nseq) != DSA_OK) return 0;
  return dsa_sparse_attn_bwd_workspace(cu_seqlens[nseq], Hq, D);
}

dsa_status_t dsa_sparse_attn_bwd_varlen(const void* dO, const void* q, const void* k, const void* v, const void* o,
                                        const float* lse, const int32_t* pool_idx, const int64_t* cu_seqlens,
                                        int nseq, int Hq, int D, int topk, float scale, void* dq, void* dk, void* dv,
                                        void* workspace, size_t ws_bytes, void* stream) {
  const dsa::CallScope scope("dsa_sparse_attn_bwd_varlen");
  const char* fn = "dsa_sparse_attn_bwd_varlen";
  dsa_status_t st = check_cu_seqlens(fn, cu_seqlens, nseq);
  if (st != DSA_OK) return st;
  if (!dO || !q || !k || !v || !o || !lse || !pool_idx || !dq || !dk || !dv)
    return fail(DSA_ERR_INVALID_ARG, "%s: null tensor pointer", fn);
  if (!aligned16(dO) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
      !aligned4(pool_idx) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(DSA_ERR_INVALID_ARG, "%s: bf16 tensors must be 16-byte aligned, pool_idx and lse 4-byte aligned", fn);
  const int64_t T = cu_seqlens[nseq];
  st = check_attn_args(fn, T, Hq, D, topk);
  if (st != DSA_OK) return st;
  const size_t need = dsa_sparse_attn_bwd_varlen_workspace(cu_seqlens, nseq, Hq, D);
  if (!workspace || ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                workspace ? ws_bytes : (size_t)0);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DSA_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", fn);
  if (!(scale > 0.f)) scale = 1.0f / sqrtf(static_cast<float>(D));
  dsa::LaunchCtx ctx;
  st = make_ctx(stream, &ctx);
  if (st != DSA_OK) return st;
  // the packed batch's fp32 dK/dV accumulators (adjacent) and Delta
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t acc_bytes = round_up(static_cast<size_t>(T) * D * sizeof(float), 256);
  float* dk_acc = reinterpret_cast<float*>(ws);
  float* dv_acc = reinterpret_cast<float*>(ws + acc_bytes);
  float* delta = reinterpret_cast<float*>(ws + 2 * acc_bytes);
  cudaError_t e = timed_launch("attn_bwd_pre", ctx.stream,
                               [&] { return dsa::launch_attn_bwd_pre(dO, o, T, T, delta, dk_acc, dv_acc, ctx); });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd_varlen: preprocess launch");
  const int64_t qrow = static_cast<int64_t>(Hq) * D * 2;
  for (int s0 = 0; s0 < nseq; s0 += dsa::kSeqBatch) {
    const int n = nseq - s0 < dsa::kSeqBatch ? nseq - s0 : dsa::kSeqBatch;
    const dsa::SeqTable tab = seq_table(cu_seqlens, s0, n);
    const int64_t r0 = tab.cu[0], rows = tab.cu[n] - r0;
    e = timed_launch("attn_bwd", ctx.stream, [&] {
      return dsa::launch_attn_bwd(static_cast<const uint8_t*>(dO) + r0 * qrow, static_cast<const uint8_t*>(q) + r0 * qrow,
                                  k, v, lse + r0 * Hq, delta + r0 * Hq, pool_idx + r0 * topk, 0, rows, topk, scale,
                                  static_cast<uint8_t*>(dq) + r0 * qrow, dk_acc, dv_acc, ctx, &tab);
    });
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd_varlen: launch");
  }
  e = timed_launch("attn_bwd_cast", ctx.stream, [&] { return dsa::launch_cast_dkdv(dk_acc, dv_acc, T * D, dk, dv, ctx); });
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_attn_bwd_varlen: cast launch");
  dsa::call_param("sequences", nseq);
  dsa::call_param("T", T);
  dsa::call_param("topk", topk);
  dsa::call_variant("atomic backward over the packed batch, one launch per 256 sequences");
  return DSA_OK;
}

dsa_status_t dsa_sync_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sync_status: stream");
  unsigned s = 0;
  e = cudaMemcpyFromSymbol(&s, g_dsa_status, sizeof(s));
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sync_status: read status");
  if (s & dsa::kStatusTimeout) return fail(DSA_ERR_TIMEOUT, "a bounded device-side wait ran out");
  if (s & dsa::kStatusInternal) return fail(DSA_ERR_INTERNAL, "a device-side check failed (malformed pool_idx?)");
  return DSA_OK;
}

dsa_status_t dsa_clear_status(void) {
  const unsigned z = 0;
  cudaError_t e = cudaMemcpyToSymbol(g_dsa_status, &z, sizeof(z));
  if (e != cudaSuccess) return cuda_fail(e, "dsa_clear_status");
  return DSA_OK;
}

int dsa_index_topk_stats(const void* workspace, size_t ws_bytes, int64_t* stats, int max_stats, void* stream) {
  if (!workspace || ws_bytes < kSyncBytes || !stats || max_stats < 1) {
    fail(DSA_ERR_INVALID_ARG, "dsa_index_topk_stats: null or short workspace, or no room for results");
    return -1;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned long long words[dsa::kIndexSyncWords];
  cudaError_t e = cudaMemcpyAsync(words, workspace, sizeof(words), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cuda_fail(e, "dsa_index_topk_stats: read counters");
    return -1;
  }
  stats[0] = static_cast<int64_t>(words[dsa::kIndexFallbackRowsWord]);
  return 1;
}

int dsa_trace_configure(void* buf, size_t bytes) {
#ifdef DSA_ITEM_TRACE
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (buf != nullptr && bytes < 64 + sizeof(dsa::IndexTraceRec)) return -1;
  g_trace_buf = buf;
  g_trace_bytes = buf ? bytes : 0;
  return 0;
#else
  (void)buf, (void)bytes;
  fail(DSA_ERR_UNSUPPORTED, "dsa_trace_configure: this library was built without DSA_ITEM_TRACE");
  return -1;
#endif
}

int dsa_fwd_tc_profile(uint64_t* counters, int ctas) {
  if (!counters || ctas < 1) {
    fail(DSA_ERR_INVALID_ARG, "dsa_fwd_tc_profile: counters must hold ctas x 32 words, ctas >= 1");
    return -1;
  }
  const int n = dsa::fwd_tc_profile_read(reinterpret_cast<unsigned long long*>(counters), ctas);
  if (n < 0) fail(DSA_ERR_UNSUPPORTED, "dsa_fwd_tc_profile: this library was built without DSA_FWD_PROFILE");
  return n;
}

void dsa_profile_enable(int on) { g_profiling.store(on ? 1 : 0); }

int dsa_profile_read(char* names, int name_len, double* ms, int64_t* launches, int max_kernels) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof);
  }
  std::map<std::string, std::pair<double, int64_t>> agg;
  std::vector<std::string> order;
  bool ok = true;
  for (ProfRec& r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      ok = false;
    if (!agg.count(r.name)) order.push_back(r.name);
    agg[r.name].first += t;
    agg[r.name].second += 1;
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  if (!ok) {
    fail(DSA_ERR_CUDA, "dsa_profile_read: event timing failed");
    return -1;
  }
  int k = 0;
  for (const std::string& n : order) {
    if (k >= max_kernels) break;
    if (names && name_len > 0) {
      snprintf(names + static_cast<size_t>(k) * name_len, name_len, "%s", n.c_str());
    }
    if (ms) ms[k] = agg[n].first;
    if (launches) launches[k] = agg[n].second;
    ++k;
  }
  return k;
}

int64_t dsa_launch_count(void) { return g_launches.load(); }

void dsa_launch_count_reset(void) { g_launches.store(0); }

}  // extern "C"
