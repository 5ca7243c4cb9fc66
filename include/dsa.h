/*
 * dsa.h -- C ABI of libdsa, the DeepSeek-Sparse-Attention (DSA) layer hot
 * path for one GB300 GPU (sm_103a): causal pooled indexer -> per-query top-k
 * of key pools -> sparse attention forward and backward.
 *
 * Sources (page title and section; the pages print no formulas or code):
 *  [SkyRL-1M]  "SkyRL 将 GLM-5.3-Flash 训练上下文扩至 100 万 token",
 *              §模型与瓶颈: DSA attends to ~2048 keys per query, while its
 *              indexer scores every query against every 4-token key pool,
 *              which moves the quadratic cost into the indexer;
 *              §1 DSA 真稀疏: the Flash variant has no positional encoding
 *              and keeps 2051 keys; the indexer is scored query chunk by
 *              query chunk (peak scoring memory ~64 GiB -> ~2.3 GiB at 32k)
 *              and sharded by query, exchanging int32 selected-pool indices.
 *  [Anyscale]  "How Lila Sciences and Anyscale Scaled GLM-5.3-Flash
 *              Training", the lesson on checking that every layer runs the
 *              kernel one expects (a sparse kernel had silently fallen back
 *              to dense attention) and the
 *              second lesson, on the indexer: sparse attention moves its
 *              quadratic cost into the indexer rather than removing it, and
 *              scoring a few hundred queries at a time keeps the score
 *              matrix under 2 GiB).
 *  [CP-lesson] "128K 的序列,激活放在哪?" (context-parallel lesson),
 *              §改进二 and evidence row ②: blockwise online softmax equals
 *              the one-shot softmax.
 *
 * The pages give no indexer formula.  This library computes
 *   Khat_p     = fp32 mean of k_idx rows 4p..4p+3, summed ((k0+k1)+(k2+k3))/4
 *   score(i,p) = sum_h w[i,h] * ReLU(q_idx[i,h,:] . Khat_p)     for 4p+3 < i
 * and selects, for every query i, the min(topk, floor(i/4)) eligible pools
 * with the largest scores (ties to the lower pool index).  Query i then
 * attends to the 4 keys of each selected pool plus its own partial pool
 * {4*floor(i/4), ..., i} (1 to 4 tokens, i itself included): up to
 * 4*topk + 4 keys.  With topk >= floor(i/4) this is dense causal attention.
 *
 * Conventions shared by every call:
 *  - Batch 1, row-major, no padding.  bf16 tensors are passed as void*.
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library allocates no device memory; scratch comes from the caller's
 *    `workspace` (sized by the *_workspace() queries).  bf16 tensors must
 *    be 16-byte aligned; fp32 and int32 tensors (w, lse, pool_idx) 4-byte
 *    aligned.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work and return; results are ready in stream order.
 *  - Arguments are checked before anything is launched; on error nothing is
 *    written and no kernel runs.  Unsupported shapes return
 *    DSA_ERR_UNSUPPORTED: there is no fallback path of any kind.
 *  - Device-side waits are bounded.  A wait that runs out sets a device
 *    status word and the kernel returns early; dsa_sync_status() reports it.
 *  - A failing call stores a message for dsa_last_error() (per host thread).
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or range  */
  DSA_ERR_UNSUPPORTED = 2,  /* shape outside what the kernels implement     */
  DSA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required   */
  DSA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed         */
  DSA_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out           */
  DSA_ERR_INTERNAL = 6      /* a device-side consistency check failed       */
} dsa_status_t;

/* Bytes of workspace dsa_index_topk is best given for sequence length S, Hi
 * indexer heads of dim Di, query chunk `chunk` and `topk`: 512 B of kernel
 * words; the pooled keys (as a bf16 hi/lo pair and as fp32, 512 B per pool);
 * a list of rows for the fallback path (4 B per query) and its 64 scratch rows
 * of scores (4 B per pool each); and a ring of min(8, ceil(S/chunk)) chunk
 * slots, which consecutive chunks take in turn.  A slot holds, for each of
 * min(chunk, S) rows (thresholds and counts padded to 128 rows), the scores of every sigma-th pool (sigma = max(2^
 * floor(log2(topk/16)), 2^ceil(log2(ceil(S/4 / 4096)))), 32 at S = 131072,
 * topk = 512), a threshold, a candidate count and up to `cap` candidates of
 * 8 B (cap = 4096 for topk <= 512).  97 MB in all at S = 131072, chunk 256,
 * topk 512; 388 MB at S = 1048576, chunk 512.  dsa_index_topk also accepts a
 * smaller workspace, down to min(2, ceil(S/chunk)) slots, and uses as many
 * slots as fit: fewer slots keep fewer chunks in flight (slower), with the
 * same result.  Returns 0 for invalid arguments. */
size_t dsa_index_topk_workspace(int64_t S, int Hi, int Di, int chunk, int topk);

/* Bytes of an index workspace that holds exactly `slots` chunk slots (1 ..
 * min(8, ceil(S/chunk))); dsa_index_topk_workspace() is this for the most
 * slots, and the least workspace dsa_index_topk accepts is this for
 * min(2, ceil(S/chunk)).  Returns 0 for invalid arguments. */
size_t dsa_index_topk_workspace_slots(int64_t S, int Hi, int Di, int chunk, int topk, int slots);

/*
 * Indexer + top-k  [SkyRL-1M §模型与瓶颈, §1 DSA 真稀疏; Anyscale, second
 * lesson (the indexer's quadratic cost)].
 *
 *  q_idx     bf16 [S, Hi, Di]  indexer queries (rows q_begin..q_end-1 read)
 *  k_idx     bf16 [S, Di]      indexer keys
 *  w         fp32 [S, Hi]      per-query head weights (any sign)
 *  S         sequence length, 1 <= S <= 2^31 - 1
 *  Hi, Di    indexer heads (1..64) and head dim (must be 64)
 *  chunk     queries scored per pass (>= 1): bounds the per-chunk scratch
 *  topk      pools kept per query (1..2048)
 *  q_begin, q_end   query range to process, 0 <= q_begin < q_end <= S; a
 *            shard of a sequence passes its own range (rows are independent)
 *  pool_idx  int32 [q_end - q_begin, topk] output: for query i the selected
 *            pools in ascending order, then -1 padding (row i holds
 *            min(topk, floor(i/4)) pools)
 *  workspace, ws_bytes  device scratch: dsa_index_topk_workspace(S, Hi, Di,
 *            chunk, topk) bytes, or fewer down to the two-slot minimum (see
 *            there); 256-byte aligned
 *
 * The score matrix is never stored.  Each row keeps, as candidates, the
 * pools whose (score, -index) is at or above a threshold taken from the
 * scores of every sigma-th pool; the row's top-k is then selected from its
 * candidates, which is exact whenever at least topk pools are candidates.
 * Rows that fall short (or overflow the candidate list) are recomputed in
 * full by a fallback kernel; dsa_index_topk_stats() counts them.
 * Selection is exact with respect to the fp32 scores the kernels compute
 * (bf16 inputs, fp32 accumulation, pooled keys carried as a bf16 hi/lo pair
 * so the product keeps ~16 more bits than a single bf16 rounding; a fallback
 * row's scores are fp32 dot products with the fp32 pooled keys).
 */
dsa_status_t dsa_index_topk(const void* q_idx, const void* k_idx, const float* w, int64_t S, int Hi, int Di,
                            int chunk, int topk, int64_t q_begin, int64_t q_end, int32_t* pool_idx,
                            void* workspace, size_t ws_bytes, void* stream);

/*
 * Sparse attention forward  [SkyRL-1M §模型与瓶颈; CP-lesson §改进二].
 *
 *  q         bf16 [S, Hq, D]  queries (Hq heads share one KV head)
 *  k, v      bf16 [S, D]      keys and values
 *  pool_idx  int32 [S, topk]  selection as written by dsa_index_topk
 *            (ascending, -1 padded, every entry < floor(i/4) for row i)
 *  Hq = 16, D = 128 (other shapes: DSA_ERR_UNSUPPORTED)
 *  scale     softmax scale; <= 0 means 1/sqrt(D)
 *  o         bf16 [S, Hq, D]  output
 *  lse       fp32 [S, Hq]     natural-log softmax normaliser of the scaled
 *                             logits (kept for the backward)
 * Online softmax in fp32 over blocks of gathered keys.
 */
dsa_status_t dsa_sparse_attn_fwd(const void* q, const void* k, const void* v, const int32_t* pool_idx, int64_t S,
                                 int Hq, int D, int topk, float scale, void* o, float* lse, void* stream);

/*
 * The same forward with both contractions on the tcgen05 tensor cores
 * (S^T = K.Q^T and O^T += V^T.P^T with fp32 accumulators in tensor memory),
 * by one persistent warp-specialised CTA per SM.  Arguments, layouts, results
 * (within rounding) and errors are those of dsa_sparse_attn_fwd.  It is the
 * measured tensor-core alternative, not the faster path: with 16 heads every
 * MMA has N = 16, and on GB300 it runs slower than dsa_sparse_attn_fwd.
 */
dsa_status_t dsa_sparse_attn_fwd_tc(const void* q, const void* k, const void* v, const int32_t* pool_idx, int64_t S,
                                    int Hq, int D, int topk, float scale, void* o, float* lse, void* stream);

/* Bytes of workspace dsa_sparse_attn_bwd needs: fp32 dK and dV accumulators
 * (2 x S x D x 4 B) plus the per-row softmax-gradient term (S x Hq x 4 B). */
size_t dsa_sparse_attn_bwd_workspace(int64_t S, int Hq, int D);

/*
 * Sparse attention backward  [SkyRL-1M §模型与瓶颈: attention over the
 * selected keys, trained end to end].
 *
 *  dO        bf16 [S, Hq, D]  upstream gradient of o
 *  q, k, v, pool_idx, S, Hq, D, topk, scale   as in the forward
 *  o, lse    the forward's outputs
 *  dq        bf16 [S, Hq, D]  output
 *  dk, dv    bf16 [S, D]      outputs
 *  workspace, ws_bytes  at least dsa_sparse_attn_bwd_workspace(S, Hq, D)
 * dK/dV contributions of every query are added into fp32 accumulators with
 * atomic reductions, so their bits may vary from run to run (within fp32
 * rounding); dq is deterministic.
 */
dsa_status_t dsa_sparse_attn_bwd(const void* dO, const void* q, const void* k, const void* v, const void* o,
                                 const float* lse, const int32_t* pool_idx, int64_t S, int Hq, int D, int topk,
                                 float scale, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                                 void* stream);

/* Bytes of workspace dsa_sparse_attn_bwd_deterministic needs: fp32 dK and dV
 * accumulators (2 x S x D x 4 B), Delta (S x Hq x 4 B), the per-pool query
 * lists (S x topk x 4 B) and their per-(pool, 1024-query block) counters
 * (about S^2 / 1024 bytes, at most 256 MiB).  0 for an unsupported shape, or
 * when S x topk exceeds 2^31 - 1 or S / 4 exceeds 2^26. */
size_t dsa_sparse_attn_bwd_deterministic_workspace(int64_t S, int Hq, int D, int topk);

/*
 * Sparse attention backward with bit-reproducible dk and dv  [SkyRL-1M
 * §模型与瓶颈: the selected-key attention is trained end to end].  The
 * arguments, shapes and results are those of dsa_sparse_attn_bwd, for the
 * whole sequence (no query range); the workspace is
 * dsa_sparse_attn_bwd_deterministic_workspace(S, Hq, D, topk) bytes,
 * 256-byte aligned.
 * dK/dV are summed key-major in a fixed order with no atomics: the selection
 * is transposed into the list of selecting queries of every pool
 * (ascending); then, span of 4096 queries by span (more per span beyond
 * S = 2^20) in ascending order, one CTA per pool adds the span's
 * contributions (its own partial-pool queries first, then its selecting
 * queries in order, split into four fixed quarters summed in order) into
 * the pool's fp32 rows.
 * The same inputs give the same dq, dk and dv bits on every run.  It reads
 * q and dO (8 KB) per (query, pool) pair, from L2 while a span is resident,
 * where the default gathers K/V and scatters with atomics.  Returns
 * DSA_ERR_UNSUPPORTED when S x topk exceeds 2^31 - 1 or S / 4 exceeds 2^26.
 */
dsa_status_t dsa_sparse_attn_bwd_deterministic(const void* dO, const void* q, const void* k, const void* v,
                                               const void* o, const float* lse, const int32_t* pool_idx, int64_t S,
                                               int Hq, int D, int topk, float scale, void* dq, void* dk, void* dv,
                                               void* workspace, size_t ws_bytes, void* stream);

/*
 * Query-range forms of the attention calls, for a rank that holds only some
 * of the sequence's queries (context parallelism [CP-lesson §改进二: the
 * sequence is split across GPUs by query rows, and each rank still needs all
 * keys]).  Queries q_begin .. q_end-1 (global positions, 0 <= q_begin <
 * q_end <= S) are processed:
 *  q, o, dO, dq   bf16 [q_end - q_begin, Hq, D]  local rows (row r = query q_begin + r)
 *  lse            fp32 [q_end - q_begin, Hq]     local rows
 *  pool_idx       int32 [q_end - q_begin, topk]  local rows, as dsa_index_topk
 *                 writes them for the same range
 *  k, v           bf16 [S, D]                   the whole sequence
 *  dk, dv         bf16 [S, D]                   this range's contribution only;
 *                 summing the ranks' contributions (a reduce-scatter or
 *                 all-reduce across ranks, which the caller runs) gives the
 *                 full gradient
 * The other arguments and the workspace are as in the unsharded calls, which
 * are these calls with the range [0, S).  Results for a query do not depend
 * on the range it is computed in (dk/dv up to fp32 summation order).
 */
dsa_status_t dsa_sparse_attn_fwd_range(const void* q, const void* k, const void* v, const int32_t* pool_idx,
                                       int64_t S, int64_t q_begin, int64_t q_end, int Hq, int D, int topk,
                                       float scale, void* o, float* lse, void* stream);
dsa_status_t dsa_sparse_attn_bwd_range(const void* dO, const void* q, const void* k, const void* v, const void* o,
                                       const float* lse, const int32_t* pool_idx, int64_t S, int64_t q_begin,
                                       int64_t q_end, int Hq, int D, int topk, float scale, void* dq, void* dk,
                                       void* dv, void* workspace, size_t ws_bytes, void* stream);

/*
 * Zig-zag query ranges of `rank` among `world` ranks  [CP-lesson §改进二,
 * zig-zag pairing]: the sequence is cut into 2*world segments
 * [j*S/(2*world), (j+1)*S/(2*world)); rank r takes segments r and
 * 2*world-1-r, so with causal masking every rank has the same amount of work
 * (exactly, when 2*world divides S).  Writes ranges = {b0, e0, b1, e1}
 * (half-open, global positions; a range may be empty for tiny S).  Each
 * range is passed to dsa_index_topk / dsa_sparse_attn_*_range as
 * q_begin/q_end; positions stay global, so pools stay aligned with their keys.
 * Host-only; DSA_ERR_INVALID_ARG unless S >= 1 and 0 <= rank < world.
 */
dsa_status_t dsa_zigzag_ranges(int64_t S, int world, int rank, int64_t* ranges);

/*
 * Packed variable-length batches.  nseq sequences lie end to end in every
 * tensor; sequence s covers rows cu_seqlens[s] .. cu_seqlens[s+1]-1
 * (cu_seqlens: HOST array of nseq+1 strictly increasing int64 offsets,
 * cu_seqlens[0] = 0; the total is the packed length).  Each sequence is its
 * own causal layer, as if passed alone: its pools, eligibility and pool_idx
 * entries count from its first token, and no query sees another sequence's
 * keys.  Tensors, scale and topk are as in the single-sequence calls, with
 * the packed length in place of S; dk/dv rows of a sequence hold that
 * sequence's gradient.  Workspaces: for the backward, the *_varlen_workspace()
 * bytes, the single-sequence workspace of the packed length (its fp32 dK/dV
 * accumulators span the batch).  For the indexer, at least one slice, the
 * single-sequence recommended workspace of the longest sequence;
 * dsa_index_topk_varlen_workspace() recommends one slice per long sequence
 * indexed at once (up to 4).  The attention calls cover the batch with one
 * launch per kernel and per 256 sequences (a table of their starts rides in
 * the launch parameters; each query finds its sequence by binary search).
 * The indexer fills the rows of every sequence of at most 4 * topk + 4
 * tokens (each row keeps all its pools) with one launch per 256 such
 * sequences, and runs once per longer sequence.  Sequences with fewer than
 * 304 indexer tiles (128 queries x 256 pools; up to ~9000 tokens) leave most
 * SMs idle in a launch of their own: when the workspace holds two or more
 * slices they run that many at once, each on a helper stream of the library
 * (forked from and joined back into `stream` by events) with a share of the
 * SMs; the others run one after another on `stream` on every SM.  Results do
 * not depend on the workspace size.  An invalid cu_seqlens or a short workspace returns
 * DSA_ERR_INVALID_ARG / DSA_ERR_WORKSPACE (and, for the query functions, 0)
 * before anything runs.  (The pages train single sequences; packing is what a
 * training data loader hands the layer.)
 */
size_t dsa_index_topk_varlen_workspace(const int64_t* cu_seqlens, int nseq, int Hi, int Di, int chunk, int topk);
dsa_status_t dsa_index_topk_varlen(const void* q_idx, const void* k_idx, const float* w, const int64_t* cu_seqlens,
                                   int nseq, int Hi, int Di, int chunk, int topk, int32_t* pool_idx, void* workspace,
                                   size_t ws_bytes, void* stream);
dsa_status_t dsa_sparse_attn_fwd_varlen(const void* q, const void* k, const void* v, const int32_t* pool_idx,
                                        const int64_t* cu_seqlens, int nseq, int Hq, int D, int topk, float scale,
                                        void* o, float* lse, void* stream);
size_t dsa_sparse_attn_bwd_varlen_workspace(const int64_t* cu_seqlens, int nseq, int Hq, int D);
dsa_status_t dsa_sparse_attn_bwd_varlen(const void* dO, const void* q, const void* k, const void* v, const void* o,
                                        const float* lse, const int32_t* pool_idx, const int64_t* cu_seqlens,
                                        int nseq, int Hq, int D, int topk, float scale, void* dq, void* dk, void* dv,
                                        void* workspace, size_t ws_bytes, void* stream);

/*
 * Indexer + top-k for callers that cannot allocate device memory.  (The
 * source pages have no counterpart to this call; it exists for users of the
 * library.)
 *
 * Same arguments, outputs and results as dsa_index_topk, but without a
 * workspace: the scratch lives in a fixed static device array of 32 MiB
 * inside the library.  Sizes run when dsa_index_topk's least workspace for
 * them (two chunk slots) fits in it -- every S <= 32768 with chunk <= 256 and
 * topk <= 512, for example; other sizes return DSA_ERR_WORKSPACE (see
 * dsa_last_error()) and nothing runs.  At the largest sizes that fit, only
 * two chunks are in flight, so the call is slower than dsa_index_topk with
 * its recommended workspace (same result).
 * Under CUDA's default lazy module loading a device reserves the array when
 * the library's module holding it is first loaded there, which happens in
 * the first call on that device (that call looks up the array's device
 * address with cudaGetSymbolAddress, with the device current); the device
 * then holds the array until the process exits.  So make the first call on
 * each device outside any region that must not allocate and before any
 * stream capture; later calls allocate nothing.  The address is cached per
 * CUDA context and looked up again after a device reset.  All calls on a
 * device share the array and leave their contents in it; nothing needs to be
 * zero beforehand.  Calls whose GPU work overlaps (e.g. on unordered
 * streams) race on the array: order them.
 */
dsa_status_t dsa_index_topk_noalloc(const void* q_idx, const void* k_idx, const float* w, int64_t S, int Hi, int Di,
                                    int chunk, int topk, int64_t q_begin, int64_t q_end, int32_t* pool_idx,
                                    void* stream);

/*
 * Counters of the last dsa_index_topk call that used `workspace` (a
 * measurement helper; no part of the layer's arithmetic).  Synchronises
 * `stream` (the stream of that call), then writes up to `max_stats` values:
 *   stats[0]  query rows whose candidates could not certify the top-k
 *             (fewer than topk, or more than the list holds), so the
 *             fallback kernel recomputed all their scores
 * Returns the number of values written, or -1 (with dsa_last_error()) for a
 * null or short workspace or a CUDA error.
 */
int dsa_index_topk_stats(const void* workspace, size_t ws_bytes, int64_t* stats, int max_stats, void* stream);

/* Synchronises `stream` and returns DSA_ERR_TIMEOUT / DSA_ERR_INTERNAL if a
 * kernel has recorded a failed bounded wait or check since the last
 * dsa_clear_status(), DSA_ERR_CUDA if the stream reports an error, else
 * DSA_OK. */
dsa_status_t dsa_sync_status(void* stream);

/* Clears the device status word (synchronous). */
dsa_status_t dsa_clear_status(void);

/*
 * What the last call on this host thread ran ([Anyscale, the lesson on
 * checking that every layer runs the kernel one expects]).  Writes one JSON
 * line describing the outermost dsa_* entry point
 * this thread called last (an entry point that calls another reports as
 * itself): {"entry": name, "variant": the path it took, "kernels": [[kernel,
 * launches], ...] in launch order (consecutive launches of one kernel
 * counted together; empty when the call failed before launching),
 * "params": {the plan: sizes, query range, chunk slots, sample stride,
 * threshold rank, candidate slots per row, spans, ...}}.  The fallback-row
 * count of the indexer is on the device (dsa_index_topk_stats).  Writes at
 * most len bytes including the terminating NUL (buf may be NULL with len 0)
 * and returns the full length without the NUL, as snprintf does.
 * Every entry point also opens an NVTX range named for it, visible to
 * profilers that record NVTX (no cost otherwise).
 */
int dsa_last_kernel_config(char* buf, size_t len);

/* Message describing the last non-OK status returned on this host thread. */
const char* dsa_last_error(void);

/* Library version string. */
const char* dsa_version(void);

/*
 * Measurement helpers (no part of the layer's arithmetic).
 *
 * dsa_profile_enable(1) makes every subsequent launch record a pair of CUDA
 * events on its stream; dsa_profile_enable(0) stops recording.
 * dsa_profile_read() synchronises those events and writes, for up to
 * `max_kernels` kernels, the kernel name into names[k*name_len ...] (NUL
 * terminated), the summed device time in ms into ms[k] and the number of
 * launches into launches[k]; it returns the number of kernels (or -1 on a
 * CUDA error) and clears the recorded events.
 * dsa_launch_count() returns the number of kernels launched by this library
 * in this process since dsa_launch_count_reset(), whether or not profiling
 * is enabled.
 */
/*
 * L2 rate probes (measurement helper).  Runs one probe kernel `iters` times
 * (after one untimed warm-up pass) on the caller's device buffer `buf` of
 * `bytes` bytes (16-byte aligned, >= 4096; size it below L2 to measure L2)
 * on `stream`, times it with CUDA events (synchronising), and returns the
 * rate in GB/s of bytes moved, or -1.0 on error:
 *   kind 0  streaming 16-byte loads over the buffer
 *   kind 1  random 1 KB blocks read whole by one warp each (the attention
 *           kernels' gather of one key pool's four 256-byte rows)
 *   kind 2  red.global.add.v4.f32 on random 2 KB blocks, each warp
 *           instruction adding 128 bytes to each of a block's four 512-byte
 *           rows (the backward's dK/dV reductions); counts bytes added
 *   kind 3  bulk reductions (cp.reduce.async.bulk .add.f32) from shared
 *           memory, one 2 KB block per operation, random blocks
 *   kind 4  the same with 512-byte operations (one row each)
 *   kind 5  red.v4 with 2 rows x 256 B per warp instruction
 *   kind 6  red.v4 with 8 rows x 64 B per warp instruction
 *   kind 7  red.v4 with 16 rows x 32 B per warp instruction (the shape of
 *           reductions issued straight from mma.sync fragments)
 *   kind 8  kind 2 and kind 3 at once, from the two halves of every CTA
 * Kinds 2..8 add into the buffer's contents.
 */
double dsa_measure_l2(int kind, void* buf, size_t bytes, int iters, void* stream);

/*
 * Tensor-core issue probe (measurement helper).  On every SM, `issuers` CTAs
 * (1..3) each have one thread issue `groups` groups of 8 back-to-back
 * tcgen05.mma (kind::f16: bf16 operands from 128-byte swizzled shared
 * memory, fp32 accumulator in tensor memory; M = 128, K = 16, N = n for n in
 * {16, 32, 64, 128, 256}; issuers * max(n, 32) <= 512), then waits for them.
 * Synchronises `stream` and returns the issuing thread's clock cycles per
 * instruction, averaged over the CTAs, or -1.0 on error.  The sparse
 * attention's products have N = 16 (one column per query head).
 */
double dsa_measure_umma(int n, int issuers, int groups, void* stream);

/*
 * Accumulator-handoff probe of the indexer (measurement helper).  One CTA of
 * the indexer's 19-warp layout: one thread issues, per head, 8 chained
 * tcgen05.mma (M = 128, N = 256, K = 16, bf16) into one of two tensor-memory
 * accumulators, and 16 epilogue warps each load their lane quarter's 64
 * columns 16 at a time and release the accumulator after the last load.
 *   mode 0  the loads alone
 *   mode 1  the loads and the indexer's fold (ReLU, packed FMA into 64 fp32
 *           sums a thread)
 *   mode 2  one warp's 32-column tensor-memory load and its wait, alone
 * Runs `heads` (>= 2) heads after one warm-up pass, synchronises `stream`
 * and returns the issuing thread's clock cycles per head (mode 2: per load),
 * or -1.0 on error.  The 8 products of one head take 1024 cycles at the
 * dense bf16 rate.
 */
double dsa_measure_fold(int mode, int heads, void* stream);

/*
 * Item trace of the persistent indexer (measurement helper; only the trace
 * build of the library, libdsa_trace.so, compiled with DSA_ITEM_TRACE, records
 * anything -- the default build returns -1).  `buf` is a device buffer of
 * `bytes`: a 64-byte header whose first 8 bytes count the records (the
 * caller zeroes it before the call it wants traced), then records of 40 bytes
 * {uint32 kind | sm << 8, uint32 chunk, uint64 t0, t1, t2, t3}: the
 * globaltimer (ns) when the epilogue took the item, ended its fold over heads
 * (= t0 for row items), ended its dependency wait, and published it.  kind:
 * 0 sample tile, 1 thresholds, 2 indexer tile, 3 top-k rows.  Records past
 * the buffer are dropped (the count keeps counting).  NULL stops tracing.
 * Returns 0, or -1.
 */
int dsa_trace_configure(void* buf, size_t bytes);

/*
 * Role counters of the last dsa_sparse_attn_fwd_tc launch (measurement
 * helper; only the trace build, compiled with DSA_FWD_PROFILE, has them --
 * the default build returns -1).  Copies ctas x 32 uint64 words into
 * `counters` (host memory), one row per CTA of the launch (the launch has
 * min(S, number of SMs) CTAs): clock cycles each warp role spent per
 * pipeline segment, summed over the blocks it handled --
 *   words 0..5   producers: row-buffer wait, selection scan, free-stage wait,
 *                block record, copy issue, drain; word 7 blocks
 *   words 8..12  issuer: full-stage wait, free-S^T wait, S^T issue, O^T
 *                products (their P^T waits included), final drain; word 15 blocks
 *   words 16..21 softmax: full-stage wait, S^T wait and load, maximum check
 *                (and rescale), P^T-buffer wait, P^T write, epilogue; word 23 blocks
 * Returns the words copied, or -1.
 */
int dsa_fwd_tc_profile(uint64_t* counters, int ctas);

void dsa_profile_enable(int on);
int dsa_profile_read(char* names, int name_len, double* ms, int64_t* launches, int max_kernels);
int64_t dsa_launch_count(void);
void dsa_launch_count_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
