// topk_row.cuh -- per-query top-k of indexer scores, as a device routine run
// by a group of 128 threads (4 warps, one named barrier) on one query row.
//
// [SkyRL-1M §1 DSA 真稀疏] each query keeps its highest-scoring pools and the
// selection travels as int32 pool indices.  For query i with n = floor(i/4)
// eligible pools the routine keeps min(topk, n) of them: every pool whose
// score is larger than the k-th largest score T, plus the lowest-indexed
// pools whose score equals T.  Kept pools are written in ascending order,
// then -1.
//
// Method (scores map to order-preserving 32-bit keys):
//   1. Threshold guess.  A strided sample of kSample keys (read as 16-byte
//      quads) is histogrammed on the top kDigitBits bits of its span; the
//      lower edge t of the bin that holds the r-th largest sample is the
//      threshold, with r chosen so that, unless the row's large scores are
//      packed into a few places, at least topk keys of the row are >= t while
//      only about a thousand are (short rows skip this: every key is a
//      candidate).
//   2. One pass over the row: each warp owns a contiguous stretch and appends
//      the keys >= t, with their indices, to its own buffer in index order
//      (slots from ballots; loads one batch ahead).
//   3. With at least topk candidates and no buffer overflowing, the exact
//      k-th largest candidate key T comes from digit rounds over the
//      candidates; once the bin holding T has at most kSmall keys they are
//      ranked against each other directly.  The candidates are then walked in
//      index order to write the kept indices.  Every key of the row that is
//      >= T is a candidate, so the result is exact.
//   4. Otherwise (the guess failed) the row takes the general path: value
//      histograms over [min, max] narrow down to T, and a stable compaction
//      pass over the whole row writes the kept indices.
// Score loads go through L2 only (__ldcg): the score buffers are rewritten by
// other CTAs between uses.
#pragma once

#include "dsa_device.cuh"

namespace dsa {
namespace topk {

constexpr int kGT = 128;                 // threads of a group
constexpr int kGW = kGT / 32;            // warps of a group
constexpr int kWarpCap = 512;            // candidate slots per warp
constexpr int kSample = 2048;            // sampled keys (4 quads per thread)
constexpr int kDigitBits = 10;           // digit rounds: 1024 bins
constexpr int kBins = 1 << kDigitBits;
constexpr int kGenBins = 1024;           // general-path value histogram
constexpr int kSmall = 64;               // a bin this small is ranked directly
constexpr int kBatch = 4;                // float4 loads in flight per lane in the candidate pass
constexpr int kPerRound = 4 * kGT;       // general-path compaction stretch

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// A float t with f >= t exactly when score_key(f) >= k, for every non-NaN
// f: the float whose key is k; -inf for k at or below the key of -inf (the
// keys below it are NaN patterns); -0 for k = 0x7FFFFFFF, the one key no
// score has (just below +0's).
__device__ __forceinline__ float key_score(uint32_t k) {
  if (k <= 0x007FFFFFu) return -INFINITY;
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

struct alignas(16) Smem {
  union {
    struct {
      uint32_t key[kGW][kWarpCap];
      uint32_t idx[kGW][kWarpCap];
    } cand;
    uint32_t samp[kSample];
    struct {
      uint32_t hist[kGenBins];
      uint32_t cand[kGenBins];
    } gen;
  } u;
  uint32_t hist[kBins];
  uint32_t small[kSmall];
  uint32_t wcount[kGW];
  uint32_t wmax[kGW];
  uint32_t wsum[2][kGW];
  uint32_t red[2 * kGW];
  uint32_t sel[4];
  uint32_t ncand;
  uint32_t nsmall;
};

// The group's threads: index within the group and the named barrier that
// synchronises exactly them.
struct Group {
  int tid;
  int bar_id;
  __device__ __forceinline__ void sync() const {
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kGT) : "memory");
  }
  __device__ __forceinline__ int lane() const { return tid & 31; }
  __device__ __forceinline__ int warp() const { return tid >> 5; }
};

// Exclusive prefix over the group of one value per thread (thread order),
// with one barrier; callers alternate `buf`.  *total gets the sum.
__device__ __forceinline__ uint32_t group_excl_scan(const Group& g, uint32_t v, uint32_t* buf, uint32_t* total) {
  const int lane = g.lane(), warp = g.warp();
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) buf[warp] = x;
  g.sync();
  uint32_t warp_base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kGW; ++w) {
    const uint32_t t = buf[w];
    warp_base += w < warp ? t : 0u;
    tot += t;
  }
  *total = tot;
  return warp_base + x - v;
}

// With a histogram of nb (<= kBins) bins, finds the bin b holding the need-th
// largest key: sm.sel = {b, count above b, count in b}.  Ends with a barrier.
// (SM: any shared-memory struct with the wsum and sel members of Smem.)
template <typename SM>
__device__ __forceinline__ void find_bin(const Group& g, const uint32_t* hist, SM& sm, uint32_t nb, uint32_t need,
                                         int& parity) {
  constexpr int kPer = kBins / kGT;  // bins per thread, in descending order
  uint32_t c[kPer], s = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int b = static_cast<int>(nb) - 1 - kPer * g.tid - q;
    c[q] = b >= 0 ? hist[b] : 0u;
    s += c[q];
  }
  uint32_t tot;
  const uint32_t excl = group_excl_scan(g, s, sm.wsum[parity], &tot);
  parity ^= 1;
  if (excl < need && excl + s >= need) {
    uint32_t cum = excl;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      if (cum + c[q] >= need) {
        sm.sel[0] = nb - 1 - kPer * g.tid - q;
        sm.sel[1] = cum;
        sm.sel[2] = c[q];
        break;
      }
      cum += c[q];
    }
  }
  g.sync();
}

template <typename SM>
__device__ __forceinline__ void group_minmax(const Group& g, uint32_t& lo, uint32_t& hi, SM& sm) {
  const int lane = g.lane(), warp = g.warp();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    sm.red[warp] = lo;
    sm.red[kGW + warp] = hi;
  }
  g.sync();
#pragma unroll
  for (int w = 0; w < kGW; ++w) {
    lo = min(lo, sm.red[w]);
    hi = max(hi, sm.red[kGW + w]);
  }
  g.sync();
}

// Exact select among keys held in shared memory: get(j, k) yields the key of
// slot j < nslots (false = empty slot); every key lies in [lo, hi] and at
// least `need` of them do.  Each round histograms the top kDigitBits bits of
// the remaining span and keeps the bin that holds the need-th largest key;
// once that bin has at most kSmall keys they are ranked against each other.
// Returns T; *take_eq = how many keys equal to T are taken.
template <typename SM, typename Get>
__device__ __forceinline__ uint32_t digit_select(const Group& g, SM& sm, uint32_t lo, uint32_t hi, uint32_t need,
                                                 int nslots, Get&& get, uint32_t* take_eq, int& parity) {
  const int tid = g.tid;
  while (true) {
    if (lo == hi) {
      *take_eq = need;
      return lo;
    }
    const uint32_t span = hi - lo;
    const int bits = 32 - __clz(span);
    const int sh = bits > kDigitBits ? bits - kDigitBits : 0;
    const uint32_t nb = (span >> sh) + 1u;
    for (uint32_t b = tid; b < nb; b += kGT) sm.hist[b] = 0u;
    if (tid == 0) sm.nsmall = 0u;
    g.sync();
    for (int j = tid; j < nslots; j += kGT) {
      uint32_t k;
      if (get(j, k) && k >= lo && k <= hi) atomicAdd(&sm.hist[(k - lo) >> sh], 1u);
    }
    g.sync();
    find_bin(g, sm.hist, sm, nb, need, parity);
    const uint32_t b = sm.sel[0], inbin = sm.sel[2];
    need -= sm.sel[1];
    const uint32_t nlo = lo + (b << sh);
    const uint64_t nhi = static_cast<uint64_t>(nlo) + ((1ull << sh) - 1ull);
    lo = nlo;
    hi = nhi < hi ? static_cast<uint32_t>(nhi) : hi;
    if (sh == 0) {  // the bin is one key value
      *take_eq = need;
      return lo;
    }
    if (inbin > static_cast<uint32_t>(kSmall)) continue;
    // few keys left in the bin (exactly inbin of them lie in [lo, hi])
    for (int j = tid; j < nslots; j += kGT) {
      uint32_t k;
      if (get(j, k) && k >= lo && k <= hi) sm.small[atomicAdd(&sm.nsmall, 1u)] = k;
    }
    g.sync();
    const int ns = static_cast<int>(sm.nsmall);
    if (tid < ns) {
      const uint32_t kj = sm.small[tid];
      uint32_t gt = 0, eq = 0;
      for (int q = 0; q < ns; ++q) {
        const uint32_t kq = sm.small[q];
        gt += kq > kj;
        eq += kq == kj;
      }
      if (gt < need && need <= gt + eq) {  // kj is T; every thread holding T writes the same values
        sm.sel[0] = kj;
        sm.sel[1] = need - gt;
      }
    }
    g.sync();
    *take_eq = sm.sel[1];
    return sm.sel[0];
  }
}

// keys of elements j .. j+3; elements >= n read as 0
__device__ __forceinline__ uint4 load_keys4(const float* srow, int j, int n) {
  if (j + 3 < n) {
    const float4 f = __ldcg(reinterpret_cast<const float4*>(srow + j));
    return make_uint4(score_key(f.x), score_key(f.y), score_key(f.z), score_key(f.w));
  }
  uint4 k;
  k.x = j < n ? score_key(__ldcg(srow + j)) : 0u;
  k.y = j + 1 < n ? score_key(__ldcg(srow + j + 1)) : 0u;
  k.z = j + 2 < n ? score_key(__ldcg(srow + j + 2)) : 0u;
  k.w = j + 3 < n ? score_key(__ldcg(srow + j + 3)) : 0u;
  return k;
}

// General path: histogram narrowing over the whole row, then a stable
// compaction pass (re-reads the scores).
__device__ __noinline__ void general(const Group& g, Smem& sm, const float* srow, int n, int topk, int32_t* orow,
                                     int& parity) {
  const int tid = g.tid;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int j = 4 * tid; j < n; j += kPerRound) {
    const uint4 k = load_keys4(srow, j, n);
    const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (j + q < n) {
        lo = min(lo, kk[q]);
        hi = max(hi, kk[q]);
      }
  }
  group_minmax(g, lo, hi, sm);
  uint32_t need = static_cast<uint32_t>(topk);
  uint32_t T = lo, take_eq = need;
  while (true) {
    if (lo == hi) {
      T = lo;
      take_eq = need;
      break;
    }
    const uint64_t range = static_cast<uint64_t>(hi - lo) + 1u;
    for (int b = tid; b < kGenBins; b += kGT) sm.u.gen.hist[b] = 0u;
    g.sync();
    for (int j = 4 * tid; j < n; j += kPerRound) {
      const uint4 k = load_keys4(srow, j, n);
      const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (j + q < n && kk[q] >= lo && kk[q] <= hi)
          atomicAdd(&sm.u.gen.hist[static_cast<uint32_t>((static_cast<uint64_t>(kk[q] - lo) * kGenBins) / range)],
                    1u);
    }
    g.sync();
    find_bin(g, sm.u.gen.hist, sm, kGenBins, need, parity);
    const uint32_t b = sm.sel[0], inbin = sm.sel[2];
    need -= sm.sel[1];
    const uint32_t nlo = lo + static_cast<uint32_t>((static_cast<uint64_t>(b) * range + kGenBins - 1) / kGenBins);
    const uint32_t nhi =
        lo + static_cast<uint32_t>((static_cast<uint64_t>(b + 1) * range + kGenBins - 1) / kGenBins) - 1u;
    lo = nlo;
    hi = nhi;
    g.sync();
    if (inbin > static_cast<uint32_t>(kGenBins)) continue;
    if (tid == 0) sm.ncand = 0;
    g.sync();
    for (int j = 4 * tid; j < n; j += kPerRound) {
      const uint4 k = load_keys4(srow, j, n);
      const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (j + q < n && kk[q] >= lo && kk[q] <= hi) sm.u.gen.cand[atomicAdd(&sm.ncand, 1u)] = kk[q];
    }
    g.sync();
    const int nc = static_cast<int>(sm.ncand);
    T = digit_select(
        g, sm, lo, hi, need, nc,
        [&](int j, uint32_t& k) {
          k = sm.u.gen.cand[j];
          return true;
        },
        &take_eq, parity);
    break;
  }
  g.sync();
  uint32_t gt_base = 0, eq_base = 0;
  const int rounds = (n + kPerRound - 1) / kPerRound;
  for (int m = 0; m < rounds; ++m) {
    const int j = m * kPerRound + 4 * tid;
    const uint4 k = j < n ? load_keys4(srow, j, n) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t kk[4] = {k.x, k.y, k.z, k.w};
    uint32_t gt[4], eq[4], c_gt = 0, c_eq = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bool v = j + q < n;
      gt[q] = v && kk[q] > T;
      eq[q] = v && kk[q] == T;
      c_gt += gt[q];
      c_eq += eq[q];
    }
    uint32_t tot;
    const uint32_t pre = group_excl_scan(g, (c_gt << 16) | c_eq, sm.wsum[parity], &tot);
    parity ^= 1;
    uint32_t gt_before = gt_base + (pre >> 16), eq_before = eq_base + (pre & 0xFFFFu);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (gt[q] || (eq[q] && eq_before < take_eq)) orow[gt_before + min(eq_before, take_eq)] = j + q;
      gt_before += gt[q];
      eq_before += eq[q];
    }
    gt_base += tot >> 16;
    eq_base += tot & 0xFFFFu;
  }
  g.sync();
}

// Top-k of one row: srow holds the n = floor(i/4) eligible scores of query i;
// writes orow[0 .. topk).  All threads of the group call it together; it ends
// with a group barrier (the shared buffers are reused by the next row).  A
// row that takes the general path adds one to *general_rows.
__device__ __noinline__ void row(const Group& g, Smem& sm, const float* srow, int n, int topk, int32_t* orow,
                                 unsigned long long* general_rows) {
  const int tid = g.tid, lane = g.lane(), warp = g.warp();
  if (n <= topk) {
    for (int j = tid; j < topk; j += kGT) orow[j] = j < n ? j : -1;
    return;
  }
  int parity = 0;
  // each warp owns the stretch [seg0, seg1) of the row, a multiple of 4 long
  const int seg = ((n + kGW - 1) / kGW + 3) & ~3;
  const int seg0 = min(n, warp * seg), seg1 = min(n, seg0 + seg);

  // ---- 1. threshold guess
  uint32_t t_lo = 0u;
  if (seg > kWarpCap) {
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    // kSample keys as kSample / 4 strided 16-byte quads (whole quads of the
    // row; n > 2048 here, so they are distinct), every load in flight at once
    constexpr int kQuads = kSample / 4, kQPer = kQuads / kGT;
    const int64_t nq = n >> 2;
    float4 sv[kQPer];
#pragma unroll
    for (int s = 0; s < kQPer; ++s)
      sv[s] = __ldcg(reinterpret_cast<const float4*>(srow) +
                     static_cast<int>((static_cast<int64_t>(tid + s * kGT) * nq) / kQuads));
#pragma unroll
    for (int s = 0; s < kQPer; ++s) {
      const uint32_t k4[4] = {score_key(sv[s].x), score_key(sv[s].y), score_key(sv[s].z), score_key(sv[s].w)};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        sm.u.samp[4 * (tid + s * kGT) + q] = k4[q];
        lo = min(lo, k4[q]);
        hi = max(hi, k4[q]);
      }
    }
    group_minmax(g, lo, hi, sm);  // its barriers also publish the samples
    // expected keys of the row above the r-th largest sample: r * n / kSample
    const float r0 = static_cast<float>(topk) * kSample / static_cast<float>(n);
    const uint32_t r = min(static_cast<uint32_t>(kSample),
                           static_cast<uint32_t>(ceilf(r0 + 4.f * sqrtf(r0) + 4.f)));
    t_lo = lo;
    if (hi > lo) {
      const uint32_t span = hi - lo;
      const int bits = 32 - __clz(span);
      const int sh = bits > kDigitBits ? bits - kDigitBits : 0;
      const uint32_t nb = (span >> sh) + 1u;
      for (uint32_t b = tid; b < nb; b += kGT) sm.hist[b] = 0u;
      g.sync();
      for (int s = 0; s < kSample / kGT; ++s) atomicAdd(&sm.hist[(sm.u.samp[tid + s * kGT] - lo) >> sh], 1u);
      g.sync();
      find_bin(g, sm.hist, sm, nb, r, parity);
      t_lo = lo + (sm.sel[0] << sh);
    }
    g.sync();  // the samples share storage with the candidate buffers
  }

  // ---- 2. one pass: per-warp candidate buffers in index order
  uint32_t cnt = 0, cmax = 0;
  // Scores are compared as floats against the threshold's float (the key
  // order is the float order, -0 and +0 being one key), and only candidates
  // are turned into keys.  A candidate's slot is the warp's count so far plus
  // the candidates of lower lanes (four ballots, one per quad element) plus
  // its own earlier ones: no shuffle chain.
  // Loads are plain 16-byte loads with no branch, issued a whole batch ahead
  // of the batch being compared; a load past the stretch is clamped to its
  // last aligned quad (rows are allocated in whole 256-float tiles, so the
  // quad is inside the row) and its elements are masked below.
  const float t_f = key_score(t_lo);
  const uint32_t lt = (1u << lane) - 1u;
  const int jmax = seg1 > 0 ? ((seg1 - 1) & ~3) : 0;
  float4 nx[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u)
    nx[u] = __ldcg(reinterpret_cast<const float4*>(srow + min(seg0 + 128 * u + 4 * lane, jmax)));
  for (int base = seg0; base < seg1; base += 128 * kBatch) {
    float4 fv[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      fv[u] = nx[u];
      nx[u] = __ldcg(reinterpret_cast<const float4*>(srow + min(base + 128 * (kBatch + u) + 4 * lane, jmax)));
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = base + 128 * u + 4 * lane;
      const float v[4] = {fv[u].x, fv[u].y, fv[u].z, fv[u].w};
      bool hit[4];
      uint32_t below = 0, total = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        hit[q] = j + q < seg1 && v[q] >= t_f;
        const uint32_t b = __ballot_sync(0xffffffffu, hit[q]);
        below += __popc(b & lt);
        total += __popc(b);
      }
      uint32_t pos = cnt + below;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (hit[q]) {
          if (pos < kWarpCap) {
            const uint32_t k = score_key(v[q]);
            sm.u.cand.key[warp][pos] = k;
            sm.u.cand.idx[warp][pos] = j + q;
            cmax = max(cmax, k);
          }
          ++pos;
        }
      cnt += total;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
  if (lane == 0) {
    sm.wcount[warp] = cnt;
    sm.wmax[warp] = cmax;
  }
  g.sync();
  uint32_t total = 0, hi = 0;
  bool overflow = false;
#pragma unroll
  for (int w = 0; w < kGW; ++w) {
    total += sm.wcount[w];
    overflow |= sm.wcount[w] > static_cast<uint32_t>(kWarpCap);
    hi = max(hi, sm.wmax[w]);
  }
  if (overflow || total < static_cast<uint32_t>(topk)) {
    if (tid == 0) atomicAdd(general_rows, 1ull);
    general(g, sm, srow, n, topk, orow, parity);
    return;
  }

  // ---- 3. exact select among the candidates
  uint32_t take_eq;
  const uint32_t T = digit_select(
      g, sm, t_lo, hi, topk, kGW * kWarpCap,
      [&](int j, uint32_t& k) {
        const int w = j / kWarpCap, p = j % kWarpCap;
        if (p >= static_cast<int>(sm.wcount[w])) return false;
        k = sm.u.cand.key[w][p];
        return true;
      },
      &take_eq, parity);

  // walk the candidates in index order: warp w takes its own buffer
  const int myc = static_cast<int>(sm.wcount[warp]);
  uint32_t c_gt = 0, c_eq = 0;
  for (int p = lane; p < myc; p += 32) {
    const uint32_t k = sm.u.cand.key[warp][p];
    c_gt += k > T;
    c_eq += k == T;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    c_gt += __shfl_xor_sync(0xffffffffu, c_gt, o);
    c_eq += __shfl_xor_sync(0xffffffffu, c_eq, o);
  }
  // exclusive prefix over warps of the packed (gt, eq) counts
  uint32_t tot;
  const uint32_t pre = group_excl_scan(g, lane == 31 ? ((c_gt << 16) | c_eq) : 0u, sm.wsum[parity], &tot);
  parity ^= 1;
  const uint32_t wpre = __shfl_sync(0xffffffffu, pre, 31);  // exclusive prefix of this warp's totals
  uint32_t gt_before = wpre >> 16, eq_before = wpre & 0xFFFFu;
  for (int p0 = 0; p0 < myc; p0 += 32) {
    const int p = p0 + lane;
    const bool v = p < myc;
    const uint32_t k = v ? sm.u.cand.key[warp][p] : 0u;
    const bool gt = v && k > T, eq = v && k == T;
    const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    const uint32_t below = (1u << lane) - 1u;
    const uint32_t g_pre = gt_before + __popc(bg & below), e_pre = eq_before + __popc(be & below);
    if (gt || (eq && e_pre < take_eq)) orow[g_pre + min(e_pre, take_eq)] = static_cast<int32_t>(sm.u.cand.idx[warp][p]);
    gt_before += __popc(bg);
    eq_before += __popc(be);
  }
  g.sync();
}

}  // namespace topk
}  // namespace dsa
