// ts_warp.cuh -- warp-per-row sampler for rows of up to 4096 bf16 / 2048 fp32
// logits with a top-k cap of at most 64 (the serving configuration: top_k 30
// under the default cap 64, Drama 3 article sections "测试口径" and
// "能跑通的命令，和文档写明的边界").
//
// One warp owns one row (four rows per 128-thread block, no block barrier).
// The row is staged in shared memory by asynchronous 16-byte copies; each
// lane's two largest logits give, through the k_eff-th largest of the 64
// per-lane maxima, a lower bound of the row's k_eff-th largest logit; the
// logits at or above it (the top-k set with all its ties, about 35 words for
// top_k 30 of 1024 gaussian logits) are bitonic-sorted by the warp as (key,
// inverted index) words, and the warp computes the fixed-point weights, the
// nucleus cutoff and the draw.  Rows with huge ties take an exact radix-select
// slow path over the staged keys.
#pragma once

#include <cuda_bf16.h>

#include "ts_device.cuh"

namespace ts {

constexpr int kWarpHistBins = 1024;
constexpr int kWarpCandMax = 128;

// Sort word: key in the high part, bit-inverted row index in the low part, so
// that descending word order is (key desc, index asc).  A zero word sorts
// after every real key (real keys are >= the -inf key).
template <class K>
struct SortWord;

template <>
struct SortWord<KeyBF16> {  // rows of at most 65536 tokens
  using T = uint32_t;
  __device__ __forceinline__ static T make(uint32_t key, uint32_t idx) {
    return (key << 16) | (0xFFFFu - idx);
  }
  __device__ __forceinline__ static uint32_t key(T w) { return w >> 16; }
  __device__ __forceinline__ static uint32_t idx(T w) { return 0xFFFFu - (w & 0xFFFFu); }
};

template <>
struct SortWord<KeyF32> {
  using T = unsigned long long;
  __device__ __forceinline__ static T make(uint32_t key, uint32_t idx) {
    return (static_cast<T>(key) << 32) | (0xFFFFFFFFu - idx);
  }
  __device__ __forceinline__ static uint32_t key(T w) { return static_cast<uint32_t>(w >> 32); }
  __device__ __forceinline__ static uint32_t idx(T w) {
    return 0xFFFFFFFFu - static_cast<uint32_t>(w);
  }
};

// Warp inclusive scan of a 64-bit value.
__device__ __forceinline__ uint64_t warp_incl_scan_u64(uint64_t v) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= static_cast<uint32_t>(o)) v += t;
  }
  return v;
}

__device__ __forceinline__ uint32_t warp_excl_scan_u32(uint32_t v, uint32_t *total) {
  const uint32_t lane = lane_id();
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= static_cast<uint32_t>(o)) x += t;
  }
  *total = __shfl_sync(0xFFFFFFFFu, x, 31);
  return x - v;
}

// Inclusive suffix sum over lanes (lane l gets the sum over lanes >= l).
__device__ __forceinline__ uint32_t warp_incl_suffix_u32(uint32_t v) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, v, o);
    if (lane + o < 32) v += t;
  }
  return v;
}

// Descending bitonic sort of 32*R words held as v[i] = element i*32 + lane.
template <class T, int R>
__device__ __forceinline__ void bitonic_desc(T (&v)[R]) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int size = 2; size <= 32 * R; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        const int jj = j >> 5;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          if ((i & jj) == 0) {
            const bool desc = ((i * 32) & size) == 0;
            const T a = v[i], b = v[i | jj];
            const T hi = a > b ? a : b, lo = a > b ? b : a;
            v[i] = desc ? hi : lo;
            v[i | jj] = desc ? lo : hi;
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const T o = __shfl_xor_sync(0xFFFFFFFFu, v[i], j);
          const bool lower = (lane & j) == 0;
          const bool desc = ((static_cast<uint32_t>(i * 32) + lane) & size) == 0;
          v[i] = (lower == desc) ? (v[i] > o ? v[i] : o) : (v[i] < o ? v[i] : o);
        }
      }
    }
  }
}

// Nucleus cutoff and draw over the sorted top-k set (positions lane and
// lane + 32 hold s0 and s1; k_eff = kq <= 64), then the outputs.
template <class K>
__device__ __forceinline__ void warp_tail(const Params &p, int r, const Row &w,
                                          typename SortWord<K>::T s0,
                                          typename SortWord<K>::T s1, int kq, uint32_t u24) {
  using SW = SortWord<K>;
  const uint32_t lane = lane_id();
  const float m = K::value(SW::key(__shfl_sync(0xFFFFFFFFu, s0, 0)));
  const bool has1 = kq > 32;
  const int p0 = static_cast<int>(lane), p1 = static_cast<int>(lane) + 32;
  float w0 = 0.f, w1 = 0.f;
  if (!w.greedy) {
    if (p0 < kq) w0 = kept_weight(K::value(SW::key(s0)), m, w.temp, w.inv_temp);
    if (has1 && p1 < kq) w1 = kept_weight(K::value(SW::key(s1)), m, w.temp, w.inv_temp);
  }
  // prefix masses in 2^-40 units, as four interleaved 32-bit scans of the
  // 20-bit halves (sums of 64 halves stay below 2^27)
  const uint64_t f0 = to_fixed(w0), f1 = to_fixed(w1);
  uint32_t h0 = static_cast<uint32_t>(f0 >> 20), l0 = static_cast<uint32_t>(f0 & 0xFFFFFu);
  uint32_t h1 = static_cast<uint32_t>(f1 >> 20), l1 = static_cast<uint32_t>(f1 & 0xFFFFFu);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t a = __shfl_up_sync(0xFFFFFFFFu, h0, o), b = __shfl_up_sync(0xFFFFFFFFu, l0, o);
    const uint32_t cc = __shfl_up_sync(0xFFFFFFFFu, h1, o), d = __shfl_up_sync(0xFFFFFFFFu, l1, o);
    if (lane >= static_cast<uint32_t>(o)) {
      h0 += a;
      l0 += b;
      h1 += cc;
      l1 += d;
    }
  }
  const uint64_t c0 = (static_cast<uint64_t>(h0) << 20) + l0;
  const uint64_t tot0 = __shfl_sync(0xFFFFFFFFu, c0, 31);
  const uint64_t c1 = (static_cast<uint64_t>(h1) << 20) + l1 + tot0;
  const uint64_t s_k = __shfl_sync(0xFFFFFFFFu, c1, 31);

  int n_p = 1, pick = 0;
  if (!w.greedy) {
    if (w.top_p >= 1.0f) {
      n_p = kq;
    } else if (w.top_p > 0.0f) {
      const uint64_t cut_i = ceil_mul_p(w.top_p, s_k);  // C reaches top_p * S_k iff C >= cut_i
      const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, p0 < kq && c0 < cut_i);
      const uint32_t b1 = __ballot_sync(0xFFFFFFFFu, p1 < kq && c1 < cut_i);
      n_p = min(__popc(b0) + __popc(b1) + 1, kq);
    }
    const int last = n_p - 1;
    const uint64_t s_p = last < 32 ? __shfl_sync(0xFFFFFFFFu, c0, last)
                                   : __shfl_sync(0xFFFFFFFFu, c1, last - 32);
    const uint64_t target = scale_u24(u24, s_p);
    const uint32_t le0 = __ballot_sync(0xFFFFFFFFu, p0 < n_p && c0 <= target);
    const uint32_t le1 = __ballot_sync(0xFFFFFFFFu, p1 < n_p && c1 <= target);
    pick = __popc(le0) + __popc(le1);
  }
  const typename SW::T pw = pick < 32 ? __shfl_sync(0xFFFFFFFFu, s0, pick)
                                      : __shfl_sync(0xFFFFFFFFu, s1, pick - 32);
  if (lane == 0) finish_row(p, r, w, static_cast<int32_t>(SW::idx(pw)), 0u);

  if (p.kept_ids) {
    const float s_real = static_cast<float>(static_cast<double>(s_k) * (1.0 / 1099511627776.0));
    const int64_t rb = static_cast<int64_t>(r) * p.max_keep;
    if (p0 < kq && p0 < p.max_keep) {
      p.kept_ids[rb + p0] = static_cast<int32_t>(SW::idx(s0));
      p.kept_probs[rb + p0] = w.greedy ? (p0 == 0 ? 1.f : 0.f) : __fdiv_rn(w0, s_real);
    }
    if (has1 && p1 < kq && p1 < p.max_keep) {
      p.kept_ids[rb + p1] = static_cast<int32_t>(SW::idx(s1));
      p.kept_probs[rb + p1] = w.greedy ? 0.f : __fdiv_rn(w1, s_real);
    }
    if (lane == 0) {
      p.n_kept[r] = kq;
      p.n_nucleus[r] = n_p;
    }
  }
}

// Exact slow path for rows the fast path declines (more than kWarpCandMax
// keys at or above the candidate threshold, i.e. huge ties): 8-bit radix
// select over the row's keys (keys(q) returns the keys of body chunk q, read
// again from memory), then the top-k set collected in index order (keys
// equal to the threshold taken by lowest index), sorted, and the common tail.
template <class K, class Loader>
__device__ __noinline__ void warp_slow_path(const Params &p, int r, const Row &w, uint32_t *hist,
                                            typename SortWord<K>::T *cand, const Loader keys,
                                            int nq, int head, int tail, int eidx, uint32_t ekey,
                                            uint32_t u24) {
  using SW = SortWord<K>;
  constexpr int EPC = K::kPerChunk;
  const uint32_t lane = lane_id();
  const int rounds = (nq + 31) >> 5;

  uint32_t prefix = 0, pmask = 0;
  uint32_t kk = static_cast<uint32_t>(w.k_eff);
#pragma unroll 1
  for (int pass = 0; pass < K::kBits / 8; ++pass) {
    const int shift = K::kBits - 8 * (pass + 1);
    reinterpret_cast<uint4 *>(hist)[lane * 2] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4 *>(hist)[lane * 2 + 1] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
#pragma unroll 1
    for (int q = static_cast<int>(lane); q < nq; q += 32) {
      const uint4 v = keys(q);
      const uint32_t c[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        const uint32_t k = K::elem(c, e);
        if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFFu], 1u);
      }
    }
    if (eidx < w.vocab && (ekey & pmask) == prefix)
      atomicAdd(&hist[(ekey >> shift) & 0xFFu], 1u);
    __syncwarp();
    const uint4 h0 = reinterpret_cast<const uint4 *>(hist)[lane * 2];
    const uint4 h1 = reinterpret_cast<const uint4 *>(hist)[lane * 2 + 1];
    const uint32_t hb[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    uint32_t s = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) s += hb[b];
    const uint32_t suf = warp_incl_suffix_u32(s);
    const uint32_t owner = 31 - __clz(__ballot_sync(0xFFFFFFFFu, suf >= kk));
    uint32_t run = suf - s, dsel = 0, asel = 0;
    bool found = false;
#pragma unroll
    for (int b = 7; b >= 0; --b) {
      const bool hit = !found && run + hb[b] >= kk;
      if (hit) {
        dsel = lane * 8 + b;
        asel = run;
      }
      found |= hit;
      run += hb[b];
    }
    dsel = __shfl_sync(0xFFFFFFFFu, dsel, owner);
    asel = __shfl_sync(0xFFFFFFFFu, asel, owner);
    kk -= asel;
    prefix |= dsel << shift;
    pmask |= 0xFFu << shift;
    __syncwarp();
  }
  const uint32_t thr = prefix;  // k_eff-th largest key
  const uint32_t need = kk;     // keys equal to thr that are kept

  uint32_t base = 0, eq_base = 0;
  const uint32_t lt = lanemask_lt();
  const bool has_e = eidx < w.vocab;
  {  // head elements (indices 0 .. head-1 live in lanes 0 .. head-1)
    const bool in = has_e && static_cast<int>(lane) < head;
    const bool gt = in && ekey > thr, eq = in && ekey == thr;
    const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, eq);
    const bool take = gt || (eq && eq_base + __popc(eqm & lt) < need);
    const uint32_t sm = __ballot_sync(0xFFFFFFFFu, take);
    const uint32_t at = base + __popc(sm & lt);
    if (take && at < 64) cand[at] = SW::make(ekey, static_cast<uint32_t>(eidx));
    base += __popc(sm);
    eq_base += __popc(eqm);
  }
#pragma unroll 1
  for (int j = 0; j < rounds; ++j) {
    const int q = static_cast<int>(lane) + 32 * j;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (q < nq) v = keys(q);
    const uint32_t c[4] = {v.x, v.y, v.z, v.w};
    uint32_t ng = 0, ne = 0;
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
      const uint32_t k = K::elem(c, e);
      ng += k > thr;
      ne += k == thr;
    }
    if (__ballot_sync(0xFFFFFFFFu, (ng | ne) != 0) == 0) continue;
    uint32_t eq_tot, eqr = warp_excl_scan_u32(ne, &eq_tot) + eq_base;
    uint32_t ns = ng, er = eqr;
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
      if (K::elem(c, e) == thr) {
        ns += er < need;
        ++er;
      }
    }
    uint32_t sel_tot, pos = warp_excl_scan_u32(ns, &sel_tot) + base;
    const uint32_t idx0 = static_cast<uint32_t>(head + q * EPC);
    er = eqr;
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
      const uint32_t k = K::elem(c, e);
      bool take = k > thr;
      if (k == thr) {
        take = er < need;
        ++er;
      }
      if (take) {
        if (pos < 64) cand[pos] = SW::make(k, idx0 + e);
        ++pos;
      }
    }
    base += sel_tot;
    eq_base += eq_tot;
  }
  {  // tail elements, in lane order after the chunks
    const bool in = has_e && static_cast<int>(lane) >= head && static_cast<int>(lane) < head + tail;
    const bool gt = in && ekey > thr, eq = in && ekey == thr;
    const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, eq);
    const bool take = gt || (eq && eq_base + __popc(eqm & lt) < need);
    const uint32_t sm = __ballot_sync(0xFFFFFFFFu, take);
    const uint32_t at = base + __popc(sm & lt);
    if (take && at < 64) cand[at] = SW::make(ekey, static_cast<uint32_t>(eidx));
  }
  __syncwarp();
  const int kq = w.k_eff;
  typename SW::T s[2];
  s[0] = static_cast<int>(lane) < kq ? cand[lane] : 0;
  s[1] = static_cast<int>(lane) + 32 < kq ? cand[lane + 32] : 0;
  __syncwarp();
  if (kq <= 32) {
    typename SW::T one[1] = {s[0]};
    bitonic_desc<typename SW::T, 1>(one);
    s[0] = one[0];
  } else {
    bitonic_desc<typename SW::T, 2>(s);
  }
  warp_tail<K>(p, r, w, s[0], s[1], kq, u24);
}

// Sorts the n (<= 32 * R) candidate words in `cand`; s0 / s1 get the first
// 64 in descending order (lane l holds positions l and l + 32).
template <class K, int R>
__device__ __forceinline__ void warp_sort_cand(const typename SortWord<K>::T *cand, int n,
                                               typename SortWord<K>::T &s0,
                                               typename SortWord<K>::T &s1) {
  using T = typename SortWord<K>::T;
  const uint32_t lane = lane_id();
  T v[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int e = i * 32 + static_cast<int>(lane);
    v[i] = e < n ? cand[e] : T(0);
  }
  bitonic_desc<T, R>(v);
  s0 = v[0];
  s1 = T(0);
  if constexpr (R > 1) s1 = v[1];
}

// Warp-path kernel.  A row is owned by one warp, or shared by 2 or 4 warps
// (kTowerWarps / WPR rows per block; the warps of a row meet at a named
// barrier of their own, never at a block barrier):
//   1. the row is copied into its shared-memory stage with 16-byte
//      asynchronous copies (lane l: body chunks l, l + 32, ...), all in
//      flight at once; the unaligned head and tail elements are read one per
//      lane; lane 0 computes the Philox draw meanwhile;
//   2. each lane keeps the two largest logits it has seen (packed bf16 or
//      fp32 min / max); the k_eff-th largest of these 64 values t0 is a lower
//      bound of the row's k_eff-th largest logit (at least k_eff of the row's
//      logits are >= t0), so every logit >= t0 is a candidate and the
//      candidates hold the whole top-k set with every tie at its end;
//   3. an unordered compare with t0 (so that a NaN is flagged too) marks the
//      chunks that hold a candidate; only those are unpacked into (key,
//      inverted index) words, about 35 for top_k 30 of 1024 gaussian logits,
//      which the warp bitonic-sorts: the first k_eff are the top-k set in
//      (logit desc, index asc) order;
//   4. the warp forms fixed-point weights, scans them, cuts the nucleus and
//      draws.
// Rows with more than kWarpCandMax candidates (huge ties) take the exact
// radix-select slow path over the staged keys.
constexpr int kTowerWarps = 4;
constexpr int kTowerThreads = 32 * kTowerWarps;
constexpr int kRowThreads = kTowerThreads;


// Per-dtype chunk helpers: the two largest values of a chunk folded into a
// running pair, and the unordered >= mask of a chunk against a threshold.
template <class K>
struct Top2;

template <>
struct Top2<KeyBF16> {
  using V = uint32_t;  // packed bf16x2
  static constexpr uint32_t kInit = 0xFF80FF80u;  // -inf, -inf
  __device__ __forceinline__ static __nv_bfloat162 b2(uint32_t x) {
    return *reinterpret_cast<__nv_bfloat162 *>(&x);
  }
  __device__ __forceinline__ static uint32_t u(__nv_bfloat162 x) {
    return *reinterpret_cast<uint32_t *>(&x);
  }
  __device__ __forceinline__ static void fold(uint32_t w, uint32_t &m1, uint32_t &m2) {
    m2 = u(__hmax2(b2(m2), __hmin2(b2(m1), b2(w))));
    m1 = u(__hmax2(b2(m1), b2(w)));
  }
  __device__ __forceinline__ static void fold_chunk(const uint4 &c, uint32_t &m1, uint32_t &m2) {
    fold(c.x, m1, m2);
    fold(c.y, m1, m2);
    fold(c.z, m1, m2);
    fold(c.w, m1, m2);
  }
  // (m1, m2) <- the two largest of the pairs (m1, m2) and (n1, n2), per half
  __device__ __forceinline__ static void merge(uint32_t &m1, uint32_t &m2, uint32_t n1,
                                               uint32_t n2) {
    m2 = u(__hmax2(__hmin2(b2(m1), b2(n1)), __hmax2(b2(m2), b2(n2))));
    m1 = u(__hmax2(b2(m1), b2(n1)));
  }
  // the lane's two largest keys from the packed pair
  __device__ __forceinline__ static void keys2(uint32_t m1, uint32_t m2, uint32_t &k1,
                                               uint32_t &k2) {
    const uint32_t a = KeyBF16::key(m1 & 0xFFFFu), b = KeyBF16::key(m1 >> 16);
    const uint32_t c = KeyBF16::key(m2 & 0xFFFFu), d = KeyBF16::key(m2 >> 16);
    k1 = max(a, b);
    k2 = max(min(a, b), max(c, d));
  }
  __device__ __forceinline__ static uint32_t splat(uint32_t key) {
    const uint32_t bits = key ^ ((key & 0x8000u) ? 0x8000u : 0xFFFFu);
    return bits | (bits << 16);
  }
  __device__ __forceinline__ static bool flagged(const uint4 &c, uint32_t t2) {
    const uint32_t m = __hgeu2_mask(b2(c.x), b2(t2)) | __hgeu2_mask(b2(c.y), b2(t2)) |
                       __hgeu2_mask(b2(c.z), b2(t2)) | __hgeu2_mask(b2(c.w), b2(t2));
    return m != 0u;
  }
};

template <>
struct Top2<KeyF32> {
  static constexpr uint32_t kInit = 0xFF800000u;  // -inf
  __device__ __forceinline__ static void fold(uint32_t w, uint32_t &m1, uint32_t &m2) {
    const float x = __uint_as_float(w), a = __uint_as_float(m1), b = __uint_as_float(m2);
    m2 = __float_as_uint(fmaxf(b, fminf(a, x)));
    m1 = __float_as_uint(fmaxf(a, x));
  }
  __device__ __forceinline__ static void fold_chunk(const uint4 &c, uint32_t &m1, uint32_t &m2) {
    fold(c.x, m1, m2);
    fold(c.y, m1, m2);
    fold(c.z, m1, m2);
    fold(c.w, m1, m2);
  }
  __device__ __forceinline__ static void merge(uint32_t &m1, uint32_t &m2, uint32_t n1,
                                               uint32_t n2) {
    const float a = __uint_as_float(m1), c = __uint_as_float(m2);
    const float x = __uint_as_float(n1), y = __uint_as_float(n2);
    m2 = __float_as_uint(fmaxf(fminf(a, x), fmaxf(c, y)));
    m1 = __float_as_uint(fmaxf(a, x));
  }
  __device__ __forceinline__ static void keys2(uint32_t m1, uint32_t m2, uint32_t &k1,
                                               uint32_t &k2) {
    k1 = KeyF32::key(m1);
    k2 = KeyF32::key(m2);
  }
  __device__ __forceinline__ static uint32_t splat(uint32_t key) {
    return key ^ ((key & 0x80000000u) ? 0x80000000u : 0xFFFFFFFFu);
  }
  __device__ __forceinline__ static bool flagged(const uint4 &c, uint32_t t) {
    const float tv = __uint_as_float(t);
    return !(__uint_as_float(c.x) < tv) || !(__uint_as_float(c.y) < tv) ||
           !(__uint_as_float(c.z) < tv) || !(__uint_as_float(c.w) < tv);
  }
};

template <class K, int MAXNCH>
struct TowerShared {
  using T = typename SortWord<K>::T;
  uint4 stage[32 * MAXNCH];
  T cand[kWarpCandMax];
  uint32_t hist[256];
  uint32_t xm1[4 * 32];  // per-lane running pairs of each warp (rows shared by warps)
  uint32_t xm2[4 * 32];
  uint32_t xb[4];    // the row's candidate bound and largest key
  uint32_t xt[4];
  uint32_t xn[4];    // per-warp candidate counts
  uint32_t xu;       // the row's draw (computed by warp 1 when the row has several)
  uint32_t xbad[4];  // per-warp NaN / +inf flags
};

// Barrier of the WPR warps that share a row (group grp of the block).
template <int WPR>
__device__ __forceinline__ void row_sync(int grp) {
  if constexpr (WPR == 1) {
    __syncwarp();
  } else if constexpr (WPR == 4) {
    asm volatile("bar.sync 1, 128;" ::: "memory");
  } else {  // two rows per block: barriers 1 and 2 (constant ids)
    if (grp == 0)
      asm volatile("bar.sync 1, 64;" ::: "memory");
    else
      asm volatile("bar.sync 2, 64;" ::: "memory");
  }
}

// The row body for rows of at most 32 * nch body chunks (nch <= 16).  One
// body serves every row width, so that warps on other widths share its code
// in the instruction cache.  With WPR > 1 the row is shared by WPR warps:
// warp `sub` owns the chunk columns j = sub, sub + WPR, ...; lane l's running
// pairs of all the warps are merged, so the bound is the one a single warp
// would find; the candidate counts are exchanged so that every warp writes
// its candidates to its own range, and warp 0 sorts and runs the tail.
template <class K, int WPR, class SH>
__device__ __forceinline__ void tower_body(const Params &p, int r, const Row &w, uint32_t u24,
                                           SH &sh, int head, int nq, int tail, const char *rowp,
                                           int nch, int sub, int grp) {
  // u24: the draw when WPR == 1; with several warps it arrives below
  using SW = SortWord<K>;
  using TT = Top2<K>;
  constexpr int EPC = K::kPerChunk;
  const uint32_t lane = lane_id();
  const int V = w.vocab;
  const char *body = rowp + head * K::kElemBytes;
  // ---- this warp's columns into the stage, all copies in flight ----
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int j = sub + i * WPR;
    if (j >= nch) break;
    const int q = static_cast<int>(lane) + 32 * j;
    if (q < nq) cp_async16(&sh.stage[q], body + static_cast<size_t>(q) * 16);
  }
  // head / tail element of this lane of warp 0 (at most 7 + 7 of them)
  int eidx = 0x7FFFFFFF;
  if (sub == 0) {
    if (static_cast<int>(lane) < head)
      eidx = static_cast<int>(lane);
    else if (static_cast<int>(lane) < head + tail)
      eidx = nq * EPC + static_cast<int>(lane);
  }
  const bool has_e = eidx < V;
  const uint32_t ebits = has_e ? K::load_one(rowp, eidx) : 0u;
  if constexpr (WPR > 1) {
    // the draw, by warp 1 while its copies are in flight: off warp 0's path
    if (sub == 1 && lane == 0 && !w.greedy)
      sh.xu = philox_u24(p.seed[r], p.request[r], static_cast<uint64_t>(p.step[w.stream]),
                         static_cast<uint64_t>(static_cast<int64_t>(p.codebook[r])));
  }
  const uint32_t ekey = has_e ? K::key(ebits) : 0u;
  cp_async_wait_all();
  __syncwarp();

  // ---- the two largest logits per lane ----
  uint32_t m1 = TT::kInit, m2 = TT::kInit;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int j = sub + i * WPR;
    if (j >= nch) break;
    const int q = static_cast<int>(lane) + 32 * j;
    if (q < nq) TT::fold_chunk(sh.stage[q], m1, m2);
  }
  if constexpr (WPR > 1) {
    sh.xm1[sub * 32 + lane] = m1;
    sh.xm2[sub * 32 + lane] = m2;
    row_sync<WPR>(grp);
    if (!w.greedy) u24 = sh.xu;  // written by warp 1 before this barrier
  }
  const int kq = w.k_eff;
  uint32_t t0 = 0, top = 0;
  if (sub == 0) {
    if constexpr (WPR > 1) {
#pragma unroll
      for (int s2 = 1; s2 < WPR; ++s2) TT::merge(m1, m2, sh.xm1[s2 * 32 + lane], sh.xm2[s2 * 32 + lane]);
    }
    uint32_t rep[2];
    TT::keys2(m1, m2, rep[0], rep[1]);
    if (has_e) {  // the lane's head / tail element joins its pair
      rep[1] = max(rep[1], min(rep[0], ekey));
      rep[0] = max(rep[0], ekey);
    }
    // ---- the k_eff-th largest of the 64 per-lane maxima: a lower bound ----
    bitonic_desc<uint32_t, 2>(rep);
    top = __shfl_sync(0xFFFFFFFFu, rep[0], 0);
    t0 = kq <= 32 ? __shfl_sync(0xFFFFFFFFu, rep[0], kq - 1)
                  : __shfl_sync(0xFFFFFFFFu, rep[1], kq - 33);
    // a NaN as t0 would flag nothing (NaN rows are caught below either way)
    if (t0 < K::kNegInf || t0 > K::kPosInf) t0 = K::kNegInf;
    if constexpr (WPR > 1) {
      if (lane == 0) {
        sh.xb[0] = t0;
        sh.xt[0] = top;
      }
    }
  }
  if constexpr (WPR > 1) {
    row_sync<WPR>(grp);
    t0 = sh.xb[0];
    top = sh.xt[0];
  }
  const uint32_t t2 = TT::splat(t0);
  // ---- candidates: chunks holding a logit >= t0 (or a NaN) ----
  uint32_t fmask = 0;  // bit i: chunk lane + 32 (sub + i WPR) is flagged
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int j = sub + i * WPR;
    if (j >= nch) break;
    const int q = static_cast<int>(lane) + 32 * j;
    if (q < nq && TT::flagged(sh.stage[q], t2)) fmask |= 1u << i;
  }
  // keys of the flagged chunks: count, then write
  uint32_t mine = 0, bad = 0;
  for (uint32_t fm = fmask; fm; fm &= fm - 1u) {
    const int q = static_cast<int>(lane) + 32 * (sub + (__ffs(fm) - 1) * WPR);
    const uint4 v = sh.stage[q];
    const uint32_t c[4] = {K::key_word(v.x), K::key_word(v.y), K::key_word(v.z), K::key_word(v.w)};
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
      const uint32_t k = K::elem(c, e);
      bad |= (k < K::kNegInf) | (k > K::kPosInf - 1u);
      mine += k >= t0 && k < K::kPosInf;
    }
  }
  if (has_e) {
    bad |= (ekey < K::kNegInf) | (ekey >= K::kPosInf);
    mine += ekey >= t0 && ekey < K::kPosInf;
  }
  uint32_t total;
  uint32_t pos = warp_excl_scan_u32(mine, &total);
  bool any_bad = __any_sync(0xFFFFFFFFu, bad);
  if constexpr (WPR > 1) {
    if (lane == 0) {
      sh.xn[sub] = total;
      sh.xbad[sub] = any_bad ? 1u : 0u;
    }
    row_sync<WPR>(grp);
    total = 0;
#pragma unroll
    for (int s2 = 0; s2 < WPR; ++s2) {
      const uint32_t n2 = sh.xn[s2];
      if (s2 < sub) pos += n2;
      total += n2;
      any_bad |= sh.xbad[s2] != 0u;
    }
  }
  if (any_bad || top <= K::kNegInf) {  // a NaN / +inf, or no finite logit
    if (sub == 0 && lane == 0) finish_row(p, r, w, -1, kRowNonFinite);
    return;
  }
  if (total > static_cast<uint32_t>(kWarpCandMax)) {
    // every warp of the row has staged its columns (the exchange above
    // ordered them), so warp 0 may read the whole row
    if (sub != 0) return;
    auto keys = [&](int q) {
      const uint4 v = sh.stage[q];
      return make_uint4(K::key_word(v.x), K::key_word(v.y), K::key_word(v.z), K::key_word(v.w));
    };
    warp_slow_path<K>(p, r, w, sh.hist, sh.cand, keys, nq, head, tail, eidx, ekey, u24);
    return;
  }
  for (uint32_t fm = fmask; fm; fm &= fm - 1u) {
    const int q = static_cast<int>(lane) + 32 * (sub + (__ffs(fm) - 1) * WPR);
    const uint4 v = sh.stage[q];
    const uint32_t c[4] = {K::key_word(v.x), K::key_word(v.y), K::key_word(v.z), K::key_word(v.w)};
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
      const uint32_t k = K::elem(c, e);
      if (k >= t0) sh.cand[pos++] = SW::make(k, static_cast<uint32_t>(head + q * EPC + e));
    }
  }
  if (has_e && ekey >= t0) sh.cand[pos] = SW::make(ekey, static_cast<uint32_t>(eidx));
  row_sync<WPR>(grp);
  if (sub != 0) return;
  const int nc = static_cast<int>(total);
  typename SortWord<K>::T s0, s1;
  if (nc <= 32)
    warp_sort_cand<K, 1>(sh.cand, nc, s0, s1);
  else if (nc <= 64)
    warp_sort_cand<K, 2>(sh.cand, nc, s0, s1);
  else
    warp_sort_cand<K, 4>(sh.cand, nc, s0, s1);
  warp_tail<K>(p, r, w, s0, s1, w.k_eff, u24);
}

// MAXNCH = most 16-byte chunks per lane of any row in the launch (1, 2, 4, 8
// or 16) sizes the shared-memory stage; every row runs the same body with
// its own chunk count.  WPR = warps per row (1, 2 or 4): a block of four
// warps samples 4 / WPR rows.
template <class K, int MAXNCH, int WPR>
__global__ void __launch_bounds__(kTowerThreads, WPR == 4 ? 9 : 1) row_sampler_kernel(const Params p) {
  constexpr int EPC = K::kPerChunk;
  constexpr int RPB = kTowerWarps / WPR;
  __shared__ __align__(16) TowerShared<K, MAXNCH> shared_rows[RPB];
  const int warp = static_cast<int>(threadIdx.x) >> 5;
  const int grp = warp / WPR, sub = warp % WPR;
  const uint32_t lane = lane_id();
  const int r = static_cast<int>(blockIdx.x) * RPB + grp;
  pdl_wait_and_release();
  if (r >= p.n_rows) return;  // every warp of the row: its barriers are not reached
  const Row w = load_row(p, r);
  if (w.err) {
    if (sub == 0 && lane == 0) finish_row(p, r, w, -1, w.err);
    return;
  }
  const int V = w.vocab;
  const char *rowp = static_cast<const char *>(p.logits) + w.off * K::kElemBytes;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
  int head = static_cast<int>(((16u - (addr & 15u)) & 15u) / K::kElemBytes);
  head = min(head, V);
  const int nq = (V - head) / EPC;
  const int tail = V - head - nq * EPC;
  TowerShared<K, MAXNCH> &sh = shared_rows[grp];
  // the draw, on lane 0 (its result is needed only by the tail); a row
  // shared by several warps has warp 1 compute it inside the body
  uint32_t u24 = 0;
  if (WPR == 1 && lane == 0 && !w.greedy)
    u24 = philox_u24(p.seed[r], p.request[r], static_cast<uint64_t>(p.step[w.stream]),
                     static_cast<uint64_t>(static_cast<int64_t>(p.codebook[r])));
  u24 = __shfl_sync(0xFFFFFFFFu, u24, 0);
  tower_body<K, WPR>(p, r, w, u24, sh, head, nq, tail, rowp, min((nq + 31) >> 5, MAXNCH), sub,
                     grp);
}

}  // namespace ts
