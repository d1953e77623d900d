// ts_warp.cuh -- warp-per-row sampler for rows of up to 4096 bf16 / 2048 fp32
// logits with a top-k cap of at most 64 (the serving configuration: top_k 30
// under the default cap 64, Drama 3 article sections "测试口径" and
// "能跑通的命令，和文档写明的边界").
//
// One block of 128 threads owns one row.  Fast path (every realistic row):
//   1. the row is read once with 16-byte streaming loads (thread t issues
//      chunks t, t+128, ..., all in flight at once); the Philox draw is
//      computed while they are in flight;
//   2. keys stay in registers (and are staged in shared memory for the slow
//      path) and feed a 1024-bin histogram of their top 10 bits (sign,
//      exponent and one mantissa bit: half-binade bins);
//   3. warp 0 finds the bin holding the k_eff-th largest key by a two-level
//      suffix scan; bins 0, 1022 and 1023 hold only NaN / +inf keys and bin 1
//      only -inf / NaN keys, so the same histogram validates the row; a
//      second 64-bin histogram over the next 6 key bits of that bin narrows
//      the threshold (for bf16 to the exact k_eff-th largest key);
//   4. every key at or above the threshold (k_eff plus any ties) is packed
//      with its index into one word (key high, inverted index low) and warp
//      0 bitonic-sorts the words: the first k_eff are the top-k set in
//      (logit desc, index asc) order, ties included;
//   5. warp 0 forms fixed-point weights, scans them, cuts the nucleus and
//      draws (the Philox draw itself is computed by warp 1 while warp 0
//      searches the histogram).
// Rows whose threshold would leave more than 128 candidates (huge ties) or
// whose threshold is -inf take an exact slow path on warp 0: 8-bit radix
// select over the staged keys with index-ordered tie ranking, then the same
// sort and tail.
#pragma once

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

// Exact slow path for rows the fast path declines (threshold at -inf, or a
// threshold bin with more than kWarpCandMax keys): 8-bit radix select over the
// staged keys, then the top-k set collected in index order (keys equal to
// the threshold taken by lowest index), sorted, and the common tail.
template <class K>
__device__ __noinline__ void warp_slow_path(const Params &p, int r, const Row &w, uint32_t *hist,
                                            typename SortWord<K>::T *cand, const uint4 *keys,
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
      const uint4 v = keys[q];
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
    if (q < nq) v = keys[q];
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

// Sorts the n (<= 32 * R) candidate words in `cand` and runs the tail.
template <class K, int R>
__device__ __forceinline__ void warp_sort_and_tail(const Params &p, int r, const Row &w,
                                                   const typename SortWord<K>::T *cand, int n,
                                                   uint32_t u24) {
  using T = typename SortWord<K>::T;
  const uint32_t lane = lane_id();
  T v[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int e = i * 32 + static_cast<int>(lane);
    v[i] = e < n ? cand[e] : T(0);
  }
  bitonic_desc<T, R>(v);
  T second = T(0);
  if constexpr (R > 1) second = v[1];
  warp_tail<K>(p, r, w, v[0], second, w.k_eff, u24);
}

// Histogram bin b lives at b + b / 32, so that a lane reading 32 consecutive
// bins touches 32 different banks.
__device__ __forceinline__ uint32_t hist_slot(uint32_t b) { return b + (b >> 5); }
constexpr int kRowHistWords = kWarpHistBins + kWarpHistBins / 32;

// Shared state of one row in a block.
constexpr int kSubBins = 64;  // second-level histogram: the next 6 key bits
template <class K>
struct RowShared {
  using T = typename SortWord<K>::T;
  uint32_t hist[kRowHistWords];
  uint32_t sub[kSubBins];
  T cand[kWarpCandMax];
  uint32_t n_cand;
  uint32_t b1;
  uint32_t above1;  // keys in bins above b1
  uint32_t thr;     // candidate threshold key after the second level
  uint32_t n_sel;   // keys >= thr
  uint32_t u24;
};

// One block of kRowThreads threads per row.
constexpr int kRowThreads = 128;

// The row body for rows of at most NCH 16-byte chunks per thread.
template <class K, int NCH>
__device__ __forceinline__ void row_body(const Params &p, int r, const Row &w, int64_t step,
                                         RowShared<K> &sh, uint4 *keys, int head, int nq,
                                         int tail, const char *rowp) {
  using SW = SortWord<K>;
  using T = typename SW::T;
  constexpr int EPC = K::kPerChunk;
  constexpr int kShift = K::kBits - 10;  // top 10 key bits select the bin
  constexpr int kShift2 = kShift - 6;    // the next 6 select the sub-bin
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t lane = lane_id();
  const int warp = t >> 5;
  const int V = w.vocab;
  const char *body = rowp + head * K::kElemBytes;
  const uint64_t pol = l2_evict_first();

  // ---- issue every load of the row (thread t: chunks t, t+128, ...) ----
  uint4 v[NCH];
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int q = t + kRowThreads * j;
    v[j] = make_uint4(0u, 0u, 0u, 0u);
    if (q < nq) v[j] = ld_stream_v4(body + static_cast<size_t>(q) * 16, pol);
  }
  int eidx = 0x7FFFFFFF;  // head / tail elements live in the first threads
  if (t < head)
    eidx = t;
  else if (t < head + tail)
    eidx = nq * EPC + t;
  uint32_t ebits = 0;
  if (eidx < V) ebits = K::load_one(rowp, eidx);
  __syncthreads();  // histograms cleared

  // ---- keys: to registers (packed) and shared memory; 10-bit histogram ----
  uint32_t c[NCH][4];
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int q = t + kRowThreads * j;
    c[j][0] = K::key_word(v[j].x);
    c[j][1] = K::key_word(v[j].y);
    c[j][2] = K::key_word(v[j].z);
    c[j][3] = K::key_word(v[j].w);
    if (q < nq) {
      keys[q] = make_uint4(c[j][0], c[j][1], c[j][2], c[j][3]);
#pragma unroll
      for (int e = 0; e < EPC; ++e) atomicAdd(&sh.hist[hist_slot(K::elem(c[j], e) >> kShift)], 1u);
    }
  }
  const uint32_t ekey = eidx < V ? K::key(ebits) : 0u;
  if (eidx < V) atomicAdd(&sh.hist[hist_slot(ekey >> kShift)], 1u);
  __syncthreads();

  // ---- validity: bins 0, 1022, 1023 hold only NaN/+inf keys; bin 1 holds
  // -inf and negative NaNs ----
  const uint32_t h_nan = sh.hist[hist_slot(0)] + sh.hist[hist_slot(kWarpHistBins - 2)] +
                         sh.hist[hist_slot(kWarpHistBins - 1)];
  const uint32_t h_ninf = sh.hist[hist_slot(1)];
  bool bad = h_nan != 0;
  if (!bad && h_ninf != 0) {  // uniform branch
    bool nan = false;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      if (t + kRowThreads * j < nq) {
#pragma unroll
        for (int e = 0; e < EPC; ++e) nan |= K::elem(c[j], e) < K::kNegInf;
      }
    }
    if (eidx < V) nan |= ekey < K::kNegInf;
    bad = __syncthreads_or(nan) != 0;
  }
  if (bad || static_cast<uint32_t>(V) == h_ninf) {
    if (t == 0) finish_row(p, r, w, -1, kRowNonFinite);
    return;
  }

  // ---- warp 0: the bin of the k_eff-th largest key; warp 1: the draw ----
  const uint32_t kk = static_cast<uint32_t>(w.k_eff);
  if (warp == 0) {
    const uint32_t *hb = &sh.hist[lane * 33];
    uint32_t part[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 32; ++i) part[i & 3] += hb[i];
    const uint32_t s = part[0] + part[1] + part[2] + part[3];
    const uint32_t suf = warp_incl_suffix_u32(s);
    const uint32_t big = 31 - __clz(__ballot_sync(0xFFFFFFFFu, suf >= kk));
    const uint32_t above_lane = __shfl_sync(0xFFFFFFFFu, suf - s, big);
    const uint32_t cb = sh.hist[big * 33 + lane];
    const uint32_t suf2 = warp_incl_suffix_u32(cb) + above_lane;
    const uint32_t sub = 31 - __clz(__ballot_sync(0xFFFFFFFFu, suf2 >= kk));
    const uint32_t above1 = __shfl_sync(0xFFFFFFFFu, suf2 - cb, sub);
    if (lane == 0) {
      sh.b1 = big * 32 + sub;
      sh.above1 = above1;
    }
  } else if (warp == 1 && lane == 0) {
    sh.u24 = philox_u24(p.seed[r], p.request[r], static_cast<uint64_t>(step),
                        static_cast<uint64_t>(static_cast<int64_t>(p.codebook[r])));
  }
  __syncthreads();
  const uint32_t b1 = sh.b1;
  if (b1 < 2) {  // threshold at -inf: exact slow path
    if (warp == 0)
      warp_slow_path<K>(p, r, w, sh.hist, sh.cand, keys, nq, head, tail, eidx, ekey, sh.u24);
    return;
  }

  // ---- second level inside bin b1: the next 6 key bits ----
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    if (t + kRowThreads * j < nq) {
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        const uint32_t k = K::elem(c[j], e);
        if ((k >> kShift) == b1) atomicAdd(&sh.sub[(k >> kShift2) & (kSubBins - 1)], 1u);
      }
    }
  }
  if (eidx < V && (ekey >> kShift) == b1)
    atomicAdd(&sh.sub[(ekey >> kShift2) & (kSubBins - 1)], 1u);
  __syncthreads();
  if (warp == 0) {
    const uint32_t kk2 = kk - sh.above1;  // ranks still needed inside bin b1
    const uint32_t lo = sh.sub[2 * lane], hi = sh.sub[2 * lane + 1];
    const uint32_t s = lo + hi;
    const uint32_t suf = warp_incl_suffix_u32(s);
    const uint32_t own = 31 - __clz(__ballot_sync(0xFFFFFFFFu, suf >= kk2));
    const uint32_t above_lane = suf - s;  // counts in sub-bins above this lane's pair
    // within the owning lane: sub-bin 2*own+1 first, then 2*own
    const bool top = above_lane + hi >= kk2;
    const uint32_t b2 = 2 * lane + (top ? 1u : 0u);
    const uint32_t n_sel = sh.above1 + (top ? above_lane + hi : suf);
    if (lane == own) {
      sh.thr = ((b1 << 6) | b2) << kShift2;
      sh.n_sel = n_sel;
    }
  }
  __syncthreads();
  const uint32_t tkey = sh.thr, n_sel = sh.n_sel;
  if (n_sel > static_cast<uint32_t>(kWarpCandMax)) {  // huge ties: exact slow path
    if (warp == 0)
      warp_slow_path<K>(p, r, w, sh.hist, sh.cand, keys, nq, head, tail, eidx, ekey, sh.u24);
    return;
  }

  // ---- every key >= tkey joins the candidates (any order: sorted next) ----
  uint32_t mine = 0;
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    if (t + kRowThreads * j < nq) {
#pragma unroll
      for (int e = 0; e < EPC; ++e) mine += K::elem(c[j], e) >= tkey;
    }
  }
  const bool e_in = eidx < V && ekey >= tkey;
  mine += e_in;
  if (mine) {
    uint32_t pos = atomicAdd(&sh.n_cand, mine);
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int q = t + kRowThreads * j;
      if (q < nq) {
#pragma unroll
        for (int e = 0; e < EPC; ++e) {
          const uint32_t k = K::elem(c[j], e);
          if (k >= tkey) {
            if (pos < static_cast<uint32_t>(kWarpCandMax))
              sh.cand[pos] = SW::make(k, static_cast<uint32_t>(head + q * EPC + e));
            ++pos;
          }
        }
      }
    }
    if (e_in && pos < static_cast<uint32_t>(kWarpCandMax))
      sh.cand[pos] = SW::make(ekey, static_cast<uint32_t>(eidx));
  }
  __syncthreads();
  if (warp != 0) return;
  const int nc = static_cast<int>(n_sel);
  if (nc <= 32)
    warp_sort_and_tail<K, 1>(p, r, w, sh.cand, nc, sh.u24);
  else if (nc <= 64)
    warp_sort_and_tail<K, 2>(p, r, w, sh.cand, nc, sh.u24);
  else
    warp_sort_and_tail<K, 4>(p, r, w, sh.cand, nc, sh.u24);
}

// MAXNCH = most 16-byte chunks per thread of any row in the launch; each row
// runs the body sized for its own width.
template <class K, int MAXNCH>
__global__ void __launch_bounds__(kRowThreads, 10) row_sampler_kernel(const Params p) {
  constexpr int EPC = K::kPerChunk;
  __shared__ __align__(16) RowShared<K> sh;
  __shared__ __align__(16) uint4 keys[MAXNCH * kRowThreads];
  const int r = static_cast<int>(blockIdx.x);
  const int t = static_cast<int>(threadIdx.x);
  pdl_wait_and_release();
  if (r >= p.n_rows) return;

  for (int i = t; i < kRowHistWords; i += kRowThreads) sh.hist[i] = 0u;
  if (t < kSubBins) sh.sub[t] = 0u;
  if (t == 0) sh.n_cand = 0;

  const Row w = load_row(p, r);
  if (w.err) {
    if (t == 0) finish_row(p, r, w, -1, w.err);
    return;
  }
  const int64_t step = (t >> 5) == 1 ? p.step[w.stream] : 0;  // for the draw (warp 1)
  const int V = w.vocab;
  const char *rowp = static_cast<const char *>(p.logits) + w.off * K::kElemBytes;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
  int head = static_cast<int>(((16u - (addr & 15u)) & 15u) / K::kElemBytes);
  head = min(head, V);
  const int nq = (V - head) / EPC;
  const int tail = V - head - nq * EPC;
  if (MAXNCH == 1 || nq <= kRowThreads)
    row_body<K, 1>(p, r, w, step, sh, keys, head, nq, tail, rowp);
  else if (MAXNCH == 2 || nq <= 2 * kRowThreads)
    row_body<K, (MAXNCH >= 2 ? 2 : 1)>(p, r, w, step, sh, keys, head, nq, tail, rowp);
  else
    row_body<K, MAXNCH>(p, r, w, step, sh, keys, head, nq, tail, rowp);
}

}  // namespace ts
