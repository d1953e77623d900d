// ts_warp.cuh -- warp-per-row sampler for rows of up to 4096 bf16 / 2048 fp32
// logits with a top-k cap of at most 64 (the serving configuration: top_k 30
// under the default cap 64, Drama 3 article sections "测试口径" and
// "能跑通的命令，和文档写明的边界").
//
// One warp owns one row.  The row is read once with 16-byte streaming loads
// (lane l issues chunks l, l+32, ..., all in flight at once), turned into
// order-preserving keys in a per-warp shared-memory buffer, and the k-th
// largest key is found by 8-bit radix select over a per-warp histogram (no
// sort of the row).  The
// k_eff <= 64 survivors (ties at the threshold taken by lowest index) are
// bitonic-sorted across the warp by (key desc, index asc); the warp then
// forms fixed-point weights, scans them, cuts the nucleus and draws.
#pragma once

#include "ts_device.cuh"

namespace ts {

constexpr int kWarpRowsPerBlock = 8;

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

// Descending bitonic sort of one 64-bit value per lane.
__device__ __forceinline__ uint64_t bitonic32_desc(uint64_t v) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, v, j);
      const bool lower = (lane & j) == 0;
      const bool desc = (lane & size) == 0;
      v = (lower == desc) ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// Descending bitonic sort of 64 values: v0 at position lane, v1 at lane + 32.
__device__ __forceinline__ void bitonic64_desc(uint64_t &v0, uint64_t &v1) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      if (j == 32) {
        const uint64_t hi = v0 > v1 ? v0 : v1, lo = v0 > v1 ? v1 : v0;
        v0 = hi;
        v1 = lo;
      } else {
        const uint64_t o0 = __shfl_xor_sync(0xFFFFFFFFu, v0, j);
        const uint64_t o1 = __shfl_xor_sync(0xFFFFFFFFu, v1, j);
        const bool lower = (lane & j) == 0;
        const bool d0 = (lane & size) == 0;
        const bool d1 = ((lane + 32) & size) == 0;
        v0 = (lower == d0) ? (v0 > o0 ? v0 : o0) : (v0 < o0 ? v0 : o0);
        v1 = (lower == d1) ? (v1 > o1 ? v1 : o1) : (v1 < o1 ? v1 : o1);
      }
    }
  }
}

// Candidate word: key in the high half, bit-inverted index in the low half,
// so that a descending order is (key desc, index asc).
__device__ __forceinline__ uint64_t cand_word(uint32_t key, uint32_t idx) {
  return (static_cast<uint64_t>(key) << 32) | (0xFFFFFFFFu - idx);
}

// Radix select, top-k collection, sort, nucleus and draw for one row whose
// keys sit in `keys` (nq full chunks; head/tail element ekey at index eidx).
template <class K>
__device__ __noinline__ void warp_select_and_draw(const Params &p, int r, const Row &w,
                                                  uint32_t *hist, uint64_t *cand,
                                                  const uint4 *keys, int nq, int rounds,
                                                  int head, int tail, int eidx, uint32_t ekey) {
  constexpr int EPC = K::kPerChunk;
  const uint32_t lane = lane_id();

  // ---- radix select of the k_eff-th largest key, 8 bits per pass ----
  uint32_t prefix = 0, pmask = 0;
  uint32_t kk = static_cast<uint32_t>(w.k_eff);
#pragma unroll 1
  for (int pass = 0; pass < K::kBits / 8; ++pass) {
    const int shift = K::kBits - 8 * (pass + 1);
    reinterpret_cast<uint4 *>(hist)[lane * 2] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4 *>(hist)[lane * 2 + 1] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
#pragma unroll 4
    for (int q = static_cast<int>(lane); q < nq; q += 32) {
      const uint4 v = keys[q];
      const uint32_t c[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        const uint32_t k = K::elem(c, e);
        if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFFu], 1u);
      }
    }
    if ((ekey & pmask) == prefix) atomicAdd(&hist[(ekey >> shift) & 0xFFu], 1u);
    __syncwarp();
    // lane l owns bins 8l .. 8l+7; find the bin where the count from the top
    // reaches kk
    const uint4 h0 = reinterpret_cast<const uint4 *>(hist)[lane * 2];
    const uint4 h1 = reinterpret_cast<const uint4 *>(hist)[lane * 2 + 1];
    const uint32_t hb[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    uint32_t s = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) s += hb[b];
    uint32_t suf = s;  // sum over lanes >= this lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, suf, o);
      if (lane + o < 32) suf += t;
    }
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
  const uint32_t need = kk;     // how many keys equal to thr are kept

  // ---- collect the top-k set in index order: head, chunks, tail ----
  uint32_t base = 0, eq_base = 0;
  const uint32_t lt = lanemask_lt();
  {  // head elements (indices 0 .. head-1 live in lanes 0 .. head-1)
    const bool in = static_cast<int>(lane) < head;
    const bool gt = in && ekey > thr, eq = in && ekey == thr;
    const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, eq);
    const bool take = gt || (eq && eq_base + __popc(eqm & lt) < need);
    const uint32_t sm = __ballot_sync(0xFFFFFFFFu, take);
    const uint32_t at = base + __popc(sm & lt);
    if (take && at < 64) cand[at] = cand_word(ekey, static_cast<uint32_t>(eidx));
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
        if (pos < 64) cand[pos] = cand_word(k, idx0 + e);
        ++pos;
      }
    }
    base += sel_tot;
    eq_base += eq_tot;
  }
  {  // tail elements, in lane order after the chunks
    const bool in = static_cast<int>(lane) >= head && static_cast<int>(lane) < head + tail;
    const bool gt = in && ekey > thr, eq = in && ekey == thr;
    const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, eq);
    const bool take = gt || (eq && eq_base + __popc(eqm & lt) < need);
    const uint32_t sm = __ballot_sync(0xFFFFFFFFu, take);
    const uint32_t at = base + __popc(sm & lt);
    if (take && at < 64) cand[at] = cand_word(ekey, static_cast<uint32_t>(eidx));
    base += __popc(sm);
  }
  __syncwarp();

  // ---- sort the <= 64 survivors by (key desc, index asc) ----
  const int kq = w.k_eff;  // == base
  uint64_t v0, v1 = 0;
  if (kq <= 32) {
    v0 = static_cast<int>(lane) < kq ? cand[lane] : 0ull;
    v0 = bitonic32_desc(v0);
  } else {
    v0 = cand[lane];
    v1 = static_cast<int>(lane) + 32 < kq ? cand[lane + 32] : 0ull;
    bitonic64_desc(v0, v1);
  }
  __syncwarp();

  // ---- weights, prefix masses, nucleus and draw ----
  const uint32_t top_key = static_cast<uint32_t>(__shfl_sync(0xFFFFFFFFu, v0, 0) >> 32);
  const float m = K::value(top_key);
  const bool has1 = kq > 32;
  const int p0 = static_cast<int>(lane), p1 = static_cast<int>(lane) + 32;
  float w0 = 0.f, w1 = 0.f;
  if (!w.greedy) {
    if (p0 < kq) w0 = kept_weight(K::value(static_cast<uint32_t>(v0 >> 32)), m, w.temp);
    if (has1 && p1 < kq) w1 = kept_weight(K::value(static_cast<uint32_t>(v1 >> 32)), m, w.temp);
  }
  const uint64_t f0 = to_fixed(w0), f1 = to_fixed(w1);
  const uint64_t c0 = warp_incl_scan_u64(f0);
  const uint64_t tot0 = __shfl_sync(0xFFFFFFFFu, c0, 31);
  const uint64_t c1 = has1 ? warp_incl_scan_u64(f1) + tot0 : tot0;
  const uint64_t s_k = has1 ? __shfl_sync(0xFFFFFFFFu, c1, 31) : tot0;

  int n_p = 1, pick = 0;
  if (!w.greedy) {
    if (w.top_p >= 1.0f) {
      n_p = kq;
    } else {
      const double cut = static_cast<double>(w.top_p) * static_cast<double>(s_k);
      const uint32_t below0 = __ballot_sync(0xFFFFFFFFu, p0 < kq && static_cast<double>(c0) < cut);
      const uint32_t below1 = __ballot_sync(0xFFFFFFFFu, p1 < kq && static_cast<double>(c1) < cut);
      n_p = min(__popc(below0) + __popc(below1) + 1, kq);
    }
    const int last = n_p - 1;
    const uint64_t s_p = last < 32 ? __shfl_sync(0xFFFFFFFFu, c0, last)
                                   : __shfl_sync(0xFFFFFFFFu, c1, last - 32);
    const uint32_t u24 = philox_u24(p.seed[r], p.request[r],
                                    static_cast<uint64_t>(p.step[w.stream]),
                                    static_cast<uint64_t>(static_cast<int64_t>(p.codebook[r])));
    const uint64_t target = scale_u24(u24, s_p);
    const uint32_t le0 = __ballot_sync(0xFFFFFFFFu, p0 < n_p && c0 <= target);
    const uint32_t le1 = __ballot_sync(0xFFFFFFFFu, p1 < n_p && c1 <= target);
    pick = __popc(le0) + __popc(le1);
  }
  const uint64_t pw = pick < 32 ? __shfl_sync(0xFFFFFFFFu, v0, pick)
                                : __shfl_sync(0xFFFFFFFFu, v1, pick - 32);
  const int32_t id = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(pw));
  if (lane == 0) finish_row(p, r, w, id, 0u);

  if (p.kept_ids) {
    const float s_real = static_cast<float>(static_cast<double>(s_k) * (1.0 / 1099511627776.0));
    const int64_t rb = static_cast<int64_t>(r) * p.max_keep;
    if (p0 < kq && p0 < p.max_keep) {
      p.kept_ids[rb + p0] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(v0));
      p.kept_probs[rb + p0] = w.greedy ? (p0 == 0 ? 1.f : 0.f) : __fdiv_rn(w0, s_real);
    }
    if (has1 && p1 < kq && p1 < p.max_keep) {
      p.kept_ids[rb + p1] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(v1));
      p.kept_probs[rb + p1] = w.greedy ? 0.f : __fdiv_rn(w1, s_real);
    }
    if (lane == 0) {
      p.n_kept[r] = kq;
      p.n_nucleus[r] = n_p;
    }
  }
}

// NCH = most 16-byte chunks per lane (the row holds at most
// NCH * 32 * kPerChunk elements).  `keys` is this warp's staging buffer of
// NCH * 32 chunks.
template <class K, int NCH>
__device__ void warp_row(const Params &p, int r, uint32_t *hist, uint64_t *cand, uint4 *keys) {
  constexpr int EPC = K::kPerChunk;
  const uint32_t lane = lane_id();
  const Row w = load_row(p, r);
  if (w.err) {
    if (lane == 0) finish_row(p, r, w, -1, w.err);
    return;
  }
  const int V = w.vocab;
  const char *rowp = static_cast<const char *>(p.logits) + w.off * K::kElemBytes;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
  int head = static_cast<int>(((16u - (addr & 15u)) & 15u) / K::kElemBytes);
  head = min(head, V);
  const int nq = (V - head) / EPC;
  const int tail = V - head - nq * EPC;
  const char *body = rowp + head * K::kElemBytes;
  const int rounds = (nq + 31) >> 5;  // warp-uniform chunk rounds

  // ---- load: interior chunks by 16-byte loads (all in flight), head/tail by
  // single loads; keys go to this warp's shared buffer ----
  {
    uint4 v[NCH];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int q = static_cast<int>(lane) + 32 * j;
      v[j] = make_uint4(0u, 0u, 0u, 0u);
      if (q < nq) v[j] = ld_stream_v4(body + static_cast<size_t>(q) * 16);
    }
    bool bad = false, finite = false;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int q = static_cast<int>(lane) + 32 * j;
      if (q < nq) {
        const uint32_t c[4] = {K::key_word(v[j].x), K::key_word(v[j].y), K::key_word(v[j].z),
                               K::key_word(v[j].w)};
#pragma unroll
        for (int e = 0; e < EPC; ++e) {
          const uint32_t k = K::elem(c, e);
          bad |= (k < K::kNegInf) | (k >= K::kPosInf);
          finite |= k > K::kNegInf;
        }
        keys[q] = make_uint4(c[0], c[1], c[2], c[3]);
      }
    }
    // the head/tail element of this lane, if any
    int eidx = 0x7FFFFFFF;
    if (static_cast<int>(lane) < head)
      eidx = static_cast<int>(lane);
    else if (static_cast<int>(lane) < head + tail)
      eidx = nq * EPC + static_cast<int>(lane);
    uint32_t ekey = 0;
    if (eidx < V) {
      ekey = K::key(K::load_one(rowp, eidx));
      bad |= (ekey < K::kNegInf) | (ekey >= K::kPosInf);
      finite |= ekey > K::kNegInf;
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    finite = __any_sync(0xFFFFFFFFu, finite);
    if (bad || !finite) {
      if (lane == 0) finish_row(p, r, w, -1, kRowNonFinite);
      return;
    }
    __syncwarp();
    warp_select_and_draw<K>(p, r, w, hist, cand, keys, nq, rounds, head, tail, eidx, ekey);
  }
}

template <class K, int NCH>
__global__ void __launch_bounds__(kWarpRowsPerBlock * 32)
    warp_sampler_kernel(const Params p) {
  __shared__ __align__(16) uint32_t hist[kWarpRowsPerBlock][256];
  __shared__ __align__(16) uint64_t cand[kWarpRowsPerBlock][64];
  extern __shared__ __align__(16) uint4 warp_keys[];
  const int wid = static_cast<int>(threadIdx.x >> 5);
  const int r = static_cast<int>(blockIdx.x) * kWarpRowsPerBlock + wid;
  if (r >= p.n_rows) return;
  warp_row<K, NCH>(p, r, hist[wid], cand[wid], warp_keys + wid * NCH * 32);
}

}  // namespace ts
