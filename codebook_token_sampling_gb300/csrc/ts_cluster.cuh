// ts_cluster.cuh -- CTA-per-row / cluster-per-row sampler for any top-k cap up
// to 4096 (the cap may be any power of two in [32, 4096]: Drama 3 article,
// section "能跑通的命令，和文档写明的边界") and rows up to 163,840 bf16 /
// 81,920 fp32 logits.
//
// A row is split into G contiguous slices, one per CTA of a thread-block
// cluster (G = 1: a plain CTA).  Each CTA streams its slice once from HBM
// into shared memory as order-preserving keys, building the first radix
// histogram on the fly.  The threshold key (the k_eff-th largest) is found
// by radix select (11 + 5 bits for bf16, 11 + 11 + 10 for fp32) whose
// histograms are merged across the cluster through distributed shared
// memory.  The top-k set (ties at the threshold by lowest index, ranked with
// an index-ordered block scan and a cluster prefix) is written into the
// leader CTA's shared memory.  The leader then finds the nucleus cutoff and
// the drawn token without sorting: a radix descent over the offset
// (max key - key) with exact 2^-40 fixed-point mass histograms, then a rank
// select among equal keys in index order.
#pragma once

#include "ts_device.cuh"

namespace ts {

constexpr int kClusterThreads = 512;
constexpr int kClusterWarps = kClusterThreads / 32;
constexpr int kHistWords = 4096;  // words per histogram buffer
static_assert(kHistWords >= 4096, "the leader keeps up to 4096 kept weights in hist_b");
constexpr int kMassBins = 1024;   // bins per level of the mass descent
constexpr int kSliceMaxBF16 = 20480;
constexpr int kSliceMaxF32 = 10240;

struct ClusterLayout {
  uint32_t keys, hist_a, hist_b, cand, misc, total;
};

__host__ __device__ inline uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }

__host__ __device__ inline ClusterLayout cluster_layout(int slice, int cap, int elem_bytes,
                                                        int per_chunk) {
  ClusterLayout l;
  uint32_t o = 0;
  l.keys = o;
  o += align16(static_cast<uint32_t>((slice + 2 * per_chunk) * elem_bytes));
  l.hist_a = o;
  o += kHistWords * 4;
  l.hist_b = o;
  o += kHistWords * 4;
  l.cand = o;  // (key, index) pairs
  o += align16(static_cast<uint32_t>(cap) * 8u);
  l.misc = o;
  o += 1024;
  l.total = o;
  return l;
}

// misc word slots
constexpr int kMiscDigit = 0, kMiscAbove = 1, kMiscCount = 2, kMiscBad = 3, kMiscFinite = 4;
constexpr int kMiscTotGt = 8, kMiscTotEq = 9, kMiscBaseGt = 10, kMiscBaseEq = 11;
constexpr int kMiscId = 12, kMiscMax = 13;
constexpr int kMiscWide = 16;     // 2 x u64 slots (words 16..19)
constexpr int kMiscScratch = 32;  // block-scan scratch (u64 x 17 -> words 32..67)

// Block-wide exclusive scan (64-bit) over kClusterThreads threads.
__device__ __forceinline__ uint64_t block_excl_scan_u64(uint64_t v, uint64_t *scratch,
                                                        uint64_t *total) {
  const uint32_t lane = lane_id(), wid = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= static_cast<uint32_t>(o)) x += t;
  }
  __syncthreads();  // scratch may still be read by a previous call
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint64_t s = lane < kClusterWarps ? scratch[lane] : 0ull;
    uint64_t inc = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
      if (lane >= static_cast<uint32_t>(o)) inc += t;
    }
    if (lane < kClusterWarps) scratch[lane] = inc - s;
    if (lane == kClusterWarps - 1) scratch[kClusterWarps] = inc;
  }
  __syncthreads();
  *total = scratch[kClusterWarps];
  return scratch[wid] + x - v;
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint64_t *scratch) {
  uint32_t x = __reduce_max_sync(0xFFFFFFFFu, v);
  const uint32_t lane = lane_id(), wid = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[wid] = x;
  __syncthreads();
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < kClusterWarps; ++i) r = max(r, static_cast<uint32_t>(scratch[i]));
  return r;
}

template <class K>
__device__ __forceinline__ void chunk_from_keys(uint32_t (&cw)[4], const uint32_t (&k)[K::kPerChunk]) {
  if constexpr (K::kPerChunk == 8) {
#pragma unroll
    for (int x = 0; x < 4; ++x) cw[x] = k[2 * x] | (k[2 * x + 1] << 16);
  } else {
#pragma unroll
    for (int x = 0; x < 4; ++x) cw[x] = k[x];
  }
}

// Merged (cluster-wide) radix step: sums histogram `h` (nbins <= 2048) over
// the G CTAs, finds the bin where the count from the top reaches kk, and
// leaves (digit, count above the digit, count in the digit) in misc.
template <int G>
__device__ void merged_select(const uint32_t *h, int nbins, uint32_t kk, uint32_t *misc,
                              uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  uint32_t hb[4] = {0u, 0u, 0u, 0u};
  if (4 * t < nbins) {  // nbins is a multiple of 4
    if constexpr (G == 1) {
      const uint4 v = reinterpret_cast<const uint4 *>(h)[t];
      hb[0] = v.x;
      hb[1] = v.y;
      hb[2] = v.z;
      hb[3] = v.w;
    } else {
      uint4 v[G];
      const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&h[4 * t]));
#pragma unroll
      for (int c = 0; c < G; ++c) {
        uint32_t ra;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(c));
        v[c] = dsmem_ld_v4(ra);
      }
#pragma unroll
      for (int c = 0; c < G; ++c) {
        hb[0] += v[c].x;
        hb[1] += v[c].y;
        hb[2] += v[c].z;
        hb[3] += v[c].w;
      }
    }
  }
  const uint32_t s = hb[0] + hb[1] + hb[2] + hb[3];
  uint64_t tot64;
  const uint32_t excl = static_cast<uint32_t>(block_excl_scan_u64(s, scratch, &tot64));
  const uint32_t total = static_cast<uint32_t>(tot64);
  const uint32_t above_me = total - excl - s;  // count in bins above this thread's
  if (s != 0 && above_me < kk && above_me + s >= kk) {
    uint32_t run = above_me;
#pragma unroll
    for (int b = 3; b >= 0; --b) {
      if (run + hb[b] >= kk) {
        misc[kMiscDigit] = static_cast<uint32_t>(4 * t + b);
        misc[kMiscAbove] = run;
        misc[kMiscCount] = hb[b];
        break;
      }
      run += hb[b];
    }
  }
  __syncthreads();
}

// Radix descent over offsets (max key - key) of the kept set with exact
// fixed-point masses.  cut_mode: first position whose cumulative mass
// reaches `cut` (i.e. is >= cut); else first position whose cumulative mass
// exceeds `target`.  Returns the key of that position's group and writes the
// mass of all keys above that group to *above_out.
//
// Levels take 10 offset bits each.  At the last level a bin is one key, so
// its mass is (count x weight of that key); above it a bin mixes keys and
// its mass is kept as three 32-bit partial sums (weight bits 0-12, 13-25 and
// 26+), so only native 32-bit shared-memory atomics are used.
// descend_levels continues a descent whose levels above have put the
// position in offsets off_lo .. off_lo + 2^span - 1 with mass `above` before
// them; its next level bins those offsets >> shift.  wt: the kept weights.
template <class K>
__device__ uint32_t descend_levels(const uint2 *cand, const float *wt, int kq, uint32_t maxk,
                                   float m, float temp, float inv_temp, bool cut_mode, uint64_t cut,
                                   uint64_t target, uint32_t off_lo, int span, int shift,
                                   uint64_t above, uint32_t *h, uint32_t *misc, uint64_t *scratch,
                                   uint64_t *above_out) {
  const int t = static_cast<int>(threadIdx.x);
  uint64_t *wide = reinterpret_cast<uint64_t *>(misc + kMiscWide);
  for (;;) {
    const bool exact = shift == 0;
    __syncthreads();
    for (int i = t; i < (exact ? kMassBins : 3 * kMassBins); i += kClusterThreads) h[i] = 0u;
    __syncthreads();
    for (int i = t; i < kq; i += kClusterThreads) {
      const uint32_t key = cand[i].x;
      const uint32_t off = maxk - key;
      if (off >= off_lo && static_cast<uint64_t>(off - off_lo) < (1ull << span)) {
        const uint32_t d = (off - off_lo) >> shift;
        if (exact) {
          atomicAdd(&h[d], 1u);
        } else {
          const uint64_t f = to_fixed(wt[i]);
          if (f) {
            atomicAdd(&h[d], static_cast<uint32_t>(f & 0x1FFFu));
            atomicAdd(&h[kMassBins + d], static_cast<uint32_t>((f >> 13) & 0x1FFFu));
            atomicAdd(&h[2 * kMassBins + d], static_cast<uint32_t>(f >> 26));
          }
        }
      }
    }
    __syncthreads();
    uint64_t ab[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const uint32_t d = static_cast<uint32_t>(2 * t + x);
      if (exact) {
        const uint32_t n = h[d];
        ab[x] = n ? n * to_fixed(kept_weight(K::value(maxk - off_lo - d), m, temp, inv_temp)) : 0ull;
      } else {
        ab[x] = (static_cast<uint64_t>(h[2 * kMassBins + d]) << 26) +
                (static_cast<uint64_t>(h[kMassBins + d]) << 13) + h[d];
      }
    }
    const uint64_t a = ab[0], b = ab[1];
    uint64_t tot;
    const uint64_t excl = block_excl_scan_u64(a + b, scratch, &tot);
    auto reached = [&](uint64_t cum) {
      return cut_mode ? cum >= cut : cum > target;
    };
    const uint64_t p0 = above + excl, p1 = p0 + a, p2 = p1 + b;
    if (!reached(p0) && reached(p1)) {
      misc[kMiscDigit] = static_cast<uint32_t>(2 * t);
      wide[0] = p0;
    } else if (!reached(p1) && reached(p2)) {
      misc[kMiscDigit] = static_cast<uint32_t>(2 * t + 1);
      wide[0] = p1;
    }
    __syncthreads();
    off_lo += misc[kMiscDigit] << shift;
    above = wide[0];
    if (shift == 0) break;
    span = shift;
    shift = shift > 10 ? shift - 10 : 0;
  }
  *above_out = above;
  return maxk - off_lo;
}

// The descent from its first level: offsets 0 .. 2^bits - 1, bits = the bit
// width of range = maxk - (smallest kept key).
template <class K>
__device__ uint32_t mass_descent(const uint2 *cand, const float *wt, int kq, uint32_t maxk,
                                 uint32_t range, float m, float temp, float inv_temp, bool cut_mode,
                                 uint64_t cut, uint64_t target,
                                 uint32_t *h, uint32_t *misc, uint64_t *scratch,
                                 uint64_t *above_out) {
  const int bits = range ? 32 - __clz(range) : 0;
  return descend_levels<K>(cand, wt, kq, maxk, m, temp, inv_temp, cut_mode, cut, target, 0u, bits,
                           bits > 10 ? bits - 10 : 0, 0ull, h, misc, scratch, above_out);
}

// The first level of a descent whose offsets need more than one level
// (shift1 = bits - 10 > 0), from the level's bin masses that the caller has
// built once for both descents: thread t holds bins 2t and 2t + 1, their
// masses a and b and the exclusive prefix p0 of bin 2t.  The bin where the
// cumulative mass reaches `cut` (cut_mode) or passes `target` is found, and
// the descent goes on below it.
template <class K>
__device__ uint32_t mass_descent_from_l1(const uint2 *cand, const float *wt, int kq, uint32_t maxk,
                                         float m, float temp, float inv_temp, bool cut_mode,
                                         uint64_t cut, uint64_t target, int shift1, uint64_t p0,
                                         uint64_t a, uint64_t b, uint32_t *h, uint32_t *misc,
                                         uint64_t *scratch, uint64_t *above_out) {
  const int t = static_cast<int>(threadIdx.x);
  uint64_t *wide = reinterpret_cast<uint64_t *>(misc + kMiscWide);
  auto reached = [&](uint64_t cum) { return cut_mode ? cum >= cut : cum > target; };
  const uint64_t p1 = p0 + a, p2 = p1 + b;
  __syncthreads();  // misc may still be read
  if (!reached(p0) && reached(p1)) {
    misc[kMiscDigit] = static_cast<uint32_t>(2 * t);
    wide[0] = p0;
  } else if (!reached(p1) && reached(p2)) {
    misc[kMiscDigit] = static_cast<uint32_t>(2 * t + 1);
    wide[0] = p1;
  }
  __syncthreads();
  const uint32_t off_lo = misc[kMiscDigit] << shift1;
  const uint64_t above = wide[0];
  return descend_levels<K>(cand, wt, kq, maxk, m, temp, inv_temp, cut_mode, cut, target, off_lo,
                           shift1, shift1 > 10 ? shift1 - 10 : 0, above, h, misc, scratch,
                           above_out);
}

// Index (token id) of the `rank`-th kept token, in index order, among those
// with key == key_sel.  Candidates are stored in index order within each key.
__device__ int32_t rank_select(const uint2 *cand, int kq, uint32_t key_sel, uint64_t rank,
                               uint32_t *misc, uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  const int per = (kq + kClusterThreads - 1) / kClusterThreads;
  const int lo = min(t * per, kq), hi = min(lo + per, kq);
  uint32_t c = 0;
  for (int i = lo; i < hi; ++i) c += cand[i].x == key_sel;
  uint64_t tot;
  const uint64_t excl = block_excl_scan_u64(c, scratch, &tot);
  if (rank >= excl && rank < excl + c) {
    uint64_t seen = excl;
    for (int i = lo; i < hi; ++i) {
      if (cand[i].x == key_sel) {
        if (seen == rank) misc[kMiscId] = cand[i].y;
        ++seen;
      }
    }
  }
  __syncthreads();
  return static_cast<int32_t>(misc[kMiscId]);
}

template <class K, int G>
__global__ void __launch_bounds__(kClusterThreads, 2) cluster_sampler_kernel(const Params p) {
  constexpr int EPC = K::kPerChunk;
  constexpr int NPASS = K::kBits == 16 ? 2 : 3;
  using KT = typename std::conditional<K::kBits == 16, uint16_t, uint32_t>::type;
  extern __shared__ __align__(16) unsigned char smem[];
  const ClusterLayout lay = cluster_layout(p.slice, p.cap, K::kElemBytes, EPC);
  KT *kbuf = reinterpret_cast<KT *>(smem + lay.keys);
  uint32_t *hist_a = reinterpret_cast<uint32_t *>(smem + lay.hist_a);
  uint32_t *hist_b = reinterpret_cast<uint32_t *>(smem + lay.hist_b);
  uint2 *cand = reinterpret_cast<uint2 *>(smem + lay.cand);
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + lay.misc);
  uint64_t *scratch = reinterpret_cast<uint64_t *>(misc + kMiscScratch);

  const uint32_t rank = G > 1 ? cluster_rank() : 0u;
  const int r = G > 1 ? static_cast<int>(cluster_index()) : static_cast<int>(blockIdx.x);
  const int tid = static_cast<int>(threadIdx.x);
  pdl_wait_and_release();
  if (r >= p.n_rows) return;  // whole cluster (grid is sized exactly)
  const Row w = load_row(p, r);
  if (w.err || w.fin) {  // identical in every CTA of the cluster: all leave before any barrier
    if (rank == 0 && tid == 0) finish_row(p, r, w, -1, w.err);
    return;
  }

  for (int i = tid; i < 2 * kHistWords / 4; i += kClusterThreads)
    reinterpret_cast<uint4 *>(hist_a)[i] = make_uint4(0u, 0u, 0u, 0u);  // hist_a and hist_b
  __syncthreads();

  // ---- slice geometry: smem slot P holds slice element P - pad ----
  const int S = p.slice;
  const int s_begin = static_cast<int>(rank) * S;
  const int sc = max(0, min(S, w.vocab - s_begin));
  const char *sp = static_cast<const char *>(p.logits) + (w.off + s_begin) * K::kElemBytes;
  const int pad = static_cast<int>((reinterpret_cast<uintptr_t>(sp) & 15u) / K::kElemBytes);
  const char *cbase = sp - pad * K::kElemBytes;
  const int nq = sc > 0 ? (sc + pad + EPC - 1) / EPC : 0;

  // ---- stream the slice in; keys to smem; first radix histogram ----
  constexpr int kShift0 = K::kBits - 11;
  const uint64_t pol = l2_evict_first();
  uint32_t nbad = 0, nfin = 0;
  for (int m = tid; m < nq; m += kClusterThreads) {
    uint32_t cw[4];
    const bool interior = m * EPC >= pad && (m + 1) * EPC <= sc + pad;
    if (interior) {
      const uint4 v = ld_stream_v4(cbase + static_cast<size_t>(m) * 16, pol);
      cw[0] = K::key_word(v.x);
      cw[1] = K::key_word(v.y);
      cw[2] = K::key_word(v.z);
      cw[3] = K::key_word(v.w);
    } else {
      uint32_t k[EPC];
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        const int slot = m * EPC + e;
        k[e] = (slot >= pad && slot < sc + pad) ? K::key(K::load_one(sp, slot - pad)) : 0u;
      }
      chunk_from_keys<K>(cw, k);
    }
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
      const int slot = m * EPC + e;
      if (interior || (slot >= pad && slot < sc + pad)) {
        const uint32_t k = K::elem(cw, e);
        nbad += (k < K::kNegInf) | (k >= K::kPosInf);
        nfin += k > K::kNegInf;
        atomicAdd(&hist_a[k >> kShift0], 1u);
      }
    }
    reinterpret_cast<uint4 *>(kbuf)[m] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  }
  nbad = __reduce_add_sync(0xFFFFFFFFu, nbad);
  nfin = __reduce_add_sync(0xFFFFFFFFu, nfin);
  if (lane_id() == 0) {
    if (nbad) atomicAdd(&hist_a[2048], nbad);
    if (nfin) atomicAdd(&hist_a[2049], nfin);
  }
  __syncthreads();
  if constexpr (G > 1) cluster_sync_all();

  // ---- pass 1 merge; value checks are cluster-wide ----
  if (tid == 0) {
    uint32_t bad = 0, fin = 0;
#pragma unroll
    for (int c = 0; c < G; ++c) {
      if constexpr (G == 1) {
        bad += hist_a[2048];
        fin += hist_a[2049];
      } else {
        bad += dsmem_ld_u32(dsmem_addr(&hist_a[2048], c));
        fin += dsmem_ld_u32(dsmem_addr(&hist_a[2049], c));
      }
    }
    misc[kMiscBad] = bad;
    misc[kMiscFinite] = fin;
  }
  uint32_t kk = static_cast<uint32_t>(w.k_eff);
  merged_select<G>(hist_a, 2048, kk, misc, scratch);
  if (misc[kMiscBad] != 0 || misc[kMiscFinite] == 0) {
    if constexpr (G > 1) cluster_sync_all();  // peers may still read our histogram
    if (rank == 0 && tid == 0) finish_row(p, r, w, -1, kRowNonFinite);
    return;
  }
  uint32_t prefix = misc[kMiscDigit] << kShift0;
  kk -= misc[kMiscAbove];

  // ---- remaining radix passes over the keys in shared memory ----
#pragma unroll 1
  for (int pass = 1; pass < NPASS; ++pass) {
    const int width = (K::kBits == 16) ? 5 : (pass == 1 ? 11 : 10);
    const int shift = (K::kBits == 16) ? 0 : (pass == 1 ? 10 : 0);
    const int hi_shift = shift + width;
    uint32_t *h = (pass & 1) ? hist_b : hist_a;
    if (pass >= 2) {  // hist_a: every peer finished reading it before the last barrier
      for (int i = tid; i < 2048 + 2; i += kClusterThreads) h[i] = 0u;
      __syncthreads();
    }
    const uint32_t want = prefix >> hi_shift;
    const uint32_t mask = (1u << width) - 1u;
    for (int m = tid; m < nq; m += kClusterThreads) {
      const uint4 v = reinterpret_cast<const uint4 *>(kbuf)[m];
      const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        const uint32_t k = K::elem(cw, e);
        if ((k >> hi_shift) == want) atomicAdd(&h[(k >> shift) & mask], 1u);
      }
    }
    __syncthreads();
    if constexpr (G > 1) cluster_sync_all();
    merged_select<G>(h, 1 << width, kk, misc, scratch);
    prefix |= misc[kMiscDigit] << shift;
    kk -= misc[kMiscAbove];
  }
  const uint32_t thr = prefix;            // k_eff-th largest key
  const uint32_t need = kk;               // keys equal to thr that are kept
  const uint32_t n_gt = static_cast<uint32_t>(w.k_eff) - need;

  // ---- top-k set: counts per chunk, index-ordered scan, cluster prefix ----
  uint32_t *cnt = (NPASS % 2 == 0) ? hist_a : hist_b;  // not read by peers any more
  const int nj = (nq + kClusterThreads - 1) / kClusterThreads;
  uint32_t my_cnt[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int m = tid + j * kClusterThreads;
    uint32_t packed = 0;
    if (j < nj && m < nq) {
      const uint4 v = reinterpret_cast<const uint4 *>(kbuf)[m];
      const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
      uint32_t ng = 0, ne = 0;
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        const uint32_t k = K::elem(cw, e);
        ng += k > thr;
        ne += k == thr;
      }
      packed = ng | (ne << 16);
    }
    my_cnt[j] = packed;
    if (j < nj) cnt[m] = packed;
  }
  __syncthreads();
  {  // exclusive scan over chunk order m (thread u scans entries [u*nj, u*nj + nj))
    uint32_t local[8];
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      local[i] = (i < nj) ? cnt[tid * nj + i] : 0u;
      s += local[i];
    }
    uint64_t tot;
    uint32_t run = static_cast<uint32_t>(block_excl_scan_u64(s, scratch, &tot));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < nj) cnt[tid * nj + i] = run;
      run += local[i];
    }
    if (tid == 0) {
      misc[kMiscTotGt] = static_cast<uint32_t>(tot) & 0xFFFFu;
      misc[kMiscTotEq] = static_cast<uint32_t>(tot) >> 16;
    }
  }
  __syncthreads();
  if constexpr (G > 1) {
    cluster_sync_all();
    if (tid < 32) {  // lane c < rank reads CTA c's totals
      uint32_t bg = 0, be = 0;
      if (static_cast<uint32_t>(tid) < rank) {
        bg = dsmem_ld_u32(dsmem_addr(&misc[kMiscTotGt], tid));
        be = dsmem_ld_u32(dsmem_addr(&misc[kMiscTotEq], tid));
      }
      bg = __reduce_add_sync(0xFFFFFFFFu, bg);
      be = __reduce_add_sync(0xFFFFFFFFu, be);
      if (tid == 0) {
        misc[kMiscBaseGt] = bg;
        misc[kMiscBaseEq] = be;
      }
    }
  } else if (tid == 0) {
    misc[kMiscBaseGt] = 0;
    misc[kMiscBaseEq] = 0;
  }
  __syncthreads();
  const uint32_t base_gt = misc[kMiscBaseGt], base_eq = misc[kMiscBaseEq];
  const uint32_t idx_base = static_cast<uint32_t>(s_begin - pad);
  uint32_t cand_remote = 0;
  if constexpr (G > 1) cand_remote = dsmem_addr(cand, 0);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int m = tid + j * kClusterThreads;
    if (j < nj && m < nq && my_cnt[j] != 0) {
      const uint32_t off = cnt[m];
      uint32_t og = base_gt + (off & 0xFFFFu), oe = base_eq + (off >> 16);
      const uint4 v = reinterpret_cast<const uint4 *>(kbuf)[m];
      const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        const uint32_t k = K::elem(cw, e);
        uint32_t pos = 0xFFFFFFFFu;
        if (k > thr) {
          pos = og++;
        } else if (k == thr) {
          if (oe < need) pos = n_gt + oe;
          ++oe;
        }
        if (pos < static_cast<uint32_t>(p.cap)) {
          const uint32_t idx = idx_base + static_cast<uint32_t>(m * EPC + e);
          if constexpr (G == 1) {
            cand[pos] = make_uint2(k, idx);
          } else {
            dsmem_st_v2(cand_remote + 8u * pos, k, idx);
          }
        }
      }
    }
  }
  __syncthreads();
  if constexpr (G > 1) cluster_sync_all();
  if (rank != 0) return;

  // ---- leader: weights, nucleus cutoff and draw over the k_eff candidates ----
  const int kq = w.k_eff;
  uint32_t mloc = 0;
  for (int i = tid; i < kq; i += kClusterThreads) mloc = max(mloc, cand[i].x);
  const uint32_t maxk = block_max_u32(mloc, scratch);
  const float mval = K::value(maxk);
  uint32_t *mh = hist_a;  // mass histograms (hist_a is free again)
  int32_t id;
  int n_p = 1;
  uint64_t s_k = 0;
  // the kept weights, computed once (hist_b is free once the top-k set is in)
  float *wt = reinterpret_cast<float *>(hist_b);
  if (w.greedy) {
    id = rank_select(cand, kq, maxk, 0, misc, scratch);
  } else {
    // the descents' first level, when their offsets need more than one: the
    // kept masses binned by (maxk - key) >> shift1, built with the weights
    const uint32_t range = maxk - thr;
    const int bits = range ? 32 - __clz(range) : 0;
    const int shift1 = bits > 10 ? bits - 10 : 0;
    if (shift1 > 0) {
      for (int i = tid; i < 3 * kMassBins; i += kClusterThreads) mh[i] = 0u;
      __syncthreads();
    }
    uint64_t part = 0;
    for (int i = tid; i < kq; i += kClusterThreads) {
      const uint32_t key = cand[i].x;
      const float wi = kept_weight(K::value(key), mval, w.temp, w.inv_temp);
      wt[i] = wi;
      const uint64_t f = to_fixed(wi);
      part += f;
      if (shift1 > 0 && f) {
        const uint32_t d = (maxk - key) >> shift1;
        atomicAdd(&mh[d], static_cast<uint32_t>(f & 0x1FFFu));
        atomicAdd(&mh[kMassBins + d], static_cast<uint32_t>((f >> 13) & 0x1FFFu));
        atomicAdd(&mh[2 * kMassBins + d], static_cast<uint32_t>(f >> 26));
      }
    }
    block_excl_scan_u64(part, scratch, &s_k);  // its first barrier: every bin is in
    uint64_t l1_p0 = 0, l1_a = 0, l1_b = 0;    // this thread's two first-level bins
    if (shift1 > 0) {
      auto bin_mass = [&](int d) {
        return (static_cast<uint64_t>(mh[2 * kMassBins + d]) << 26) +
               (static_cast<uint64_t>(mh[kMassBins + d]) << 13) + mh[d];
      };
      l1_a = bin_mass(2 * tid);
      l1_b = bin_mass(2 * tid + 1);
      uint64_t tot1;
      l1_p0 = block_excl_scan_u64(l1_a + l1_b, scratch, &tot1);
    }
    uint64_t s_p;
    if (w.top_p >= 1.0f) {
      n_p = kq;
      s_p = s_k;
    } else if (!(w.top_p > 0.0f)) {
      n_p = 1;
      s_p = to_fixed(kept_weight(mval, mval, w.temp, w.inv_temp));
    } else {
      const uint64_t cut = ceil_mul_p(w.top_p, s_k);  // C reaches top_p * S_k iff C >= cut
      uint64_t above;
      const uint32_t key_c =
          shift1 > 0 ? mass_descent_from_l1<K>(cand, wt, kq, maxk, mval, w.temp, w.inv_temp, true,
                                               cut, 0, shift1, l1_p0, l1_a, l1_b, mh, misc,
                                               scratch, &above)
                     : mass_descent<K>(cand, wt, kq, maxk, range, mval, w.temp, w.inv_temp, true,
                                       cut, 0, mh, misc, scratch, &above);
      const uint64_t wc = to_fixed(kept_weight(K::value(key_c), mval, w.temp, w.inv_temp));
      // smallest n >= 1 with above + n * wc >= cut (above < cut; the crossing
      // group has positive mass, the guard only protects the division)
      uint64_t n_c = wc > 0 ? (cut - above + wc - 1) / wc : 1;
      if (n_c < 1) n_c = 1;
      uint32_t gt_loc = 0;
      for (int i = tid; i < kq; i += kClusterThreads) gt_loc += cand[i].x > key_c;
      uint64_t n_above;
      block_excl_scan_u64(gt_loc, scratch, &n_above);
      n_p = static_cast<int>(n_above + n_c);
      s_p = above + n_c * wc;
    }
    const uint32_t u24 = philox_u24(p.seed[r], p.request[r],
                                    static_cast<uint64_t>(p.step[w.stream]),
                                    static_cast<uint64_t>(static_cast<int64_t>(p.codebook[r])));
    const uint64_t target = scale_u24(u24, s_p);
    uint64_t above_d;
    const uint32_t key_d =
        shift1 > 0 ? mass_descent_from_l1<K>(cand, wt, kq, maxk, mval, w.temp, w.inv_temp, false, 0,
                                             target, shift1, l1_p0, l1_a, l1_b, mh, misc, scratch,
                                             &above_d)
                   : mass_descent<K>(cand, wt, kq, maxk, range, mval, w.temp, w.inv_temp, false, 0,
                                     target, mh, misc, scratch, &above_d);
    const uint64_t wd = to_fixed(kept_weight(K::value(key_d), mval, w.temp, w.inv_temp));
    id = rank_select(cand, kq, key_d, wd > 0 ? (target - above_d) / wd : 0, misc, scratch);
  }
  if (tid == 0) finish_row(p, r, w, id, 0u);
  if (p.kept_ids) {
    const float s_real = static_cast<float>(static_cast<double>(s_k) * (1.0 / 1099511627776.0));
    const int64_t rb = static_cast<int64_t>(r) * p.max_keep;
    for (int i = tid; i < kq && i < p.max_keep; i += kClusterThreads) {
      const int32_t tok = static_cast<int32_t>(cand[i].y);
      p.kept_ids[rb + i] = tok;
      p.kept_probs[rb + i] =
          w.greedy ? (tok == id ? 1.f : 0.f)
                   : __fdiv_rn(wt[i], s_real);
    }
    if (tid == 0) {
      p.n_kept[r] = kq;
      p.n_nucleus[r] = n_p;
    }
  }
}

}  // namespace ts
