// ts_wide.cuh -- single-pass sampler for wide bf16 rows (backbone vocabularies
// such as 151,936 tokens) under any top-k cap up to 4096 (Drama 3 article,
// section "能跑通的命令，和文档写明的边界": the cap may be any power of two in
// [32, 4096]).
//
// A row is split into G contiguous slices, one CTA each, forming a
// thread-block cluster.  The row is read from HBM exactly once:
//
//  1. Threshold estimate.  Every CTA reads the same evenly spaced sample of
//     the row (1024 16-byte chunks; these lines stay in L2 for the pass that
//     follows) and takes, by an exact two-level radix select, the sample's
//     r-th largest key t with r sized so that about 1.4 k_eff row elements
//     are expected at or above t.  This is the sampling step of Floyd and
//     Rivest's selection algorithm ("Expected time bounds for selection",
//     CACM 18(3), 1975): only its speed depends on the sample, never its
//     result.  Rows no wider than the candidate buffer skip it (t = lowest key).
//  2. Filter.  Each CTA streams its slice with 16-byte loads, compares eight
//     logits per chunk against t with packed bf16 compares (an unordered
//     compare, so a NaN is flagged too), stages the flagged chunks per warp
//     and appends every element >= t as (key << 16 | slice index) to its own
//     candidate buffer in shared memory.
//  3. Check and gather.  After a cluster barrier every CTA reads all
//     candidate counts through distributed shared memory.  If the row holds a
//     NaN or +inf it is an error.  If the candidates number at least k_eff
//     (so they hold the whole top-k set and every key tied with its last
//     member) and fit the leader's buffer, each CTA copies its candidates
//     into the leader CTA and leaves.  Otherwise (an unlucky or adversarial
//     sample) the cluster runs an exact radix select over the slice again
//     and collects exactly the top-k set, ties taken by lowest index.
//  4. Leader tail, order-free.  The leader finds the threshold key and the
//     number of kept tokens tied at it by radix select over the candidates,
//     sums 2^-40 fixed-point weights (which depend only on the key), finds
//     the nucleus cutoff and the draw by a radix descent over (max key - key)
//     with exact masses, and picks the token inside the drawn key group by a
//     radix select on the token index.  No step depends on the order in
//     which candidates were appended, so the result is the same for every
//     cluster size and equal to the other kernels' bit for bit.
#pragma once

#include <cuda_bf16.h>

#include "ts_device.cuh"

namespace ts {

constexpr int kWideThreads = 256;
constexpr int kWideWarps = kWideThreads / 32;
constexpr int kWideCandMax = 8192;        // candidate entries per CTA, G <= 2 (32 KB)
constexpr int kWideCandMaxWide = 4096;    // ... G >= 4 (16 KB)
constexpr int kWideU = 4;                 // 16-byte chunks per lane per iteration
constexpr int kWideRing = 64;             // staged words per warp (a ring)
constexpr int kWideSampleChunks = 512;    // 4,096 sampled logits
constexpr int kWideSliceMax = 65536;      // slice index fits 16 bits
constexpr int kWideBins = 2048;           // per-key counts: keys t .. t + 2047
constexpr int kWideMaxG = 16;
// work area: [staging rings 4 KB][per-key counts, packed 16-bit pairs 4 KB]
//            [sample / rank-select histogram 8 KB][counts by key >> 8 1 KB]
//            [spare 1 KB]; the exact path and the distributed tail reuse the
//            first 8 KB once the filter is done with it
constexpr uint32_t kWideRingBytes = kWideWarps * kWideRing * 8;
constexpr uint32_t kWideLhOff = kWideRingBytes;
constexpr uint32_t kWideMhOff = kWideLhOff + kWideBins * 2;
constexpr uint32_t kWidePgOff = kWideMhOff + 8192;  // candidate counts by key >> 8 (256)
constexpr uint32_t kWideWorkBytes = 18432;
constexpr uint32_t kWideMiscWords = 256;
// candidate entries each CTA holds; CTAs of a cluster never pool them
__host__ __device__ constexpr int wide_cap(int g) { return g >= 4 ? kWideCandMaxWide : kWideCandMax; }
__host__ __device__ constexpr uint32_t wide_smem_bytes(int g) {
  return static_cast<uint32_t>(wide_cap(g)) * 4u + kWideWorkBytes + kWideMiscWords * 4u;
}

// misc word slots
constexpr int kWN = 0;        // local candidate count (may exceed the buffer)
constexpr int kWBad = 1;      // NaN / +inf seen in this slice
constexpr int kWTKey = 2;     // threshold key t
constexpr int kWU24 = 3;      // the row's draw
constexpr int kWTotal = 4;    // candidates over the cluster
constexpr int kWFast = 5;     // 1: per-key tail, 3: gathered tail, 2: row error, 0: exact path
constexpr int kWRange = 6;    // a candidate key beyond t + kWideBins - 1
constexpr int kWDigit = 8, kWAbove = 9, kWCount = 10, kWId = 11;
constexpr int kWFin = 12;     // finite logits in this slice (exact path)
constexpr int kWEq = 13;      // keys equal to the threshold in this slice (exact path)
constexpr int kWTake = 14;    // ... of which this slice keeps (exact path)
constexpr int kWMaxK = 15;
constexpr int kWWide = 16;    // 2 x u64 (words 16..19)
constexpr int kWSeg = 24;     // G + 1 segment offsets (words 24..40)
constexpr int kWHist2 = 64;   // 32-bin second-level histogram (words 64..95)
constexpr int kWThrB = 96, kWNeed = 97, kWNp = 98, kWDrawB = 99, kWRho = 100;
constexpr int kWOwner = 101, kWRho2 = 102, kWKept = 103, kWSelIdx = 104, kWMaxB = 105;
constexpr int kWSp = 106;     // u64 (words 106..107)
constexpr int kWScan = 128;   // block-scan scratch: u64 x (kWideWarps + 1)

// Keys of the wide path are KeyBF16's (-0 takes the key of +0).
__device__ __forceinline__ uint32_t wkey(uint32_t bits16) { return KeyBF16::key(bits16); }
__device__ __forceinline__ uint32_t wkey_word(uint32_t w) { return KeyBF16::key_word(w); }

// bf16 bits of the value whose key is k (k = 0 stands for "every element":
// -inf, so that an unordered compare flags every logit).
__device__ __forceinline__ uint32_t wkey_bits(uint32_t k) {
  if (k == 0u) return 0xFF80u;
  return k ^ ((k & 0x8000u) ? 0x8000u : 0xFFFFu);
}

__device__ __forceinline__ uint32_t hgeu_mask(uint32_t w, uint32_t t2) {
  return __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w),
                      *reinterpret_cast<const __nv_bfloat162 *>(&t2));
}

// Cluster barrier preceded by a block barrier, so that every warp arrives
// converged (the cluster barrier is the warp-aligned form).
__device__ __forceinline__ void wide_cluster_sync() {
  __syncthreads();
  cluster_sync_all();
}

// ---------------------------------------------------------------------------
// Block primitives for kWideThreads threads.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t wide_excl_scan_u64(uint64_t v, uint64_t *scratch,
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
    const uint64_t s = lane < kWideWarps ? scratch[lane] : 0ull;
    uint64_t inc = s;
#pragma unroll
    for (int o = 1; o < kWideWarps; o <<= 1) {
      const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
      if (lane >= static_cast<uint32_t>(o)) inc += t;
    }
    if (lane < kWideWarps) scratch[lane] = inc - s;
    if (lane == kWideWarps - 1) scratch[kWideWarps] = inc;
  }
  __syncthreads();
  *total = scratch[kWideWarps];
  return scratch[wid] + x - v;
}

__device__ __forceinline__ uint32_t wide_max_u32(uint32_t v, uint64_t *scratch) {
  const uint32_t x = __reduce_max_sync(0xFFFFFFFFu, v);
  const uint32_t lane = lane_id(), wid = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[wid] = x;
  __syncthreads();
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < kWideWarps; ++i) r = max(r, static_cast<uint32_t>(scratch[i]));
  return r;
}

// Selects, from a histogram of PER * kWideThreads bins in ascending key
// order (thread t owns bins [t*PER, t*PER + PER)), the bin holding the kk-th
// largest element (1-based).  Writes the bin, the count above it and its
// count to misc.  `h` may live in another CTA of the cluster when G > 1
// (distributed shared memory, summed over the G CTAs).
template <int PER, int G>
__device__ void wide_select_top(const uint32_t *h, uint32_t kk, uint32_t *misc,
                                uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  uint32_t hb[PER];
#pragma unroll
  for (int b = 0; b < PER; ++b) hb[b] = 0u;
  if constexpr (G == 1) {
#pragma unroll
    for (int b = 0; b < PER; ++b) hb[b] = h[t * PER + b];
  } else {
#pragma unroll
    for (int c = 0; c < G; ++c) {
#pragma unroll
      for (int b = 0; b < PER; ++b) hb[b] += dsmem_ld_u32(dsmem_addr(&h[t * PER + b], c));
    }
  }
  uint32_t s = 0;
#pragma unroll
  for (int b = 0; b < PER; ++b) s += hb[b];
  uint64_t tot64;
  const uint32_t excl = static_cast<uint32_t>(wide_excl_scan_u64(s, scratch, &tot64));
  const uint32_t above_me = static_cast<uint32_t>(tot64) - excl - s;
  if (s != 0 && above_me < kk && above_me + s >= kk) {
    uint32_t run = above_me;
#pragma unroll
    for (int b = PER - 1; b >= 0; --b) {
      if (run < kk && run + hb[b] >= kk) {
        misc[kWDigit] = static_cast<uint32_t>(t * PER + b);
        misc[kWAbove] = run;
        misc[kWCount] = hb[b];
      }
      run += hb[b];
    }
  }
  __syncthreads();
}

// Exact r-th largest canonical key of an evenly spaced sample of the row
// (every CTA of the cluster computes the same value from the same sample):
// up to 512 16-byte chunks, taken as runs of RUN consecutive chunks at
// evenly spaced starts (RUN = 8: 128-byte runs, a fraction of the DRAM
// sectors that 512 scattered chunks touch).  Returns 0 ("every element") when
// the sample cannot give a useful bound.
template <int RUN = 1>
__device__ uint32_t wide_sample_threshold(const char *rowp, int V, int k_eff, int G,
                                          uint32_t *hist, uint32_t *misc, uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  const int head_r =
      min(V, static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(rowp) & 15u)) & 15u) / 2u));
  const int nq_r = (V - head_r) / 8;
  const int n_runs = min(nq_r, kWideSampleChunks) / RUN;
  const int n_chunks = n_runs * RUN;
  const int stride = n_runs > 0 ? nq_r / n_runs : 0;  // >= RUN
  const int n_s = 8 * n_chunks;
  if (n_chunks <= 0) return 0u;
  // r such that about 1.6 k_eff row elements (at most 3/4 of the cluster's
  // candidate buffers) are expected at or above it
  const long long expect10 = min(16ll * k_eff, 75ll * wide_cap(G) * G / 10);
  const long long want = (expect10 * n_s + 10ll * V - 1) / (10ll * V);
  const int r = static_cast<int>(max(32ll, want));
  if (r > n_s) return 0u;
  const char *body = rowp + 2 * head_r;
  constexpr int kPerT = kWideSampleChunks / kWideThreads;
  for (int i = t; i < 2048; i += kWideThreads) hist[i] = 0u;
  if (t < 32) misc[kWHist2 + t] = 0u;
  __syncthreads();
  uint32_t kw[kPerT][4];
#pragma unroll
  for (int i = 0; i < kPerT; ++i) {
    const int j = t + i * kWideThreads;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (j < n_chunks) {
      const long long q = RUN == 1 ? static_cast<long long>(j) * nq_r / n_chunks
                                   : static_cast<long long>(j / RUN) * stride + j % RUN;
      v = __ldg(reinterpret_cast<const uint4 *>(body + 16 * q));
    }
    kw[i][0] = wkey_word(v.x);
    kw[i][1] = wkey_word(v.y);
    kw[i][2] = wkey_word(v.z);
    kw[i][3] = wkey_word(v.w);
  }
#pragma unroll
  for (int i = 0; i < kPerT; ++i) {
    if (t + i * kWideThreads < n_chunks) {
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        atomicAdd(&hist[(kw[i][x] & 0xFFFFu) >> 5], 1u);
        atomicAdd(&hist[kw[i][x] >> 21], 1u);
      }
    }
  }
  __syncthreads();
  wide_select_top<8, 1>(hist, static_cast<uint32_t>(r), misc, scratch);
  const uint32_t b1 = misc[kWDigit];
  const uint32_t above = misc[kWAbove];
#pragma unroll
  for (int i = 0; i < kPerT; ++i) {
    if (t + i * kWideThreads < n_chunks) {
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const uint32_t lo = kw[i][x] & 0xFFFFu, hi = kw[i][x] >> 16;
        if ((lo >> 5) == b1) atomicAdd(&misc[kWHist2 + (lo & 31u)], 1u);
        if ((hi >> 5) == b1) atomicAdd(&misc[kWHist2 + (hi & 31u)], 1u);
      }
    }
  }
  __syncthreads();
  // 32 bins: threads 0..31 own one bin each (PER = 1 over the first 32 threads)
  uint32_t d2 = 0;
  if (t < 32) {
    const uint32_t kk = static_cast<uint32_t>(r) - above;
    const uint32_t c = misc[kWHist2 + t];
    // suffix count over bins >= t
    uint32_t suf = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_down_sync(0xFFFFFFFFu, suf, o);
      if (t + o < 32) suf += x;
    }
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, suf >= kk);
    d2 = 31u - __clz(hit);
  }
  __syncthreads();  // everyone has read misc before it is reused
  uint32_t tk = (b1 << 5) | d2;
  if (t >= 32) tk = 0;  // only warp 0 holds d2; broadcast below
  if (t == 0) misc[kWTKey] = tk;
  __syncthreads();
  tk = misc[kWTKey];
  if (tk < KeyBF16::kNegInf || tk >= KeyBF16::kPosInf) tk = 0u;
  return tk;
}

// One candidate: its entry (key << 16 | slice index), its per-key count, its
// count by key >> 8 and the running maximum key.
// The count keeps growing past the buffer (the caller compares it with
// the capacity) and the entry is then dropped; a key beyond the counted
// window raises `range`.
__device__ __forceinline__ void wide_keep(uint32_t key, uint32_t idx, uint32_t pos,
                                          uint32_t t_key, uint32_t *cand, uint32_t cap,
                                          uint32_t *lh, uint32_t *pg, uint32_t &range,
                                          uint32_t &kmax) {
  if (pos < cap) cand[pos] = (key << 16) | idx;
  atomicAdd(&pg[key >> 8], 1u);
  kmax = max(kmax, key);
  const uint32_t off = key - t_key;
  if (off < static_cast<uint32_t>(kWideBins))
    atomicAdd(&lh[off >> 1], 1u << ((off & 1u) * 16u));
  else
    range = 1u;
}

// Drains n <= 32 staged words (two logits each) from a warp's ring: lane l
// takes entry head + l; every element with key >= t_key becomes a
// candidate.  NaN / +inf keys raise `bad`.
__device__ __forceinline__ void wide_drain(const uint2 *ring, uint32_t head, uint32_t n,
                                           uint32_t t_key, uint32_t *cand, uint32_t cap,
                                           uint32_t *lh, uint32_t *pg, uint32_t *counter,
                                           uint32_t &bad, uint32_t &range, uint32_t &kmax) {
  const uint32_t lane = lane_id();
  bool f0 = false, f1 = false;
  uint32_t k0 = 0, k1 = 0, idx0 = 0;
  if (lane < n) {
    const uint2 e = ring[(head + lane) & (kWideRing - 1)];
    const uint32_t kw = wkey_word(e.x);
    k0 = kw & 0xFFFFu;
    k1 = kw >> 16;
    idx0 = e.y;
    const bool nf0 = k0 < KeyBF16::kNegInf || k0 >= KeyBF16::kPosInf;
    const bool nf1 = k1 < KeyBF16::kNegInf || k1 >= KeyBF16::kPosInf;
    bad |= nf0 | nf1;
    f0 = !nf0 && k0 >= t_key;
    f1 = !nf1 && k1 >= t_key;
  }
  const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, f0), b1 = __ballot_sync(0xFFFFFFFFu, f1);
  const uint32_t total = __popc(b0) + __popc(b1);
  if (total == 0) return;
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(counter, total);
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  const uint32_t lt = lanemask_lt();
  const uint32_t pos = base + __popc(b0 & lt) + __popc(b1 & lt);
  if (f0) wide_keep(k0, idx0, pos, t_key, cand, cap, lh, pg, range, kmax);
  if (f1) wide_keep(k1, idx0 + 1u, pos + (f0 ? 1u : 0u), t_key, cand, cap, lh, pg, range, kmax);
}

// One element of a slice's unaligned head or tail.
__device__ __forceinline__ void wide_append_one(const char *sp, int idx, uint32_t t_key,
                                                uint32_t *cand, uint32_t cap, uint32_t *lh,
                                                uint32_t *pg, uint32_t *counter, uint32_t &bad,
                                                uint32_t &range, uint32_t &kmax) {
  const uint32_t k = wkey(KeyBF16::load_one(sp, idx));
  const bool nonfinite = k < KeyBF16::kNegInf || k >= KeyBF16::kPosInf;
  bad |= nonfinite;
  if (!nonfinite && k >= t_key)
    wide_keep(k, static_cast<uint32_t>(idx), atomicAdd(counter, 1u), t_key, cand, cap, lh, pg,
              range, kmax);
}

// Appends one entry of the exact path (at most k_eff <= 4096 per CTA, so
// within every capacity); out-of-range positions are dropped defensively.
__device__ __forceinline__ void wide_put(uint32_t *cand, uint32_t *counter, uint32_t e) {
  const uint32_t pos = atomicAdd(counter, 1u);
  if (pos < static_cast<uint32_t>(kWideCandMaxWide)) cand[pos] = e;
}

// Exact path of a cluster (rare: the sample's threshold left fewer than
// k_eff candidates or more than the buffer holds): radix select over the
// slices re-read from global memory (11 + 5 key bits, histograms merged
// through distributed shared memory), then the exact top-k set collected
// into each CTA's candidate buffer: every key above the threshold, and the
// lowest-index keys equal to it (ranked in index order across the cluster).
// Returns false when the row has no finite logit or holds a NaN / +inf
// (the caller reports the error), true otherwise.
template <int G>
__device__ bool wide_exact_collect(const char *sp, int head, int nq, int tail, uint32_t rank,
                                   uint32_t k_eff, uint32_t *cand, uint32_t *hist, uint32_t *pg,
                                   uint32_t *misc, uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  const char *body = sp + 2 * head;
  for (int i = t; i < 2048; i += kWideThreads) hist[i] = 0u;
  if (t < 32) misc[kWHist2 + t] = 0u;
  if (t == 0) {
    misc[kWBad] = 0u;
    misc[kWFin] = 0u;
  }
  __syncthreads();
  // pass 1: 11-bit histogram, NaN / +inf and finite counts
  uint32_t nbad = 0, nfin = 0;
  auto count1 = [&](uint32_t k) {
    nbad += (k < KeyBF16::kNegInf) | (k >= KeyBF16::kPosInf);
    nfin += k > KeyBF16::kNegInf;
    atomicAdd(&hist[k >> 5], 1u);
  };
  for (int m = t; m < nq; m += kWideThreads) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(body + 16 * static_cast<size_t>(m)));
    const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const uint32_t kw = wkey_word(wds[x]);
      count1(kw & 0xFFFFu);
      count1(kw >> 16);
    }
  }
  if (t < head + tail) {
    const int idx = t < head ? t : head + 8 * nq + (t - head);
    count1(wkey(KeyBF16::load_one(sp, idx)));
  }
  nbad = __reduce_add_sync(0xFFFFFFFFu, nbad);
  nfin = __reduce_add_sync(0xFFFFFFFFu, nfin);
  if (lane_id() == 0) {
    if (nbad) atomicAdd(&misc[kWBad], nbad);
    if (nfin) atomicAdd(&misc[kWFin], nfin);
  }
  __syncthreads();
  if constexpr (G > 1) wide_cluster_sync();
  uint32_t bad = 0, fin = 0;
#pragma unroll
  for (int c = 0; c < G; ++c) {
    if constexpr (G == 1) {
      bad += misc[kWBad];
      fin += misc[kWFin];
    } else {
      bad += dsmem_ld_u32(dsmem_addr(&misc[kWBad], c));
      fin += dsmem_ld_u32(dsmem_addr(&misc[kWFin], c));
    }
  }
  wide_select_top<8, G>(hist, k_eff, misc, scratch);
  if (bad != 0 || fin == 0) {
    if constexpr (G > 1) wide_cluster_sync();  // peers may still read our histogram
    return false;
  }
  const uint32_t b1 = misc[kWDigit];
  uint32_t kk = k_eff - misc[kWAbove];
  // pass 2: the low 5 key bits inside bin b1
  auto count2 = [&](uint32_t k) {
    if ((k >> 5) == b1) atomicAdd(&misc[kWHist2 + (k & 31u)], 1u);
  };
  for (int m = t; m < nq; m += kWideThreads) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(body + 16 * static_cast<size_t>(m)));
    const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const uint32_t kw = wkey_word(wds[x]);
      count2(kw & 0xFFFFu);
      count2(kw >> 16);
    }
  }
  if (t < head + tail) {
    const int idx = t < head ? t : head + 8 * nq + (t - head);
    count2(wkey(KeyBF16::load_one(sp, idx)));
  }
  __syncthreads();
  if constexpr (G > 1) wide_cluster_sync();
  // merged 32-bin select by warp 0
  if (t < 32) {
    uint32_t c = 0;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if constexpr (G == 1)
        c += misc[kWHist2 + t];
      else
        c += dsmem_ld_u32(dsmem_addr(&misc[kWHist2 + t], g));
    }
    uint32_t suf = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_down_sync(0xFFFFFFFFu, suf, o);
      if (t + o < 32) suf += x;
    }
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, suf >= kk);
    const uint32_t d2 = 31u - __clz(hit);
    const uint32_t above2 = __shfl_sync(0xFFFFFFFFu, suf - c, d2);
    // keys equal to the threshold in lower-ranked CTAs (index order)
    uint32_t eq_before = 0;
    if (t < static_cast<int>(rank)) {
      if constexpr (G > 1) eq_before = dsmem_ld_u32(dsmem_addr(&misc[kWHist2 + d2], t));
    }
    eq_before = __reduce_add_sync(0xFFFFFFFFu, eq_before);
    if (t == 0) {
      const uint32_t need = kk - above2;  // keys equal to the threshold that are kept
      const uint32_t mine = misc[kWHist2 + d2];
      const uint32_t take = need > eq_before ? min(need - eq_before, mine) : 0u;
      misc[kWTKey] = (b1 << 5) | d2;
      misc[kWTake] = take;
      misc[kWN] = 0u;
    }
  }
  pg[threadIdx.x] = 0u;  // kWideThreads == 256 page counts, rebuilt for the exact set
  __syncthreads();
  if constexpr (G > 1) wide_cluster_sync();  // peers are done reading our histograms
  const uint32_t thr = misc[kWTKey];
  const uint32_t take = misc[kWTake];
  uint32_t *counter = &misc[kWN];
  uint32_t kmax = 0;
  auto put = [&](uint32_t k, uint32_t idx) {
    wide_put(cand, counter, (k << 16) | idx);
    atomicAdd(&pg[k >> 8], 1u);
    kmax = max(kmax, k);
  };
  // pass 3: collect.  Keys above thr in any order; keys equal to thr in
  // index order until `take` of them.  Head elements first (thread 0, in
  // order), then the body in rounds of kWideThreads chunks, then the tail.
  uint32_t eq_seen = 0;  // uniform: equal keys already met in this slice
  if (t == 0) {
    for (int idx = 0; idx < head; ++idx) {
      const uint32_t k = wkey(KeyBF16::load_one(sp, idx));
      bool keep = k > thr;
      if (k == thr) keep = eq_seen++ < take;
      if (keep) put(k, static_cast<uint32_t>(idx));
    }
    misc[kWEq] = eq_seen;
  }
  __syncthreads();
  eq_seen = misc[kWEq];
  const int rounds = (nq + kWideThreads - 1) / kWideThreads;
#pragma unroll 1
  for (int j = 0; j < rounds; ++j) {
    const int m = j * kWideThreads + t;
    uint32_t k[8];
    uint32_t ne = 0;
    if (m < nq) {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(body + 16 * static_cast<size_t>(m)));
      const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const uint32_t kw = wkey_word(wds[x]);
        k[2 * x] = kw & 0xFFFFu;
        k[2 * x + 1] = kw >> 16;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) ne += k[e] == thr;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) k[e] = 0u;
    }
    uint64_t tot;
    uint32_t er = eq_seen + static_cast<uint32_t>(wide_excl_scan_u64(ne, scratch, &tot));
    if (m < nq) {
      const uint32_t idx0 = static_cast<uint32_t>(head) + 8u * static_cast<uint32_t>(m);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        bool keep = k[e] > thr;
        if (k[e] == thr) keep = er++ < take;
        if (keep) put(k[e], idx0 + e);
      }
    }
    eq_seen += static_cast<uint32_t>(tot);
  }
  __syncthreads();
  if (t == 0) {
    for (int j = 0; j < tail; ++j) {
      const int idx = head + 8 * nq + j;
      const uint32_t k = wkey(KeyBF16::load_one(sp, idx));
      bool keep = k > thr;
      if (k == thr) keep = eq_seen++ < take;
      if (keep) put(k, static_cast<uint32_t>(idx));
    }
  }
  kmax = wide_max_u32(kmax, scratch);
  if (threadIdx.x == 0) misc[kWMaxK] = kmax;
  __syncthreads();
  return true;
}

// The rho-th smallest (0-based) slice index among this CTA's candidates
// with key `key_sel`: a two-level radix select on the 16-bit slice index
// (256 bins per level).  Order-free.
__device__ uint32_t wide_local_rank_select(const uint32_t *cand, int n, uint32_t key_sel,
                                           uint32_t rho, uint32_t *h, uint32_t *misc,
                                           uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  uint32_t b1 = 0, below = 0;
#pragma unroll 1
  for (int level = 0; level < 2; ++level) {
    __syncthreads();
    h[t] = 0u;  // kWideThreads == 256 bins
    __syncthreads();
    for (int i = t; i < n; i += kWideThreads) {
      const uint32_t e = cand[i];
      if ((e >> 16) != key_sel) continue;
      const uint32_t idx = e & 0xFFFFu;
      if (level == 0)
        atomicAdd(&h[idx >> 8], 1u);
      else if ((idx >> 8) == b1)
        atomicAdd(&h[idx & 255u], 1u);
    }
    __syncthreads();
    const uint32_t want = rho - below;
    const uint32_t c = h[t];
    uint64_t tot;
    const uint32_t ex = static_cast<uint32_t>(wide_excl_scan_u64(c, scratch, &tot));
    if (ex <= want && want < ex + c) {
      misc[kWDigit] = static_cast<uint32_t>(t);
      misc[kWAbove] = ex;
    }
    __syncthreads();
    if (level == 0) {
      b1 = misc[kWDigit];
      below = misc[kWAbove];
    } else {
      return (b1 << 8) | misc[kWDigit];
    }
  }
  return 0;
}

__device__ __forceinline__ uint32_t dsmem_atomic_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

// Fast tail.  Every CTA of the cluster merges the G per-key candidate counts
// (keys t .. t + kWideBins - 1) and, redundantly so that none waits for
// another, finds the threshold key and the kept count tied at it, the
// masses (one weight per key), the nucleus cutoff and the draw; the CTA that
// holds the drawn token (index order = CTA order) picks it from its own
// candidates.  Bins: thread j owns keys t + 8j .. t + 8j + 7.
template <int G>
__device__ void wide_fast_tail(const Params &p, int r, const Row &w, uint32_t rank, int S,
                               uint32_t t_key, const uint32_t *cand, int n_loc,
                               const uint32_t *lh, uint32_t *hsel, uint32_t *misc,
                               uint64_t *scratch) {
  constexpr int kPer = kWideBins / kWideThreads;
  static_assert(kPer == 8, "two packed words per uint4 load");
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t lane = lane_id();
  const uint32_t k_eff = static_cast<uint32_t>(w.k_eff);
  uint64_t *m64 = reinterpret_cast<uint64_t *>(misc);

  // ---- merged per-key counts (packed 16-bit pairs add without carries) ----
  uint32_t c[kPer];
  {
    uint4 acc = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      uint4 v;
      if constexpr (G == 1)
        v = reinterpret_cast<const uint4 *>(lh)[t];
      else
        v = dsmem_ld_v4(dsmem_addr(&lh[4 * t], g));
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const uint32_t wd[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      c[2 * j] = wd[j] & 0xFFFFu;
      c[2 * j + 1] = wd[j] >> 16;
    }
  }
  // ---- highest populated key, threshold key (k_eff-th largest) ----
  uint32_t s = 0, hi = 0;
#pragma unroll
  for (int b = 0; b < kPer; ++b) {
    s += c[b];
    if (c[b]) hi = static_cast<uint32_t>(kPer * t + b) + 1u;
  }
  const uint32_t maxb = wide_max_u32(hi, scratch) - 1u;
  if (t_key + maxb <= KeyBF16::kNegInf) {  // every candidate is -inf: no finite logit in the row
    if (rank == 0 && t == 0) finish_row(p, r, w, -1, kRowNonFinite);
    return;
  }
  uint64_t tot;
  const uint32_t excl = static_cast<uint32_t>(wide_excl_scan_u64(s, scratch, &tot));
  const uint32_t above_cnt = static_cast<uint32_t>(tot) - excl - s;  // kept above my keys
  if (s != 0 && above_cnt < k_eff && above_cnt + s >= k_eff) {
    uint32_t run = above_cnt;
#pragma unroll
    for (int b = kPer - 1; b >= 0; --b) {
      if (run < k_eff && run + c[b] >= k_eff) {
        misc[kWThrB] = static_cast<uint32_t>(kPer * t + b);
        misc[kWNeed] = k_eff - run;
      }
      run += c[b];
    }
  }
  __syncthreads();
  const uint32_t thr_b = misc[kWThrB], need = misc[kWNeed];
  const float m = KeyBF16::value(t_key + maxb);
  const uint32_t u24 = misc[kWU24];
  uint32_t draw_b = maxb, rho = 0, n_p = 1;
  uint64_t s_k = 0;
  if (!w.greedy) {
    // ---- masses: count x weight of the key (the threshold key: need) ----
    uint64_t mass[kPer];
    uint64_t st = 0;
#pragma unroll
    for (int b = 0; b < kPer; ++b) {
      const uint32_t bin = static_cast<uint32_t>(kPer * t + b);
      const uint32_t cnt = bin > thr_b ? c[b] : (bin == thr_b ? need : 0u);
      mass[b] = cnt ? cnt * to_fixed(kept_weight(KeyBF16::value(t_key + bin), m, w.temp,
                                                 w.inv_temp))
                    : 0ull;
      st += mass[b];
    }
    const uint64_t ex_m = wide_excl_scan_u64(st, scratch, &s_k);
    const uint64_t above_m = s_k - ex_m - st;  // mass above my keys
    // ---- nucleus cutoff ----
    uint64_t s_p;
    if (w.top_p >= 1.0f) {
      n_p = k_eff;
      s_p = s_k;
    } else if (!(w.top_p > 0.0f)) {
      n_p = 1;
      s_p = to_fixed(kept_weight(m, m, w.temp, w.inv_temp));
    } else {
      const uint64_t cut = ceil_mul_p(w.top_p, s_k);  // C reaches top_p * S_k iff C >= cut
      if (st != 0 && above_m < cut && above_m + st >= cut) {
        uint64_t cum = above_m;
        uint32_t cnt_above = above_cnt;
#pragma unroll
        for (int b = kPer - 1; b >= 0; --b) {
          if (cum < cut && cum + mass[b] >= cut) {
            const uint32_t bin = static_cast<uint32_t>(kPer * t + b);
            const uint64_t wb =
                to_fixed(kept_weight(KeyBF16::value(t_key + bin), m, w.temp, w.inv_temp));
            uint64_t n_c = (cut - cum + wb - 1) / wb;
            if (n_c < 1) n_c = 1;
            m64[kWSp / 2] = cum + n_c * wb;
            misc[kWNp] = cnt_above + static_cast<uint32_t>(n_c);
          }
          cum += mass[b];
          cnt_above += c[b];
        }
      }
      __syncthreads();
      s_p = m64[kWSp / 2];
      n_p = misc[kWNp];
    }
    // ---- draw: the key group whose cumulative mass first exceeds target ----
    const uint64_t target = scale_u24(u24, s_p);
    if (st != 0 && above_m <= target && target < above_m + st) {
      uint64_t cum = above_m;
#pragma unroll
      for (int b = kPer - 1; b >= 0; --b) {
        if (cum <= target && target < cum + mass[b]) {
          const uint32_t bin = static_cast<uint32_t>(kPer * t + b);
          const uint64_t wb =
              to_fixed(kept_weight(KeyBF16::value(t_key + bin), m, w.temp, w.inv_temp));
          misc[kWDrawB] = bin;
          misc[kWRho] = static_cast<uint32_t>((target - cum) / wb);
        }
        cum += mass[b];
      }
    }
    __syncthreads();
    draw_b = misc[kWDrawB];
    rho = misc[kWRho];
  }
  // ---- the CTA holding the drawn token (index order = CTA order) ----
  if (t < 32) {
    uint32_t cnt = 0;
    if (lane < static_cast<uint32_t>(G)) {
      uint32_t word;
      if constexpr (G == 1)
        word = lh[draw_b >> 1];
      else
        word = dsmem_ld_u32(dsmem_addr(&lh[draw_b >> 1], lane));
      cnt = (word >> ((draw_b & 1u) * 16u)) & 0xFFFFu;
    }
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= static_cast<uint32_t>(o)) incl += x;
    }
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl > rho && lane < static_cast<uint32_t>(G));
    const uint32_t owner = hit ? static_cast<uint32_t>(__ffs(hit) - 1) : 0u;
    const uint32_t before = __shfl_sync(0xFFFFFFFFu, incl - cnt, owner);
    if (t == 0) {
      misc[kWOwner] = owner;
      misc[kWRho2] = rho - before;
    }
  }
  __syncthreads();
  const uint32_t owner = misc[kWOwner];
  uint32_t sel = 0xFFFFFFFFu;
  if (rank == owner) {
    sel = wide_local_rank_select(cand, n_loc, t_key + draw_b, misc[kWRho2], hsel, misc, scratch);
    if (t == 0) finish_row(p, r, w, static_cast<int32_t>(rank * S + sel), 0u);
  }
  if (p.kept_ids) {
    // this CTA's share of the keys tied at the threshold: the lowest indices
    // of the row first, and CTA order is index order
    if (t < 32) {
      uint32_t e = 0;
      if (lane < rank) {
        if constexpr (G > 1) {
          const uint32_t word = dsmem_ld_u32(dsmem_addr(&lh[thr_b >> 1], lane));
          e = (word >> ((thr_b & 1u) * 16u)) & 0xFFFFu;
        }
      }
      const uint32_t before = __reduce_add_sync(0xFFFFFFFFu, e);
      if (t == 0) {
        const uint32_t mine = (lh[thr_b >> 1] >> ((thr_b & 1u) * 16u)) & 0xFFFFu;
        misc[kWTake] = need > before ? min(need - before, mine) : 0u;
        misc[kWEq] = mine;
      }
    }
    __syncthreads();
    const uint32_t take = misc[kWTake], mine = misc[kWEq];
    uint32_t cut_idx = take ? 0xFFFFu : 0u;
    if (take != 0 && take < mine)
      cut_idx = wide_local_rank_select(cand, n_loc, t_key + thr_b, take - 1, hsel, misc, scratch);
    const float s_real = static_cast<float>(static_cast<double>(s_k) * (1.0 / 1099511627776.0));
    const int64_t rb = static_cast<int64_t>(r) * p.max_keep;
    const uint32_t kept_addr = G > 1 ? dsmem_addr(&misc[kWKept], 0) : 0u;
    for (int i = t; i < n_loc; i += kWideThreads) {
      const uint32_t e = cand[i];
      const uint32_t key = e >> 16, idx = e & 0xFFFFu;
      const uint32_t bin = key - t_key;
      const bool keep = bin > thr_b || (bin == thr_b && take != 0 && idx <= cut_idx);
      if (!keep) continue;
      uint32_t pos;
      if constexpr (G > 1)
        pos = dsmem_atomic_add(kept_addr, 1u);
      else
        pos = atomicAdd(&misc[kWKept], 1u);
      if (pos < static_cast<uint32_t>(p.max_keep)) {
        p.kept_ids[rb + pos] = static_cast<int32_t>(rank * S + idx);
        p.kept_probs[rb + pos] =
            w.greedy ? ((rank == owner && idx == sel) ? 1.f : 0.f)
                     : __fdiv_rn(kept_weight(KeyBF16::value(key), m, w.temp, w.inv_temp), s_real);
      }
    }
    if (rank == 0 && t == 0) {
      p.n_kept[r] = static_cast<int32_t>(k_eff);
      p.n_nucleus[r] = static_cast<int32_t>(n_p);
    }
  }
}

// Reads word `i` of CTA c's shared array `a` (c == this CTA when G == 1).
template <int G>
__device__ __forceinline__ uint32_t wide_peer_u32(const uint32_t *a, int i, int c) {
  if constexpr (G == 1)
    return a[i];
  else
    return dsmem_ld_u32(dsmem_addr(&a[i], c));
}
template <int G>
__device__ __forceinline__ uint4 wide_peer_v4(const uint32_t *a, int i, int c) {
  if constexpr (G == 1)
    return *reinterpret_cast<const uint4 *>(&a[i]);
  else
    return dsmem_ld_v4(dsmem_addr(&a[i], c));
}

// Cluster barrier (or a block barrier for a single CTA).
template <int G>
__device__ __forceinline__ void wide_sync_all() {
  if constexpr (G > 1)
    wide_cluster_sync();
  else
    __syncthreads();
}

// Sum over the G CTAs of word i of the shared arrays a[0..N-1]; every
// remote load is issued before any is used.
template <int G, int N>
__device__ __forceinline__ void wide_sum_peers(const uint32_t *const (&a)[N], int i,
                                               uint32_t (&out)[N]) {
  if constexpr (G == 1) {
#pragma unroll
    for (int j = 0; j < N; ++j) out[j] = a[j][i];
  } else {
    uint32_t v[N][G];
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(&a[j][i]));
#pragma unroll
      for (int c = 0; c < G; ++c) {
        uint32_t ra;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(base), "r"(c));
        v[j][c] = dsmem_ld_u32(ra);
      }
    }
#pragma unroll
    for (int j = 0; j < N; ++j) {
      uint32_t sum = 0;
#pragma unroll
      for (int c = 0; c < G; ++c) sum += v[j][c];
      out[j] = sum;
    }
  }
}

template <int G>
__device__ __forceinline__ uint32_t wide_sum_peers1(const uint32_t *a, int i) {
  const uint32_t *arr[1] = {a};
  uint32_t out[1];
  wide_sum_peers<G, 1>(arr, i, out);
  return out[0];
}

// 256 bins in ascending key order, bin t held by thread t: the bin holding
// the kk-th largest element (bin -> misc[kWDigit], count above it ->
// misc[kWAbove]).  Ends with a block barrier.
__device__ __forceinline__ void wide_select256(uint32_t c, uint32_t kk, uint32_t *misc,
                                               uint64_t *scratch) {
  uint64_t tot;
  const uint32_t ex = static_cast<uint32_t>(wide_excl_scan_u64(c, scratch, &tot));
  const uint32_t above = static_cast<uint32_t>(tot) - ex - c;
  if (c != 0 && above < kk && above + c >= kk) {
    misc[kWDigit] = threadIdx.x;
    misc[kWAbove] = above;
  }
  __syncthreads();
}

// This CTA's kept-key counts inside coarse bin `bin` (keys maxk - (bin <<
// shift) - j, j < 2^shift <= 256; the key at thr is counted apart).
__device__ __forceinline__ void wide_local_level2(const uint32_t *cand, int n, uint32_t maxk,
                                                  uint32_t thr, int shift, uint32_t bin,
                                                  uint32_t *l2) {
  const int t = static_cast<int>(threadIdx.x);
  l2[t] = 0u;
  __syncthreads();
#pragma unroll 4
  for (int i = t; i < n; i += kWideThreads) {
    const uint32_t key = cand[i] >> 16;
    const uint32_t off = maxk - key;
    if (key > thr && (off >> shift) == bin) atomicAdd(&l2[off & ((1u << shift) - 1u)], 1u);
  }
}

// Merged second level: thread j weighs key base - j (the G CTAs' counts plus
// the `need` kept tokens at thr); finds the key where the cumulative mass
// from the top (starting at `above`) first reaches `goal` (cut_mode) or first
// exceeds it.  Writes the key, the mass above it and the kept count above it
// inside the bin to misc.  Ends with a block barrier.
template <int G>
__device__ void wide_merge_level2(const uint32_t *l2, uint32_t maxk, uint32_t thr, uint32_t need,
                                  int shift, uint32_t bin, float m, float temp, float inv_temp,
                                  bool cut_mode, uint64_t goal, uint64_t above, uint32_t *misc,
                                  uint64_t *scratch) {
  const uint32_t j = threadIdx.x;
  uint64_t *m64 = reinterpret_cast<uint64_t *>(misc);
  const uint32_t base = maxk - (bin << shift);
  uint32_t c = 0;
  if (j < (1u << shift)) {
    c = wide_sum_peers1<G>(l2, static_cast<int>(j));
    if (((maxk - thr) >> shift) == bin && j == ((maxk - thr) & ((1u << shift) - 1u))) c += need;
  }
  const uint64_t ms = c ? c * to_fixed(kept_weight(KeyBF16::value(base - j), m, temp, inv_temp)) : 0ull;
  uint64_t tm, tc;
  const uint64_t cum = above + wide_excl_scan_u64(ms, scratch, &tm);
  const uint32_t ccum = static_cast<uint32_t>(wide_excl_scan_u64(c, scratch, &tc));
  const uint64_t nxt = cum + ms;
  const bool hit = cut_mode ? (cum < goal && nxt >= goal) : (cum <= goal && goal < nxt);
  if (hit) {
    misc[kWDigit] = base - j;
    m64[kWSp / 2] = cum;
    misc[kWCount] = ccum;
  }
  __syncthreads();
}

// Distributed tail (any key range).  Every CTA of the cluster keeps its own
// candidates (together a superset of the top-k set that holds every key
// tied with the k_eff-th largest); each pass runs over the CTA's own
// candidates and 256-bin histograms are merged through distributed shared
// memory, every CTA reaching the same decisions:
//   1. counts by key >> 8 (built during the filter) -> the threshold's page;
//   2. the low key byte inside that page -> the threshold key thr and
//      `need`, the kept tokens tied at it (the lowest indices of the row);
//   3. kept masses and counts over (maxk - key) >> shift (256 coarse bins;
//      the only pass that evaluates exp per token) -> S_k and the coarse
//      bins of the nucleus cutoff and of the draw;
//   4. an exact level inside each of those two bins (when shift > 0);
//   5. the CTA holding the drawn token (index order = CTA order) picks it by
//      a radix select on its slice index.
// The caller ends with a cluster barrier (peers read this CTA's histograms).
template <int G>
__device__ void wide_dist_tail(const Params &p, int r, const Row &w, uint32_t rank, int S,
                               const uint32_t *cand, int n, uint32_t *hw, const uint32_t *pg,
                               uint32_t *misc, uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t lane = lane_id();
  const uint32_t k_eff = static_cast<uint32_t>(w.k_eff);
  uint64_t *m64 = reinterpret_cast<uint64_t *>(misc);
  uint32_t *bB = hw;  // low key bytes inside the threshold's page
  uint32_t *plo = hw + 256, *pmid = hw + 512, *phi = hw + 768, *pcnt = hw + 1024;
  uint32_t *lD = hw + 1280;  // second level of the cutoff's coarse bin
  uint32_t *lE = hw + 1536;  // second level of the draw's coarse bin
  uint32_t *rs = hw + 1792;  // rank select

  // ---- 1. the threshold's page, the maximum key ----
  bB[t] = 0u;
  const uint32_t cpage = wide_sum_peers1<G>(pg, t);
  if (t < 32) {
    uint32_t mk = 0;
    if (lane < static_cast<uint32_t>(G)) mk = wide_peer_u32<G>(misc, kWMaxK, static_cast<int>(lane));
    mk = __reduce_max_sync(0xFFFFFFFFu, mk);
    if (t == 0) misc[kWMaxB] = mk;
  }
  wide_select256(cpage, k_eff, misc, scratch);
  const uint32_t maxk = misc[kWMaxB];
  if (maxk <= KeyBF16::kNegInf) {  // every candidate is -inf: no finite logit in the row
    if (rank == 0 && t == 0) finish_row(p, r, w, -1, kRowNonFinite);
    return;
  }
  const uint32_t page = misc[kWDigit];
  const uint32_t kk = k_eff - misc[kWAbove];
  // ---- 2. the threshold key inside that page ----
#pragma unroll 4
  for (int i = t; i < n; i += kWideThreads) {
    const uint32_t key = cand[i] >> 16;
    if ((key >> 8) == page) atomicAdd(&bB[key & 255u], 1u);
  }
  wide_sync_all<G>();
  wide_select256(wide_sum_peers1<G>(bB, t), kk, misc, scratch);
  const uint32_t lowb = misc[kWDigit];
  const uint32_t thr = (page << 8) | lowb;
  const uint32_t need = kk - misc[kWAbove];
  if (t < 32) {  // keys at thr in lower-ranked CTAs (lower token indices)
    uint32_t eb = 0;
    if (lane < rank) eb = wide_peer_u32<G>(bB, static_cast<int>(lowb), static_cast<int>(lane));
    eb = __reduce_add_sync(0xFFFFFFFFu, eb);
    if (t == 0) misc[kWEq] = eb;
  }
  __syncthreads();
  const uint32_t eq_before = misc[kWEq], eq_mine = bB[lowb];
  const float m = KeyBF16::value(maxk);
  const uint32_t u24 = misc[kWU24];
  uint32_t key_d = maxk, rho = 0, n_p = 1;
  uint64_t s_k = 0;
  int shift = 0;
  uint32_t d1 = 0;
  if (!w.greedy) {
    // ---- 3. coarse kept masses and counts over (maxk - key) >> shift ----
    const uint32_t range = maxk - thr;
    const int bits = range ? 32 - __clz(range) : 0;
    shift = bits > 8 ? bits - 8 : 0;
    plo[t] = 0u;
    pmid[t] = 0u;
    phi[t] = 0u;
    pcnt[t] = 0u;
    __syncthreads();
#pragma unroll 4
    for (int i = t; i < n; i += kWideThreads) {
      const uint32_t key = cand[i] >> 16;
      if (key <= thr) continue;
      const uint32_t d = (maxk - key) >> shift;
      atomicAdd(&pcnt[d], 1u);
      if (shift) {
        const uint64_t f = to_fixed(kept_weight(KeyBF16::value(key), m, w.temp, w.inv_temp));
        if (f) {
          atomicAdd(&plo[d], static_cast<uint32_t>(f & 0x1FFFu));
          atomicAdd(&pmid[d], static_cast<uint32_t>((f >> 13) & 0x1FFFu));
          atomicAdd(&phi[d], static_cast<uint32_t>(f >> 26));
        }
      }
    }
    wide_sync_all<G>();
    const uint32_t dthr = (maxk - thr) >> shift;
    uint32_t cs;
    uint64_t ms;
    if (shift == 0) {
      cs = wide_sum_peers1<G>(pcnt, t) + (static_cast<uint32_t>(t) == dthr ? need : 0u);
      ms = cs ? cs * to_fixed(kept_weight(KeyBF16::value(maxk - t), m, w.temp, w.inv_temp)) : 0ull;
    } else {
      const uint32_t *arr[4] = {pcnt, plo, pmid, phi};
      uint32_t v[4];
      wide_sum_peers<G, 4>(arr, t, v);
      cs = v[0];
      ms = (static_cast<uint64_t>(v[3]) << 26) + (static_cast<uint64_t>(v[2]) << 13) + v[1];
      if (static_cast<uint32_t>(t) == dthr && need) {
        cs += need;
        ms += need * to_fixed(kept_weight(KeyBF16::value(thr), m, w.temp, w.inv_temp));
      }
    }
    const uint64_t cum_t = wide_excl_scan_u64(ms, scratch, &s_k);
    uint64_t n_all64;
    const uint32_t ccum_t = static_cast<uint32_t>(wide_excl_scan_u64(cs, scratch, &n_all64));
    // ---- nucleus cutoff ----
    uint64_t s_p;
    if (w.top_p >= 1.0f) {
      n_p = k_eff;
      s_p = s_k;
    } else if (!(w.top_p > 0.0f)) {
      n_p = 1;
      s_p = to_fixed(kept_weight(m, m, w.temp, w.inv_temp));
    } else {
      const uint64_t cut = ceil_mul_p(w.top_p, s_k);  // C reaches top_p * S_k iff C >= cut
      if (cum_t < cut && cum_t + ms >= cut) {
        misc[kWThrB] = static_cast<uint32_t>(t);
        m64[kWWide / 2] = cum_t;
        misc[kWNeed] = ccum_t;
      }
      __syncthreads();
      const uint32_t c1 = misc[kWThrB];
      const uint64_t above_c = m64[kWWide / 2];
      const uint32_t cnt_c = misc[kWNeed];
      uint32_t key_c;
      uint64_t above_k;
      uint32_t cnt_k;
      if (shift == 0) {
        key_c = maxk - c1;
        above_k = above_c;
        cnt_k = cnt_c;
      } else {
        wide_local_level2(cand, n, maxk, thr, shift, c1, lD);
        wide_sync_all<G>();
        wide_merge_level2<G>(lD, maxk, thr, need, shift, c1, m, w.temp, w.inv_temp, true, cut,
                             above_c, misc, scratch);
        key_c = misc[kWDigit];
        above_k = m64[kWSp / 2];
        cnt_k = cnt_c + misc[kWCount];
      }
      const uint64_t wc = to_fixed(kept_weight(KeyBF16::value(key_c), m, w.temp, w.inv_temp));
      uint64_t n_c = wc > 0 ? (cut - above_k + wc - 1) / wc : 1;
      if (n_c < 1) n_c = 1;
      n_p = cnt_k + static_cast<uint32_t>(n_c);
      s_p = above_k + n_c * wc;
      __syncthreads();  // misc is read before it is reused
    }
    // ---- draw ----
    const uint64_t target = scale_u24(u24, s_p);
    if (cum_t <= target && target < cum_t + ms) {
      misc[kWDrawB] = static_cast<uint32_t>(t);
      m64[kWWide / 2] = cum_t;
    }
    __syncthreads();
    d1 = misc[kWDrawB];
    uint64_t above_d = m64[kWWide / 2];
    if (shift == 0) {
      key_d = maxk - d1;
    } else {
      wide_local_level2(cand, n, maxk, thr, shift, d1, lE);
      wide_sync_all<G>();
      wide_merge_level2<G>(lE, maxk, thr, need, shift, d1, m, w.temp, w.inv_temp, false, target,
                           above_d, misc, scratch);
      key_d = misc[kWDigit];
      above_d = m64[kWSp / 2];
    }
    const uint64_t wd = to_fixed(kept_weight(KeyBF16::value(key_d), m, w.temp, w.inv_temp));
    rho = wd > 0 ? static_cast<uint32_t>((target - above_d) / wd) : 0u;
  }
  // ---- 5. the CTA holding the drawn token ----
  // per-CTA counts of key_d: in the threshold's page the low-byte counts;
  // above it the coarse counts (one key per bin when shift == 0) or the
  // draw bin's second level.  A greedy row whose maximum lies above the
  // threshold's page counts its maximum in one more local pass.
  const bool greedy_pass = w.greedy && (maxk >> 8) != page;
  if (greedy_pass) {
    if (t == 0) misc[kWCount] = 0u;
    __syncthreads();
    uint32_t c = 0;
    for (int i = t; i < n; i += kWideThreads) c += (cand[i] >> 16) == maxk;
    if (c) atomicAdd(&misc[kWCount], c);
    wide_sync_all<G>();
  }
  if (t < 32) {
    uint32_t cnt = 0;
    if (lane < static_cast<uint32_t>(G)) {
      const int g = static_cast<int>(lane);
      if (greedy_pass)
        cnt = wide_peer_u32<G>(misc, kWCount, g);
      else if ((key_d >> 8) == page && (w.greedy || key_d == thr))
        cnt = wide_peer_u32<G>(bB, static_cast<int>(key_d & 255u), g);
      else if (shift == 0)
        cnt = wide_peer_u32<G>(pcnt, static_cast<int>(d1), g);
      else
        cnt = wide_peer_u32<G>(lE, static_cast<int>((maxk - key_d) & ((1u << shift) - 1u)), g);
    }
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= static_cast<uint32_t>(o)) incl += x;
    }
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl > rho && lane < static_cast<uint32_t>(G));
    const uint32_t owner = hit ? static_cast<uint32_t>(__ffs(hit) - 1) : 0u;
    const uint32_t before = __shfl_sync(0xFFFFFFFFu, incl - cnt, owner);
    if (t == 0) {
      misc[kWOwner] = owner;
      misc[kWRho2] = rho - before;
    }
  }
  __syncthreads();
  const uint32_t owner = misc[kWOwner];
  uint32_t sel = 0xFFFFFFFFu;
  if (rank == owner) {
    sel = wide_local_rank_select(cand, n, key_d, misc[kWRho2], rs, misc, scratch);
    if (t == 0) finish_row(p, r, w, static_cast<int32_t>(rank * S + sel), 0u);
  }
  if (p.kept_ids) {
    // keys above thr, and this CTA's share of the `need` lowest-index keys at thr
    const uint32_t take = need > eq_before ? min(need - eq_before, eq_mine) : 0u;
    uint32_t cut_idx = take ? 0xFFFFu : 0u;
    if (take != 0 && take < eq_mine)
      cut_idx = wide_local_rank_select(cand, n, thr, take - 1, rs, misc, scratch);
    const float s_real = static_cast<float>(static_cast<double>(s_k) * (1.0 / 1099511627776.0));
    const int64_t rb = static_cast<int64_t>(r) * p.max_keep;
    const uint32_t kept_addr = G > 1 ? dsmem_addr(&misc[kWKept], 0) : 0u;
    for (int i = t; i < n; i += kWideThreads) {
      const uint32_t e = cand[i];
      const uint32_t key = e >> 16, idx = e & 0xFFFFu;
      const bool keep = key > thr || (key == thr && take != 0 && idx <= cut_idx);
      if (!keep) continue;
      uint32_t pos;
      if constexpr (G > 1)
        pos = dsmem_atomic_add(kept_addr, 1u);
      else
        pos = atomicAdd(&misc[kWKept], 1u);
      if (pos < static_cast<uint32_t>(p.max_keep)) {
        p.kept_ids[rb + pos] = static_cast<int32_t>(rank * S + idx);
        p.kept_probs[rb + pos] =
            w.greedy ? ((rank == owner && idx == sel) ? 1.f : 0.f)
                     : __fdiv_rn(kept_weight(KeyBF16::value(key), m, w.temp, w.inv_temp), s_real);
      }
    }
    if (rank == 0 && t == 0) {
      p.n_kept[r] = static_cast<int32_t>(k_eff);
      p.n_nucleus[r] = static_cast<int32_t>(n_p);
    }
  }
}

template <int G>
__global__ void __launch_bounds__(kWideThreads, 4) wide_sampler_kernel(const Params p) {
  constexpr uint32_t kCap = static_cast<uint32_t>(wide_cap(G));
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t *cand = reinterpret_cast<uint32_t *>(smem);
  unsigned char *work = smem + kCap * 4;
  uint32_t *misc = reinterpret_cast<uint32_t *>(work + kWideWorkBytes);
  uint64_t *scratch = reinterpret_cast<uint64_t *>(misc + kWScan);
  uint32_t *lh = reinterpret_cast<uint32_t *>(work + kWideLhOff);  // per-key counts
  uint32_t *mh = reinterpret_cast<uint32_t *>(work + kWideMhOff);  // sample / select histograms
  uint32_t *pg = reinterpret_cast<uint32_t *>(work + kWidePgOff);  // candidate counts by key >> 8

  const uint32_t rank = G > 1 ? cluster_rank() : 0u;
  const int r = G > 1 ? static_cast<int>(cluster_index()) : static_cast<int>(blockIdx.x);
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t lane = lane_id();
  const int warp = t >> 5;
  pdl_wait_and_release();
  if (r >= p.n_rows) return;  // whole cluster (grid is sized exactly)
  const Row w = load_row(p, r);
  if (w.err || w.fin) {  // identical in every CTA of the cluster: all leave before any barrier
    if (rank == 0 && t == 0) finish_row(p, r, w, -1, w.err);
    return;
  }
  if (t == 32) {  // the draw, off the critical path (every CTA may need it)
    misc[kWU24] = philox_u24(p.seed[r], p.request[r], static_cast<uint64_t>(p.step[w.stream]),
                             static_cast<uint64_t>(static_cast<int64_t>(p.codebook[r])));
  }

  // ---- slice geometry ----
  const int V = w.vocab;
  const int S = p.slice;
  const int s_begin = static_cast<int>(rank) * S;
  const int sc = max(0, min(S, V - s_begin));
  const char *rowp = static_cast<const char *>(p.logits) + w.off * 2;
  const char *sp = rowp + 2 * static_cast<int64_t>(s_begin);
  const int head =
      min(sc, static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(sp) & 15u)) & 15u) / 2u));
  const int nq = (sc - head) / 8;
  const int tail = sc - head - 8 * nq;
  const char *body = sp + 2 * head;
  const uint32_t k_eff = static_cast<uint32_t>(w.k_eff);

  // ---- first loads of the slice in flight before the threshold estimate ----
  const uint64_t pol = l2_evict_first();
  constexpr int kPerIter = kWideThreads * kWideU;
  const int n_it = (nq + kPerIter - 1) / kPerIter;
  uint4 cur[kWideU];
#pragma unroll
  for (int u = 0; u < kWideU; ++u) {
    const int m = u * kWideThreads + t;
    cur[u] = m < nq ? ld_stream_v4(body + 16 * static_cast<size_t>(m), pol)
                    : make_uint4(0u, 0u, 0u, 0u);
  }

  // a slice no longer than the buffer keeps every element (no sample)
  uint32_t t_key = 0;
  if (S > static_cast<int>(kCap) && !p.wide_exact)
    t_key = wide_sample_threshold(rowp, V, w.k_eff, G, mh, misc, scratch);
  for (int i = t; i < kWideBins / 2; i += kWideThreads) lh[i] = 0u;
  pg[t] = 0u;  // kWideThreads == 256 pages
  if (t < 16) misc[kWThrB + t] = 0u;  // fast-tail results and the kept-set counter
  if (t == 0) {
    misc[kWN] = 0u;
    misc[kWBad] = 0u;
    misc[kWRange] = 0u;
  }
  __syncthreads();

  // ---- filter: every element with key >= t_key becomes a candidate ----
  uint32_t bad = 0, range = 0, kmax = 0;
  if (!p.wide_exact) {
    const uint32_t tb = wkey_bits(t_key);
    const uint32_t t2 = tb | (tb << 16);
    uint2 *ring = reinterpret_cast<uint2 *>(work) + warp * kWideRing;
    const uint32_t lt = lanemask_lt();
    uint32_t rh = 0, rt = 0;  // warp-uniform ring head (drained) and tail (staged)
#pragma unroll 1
    for (int it = 0; it < n_it; ++it) {
      uint4 nxt[kWideU];
#pragma unroll
      for (int u = 0; u < kWideU; ++u) {
        const int m = (it + 1) * kPerIter + u * kWideThreads + t;
        nxt[u] = m < nq ? ld_stream_v4(body + 16 * static_cast<size_t>(m), pol)
                        : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kWideU; ++u) {
        const int m = it * kPerIter + u * kWideThreads + t;
        const uint32_t wd[4] = {cur[u].x, cur[u].y, cur[u].z, cur[u].w};
        uint32_t mk[4] = {0u, 0u, 0u, 0u};
        if (m < nq) {
#pragma unroll
          for (int x = 0; x < 4; ++x) mk[x] = hgeu_mask(wd[x], t2);
        }
        if (!__any_sync(0xFFFFFFFFu, (mk[0] | mk[1] | mk[2] | mk[3]) != 0u)) continue;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const bool f = mk[x] != 0u;
          const uint32_t bal = __ballot_sync(0xFFFFFFFFu, f);
          if (f)
            ring[(rt + __popc(bal & lt)) & (kWideRing - 1)] =
                make_uint2(wd[x], static_cast<uint32_t>(head + 8 * m + 2 * x));
          rt += __popc(bal);
          if (rt - rh >= 32u) {
            __syncwarp();
            wide_drain(ring, rh, 32u, t_key, cand, kCap, lh, pg, &misc[kWN], bad, range, kmax);
            rh += 32u;
            __syncwarp();
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kWideU; ++u) cur[u] = nxt[u];
    }
    __syncwarp();
    if (rt != rh)
      wide_drain(ring, rh, rt - rh, t_key, cand, kCap, lh, pg, &misc[kWN], bad, range, kmax);
    if (t < head + tail) {
      const int idx = t < head ? t : head + 8 * nq + (t - head);
      wide_append_one(sp, idx, t_key, cand, kCap, lh, pg, &misc[kWN], bad, range, kmax);
    }
    if (bad) atomicOr(&misc[kWBad], 1u);
    if (range) atomicOr(&misc[kWRange], 1u);
  }
  kmax = wide_max_u32(kmax, scratch);
  if (t == 0) misc[kWMaxK] = kmax;
  if constexpr (G > 1)
    wide_cluster_sync();
  else
    __syncthreads();

  // ---- check: counts and flags of every CTA ----
  if (t < 32) {
    uint32_t n = 0, b = 0, rg = 0;
    if (lane < static_cast<uint32_t>(G)) {
      if constexpr (G == 1) {
        n = misc[kWN];
        b = misc[kWBad];
        rg = misc[kWRange];
      } else {
        n = dsmem_ld_u32(dsmem_addr(&misc[kWN], lane));
        b = dsmem_ld_u32(dsmem_addr(&misc[kWBad], lane));
        rg = dsmem_ld_u32(dsmem_addr(&misc[kWRange], lane));
      }
    }
    uint32_t incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= static_cast<uint32_t>(o)) incl += x;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const bool any_bad = __any_sync(0xFFFFFFFFu, b != 0);
    const bool any_range = __any_sync(0xFFFFFFFFu, rg != 0);
    const bool any_full = __any_sync(0xFFFFFFFFu, n > kCap);
    if (t == 0) {
      uint32_t mode = 0u;
      if (!p.wide_exact) {
        if (any_bad)
          mode = 2u;
        else if (total >= k_eff && total <= 65535u && !any_full && !any_range)
          mode = 1u;
        else if (total >= k_eff && !any_full)
          mode = 3u;  // key range too wide for the per-key counts
      }
      misc[kWFast] = mode;
    }
  }
  __syncthreads();
  const uint32_t mode = misc[kWFast];
  if (mode == 2u) {
    if constexpr (G > 1) wide_cluster_sync();  // peers may still read our counters
    if (rank == 0 && t == 0) finish_row(p, r, w, -1, kRowNonFinite);
    return;
  }
  if (mode == 1u) {
    wide_fast_tail<G>(p, r, w, rank, S, t_key, cand, static_cast<int>(misc[kWN]), lh, mh, misc,
                      scratch);
    if constexpr (G > 1) wide_cluster_sync();  // peers read our counts and the leader's counter
    return;
  }
  uint32_t *hw = reinterpret_cast<uint32_t *>(work);
  if (mode == 0u) {
    // the exact top-k set collected anew by re-reading the slice
    if constexpr (G > 1) wide_cluster_sync();  // peers may still read our counters
    const bool ok = wide_exact_collect<G>(sp, head, nq, tail, rank, k_eff, cand, hw, pg, misc,
                                          scratch);
    if (!ok) {
      if (rank == 0 && t == 0) finish_row(p, r, w, -1, kRowNonFinite);
      return;
    }
  }
  if (mode == 0u) wide_sync_all<G>();  // the exact set's page counts are complete everywhere
  wide_dist_tail<G>(p, r, w, rank, S, cand, static_cast<int>(min(misc[kWN], kCap)), hw, pg, misc,
                    scratch);
  if constexpr (G > 1) wide_cluster_sync();  // peers read our histograms and the leader's counter
}

}  // namespace ts
