// ts_split.cuh -- the wide-row sampler as three kernels over a workspace
// (bf16 rows such as the 151,936-token backbone vocabulary, any top-k cap up
// to 4096: Drama 3 article, section "能跑通的命令，和文档写明的边界").
//
// Kernel A (one CTA per row) reads an evenly spaced sample of the row (64
// runs of 64 logits) and stores the threshold key t (the sampling step of
// Floyd and Rivest's selection, "Expected time bounds for selection", CACM
// 18(3), 1975); it also clears the row's candidate counter.
//
// Kernel B (U CTAs per row, one contiguous slice each) streams its slice
// once with 16-byte loads and keeps every logit that compares >= t or is a
// NaN, as raw entries (bf16 bits << 16 | slice index): each warp compacts
// the flags of four chunks per lane at once, and the CTA appends its entries
// to the row's candidate array with one atomic on the row's counter.  It
// does nothing else, so the streaming CTAs never wait for one another or
// hold an SM for a row's tail.
//
// For launches of few CTAs, kernel A is skipped and every CTA of kernel B
// takes the same sample itself (the threshold kernel's launch would cost
// more than the duplicated sample).  Kernel C clears each row's counter
// after use, so the counters are zero at the start of every call either way.
//
// Kernel C (one CTA per row) copies the row's candidate array (a few
// thousand entries, from L2) into shared memory in the same round of loads
// as the units' records, and runs the row's tail:
//   - keys, page counts, the maximum and the NaN / +inf check of the
//     candidates; the threshold key's page from the page counts and the
//     candidates counted per key;
//   - the keys that occur, compacted in key order, so that one block scan
//     over them gives the threshold key thr (the k_eff-th largest) and
//     `need`, the kept tokens tied at it, and one more the kept masses (2^-40
//     fixed point, depending only on the key), the nucleus cutoff and the
//     draw;
//   - the drawn token: the rho-th lowest token index among the candidates
//     that share the drawn key.
// If the sample misled t (fewer than k_eff candidates, or more than the
// buffers hold) kernel C re-reads the row and selects exactly.  Candidates
// spread over too many keys take a coarse-bin tail instead.
#pragma once

#include "ts_wide.cuh"

namespace ts {

constexpr int kSplitThreads = 256;
constexpr int kSplitUnitCap = 4096;     // candidates one CTA may hand over
constexpr int kSplitRowCap = 8192;      // candidates the tail CTA gathers
constexpr int kSplitMaxUnits = 16;
constexpr int kSplitU = 4;              // 16-byte chunks per lane per iteration
constexpr int kSplitKeyPages = 32;       // per-key counts for up to 32 pages of 256 keys
constexpr int kSplitListCap = 1024;      // distinct candidate keys the compact tail takes
constexpr int kSplitSampleRun = 8;       // kernel A samples 128-byte runs of the row
static_assert(kSplitThreads == kWideThreads, "the block scans assume 8 warps");

// Kernel B's dynamic shared memory: the unit's candidates, each thread's
// last four chunks (for the element lookups of the compaction) and
// bookkeeping (33 KB).
constexpr uint32_t kStreamCandOff = 0;
constexpr uint32_t kStreamStageOff = kSplitUnitCap * 4;
constexpr uint32_t kStreamMiscOff = kStreamStageOff + kSplitU * kSplitThreads * 16;
constexpr uint32_t kStreamSmemBytes = kStreamMiscOff + kWideMiscWords * 4;

// Kernel C's: the gathered candidates (32 KB), a 16 KB work area (per-key
// counts, then the coarse-bin tail, the exact path's histogram or the rank
// lists), the compacted key list, page counts, page <-> slot maps, unit
// segments and their units, and bookkeeping (55.4 KB: four CTAs per SM).
constexpr uint32_t kTailCandOff = 0;
constexpr uint32_t kTailHwOff = kSplitRowCap * 4;
constexpr uint32_t kTailListOff = kTailHwOff + 16384;
constexpr uint32_t kTailPgOff = kTailListOff + kSplitListCap * 4;
constexpr uint32_t kTailPageSlotOff = kTailPgOff + 1024;
constexpr uint32_t kTailSlotPageOff = kTailPageSlotOff + 1024;
constexpr uint32_t kTailSegOff = kTailSlotPageOff + kSplitKeyPages * 4;
constexpr uint32_t kTailMiscOff = kTailSegOff + 256;
constexpr uint32_t kTailSmemBytes = kTailMiscOff + kWideMiscWords * 4;

// Workspace layout (every region 16-byte aligned).
struct SplitRowMeta {
  uint32_t t_key;
  uint32_t count;  // candidate entries appended so far (cleared by kernel A)
  uint32_t pad[2];
};
struct SplitUnitMeta {
  uint32_t n;     // entries the unit kept (may exceed kSplitUnitCap)
  uint32_t base;  // where its run starts in the row's candidate array
  uint32_t pad[2];
};

// Row records for max_rows rows, unit records for max_units units (a
// launch's CTAs: unit r * U + u is slice u of row r), then each row's
// candidate array of kSplitRowCap entries.
__host__ __device__ constexpr size_t split_workspace_bytes(int max_rows, int max_units) {
  const size_t rows = static_cast<size_t>(max_rows), units = static_cast<size_t>(max_units);
  return rows * sizeof(SplitRowMeta) + units * sizeof(SplitUnitMeta) + rows * kSplitRowCap * 4;
}

struct SplitWs {
  SplitRowMeta *row;
  SplitUnitMeta *unit;
  uint32_t *cand;  // [row][kSplitRowCap]
};

__device__ __forceinline__ SplitWs split_ws(void *base, int max_rows, int max_units) {
  SplitWs ws;
  char *b = static_cast<char *>(base);
  const size_t rows = static_cast<size_t>(max_rows), units = static_cast<size_t>(max_units);
  ws.row = reinterpret_cast<SplitRowMeta *>(b);
  b += rows * sizeof(SplitRowMeta);
  ws.unit = reinterpret_cast<SplitUnitMeta *>(b);
  b += units * sizeof(SplitUnitMeta);
  ws.cand = reinterpret_cast<uint32_t *>(b);
  return ws;
}

// ---------------------------------------------------------------------------
// Kernel A: the row's threshold key from its sample; clears its counter.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSplitThreads) split_threshold_kernel(const Params p) {
  __shared__ __align__(16) uint32_t hist[2048];
  __shared__ __align__(16) uint32_t misc[kWideMiscWords];
  const int r = static_cast<int>(blockIdx.x);
  const int t = static_cast<int>(threadIdx.x);
  pdl_wait_and_release();
  if (r >= p.n_rows) return;
  SplitWs ws = split_ws(p.workspace, p.ws_rows, p.ws_units);
  const Row w = load_row(p, r);
  uint32_t t_key = 0;
  if (!w.err && !w.fin && !p.wide_exact) {
    const char *rowp = static_cast<const char *>(p.logits) + w.off * 2;
    // a row the tail CTA can gather whole, in slices each CTA can hold,
    // keeps every logit (t = lowest key); others sample
    if (w.vocab > kSplitRowCap || p.slice > kSplitUnitCap)
      t_key = wide_sample_threshold<kSplitSampleRun>(rowp, w.vocab, w.k_eff, 1, hist, misc,
                                                     reinterpret_cast<uint64_t *>(misc + kWScan));
  }
  if (t == 0) {
    ws.row[r].t_key = t_key;
    ws.row[r].count = 0u;
  }
}

// Candidate entries are grouped in segments, one per unit: segment k is
// entries seg[k] .. seg[k + 1] - 1 and came from unit seg[kSplitUmapOff + k]
// (their low 16 bits index that unit's slice).
constexpr int kSplitUmapOff = kSplitMaxUnits + 1;

// The segment holding entry i, for nondecreasing seg[0 .. U] with seg[0] = 0
// <= i < seg[U] and U <= 16: a binary search of four fixed steps (no
// data-dependent loop, so the lanes of a warp stay converged).
__device__ __forceinline__ int split_unit_of(const uint32_t *seg, int U, uint32_t i) {
  int c = 0;
#pragma unroll
  for (int step = 8; step >= 1; step >>= 1)
    if (c + step < U && i >= seg[c + step]) c += step;
  return c;
}

// The token index of entry e, the i-th candidate.
__device__ __forceinline__ uint32_t split_gidx(const uint32_t *seg, int U, int S, uint32_t i,
                                               uint32_t e) {
  return seg[kSplitUmapOff + split_unit_of(seg, U, i)] * static_cast<uint32_t>(S) + (e & 0xFFFFu);
}

// The rho-th smallest (0-based) token index among the gathered candidates
// with key `key_sel`; segment c of the array came from unit c, whose slice
// starts at token c * S.  Two-level radix select on the 18-bit index.
__device__ uint32_t split_rank_select(const uint32_t *cand, int n, const uint32_t *seg, int U,
                                      int S, uint32_t key_sel, uint32_t rho, uint32_t *h,
                                      uint32_t *misc, uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  uint32_t b1 = 0, below = 0;
#pragma unroll 1
  for (int level = 0; level < 2; ++level) {
    __syncthreads();
    h[2 * t] = 0u;
    h[2 * t + 1] = 0u;
    __syncthreads();
#pragma unroll 4
    for (int base = 0; base < n; base += kSplitThreads) {
      const int i = base + t;
      const uint32_t e = i < n ? cand[i] : 0u;
      if (i < n && (e >> 16) == key_sel) {
        const uint32_t g = split_gidx(seg, U, S, static_cast<uint32_t>(i), e);
        if (level == 0)
          atomicAdd(&h[g >> 9], 1u);
        else if ((g >> 9) == b1)
          atomicAdd(&h[g & 511u], 1u);
      }
    }
    __syncthreads();
    const uint32_t want = rho - below;
    const uint32_t h0 = h[2 * t], h1 = h[2 * t + 1];
    uint64_t tot;
    const uint32_t ex = static_cast<uint32_t>(wide_excl_scan_u64(h0 + h1, scratch, &tot));
    if (ex <= want && want < ex + h0) {
      misc[kWDigit] = 2 * t;
      misc[kWAbove] = ex;
    } else if (ex + h0 <= want && want < ex + h0 + h1) {
      misc[kWDigit] = 2 * t + 1;
      misc[kWAbove] = ex + h0;
    }
    __syncthreads();
    if (level == 0) {
      b1 = misc[kWDigit];
      below += misc[kWAbove];
    } else {
      return (b1 << 9) | misc[kWDigit];
    }
  }
  return 0;
}

// The row's tail over the gathered candidates (any key range): see the file
// comment.  pgc[256] holds the candidate counts by key >> 8, maxk the largest
// candidate key.
__device__ void split_row_tail(const Params &p, int r, const Row &w, const uint32_t *cand, int n,
                               const uint32_t *seg, int U, int S, const uint32_t *pgc,
                               uint32_t maxk, uint32_t *hw, uint32_t *misc, uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t k_eff = static_cast<uint32_t>(w.k_eff);
  uint64_t *m64 = reinterpret_cast<uint64_t *>(misc);
  uint32_t *bB = hw;  // low key bytes inside the threshold's page
  uint32_t *plo = hw + 256, *pmid = hw + 512, *phi = hw + 768, *pcnt = hw + 1024;
  uint32_t *lD = hw + 1280, *lE = hw + 1536;  // second levels of the cutoff's / draw's bin
  uint32_t *rs = hw + 1024;                   // rank select (after the coarse counts)
  if (maxk <= KeyBF16::kNegInf) {  // every candidate is -inf: no finite logit in the row
    if (t == 0) finish_row(p, r, w, -1, kRowNonFinite);
    return;
  }
  // ---- the threshold key: its page, then its low byte ----
  bB[t] = 0u;
  wide_select256(pgc[t], k_eff, misc, scratch);
  const uint32_t page = misc[kWDigit];
  const uint32_t kk = k_eff - misc[kWAbove];
#pragma unroll 4
  for (int i = t; i < n; i += kSplitThreads) {
    const uint32_t key = cand[i] >> 16;
    if ((key >> 8) == page) atomicAdd(&bB[key & 255u], 1u);
  }
  __syncthreads();
  wide_select256(bB[t], kk, misc, scratch);
  const uint32_t thr = (page << 8) | misc[kWDigit];
  const uint32_t need = kk - misc[kWAbove];
  const float m = KeyBF16::value(maxk);
  const uint32_t u24 = misc[kWU24];
  uint32_t key_d = maxk, rho = 0, n_p = 1;
  uint64_t s_k = 0;
  if (!w.greedy) {
    // ---- coarse kept masses and counts over (maxk - key) >> shift ----
    const uint32_t range = maxk - thr;
    const int bits = range ? 32 - __clz(range) : 0;
    const int shift = bits > 8 ? bits - 8 : 0;
    plo[t] = 0u;
    pmid[t] = 0u;
    phi[t] = 0u;
    pcnt[t] = 0u;
    __syncthreads();
#pragma unroll 4
    for (int i = t; i < n; i += kSplitThreads) {
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
    __syncthreads();
    const uint32_t dthr = (maxk - thr) >> shift;
    uint32_t cs = pcnt[t] + (static_cast<uint32_t>(t) == dthr ? need : 0u);
    uint64_t ms;
    if (shift == 0) {
      ms = cs ? cs * to_fixed(kept_weight(KeyBF16::value(maxk - t), m, w.temp, w.inv_temp)) : 0ull;
    } else {
      ms = (static_cast<uint64_t>(phi[t]) << 26) + (static_cast<uint64_t>(pmid[t]) << 13) + plo[t];
      if (static_cast<uint32_t>(t) == dthr && need)
        ms += need * to_fixed(kept_weight(KeyBF16::value(thr), m, w.temp, w.inv_temp));
    }
    const uint64_t cum_t = wide_excl_scan_u64(ms, scratch, &s_k);
    uint64_t n_all64;
    const uint32_t ccum_t = static_cast<uint32_t>(wide_excl_scan_u64(cs, scratch, &n_all64));
    // ---- nucleus cutoff ----
    uint64_t s_p;
    uint32_t c1 = 0xFFFFFFFFu;
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
      c1 = misc[kWThrB];
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
        __syncthreads();
        wide_merge_level2<1>(lD, maxk, thr, need, shift, c1, m, w.temp, w.inv_temp, true, cut,
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
    const uint32_t d1 = misc[kWDrawB];
    uint64_t above_d = m64[kWWide / 2];
    if (shift == 0) {
      key_d = maxk - d1;
    } else {
      // the cutoff's second level serves the draw too when both fall in one bin
      uint32_t *l2 = lD;
      if (d1 != c1) {
        wide_local_level2(cand, n, maxk, thr, shift, d1, lE);
        __syncthreads();
        l2 = lE;
      }
      wide_merge_level2<1>(l2, maxk, thr, need, shift, d1, m, w.temp, w.inv_temp, false, target,
                           above_d, misc, scratch);
      key_d = misc[kWDigit];
      above_d = m64[kWSp / 2];
    }
    const uint64_t wd = to_fixed(kept_weight(KeyBF16::value(key_d), m, w.temp, w.inv_temp));
    rho = wd > 0 ? static_cast<uint32_t>((target - above_d) / wd) : 0u;
  }
  const uint32_t id = split_rank_select(cand, n, seg, U, S, key_d, rho, rs, misc, scratch);
  if (t == 0) finish_row(p, r, w, static_cast<int32_t>(id), 0u);
  if (p.kept_ids) {
    // keys above thr, and the `need` lowest-index keys at thr
    const uint32_t idx_cut =
        need ? split_rank_select(cand, n, seg, U, S, thr, need - 1, rs, misc, scratch) : 0u;
    if (t == 0) misc[kWKept] = 0u;
    __syncthreads();
    const float s_real = static_cast<float>(static_cast<double>(s_k) * (1.0 / 1099511627776.0));
    const int64_t rb = static_cast<int64_t>(r) * p.max_keep;
    for (int i = t; i < n; i += kSplitThreads) {
      const uint32_t e = cand[i];
      const uint32_t key = e >> 16;
      const uint32_t g = split_gidx(seg, U, S, static_cast<uint32_t>(i), e);
      if (key > thr || (key == thr && need && g <= idx_cut)) {
        const uint32_t pos = atomicAdd(&misc[kWKept], 1u);
        if (pos < static_cast<uint32_t>(p.max_keep)) {
          p.kept_ids[rb + pos] = static_cast<int32_t>(g);
          p.kept_probs[rb + pos] =
              w.greedy ? (g == id ? 1.f : 0.f)
                       : __fdiv_rn(kept_weight(KeyBF16::value(key), m, w.temp, w.inv_temp), s_real);
        }
      }
    }
    if (t == 0) {
      p.n_kept[r] = static_cast<int32_t>(k_eff);
      p.n_nucleus[r] = static_cast<int32_t>(n_p);
    }
  }
}

// The threshold key's page (the page holding the k_eff-th largest candidate,
// from the counts by key >> 8) and a slot of 256 packed 16-bit per-key counts
// for each occupied page at or above it, cleared.  Returns the number of
// such pages; above kSplitKeyPages nothing is cleared and the caller takes
// the coarse-bin tail.  misc[kWDigit] = the page.
__device__ int split_key_setup(const uint32_t *pgc, uint32_t k_eff, uint32_t *kc,
                               uint32_t *page_slot, uint32_t *slot_page, uint32_t *misc,
                               uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t c = pgc[t];
  wide_select256(c, k_eff, misc, scratch);
  const uint32_t page = misc[kWDigit];
  const bool occ = static_cast<uint32_t>(t) >= page && c != 0u;
  uint64_t n_occ;
  const uint32_t slot = static_cast<uint32_t>(wide_excl_scan_u64(occ ? 1u : 0u, scratch, &n_occ));
  const int up = static_cast<int>(n_occ);
  if (up > kSplitKeyPages) return up;
  page_slot[t] = occ ? slot : 0u;
  if (occ) slot_page[slot] = static_cast<uint32_t>(t);
  for (int i = t; i < up * 128; i += kSplitThreads) kc[i] = 0u;
  __syncthreads();
  return up;
}

// Counts one candidate key (at or above the threshold's page) in its slot.
__device__ __forceinline__ void split_key_count(uint32_t key, uint32_t page,
                                                const uint32_t *page_slot, uint32_t *kc) {
  if ((key >> 8) >= page)
    atomicAdd(&kc[page_slot[key >> 8] * 128u + ((key & 255u) >> 1)], 1u << ((key & 1u) * 16u));
}

// Exclusive block scans of two values at once (one pass of barriers).
__device__ __forceinline__ void split_excl_scan2(uint64_t a, uint32_t b, uint64_t *scratch,
                                                 uint64_t *ex_a, uint64_t *tot_a, uint32_t *ex_b,
                                                 uint32_t *tot_b) {
  const uint32_t lane = lane_id(), wid = threadIdx.x >> 5;
  uint64_t x = a;
  uint32_t y = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t tx = __shfl_up_sync(0xFFFFFFFFu, x, o);
    const uint32_t ty = __shfl_up_sync(0xFFFFFFFFu, y, o);
    if (lane >= static_cast<uint32_t>(o)) {
      x += tx;
      y += ty;
    }
  }
  __syncthreads();  // scratch may still be read by a previous scan
  if (lane == 31) {
    scratch[wid] = x;
    scratch[16 + wid] = y;
  }
  __syncthreads();
  if (wid == 0) {
    const uint64_t sa = lane < kWideWarps ? scratch[lane] : 0ull;
    const uint64_t sb = lane < kWideWarps ? scratch[16 + lane] : 0ull;
    uint64_t ia = sa, ib = sb;
#pragma unroll
    for (int o = 1; o < kWideWarps; o <<= 1) {
      const uint64_t ta = __shfl_up_sync(0xFFFFFFFFu, ia, o);
      const uint64_t tb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
      if (lane >= static_cast<uint32_t>(o)) {
        ia += ta;
        ib += tb;
      }
    }
    if (lane < kWideWarps) {
      scratch[lane] = ia - sa;
      scratch[16 + lane] = ib - sb;
    }
    if (lane == kWideWarps - 1) {
      scratch[kWideWarps] = ia;
      scratch[16 + kWideWarps] = ib;
    }
  }
  __syncthreads();
  *ex_a = scratch[wid] + x - a;
  *tot_a = scratch[kWideWarps];
  *ex_b = static_cast<uint32_t>(scratch[16 + wid]) + y - b;
  *tot_b = static_cast<uint32_t>(scratch[16 + kWideWarps]);
}

// The rho-th smallest token index among the n_key candidates with key `key`
// (n_key <= kSplitThreads): the indices are collected, and the one with
// exactly rho smaller ones is it.  rl: n_key words of scratch.
__device__ uint32_t split_small_rank(const uint32_t *cand, int n, const uint32_t *seg, int U,
                                     int S, uint32_t key, uint32_t n_key, uint32_t rho,
                                     uint32_t *rl, uint32_t *misc) {
  const int t = static_cast<int>(threadIdx.x);
  if (t == 0) misc[kWN] = 0u;
  __syncthreads();
#pragma unroll 4
  for (int base = 0; base < n; base += kSplitThreads) {
    const int i = base + t;
    const uint32_t e = i < n ? cand[i] : 0u;
    if (i < n && (e >> 16) == key) {
      const uint32_t pos = atomicAdd(&misc[kWN], 1u);
      if (pos < n_key)
        rl[pos] = split_gidx(seg, U, S, static_cast<uint32_t>(i), e);
    }
  }
  __syncthreads();
  if (static_cast<uint32_t>(t) < n_key) {
    const uint32_t g = rl[t];
    uint32_t below = 0;
    for (uint32_t j = 0; j < n_key; ++j) below += rl[j] < g ? 1u : 0u;
    if (below == rho) misc[kWSelIdx] = g;
  }
  __syncthreads();
  return misc[kWSelIdx];
}

// The row's tail from the per-key counts of split_key_setup: the occupied
// keys are compacted in key order (one entry, key << 16 | count, per key
// that occurs), and each thread takes up to four consecutive entries in
// descending key order, so that block scans over the entries give the
// threshold key and `need`, S_k, the nucleus cutoff and the draw, with one
// weight evaluation per key.  Returns false (nothing written) when more than
// kSplitListCap keys occur; the caller then runs split_row_tail.
__device__ bool split_key_tail(const Params &p, int r, const Row &w, const uint32_t *cand, int n,
                               const uint32_t *seg, int U, int S, uint32_t maxk, int up,
                               uint32_t u24, uint32_t *kc, uint32_t *list,
                               const uint32_t *slot_page, uint32_t *misc, uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t k_eff = static_cast<uint32_t>(w.k_eff);
  uint64_t *m64 = reinterpret_cast<uint64_t *>(misc);
  auto bin_cnt = [&](int b) { return (kc[b >> 1] >> ((b & 1) * 16)) & 0xFFFFu; };
  // ---- the keys that occur, in ascending order (thread t owns bins
  // [t * up, t * up + up), bin b = slot b >> 8, low byte b & 255) ----
  const int b0 = t * up;
  uint32_t occ = 0;
#pragma unroll 8
  for (int j = 0; j < up; ++j) occ += bin_cnt(b0 + j) != 0u ? 1u : 0u;
  uint64_t n_list;
  uint32_t pos = static_cast<uint32_t>(wide_excl_scan_u64(occ, scratch, &n_list));
  const int L = static_cast<int>(n_list);
  if (L > kSplitListCap) return false;
#pragma unroll 8
  for (int j = 0; j < up; ++j) {
    const int b = b0 + j;
    const uint32_t c = bin_cnt(b);
    if (c) list[pos++] = (((slot_page[b >> 8] << 8) | static_cast<uint32_t>(b & 255)) << 16) | c;
  }
  __syncthreads();
  // ---- entries j0 .. j0 + E - 1 in descending key order ----
  const int E = (L + kSplitThreads - 1) / kSplitThreads;  // <= 4
  const int j0 = t * E;
  uint32_t ek[4], ec[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = j0 + q;
    const uint32_t e = q < E && j < L ? list[L - 1 - j] : 0u;
    ek[q] = e >> 16;
    ec[q] = e & 0xFFFFu;
  }
  // ---- threshold key (k_eff-th largest) and `need` ----
  const uint32_t s = ec[0] + ec[1] + ec[2] + ec[3];
  uint64_t tot;
  const uint32_t above = static_cast<uint32_t>(wide_excl_scan_u64(s, scratch, &tot));
  if (s != 0 && above < k_eff && above + s >= k_eff) {
    uint32_t run = above;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (ec[q] && run < k_eff && run + ec[q] >= k_eff) {
        misc[kWTKey] = ek[q];
        misc[kWTake] = k_eff - run;
      }
      run += ec[q];
    }
  }
  __syncthreads();
  const uint32_t thr = misc[kWTKey];
  const uint32_t need = misc[kWTake];
  const float m = KeyBF16::value(maxk);
  uint32_t key_d = maxk, rho = 0, n_p = 1;
  uint32_t c_d = list[L - 1] & 0xFFFFu;  // candidates with the largest key
  uint64_t s_k = 0;
  if (!w.greedy) {
    uint32_t kq[4];
    uint64_t wq[4];
    uint64_t st = 0;
    uint32_t ct = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      kq[q] = ec[q] == 0u ? 0u : ek[q] > thr ? ec[q] : ek[q] == thr ? need : 0u;
      wq[q] = kq[q] ? to_fixed(kept_weight(KeyBF16::value(ek[q]), m, w.temp, w.inv_temp)) : 0ull;
      st += kq[q] * wq[q];
      ct += kq[q];
    }
    uint64_t ex_m;
    uint32_t ex_c, n_kept;
    split_excl_scan2(st, ct, scratch, &ex_m, &s_k, &ex_c, &n_kept);
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
      if (st != 0 && ex_m < cut && ex_m + st >= cut) {
        uint64_t cum = ex_m;
        uint32_t ccum = ex_c;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint64_t mb = kq[q] * wq[q];
          if (mb && cum < cut && cum + mb >= cut) {
            uint64_t n_c = (cut - cum + wq[q] - 1) / wq[q];
            if (n_c < 1) n_c = 1;
            m64[kWSp / 2] = cum + n_c * wq[q];
            misc[kWNp] = ccum + static_cast<uint32_t>(n_c);
          }
          cum += mb;
          ccum += kq[q];
        }
      }
      __syncthreads();
      s_p = m64[kWSp / 2];
      n_p = misc[kWNp];
    }
    // ---- draw ----
    const uint64_t target = scale_u24(u24, s_p);
    if (st != 0 && ex_m <= target && target < ex_m + st) {
      uint64_t cum = ex_m;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint64_t mb = kq[q] * wq[q];
        if (mb && cum <= target && target < cum + mb) {
          misc[kWDrawB] = ek[q];
          misc[kWRho] = static_cast<uint32_t>((target - cum) / wq[q]);
          misc[kWCount] = ec[q];
        }
        cum += mb;
      }
    }
    __syncthreads();
    key_d = misc[kWDrawB];
    rho = misc[kWRho];
    c_d = misc[kWCount];
  }
  // ---- the drawn token (kc is free once the list is built) ----
  const uint32_t id = c_d <= static_cast<uint32_t>(kSplitThreads)
                          ? split_small_rank(cand, n, seg, U, S, key_d, c_d, rho, kc, misc)
                          : split_rank_select(cand, n, seg, U, S, key_d, rho, kc, misc, scratch);
  if (t == 0) finish_row(p, r, w, static_cast<int32_t>(id), 0u);
  if (p.kept_ids) {
    // keys above thr, and the `need` lowest-index keys at thr
    const uint32_t idx_cut =
        need ? split_rank_select(cand, n, seg, U, S, thr, need - 1, kc, misc, scratch) : 0u;
    if (t == 0) misc[kWKept] = 0u;
    __syncthreads();
    const float s_real = static_cast<float>(static_cast<double>(s_k) * (1.0 / 1099511627776.0));
    const int64_t rb = static_cast<int64_t>(r) * p.max_keep;
    for (int i = t; i < n; i += kSplitThreads) {
      const uint32_t e = cand[i];
      const uint32_t key = e >> 16;
      const uint32_t g = split_gidx(seg, U, S, static_cast<uint32_t>(i), e);
      if (key > thr || (key == thr && need && g <= idx_cut)) {
        const uint32_t at = atomicAdd(&misc[kWKept], 1u);
        if (at < static_cast<uint32_t>(p.max_keep)) {
          p.kept_ids[rb + at] = static_cast<int32_t>(g);
          p.kept_probs[rb + at] =
              w.greedy ? (g == id ? 1.f : 0.f)
                       : __fdiv_rn(kept_weight(KeyBF16::value(key), m, w.temp, w.inv_temp), s_real);
        }
      }
    }
    if (t == 0) {
      p.n_kept[r] = static_cast<int32_t>(k_eff);
      p.n_nucleus[r] = static_cast<int32_t>(n_p);
    }
  }
  return true;
}

// Exact fallback of kernel C: the whole row read again, the k_eff-th
// largest key by radix select (11 + 5 bits), and the exact top-k set
// collected in token order, ties at the threshold by lowest index, as
// (key << 16 | slice index) entries grouped by unit (unit c's entries are
// cand[seg[c] .. seg[c + 1])).  Returns false for a row with a NaN / +inf
// or without a finite logit.  Also fills pgc (counts by key >> 8) and
// *maxk for the tail.
__device__ bool split_exact(const char *rowp, int V, int U, int S, uint32_t k_eff, uint32_t *cand,
                            uint32_t *seg, uint32_t *pgc, uint32_t *maxk_out, uint32_t *hist,
                            uint32_t *misc, uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  if (t < kSplitMaxUnits) seg[kSplitUmapOff + t] = static_cast<uint32_t>(t);  // units in order
  const int head = min(V, static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(rowp) & 15u)) & 15u) / 2u));
  const int nq = (V - head) / 8;
  const int tail = V - head - 8 * nq;
  const char *body = rowp + 2 * head;
  auto key_at = [&](int idx) { return KeyBF16::key(KeyBF16::load_one(rowp, idx)); };
  // pass 1: 11-bit histogram, NaN / +inf and finite counts
  for (int i = t; i < 2048; i += kSplitThreads) hist[i] = 0u;
  if (t < 32) misc[kWHist2 + t] = 0u;
  if (t == 0) {
    misc[kWBad] = 0u;
    misc[kWFin] = 0u;
  }
  __syncthreads();
  uint32_t nbad = 0, nfin = 0;
  auto count1 = [&](uint32_t k) {
    nbad += (k < KeyBF16::kNegInf) | (k >= KeyBF16::kPosInf);
    nfin += k > KeyBF16::kNegInf;
    atomicAdd(&hist[k >> 5], 1u);
  };
  for (int q = t; q < nq; q += kSplitThreads) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(body + 16 * static_cast<size_t>(q)));
    const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const uint32_t kw = KeyBF16::key_word(wds[x]);
      count1(kw & 0xFFFFu);
      count1(kw >> 16);
    }
  }
  if (t < head + tail) count1(key_at(t < head ? t : head + 8 * nq + (t - head)));
  nbad = __reduce_add_sync(0xFFFFFFFFu, nbad);
  nfin = __reduce_add_sync(0xFFFFFFFFu, nfin);
  if (lane_id() == 0) {
    if (nbad) atomicAdd(&misc[kWBad], nbad);
    if (nfin) atomicAdd(&misc[kWFin], nfin);
  }
  __syncthreads();
  if (misc[kWBad] != 0u || misc[kWFin] == 0u) return false;
  wide_select_top<8, 1>(hist, k_eff, misc, scratch);
  const uint32_t b1 = misc[kWDigit];
  const uint32_t kk = k_eff - misc[kWAbove];
  // pass 2: the low 5 key bits inside bin b1
  for (int q = t; q < nq; q += kSplitThreads) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(body + 16 * static_cast<size_t>(q)));
    const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const uint32_t kw = KeyBF16::key_word(wds[x]);
      const uint32_t a = kw & 0xFFFFu, b = kw >> 16;
      if ((a >> 5) == b1) atomicAdd(&misc[kWHist2 + (a & 31u)], 1u);
      if ((b >> 5) == b1) atomicAdd(&misc[kWHist2 + (b & 31u)], 1u);
    }
  }
  if (t < head + tail) {
    const uint32_t k = key_at(t < head ? t : head + 8 * nq + (t - head));
    if ((k >> 5) == b1) atomicAdd(&misc[kWHist2 + (k & 31u)], 1u);
  }
  __syncthreads();
  if (t < 32) {
    const uint32_t c = misc[kWHist2 + t];
    uint32_t suf = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_down_sync(0xFFFFFFFFu, suf, o);
      if (t + o < 32) suf += x;
    }
    const uint32_t d2 = 31u - __clz(__ballot_sync(0xFFFFFFFFu, suf >= kk));
    const uint32_t above2 = __shfl_sync(0xFFFFFFFFu, suf - c, d2);
    if (t == 0) {
      misc[kWTKey] = (b1 << 5) | d2;
      misc[kWTake] = kk - above2;
    }
  }
  pgc[t] = 0u;
  __syncthreads();
  const uint32_t thr = misc[kWTKey];
  const uint32_t take = misc[kWTake];  // keys equal to thr that are kept (lowest indices)
  // pass 3: collect in token order, unit by unit, in rounds of 8 consecutive
  // tokens per thread; keys at thr are ranked by an exclusive scan
  uint32_t n = 0, eq_seen = 0, kmax = 0;
  for (int c = 0; c < U; ++c) {
    if (t == 0) seg[c] = n;
    const int lo = c * S, hi = min(V, lo + S);
    for (int base = lo; base < hi; base += 8 * kSplitThreads) {
      const int i0 = base + 8 * t;
      uint32_t k[8];
      uint32_t ne = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        k[e] = i0 + e < hi ? key_at(i0 + e) : 0u;
        ne += i0 + e < hi && k[e] == thr;
      }
      uint64_t tot_eq;
      uint32_t er = eq_seen + static_cast<uint32_t>(wide_excl_scan_u64(ne, scratch, &tot_eq));
      uint32_t keepm = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (i0 + e >= hi) continue;
        bool keep = k[e] > thr;
        if (k[e] == thr) keep = er++ < take;
        keepm |= (keep ? 1u : 0u) << e;
      }
      uint64_t tot_keep;
      uint32_t at = n + static_cast<uint32_t>(wide_excl_scan_u64(__popc(keepm), scratch, &tot_keep));
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (!(keepm & (1u << e))) continue;
        if (at < static_cast<uint32_t>(kSplitRowCap)) {
          cand[at] = (k[e] << 16) | static_cast<uint32_t>(i0 + e - lo);
          atomicAdd(&pgc[k[e] >> 8], 1u);
          kmax = max(kmax, k[e]);
        }
        ++at;
      }
      n += static_cast<uint32_t>(tot_keep);
      eq_seen += static_cast<uint32_t>(tot_eq);
    }
  }
  if (t == 0) seg[U] = n;
  kmax = wide_max_u32(kmax, scratch);
  if (t == 0) *maxk_out = kmax;
  __syncthreads();
  return true;
}

// ---------------------------------------------------------------------------
// Kernel B: stream the slice once and hand its candidates over.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSplitThreads, 4) split_stream_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t *cand = reinterpret_cast<uint32_t *>(smem + kStreamCandOff);
  uint4 *stage = reinterpret_cast<uint4 *>(smem + kStreamStageOff);
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + kStreamMiscOff);

  const int U = p.ws_units_per_row;
  const int r = static_cast<int>(blockIdx.x) / U;
  const int u = static_cast<int>(blockIdx.x) - r * U;
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t lane = lane_id();
  if (r >= p.n_rows) {
    pdl_wait_and_release();
    return;
  }
  const Row w = load_row(p, r);
  if (w.err || w.fin) {  // kernel C reports it
    pdl_wait_and_release();
    return;
  }
  // ---- slice geometry; the first loads go out before the threshold arrives
  // (the logits were complete before the threshold kernel started) ----
  const int V = w.vocab;
  const int S = p.slice;
  const int s_begin = u * S;
  const int sc = max(0, min(S, V - s_begin));
  const char *rowp = static_cast<const char *>(p.logits) + w.off * 2;
  const char *sp = rowp + 2 * static_cast<int64_t>(s_begin);
  const int head =
      min(sc, static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(sp) & 15u)) & 15u) / 2u));
  const int nq = (sc - head) / 8;
  const int tail = sc - head - 8 * nq;
  const char *body = sp + 2 * head;
  const uint64_t pol = l2_evict_first();
  constexpr int kPerIter = kSplitThreads * kSplitU;
  const int n_it = (nq + kPerIter - 1) / kPerIter;
  uint4 cur[kSplitU];
#pragma unroll
  for (int j = 0; j < kSplitU; ++j) {
    const int m = j * kSplitThreads + t;
    cur[j] = m < nq ? ld_stream_v4(body + 16 * static_cast<size_t>(m), pol)
                    : make_uint4(0u, 0u, 0u, 0u);
  }
  if (t == 0) misc[kWN] = 0u;
  pdl_wait_and_release();  // the threshold kernel (if any) has finished
  SplitWs ws = split_ws(p.workspace, p.ws_rows, p.ws_units);
  uint32_t t_key = 0;
  if (p.split_inline) {
    // small launches: every CTA of the row takes the same sample itself
    // (the staging area holds the histogram), saving the threshold kernel
    if (!p.wide_exact && (V > kSplitRowCap || S > kSplitUnitCap))
      t_key = wide_sample_threshold<kSplitSampleRun>(rowp, V, w.k_eff, 1,
                                                     reinterpret_cast<uint32_t *>(stage), misc,
                                                     reinterpret_cast<uint64_t *>(misc + kWScan));
  } else {
    t_key = __ldcg(&ws.row[r].t_key);
  }
  __syncthreads();

  // ---- filter: every logit that compares >= t (NaN included) is kept as
  // a raw entry; a lane's flags for its four chunks of an iteration form one
  // 32-bit mask, and the warp compacts them once per iteration ----
  if (!p.wide_exact) {
    const uint32_t tb = wkey_bits(t_key);
    const uint32_t t2 = tb | (tb << 16);
    const uint32_t lt = lanemask_lt();
    const uint16_t *st16 = reinterpret_cast<const uint16_t *>(stage);
#pragma unroll 1
    for (int it = 0; it < n_it; ++it) {
      uint4 nxt[kSplitU];
#pragma unroll
      for (int j = 0; j < kSplitU; ++j) {
        const int m = (it + 1) * kPerIter + j * kSplitThreads + t;
        nxt[j] = m < nq ? ld_stream_v4(body + 16 * static_cast<size_t>(m), pol)
                        : make_uint4(0u, 0u, 0u, 0u);
      }
      uint32_t f = 0;  // bit 8 j + e: element e of chunk j
#pragma unroll
      for (int j = 0; j < kSplitU; ++j) {
        const int m = it * kPerIter + j * kSplitThreads + t;
        if (m < nq) {
          const uint32_t m0 = hgeu_mask(cur[j].x, t2), m1 = hgeu_mask(cur[j].y, t2);
          const uint32_t m2 = hgeu_mask(cur[j].z, t2), m3 = hgeu_mask(cur[j].w, t2);
          const uint32_t fj = (m0 & 1u) | ((m0 >> 30) & 2u) | ((m1 & 1u) << 2) |
                              ((m1 >> 28) & 8u) | ((m2 & 1u) << 4) | ((m2 >> 26) & 32u) |
                              ((m3 & 1u) << 6) | ((m3 >> 24) & 128u);
          f |= fj << (8 * j);
        }
      }
      const uint32_t c = __popc(f);
      const uint32_t wsum = __reduce_add_sync(0xFFFFFFFFu, c);
      if (wsum != 0u) {
        if (f) {  // the lane's chunks, for its own element lookups below
#pragma unroll
          for (int j = 0; j < kSplitU; ++j) stage[j * kSplitThreads + t] = cur[j];
        }
        // exclusive prefix of c over the warp's lanes, from its six bits
        uint32_t pre = 0;
#pragma unroll
        for (int bb = 0; bb < 6; ++bb)
          pre += static_cast<uint32_t>(__popc(__ballot_sync(0xFFFFFFFFu, (c >> bb) & 1u) & lt))
                 << bb;
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(&misc[kWN], wsum);
        uint32_t pos = __shfl_sync(0xFFFFFFFFu, base, 0) + pre;
        const uint32_t cmax = __reduce_max_sync(0xFFFFFFFFu, c);
        for (uint32_t q = 0; q < cmax; ++q) {  // the same trip count in every lane
          if (f) {
            const uint32_t e = static_cast<uint32_t>(__ffs(f) - 1);
            f &= f - 1u;
            const uint32_t j = e >> 3, k8 = e & 7u;
            const uint32_t bits = st16[(j * kSplitThreads + t) * 8u + k8];
            const uint32_t idx =
                static_cast<uint32_t>(head + 8 * (it * kPerIter + static_cast<int>(j) * kSplitThreads + t)) + k8;
            if (pos < static_cast<uint32_t>(kSplitUnitCap)) cand[pos] = (bits << 16) | idx;
            ++pos;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kSplitU; ++j) cur[j] = nxt[j];
    }
    if (t < head + tail) {
      const int idx = t < head ? t : head + 8 * nq + (t - head);
      const uint32_t bits = KeyBF16::load_one(sp, idx);
      const uint32_t k = KeyBF16::key(bits);
      if (k >= t_key || k < KeyBF16::kNegInf || k >= KeyBF16::kPosInf) {
        const uint32_t pos = atomicAdd(&misc[kWN], 1u);
        if (pos < static_cast<uint32_t>(kSplitUnitCap)) cand[pos] = (bits << 16) | static_cast<uint32_t>(idx);
      }
    }
  }
  __syncthreads();
  // ---- hand over: the unit's entries go to the row's candidate array at a
  // run reserved with one atomic ----
  const size_t ui = static_cast<size_t>(r) * U + u;  // == blockIdx.x
  const uint32_t n_loc = misc[kWN];
  const uint32_t n_copy = min(n_loc, static_cast<uint32_t>(kSplitUnitCap));
  if (t == 0) misc[kWFast] = atomicAdd(&ws.row[r].count, n_copy);
  __syncthreads();
  const uint32_t base = misc[kWFast];
  uint32_t *gc = ws.cand + static_cast<size_t>(r) * kSplitRowCap;
  for (uint32_t i = static_cast<uint32_t>(t); i < n_copy; i += kSplitThreads)
    if (base + i < static_cast<uint32_t>(kSplitRowCap)) __stcg(&gc[base + i], cand[i]);
  if (t == 0) {
    SplitUnitMeta mt;
    mt.n = n_loc;
    mt.base = base;
    mt.pad[0] = 0u;
    mt.pad[1] = 0u;
    __stcg(reinterpret_cast<uint4 *>(&ws.unit[ui]), *reinterpret_cast<uint4 *>(&mt));
  }
}

// ---------------------------------------------------------------------------
// Kernel C: one CTA per row gathers the units' candidates and runs the tail.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSplitThreads, 4) split_tail_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t *cand = reinterpret_cast<uint32_t *>(smem + kTailCandOff);
  uint32_t *hw = reinterpret_cast<uint32_t *>(smem + kTailHwOff);
  uint32_t *list = reinterpret_cast<uint32_t *>(smem + kTailListOff);
  uint32_t *pgc = reinterpret_cast<uint32_t *>(smem + kTailPgOff);
  uint32_t *page_slot = reinterpret_cast<uint32_t *>(smem + kTailPageSlotOff);
  uint32_t *slot_page = reinterpret_cast<uint32_t *>(smem + kTailSlotPageOff);
  uint32_t *seg = reinterpret_cast<uint32_t *>(smem + kTailSegOff);
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + kTailMiscOff);
  uint64_t *scratch = reinterpret_cast<uint64_t *>(misc + kWScan);

  const int r = static_cast<int>(blockIdx.x);
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t lane = lane_id();
  if (r >= p.n_rows) {
    pdl_wait_and_release();
    return;
  }
  // the inputs were complete before the threshold kernel started
  const Row w = load_row(p, r);
  if (t == 32 && !w.err && !w.fin && !w.greedy)
    misc[kWU24] = philox_u24(p.seed[r], p.request[r], static_cast<uint64_t>(w.stepv),
                             static_cast<uint64_t>(static_cast<int64_t>(p.codebook[r])));
  pdl_wait_and_release();  // the streaming kernel has finished
  if (t == 0) {  // the row's counter starts at zero for the next call
    SplitWs ws0 = split_ws(p.workspace, p.ws_rows, p.ws_units);
    ws0.row[r].count = 0u;
  }
  if (w.err || w.fin) {
    if (t == 0) finish_row(p, r, w, -1, w.err);
    return;
  }
  const int U = p.ws_units_per_row;
  const int S = p.slice;
  const int V = w.vocab;
  const uint32_t k_eff = static_cast<uint32_t>(w.k_eff);
  SplitWs ws = split_ws(p.workspace, p.ws_rows, p.ws_units);
  const size_t u0 = static_cast<size_t>(r) * U;

  // ---- one round of loads: the row's whole candidate array, whatever its
  // count, copied straight into shared memory, and the units' records ----
  if (!p.wide_exact) {
    const uint32_t *src = ws.cand + static_cast<size_t>(r) * kSplitRowCap;
#pragma unroll
    for (int j = 0; j < kSplitRowCap / (4 * kSplitThreads); ++j) {
      const int q = j * kSplitThreads + t;
      cp_async16(&cand[4 * q], &src[4 * q]);
    }
  }
  pgc[t] = 0u;
  if (t < 32) {
    uint4 mt = make_uint4(0u, 0u, 0u, 0u);
    if (t < U) mt = __ldcg(reinterpret_cast<const uint4 *>(&ws.unit[u0 + t]));
    const uint32_t nc = min(mt.x, static_cast<uint32_t>(kSplitUnitCap));  // entries written
    const uint32_t tot = __reduce_add_sync(0xFFFFFFFFu, nc);
    const bool fl = __any_sync(0xFFFFFFFFu, mt.x > static_cast<uint32_t>(kSplitUnitCap));
    // segments: the units that wrote entries, in the order of their runs
    const bool has = t < U && nc != 0u;
    const uint32_t bkey = has ? mt.y : 0xFFFFFFFFu;
    uint32_t rank = 0;
#pragma unroll
    for (int o = 0; o < kSplitMaxUnits; ++o) rank += __shfl_sync(0xFFFFFFFFu, bkey, o) < bkey ? 1u : 0u;
    const uint32_t n_has = static_cast<uint32_t>(__popc(__ballot_sync(0xFFFFFFFFu, has)));
    if (has) {
      seg[rank] = mt.y;
      seg[kSplitUmapOff + rank] = static_cast<uint32_t>(t);
    }
    if (static_cast<uint32_t>(t) >= n_has && t <= U) seg[t] = tot;
    if (t == 0) {
      misc[kWTotal] = tot;
      misc[kWRange] = fl ? 1u : 0u;
    }
  }
  cp_async_wait_all();
  __syncthreads();
  const uint32_t total = misc[kWTotal], full = misc[kWRange];
  const uint32_t u24 = misc[kWU24];
  uint32_t maxk = 0;
  int n = 0, up = 0;
  if (!p.wide_exact && !full && total >= k_eff && total <= static_cast<uint32_t>(kSplitRowCap)) {
    // ---- keys, page counts, maximum and the NaN / +inf check ----
    n = static_cast<int>(total);
    uint32_t nbad = 0, kmax = 0;
#pragma unroll 4
    for (int i = t; i < n; i += kSplitThreads) {
      const uint32_t e = cand[i];
      const uint32_t k = KeyBF16::key(e >> 16);
      nbad |= (k < KeyBF16::kNegInf || k >= KeyBF16::kPosInf) ? 1u : 0u;
      kmax = max(kmax, k);
      cand[i] = (k << 16) | (e & 0xFFFFu);
      atomicAdd(&pgc[k >> 8], 1u);
    }
    if (__syncthreads_or(nbad != 0u)) {
      if (t == 0) finish_row(p, r, w, -1, kRowNonFinite);
      return;
    }
    maxk = wide_max_u32(kmax, scratch);
    up = split_key_setup(pgc, k_eff, hw, page_slot, slot_page, misc, scratch);
    if (up <= kSplitKeyPages) {
      const uint32_t page = misc[kWDigit];
#pragma unroll 4
      for (int i = t; i < n; i += kSplitThreads) split_key_count(cand[i] >> 16, page, page_slot, hw);
    }
  } else {
    const char *rowp = static_cast<const char *>(p.logits) + w.off * 2;
    uint32_t *mk = &misc[kWMaxK];
    if (!split_exact(rowp, V, U, S, k_eff, cand, seg, pgc, mk, hw, misc, scratch)) {
      if (t == 0) finish_row(p, r, w, -1, kRowNonFinite);
      return;
    }
    maxk = *mk;
    n = static_cast<int>(min(seg[U], static_cast<uint32_t>(kSplitRowCap)));
    up = split_key_setup(pgc, k_eff, hw, page_slot, slot_page, misc, scratch);
    if (up <= kSplitKeyPages) {
      const uint32_t page = misc[kWDigit];
#pragma unroll 4
      for (int i = t; i < n; i += kSplitThreads) split_key_count(cand[i] >> 16, page, page_slot, hw);
    }
  }
  __syncthreads();
  if (maxk <= KeyBF16::kNegInf) {  // every candidate is -inf: no finite logit in the row
    if (t == 0) finish_row(p, r, w, -1, kRowNonFinite);
    return;
  }
  if (up > kSplitKeyPages ||
      !split_key_tail(p, r, w, cand, n, seg, U, S, maxk, up, u24, hw, list, slot_page, misc,
                      scratch)) {
    __syncthreads();
    split_row_tail(p, r, w, cand, n, seg, U, S, pgc, maxk, hw, misc, scratch);
  }
}

}  // namespace ts
