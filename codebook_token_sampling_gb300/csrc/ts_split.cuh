// ts_split.cuh -- the wide-row sampler as two kernels over a workspace (bf16
// rows such as the 151,936-token backbone vocabulary, any top-k cap up to
// 4096: Drama 3 article, section "能跑通的命令，和文档写明的边界").
//
// Kernel A (one CTA per row) reads an evenly spaced sample of the row and
// stores the threshold key t (the sampling step of Floyd and Rivest's
// selection, "Expected time bounds for selection", CACM 18(3), 1975); it
// also resets the row's arrival counter.
//
// Kernel B (U CTAs per row, one contiguous slice each) streams its slice
// once with 16-byte loads and keeps every logit >= t: candidates (key << 16 |
// slice index), their counts by key >> 8, the maximum key and a NaN / +inf
// flag go to the workspace.  A CTA that is not the last of its row to arrive
// leaves at once, so the streaming CTAs never wait for one another.  The
// last one gathers the row's candidates (a few thousand, from L2) and runs
// the row's tail alone:
//   - the threshold key thr (the k_eff-th largest) and `need`, the kept
//     tokens tied at it, from the page counts and one 256-bin pass;
//   - the kept masses (2^-40 fixed point, depending only on the key) over
//     256 coarse bins of (max key - key) >> shift, then an exact level inside
//     the bins of the nucleus cutoff and of the draw;
//   - the drawn token by a radix select on the token index.
// If the sample misled t (fewer than k_eff candidates, or more than the
// buffers hold) the last CTA re-reads the row and selects exactly.  Nothing
// waits on another CTA: the only cross-CTA step is an atomic counter.
#pragma once

#include "ts_wide.cuh"

namespace ts {

constexpr int kSplitThreads = 256;
constexpr int kSplitUnitCap = 4096;     // candidates one CTA may hand over
constexpr int kSplitRowCap = 8192;      // candidates the last CTA gathers
constexpr int kSplitMaxUnits = 16;
constexpr int kSplitU = 4;              // 16-byte chunks per lane per iteration
// dynamic shared memory: the gathered candidates (32 KB; the streaming phase
// keeps its own candidates and staging rings there), the tail's histograms
// (20 KB), page counts and bookkeeping
constexpr uint32_t kSplitCandOff = 0;
constexpr uint32_t kSplitRingOff = kSplitUnitCap * 4;                       // streaming only
constexpr int kSplitKeyPages = 32;       // per-key counts for up to 32 pages of 256 keys
constexpr uint32_t kSplitHwOff = kSplitRowCap * 4;                          // 20 KB
constexpr uint32_t kSplitPgOff = kSplitHwOff + 20480;                       // 256 words
constexpr uint32_t kSplitSegOff = kSplitPgOff + 1024;                       // 32 words
constexpr uint32_t kSplitMiscOff = kSplitSegOff + 128;                      // 256 words
constexpr uint32_t kSplitSmemBytes = kSplitMiscOff + kWideMiscWords * 4;

// Workspace layout, in 4-byte words (every region 16-byte aligned).
struct SplitRowMeta {
  uint32_t t_key;
  uint32_t arrived;
  uint32_t pad[2];
};
struct SplitUnitMeta {
  uint32_t n;     // candidates of the unit (may exceed kSplitUnitCap)
  uint32_t maxk;  // largest candidate key
  uint32_t bad;   // a NaN / +inf was met
  uint32_t pad;
};

// Row records for max_rows rows, then unit records for max_units units (a
// launch's CTAs: unit r * U + u is slice u of row r).
__host__ __device__ inline size_t split_workspace_bytes(int max_rows, int max_units) {
  const size_t rows = static_cast<size_t>(max_rows), units = static_cast<size_t>(max_units);
  return rows * sizeof(SplitRowMeta) + units * sizeof(SplitUnitMeta) + units * 256 * 4 +
         units * kSplitUnitCap * 4;
}

struct SplitWs {
  SplitRowMeta *row;
  SplitUnitMeta *unit;
  uint32_t *pg;    // [unit][256]
  uint32_t *cand;  // [unit][kSplitUnitCap]
};

__device__ __forceinline__ SplitWs split_ws(void *base, int max_rows, int max_units) {
  SplitWs ws;
  char *b = static_cast<char *>(base);
  const size_t rows = static_cast<size_t>(max_rows), units = static_cast<size_t>(max_units);
  ws.row = reinterpret_cast<SplitRowMeta *>(b);
  b += rows * sizeof(SplitRowMeta);
  ws.unit = reinterpret_cast<SplitUnitMeta *>(b);
  b += units * sizeof(SplitUnitMeta);
  ws.pg = reinterpret_cast<uint32_t *>(b);
  b += units * 256 * 4;
  ws.cand = reinterpret_cast<uint32_t *>(b);
  return ws;
}

// ---------------------------------------------------------------------------
// Kernel A: the row's threshold key from its sample; resets the counter.
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
  if (!w.err && !p.wide_exact) {
    const char *rowp = static_cast<const char *>(p.logits) + w.off * 2;
    // a row the last CTA can gather whole, in slices each CTA can hold,
    // keeps every logit (t = lowest key); others sample
    if (w.vocab > kSplitRowCap || p.slice > kSplitUnitCap)
      t_key = wide_sample_threshold(rowp, w.vocab, w.k_eff, 1, hist, misc,
                                    reinterpret_cast<uint64_t *>(misc + kWScan));
  }
  if (t == 0) {
    ws.row[r].t_key = t_key;
    ws.row[r].arrived = 0u;
  }
}

// One candidate of the streaming phase: its entry, its page count and the
// running maximum.
__device__ __forceinline__ void split_keep(uint32_t key, uint32_t idx, uint32_t pos,
                                           uint32_t *cand, uint32_t *pg, uint32_t &kmax) {
  if (pos < static_cast<uint32_t>(kSplitUnitCap)) cand[pos] = (key << 16) | idx;
  atomicAdd(&pg[key >> 8], 1u);
  kmax = max(kmax, key);
}

// Drains n <= 32 staged words (two logits each) from a warp's ring.
__device__ __forceinline__ void split_drain(const uint2 *ring, uint32_t head, uint32_t n,
                                            uint32_t t_key, uint32_t *cand, uint32_t *pg,
                                            uint32_t *counter, uint32_t &bad, uint32_t &kmax) {
  const uint32_t lane = lane_id();
  bool f0 = false, f1 = false;
  uint32_t k0 = 0, k1 = 0, idx0 = 0;
  if (lane < n) {
    const uint2 e = ring[(head + lane) & (kWideRing - 1)];
    const uint32_t kw = KeyBF16::key_word(e.x);
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
  if (f0) split_keep(k0, idx0, pos, cand, pg, kmax);
  if (f1) split_keep(k1, idx0 + 1u, pos + (f0 ? 1u : 0u), cand, pg, kmax);
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
    int c = 0;
    for (int i = t; i < n; i += kSplitThreads) {
      while (c + 1 < U && static_cast<uint32_t>(i) >= seg[c + 1]) ++c;
      const uint32_t e = cand[i];
      if ((e >> 16) != key_sel) continue;
      const uint32_t g = static_cast<uint32_t>(c * S) + (e & 0xFFFFu);
      if (level == 0)
        atomicAdd(&h[g >> 9], 1u);
      else if ((g >> 9) == b1)
        atomicAdd(&h[g & 511u], 1u);
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
    int c = 0;
    for (int i = t; i < n; i += kSplitThreads) {
      while (c + 1 < U && static_cast<uint32_t>(i) >= seg[c + 1]) ++c;
      const uint32_t e = cand[i];
      const uint32_t key = e >> 16;
      const uint32_t g = static_cast<uint32_t>(c * S) + (e & 0xFFFFu);
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

// The row's tail from per-key counts: every page (256 keys, key >> 8) at or
// above the threshold's page that holds a candidate gets a slot of 256
// packed 16-bit counts; one pass counts the candidates per key, and block
// scans over those keys (in key order) give the threshold key and `need`,
// S_k, the nucleus cutoff and the draw, with one weight evaluation per key
// that occurs.  Returns false (nothing written) when more than
// kSplitKeyPages pages are occupied; the caller then runs split_row_tail.
__device__ bool split_key_tail(const Params &p, int r, const Row &w, const uint32_t *cand, int n,
                               const uint32_t *seg, int U, int S, const uint32_t *pgc,
                               uint32_t maxk, uint32_t *hw, uint32_t *misc, uint64_t *scratch) {
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t k_eff = static_cast<uint32_t>(w.k_eff);
  uint64_t *m64 = reinterpret_cast<uint64_t *>(misc);
  uint32_t *kc = hw;                           // [slot][128] packed counts (16 KB)
  uint32_t *page_slot = hw + kSplitKeyPages * 128;
  uint32_t *slot_page = page_slot + 256;       // 32
  uint32_t *rs = slot_page + 32;               // rank select (512)
  // ---- the threshold's page; slots for the occupied pages at or above it ----
  const uint32_t c = pgc[t];
  wide_select256(c, k_eff, misc, scratch);
  const uint32_t page = misc[kWDigit];
  const bool occ = static_cast<uint32_t>(t) >= page && c != 0u;
  uint64_t n_occ;
  const uint32_t slot = static_cast<uint32_t>(wide_excl_scan_u64(occ ? 1u : 0u, scratch, &n_occ));
  const int up = static_cast<int>(n_occ);
  if (up > kSplitKeyPages) return false;
  page_slot[t] = occ ? slot : 0xFFFFFFFFu;
  if (occ) slot_page[slot] = static_cast<uint32_t>(t);
  for (int i = t; i < up * 128; i += kSplitThreads) kc[i] = 0u;
  __syncthreads();
#pragma unroll 4
  for (int i = t; i < n; i += kSplitThreads) {
    const uint32_t key = cand[i] >> 16;
    if ((key >> 8) < page) continue;
    const uint32_t sl = page_slot[key >> 8];
    atomicAdd(&kc[sl * 128 + ((key & 255u) >> 1)], 1u << ((key & 1u) * 16u));
  }
  __syncthreads();
  // bins in key order: bin b = slot b >> 8, low byte b & 255; thread t owns
  // bins [t * up, t * up + up)
  auto bin_key = [&](int b) { return (slot_page[b >> 8] << 8) | static_cast<uint32_t>(b & 255); };
  auto bin_cnt = [&](int b) {
    return (kc[(b >> 8) * 128 + ((b & 255) >> 1)] >> ((b & 1) * 16)) & 0xFFFFu;
  };
  const int b0 = t * up;
  // ---- threshold key (k_eff-th largest) and `need` ----
  uint32_t s = 0;
  for (int b = b0; b < b0 + up; ++b) s += bin_cnt(b);
  uint64_t tot;
  uint32_t ex = static_cast<uint32_t>(wide_excl_scan_u64(s, scratch, &tot));
  uint32_t above = static_cast<uint32_t>(tot) - ex - s;
  if (s != 0 && above < k_eff && above + s >= k_eff) {
    uint32_t run = above;
    for (int b = b0 + up - 1; b >= b0; --b) {
      const uint32_t cb = bin_cnt(b);
      if (run < k_eff && run + cb >= k_eff) {
        misc[kWTKey] = bin_key(b);
        misc[kWTake] = k_eff - run;
      }
      run += cb;
    }
  }
  __syncthreads();
  const uint32_t thr = misc[kWTKey];
  const uint32_t need = misc[kWTake];
  const float m = KeyBF16::value(maxk);
  const uint32_t u24 = misc[kWU24];
  uint32_t key_d = maxk, rho = 0, n_p = 1;
  uint64_t s_k = 0;
  if (!w.greedy) {
    auto kept = [&](int b, uint32_t key) {
      return key > thr ? bin_cnt(b) : (key == thr ? need : 0u);
    };
    auto weight = [&](uint32_t key) {
      return to_fixed(kept_weight(KeyBF16::value(key), m, w.temp, w.inv_temp));
    };
    uint64_t st = 0;
    uint32_t ct = 0;
    for (int b = b0; b < b0 + up; ++b) {
      const uint32_t key = bin_key(b), cnt = kept(b, key);
      if (cnt) {
        st += cnt * weight(key);
        ct += cnt;
      }
    }
    const uint64_t ex_m = wide_excl_scan_u64(st, scratch, &s_k);
    const uint64_t above_m = s_k - ex_m - st;
    uint64_t n_kept;
    const uint32_t ex_c = static_cast<uint32_t>(wide_excl_scan_u64(ct, scratch, &n_kept));
    const uint32_t above_c = static_cast<uint32_t>(n_kept) - ex_c - ct;
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
        uint32_t ccum = above_c;
        for (int b = b0 + up - 1; b >= b0; --b) {
          const uint32_t key = bin_key(b), cnt = kept(b, key);
          if (!cnt) continue;
          const uint64_t wb = weight(key), mb = cnt * wb;
          if (cum < cut && cum + mb >= cut) {
            uint64_t n_c = wb > 0 ? (cut - cum + wb - 1) / wb : 1;
            if (n_c < 1) n_c = 1;
            m64[kWSp / 2] = cum + n_c * wb;
            misc[kWNp] = ccum + static_cast<uint32_t>(n_c);
          }
          cum += mb;
          ccum += cnt;
        }
      }
      __syncthreads();
      s_p = m64[kWSp / 2];
      n_p = misc[kWNp];
    }
    // ---- draw ----
    const uint64_t target = scale_u24(u24, s_p);
    if (st != 0 && above_m <= target && target < above_m + st) {
      uint64_t cum = above_m;
      for (int b = b0 + up - 1; b >= b0; --b) {
        const uint32_t key = bin_key(b), cnt = kept(b, key);
        if (!cnt) continue;
        const uint64_t wb = weight(key), mb = cnt * wb;
        if (cum <= target && target < cum + mb) {
          misc[kWDrawB] = key;
          misc[kWRho] = static_cast<uint32_t>((target - cum) / wb);
        }
        cum += mb;
      }
    }
    __syncthreads();
    key_d = misc[kWDrawB];
    rho = misc[kWRho];
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
    int cs = 0;
    for (int i = t; i < n; i += kSplitThreads) {
      while (cs + 1 < U && static_cast<uint32_t>(i) >= seg[cs + 1]) ++cs;
      const uint32_t e = cand[i];
      const uint32_t key = e >> 16;
      const uint32_t g = static_cast<uint32_t>(cs * S) + (e & 0xFFFFu);
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
  return true;
}

// Exact fallback of the last CTA: the whole row read again, the k_eff-th
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
// Kernel B: stream, hand over, and (last CTA of the row) the tail.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSplitThreads, 4) split_stream_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t *cand = reinterpret_cast<uint32_t *>(smem + kSplitCandOff);
  uint2 *rings = reinterpret_cast<uint2 *>(smem + kSplitRingOff);
  uint32_t *hw = reinterpret_cast<uint32_t *>(smem + kSplitHwOff);
  uint32_t *pg = reinterpret_cast<uint32_t *>(smem + kSplitPgOff);
  uint32_t *seg = reinterpret_cast<uint32_t *>(smem + kSplitSegOff);
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + kSplitMiscOff);
  uint64_t *scratch = reinterpret_cast<uint64_t *>(misc + kWScan);

  const int U = p.ws_units_per_row;
  const int r = static_cast<int>(blockIdx.x) / U;
  const int u = static_cast<int>(blockIdx.x) - r * U;
  const int t = static_cast<int>(threadIdx.x);
  const uint32_t lane = lane_id();
  const int warp = t >> 5;
  if (r >= p.n_rows) {
    pdl_wait_and_release();
    return;
  }
  const Row w = load_row(p, r);
  if (w.err) {
    pdl_wait_and_release();
    if (u == 0 && t == 0) finish_row(p, r, w, -1, w.err);
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
  pg[t] = 0u;  // kSplitThreads == 256 pages
  if (t == 0) misc[kWN] = 0u;
  if (t == 32 && !w.greedy)
    misc[kWU24] = philox_u24(p.seed[r], p.request[r], static_cast<uint64_t>(p.step[w.stream]),
                             static_cast<uint64_t>(static_cast<int64_t>(p.codebook[r])));
  pdl_wait_and_release();  // the threshold kernel has finished
  SplitWs ws = split_ws(p.workspace, p.ws_rows, p.ws_units);
  const uint32_t t_key = __ldcg(&ws.row[r].t_key);
  __syncthreads();

  // ---- filter: every logit with key >= t_key becomes a candidate ----
  uint32_t bad = 0, kmax = 0;
  if (!p.wide_exact) {
    const uint32_t tb = wkey_bits(t_key);
    const uint32_t t2 = tb | (tb << 16);
    uint2 *ring = rings + warp * kWideRing;
    const uint32_t lt = lanemask_lt();
    uint32_t rh = 0, rt = 0;
#pragma unroll 1
    for (int it = 0; it < n_it; ++it) {
      uint4 nxt[kSplitU];
#pragma unroll
      for (int j = 0; j < kSplitU; ++j) {
        const int m = (it + 1) * kPerIter + j * kSplitThreads + t;
        nxt[j] = m < nq ? ld_stream_v4(body + 16 * static_cast<size_t>(m), pol)
                        : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < kSplitU; ++j) {
        const int m = it * kPerIter + j * kSplitThreads + t;
        const uint32_t wd[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
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
            split_drain(ring, rh, 32u, t_key, cand, pg, &misc[kWN], bad, kmax);
            rh += 32u;
            __syncwarp();
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kSplitU; ++j) cur[j] = nxt[j];
    }
    __syncwarp();
    if (rt != rh) split_drain(ring, rh, rt - rh, t_key, cand, pg, &misc[kWN], bad, kmax);
    if (t < head + tail) {
      const int idx = t < head ? t : head + 8 * nq + (t - head);
      const uint32_t k = KeyBF16::key(KeyBF16::load_one(sp, idx));
      const bool nf = k < KeyBF16::kNegInf || k >= KeyBF16::kPosInf;
      bad |= nf;
      if (!nf && k >= t_key) split_keep(k, static_cast<uint32_t>(idx), atomicAdd(&misc[kWN], 1u),
                                        cand, pg, kmax);
    }
  }
  kmax = wide_max_u32(kmax, scratch);
  // ---- hand the unit's results over ----
  const size_t ui = static_cast<size_t>(r) * U + u;  // == blockIdx.x
  const uint32_t n_loc = misc[kWN];
  const int n_copy = static_cast<int>(min(n_loc, static_cast<uint32_t>(kSplitUnitCap)));
  uint32_t *gc = ws.cand + ui * kSplitUnitCap;
  for (int i = t; i < n_copy; i += kSplitThreads) __stcg(&gc[i], cand[i]);
  __stcg(&ws.pg[ui * 256 + t], pg[t]);
  const uint32_t bad_any = __syncthreads_or(bad != 0u);
  if (t == 0) {
    SplitUnitMeta mt;
    mt.n = n_loc;
    mt.maxk = kmax;
    mt.bad = bad_any;
    mt.pad = 0u;
    __stcg(reinterpret_cast<uint4 *>(&ws.unit[ui]), *reinterpret_cast<uint4 *>(&mt));
  }
  __threadfence();
  __syncthreads();
  if (t == 0) misc[kWFast] = atomicAdd(&ws.row[r].arrived, 1u) == static_cast<uint32_t>(U - 1);
  __syncthreads();
  if (!misc[kWFast]) return;
  __threadfence();

  // ---- last CTA of the row: gather and tail (every load of a step is issued
  // before any is used: the units' records are independent) ----
  const size_t u0 = static_cast<size_t>(r) * U;
  if (t < 32) {
    uint4 mt = make_uint4(0u, 0u, 0u, 0u);
    if (t < U) mt = __ldcg(reinterpret_cast<const uint4 *>(&ws.unit[u0 + t]));
    uint32_t incl = mt.x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= static_cast<uint32_t>(o)) incl += x;
    }
    const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, mt.y);
    const bool bd = __any_sync(0xFFFFFFFFu, mt.z != 0u);
    const bool fl = __any_sync(0xFFFFFFFFu, mt.x > static_cast<uint32_t>(kSplitUnitCap));
    if (t <= U) seg[t] = incl - mt.x;  // exclusive offsets; seg[U] = total
    if (t == 0) {
      misc[kWTotal] = tot;
      misc[kWMaxB] = mk;
      misc[kWBad] = bd ? 1u : 0u;
      misc[kWRange] = fl ? 1u : 0u;
    }
  }
  __syncthreads();
  const uint32_t total = misc[kWTotal], any_bad = misc[kWBad], full = misc[kWRange];
  uint32_t maxk = misc[kWMaxB];
  if (any_bad) {
    if (t == 0) finish_row(p, r, w, -1, kRowNonFinite);
    return;
  }
  uint32_t *pgc = pg;  // merged page counts
  int n = 0;
  const uint32_t k_eff = static_cast<uint32_t>(w.k_eff);
  if (!p.wide_exact && !full && total >= k_eff && total <= static_cast<uint32_t>(kSplitRowCap)) {
    uint32_t v[kSplitMaxUnits];
#pragma unroll
    for (int c = 0; c < kSplitMaxUnits; ++c)
      v[c] = c < U ? __ldcg(&ws.pg[(u0 + c) * 256 + t]) : 0u;
    uint32_t sum = 0;
#pragma unroll
    for (int c = 0; c < kSplitMaxUnits; ++c) sum += v[c];
    pgc[t] = sum;
    // the candidates, flattened over the units: entry i of the row is entry
    // i - seg[c] of unit c (seg is increasing in i for each thread)
    const uint32_t *src0 = ws.cand + u0 * kSplitUnitCap;
    constexpr int kBatch = 8;
    int c = 0;
    for (uint32_t base = t; base < total; base += kBatch * kSplitThreads) {
      uint32_t val[kBatch];
      uint32_t dst[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const uint32_t i = base + j * kSplitThreads;
        dst[j] = i;
        val[j] = 0u;
        if (i < total) {
          while (c + 1 < U && i >= seg[c + 1]) ++c;
          val[j] = __ldcg(&src0[static_cast<size_t>(c) * kSplitUnitCap + (i - seg[c])]);
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (dst[j] < total) cand[dst[j]] = val[j];
    }
    n = static_cast<int>(total);
  } else {
    uint32_t *mk = &misc[kWMaxK];
    if (!split_exact(rowp, V, U, S, k_eff, cand, seg, pgc, mk, hw, misc, scratch)) {
      if (t == 0) finish_row(p, r, w, -1, kRowNonFinite);
      return;
    }
    maxk = *mk;
    n = static_cast<int>(min(seg[U], static_cast<uint32_t>(kSplitRowCap)));
  }
  __syncthreads();
  if (maxk <= KeyBF16::kNegInf) {  // every candidate is -inf: no finite logit in the row
    if (t == 0) finish_row(p, r, w, -1, kRowNonFinite);
    return;
  }
  if (!split_key_tail(p, r, w, cand, n, seg, U, S, pgc, maxk, hw, misc, scratch)) {
    __syncthreads();
    split_row_tail(p, r, w, cand, n, seg, U, S, pgc, maxk, hw, misc, scratch);
  }
}

}  // namespace ts
