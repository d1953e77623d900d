// ts_warp.cuh -- warp-path sampler for rows of up to 4096 bf16 or fp32
// logits with a top-k cap of at most 64 (the serving configuration: top_k 30
// under the default cap 64, Drama 3 article sections "测试口径" and
// "能跑通的命令，和文档写明的边界").
//
// A row is owned by one warp, or shared by 2 or 4 warps of a 128-thread
// block.  Per row:
//   1. its 16-byte chunks are copied into the row's shared-memory stage by
//      asynchronous copies, all in flight at once (the unaligned head and
//      tail elements are read one per lane);
//   2. every lane keeps the two largest logits of each of its two value
//      streams (the low and high halves of its bf16 words, or the even and
//      odd elements of its fp32 chunks): 128 sample values per row, among
//      them the row's maximum;
//   3. the k_eff-th largest sample value t0 is found by bisection on the
//      order-preserving key (warp-wide counts by redux.sync).  At least k_eff
//      logits of the row are >= t0, so the logits >= t0 (the candidates)
//      hold the whole top-k set with all its ties; for top_k 30 of 1024
//      gaussian logits they are about 31;
//   4. one packed compare per word marks the candidates in a per-lane
//      bitmap; the marked logits are written out as (key, inverted index)
//      words and bitonic-sorted by one warp (32, 64 or 128 slots);
//   5. the first k_eff sorted words are the top-k set in (logit desc, index
//      asc) order: fixed-point weights, one warp scan, the nucleus cutoff and
//      the draw, then the outputs.
// Rows with more than kWarpCandMax candidates (huge ties) take an exact
// radix-select slow path over the staged keys.
//
// The kernel walks its rows in batches of up to 32 consecutive rows: with G
// row groups (the warps sharing a row) in the grid and B rows per batch,
// group g takes batches g, g + G, g + 2G, ...  Lane i loads the parameters of
// the batch's i-th row and computes its Philox draw, so these cost one round
// of loads and one Philox evaluation per lane for up to 32 rows.  A launch may also span several decode steps (the
// multi-step mode): row g is row g mod n_rows of step g / n_rows.  With ready
// flags, a step's rows are sampled exactly when its flag is seen set; a warp
// waits up to the time limit for a flag only until the first one that does
// not come, and then looks at later flags once.
#pragma once

#include <cuda_bf16.h>

#include "ts_device.cuh"

namespace ts {

constexpr int kWarpCandMax = 128;
constexpr int kTowerWarps = 4;
constexpr int kTowerThreads = 32 * kTowerWarps;

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

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
  return __reduce_add_sync(0xFFFFFFFFu, v);
}
__device__ __forceinline__ uint32_t warp_max(uint32_t v) {
  return __reduce_max_sync(0xFFFFFFFFu, v);
}
__device__ __forceinline__ uint32_t warp_min(uint32_t v) {
  return __reduce_min_sync(0xFFFFFFFFu, v);
}

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

// Descending bitonic sort of 32 * R words; lane l holds positions R*l .. R*l +
// R - 1 in v[0 .. R-1].  Partners R or more positions apart are in another
// lane (a shuffle); closer ones are in the same lane.
template <class T, int R>
__device__ __forceinline__ void bitonic_desc(T (&v)[R]) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int size = 2; size <= 32 * R; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      if (j < R) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
          if ((i & j) == 0) {
            const bool desc = ((static_cast<uint32_t>(R) * lane + i) & size) == 0;
            const T a = v[i], b = v[i | j];
            const T hi = a > b ? a : b, lo = a > b ? b : a;
            v[i] = desc ? hi : lo;
            v[i | j] = desc ? lo : hi;
          }
        }
      } else {
        const int jl = j / R;
        const bool lower = (lane & static_cast<uint32_t>(jl)) == 0;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const T o = __shfl_xor_sync(0xFFFFFFFFu, v[i], jl);
          const bool desc = ((static_cast<uint32_t>(R) * lane + i) & size) == 0;
          v[i] = (lower == desc) ? (v[i] > o ? v[i] : o) : (v[i] < o ? v[i] : o);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Per-dtype lane helpers: the running top-2 of the lane's two value streams,
// the four sample keys, and the candidate bitmap of a chunk.
// ---------------------------------------------------------------------------
template <class K>
struct Lane;

template <>
struct Lane<KeyBF16> {
  // m1 >= m2 per half: the low halves of the lane's words are one stream,
  // the high halves the other.  m1 keeps a NaN once it has met one (a NaN
  // row is an error; m2 then no longer matters).
  struct Acc {
    uint32_t m1, m2;
  };
  static constexpr int kChunksPerMap = 4;  // a bitmap word covers 4 chunks (32 logits)
  static constexpr uint32_t kNeutral = 0xFF80FF80u;  // a word that folds to nothing (-inf, -inf)
  __device__ __forceinline__ static __nv_bfloat162 b2(uint32_t x) {
    return *reinterpret_cast<__nv_bfloat162 *>(&x);
  }
  __device__ __forceinline__ static uint32_t u(__nv_bfloat162 x) {
    return *reinterpret_cast<uint32_t *>(&x);
  }
  __device__ __forceinline__ static Acc init() { return {0xFF80FF80u, 0xFF80FF80u}; }
  __device__ __forceinline__ static void fold(uint32_t w, Acc &a) {
    a.m2 = u(__hmax2(b2(a.m2), __hmin2(b2(a.m1), b2(w))));
    a.m1 = u(__hmax2_nan(b2(a.m1), b2(w)));
  }
  __device__ __forceinline__ static void fold_chunk(const uint4 &c, Acc &a) {
    fold(c.x, a);
    fold(c.y, a);
    fold(c.z, a);
    fold(c.w, a);
  }
  __device__ __forceinline__ static void merge(Acc &a, const Acc &b) {
    a.m2 = u(__hmax2(__hmin2(b2(a.m1), b2(b.m1)), __hmax2(b2(a.m2), b2(b.m2))));
    a.m1 = u(__hmax2_nan(b2(a.m1), b2(b.m1)));
  }
  // a NaN among the logits folded into this lane's streams
  __device__ __forceinline__ static bool has_nan(const Acc &a) {
    return ((a.m1 & 0x7FFFu) > 0x7F80u) || ((a.m1 & 0x7FFF0000u) > 0x7F800000u);
  }
  __device__ __forceinline__ static void store(uint32_t *dst, const Acc &a) {
    dst[0] = a.m1;
    dst[1] = a.m2;
  }
  __device__ __forceinline__ static Acc load(const uint32_t *src) { return {src[0], src[1]}; }
  __device__ __forceinline__ static void sample_keys(const Acc &a, uint32_t (&k)[4]) {
    k[0] = KeyBF16::key(a.m1 & 0xFFFFu);
    k[1] = KeyBF16::key(a.m1 >> 16);
    k[2] = KeyBF16::key(a.m2 & 0xFFFFu);
    k[3] = KeyBF16::key(a.m2 >> 16);
  }
  // the threshold as a packed pair of bf16 values
  __device__ __forceinline__ static uint32_t splat(uint32_t key) {
    const uint32_t bits = key ^ ((key & 0x8000u) ? 0x8000u : 0xFFFFu);
    return bits | (bits << 16);
  }
  // bitmap bits of the logits >= t (unordered: a NaN is marked too) in chunk
  // slot cs (0..3) of a map word: word i of the chunk is map word w = 4 cs +
  // i, its low half at bit w and its high half at bit w + 16
  __device__ __forceinline__ static uint32_t flags(const uint4 &c, uint32_t t2, int cs) {
    const int w = 4 * cs;
    return (__hgeu2_mask(b2(c.x), b2(t2)) & (0x00010001u << w)) |
           (__hgeu2_mask(b2(c.y), b2(t2)) & (0x00010001u << (w + 1))) |
           (__hgeu2_mask(b2(c.z), b2(t2)) & (0x00010001u << (w + 2))) |
           (__hgeu2_mask(b2(c.w), b2(t2)) & (0x00010001u << (w + 3)));
  }
  // (chunk slot, element of the chunk) of a bitmap bit
  __device__ __forceinline__ static void bit_elem(int b, int &cs, int &e) {
    const int w = b & 15;
    cs = w >> 2;
    e = 2 * (w & 3) + (b >> 4);
  }
  // 16 times the number of the lane's four sample values whose key is >= c:
  // two packed compares against the value of key c (the row has no NaN here)
  __device__ __forceinline__ static uint32_t count16_ge(const Acc &a, uint32_t c) {
    const uint32_t bits = c ^ (0xFFFFu - (c >> 15) * 0x7FFFu);
    const uint32_t c2 = __byte_perm(bits, 0u, 0x1010);
    return __popc(__hge2_mask(b2(a.m1), b2(c2))) + __popc(__hge2_mask(b2(a.m2), b2(c2)));
  }
};

template <>
struct Lane<KeyF32> {
  // stream A: elements 0 and 2 of the lane's chunks, stream B: 1 and 3;
  // a1 / b1 keep a NaN once they have met one
  struct Acc {
    uint32_t a1, a2, b1, b2;
  };
  __device__ __forceinline__ static float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
  }
  static constexpr int kChunksPerMap = 8;  // a bitmap word covers 8 chunks (32 logits)
  static constexpr uint32_t kNeutral = 0xFF800000u;  // a word that folds to nothing (-inf)
  __device__ __forceinline__ static Acc init() {
    return {0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u};
  }
  __device__ __forceinline__ static void fold1(uint32_t w, uint32_t &m1, uint32_t &m2) {
    const float x = __uint_as_float(w), a = __uint_as_float(m1), b = __uint_as_float(m2);
    m2 = __float_as_uint(fmaxf(b, fminf(a, x)));
    m1 = __float_as_uint(max_nan(a, x));
  }
  __device__ __forceinline__ static void fold_chunk(const uint4 &c, Acc &a) {
    fold1(c.x, a.a1, a.a2);
    fold1(c.y, a.b1, a.b2);
    fold1(c.z, a.a1, a.a2);
    fold1(c.w, a.b1, a.b2);
  }
  __device__ __forceinline__ static void merge2(uint32_t &m1, uint32_t &m2, uint32_t n1,
                                                uint32_t n2) {
    const float a = __uint_as_float(m1), c = __uint_as_float(m2);
    const float x = __uint_as_float(n1), y = __uint_as_float(n2);
    m2 = __float_as_uint(fmaxf(fminf(a, x), fmaxf(c, y)));
    m1 = __float_as_uint(max_nan(a, x));
  }
  __device__ __forceinline__ static void merge(Acc &a, const Acc &b) {
    merge2(a.a1, a.a2, b.a1, b.a2);
    merge2(a.b1, a.b2, b.b1, b.b2);
  }
  __device__ __forceinline__ static bool has_nan(const Acc &a) {
    return (a.a1 & 0x7FFFFFFFu) > 0x7F800000u || (a.b1 & 0x7FFFFFFFu) > 0x7F800000u;
  }
  __device__ __forceinline__ static void store(uint32_t *dst, const Acc &a) {
    dst[0] = a.a1;
    dst[1] = a.a2;
    dst[2] = a.b1;
    dst[3] = a.b2;
  }
  __device__ __forceinline__ static Acc load(const uint32_t *src) {
    return {src[0], src[1], src[2], src[3]};
  }
  __device__ __forceinline__ static void sample_keys(const Acc &a, uint32_t (&k)[4]) {
    k[0] = KeyF32::key(a.a1);
    k[1] = KeyF32::key(a.b1);
    k[2] = KeyF32::key(a.a2);
    k[3] = KeyF32::key(a.b2);
  }
  __device__ __forceinline__ static uint32_t splat(uint32_t key) {
    return key ^ ((key & 0x80000000u) ? 0x80000000u : 0xFFFFFFFFu);
  }
  // bit 4 cs + e for element e of chunk slot cs (0..7) when it is >= t
  // (unordered: a NaN is marked too)
  __device__ __forceinline__ static uint32_t flags(const uint4 &c, uint32_t t, int cs) {
    const float tv = __uint_as_float(t);
    const int b = 4 * cs;
    return (static_cast<uint32_t>(!(__uint_as_float(c.x) < tv)) << b) |
           (static_cast<uint32_t>(!(__uint_as_float(c.y) < tv)) << (b + 1)) |
           (static_cast<uint32_t>(!(__uint_as_float(c.z) < tv)) << (b + 2)) |
           (static_cast<uint32_t>(!(__uint_as_float(c.w) < tv)) << (b + 3));
  }
  __device__ __forceinline__ static void bit_elem(int b, int &cs, int &e) {
    cs = b >> 2;
    e = b & 3;
  }
  __device__ __forceinline__ static uint32_t count16_ge(const Acc &a, uint32_t c) {
    uint32_t k[4];
    sample_keys(a, k);
    return 16u * (static_cast<uint32_t>(k[0] >= c) + static_cast<uint32_t>(k[1] >= c) +
                  static_cast<uint32_t>(k[2] >= c) + static_cast<uint32_t>(k[3] >= c));
  }
};

template <class K>
__host__ __device__ constexpr int acc_words() {
  return sizeof(typename Lane<K>::Acc) / 4;
}

// The kq-th largest of the warp's sample values (four per lane in `a`: the
// two streams' two largest; plus `ex` on lanes that hold a head or tail
// element), as a key, searched on the key's top 16 bits: for bf16 the exact
// key, for fp32 that key with its low 16 bits cleared (still a lower bound).
// The search starts from [lo, top], lo a key with at least kq sample keys >=
// it and top the largest sample key.
template <class K>
__device__ __forceinline__ uint32_t sample_kth(const typename Lane<K>::Acc &a, uint32_t ex,
                                               bool any_ex, int kq, uint32_t lo, uint32_t top) {
  constexpr int kShift = K::kBits - 16;
  const uint32_t lo16 = lo >> kShift, hi16 = top >> kShift;
  const uint32_t diff = lo16 ^ hi16;
  if (diff == 0) return lo16 << kShift;
  int b = 31 - __clz(diff);
  // the common prefix of lo and top, lower bits clear: <= lo
  uint32_t t16 = hi16 & ~((2u << b) - 1u);
  const uint32_t need = static_cast<uint32_t>(kq);
  // two bits per round: the counts at the three thresholds t16 + {1, 2, 3}
  // << (b - 1), packed in 8-bit fields (at most 5 keys per lane, 160 per
  // warp), go through one warp reduction
#pragma unroll 1
  for (; b >= 1; b -= 2) {
    const uint32_t c1 = (t16 | (1u << (b - 1))) << kShift;
    const uint32_t c2 = (t16 | (2u << (b - 1))) << kShift;
    const uint32_t c3 = (t16 | (3u << (b - 1))) << kShift;
    uint32_t n = (Lane<K>::count16_ge(a, c1) >> 4) | ((Lane<K>::count16_ge(a, c2) >> 4) << 8) |
                 ((Lane<K>::count16_ge(a, c3) >> 4) << 16);
    if (any_ex) n += (ex >= c1 ? 1u : 0u) + (ex >= c2 ? 0x100u : 0u) + (ex >= c3 ? 0x10000u : 0u);
    const uint32_t tot = warp_sum(n);
    const uint32_t step = (tot >> 16) >= need ? 3u : ((tot >> 8) & 0xFFu) >= need ? 2u
                        : (tot & 0xFFu) >= need ? 1u : 0u;
    t16 |= step << (b - 1);
  }
  if (b == 0) {
    const uint32_t c = (t16 | 1u) << kShift;
    uint32_t n = Lane<K>::count16_ge(a, c) >> 4;
    if (any_ex) n += ex >= c ? 1u : 0u;
    if (warp_sum(n) >= need) t16 |= 1u;
  }
  return t16 << kShift;
}

// The repetition penalty (Keskar et al. 2019, CTRL) on one logit's bits: a
// positive logit divided by theta, another multiplied by it, in fp32, the
// result rounded to the logits' type (nearest even for bf16).
template <class K>
__device__ __forceinline__ uint32_t penalised_bits(uint32_t bits, float theta);
template <>
__device__ __forceinline__ uint32_t penalised_bits<KeyBF16>(uint32_t bits, float theta) {
  const float f = __uint_as_float(bits << 16);
  const float pen = f > 0.0f ? __fdiv_rn(f, theta) : __fmul_rn(f, theta);
  const __nv_bfloat16 h = __float2bfloat16_rn(pen);
  return static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(&h));
}
template <>
__device__ __forceinline__ uint32_t penalised_bits<KeyF32>(uint32_t bits, float theta) {
  const float f = __uint_as_float(bits);
  return __float_as_uint(f > 0.0f ? __fdiv_rn(f, theta) : __fmul_rn(f, theta));
}

// ---------------------------------------------------------------------------
// One row's parameters, as one lane of the batch holds them.  The fields the
// row body needs early (offset, width, k_eff, flags) are broadcast when the
// row starts; the tail's (temperature, top_p, slot, EOS id) when it runs.
// ---------------------------------------------------------------------------
struct RowParams {
  int64_t off;    // element offset of the row (its step's logits included)
  int64_t t;      // the row's step (Philox counter word 0)
  int32_t r;      // row of the batch
  int32_t s;      // step index within the launch
  int32_t stream; // index into step[] (valid when the row has no shape error)
  uint32_t meta;  // vocab (bits 0-12) | k_eff (13-19) | greedy (20) | error bits (21-25)
                  // | finish reason (26-27)
  int32_t slot;   // write-back slot (its step's frame included), -1 = none
  int32_t eos;
  float temp;
  float top_p;
};
// 48 bytes: a block's four batches of 32 rows take 6 KB of shared memory, and
// the 16-column variant keeps five blocks per SM (the next step's blocks start
// beside the current step's).
static_assert(sizeof(RowParams) == 48, "RowParams is sized for the block's shared memory");

__device__ __forceinline__ int meta_vocab(uint32_t m) { return static_cast<int>(m & 0x1FFFu); }
__device__ __forceinline__ int meta_keff(uint32_t m) { return static_cast<int>((m >> 13) & 0x7Fu); }
__device__ __forceinline__ bool meta_greedy(uint32_t m) { return ((m >> 20) & 1u) != 0u; }
__device__ __forceinline__ uint32_t meta_err(uint32_t m) { return (m >> 21) & 0x1Fu; }
__device__ __forceinline__ uint32_t meta_fin(uint32_t m) { return m >> 26; }

// The parameters of row g of the launch (row g mod n_rows of step g / n_rows).
// Every check that the warp path needs is made here: a row whose width
// exceeds the launch's maximum is a shape error, so width and k_eff fit their
// fields.
__device__ __forceinline__ RowParams load_params(const Params &p, int64_t g) {
  RowParams w;
  const int s = p.n_steps == 1 ? 0 : static_cast<int>(g / p.n_rows);
  const int r = static_cast<int>(g - static_cast<int64_t>(s) * p.n_rows);
  w.r = r;
  w.s = s;
  const int32_t vocab = p.row_vocab[r];
  w.off = p.row_offsets[r];
  w.temp = p.temp[r];
  w.top_p = p.top_p[r];
  const int32_t stream = p.row_stream[r];
  w.stream = stream;
  const int32_t slot = p.feedback_buf ? p.feedback_slot[r] : -1;
  w.eos = p.eos_id ? p.eos_id[r] : -1;
  const int32_t tk = p.top_k[r];
  uint32_t e = 0;
  if (w.off < 0) e |= kRowBadShape;
  w.off += static_cast<int64_t>(s) * p.logits_step_stride;
  if (vocab <= 0 || vocab > p.max_row_vocab || w.off > p.logits_len - static_cast<int64_t>(vocab))
    e |= kRowBadShape;
  if (stream < 0 || stream >= p.n_streams) e |= kRowBadShape;
  uint32_t fin = 0;
  w.t = 0;
  if (isnan(w.temp) || isinf(w.temp) || isnan(w.top_p)) e |= kRowBadParam;
  if (slot >= 0 && static_cast<int64_t>(slot) >= p.feedback_len) e |= kRowBadSlot;
  w.slot = slot >= 0 ? static_cast<int32_t>(slot + static_cast<int64_t>(s) * p.feedback_step_stride)
                     : -1;
  if (p.hist_ring) {  // the history column and the penalty (read again where used)
    const int32_t cb = p.codebook[r];
    const float pen = p.rep_penalty[r];
    if (cb < 0 || cb >= p.hist_q) e |= kRowBadShape;
    if (isnan(pen) || isinf(pen) || !(pen > 0.0f)) e |= kRowBadParam;
  }
  // the finish rule and the history ring need the row's step now; without
  // them the step is read by the draw, while the row's logits are on their way
  if ((p.stop_step || p.max_steps || p.hist_ring) && !(e & (kRowBadShape | kRowBadSlot))) {
    w.t = p.step[stream] + s;
    fin = finish_rule(p, stream, w.t);
    if (fin) e = 0;  // a finished row's logits and parameters are not looked at
  }
  const int32_t v = (e || fin) ? 1 : vocab;
  int32_t k = tk > 0 ? tk : v;
  k = min(k, p.cap);
  k = min(k, v);
  const bool greedy = !(w.temp > 0.0f) || k == 1;
  w.meta = static_cast<uint32_t>(v) | (static_cast<uint32_t>(k) << 13) |
           (greedy ? (1u << 20) : 0u) | (e << 21) | (fin << 26);
  return w;
}

// The row's outputs: id, EOS flag and write-back (its step's slots), or the
// error marks.  `out` = the row's output index; eos / slot are used only
// without an error.
__device__ __forceinline__ void row_outputs(const Params &p, int r, int64_t out, int32_t eos,
                                            int32_t slot, int32_t id, uint32_t err,
                                            int32_t stream = 0, int64_t t = 0) {
  if (err) {
    p.out_ids[out] = -1;
    p.out_eos[out] = 0;
    atomicOr(p.status, err);
    if (p.kept_ids) {
      p.n_kept[r] = 0;
      p.n_nucleus[r] = 0;
    }
    return;
  }
  p.out_ids[out] = id;
  const bool is_eos = eos >= 0 && id == eos;
  p.out_eos[out] = static_cast<uint8_t>(is_eos);
  if (slot >= 0) p.feedback_buf[slot] = id;
  if (is_eos) {  // the stream stops: its rows pad from the next step on
    if (p.stop_step) p.stop_step[stream] = t;
    if (p.finish_reason) p.finish_reason[stream] = 1u;
  }
}

// The row's draw joins its history column at the slot of its step.
__device__ __forceinline__ void history_write(const Params &p, int32_t stream, int32_t cb,
                                              int64_t t, int32_t id) {
  const int64_t j = ((t % p.hist_len) + p.hist_len) % p.hist_len;
  p.hist_ring[(static_cast<int64_t>(stream) * p.hist_len + j) * p.hist_q + cb] = id;
}

// A finished stream's row: the pad id, no EOS flag, the reason.
__device__ __forceinline__ void row_padded(const Params &p, int r, int64_t out, int32_t slot,
                                           int32_t stream, uint32_t fin) {
  p.out_ids[out] = p.pad_id;
  p.out_eos[out] = 0;
  if (slot >= 0) p.feedback_buf[slot] = p.pad_id;
  if (p.finish_reason) p.finish_reason[stream] = static_cast<uint8_t>(fin);
  if (p.kept_ids) {
    p.n_kept[r] = 0;
    p.n_nucleus[r] = 0;
  }
}

// What the tail needs of a row: the row's parameters where the warp's batch
// keeps them (shared memory), read where they are used, so that none of them
// holds a register through the sort.
using TailParams = RowParams;

// Waits (lane 0, bounded) for a step's ready flag; true once it is set.  A
// zero limit looks at the flag once.
// The flag is read with acquire semantics at system scope, so that a flag
// written by the host (or by a copy) orders the step's logits before the
// loads that follow.
__device__ __forceinline__ bool wait_ready(const uint32_t *flag, uint64_t timeout_ns) {
  uint32_t ok = 0;
  if (lane_id() == 0) {
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
#pragma unroll 1
    for (uint32_t it = 0; it < (1u << 24); ++it) {
      uint32_t v;
      asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
      if (v) {
        ok = 1;
        break;
      }
      uint64_t t1;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
      if (t1 - t0 > timeout_ns) break;
      __nanosleep(200);
    }
  }
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// ---------------------------------------------------------------------------
// The tail: the sorted top-k set (kq <= 64 positions, lane l holds positions
// R*l .. R*l + R - 1), fixed-point weights, the nucleus cutoff and the draw.
// ---------------------------------------------------------------------------
template <class K, int R>
__device__ __forceinline__ void warp_tail(const Params &p, const TailParams &w,
                                          typename SortWord<K>::T (&v)[R], int kq,
                                          uint32_t u24) {
  using SW = SortWord<K>;
  using T = typename SW::T;
  const uint32_t lane = lane_id();
  const int pos0 = R * static_cast<int>(lane);
  const float m = K::value(SW::key(__shfl_sync(0xFFFFFFFFu, v[0], 0)));
  const bool greedy = meta_greedy(w.meta);
  const float inv_temp = greedy ? 1.0f : 1.0f / w.temp;
  float wt[R];
  uint64_t c[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    wt[i] = 0.f;
    if (!greedy && pos0 + i < kq) wt[i] = kept_weight(K::value(SW::key(v[i])), m, w.temp, inv_temp);
    c[i] = to_fixed(wt[i]);
    if (i > 0) c[i] += c[i - 1];
  }
  // prefix masses in 2^-40 units: the lane's inclusive local sums plus the
  // warp's exclusive scan of the lane totals
  const uint64_t incl = warp_incl_scan_u64(c[R - 1]);
  const uint64_t excl = incl - c[R - 1];
#pragma unroll
  for (int i = 0; i < R; ++i) c[i] += excl;
  const uint64_t s_k = __shfl_sync(0xFFFFFFFFu, incl, 31);

  int n_p = 1, pick = 0;
  if (!greedy) {
    if (w.top_p >= 1.0f) {
      n_p = kq;
    } else if (w.top_p > 0.0f) {
      const uint64_t cut_i = ceil_mul_p(w.top_p, s_k);  // C reaches top_p * S_k iff C >= cut_i
      uint32_t below = 0;
#pragma unroll
      for (int i = 0; i < R; ++i) below += (pos0 + i < kq && c[i] < cut_i) ? 1u : 0u;
      n_p = min(static_cast<int>(warp_sum(below)) + 1, kq);
    }
    const int last = n_p - 1;
    uint64_t cl = c[0];
#pragma unroll
    for (int i = 1; i < R; ++i)
      if ((last % R) == i) cl = c[i];
    const uint64_t s_p = __shfl_sync(0xFFFFFFFFu, cl, last / R);
    const uint64_t target = scale_u24(u24, s_p);
    uint32_t le = 0;
#pragma unroll
    for (int i = 0; i < R; ++i) le += (pos0 + i < n_p && c[i] <= target) ? 1u : 0u;
    pick = static_cast<int>(warp_sum(le));
  }
  T vp = v[0];
#pragma unroll
  for (int i = 1; i < R; ++i)
    if ((pick % R) == i) vp = v[i];
  const T pw = __shfl_sync(0xFFFFFFFFu, vp, pick / R);
  if (lane == 0) {
    const int32_t id = static_cast<int32_t>(SW::idx(pw));
    row_outputs(p, w.r, static_cast<int64_t>(w.s) * p.out_step_stride + w.r, w.eos, w.slot, id,
                0u, w.stream, w.t);
    if (p.hist_ring) history_write(p, w.stream, p.codebook[w.r], w.t, id);
  }

  if (p.kept_ids) {
    const float s_real = static_cast<float>(static_cast<double>(s_k) * (1.0 / 1099511627776.0));
    const int64_t rb = static_cast<int64_t>(w.r) * p.max_keep;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int q = pos0 + i;
      if (q < kq && q < p.max_keep) {
        p.kept_ids[rb + q] = static_cast<int32_t>(SW::idx(v[i]));
        p.kept_probs[rb + q] = greedy ? (q == 0 ? 1.f : 0.f) : __fdiv_rn(wt[i], s_real);
      }
    }
    if (lane == 0) {
      p.n_kept[w.r] = kq;
      p.n_nucleus[w.r] = n_p;
    }
  }
}

// Sorts the nc candidate words of `cand` and runs the tail on the first kq.
template <class K, int R>
__device__ __forceinline__ void sort_and_tail(const Params &p, const TailParams &w,
                                              const typename SortWord<K>::T *cand, int nc,
                                              uint32_t u24) {
  using T = typename SortWord<K>::T;
  const int pos0 = R * static_cast<int>(lane_id());
  T v[R];
#pragma unroll
  for (int i = 0; i < R; ++i) v[i] = pos0 + i < nc ? cand[pos0 + i] : T(0);
  if (nc > 1) bitonic_desc<T, R>(v);
  if constexpr (R <= 2) {
    warp_tail<K, R>(p, w, v, meta_keff(w.meta), u24);
  } else {
    // k_eff <= 64: the first 64 sorted positions, two per lane.  Position
    // 2l + h lives in lane (2l + h) / R, slot (2l + h) % R; readers want
    // different slots of one lane, so every slot is shuffled and the reader
    // keeps its own.
    T v2[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = 2 * static_cast<int>(lane_id()) + h;
      T x = T(0);
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const T y = __shfl_sync(0xFFFFFFFFu, v[i], q / R);
        if ((q % R) == i) x = y;
      }
      v2[h] = x;
    }
    warp_tail<K, 2>(p, w, v2, meta_keff(w.meta), u24);
  }
}

// The 128-slot sort (rows with 65 to 128 candidates).
template <class K>
__device__ __forceinline__ void sort_and_tail_128(const Params &p, const TailParams &w,
                                               const typename SortWord<K>::T *cand, int nc,
                                               uint32_t u24) {
  sort_and_tail<K, 4>(p, w, cand, nc, u24);
}

// Exact slow path for rows whose candidate count exceeds kWarpCandMax (huge
// ties): 8-bit radix select over the row's keys (keys(q) returns the keys of
// body chunk q, read again from the stage), then the top-k set collected in
// index order (keys equal to the threshold taken by lowest index) into
// cand[0 .. k_eff).
template <class K, class Loader>
__device__ __forceinline__ void warp_slow_select(int vocab, int k_eff, uint32_t *hist,
                                              typename SortWord<K>::T *cand, const Loader keys,
                                              int nq, int head, int tail, int eidx,
                                              uint32_t ekey) {
  using SW = SortWord<K>;
  constexpr int EPC = K::kPerChunk;
  const uint32_t lane = lane_id();
  const int rounds = (nq + 31) >> 5;

  uint32_t prefix = 0, pmask = 0;
  uint32_t kk = static_cast<uint32_t>(k_eff);
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
    if (eidx < vocab && (ekey & pmask) == prefix)
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
  const bool has_e = eidx < vocab;
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
}

// Shared memory of one row group: a stage of STG chunk columns (32 * STG
// chunks).  The slow path's histogram and the candidate words are never live
// at once, so they share storage.
template <class K, int STG, int WPR>
struct TowerShared {
  using T = typename SortWord<K>::T;
  uint4 stage[32 * STG];
  union {
    T cand[kWarpCandMax];
    uint32_t hist[256];
  } u;
  uint32_t xacc[(WPR > 1 ? WPR - 1 : 1) * 32 * acc_words<K>()];  // warps 1.. running pairs
  uint32_t xu[32];    // the batch's draws
  uint32_t xt0, xtop;
  uint32_t xready;    // the current step's ready flag came in time
  uint32_t xcnt;      // candidate slots taken so far
  uint32_t xbad[1];   // the row holds a NaN or +inf
};

// Barrier of the WPR warps that share a row (group grp of the block).
template <int WPR>
__device__ __forceinline__ void row_sync(int grp) {
  if constexpr (WPR == 1) {
    __syncwarp();
  } else if constexpr (WPR == 4) {
    asm volatile("bar.sync 1, 128;" ::: "memory");
  } else {  // two groups per block: barriers 1 and 2 (constant ids)
    if (grp == 0)
      asm volatile("bar.sync 1, 64;" ::: "memory");
    else
      asm volatile("bar.sync 2, 64;" ::: "memory");
  }
}

// After every block of the launch has read step[]: the last block to arrive
// adds n_steps to step_out[0 .. n_streams) and re-arms the ticket.  No block
// waits for another; every thread of the block must reach this call.
// Only the last block writes step_out, so every block reads the values it
// would add to before its ticket, while the block's other warps finish: the
// last block then only stores (one round trip less after the ticket).
// The ticket is taken with an acquire-release atomic at GPU scope: the block's
// reads of step[] (ordered before it by the block barrier) happen before the
// last block's acquire, so its increments cannot reach a reader of this
// launch.  The next launch in the stream sees them (and the re-armed ticket)
// once this grid has completed.
__device__ __forceinline__ void advance_steps_last_block(const Params &p) {
  __shared__ uint32_t last;
  const int tid = static_cast<int>(threadIdx.x);
  const bool one_pass = p.n_streams <= static_cast<int>(blockDim.x);
  int64_t cur = 0;
  if (one_pass && tid < p.n_streams) cur = p.step_out[tid];
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(old) : "l"(p.ticket) : "memory");
    last = old == gridDim.x - 1 ? 1u : 0u;
  }
  __syncthreads();
  if (!last) return;
  if (one_pass) {
    if (tid < p.n_streams) p.step_out[tid] = cur + p.n_steps;
  } else {
    for (int i = tid; i < p.n_streams; i += static_cast<int>(blockDim.x)) p.step_out[i] += p.n_steps;
  }
  if (threadIdx.x == 0) *p.ticket = 0u;
}

// MAXNCH = most 16-byte chunks per lane of any row in the launch (1, 2, 4, 8,
// 16, or 32 for fp32 rows wider than 2048); WPR = warps per row (1, 2 or 4);
// STG = chunk columns the stage
// holds (MAXNCH, or fewer for one warp per row: wider rows then go through
// the stage in segments of STG columns, read twice, the second time from L2;
// a smaller stage lets more warps share an SM).  A block of four warps holds
// 4 / WPR row groups; a group walks its rows in batches of up to 32.
template <class K, int MAXNCH, int WPR, int STG = MAXNCH>
__global__ void __launch_bounds__(kTowerThreads, 8) row_sampler_kernel(const Params p) {
  using SW = SortWord<K>;
  using T = typename SW::T;
  using LN = Lane<K>;
  using Acc = typename LN::Acc;
  constexpr int EPC = K::kPerChunk;
  constexpr int RPB = kTowerWarps / WPR;
  constexpr int NCHW = (MAXNCH + WPR - 1) / WPR;          // chunk columns per warp
  constexpr int CPM = LN::kChunksPerMap;
  constexpr int AW = acc_words<K>();
  constexpr bool kSeg = STG < MAXNCH;
  constexpr int NSEG = MAXNCH / STG;
  constexpr int NCC = kSeg ? STG : NCHW;  // chunk columns a warp folds per segment
  constexpr int LG = NCC < 4 ? NCC : 4;   // chunks loaded together
  static_assert(!kSeg || (WPR == 1 && MAXNCH % STG == 0 && STG % CPM == 0),
                "segments: one warp per row, whole map words per segment");
  __shared__ __align__(16) TowerShared<K, STG, WPR> shared_rows[RPB];
  // each warp's copy of its batch's row parameters (lane i: the i-th row)
  __shared__ __align__(16) RowParams batch_rows[kTowerWarps][32];
  const int warp = static_cast<int>(threadIdx.x) >> 5;
  const int grp = warp / WPR, sub = warp % WPR;
  const uint32_t lane = lane_id();
  TowerShared<K, STG, WPR> &sh = shared_rows[grp];
  const int64_t total = static_cast<int64_t>(p.n_rows) * p.n_steps;
  const int64_t n_groups = static_cast<int64_t>(gridDim.x) * RPB;
  pdl_wait_and_release();

  // a second step array: each thread stores the advanced step of at most one
  // stream, its load sent out with the first batch's parameter loads
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  bool next_due = p.step_next != nullptr && gtid < p.n_streams;
  const int64_t next_v = next_due ? p.step[gtid] : 0;

  int seen_step = -1;      // last step whose ready flag this warp has checked
  bool step_ok = true;     // that step's flag was seen set
  bool gave_up = false;    // a flag did not come in time: later flags get one look
  bool first_row = true;
  // batches of B consecutive rows (B <= 32, about the rows per group): batch
  // k covers rows [k B, k B + B), and group g takes batches g, g + G, ...
  // Consecutive rows mix a frame's codebooks, so the groups' loads match
  const int64_t per_group = (total + n_groups - 1) / n_groups;
  const int bsz = per_group < 32 ? static_cast<int>(per_group) : 32;
#pragma unroll 1
  for (int64_t base = (static_cast<int64_t>(blockIdx.x) * RPB + grp) * bsz; base < total;
       base += n_groups * bsz) {
    const int nb = total - base < bsz ? static_cast<int>(total - base) : bsz;
    // lane i: the parameters of the batch's i-th row
    RowParams *rows = batch_rows[warp];
    // every warp of a group loads its own copy: no barrier before the rows
    if (static_cast<int>(lane) < nb) rows[lane] = load_params(p, base + lane);
    __syncwarp();
    if (next_due) {
      p.step_next[gtid] = next_v + p.n_steps;
      next_due = false;
    }
    bool drawn = false;
#pragma unroll 1
    for (int i = 0; i < nb; ++i) {
      const uint32_t meta = rows[i].meta;
      const int wstep = rows[i].s;
      // a group sharing a row: the previous row's readers of the stage and
      // the candidate words are done before they are overwritten
      if (WPR > 1 && !first_row) row_sync<WPR>(grp);
      first_row = false;
      uint32_t err = meta_err(meta);
      if (!err && p.ready) {
        // warp 0 waits for the step's flag and tells the group (every warp
        // of the group takes this branch for the same rows).  After its
        // first flag that did not come in time, a group only looks at the
        // later steps' flags once, without waiting.
        if (wstep != seen_step) {
          seen_step = wstep;
          if (sub == 0) {
            const bool ok = wait_ready(p.ready + wstep, gave_up ? 0ull : p.ready_timeout_ns);
            if (lane == 0) sh.xready = ok ? 1u : 0u;
          }
          row_sync<WPR>(grp);
          step_ok = sh.xready != 0u;
          gave_up |= !step_ok;
        }
        if (!step_ok) err = kRowNotReady;
      }
      // ---- this warp's columns into the stage, all copies in flight ----
      const int V = meta_vocab(meta);
      const int64_t woff = rows[i].off;
      const char *rowp = static_cast<const char *>(p.logits) + woff * K::kElemBytes;
      const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
      int head = static_cast<int>(((16u - (addr & 15u)) & 15u) / K::kElemBytes);
      head = min(head, V);
      const int nq = err ? 0 : (V - head) / EPC;
      const int tail = V - head - nq * EPC;
      const int nch = min((nq + 31) >> 5, MAXNCH);
      const char *body = rowp + head * K::kElemBytes;
      // this warp's column c is chunk column j = sub + c WPR of the row,
      // chunk q = lane + 32 j, held in stage slot lane + 32 (j mod STG)
      const auto issue = [&](int seg) {
#pragma unroll
        for (int cc = 0; cc < (kSeg ? STG : NCHW); ++cc) {
          const int c = seg * STG + cc;
          const int j = sub + c * WPR;
          if (j >= nch) break;  // uniform: narrower rows leave the unrolled loop early
          const int q = static_cast<int>(lane) + 32 * j;
          if (q < nq)
            cp_async16(&sh.stage[lane + 32 * (j % STG)], body + static_cast<size_t>(q) * 16);
        }
      };
      if (!err) issue(0);
      // the batch's draws, while the first row's copies are in flight: lane
      // i of the group's last warp draws for the batch's i-th row
      if (!drawn) {
        drawn = true;
        if (sub == WPR - 1) {
          uint32_t u24 = 0;
          if (static_cast<int>(lane) < nb) {
            const RowParams &mine = rows[lane];
            if (!meta_err(mine.meta) && !meta_fin(mine.meta) && !meta_greedy(mine.meta)) {
              const int r = mine.r;
              const int64_t t = (p.stop_step || p.max_steps) ? mine.t : p.step[mine.stream] + mine.s;
              u24 = philox_u24(p.seed[r], p.request[r], static_cast<uint64_t>(t),
                               static_cast<uint64_t>(static_cast<int64_t>(p.codebook[r])));
            }
          }
          sh.xu[lane] = u24;
        }
      }
      if (err) {
        const int wr = rows[i].r;
        if (sub == 0 && lane == 0)
          row_outputs(p, wr, static_cast<int64_t>(wstep) * p.out_step_stride + wr, -1, -1, -1, err);
        continue;
      }
      if (meta_fin(meta)) {  // a finished stream: no draw
        const RowParams &rp = rows[i];
        if (sub == 0 && lane == 0)
          row_padded(p, rp.r, static_cast<int64_t>(wstep) * p.out_step_stride + rp.r, rp.slot,
                     rp.stream, meta_fin(meta));
        continue;
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
      uint32_t ebits = has_e ? K::load_one(rowp, eidx) : 0u;
      // the row's penalty and history column (lane j: the frame in slot j),
      // fetched while the row's logits arrive
      float pen = 1.0f;
      int hx = -1;
      if (p.hist_ring) {
        const int rr = rows[i].r;
        pen = p.rep_penalty[rr];
        if (sub == 0 && static_cast<int>(lane) < p.hist_len)
          hx = p.hist_ring[(static_cast<int64_t>(rows[i].stream) * p.hist_len + lane) * p.hist_q +
                           p.codebook[rr]];
      }
      cp_async_wait_all();
      __syncwarp();
      // ---- the repetition penalty over the row's history column ----
      if (p.hist_ring) {
        if (pen != 1.0f) {
          if constexpr (WPR > 1) row_sync<WPR>(grp);  // every warp's columns are staged
          if (sub == 0) {
            const int x = hx;
            const bool valid = x >= 0 && x < V;
            // one lane per distinct token penalises it
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, valid ? x : -1 - static_cast<int>(lane));
            if (valid && __ffs(peers) - 1 == static_cast<int>(lane) && x >= head &&
                x < head + nq * EPC) {
              const int q = (x - head) / EPC, e = (x - head) % EPC;
              const int idx = ((q & 31) + 32 * ((q >> 5) % STG)) * EPC + e;
              if (K::kElemBytes == 2) {
                uint16_t *el = reinterpret_cast<uint16_t *>(sh.stage) + idx;
                *el = static_cast<uint16_t>(penalised_bits<K>(*el, pen));
              } else {
                uint32_t *el = reinterpret_cast<uint32_t *>(sh.stage) + idx;
                *el = penalised_bits<K>(*el, pen);
              }
            }
            // head / tail elements: their owning lanes look for them
            if (__any_sync(0xFFFFFFFFu, has_e)) {
              bool hit = false;
              for (int j = 0; j < p.hist_len; ++j)
                hit |= __shfl_sync(0xFFFFFFFFu, valid ? x : -1, j) == eidx;
              if (has_e && hit) ebits = penalised_bits<K>(ebits, pen);
            }
          }
          row_sync<WPR>(grp);
        }
      }
      const uint32_t ekey = has_e ? K::key(ebits) : 0u;

      // ---- the two largest logits of each of the lane's two streams ----
      // two independent running pairs (even and odd columns), then merged
      Acc acc = LN::init(), acc_odd = LN::init();
#pragma unroll
      for (int seg = 0; seg < NSEG; ++seg) {
        if (seg > 0) {  // the next segment over the same stage
          if (seg * STG >= nch) break;
          __syncwarp();
          issue(seg);
          cp_async_wait_all();
          __syncwarp();
        }
        // LG chunks at a time: their loads go out together (a stage slot is
        // read whatever the column; a chunk past the row folds as -inf)
#pragma unroll
        for (int c0 = 0; c0 < NCC; c0 += LG) {
          if (sub + (seg * STG + c0) * WPR >= nch) break;  // uniform
          uint4 x[LG];
#pragma unroll
          for (int k = 0; k < LG; ++k)
            x[k] = sh.stage[lane + 32 * ((sub + (seg * STG + c0 + k) * WPR) % STG)];
#pragma unroll
          for (int k = 0; k < LG; ++k) {
            const int c = seg * STG + c0 + k;
            const int j = sub + c * WPR;
            const int q = static_cast<int>(lane) + 32 * j;
            const uint4 v = (c0 + k < NCC && j < nch && q < nq)
                                ? x[k] : make_uint4(LN::kNeutral, LN::kNeutral, LN::kNeutral, LN::kNeutral);
            LN::fold_chunk(v, (c & 1) ? acc_odd : acc);
          }
        }
      }
      if (NCHW > 1) LN::merge(acc, acc_odd);
      if constexpr (WPR > 1) {
        if (sub > 0) LN::store(&sh.xacc[((sub - 1) * 32 + lane) * AW], acc);
        row_sync<WPR>(grp);
      }
      const int kq = meta_keff(meta);
      uint32_t t0 = 0, top = 0;
      bool bad = false;
      if (sub == 0) {
        if constexpr (WPR > 1) {
#pragma unroll
          for (int s2 = 1; s2 < WPR; ++s2) LN::merge(acc, LN::load(&sh.xacc[((s2 - 1) * 32 + lane) * AW]));
        }
        uint32_t sk[4];
        LN::sample_keys(acc, sk);
        // a NaN anywhere in the row reaches a lane's first maxima; +inf
        // (or a positive NaN) is the row's maximum
        const uint32_t ex = has_e ? ekey : 0u;
        bad = __any_sync(0xFFFFFFFFu, LN::has_nan(acc) ||
                                          (has_e && (ekey < K::kNegInf || ekey >= K::kPosInf)));
        uint32_t t1 = max(sk[0], sk[1]), t2 = max(min(sk[0], sk[1]), max(sk[2], sk[3]));
        if (has_e) {
          t2 = max(t2, min(t1, ex));
          t1 = max(t1, ex);
        }
        top = warp_max(t1);
        bad = bad || top >= K::kPosInf;
        if (!bad && top > K::kNegInf) {
          // ---- the k_eff-th largest sample key: a lower bound ----
          // every lane holds >= 1 (>= 2) sample keys >= its t1 (t2): the
          // smallest t1 (t2) over the lanes has >= 32 (64) keys above it
          const uint32_t lo = warp_min(kq <= 32 ? t1 : t2);
          t0 = sample_kth<K>(acc, ex, __any_sync(0xFFFFFFFFu, has_e), kq, lo, top);
        }
        if (lane == 0) sh.xcnt = 0u;  // the row's candidate count
        if constexpr (WPR > 1) {
          if (lane == 0) {
            sh.xt0 = t0;
            sh.xtop = top;
            sh.xbad[0] = bad ? 1u : 0u;
          }
        } else {
          __syncwarp();
        }
      }
      if constexpr (WPR > 1) {
        row_sync<WPR>(grp);
        t0 = sh.xt0;
        top = sh.xtop;
        bad = sh.xbad[0] != 0u;
      }
      if (bad || top <= K::kNegInf) {  // a NaN / +inf, or no finite logit
        if (sub == 0 && lane == 0) {
          const RowParams &rp = rows[i];
          row_outputs(p, rp.r, static_cast<int64_t>(rp.s) * p.out_step_stride + rp.r, -1, -1, -1,
                      kRowNonFinite);
        }
        continue;
      }
      // ---- candidates: the logits >= t0, CPM chunks (32 logits per lane) at
      // a time: the group's map word per lane, a run of slots reserved with
      // one shared atomic, the marked logits written out as sort words (in
      // any order: they are sorted next) ----
      const uint32_t t2 = LN::splat(t0);
      const int ncol = sub < nch ? (nch - sub + WPR - 1) / WPR : 0;  // this warp's columns
      // segments: the one in the stage first, then the others copied again
      const int nseg = kSeg ? (ncol + STG - 1) / STG : 1;
      constexpr int GPS = (kSeg ? STG : NCHW + CPM - 1) / CPM;  // map words per segment
#pragma unroll 1
      for (int k = 0; k < nseg; ++k) {
        const int seg = nseg - 1 - k;
        if (k > 0) {
          __syncwarp();
          issue(seg);
          cp_async_wait_all();
          __syncwarp();
        }
        uint32_t bm[GPS];
#pragma unroll
        for (int g = 0; g < GPS; ++g) bm[g] = 0u;
#pragma unroll
        for (int g = 0; g < GPS; ++g) {
          if (seg * STG + g * CPM >= ncol) break;  // uniform
          // LG chunks at a time, their loads together; a chunk past the row
          // marks nothing
#pragma unroll
          for (int c0 = 0; c0 < CPM; c0 += LG) {
            uint4 x[LG];
#pragma unroll
            for (int k = 0; k < LG; ++k)
              x[k] = sh.stage[lane + 32 * ((sub + (seg * STG + g * CPM + c0 + k) * WPR) % STG)];
#pragma unroll
            for (int k = 0; k < LG; ++k) {
              const int cs = c0 + k;
              const int c = seg * STG + g * CPM + cs;
              const int j = sub + c * WPR;
              const int q = static_cast<int>(lane) + 32 * j;
              const uint32_t fl = LN::flags(x[k], t2, cs);
              bm[g] |= (cs < CPM && c < ncol && q < nq) ? fl : 0u;
            }
          }
        }
        uint32_t mine_n = 0;
#pragma unroll
        for (int g = 0; g < GPS; ++g) mine_n += __popc(bm[g]);
        uint32_t at = mine_n ? atomicAdd(&sh.xcnt, mine_n) : 0u;
        // the lane's marked logits, lowest bit first over its map words taken
        // as two 64-bit words (one loop, as many turns as the lane has marks)
        static_assert(GPS <= 4, "at most four map words per segment");
        uint64_t mlo = bm[0], mhi = 0;
        if constexpr (GPS > 1) mlo |= static_cast<uint64_t>(bm[1]) << 32;
        if constexpr (GPS > 2) mhi = bm[2];
        if constexpr (GPS > 3) mhi |= static_cast<uint64_t>(bm[3]) << 32;
#pragma unroll 1
        for (uint32_t n = 0; n < mine_n; ++n) {
          const bool in_lo = mlo != 0u;
          const uint64_t cur = in_lo ? mlo : mhi;
          const int bit = __ffsll(static_cast<long long>(cur)) - 1 + (in_lo ? 0 : 64);
          if (in_lo)
            mlo &= mlo - 1u;
          else
            mhi &= mhi - 1u;
          int cs, e;
          LN::bit_elem(bit & 31, cs, e);
          const int j = sub + (seg * STG + (bit >> 5) * CPM + cs) * WPR;
          const int q = static_cast<int>(lane) + 32 * j;
          if (at < static_cast<uint32_t>(kWarpCandMax))
            sh.u.cand[at] = SW::make(K::key(K::load_one(sh.stage, (lane + 32 * (j % STG)) * EPC + e)),
                                     static_cast<uint32_t>(head + q * EPC + e));
          ++at;
        }
      }
      if (has_e && ekey >= t0) {
        const uint32_t at = atomicAdd(&sh.xcnt, 1u);
        if (at < static_cast<uint32_t>(kWarpCandMax))
          sh.u.cand[at] = SW::make(ekey, static_cast<uint32_t>(eidx));
      }
      row_sync<WPR>(grp);
      const uint32_t total_n = sh.xcnt;
      const bool over = total_n > static_cast<uint32_t>(kWarpCandMax);
      if (sub != 0) continue;
      const TailParams &tp = rows[i];
      const uint32_t u24 = sh.xu[i];
      int nc = static_cast<int>(total_n);
      if (over) {
        // the row's chunks from the stage, or (segmented) from memory again
        auto keys = [&](int q) {
          const uint4 v = kSeg ? *reinterpret_cast<const uint4 *>(body + static_cast<size_t>(q) * 16)
                               : sh.stage[q];
          return make_uint4(K::key_word(v.x), K::key_word(v.y), K::key_word(v.z), K::key_word(v.w));
        };
        warp_slow_select<K>(V, kq, sh.u.hist, sh.u.cand, keys, nq, head, tail, eidx, ekey);
        nc = kq;
      }
      if (nc <= 32)
        sort_and_tail<K, 1>(p, tp, sh.u.cand, nc, u24);
      else if (nc <= 64)
        sort_and_tail<K, 2>(p, tp, sh.u.cand, nc, u24);
      else
        sort_and_tail_128<K>(p, tp, sh.u.cand, nc, u24);
    }
  }
  if (next_due) p.step_next[gtid] = next_v + p.n_steps;  // a warp without rows
  if (p.step_next) {  // more streams than threads
    const int64_t all = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = gtid + all; i < p.n_streams; i += all) p.step_next[i] = p.step[i] + p.n_steps;
  }
  if (p.step_out) advance_steps_last_block(p);
}

}  // namespace ts
