// ts_device.cuh -- device-side building blocks shared by the sampler kernels:
// order-preserving keys, the Philox4x64-10 draw, the kept-set weight in
// fixed point, streaming loads and thread-block-cluster primitives (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ts {

constexpr uint32_t kRowBadShape = 1u;
constexpr uint32_t kRowBadParam = 2u;
constexpr uint32_t kRowNonFinite = 4u;
constexpr uint32_t kRowBadSlot = 8u;
constexpr uint32_t kRowNotReady = 16u;

// Kernel parameters, passed by value (one copy per launch).
struct Params {
  const void *logits;
  int64_t logits_len;
  int32_t n_rows;
  int32_t max_row_vocab;
  const int32_t *row_vocab;
  const int64_t *row_offsets;
  const float *temp;
  const int32_t *top_k;
  const float *top_p;
  const uint64_t *seed;
  const uint64_t *request;
  const int32_t *codebook;
  const int32_t *row_stream;
  const int64_t *step;
  int32_t n_streams;
  const int32_t *eos_id;
  int32_t *out_ids;
  uint8_t *out_eos;
  int32_t *feedback_buf;
  const int32_t *feedback_slot;
  int64_t feedback_len;
  int32_t cap;
  uint32_t *status;
  // diagnostics (kept_ids == nullptr: off)
  int32_t max_keep;
  int32_t *kept_ids;
  float *kept_probs;
  int32_t *n_kept;
  int32_t *n_nucleus;
  // CTA/cluster and wide paths: elements of a row held by one CTA
  int32_t slice;
  // wide path: 1 = always take the exact (re-reading) path (testing)
  int32_t wide_exact;
  // split wide path: the workspace and its layout (row and unit records),
  // and the units (CTAs) of each row in this launch
  void *workspace;
  int32_t ws_rows;
  int32_t ws_units;
  int32_t ws_units_per_row;
  int32_t split_inline;  // split path: the streaming CTAs compute the threshold themselves
  // multi-step launches of the warp path: steps in the launch (1 for one
  // step), the distance from one step's logits / outputs / frame to the
  // next's, per-step ready flags (null: all ready) and how long a warp waits
  // for one (nanoseconds)
  int32_t n_steps;
  int64_t logits_step_stride;
  int64_t out_step_stride;
  int64_t feedback_step_stride;
  const uint32_t *ready;
  uint64_t ready_timeout_ns;
  // step advance fused into the launch: after every block has read step[],
  // the last block to finish (by an atomic ticket) adds n_steps to
  // step_out[0 .. n_streams) and re-arms the ticket; null: no advance
  int64_t *step_out;
  uint32_t *ticket;
  // a second step array (warp path): step_next[i] = step[i] + n_steps for
  // i < n_streams, written by any thread (nothing in the launch reads it);
  // null: none
  int64_t *step_next;
  // finished streams (null: off): the step of a stream's EOS (< 0: none),
  // the length cap on a stream's step, the finish reason per stream (1 stop,
  // 2 length) and the id a finished stream's rows return
  int64_t *stop_step;
  const int64_t *max_steps;
  uint8_t *finish_reason;
  int32_t pad_id;
  // repetition penalty over the frame history (warp path; null ring: off):
  // stream s, codebook q, step t at hist_ring[(s * hist_len + t mod
  // hist_len) * hist_q + q]; the row's penalty theta in rep_penalty
  int32_t *hist_ring;
  int32_t hist_len;
  int32_t hist_q;
  const float *rep_penalty;
};

// The finish rule for a row of a stream at step t: its EOS was drawn at an
// earlier step (1, stop), else t reached its length cap (2, length), else 0.
// Rows of one step that draw EOS record t, which no row of step t reads as
// finished: the rule gives every row of a step the same answer, in any
// order of the rows.
__device__ __forceinline__ uint32_t finish_rule(const Params &p, int32_t stream, int64_t t) {
  if (p.stop_step) {
    const int64_t s = p.stop_step[stream];
    if (s >= 0 && s < t) return 1u;
  }
  if (p.max_steps && t >= p.max_steps[stream]) return 2u;
  return 0u;
}

// ---------------------------------------------------------------------------
// Order-preserving keys.  A float's bit pattern becomes an unsigned integer
// whose order is the float order: negative values have every bit flipped,
// non-negative ones only the sign bit; -0 is first made +0, so that equal
// values always have equal keys (ties then go by token index).  -inf maps to kNegInf, +inf to kPosInf;
// a NaN maps below kNegInf or above kPosInf.
// ---------------------------------------------------------------------------
struct KeyBF16 {
  static constexpr int kBits = 16;
  static constexpr int kElemBytes = 2;
  static constexpr int kPerChunk = 8;  // elements per 16-byte chunk
  static constexpr uint32_t kNegInf = 0x007Fu;
  static constexpr uint32_t kPosInf = 0xFF80u;
  // -0 and +0 are equal values, so -0 takes the key of +0.
  __device__ __forceinline__ static uint32_t key(uint32_t bits) {
    if (bits == 0x8000u) bits = 0u;
    return bits ^ ((bits & 0x8000u) ? 0xFFFFu : 0x8000u);
  }
  __device__ __forceinline__ static float value(uint32_t k) {
    uint32_t bits = k ^ ((k & 0x8000u) ? 0x8000u : 0xFFFFu);
    return __uint_as_float(bits << 16);
  }
  // Two packed bf16 values -> two packed keys, no branch.  A zero half
  // loses its sign first: the mask keeps the sign bit only where the
  // magnitude is non-zero (its sum with 0x7FFF carries into bit 15).
  __device__ __forceinline__ static uint32_t key_word(uint32_t w) {
    const uint32_t mag = w & 0x7FFF7FFFu;
    w &= (mag + 0x7FFF7FFFu) | 0x7FFF7FFFu;
    uint32_t neg = (w >> 15) & 0x00010001u;
    return w ^ ((neg * 0x7FFFu) | 0x80008000u);
  }
  __device__ __forceinline__ static uint32_t elem(const uint32_t (&c)[4], int e) {
    return (c[e >> 1] >> ((e & 1) * 16)) & 0xFFFFu;
  }
  __device__ __forceinline__ static uint32_t load_one(const void *p, int64_t i) {
    return static_cast<const uint16_t *>(p)[i];
  }
};

struct KeyF32 {
  static constexpr int kBits = 32;
  static constexpr int kElemBytes = 4;
  static constexpr int kPerChunk = 4;
  static constexpr uint32_t kNegInf = 0x007FFFFFu;
  static constexpr uint32_t kPosInf = 0xFF800000u;
  // -0 and +0 are equal values, so -0 takes the key of +0.
  __device__ __forceinline__ static uint32_t key(uint32_t bits) {
    if (bits == 0x80000000u) bits = 0u;
    return bits ^ ((bits & 0x80000000u) ? 0xFFFFFFFFu : 0x80000000u);
  }
  __device__ __forceinline__ static float value(uint32_t k) {
    return __uint_as_float(k ^ ((k & 0x80000000u) ? 0x80000000u : 0xFFFFFFFFu));
  }
  __device__ __forceinline__ static uint32_t key_word(uint32_t w) { return key(w); }
  __device__ __forceinline__ static uint32_t elem(const uint32_t (&c)[4], int e) { return c[e]; }
  __device__ __forceinline__ static uint32_t load_one(const void *p, int64_t i) {
    return static_cast<const uint32_t *>(p)[i];
  }
};

// ---------------------------------------------------------------------------
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11): per round, the words at
// positions 0 and 2 are multiplied by the two round multipliers; the high
// halves are XORed with the other two words and the round key, the low
// halves are kept; the key advances by the two Weyl increments.  Returns the
// top 24 bits of output word 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t philox_u24(uint64_t seed, uint64_t request,
                                               uint64_t step, uint64_t codebook) {
  const uint64_t kMul0 = 0xD2E7470EE14C6C93ull, kMul1 = 0xCA5A826395121157ull;
  const uint64_t kWeyl0 = 0x9E3779B97F4A7C15ull, kWeyl1 = 0xBB67AE8584CAA73Bull;
  uint64_t c0 = step, c1 = codebook, c2 = 0, c3 = 0;
  uint64_t k0 = seed, k1 = request;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t hi_a = __umul64hi(kMul0, c0), lo_a = kMul0 * c0;
    const uint64_t hi_b = __umul64hi(kMul1, c2), lo_b = kMul1 * c2;
    c0 = hi_b ^ c1 ^ k0;
    c1 = lo_b;
    c2 = hi_a ^ c3 ^ k1;
    c3 = lo_a;
    k0 += kWeyl0;
    k1 += kWeyl1;
  }
  return static_cast<uint32_t>(c0 >> 40);
}

// ---------------------------------------------------------------------------
// Kept-set weight w = exp((v - m) / T) for v <= m, T > 0 (inv_t = 1 / T).
// The argument is carried as a float pair (exact difference by two-sum, the
// quotient's remainder by fma) so that its rounding does not grow with
// |v - m|: exp(x_hi + x_lo) = exp(x_hi) * (1 + x_lo) to first order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float kept_weight(float v, float m, float t, float inv_t) {
  if (v == -INFINITY) return 0.0f;
  const float d = v - m;
  const float bv = d - v;
  const float d_err = (v - (d - bv)) + (-m - bv);
  const float x = d * inv_t;
  const float e = expf(x);
  if (e == 0.0f) return 0.0f;
  const float rem = fmaf(-x, t, d);
  const float x_lo = (rem + d_err) * inv_t;
  return fmaf(e, x_lo, e);
}

// Fixed-point mass: w * 2^40 rounded to the nearest integer, ties to even,
// for a finite w in [0, 2^23).  Sums of up to 4096 weights <= 1 stay below
// 2^53, so every prefix sum is exact and order-free.  Computed from the IEEE
// fields with integer operations: w = m * 2^(e - 150) for a normal w with
// significand m (24 bits) and biased exponent e, so w * 2^40 = m * 2^sh with
// sh = e - 110; a right shift by s = -sh rounds on the s discarded bits.
__device__ __forceinline__ uint64_t to_fixed(float w) {
  const uint32_t b = __float_as_uint(w);
  const int e = static_cast<int>(b >> 23);
  if (e == 0) return 0ull;  // zero or subnormal: w * 2^40 < 2^-86
  const uint64_t m = (b & 0x7FFFFFu) | 0x800000u;
  const int sh = e - 110;
  if (sh >= 0) return m << sh;
  if (sh < -25) return 0ull;  // below 1/4
  const int s = -sh;          // 1 <= s <= 25
  const uint64_t q = m >> s, rem = m & ((1ull << s) - 1ull), half = 1ull << (s - 1);
  return q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
}

// ceil(p * s) for an fp32 0 < p < 1 and s < 2^53, exact (128-bit product).
// A prefix mass C (an integer) reaches top_p * S exactly when C >= this.
__device__ __forceinline__ uint64_t ceil_mul_p(float p, uint64_t s) {
  const uint32_t bits = __float_as_uint(p);
  const int biased = static_cast<int>((bits >> 23) & 0xFFu);
  uint64_t mant = bits & 0x7FFFFFu;
  int sh;  // p = mant * 2^-sh
  if (biased == 0) {
    sh = 149;
  } else {
    mant |= 0x800000u;
    sh = 150 - biased;
  }
  const uint64_t lo = mant * s, hi = __umul64hi(mant, s);
  if (sh >= 128) return (hi | lo) ? 1ull : 0ull;
  uint64_t q;
  bool rem;
  if (sh >= 64) {
    const int k = sh - 64;
    q = k == 0 ? hi : (hi >> k);
    rem = lo != 0 || (k != 0 && (hi & ((1ull << k) - 1)) != 0);
  } else {  // sh >= 24 here because p < 1
    q = (lo >> sh) | (hi << (64 - sh));
    rem = (lo & ((1ull << sh) - 1)) != 0;
  }
  return q + (rem ? 1ull : 0ull);
}

// floor(u24 * s / 2^24), exact for s < 2^53.
__device__ __forceinline__ uint64_t scale_u24(uint32_t u24, uint64_t s) {
  const uint64_t lo = static_cast<uint64_t>(u24) * s;
  const uint64_t hi = __umul64hi(static_cast<uint64_t>(u24), s);
  return (hi << 40) | (lo >> 24);
}

// ---------------------------------------------------------------------------
// Memory helpers.
// ---------------------------------------------------------------------------
// An L2 policy that evicts the streamed logits first, so that the small
// per-row parameter arrays stay resident from step to step.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// Programmatic dependent launch: the next kernel in the stream may be
// scheduled as soon as every block of this one has started; this kernel in
// turn waits for its predecessor's completion (and memory) before it reads
// anything.  Without a programmatic predecessor the wait returns at once.
// 16-byte asynchronous global -> shared copies (both addresses 16-byte
// aligned) and the wait for all of this thread's copies.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_and_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Thread-block cluster primitives (sm_90+; used with cluster dims (G,1,1)).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void *local, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

// Loads and stores to a peer CTA's shared memory.  They are ordered with
// respect to the cluster barriers (which carry the memory clobber) and do not
// themselves force a wait, so a thread can have several loads in flight.
__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 dsmem_ld_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void dsmem_st_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b));
}

// ---------------------------------------------------------------------------
// Per-row parameters and the checks shared by both kernel families.
// ---------------------------------------------------------------------------
struct Row {
  int64_t off;
  int64_t stepv;  // the stream's step (Philox counter word 0)
  int32_t vocab;
  int32_t k_eff;
  int32_t stream;
  int32_t slot;
  int32_t eos;
  float temp;
  float inv_temp;
  float top_p;
  uint32_t err;
  uint32_t fin;  // finished stream: 1 stop, 2 length (the row draws nothing)
  bool greedy;
};

__device__ __forceinline__ Row load_row(const Params &p, int r) {
  Row w;
  w.vocab = p.row_vocab[r];
  w.off = p.row_offsets[r];
  w.temp = p.temp[r];
  w.top_p = p.top_p[r];
  w.stream = p.row_stream[r];
  w.slot = p.feedback_buf ? p.feedback_slot[r] : -1;
  w.eos = p.eos_id ? p.eos_id[r] : -1;
  uint32_t e = 0;
  if (w.vocab <= 0 || w.vocab > p.max_row_vocab || w.off < 0 ||
      w.off > p.logits_len - static_cast<int64_t>(w.vocab))
    e |= kRowBadShape;
  if (w.stream < 0 || w.stream >= p.n_streams) e |= kRowBadShape;
  if (isnan(w.temp) || isinf(w.temp) || isnan(w.top_p)) e |= kRowBadParam;
  if (w.slot >= 0 && static_cast<int64_t>(w.slot) >= p.feedback_len) e |= kRowBadSlot;
  w.stepv = 0;
  w.fin = 0;
  if (!(e & (kRowBadShape | kRowBadSlot))) {
    w.stepv = p.step[w.stream];
    if (p.stop_step || p.max_steps) {
      w.fin = finish_rule(p, w.stream, w.stepv);
      if (w.fin) e = 0;  // a finished row's logits and parameters are not looked at
    }
  }
  const int32_t tk = p.top_k[r];
  int32_t k = tk > 0 ? tk : w.vocab;
  k = min(k, p.cap);
  k = min(k, w.vocab);
  w.k_eff = k;
  w.greedy = !(w.temp > 0.0f) || k == 1;
  w.inv_temp = w.greedy ? 1.0f : 1.0f / w.temp;
  w.err = e;
  return w;
}

__device__ __forceinline__ void finish_row(const Params &p, int r, const Row &w, int32_t id,
                                           uint32_t err) {
  if (!err && w.fin) {  // a finished stream: the pad id, no EOS flag
    p.out_ids[r] = p.pad_id;
    p.out_eos[r] = 0;
    if (w.slot >= 0) p.feedback_buf[w.slot] = p.pad_id;
    if (p.finish_reason) p.finish_reason[w.stream] = static_cast<uint8_t>(w.fin);
    if (p.kept_ids) {
      p.n_kept[r] = 0;
      p.n_nucleus[r] = 0;
    }
    return;
  }
  if (err) {
    p.out_ids[r] = -1;
    p.out_eos[r] = 0;
    atomicOr(p.status, err);
    if (p.kept_ids) {
      p.n_kept[r] = 0;
      p.n_nucleus[r] = 0;
    }
    return;
  }
  p.out_ids[r] = id;
  const bool eos = w.eos >= 0 && id == w.eos;
  p.out_eos[r] = static_cast<uint8_t>(eos);
  if (w.slot >= 0) p.feedback_buf[w.slot] = id;
  if (eos) {  // the stream stops: its rows pad from the next step on
    if (p.stop_step) p.stop_step[w.stream] = w.stepv;
    if (p.finish_reason) p.finish_reason[w.stream] = 1u;
  }
}

}  // namespace ts
