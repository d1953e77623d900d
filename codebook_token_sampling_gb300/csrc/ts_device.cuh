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
  // CTA/cluster path: elements of a row held by one CTA
  int32_t slice;
};

// ---------------------------------------------------------------------------
// Order-preserving keys.  A float's bit pattern becomes an unsigned integer
// whose order is the float order: negative values have every bit flipped,
// non-negative ones only the sign bit.  -inf maps to kNegInf, +inf to kPosInf;
// a NaN maps below kNegInf or above kPosInf.
// ---------------------------------------------------------------------------
struct KeyBF16 {
  static constexpr int kBits = 16;
  static constexpr int kElemBytes = 2;
  static constexpr int kPerChunk = 8;  // elements per 16-byte chunk
  static constexpr uint32_t kNegInf = 0x007Fu;
  static constexpr uint32_t kPosInf = 0xFF80u;
  __device__ __forceinline__ static uint32_t key(uint32_t bits) {
    return bits ^ ((bits & 0x8000u) ? 0xFFFFu : 0x8000u);
  }
  __device__ __forceinline__ static float value(uint32_t k) {
    uint32_t bits = k ^ ((k & 0x8000u) ? 0x8000u : 0xFFFFu);
    return __uint_as_float(bits << 16);
  }
  // Two packed bf16 values -> two packed keys, no branch.
  __device__ __forceinline__ static uint32_t key_word(uint32_t w) {
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
  __device__ __forceinline__ static uint32_t key(uint32_t bits) {
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
// Kept-set weight w = exp((v - m) / T) for v <= m, T > 0.  The argument is
// carried as a float pair (exact difference by two-sum, exact division
// remainder by fma) so that its rounding does not grow with |v - m|:
// exp(x_hi + x_lo) = exp(x_hi) * (1 + x_lo) to first order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float kept_weight(float v, float m, float t) {
  if (v == -INFINITY) return 0.0f;
  const float d = v - m;
  const float bv = d - v;
  const float d_err = (v - (d - bv)) + (-m - bv);
  const float x = __fdiv_rn(d, t);
  const float e = expf(x);
  if (e == 0.0f) return 0.0f;
  const float rem = fmaf(-x, t, d);
  const float x_lo = __fdiv_rn(rem + d_err, t);
  return fmaf(e, x_lo, e);
}

// Fixed-point mass: w * 2^40 rounded to an integer.  Sums of up to 4096
// weights stay below 2^53, so every prefix sum is exact and order-free.
__device__ __forceinline__ uint64_t to_fixed(float w) {
  return __float2ull_rn(w * 1099511627776.0f);
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
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

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

__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void dsmem_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Per-row parameters and the checks shared by both kernel families.
// ---------------------------------------------------------------------------
struct Row {
  int64_t off;
  int32_t vocab;
  int32_t k_eff;
  int32_t stream;
  int32_t slot;
  float temp;
  float top_p;
  uint32_t err;
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
  uint32_t e = 0;
  if (w.vocab <= 0 || w.vocab > p.max_row_vocab || w.off < 0 ||
      w.off > p.logits_len - static_cast<int64_t>(w.vocab))
    e |= kRowBadShape;
  if (w.stream < 0 || w.stream >= p.n_streams) e |= kRowBadShape;
  if (isnan(w.temp) || isinf(w.temp) || isnan(w.top_p)) e |= kRowBadParam;
  if (w.slot >= 0 && static_cast<int64_t>(w.slot) >= p.feedback_len) e |= kRowBadSlot;
  const int32_t tk = p.top_k[r];
  int32_t k = tk > 0 ? tk : w.vocab;
  k = min(k, p.cap);
  k = min(k, w.vocab);
  w.k_eff = k;
  w.greedy = !(w.temp > 0.0f) || k == 1;
  w.err = e;
  return w;
}

__device__ __forceinline__ void finish_row(const Params &p, int r, const Row &w, int32_t id,
                                           uint32_t err) {
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
  const int32_t eos = p.eos_id ? p.eos_id[r] : -1;
  p.out_eos[r] = static_cast<uint8_t>(eos >= 0 && id == eos);
  if (w.slot >= 0) p.feedback_buf[w.slot] = id;
}

}  // namespace ts
