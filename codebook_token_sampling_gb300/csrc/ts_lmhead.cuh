// ts_lmhead.cuh -- the LM head of a frame's rows, the step before sampling:
// row r (stream r / Q, codebook q = r mod Q) gets the logits
//   l_r[v] = sum_k h_r[k] W_q[v][k],   v < V_r,
// the product of its hidden state (bf16) and its codebook's output head (bf16,
// one row of `dim` elements per vocabulary entry), accumulated in fp32 on the
// tensor cores and stored as fp32 logits for the sampler.  The Qwen3-TTS
// handbook page ("案例一：Qwen3-TTS——三个 stage 与首包延迟", section "拓扑")
// gives the shape: hidden size 1024, 16 codebooks of 2048 entries per frame;
// the Drama 3 article (section "两阶段共享一张卡") has one forward per frame
// produce every codebook's logits, sampled on the device.
//
// One CTA computes a 32-stream x NT-entry tile of one codebook: the head's NT
// rows stream once through an NS-stage cp.async ring (KC hidden elements per
// stage), the tile's 32 hidden states ride along, and four warps each take
// NT / 4 entries with bf16 m16n8k16 MMAs (fp32 accumulators).  At the frame sizes
// of the pages (32 or 128 streams per codebook) the weights dominate the
// bytes, so the kernel is bound by what each SM takes in through L2 (its
// tiles' head rows plus a quarter as much again in hidden states), not by
// the MMAs.
//
// A row whose head does not lie inside the weights (a negative offset, an
// offset that is not a multiple of 8 elements, or fewer than V_r rows left)
// gets NaN logits, which the sampler reports as a non-finite row; a row with a
// shape error (V_r <= 0, V_r > max_row_vocab, logits outside the buffer) is not
// written, and the sampler reports it.
#pragma once

#include "ts_device.cuh"

namespace ts {

constexpr int kLmThreads = 128;            // four warps
constexpr int kLmM = 32;                   // streams of one codebook per CTA

// A tile of NT vocabulary entries (NT / 4 per warp, a multiple of 16) with an
// NS-stage ring of KC hidden elements per stage.  Shared rows are KC + 8
// elements long (a 16-byte pad), so the eight rows of an ldmatrix start 4
// banks apart.
template <int NT, int NS, int KC>
struct LmTile {
  static_assert(NT % 64 == 0 && NS >= 2 && KC % 64 == 0, "tile, ring and stage shapes");
  static constexpr int kPitch = KC + 8;
  static constexpr int kStageA = kLmM * kPitch;  // bf16 elements of hidden states per stage
  static constexpr int kStageB = NT * kPitch;    // of head rows per stage
  static constexpr uint32_t kSmemBytes = NS * (kStageA + kStageB) * 2;
};

struct LmParams {
  const uint16_t *hidden;        // [n_rows][dim] bf16 bits
  const uint16_t *weights;       // bf16 bits; head q: rows of dim elements from head_offsets[q]
  int64_t weights_len;           // elements
  const int64_t *head_offsets;   // [n_heads]
  int32_t n_heads;               // Q: row r uses head r mod Q
  int32_t dim;                   // a multiple of the tile's KC
  int32_t n_rows;                // a multiple of n_heads
  int32_t max_row_vocab;
  const int32_t *row_vocab;
  const int64_t *row_offsets;
  float *logits;
  int64_t logits_len;
};

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Four 8x8 b16 matrices from shared memory: lane i gives the address of row
// i mod 8 of matrix i / 8, and register j receives matrix j's fragment (row
// lane / 4, elements 2 (lane mod 4) and 2 (lane mod 4) + 1).
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const uint16_t *smem_row) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem_row));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a)
               : "memory");
}

// d += a b for a 16x16 bf16 tile of A (row-major), a 16x8 tile of B (column-
// major: eight rows of the head, each 16 hidden elements) and fp32 d.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// grid (ceil(max_row_vocab / NT), Q, ceil(streams / 32)), kLmThreads threads,
// LmTile<NT, NS, KC>::kSmemBytes of dynamic shared memory; dim a multiple of KC.
template <int NT, int NS, int KC>
__global__ void __launch_bounds__(kLmThreads) lm_head_kernel(const LmParams p) {
  using Tile = LmTile<NT, NS, KC>;
  constexpr int kPitch = Tile::kPitch;
  constexpr int kStageA = Tile::kStageA;
  constexpr int kStageB = Tile::kStageB;
  constexpr int kWarpN = NT / 4;       // entries per warp
  constexpr int kTilesN = kWarpN / 8;  // 8-entry MMA tiles per warp (even)
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t *sa = reinterpret_cast<uint16_t *>(smem);
  uint16_t *sb = sa + NS * kStageA;
  __shared__ int64_t tile_off[kLmM];   // the tile's rows: logits offset
  __shared__ int32_t tile_vocab[kLmM]; // and width (0: nothing to write)
  __shared__ int32_t tile_vmax, head_rows;
  __shared__ int64_t head_off;

  const int q = static_cast<int>(blockIdx.y);
  const int v0 = static_cast<int>(blockIdx.x) * NT;
  const int s0 = static_cast<int>(blockIdx.z) * kLmM;
  const int t = static_cast<int>(threadIdx.x);
  const int lane = t & 31, warp = t >> 5;
  const int n_streams = p.n_rows / p.n_heads;
  pdl_wait_and_release();

  if (warp == 0) {
    const int s = s0 + lane;
    int32_t vr = 0;
    int64_t off = -1;
    if (s < n_streams) {
      const int64_t r = static_cast<int64_t>(s) * p.n_heads + q;
      vr = p.row_vocab[r];
      off = p.row_offsets[r];
      if (vr <= 0 || vr > p.max_row_vocab || off < 0 || off > p.logits_len - vr) {
        vr = 0;
        off = -1;
      }
    }
    tile_vocab[lane] = vr;
    tile_off[lane] = off;
    const int vmax = __reduce_max_sync(0xFFFFFFFFu, vr);
    if (lane == 0) {
      tile_vmax = vmax;
      // the head's rows inside the weights (none for a negative or misaligned offset)
      const int64_t ho = p.head_offsets[q];
      int64_t rows = 0;
      if (ho >= 0 && (ho & 7) == 0 && ho <= p.weights_len) rows = (p.weights_len - ho) / p.dim;
      head_rows = static_cast<int32_t>(rows < p.max_row_vocab ? rows : p.max_row_vocab);
      head_off = ho;
    }
  }
  __syncthreads();
  if (v0 >= tile_vmax) return;  // the whole CTA: no row of the tile reaches this far
  const int wrows = head_rows;
  const int g = lane >> 2, tg = lane & 3;

  if (wrows <= 0) {  // no row of this head lies inside the weights
    for (int i = t >> 5; i < kLmM; i += kLmThreads / 32) {
      const int vr = tile_vocab[i];
      for (int v = v0 + lane; v < vr && v < v0 + NT; v += 32)
        p.logits[tile_off[i] + v] = __int_as_float(0x7FC00000);
    }
    return;
  }

  // ---- the ring: stage st holds hidden elements [KC kc, KC kc + KC) of the
  // tile's 32 hidden states and of its NT head rows (rows past the tile's
  // streams or the head's rows repeat the last one; their results are not
  // stored) ----
  const uint16_t *wbase = p.weights + head_off;
  const int nk = p.dim / KC;
  auto load_stage = [&](int kc, int st) {
    uint16_t *a = sa + st * kStageA;
    uint16_t *b = sb + st * kStageB;
    const int k0 = kc * KC;
#pragma unroll
    for (int j = 0; j < (kLmM * KC / 8) / kLmThreads; ++j) {
      const int c = t + kLmThreads * j;
      const int i = c / (KC / 8), part = c % (KC / 8);
      const int s = min(s0 + i, n_streams - 1);
      const uint16_t *src =
          p.hidden + (static_cast<int64_t>(s) * p.n_heads + q) * p.dim + k0 + part * 8;
      cp_async16(a + i * kPitch + part * 8, src);
    }
#pragma unroll
    for (int j = 0; j < (NT * KC / 8) / kLmThreads; ++j) {
      const int c = t + kLmThreads * j;
      const int i = c / (KC / 8), part = c % (KC / 8);
      const int v = min(v0 + i, wrows - 1);
      cp_async16(b + i * kPitch + part * 8,
                 wbase + static_cast<int64_t>(v) * p.dim + k0 + part * 8);
    }
  };

#pragma unroll
  for (int st = 0; st < NS - 1; ++st) {
    if (st < nk) load_stage(st, st);
    cp_async_commit();
  }
  float acc[2][kTilesN][4];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int n = 0; n < kTilesN; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[m][n][e] = 0.0f;

#pragma unroll 1
  for (int kc = 0; kc < nk; ++kc) {
    cp_async_wait_group<NS - 2>();  // this thread's copies of stage kc are in
    __syncthreads();  // everyone's are, and stage kc - 1 is no longer read
    const int nxt = kc + NS - 1;
    if (nxt < nk) load_stage(nxt, nxt % NS);
    cp_async_commit();
    const uint16_t *a = sa + (kc % NS) * kStageA;
    const uint16_t *b = sb + (kc % NS) * kStageB;
#pragma unroll
    for (int kk = 0; kk < KC / 16; ++kk) {
      // A: matrices (rows 0-7 | 8-15) x (k 0-7 | 8-15) of each 16-row tile
      uint32_t af[2][4];
#pragma unroll
      for (int m = 0; m < 2; ++m)
        ldmatrix_x4(af[m], a + (m * 16 + (lane & 15)) * kPitch + kk * 16 + (lane >> 4) * 8);
      // B: for each pair of 8-entry tiles, (tile 0 | tile 1) x (k 0-7 | 8-15)
      uint32_t bf[kTilesN][2];
#pragma unroll
      for (int pr = 0; pr < kTilesN / 2; ++pr) {
        uint32_t r4[4];
        const int n = warp * kWarpN + pr * 16 + ((lane >> 4) << 3) + (lane & 7);
        ldmatrix_x4(r4, b + n * kPitch + kk * 16 + (((lane >> 3) & 1) << 3));
        bf[2 * pr][0] = r4[0];
        bf[2 * pr][1] = r4[1];
        bf[2 * pr + 1][0] = r4[2];
        bf[2 * pr + 1][1] = r4[3];
      }
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < kTilesN; ++n) mma_bf16_16816(acc[m][n], af[m], bf[n][0], bf[n][1]);
    }
  }
  cp_async_wait_group<0>();  // the trailing (empty) groups

  // ---- the tile's logits: accumulator (m, n, 2 h + e) is stream s0 + 16 m +
  // g + 8 h, entry v0 + (NT / 4) warp + 8 n + 2 tg + e ----
#pragma unroll
  for (int m = 0; m < 2; ++m) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = m * 16 + g + 8 * h;
      const int vr = tile_vocab[i];
      const int64_t off = tile_off[i];
      const bool inside = vr <= wrows;
#pragma unroll
      for (int n = 0; n < kTilesN; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int v = v0 + warp * kWarpN + n * 8 + 2 * tg + e;
          if (v < vr) p.logits[off + v] = inside ? acc[m][n][2 * h + e] : __int_as_float(0x7FC00000);
        }
      }
    }
  }
}

}  // namespace ts
