// ts_sampler.cu -- host side of the C ABI declared in include/ts_sampler.h:
// argument validation, kernel-geometry choice and launches on the caller's
// stream.  Nothing here reads device memory, allocates or synchronises on the
// sampling path, so a decode step can be captured into a CUDA graph (Drama 3
// article, section "两阶段共享一张卡": decode steps replay as one graph, with
// no host synchronisation between steps).
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <type_traits>

#include "../../include/ts_sampler.h"
#include "ts_cluster.cuh"
#include "ts_device.cuh"
#include "ts_lmhead.cuh"
#include "ts_split.cuh"
#include "ts_warp.cuh"
#include "ts_wide.cuh"

struct ts_sampler {
  int device;
  int cap;
  int num_sms;
  int force_path;     // 0 auto, 1 warps per row, 2 CTA/cluster per row, 3 wide cluster, 4 split
  int force_cluster;  // 0 auto, else CTAs per row
  int pdl;            // launch with programmatic stream serialization
  int wide_exact;     // wide path: always take the exact path (testing)
  int force_wpr;      // warp-per-row path: 0 auto, else warps per row (1, 2, 4)
  int fail_launch;    // tests: the split path's launch of this index (2 or 3) fails once
  uint32_t *status;   // device word (first of two: the status word, then the ticket)
  uint32_t *ticket;   // the warp path's fused step advance: blocks done so far
  int occ_warp[2][5][3];  // resident blocks per SM of each warp-path variant
  int occ_seg[2];         // of the segmented 16-column, one-warp-per-row variant
  int occ_seg32;          // of the fp32 32-column variant (16 columns staged at a time)
  void *ws;           // split wide path workspace (ts_reserve), or null
  size_t ws_bytes;
  int ws_rows;        // row records it holds
  int ws_units;       // unit records it holds
  int ws_vocab;       // widest row it was sized for
};

// Scratch of ts_sample_noalloc, for callers that cannot allocate device
// memory: the split path's workspace, after a 256-byte slot that takes the row
// error bits of calls made without a status word.  Every device that loads this
// library holds it until the process exits.  In host code the name stands for
// the array; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TS_NOALLOC_SCRATCH_BYTES];

namespace {

thread_local char g_last_error[256] = "";

ts_status cuda_fail(cudaError_t e, const char *what) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s: %s", what, cudaGetErrorString(e));
  return TS_ERR_CUDA;
}

int cap_of(int requested) {
  if (requested == 0) return 64;
  if (requested < 32 || requested > 4096 || (requested & (requested - 1))) return -1;
  return requested;
}

constexpr int kWarpMaxBF16 = 4096;
constexpr int kWarpMaxF32 = 4096;
// The LM head's tile: vocabulary entries per CTA, pipeline stages and hidden
// elements per stage (the hidden size must be a multiple of it).
constexpr int kLmN = 128;
constexpr int kLmStages = 4;
constexpr int kLmKC = 64;
constexpr int kWarpMaxF32Penalty = 2048;  // rows the penalty edits in one staged pass
// bf16 rows wider than this take a single-pass wide path
constexpr int kWideMinVocab = 32768;
// split path: slices of about this many tokens at most (76 KB of bf16)
constexpr int kSplitSliceTarget = 40000;

// Units (CTAs) per row of the split path for a launch of n_rows rows of at
// most vmax tokens: slices of at most kSplitSliceTarget tokens, at least two
// units, and for few rows enough units to cover the GPU twice.
int split_units(int n_rows, int vmax, int num_sms) {
  int u = (vmax + kSplitSliceTarget - 1) / kSplitSliceTarget;
  u = std::max(u, 2);
  const int spread = (2 * num_sms + std::max(n_rows, 1) - 1) / std::max(n_rows, 1);
  u = std::max(u, std::min(spread, ts::kSplitMaxUnits));
  return std::min(u, ts::kSplitMaxUnits);
}

struct Plan {
  int path;   // 1 warp(s) per row, 2 cluster, 3 wide, 4 split
  int nch;    // warp path: 16-byte chunks per lane
  int wpr;    // warp path: warps per row
  int seg;    // warp path: 1 = the stage holds 8 of 16 columns, 2 = 16 of 32 (fp32)
  int g;      // cluster and wide paths: CTAs per row
  int slice;  // cluster and wide paths: elements per CTA
  int threads;
  int smem;
  int grid;
};

ts_status make_plan(const ts_sampler *s, const ts_batch *b, Plan *pl, int n_steps = 1) {
  const bool bf16 = b->dtype == TS_DTYPE_BF16;
  const int vmax = b->max_row_vocab;
  if (vmax > (bf16 ? TS_MAX_VOCAB_BF16 : TS_MAX_VOCAB_F32)) return TS_ERR_UNSUPPORTED;
  const int warp_max = bf16 ? kWarpMaxBF16 : kWarpMaxF32;
  const bool warp_ok = s->cap <= 64 && vmax <= warp_max;
  const int su = split_units(b->n_rows, vmax, s->num_sms);
  const bool split_ok = bf16 && s->ws && b->n_rows <= s->ws_rows &&
                        static_cast<long long>(b->n_rows) * su <= s->ws_units &&
                        (vmax + su - 1) / su <= ts::kWideSliceMax;
  int path = s->force_path;
  if (!path) path = warp_ok ? 1 : (bf16 && vmax > kWideMinVocab ? (split_ok ? 4 : 3) : 2);
  if (path == 1 && !warp_ok) return TS_ERR_INVALID_ARG;
  if (b->hist_ring && path != 1) return TS_ERR_UNSUPPORTED;  // the penalty is on the warp path
  // the penalty edits the staged row in place: rows staged in two passes
  // (fp32 wider than 2048) would lose the first pass's edits
  if (b->hist_ring && !bf16 && vmax > kWarpMaxF32Penalty) return TS_ERR_UNSUPPORTED;
  if (path == 3 && !bf16) return TS_ERR_INVALID_ARG;
  std::memset(pl, 0, sizeof *pl);
  pl->path = path;
  if (path == 4) {
    int u = s->force_cluster ? s->force_cluster : su;
    if (!bf16 || !s->ws || u < 2 || u > ts::kSplitMaxUnits || b->n_rows > s->ws_rows ||
        static_cast<long long>(b->n_rows) * u > s->ws_units)
      return TS_ERR_INVALID_ARG;
    int slice = (vmax + u - 1) / u;
    slice = (slice + 7) / 8 * 8;
    if (slice > ts::kWideSliceMax) return TS_ERR_UNSUPPORTED;
    pl->g = u;
    pl->slice = slice;
    pl->threads = ts::kSplitThreads;
    pl->smem = static_cast<int>(ts::kStreamSmemBytes);
    pl->grid = b->n_rows * u;
    return TS_OK;
  }
  if (path == 3) {
    int g = 1;
    if (s->force_cluster) {
      g = s->force_cluster;
    } else {
      while ((vmax + g - 1) / g > ts::kWideSliceMax) g *= 2;
      // few rows: spread each row over more SMs
      while (g < 8 && static_cast<long long>(b->n_rows) * g < 2LL * s->num_sms) g *= 2;
    }
    if (g != 1 && g != 2 && g != 4 && g != 8) return TS_ERR_INVALID_ARG;
    int slice = (vmax + g - 1) / g;
    slice = (slice + 7) / 8 * 8;
    if (slice > ts::kWideSliceMax) return TS_ERR_UNSUPPORTED;
    pl->g = g;
    pl->slice = slice;
    pl->threads = ts::kWideThreads;
    pl->smem = static_cast<int>(ts::wide_smem_bytes(g));
    pl->grid = b->n_rows * g;
    return TS_OK;
  }
  if (path == 1) {
    const int epc = bf16 ? 8 : 4;
    const int per_lane = (vmax + 32 * epc - 1) / (32 * epc);  // 16-byte chunks per lane
    pl->nch = per_lane <= 1 ? 1 : per_lane <= 2 ? 2 : per_lane <= 4 ? 4 : per_lane <= 8 ? 8
            : per_lane <= 16 ? 16 : 32;
    // small batches share each row among several warps (a shorter chain per
    // row while the GPU has room); large ones keep one warp per row
    const long long rows = static_cast<long long>(b->n_rows) * n_steps;
    // (measured on the 128 x 10 step: 1 warp per row 9.5 us, 2 10.2 us, 4 12.2 us)
    int wpr = s->force_wpr;
    if (!wpr) wpr = rows <= s->num_sms ? 4 : rows <= 4LL * s->num_sms ? 2 : 1;
    if (pl->nch == 32) wpr = 1;  // fp32 rows wider than 2048: one warp, two staged passes
    const int rpb = ts::kTowerWarps / wpr;
    pl->wpr = wpr;
    pl->g = wpr;
    pl->threads = ts::kTowerThreads;
    pl->smem = 0;  // static shared memory only
    // one row per row group while the grid fits on the GPU at once; beyond
    // that a resident grid whose groups walk several rows each
    const int ni = pl->nch == 1 ? 0 : pl->nch == 2 ? 1 : pl->nch == 4 ? 2 : pl->nch == 8 ? 3 : 4;
    const int occ = pl->nch == 32 ? s->occ_seg32
                                  : s->occ_warp[bf16 ? 1 : 0][ni][wpr == 1 ? 0 : wpr == 2 ? 1 : 2];
    long long resident = static_cast<long long>(s->num_sms) * std::max(occ, 1);
    if (pl->nch == 32) pl->seg = 2;
    // more rows than row groups on the GPU at once: the groups walk several
    // rows each, and the 16-column variant stages 8 columns at a time (half
    // the shared memory, so more warps per SM)
    if (wpr == 1 && pl->nch == 16 && rows > resident * rpb && !b->hist_ring) {
      pl->seg = 1;
      resident = static_cast<long long>(s->num_sms) * std::max(s->occ_seg[bf16 ? 1 : 0], 1);
    }
    pl->grid = static_cast<int>(std::min<long long>((rows + rpb - 1) / rpb, resident));
    return TS_OK;
  }
  const int slice_max = bf16 ? ts::kSliceMaxBF16 : ts::kSliceMaxF32;
  const int epc = bf16 ? 8 : 4;
  int g = 1;
  if (s->force_cluster) {
    g = s->force_cluster;
  } else {
    while ((vmax + g - 1) / g > slice_max) g *= 2;
    // few rows: spread each row over more SMs while slices stay sizeable
    while (g < 8 && static_cast<long long>(b->n_rows) * g * 2 <= s->num_sms &&
           (vmax + 2 * g - 1) / (2 * g) >= 4096)
      g *= 2;
  }
  if (g != 1 && g != 2 && g != 4 && g != 8) return TS_ERR_INVALID_ARG;
  int slice = (vmax + g - 1) / g;
  slice = (slice + epc - 1) / epc * epc;
  if (slice > slice_max) return TS_ERR_UNSUPPORTED;
  const ts::ClusterLayout lay = ts::cluster_layout(slice, s->cap, bf16 ? 2 : 4, epc);
  pl->g = g;
  pl->slice = slice;
  pl->threads = ts::kClusterThreads;
  pl->smem = static_cast<int>(lay.total);
  pl->grid = b->n_rows * g;
  return TS_OK;
}

ts_status check_batch(const ts_batch *b) {
  if (!b) return TS_ERR_INVALID_ARG;
  if (b->n_rows < 0 || b->n_streams < 0 || b->logits_len < 0 || b->feedback_len < 0)
    return TS_ERR_INVALID_ARG;
  if (b->dtype != TS_DTYPE_F32 && b->dtype != TS_DTYPE_BF16) return TS_ERR_INVALID_ARG;
  if (b->n_rows == 0) return TS_OK;
  if (b->max_row_vocab <= 0) return TS_ERR_INVALID_ARG;
  const size_t es = b->dtype == TS_DTYPE_BF16 ? 2 : 4;
  if (!b->logits || reinterpret_cast<uintptr_t>(b->logits) % es) return TS_ERR_INVALID_ARG;
  if (!b->row_vocab || !b->row_offsets || !b->temp || !b->top_k || !b->top_p || !b->seed ||
      !b->request || !b->codebook || !b->row_stream || !b->step || !b->out_ids || !b->out_eos)
    return TS_ERR_INVALID_ARG;
  if (b->n_streams == 0) return TS_ERR_INVALID_ARG;
  if (b->step_out && b->step_out != b->step) {  // a second step array must not overlap the first
    const int64_t *a = b->step, *o = b->step_out;
    if (o < a + b->n_streams && a < o + b->n_streams) return TS_ERR_INVALID_ARG;
  }
  if (b->feedback_buf && !b->feedback_slot) return TS_ERR_INVALID_ARG;
  if (b->hist_ring && (b->hist_len < 1 || b->hist_len > 32 || b->hist_codebooks < 1 ||
                       !b->rep_penalty || !b->codebook))
    return TS_ERR_INVALID_ARG;
  return TS_OK;
}

ts::Params make_params(const ts_sampler *s, const ts_batch *b) {
  ts::Params p;
  std::memset(&p, 0, sizeof p);
  p.logits = b->logits;
  p.logits_len = b->logits_len;
  p.n_rows = b->n_rows;
  p.max_row_vocab = b->max_row_vocab;
  p.row_vocab = b->row_vocab;
  p.row_offsets = b->row_offsets;
  p.temp = b->temp;
  p.top_k = b->top_k;
  p.top_p = b->top_p;
  p.seed = b->seed;
  p.request = b->request;
  p.codebook = b->codebook;
  p.row_stream = b->row_stream;
  p.step = b->step;
  p.n_streams = b->n_streams;
  p.eos_id = b->eos_id;
  p.out_ids = b->out_ids;
  p.out_eos = b->out_eos;
  p.feedback_buf = b->feedback_buf;
  p.feedback_slot = b->feedback_slot;
  p.feedback_len = b->feedback_len;
  p.cap = s->cap;
  p.status = s->status;
  p.n_steps = 1;
  p.out_step_stride = b->n_rows;
  p.stop_step = b->stop_step;
  p.max_steps = b->max_steps;
  p.finish_reason = b->finish_reason;
  p.pad_id = b->pad_id;
  p.hist_ring = b->hist_ring;
  p.hist_len = b->hist_len;
  p.hist_q = b->hist_codebooks;
  p.rep_penalty = b->rep_penalty;
  p.step_next = (b->advance_steps && b->step_out && b->step_out != b->step) ? b->step_out : nullptr;
  return p;
}

template <class K, int WPR>
void *warp_kernel_wpr(int nch) {
  if (nch == 1) return reinterpret_cast<void *>(ts::row_sampler_kernel<K, 1, WPR>);
  if (nch == 2) return reinterpret_cast<void *>(ts::row_sampler_kernel<K, 2, WPR>);
  if (nch == 4) return reinterpret_cast<void *>(ts::row_sampler_kernel<K, 4, WPR>);
  if (nch == 8) return reinterpret_cast<void *>(ts::row_sampler_kernel<K, 8, WPR>);
  return reinterpret_cast<void *>(ts::row_sampler_kernel<K, 16, WPR>);
}

template <class K>
void *warp_kernel_for(int nch, int wpr, int seg = 0) {
  if (seg == 2) {  // fp32 only: 32 columns, 16 staged at a time
    if constexpr (std::is_same<K, ts::KeyF32>::value)
      return reinterpret_cast<void *>(ts::row_sampler_kernel<ts::KeyF32, 32, 1, 16>);
    return nullptr;
  }
  if (seg) return reinterpret_cast<void *>(ts::row_sampler_kernel<K, 16, 1, 8>);
  if (wpr == 4) return warp_kernel_wpr<K, 4>(nch);
  if (wpr == 2) return warp_kernel_wpr<K, 2>(nch);
  return warp_kernel_wpr<K, 1>(nch);
}

void *wide_kernel_for(int g) {
  if (g == 1) return reinterpret_cast<void *>(ts::wide_sampler_kernel<1>);
  if (g == 2) return reinterpret_cast<void *>(ts::wide_sampler_kernel<2>);
  if (g == 4) return reinterpret_cast<void *>(ts::wide_sampler_kernel<4>);
  return reinterpret_cast<void *>(ts::wide_sampler_kernel<8>);
}

template <class K>
void *cluster_kernel_for(int g) {
  if (g == 1) return reinterpret_cast<void *>(ts::cluster_sampler_kernel<K, 1>);
  if (g == 2) return reinterpret_cast<void *>(ts::cluster_sampler_kernel<K, 2>);
  if (g == 4) return reinterpret_cast<void *>(ts::cluster_sampler_kernel<K, 4>);
  return reinterpret_cast<void *>(ts::cluster_sampler_kernel<K, 8>);
}

// Lets every kernel use the device's opt-in shared memory (less what the
// kernel declares statically).  Done once in ts_create, before any capture.
ts_status set_attributes(int device) {
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  void *fns[48];
  int n = 0;
  const int gs[4] = {1, 2, 4, 8};
  for (int i = 0; i < 4; ++i) {
    fns[n++] = cluster_kernel_for<ts::KeyBF16>(gs[i]);
    fns[n++] = cluster_kernel_for<ts::KeyF32>(gs[i]);
    fns[n++] = wide_kernel_for(gs[i]);
  }
  const int nchs[5] = {1, 2, 4, 8, 16};
  const int wprs[3] = {1, 2, 4};
  for (int i = 0; i < 5; ++i) {
    for (int k = 0; k < 3; ++k) {
      fns[n++] = warp_kernel_for<ts::KeyBF16>(nchs[i], wprs[k]);
      fns[n++] = warp_kernel_for<ts::KeyF32>(nchs[i], wprs[k]);
    }
  }
  fns[n++] = reinterpret_cast<void *>(ts::split_stream_kernel);
  fns[n++] = reinterpret_cast<void *>(ts::split_tail_kernel);
  fns[n++] = warp_kernel_for<ts::KeyF32>(32, 1, 2);
  fns[n++] = reinterpret_cast<void *>(ts::lm_head_kernel<kLmN, kLmStages, kLmKC>);
  for (int i = 0; i < n; ++i) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fns[i]);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes");
    const int dyn = optin - static_cast<int>(fa.sharedSizeBytes);
    e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  }
  return TS_OK;
}

// dst[i] = src[i] + by for i < n (dst == src: in place), one thread per stream.
__global__ void advance_steps_kernel(const int64_t *src, int64_t *dst, int32_t n, int64_t by) {
  ts::pdl_wait_and_release();
  const int i = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
  if (i < n) dst[i] = src[i] + by;
}

// step[i] += by for i < n_streams, one thread per stream.
// Resident blocks per SM of every warp-path variant (for grids that walk
// several rows per row group).  Done once in ts_create.
ts_status warp_occupancy(ts_sampler *s) {
  const int nchs[5] = {1, 2, 4, 8, 16};
  const int wprs[3] = {1, 2, 4};
  for (int d = 0; d < 2; ++d) {
    for (int i = 0; i < 5; ++i) {
      for (int k = 0; k < 3; ++k) {
        void *fn = d ? warp_kernel_for<ts::KeyBF16>(nchs[i], wprs[k])
                     : warp_kernel_for<ts::KeyF32>(nchs[i], wprs[k]);
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, ts::kTowerThreads, 0);
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        s->occ_warp[d][i][k] = n;
      }
    }
    int n = 0;
    void *fn = d ? warp_kernel_for<ts::KeyBF16>(16, 1, 1) : warp_kernel_for<ts::KeyF32>(16, 1, 1);
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, ts::kTowerThreads, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    s->occ_seg[d] = n;
  }
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &s->occ_seg32, warp_kernel_for<ts::KeyF32>(32, 1, 2), ts::kTowerThreads, 0);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  return TS_OK;
}

ts_status launch_advance(const int64_t *step, int64_t *dst, int32_t n_streams, int64_t by,
                         cudaStream_t stream) {
  if (n_streams == 0) return TS_OK;
  const int threads = 256;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>((n_streams + threads - 1) / threads));
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, advance_steps_kernel, step, dst, n_streams, by);
  return e == cudaSuccess ? TS_OK : cuda_fail(e, "advance_steps launch");
}

// pdl: launch the sampler's kernels with programmatic dependent launch (the
// sampler's option; ts_lm_head_sample turns it off for the launch that
// follows the head, see there).
ts_status launch(const ts_sampler *s, const ts_batch *b, const ts::Params &base, cudaStream_t st,
                 const Plan &pl, bool pdl);

ts_status launch(const ts_sampler *s, const ts_batch *b, const ts::Params &base, cudaStream_t st,
                 bool pdl) {
  Plan pl;
  ts_status rc = make_plan(s, b, &pl, base.n_steps);
  if (rc != TS_OK) return rc;
  if (b->advance_steps && pl.path != 1) {
    // the other paths advance the steps by one more small launch
    rc = launch(s, b, base, st, pl, pdl);
    if (rc != TS_OK) return rc;
    return launch_advance(b->step, base.step_next ? base.step_next : b->step, b->n_streams,
                          base.n_steps, st);
  }
  return launch(s, b, base, st, pl, pdl);
}

ts_status launch(const ts_sampler *s, const ts_batch *b, const ts::Params &base, cudaStream_t st) {
  return launch(s, b, base, st, s->pdl != 0);
}

ts_status launch(const ts_sampler *s, const ts_batch *b, const ts::Params &base, cudaStream_t st,
                 const Plan &pl, bool pdl) {
  ts::Params p = base;
  p.slice = pl.slice;
  p.wide_exact = s->wide_exact;
  if (pl.path == 1 && b->advance_steps && !p.step_next) {  // in place: the ticket
    p.step_out = b->step;
    p.ticket = s->ticket;
  }
  if (pl.path != 1) p.step_next = nullptr;  // the advance launch writes step_out
  const bool bf16 = b->dtype == TS_DTYPE_BF16;
  if (pl.path == 4) {
    p.workspace = s->ws;
    p.ws_rows = s->ws_rows;
    p.ws_units = s->ws_units;
    p.ws_units_per_row = pl.g;
    // few CTAs: the streaming CTAs compute the threshold themselves
    p.split_inline = static_cast<long long>(b->n_rows) * pl.g <= 2LL * s->num_sms ? 1 : 0;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cfg.stream = st;
    cfg.blockDim = dim3(ts::kSplitThreads);
    cfg.gridDim = dim3(static_cast<unsigned>(b->n_rows));
    void *args[] = {&p};
    // A launch refused after the streaming kernel was queued leaves the row
    // counters that the tail kernel would have cleared non-zero.  The row
    // records are then zeroed on the same stream, so that the next call on
    // this workspace starts from clean counters (no allocation, no sync).
    const auto fail_after_stream = [&](cudaError_t e, const char *what) {
      const ts_status rc = cuda_fail(e, what);
      const size_t bytes = static_cast<size_t>(b->n_rows) * sizeof(ts::SplitRowMeta);
      const cudaError_t e2 = cudaMemsetAsync(s->ws, 0, bytes, st);
      if (e2 != cudaSuccess) cuda_fail(e2, "split workspace reset after a failed launch");
      return rc;
    };
    // the test-only injection of ts_set_option(TS_OPT_FAIL_LAUNCH): the
    // launch is refused before anything is queued for it
    const auto injected = [&](int which) {
      if (s->fail_launch != which) return false;
      const_cast<ts_sampler *>(s)->fail_launch = 0;
      return true;
    };
    cudaError_t e = cudaSuccess;
    if (!p.split_inline) {
      e = cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(ts::split_threshold_kernel), args);
      if (e != cudaSuccess) return cuda_fail(e, "split threshold launch");
    }
    cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
    cfg.dynamicSmemBytes = static_cast<size_t>(pl.smem);
    e = injected(2) ? cudaErrorLaunchOutOfResources
                    : cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(ts::split_stream_kernel),
                                          args);
    // the threshold kernel (if it ran) cleared the counters; nothing is dirty yet
    if (e != cudaSuccess) return cuda_fail(e, "split stream launch");
    cfg.gridDim = dim3(static_cast<unsigned>(b->n_rows));
    cfg.dynamicSmemBytes = ts::kTailSmemBytes;
    e = injected(3) ? cudaErrorLaunchOutOfResources
                    : cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(ts::split_tail_kernel),
                                          args);
    if (e != cudaSuccess) return fail_after_stream(e, "split tail launch");
    return TS_OK;
  }
  void *fn = nullptr;
  if (pl.path == 1) {
    fn = bf16 ? warp_kernel_for<ts::KeyBF16>(pl.nch, pl.wpr, pl.seg)
              : warp_kernel_for<ts::KeyF32>(pl.nch, pl.wpr, pl.seg);
  } else if (pl.path == 3) {
    fn = wide_kernel_for(pl.g);
  } else {
    fn = bf16 ? cluster_kernel_for<ts::KeyBF16>(pl.g) : cluster_kernel_for<ts::KeyF32>(pl.g);
  }
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
  cfg.blockDim = dim3(static_cast<unsigned>(pl.threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(pl.smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  ++na;
  if (pl.path >= 2 && pl.g > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(pl.g);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  void *args[] = {&p};
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return cuda_fail(e, "sampler launch");
  return TS_OK;
}

// ---------------------------------------------------------------------------
// The LM head (ts_lm_head_logits / ts_lm_head_sample)
// ---------------------------------------------------------------------------
ts_status check_lm_head(const ts_lm_head *h, const ts_batch *b) {
  if (!h || !b) return TS_ERR_INVALID_ARG;
  if (b->dtype != TS_DTYPE_F32) return TS_ERR_INVALID_ARG;  // the head writes fp32 logits
  if (h->n_heads < 1 || h->dim < TS_LM_HEAD_DIM_STEP || h->dim > TS_LM_HEAD_MAX_DIM ||
      h->dim % TS_LM_HEAD_DIM_STEP || h->weights_len < 0)
    return TS_ERR_INVALID_ARG;
  if (b->n_rows % h->n_heads) return TS_ERR_INVALID_ARG;
  if (b->n_rows == 0) return TS_OK;
  if (!h->hidden || !h->weights || !h->head_offsets) return TS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(h->hidden) % 16 || reinterpret_cast<uintptr_t>(h->weights) % 16)
    return TS_ERR_INVALID_ARG;
  if (b->max_row_vocab > TS_MAX_VOCAB_F32) return TS_ERR_UNSUPPORTED;
  return TS_OK;
}

ts_status launch_lm_head(const ts_sampler *s, const ts_lm_head *h, const ts_batch *b,
                         cudaStream_t st) {
  using Tile = ts::LmTile<kLmN, kLmStages, kLmKC>;
  static_assert(kLmKC == TS_LM_HEAD_DIM_STEP, "the header's dim rule is the stage depth");
  ts::LmParams p;
  std::memset(&p, 0, sizeof p);
  p.hidden = static_cast<const uint16_t *>(h->hidden);
  p.weights = static_cast<const uint16_t *>(h->weights);
  p.weights_len = h->weights_len;
  p.head_offsets = h->head_offsets;
  p.n_heads = h->n_heads;
  p.dim = h->dim;
  p.n_rows = b->n_rows;
  p.max_row_vocab = b->max_row_vocab;
  p.row_vocab = b->row_vocab;
  p.row_offsets = b->row_offsets;
  p.logits = static_cast<float *>(const_cast<void *>(b->logits));
  p.logits_len = b->logits_len;
  const int streams = b->n_rows / h->n_heads;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>((b->max_row_vocab + kLmN - 1) / kLmN),
                     static_cast<unsigned>(h->n_heads),
                     static_cast<unsigned>((streams + ts::kLmM - 1) / ts::kLmM));
  cfg.blockDim = dim3(ts::kLmThreads);
  cfg.dynamicSmemBytes = Tile::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = s->pdl ? 1 : 0;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, ts::lm_head_kernel<kLmN, kLmStages, kLmKC>, p);
  return e == cudaSuccess ? TS_OK : cuda_fail(e, "LM head launch");
}

// ---------------------------------------------------------------------------
// ts_sample_noalloc: per-device set-up and geometry
// ---------------------------------------------------------------------------
constexpr size_t kNoallocWsOff = 256;  // the workspace follows the status slot
constexpr int kNoallocMaxDevices = 64;
// The scratch holds a fixed layout, the same for every call: row records for
// TS_NOALLOC_MAX_ROWS rows and unit records for that many rows at the most
// units per row, at fixed offsets.  A row's candidate counter therefore sits
// at the same address in every call, and the call that last used it has
// cleared it.
constexpr int kNoallocWsRows = TS_NOALLOC_MAX_ROWS;
constexpr int kNoallocWsUnits = TS_NOALLOC_MAX_ROWS * ts::kSplitMaxUnits;
static_assert(kNoallocWsOff + ts::split_workspace_bytes(kNoallocWsRows, kNoallocWsUnits) <=
                  TS_NOALLOC_SCRATCH_BYTES,
              "the no-alloc scratch must hold the split workspace of its largest call");

struct NoallocDevice {
  void *scratch;  // device address of g_noalloc_scratch; null until set up
  int num_sms;
};

std::mutex g_noalloc_mu;
NoallocDevice g_noalloc_dev[kNoallocMaxDevices];

ts_status noalloc_reject(const char *what) {
  std::snprintf(g_last_error, sizeof g_last_error, "ts_sample_noalloc: %s", what);
  return TS_ERR_UNSUPPORTED;
}

// Once per device, with the device current: the scratch array's address and
// the split kernels' dynamic shared-memory limits (the values ts_create
// sets).  Neither allocates.
ts_status noalloc_setup(int device, NoallocDevice *out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocDevice &d = g_noalloc_dev[device];
  if (!d.scratch) {
    int sms = 0, optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    const void *fns[2] = {reinterpret_cast<const void *>(ts::split_stream_kernel),
                          reinterpret_cast<const void *>(ts::split_tail_kernel)};
    for (const void *fn : fns) {
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, fn);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes");
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               optin - static_cast<int>(fa.sharedSizeBytes));
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    }
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) return cuda_fail(e, "cudaGetSymbolAddress");
    d.num_sms = sms;
    d.scratch = ptr;
  }
  *out = d;
  return TS_OK;
}

}  // namespace

extern "C" {

ts_status ts_create(int device, int max_top_k, ts_sampler **out) {
  if (!out) return TS_ERR_INVALID_ARG;
  *out = nullptr;
  const int cap = cap_of(max_top_k);
  if (cap < 0) return TS_ERR_INVALID_ARG;
  int n_dev = 0;
  cudaError_t e = cudaGetDeviceCount(&n_dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (device < 0 || device >= n_dev) return TS_ERR_INVALID_ARG;
  int prev = 0;
  cudaGetDevice(&prev);
  e = cudaSetDevice(device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  ts_sampler *s = new (std::nothrow) ts_sampler;
  if (!s) {
    cudaSetDevice(prev);
    return TS_ERR_NO_MEMORY;
  }
  s->device = device;
  s->cap = cap;
  s->force_path = 0;
  s->force_cluster = 0;
  s->pdl = 1;
  s->wide_exact = 0;
  s->force_wpr = 0;
  s->fail_launch = 0;
  s->status = nullptr;
  s->ticket = nullptr;
  std::memset(s->occ_warp, 0, sizeof s->occ_warp);
  std::memset(s->occ_seg, 0, sizeof s->occ_seg);
  s->occ_seg32 = 0;
  s->ws = nullptr;
  s->ws_bytes = 0;
  s->ws_rows = 0;
  s->ws_units = 0;
  s->ws_vocab = 0;
  ts_status rc = TS_OK;
  e = cudaDeviceGetAttribute(&s->num_sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) rc = cuda_fail(e, "cudaDeviceGetAttribute");
  if (rc == TS_OK) {
    e = cudaMalloc(reinterpret_cast<void **>(&s->status), 2 * sizeof(uint32_t));
    if (e != cudaSuccess) rc = e == cudaErrorMemoryAllocation ? TS_ERR_NO_MEMORY
                                                              : cuda_fail(e, "cudaMalloc");
  }
  if (rc == TS_OK) {
    s->ticket = s->status + 1;
    e = cudaMemset(s->status, 0, 2 * sizeof(uint32_t));
    if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemset");
  }
  if (rc == TS_OK) rc = set_attributes(device);
  if (rc == TS_OK) rc = warp_occupancy(s);
  cudaSetDevice(prev);
  if (rc != TS_OK) {
    if (s->status) cudaFree(s->status);
    delete s;
    return rc;
  }
  *out = s;
  return TS_OK;
}

ts_status ts_destroy(ts_sampler *s) {
  if (!s) return TS_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(s->device);
  cudaError_t e = cudaFree(s->status);
  if (s->ws) {
    const cudaError_t e2 = cudaFree(s->ws);
    if (e == cudaSuccess) e = e2;
  }
  cudaSetDevice(prev);
  delete s;
  return e == cudaSuccess ? TS_OK : cuda_fail(e, "cudaFree");
}

int32_t ts_max_top_k(const ts_sampler *s) { return s ? s->cap : -1; }

ts_status ts_sample(ts_sampler *s, const ts_batch *b, void *stream) {
  if (!s) return TS_ERR_INVALID_ARG;
  ts_status rc = check_batch(b);
  if (rc != TS_OK || b->n_rows == 0) return rc;
  return launch(s, b, make_params(s, b), static_cast<cudaStream_t>(stream));
}

ts_status ts_lm_head_logits(ts_sampler *s, const ts_lm_head *h, const ts_batch *b, void *stream) {
  if (!s) return TS_ERR_INVALID_ARG;
  ts_status rc = check_batch(b);
  if (rc != TS_OK) return rc;
  rc = check_lm_head(h, b);
  if (rc != TS_OK || b->n_rows == 0) return rc;
  return launch_lm_head(s, h, b, static_cast<cudaStream_t>(stream));
}

ts_status ts_lm_head_sample(ts_sampler *s, const ts_lm_head *h, const ts_batch *b, void *stream) {
  if (!s) return TS_ERR_INVALID_ARG;
  ts_status rc = check_batch(b);
  if (rc != TS_OK) return rc;
  rc = check_lm_head(h, b);
  if (rc != TS_OK || b->n_rows == 0) return rc;
  Plan pl;  // refuse what the sampler would refuse before the head runs
  rc = make_plan(s, b, &pl);
  if (rc != TS_OK) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = launch_lm_head(s, h, b, st);
  if (rc != TS_OK) return rc;
  // The sampler follows without programmatic dependent launch: scheduled
  // early, its blocks would find room only on the SMs that hold one head
  // block (two leave too little shared memory) and run crowded there once
  // the head completes (measured: 28.4 against 26.0 us per qwen3tts frame).
  return launch(s, b, make_params(s, b), st, false);
}

ts_status ts_sample_host(ts_sampler *s, const ts_batch *b, const void *host_logits,
                         int32_t *host_ids, uint8_t *host_eos, void *stream) {
  if (!s || !host_logits || !host_ids || !host_eos) return TS_ERR_INVALID_ARG;
  ts_status rc = check_batch(b);
  if (rc != TS_OK || b->n_rows == 0) return rc;
  Plan pl;  // refuse what the sampler would refuse before anything is queued
  rc = make_plan(s, b, &pl);
  if (rc != TS_OK) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t es = b->dtype == TS_DTYPE_BF16 ? 2 : 4;
  cudaError_t e = cudaMemcpyAsync(const_cast<void *>(b->logits), host_logits,
                                  static_cast<size_t>(b->logits_len) * es,
                                  cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "ts_sample_host: logits copy");
  rc = launch(s, b, make_params(s, b), st);
  if (rc != TS_OK) return rc;
  const size_t n = static_cast<size_t>(b->n_rows);
  e = cudaMemcpyAsync(host_ids, b->out_ids, n * sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "ts_sample_host: ids copy");
  e = cudaMemcpyAsync(host_eos, b->out_eos, n, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "ts_sample_host: EOS flags copy");
  e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? TS_OK : cuda_fail(e, "ts_sample_host: stream wait");
}

ts_status ts_sample_debug(ts_sampler *s, const ts_batch *b, int32_t max_keep, int32_t *kept_ids,
                          float *kept_probs, int32_t *n_kept, int32_t *n_nucleus, void *stream) {
  if (!s || max_keep <= 0 || !kept_ids || !kept_probs || !n_kept || !n_nucleus)
    return TS_ERR_INVALID_ARG;
  ts_status rc = check_batch(b);
  if (rc != TS_OK || b->n_rows == 0) return rc;
  ts::Params p = make_params(s, b);
  p.max_keep = max_keep;
  p.kept_ids = kept_ids;
  p.kept_probs = kept_probs;
  p.n_kept = n_kept;
  p.n_nucleus = n_nucleus;
  return launch(s, b, p, static_cast<cudaStream_t>(stream));
}

ts_status ts_sample_steps(ts_sampler *s, const ts_batch *b, const ts_steps *st, void *stream) {
  if (!s || !st) return TS_ERR_INVALID_ARG;
  ts_status rc = check_batch(b);
  if (rc != TS_OK) return rc;
  constexpr uint64_t kMaxTimeoutNs = 10000000000ull;
  if (st->n_steps < 1 || st->logits_step_stride < 0 || st->out_step_stride < b->n_rows ||
      st->ready_timeout_ns > kMaxTimeoutNs ||
      (b->feedback_buf && st->feedback_step_stride < b->feedback_len))
    return TS_ERR_INVALID_ARG;
  if (b->n_rows == 0) return TS_OK;
  const bool bf16 = b->dtype == TS_DTYPE_BF16;
  if (s->cap > 64 || b->max_row_vocab > (bf16 ? kWarpMaxBF16 : kWarpMaxF32))
    return TS_ERR_UNSUPPORTED;
  // a later step's rows may run before an earlier step's EOS row (or the
  // earlier step's draw into the history): the finished-stream rule and the
  // repetition penalty need one step per call
  if (b->stop_step || b->max_steps || b->hist_ring) return TS_ERR_UNSUPPORTED;
  if (s->force_path != 0 && s->force_path != 1) return TS_ERR_INVALID_ARG;
  ts::Params p = make_params(s, b);
  p.n_steps = st->n_steps;
  p.logits_step_stride = st->logits_step_stride;
  p.out_step_stride = st->out_step_stride;
  p.feedback_step_stride = st->feedback_step_stride;
  p.ready = st->ready;
  p.ready_timeout_ns = st->ready_timeout_ns ? st->ready_timeout_ns : 1000000000ull;
  return launch(s, b, p, static_cast<cudaStream_t>(stream));
}

ts_status ts_reserve(ts_sampler *s, int32_t max_rows, int32_t max_row_vocab) {
  if (!s || max_rows < 0 || max_row_vocab < 0) return TS_ERR_INVALID_ARG;
  if (max_row_vocab > TS_MAX_VOCAB_BF16) return TS_ERR_UNSUPPORTED;
  int units = 0;
  for (int rows = 1; rows <= max_rows; ++rows)
    units = std::max(units, rows * split_units(rows, std::max(max_row_vocab, 1), s->num_sms));
  if (max_rows > 0 && max_rows <= s->ws_rows && units <= s->ws_units) return TS_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaError_t e = cudaSetDevice(s->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  if (s->ws) {
    e = cudaFree(s->ws);
    s->ws = nullptr;
    s->ws_bytes = 0;
    s->ws_rows = 0;
    s->ws_units = 0;
    if (e != cudaSuccess) {
      cudaSetDevice(prev);
      return cuda_fail(e, "cudaFree");
    }
  }
  ts_status rc = TS_OK;
  if (max_rows > 0) {
    const size_t bytes = ts::split_workspace_bytes(max_rows, units);
    e = cudaMalloc(&s->ws, bytes);
    if (e == cudaSuccess) {
      e = cudaMemset(s->ws, 0, bytes);  // the per-row counters start at zero
      if (e != cudaSuccess) {
        cudaFree(s->ws);
        s->ws = nullptr;
        cudaSetDevice(prev);
        return cuda_fail(e, "cudaMemset");
      }
    }
    if (e != cudaSuccess) {
      s->ws = nullptr;
      rc = e == cudaErrorMemoryAllocation ? TS_ERR_NO_MEMORY : cuda_fail(e, "cudaMalloc");
    } else {
      s->ws_bytes = bytes;
      s->ws_rows = max_rows;
      s->ws_units = units;
      s->ws_vocab = max_row_vocab;
    }
  }
  cudaSetDevice(prev);
  return rc;
}

ts_status ts_sample_noalloc(int32_t max_top_k, const ts_batch *b, uint32_t *status,
                            void *stream) {
  const int cap = cap_of(max_top_k);
  if (cap < 0) return TS_ERR_INVALID_ARG;
  ts_status rc = check_batch(b);
  if (rc != TS_OK) return rc;
  if (b->dtype != TS_DTYPE_BF16) return noalloc_reject("bf16 logits only");
  if (b->n_rows > TS_NOALLOC_MAX_ROWS) return noalloc_reject("more than 64 rows");
  if (b->n_rows > 0 && b->max_row_vocab > TS_MAX_VOCAB_BF16)
    return noalloc_reject("max_row_vocab above TS_MAX_VOCAB_BF16");
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (device < 0 || device >= kNoallocMaxDevices) return noalloc_reject("device index above 63");
  NoallocDevice d;
  rc = noalloc_setup(device, &d);
  if (rc != TS_OK || b->n_rows == 0) return rc;

  // The split path's CTAs per row (at most kSplitMaxUnits, which the fixed
  // layout holds for every row).
  const int n = b->n_rows, vmax = b->max_row_vocab;
  const int u = split_units(n, vmax, d.num_sms);

  ts_sampler s;
  std::memset(&s, 0, sizeof s);
  s.device = device;
  s.cap = cap;
  s.num_sms = d.num_sms;
  s.force_path = 4;
  s.force_cluster = u;
  s.pdl = 1;
  s.status = status ? status : static_cast<uint32_t *>(d.scratch);
  s.ws = static_cast<char *>(d.scratch) + kNoallocWsOff;
  s.ws_bytes = TS_NOALLOC_SCRATCH_BYTES - kNoallocWsOff;
  s.ws_rows = kNoallocWsRows;
  s.ws_units = kNoallocWsUnits;
  s.ws_vocab = vmax;
  return launch(&s, b, make_params(&s, b), static_cast<cudaStream_t>(stream));
}

ts_status ts_advance_steps(int64_t *step, int32_t n_streams, void *stream) {
  if (n_streams < 0 || (n_streams > 0 && !step)) return TS_ERR_INVALID_ARG;
  return launch_advance(step, step, n_streams, 1, static_cast<cudaStream_t>(stream));
}

ts_status ts_read_status(ts_sampler *s, uint32_t *bits, void *stream) {
  if (!s || !bits) return TS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, s->status, sizeof host, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(s->status, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "ts_read_status");
  *bits = host;
  return TS_OK;
}

ts_status ts_set_option(ts_sampler *s, int32_t option, int32_t value) {
  if (!s) return TS_ERR_INVALID_ARG;
  if (option == TS_OPT_PATH) {
    if (value < 0 || value > 4) return TS_ERR_INVALID_ARG;
    s->force_path = value;
    return TS_OK;
  }
  if (option == TS_OPT_CLUSTER) {  // paths 2 / 3: 1, 2, 4 or 8; path 4: 2 .. 16 (checked at launch)
    if (value < 0 || value > ts::kSplitMaxUnits) return TS_ERR_INVALID_ARG;
    s->force_cluster = value;
    return TS_OK;
  }
  if (option == TS_OPT_PDL) {
    if (value != 0 && value != 1) return TS_ERR_INVALID_ARG;
    s->pdl = value;
    return TS_OK;
  }
  if (option == TS_OPT_WIDE_EXACT) {
    if (value != 0 && value != 1) return TS_ERR_INVALID_ARG;
    s->wide_exact = value;
    return TS_OK;
  }
  if (option == TS_OPT_WARPS_PER_ROW) {
    if (value != 0 && value != 1 && value != 2 && value != 4) return TS_ERR_INVALID_ARG;
    s->force_wpr = value;
    return TS_OK;
  }
  if (option == TS_OPT_FAIL_LAUNCH) {
    if (value != 0 && value != 2 && value != 3) return TS_ERR_INVALID_ARG;
    s->fail_launch = value;
    return TS_OK;
  }
  return TS_ERR_INVALID_ARG;
}

ts_status ts_plan(const ts_sampler *s, const ts_batch *b, int32_t *path, int32_t *ctas_per_row,
                  int32_t *threads, int32_t *smem_bytes, int32_t *grid) {
  if (!s) return TS_ERR_INVALID_ARG;
  ts_status rc = check_batch(b);
  if (rc != TS_OK) return rc;
  Plan pl;
  rc = make_plan(s, b, &pl);
  if (rc != TS_OK) return rc;
  if (path) *path = pl.path;
  if (ctas_per_row) *ctas_per_row = pl.g;
  if (threads) *threads = pl.threads;
  if (smem_bytes) *smem_bytes = pl.smem;
  if (grid) *grid = pl.grid;
  return TS_OK;
}

const char *ts_status_string(ts_status st) {
  switch (st) {
    case TS_OK: return "ok";
    case TS_ERR_INVALID_ARG: return "invalid argument";
    case TS_ERR_UNSUPPORTED: return "unsupported size";
    case TS_ERR_CUDA: return "CUDA error";
    case TS_ERR_NO_MEMORY: return "out of memory";
  }
  return "unknown status";
}

const char *ts_last_error(void) { return g_last_error; }

}  // extern "C"
