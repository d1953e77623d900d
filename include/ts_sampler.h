/*
 * ts_sampler.h -- C ABI of the GB300 (sm_103a) per-step multi-codebook token
 * sampler.
 *
 * One call samples every row of one decode step: each (stream, codebook)
 * pair of the batch is a row of logits, and each row gets one token drawn by
 * temperature -> top-k -> top-p sampling, an EOS flag, and an optional
 * write-back of the token into the frame buffer that the next step reads.
 *
 * Sources (page title, section):
 *  - "vLLM-Omni 宣布支持 Fish Audio Drama 3 ..." (AREX article), section
 *    "两阶段共享一张卡": one forward per frame for the whole batch, the
 *    backbone sampling the main codebook and the codebook tower the rest,
 *    top-k / top-p sampling fused on the device with no host synchronisation
 *    between steps, decode steps replayed as one CUDA graph.
 *  - same article, section "测试口径": temperature 1.0, top_p 0.9, top_k 30.
 *  - same article, section "能跑通的命令，和文档写明的边界": top_k is capped at
 *    64 by default and the cap may be set to any power of two in [32, 4096].
 *  - "案例一：Qwen3-TTS——三个 stage 与首包延迟" (AI-infra handbook), section
 *    "第二站：TTS 引擎": the whole frame of codes is written back into a
 *    buffer as the next step's input; section "拓扑": codec EOS id 2150.
 *  - same page, section "一个真实问题：说完了却停不下来": an EOS at p ~ 1e-14
 *    ranked outside the top-k set is never sampled.
 *
 * Semantics where the pages are silent (the plainest reading):
 *  - selection is on the raw logits; ties go to the lower token index;
 *  - k_eff = min(top_k > 0 ? top_k : V, cap, V); top_k above the cap is
 *    clamped, not rejected;
 *  - temperature only shapes probabilities: w_j = exp((l_j - l_max) / T) over
 *    the top-k set; T <= 0 or k_eff == 1 is greedy (first sorted token);
 *  - nucleus = smallest prefix of the top-k set, in (logit desc, index asc)
 *    order, whose renormalised mass reaches top_p (at least one token);
 *    top_p >= 1 keeps all k_eff, top_p <= 0 keeps one;
 *  - draw: u = (x0 >> 40) * 2^-24 with x0 the first word of
 *    Philox4x64-10(counter = (step, codebook, 0, 0), key = (seed, request))
 *    (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC'11);
 *    the token is the first nucleus position whose cumulative mass exceeds
 *    u times the nucleus mass.  Masses are summed in 2^-40 fixed point, so a
 *    result never depends on thread, block or cluster geometry.
 *
 * Every pointer in ts_batch is a DEVICE pointer owned by the caller and must
 * stay valid until the work queued on `stream` has run.  The library never
 * allocates, frees or synchronises inside ts_sample / ts_sample_debug /
 * ts_sample_steps / ts_advance_steps, so those calls may be captured into a
 * CUDA graph.  They
 * run on the device that is current when they are called, which must be the
 * device the sampler was created on.
 */
#ifndef TS_SAMPLER_H
#define TS_SAMPLER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TS_OK = 0,
  TS_ERR_INVALID_ARG = 1,  /* bad pointer, size, dtype, cap or option */
  TS_ERR_UNSUPPORTED = 2,  /* max_row_vocab beyond what the kernels hold */
  TS_ERR_CUDA = 3,         /* a CUDA runtime call failed (see ts_last_error) */
  TS_ERR_NO_MEMORY = 4     /* host or device allocation failed in ts_create */
} ts_status;

typedef enum { TS_DTYPE_F32 = 0, TS_DTYPE_BF16 = 1 } ts_dtype;

/* Per-row error bits.  A row with an error gets out_ids = -1, out_eos = 0
 * and no write-back; the bit is ORed into the sampler's device status word
 * (read with ts_read_status).  The kernels never trap or assert. */
#define TS_ROW_BAD_SHAPE 1u /* V <= 0, V > max_row_vocab, row outside logits_len,
                               or row_stream outside [0, n_streams) */
#define TS_ROW_BAD_PARAM 2u /* temperature NaN or +-inf, or top_p NaN */
#define TS_ROW_NONFINITE 4u /* a NaN or +inf logit, or no finite logit */
#define TS_ROW_BAD_SLOT 8u  /* feedback_slot >= feedback_len */

/* Largest row width each dtype supports (TS_ERR_UNSUPPORTED above it). */
#define TS_MAX_VOCAB_BF16 163840
#define TS_MAX_VOCAB_F32 81920

typedef struct ts_sampler ts_sampler; /* opaque; owns its config and a device status word */

typedef struct {
  /* Packed ragged logits: row r holds row_vocab[r] elements starting at
   * element offset row_offsets[r].  dtype selects fp32 or bf16 (raw bits).
   * `logits` must be aligned to its element size; logits_len is the number
   * of elements the buffer holds (rows reaching past it are errors). */
  const void *logits;
  int32_t dtype;
  int64_t logits_len;
  int32_t n_rows;        /* rows in this call (0 is allowed: nothing runs) */
  int32_t max_row_vocab; /* host-side upper bound on row_vocab[]; picks the
                            kernel geometry (no device read); wider rows
                            are errors */
  const int32_t *row_vocab;   /* [n_rows] */
  const int64_t *row_offsets; /* [n_rows] element offsets */
  const float *temp;          /* [n_rows] temperature */
  const int32_t *top_k;       /* [n_rows] (<= 0: no top-k; clamped to the cap) */
  const float *top_p;         /* [n_rows] */
  const uint64_t *seed;       /* [n_rows] Philox key word 0 */
  const uint64_t *request;    /* [n_rows] Philox key word 1 */
  const int32_t *codebook;    /* [n_rows] Philox counter word 1 */
  const int32_t *row_stream;  /* [n_rows] index into step[] */
  int64_t *step;              /* [n_streams] Philox counter word 0 of the stream's
                                 rows; written only when advance_steps is set */
  int32_t n_streams;
  const int32_t *eos_id;      /* [n_rows] EOS token of the row, -1 = none; may be NULL */
  int32_t *out_ids;           /* [n_rows] sampled token id, -1 on a row error */
  uint8_t *out_eos;           /* [n_rows] 1 if the sampled id is the row's EOS */
  int32_t *feedback_buf;      /* frame buffer of the next step, or NULL (no write-back) */
  const int32_t *feedback_slot; /* [n_rows] slot of the row in feedback_buf,
                                   -1 = none; required when feedback_buf is set */
  int64_t feedback_len;       /* elements in feedback_buf */
  int32_t advance_steps;      /* nonzero: once every row of the call has read its
                                 step, step[i] += 1 for i < n_streams (+= n_steps
                                 for ts_sample_steps), as ts_advance_steps would do
                                 after the call, but inside the call's own launch on
                                 the warp path (its last block to finish does it) and
                                 as one more small launch on the other paths; with
                                 step_out (below) the advanced steps go there */
  /* Finished streams (each pointer may be NULL: no stopping / no length cap /
   * no reasons).  The serving side must report how a request ended, stop at
   * its EOS or length at the generation cap, and cap the generation length
   * ("案例一：Qwen3-TTS——三个 stage 与首包延迟", section "一个真实问题：说完了
   * 却停不下来").  A row of stream s at step t = step[s] is finished when
   * 0 <= stop_step[s] < t (reason 1, stop) or else when t >= max_steps[s]
   * (reason 2, length).  A finished row draws nothing: out_ids = pad_id,
   * out_eos = 0, the frame slot gets pad_id, finish_reason[s] = the reason;
   * its logits and parameters are not read (shape and slot errors still
   * apply).  A row that draws its EOS sets stop_step[s] = t and
   * finish_reason[s] = 1, so the stream's rows pad from step t + 1 on; every
   * row of step t gets the same answer whatever order the rows run in.
   * ts_sample_steps does not take them (TS_ERR_UNSUPPORTED). */
  int64_t *stop_step;         /* [n_streams] step of the stream's EOS, < 0 = running */
  const int64_t *max_steps;   /* [n_streams] length cap on the stream's step */
  uint8_t *finish_reason;     /* [n_streams] 0 running, 1 stop, 2 length */
  int32_t pad_id;             /* id of a finished stream's rows */
  /* Repetition penalty over the fed-back frame history (NULL hist_ring: off).
   * The handbook section above names a repetition penalty among the sampling
   * knobs; the rule is the published one (Keskar et al., "CTRL", 2019): each
   * distinct token of the row's history has its logit divided by theta when
   * positive and multiplied by theta otherwise, before selection, in fp32 and
   * rounded to the logits' type.  The history is a ring [n_streams][hist_len]
   * [hist_codebooks] of token ids: the token of stream s at codebook q drawn
   * at step t sits at ((s * hist_len) + t mod hist_len) * hist_codebooks + q;
   * slots < 0 are empty and ids outside the row are ignored.  A row reads its
   * own column (its stream, its codebook[r]) and, after its draw, writes the
   * drawn id into the slot of its step (finished and error rows write
   * nothing); no two rows of a call share a column.  The caller fills the
   * ring with -1 to start.  Warp path only (top-k cap <= 64, rows up to 4096
   * bf16 / 2048 fp32: a wider fp32 row is staged in two passes and would lose
   * the first pass's edits; others return TS_ERR_UNSUPPORTED), 1 <= hist_len <= 32,
   * not in ts_sample_steps.  Row errors: codebook[r] outside [0,
   * hist_codebooks) is a shape error, theta NaN, infinite or <= 0 a parameter
   * error. */
  int32_t *hist_ring;
  int32_t hist_len;
  int32_t hist_codebooks;
  const float *rep_penalty;   /* [n_rows] theta (1: no penalty) */
  /* Where the advanced steps go when advance_steps is set.  NULL (or step
   * itself): step is advanced in place, which on the warp path needs an
   * acquire-release ticket between the launch's blocks, the last of them
   * storing the steps.  Another array of n_streams entries, not overlapping
   * step: step_out[i] = step[i] + 1 (+ n_steps for ts_sample_steps) for every
   * i < n_streams and step is only read, so no block waits for another; a
   * decode loop alternates the two arrays (step and step_out swapped from
   * one call to the next, e.g. in consecutive calls captured in one CUDA
   * graph).  Overlapping arrays are TS_ERR_INVALID_ARG. */
  int64_t *step_out;
} ts_batch;

/* Creates a sampler on CUDA device `device`.  max_top_k: 0 selects the
 * default cap 64; otherwise a power of two in [32, 4096] (else
 * TS_ERR_INVALID_ARG).  Allocates a 4-byte device status word (besides the
 * workspace of ts_reserve, the only allocation the library makes).  Call it
 * before any stream capture. */
ts_status ts_create(int device, int max_top_k, ts_sampler **out);
/* (The status word shares its 8-byte allocation with the ticket counter that
 * the warp path's fused step advance uses; both start at zero.) */

/* Frees the sampler and its status word.  NULL is accepted. */
ts_status ts_destroy(ts_sampler *s);

/* Effective top-k cap of the sampler (or -1 for NULL). */
int32_t ts_max_top_k(const ts_sampler *s);

/* Samples every row of `b` on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  Asynchronous: it validates the host-side arguments, picks the
 * kernel geometry from max_row_vocab, the cap and dtype, and launches; it
 * reads no device memory and never synchronises.  Host-side errors return a
 * status and launch nothing; per-row errors are reported through the status
 * word. */
ts_status ts_sample(ts_sampler *s, const ts_batch *b, void *stream);

/* ts_sample for logits that are in host memory, end to end in one call: the
 * host's logits_len logits (host_logits, in the batch's dtype and layout) are
 * copied into b->logits (device, caller-owned, writable), the batch is
 * sampled, the n_rows ids and EOS flags are copied back into host_ids and
 * host_eos, and the call waits for `stream` before it returns, so the results
 * can be read at once.  Pinned host memory makes the copies asynchronous DMA
 * on the stream; pageable memory also works, more slowly.  Because it waits,
 * it cannot be captured in a CUDA graph.  Host-side refusals (as for
 * ts_sample, plus a NULL host pointer) are returned before anything is
 * queued; row errors are reported through the status word as for ts_sample. */
ts_status ts_sample_host(ts_sampler *s, const ts_batch *b, const void *host_logits,
                         int32_t *host_ids, uint8_t *host_eos, void *stream);

/* Same draw as ts_sample, and additionally writes, per row r: the top-k set
 * (kept_ids[r * max_keep + j], unspecified order), each kept token's
 * probability renormalised over the top-k set (kept_probs, fp32; greedy rows
 * report 1 for the drawn token and 0 for the rest), n_kept[r] = k_eff and
 * n_nucleus[r] = nucleus size.  Rows with errors get n_kept = n_nucleus = 0.
 * Entries beyond max_keep are not written.  For parity tests and debugging. */
ts_status ts_sample_debug(ts_sampler *s, const ts_batch *b, int32_t max_keep,
                          int32_t *kept_ids, float *kept_probs, int32_t *n_kept,
                          int32_t *n_nucleus, void *stream);

/* Sizes the sampler's workspace for calls of up to max_rows rows no wider
 * than max_row_vocab (bf16).  The workspace lets wide rows (more than 32,768
 * tokens) take the split path: a threshold kernel, a streaming kernel whose
 * CTAs hand their candidates over through it, and a tail kernel with one CTA
 * per row that finishes the row.  Without it (or when a call exceeds it) wide rows take
 * the cluster path, which needs no workspace.  Allocates device memory
 * (32 KB per row plus 16 bytes per CTA of the largest launch), so call it before any stream
 * capture and not concurrently with work on the sampler; 0 rows frees the
 * workspace.  Smaller requests than the current size keep it.  Calls that
 * use the workspace share it: two such calls on one sampler must not
 * overlap on the GPU (order them on one stream or with events). */
ts_status ts_reserve(ts_sampler *s, int32_t max_rows, int32_t max_row_vocab);

/* Scratch size and row limit of ts_sample_noalloc. */
#define TS_NOALLOC_SCRATCH_BYTES 4194304
#define TS_NOALLOC_MAX_ROWS 64

/* The method's sources describe nothing like this call; it exists for callers
 * that cannot allocate device memory.  An engine that reserves almost all of
 * the GPU's memory for weights and KV cache at start-up and hands out memory
 * only from its own pool cannot let a library call cudaMalloc: the call would
 * fail, or take memory the pool does not know about.  cudaFree also waits
 * for the whole device, which stalls every other stream of such an engine.
 * Such callers can use neither ts_create (it allocates the status word) nor
 * ts_reserve (it allocates the workspace).
 *
 * ts_sample_noalloc samples every row of `b` on `stream` exactly as
 * ts_sample on a sampler of cap max_top_k would (the same ids, EOS flags and
 * write-back; results never depend on the kernel geometry).  It runs the
 * split kernels (a threshold kernel, a streaming kernel, then a tail kernel
 * with one CTA per row), and their workspace is a static device array of
 * TS_NOALLOC_SCRATCH_BYTES (4 MiB) inside this library: every GPU that loads
 * the library holds those 4 MiB until the process exits, used or not.  The
 * call allocates nothing and frees nothing, on the host or the device.
 *
 * max_top_k: as in ts_create (0 = 64, else a power of two in [32, 4096]).
 * b: as in ts_sample; bf16 logits only, at most TS_NOALLOC_MAX_ROWS (64) rows,
 *   max_row_vocab <= TS_MAX_VOCAB_BF16.  Larger requests, and fp32 logits,
 *   return TS_ERR_UNSUPPORTED and launch nothing; ts_last_error then names the
 *   limit.  Within them the scratch always suffices.
 * status: a device word owned by the caller; each row error ORs its bits into
 *   it (it is never cleared here).  NULL drops the bits; rows with errors
 *   still get out_ids = -1.
 * stream: a cudaStream_t (NULL = legacy default stream); the call is
 *   asynchronous.
 *
 * Set-up: the first call on a device (the current one) looks up the array's
 * device address and raises the streaming kernel's shared-memory limit on
 * that device; later calls reuse both.  Make that first call, which may have
 * n_rows = 0 and then does only the set-up, before any stream capture.  The
 * set-up is thread-safe; a failure returns TS_ERR_CUDA and is retried by the
 * next call.
 *
 * Sharing: all calls on a device use the one array, which keeps what the last
 * call left in it.  Its layout is fixed, the same for every call whatever its
 * row count: a 256-byte status slot, then 64 row records (16 bytes each),
 * then 1024 unit records (16 bytes each, 16 per row), then 64 candidate
 * arrays of 32 KB, each at a fixed offset (about 2 MiB of the 4 MiB in all).
 * Row r of any call uses row record r, whose candidate counter must be zero
 * when a call starts: the array starts zeroed, and the call that used a
 * counter clears it before it ends (if one of its launches is refused after
 * an earlier one was queued, the call zeroes its rows' records on the stream
 * instead).  Everything else that a call uses it writes before it reads it.
 * Calls whose kernels may overlap on the GPU (on unordered streams, or
 * from several host threads without ordering) race on the array and give
 * wrong results: order them on one stream or with events. */
ts_status ts_sample_noalloc(int32_t max_top_k, const ts_batch *b, uint32_t *status,
                            void *stream);

/* Several decode steps in one launch: ts_sample_steps samples st->n_steps
 * steps of the batch `b` in step order, as that many ts_sample calls would,
 * with step i of the launch (0 <= i < n_steps):
 *   - reading its logits at element offset row_offsets[r] + i *
 *     logits_step_stride of b->logits (rows reaching past logits_len are
 *     errors),
 *   - drawing with Philox counter word 0 = step[row_stream[r]] + i,
 *   - writing out_ids / out_eos at i * out_step_stride + r and its frame at
 *     feedback_buf[i * feedback_step_stride + feedback_slot[r]] (slots are
 *     checked against feedback_len, the length of one frame).
 * With b->advance_steps set, step[] grows by n_steps once the launch is done.
 * It serves callers that queue several steps' logits ahead (their rows are
 * streamed by one persistent grid, so the launch cost is paid once), and
 * producers that finish steps one after another: with `ready` set, the rows
 * of step i wait until ready[i] is nonzero (read with acquire semantics at
 * system scope, so a flag written by the host or by a copy engine after the
 * logits orders them).  A step's rows are sampled exactly when its flag is
 * seen set; otherwise they get out_ids = -1, out_eos = 0, no write-back and
 * the status bit TS_ROW_NOT_READY.  A warp waits at most ready_timeout_ns for
 * a flag (0: one second; at most ten seconds), and after the first flag that
 * has not come by then it looks at later flags only once, so a launch whose
 * flags never come ends within about one limit.  No kernel waits on
 * another kernel: a flag must be set by the host, by a copy, or before the
 * launch.  Only the warp path runs it: top-k cap <= 64, rows of at most 4096
 * bf16 or fp32 logits; anything else returns TS_ERR_UNSUPPORTED.
 * Asynchronous and graph-capturable like ts_sample; ts_sample_debug has no
 * multi-step form. */
#define TS_ROW_NOT_READY 16u
typedef struct {
  int32_t n_steps;               /* >= 1 */
  int64_t logits_step_stride;    /* elements from one step's logits to the next's */
  int64_t out_step_stride;       /* entries from one step's outputs to the next's (>= n_rows) */
  int64_t feedback_step_stride;  /* entries from one step's frame to the next's
                                    (>= feedback_len when feedback_buf is set) */
  const uint32_t *ready;         /* [n_steps] device-visible flags, or NULL: all ready */
  uint64_t ready_timeout_ns;
} ts_steps;
ts_status ts_sample_steps(ts_sampler *s, const ts_batch *b, const ts_steps *st, void *stream);

/* The LM head of a frame's rows, the step before sampling.  The Qwen3-TTS
 * handbook page ("案例一：Qwen3-TTS——三个 stage 与首包延迟", section "拓扑")
 * gives the shape: a hidden size of 1024, 16 codebooks of 2048 entries per
 * frame, each codebook's logits the product of a hidden state and that
 * codebook's output head; the Drama 3 article (section "两阶段共享一张卡")
 * has one forward per frame produce every codebook's logits and sample them
 * on the device with no host synchronisation.
 *
 * Rows are a frame in stream-major order: n_rows = streams x n_heads and row r
 * (stream r / n_heads) uses head q = r mod n_heads.  Row r's logits are
 *   l_r[v] = sum_k hidden[r * dim + k] * weights[head_offsets[q] + v * dim + k]
 * for v < row_vocab[r], bf16 products accumulated in fp32 on the tensor cores
 * (in an order the kernel fixes, so they differ from the exactly rounded sum
 * by a few fp32 roundings), written as fp32 to the batch's logits at
 * row_offsets[r].  Rows of one head may have different widths; head q must
 * then hold as many rows as its widest row.
 *
 * Every pointer is a device pointer owned by the caller.  hidden: [n_rows]
 * [dim] bf16 bits, 16-byte aligned.  weights: bf16 bits, 16-byte aligned,
 * weights_len elements; head q's rows of dim elements start at element
 * head_offsets[q] (a device array of n_heads entries).  dim: a multiple of
 * TS_LM_HEAD_DIM_STEP up to TS_LM_HEAD_MAX_DIM.
 *
 * Errors.  Host side (nothing launched): TS_ERR_INVALID_ARG for a NULL or
 * misaligned pointer, a dim or n_heads outside the rules, n_rows not a
 * multiple of n_heads, or a batch whose dtype is not TS_DTYPE_F32 (the head
 * writes fp32 logits); TS_ERR_UNSUPPORTED for max_row_vocab above
 * TS_MAX_VOCAB_F32.  Per row: a head that does not lie inside the weights
 * (a negative offset, an offset that is not a multiple of 8 elements, or
 * fewer than row_vocab[r] rows before weights_len) gives NaN logits, which
 * sampling reports as TS_ROW_NONFINITE; a row with a shape error (width <= 0
 * or above max_row_vocab, logits outside the buffer) is not written and
 * sampling reports TS_ROW_BAD_SHAPE. */
#define TS_LM_HEAD_DIM_STEP 64
#define TS_LM_HEAD_MAX_DIM 16384
typedef struct {
  const void *hidden;            /* [n_rows][dim] bf16 bits */
  const void *weights;           /* bf16 bits, the heads' rows */
  int64_t weights_len;           /* elements in weights */
  const int64_t *head_offsets;   /* [n_heads] element offset of each head's first row */
  int32_t dim;                   /* hidden size */
  int32_t n_heads;               /* codebooks per frame */
} ts_lm_head;

/* Writes the LM head's fp32 logits into b->logits (which must be writable
 * device memory of logits_len floats) on `stream`; samples nothing.  Only the
 * batch's shape fields are used (n_rows, max_row_vocab, row_vocab,
 * row_offsets, logits, logits_len, dtype), but the batch must pass the checks
 * of ts_sample.  Asynchronous, graph-capturable, no allocation. */
ts_status ts_lm_head_logits(ts_sampler *s, const ts_lm_head *h, const ts_batch *b, void *stream);

/* ts_lm_head_logits, then ts_sample on the same batch, in one call: two
 * launches on `stream`.  The head is launched like the sampler's kernels
 * (programmatic dependent launch unless TS_OPT_PDL is 0); the sampler follows
 * it plainly, so that its blocks are placed once the head's shared memory is
 * free.  The logits (a few MB per frame) go through L2 between the two; a
 * host-side refusal of the sampler is returned before the head launches. */
ts_status ts_lm_head_sample(ts_sampler *s, const ts_lm_head *h, const ts_batch *b, void *stream);

/* step[i] += 1 for i < n_streams, on the device (graph-capturable).  Call it
 * after the step's ts_sample so that sibling rows of one stream share a step
 * (or set ts_batch.advance_steps, which does the same inside the call). */
ts_status ts_advance_steps(int64_t *step, int32_t n_streams, void *stream);

/* Reads the OR of all row error bits since the last read, then clears it.
 * Synchronises `stream`: for tests and debugging, not for the decode loop. */
ts_status ts_read_status(ts_sampler *s, uint32_t *bits, void *stream);

/* Testing / tuning options.  TS_OPT_PATH: 0 = automatic, 1 = one to four
 * warps per row with a bounded candidate set (requires cap <= 64 and
 * max_row_vocab <= 4096; fp32 rows wider than 2048 always take one warp per
 * row), 2 = CTA or cluster per row that
 * holds the row in shared memory, 3 = the single-pass wide-row cluster path
 * (bf16 only; automatic for bf16 rows wider than 32,768 without a
 * workspace), 4 = the split wide-row path (bf16 only; needs ts_reserve;
 * automatic for bf16 rows wider than 32,768 when the workspace fits).
 * TS_OPT_CLUSTER: 0 = automatic, else the CTAs per row of paths 2 and 3 (1,
 * 2, 4 or 8; path 3 needs max_row_vocab / CTAs <= 65,536) or of path 4 (2 ..
 * 16).  TS_OPT_PDL: 1 (default) launches
 * with programmatic dependent launch, so that a step's kernel is scheduled
 * while the previous kernel in the stream drains (each kernel still waits
 * for its predecessor before touching memory); 0 launches plainly.
 * TS_OPT_WIDE_EXACT: 1 makes paths 3 and 4 skip their sampled threshold and
 * always take their exact re-reading select (for tests).
 * TS_OPT_WARPS_PER_ROW: path 1's warps per row, 0 = automatic (4 for calls of
 * up to 1 row per SM, 2 up to 4, else 1), or 1, 2 or 4.  Results never
 * depend on any option. */
#define TS_OPT_PATH 1
#define TS_OPT_CLUSTER 2
#define TS_OPT_PDL 3
#define TS_OPT_WIDE_EXACT 4
#define TS_OPT_WARPS_PER_ROW 5
/* TS_OPT_FAIL_LAUNCH (tests only): 2 or 3 makes the next split-path call
 * refuse its streaming (2) or tail (3) launch on the host, before anything is
 * queued for it, and return TS_ERR_CUDA, as a failed cudaLaunchKernelExC
 * would; 0 disarms it.  When the tail launch fails after the streaming kernel
 * was queued, the call zeroes the rows' workspace records on the stream
 * before it returns, so the next call starts from clean counters. */
#define TS_OPT_FAIL_LAUNCH 6
ts_status ts_set_option(ts_sampler *s, int32_t option, int32_t value);

/* Describes the kernel that ts_sample would launch for `b` (path 1 .. 4,
 * CTAs per row (path 1: warps per row), threads per CTA, dynamic shared
 * memory bytes, grid size).
 * Any output pointer may be NULL. */
ts_status ts_plan(const ts_sampler *s, const ts_batch *b, int32_t *path,
                  int32_t *ctas_per_row, int32_t *threads, int32_t *smem_bytes,
                  int32_t *grid);

/* Static strings; ts_last_error describes the last TS_ERR_CUDA of this thread,
 * or the limit that its last rejected ts_sample_noalloc call exceeded. */
const char *ts_status_string(ts_status st);
const char *ts_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TS_SAMPLER_H */
