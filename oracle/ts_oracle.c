/*
 * ts_oracle.c -- plain, slow CPU oracle for the per-step multi-codebook token
 * sampler.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU
 * baseline leg of the benchmark call it; the product path never does.  It
 * shares no code, header, table or constant generator with the CUDA library.
 *
 * What it computes, per row, written as the plain definition (full sort,
 * explicit fp64 renormalisation, inverse-CDF draw):
 *
 *   sources (the pages this follows, by title and section):
 *   [D3-run]   "vLLM-Omni 宣布支持 Fish Audio Drama 3 ..." (AREX article),
 *              section "两阶段共享一张卡": every request of the batch is sampled
 *              on the device by one fused top-k / top-p step per frame, with
 *              no host synchronisation between steps; the backbone samples
 *              the main codebook and the codebook tower the other nine.
 *   [D3-proto] same article, section "测试口径": serving parameters
 *              temperature 1.0, top_p 0.9, top_k 30, max_new_tokens 500.
 *   [D3-limit] same article, section "能跑通的命令，和文档写明的边界": the fused
 *              kernel caps top_k at 64 by default; the cap can be set to any
 *              power of two from 32 to 4096.
 *   [QT-engine] "案例一：Qwen3-TTS——三个 stage 与首包延迟" (AI-infra handbook),
 *              section "第二站：TTS 引擎": the whole frame of codes is written
 *              back into a buffer as the next step's input.
 *   [QT-eos]   same page, section "一个真实问题：说完了却停不下来": an EOS whose
 *              probability has collapsed to ~1e-14 and ranks outside top-k is
 *              never sampled; the serving side must report how a request
 *              ended (stop at EOS, or length at the generation cap) and cap
 *              the generation length.
 *              The same section names a repetition penalty among the
 *              sampling knobs (it cannot lift the starved EOS either).
 *   [CTRL]     Keskar et al., "CTRL: A Conditional Transformer Language Model
 *              for Controllable Generation", 2019: the repetition penalty
 *              divides a previously generated token's logit by theta when it
 *              is positive and multiplies it by theta otherwise.
 *   [Philox]   Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 *              as 1, 2, 3", SC'11: the Philox4x64 bijection, 10 rounds.
 *   [QT-topo]  "案例一：Qwen3-TTS——三个 stage 与首包延迟", section "拓扑": the
 *              talker's hidden size is 1024 and a frame has 16 codebooks of
 *              2048 entries; the logits each codebook samples from are the
 *              product of a hidden state and that codebook's output head.
 *
 *   Readings where the pages are silent (all listed in the design notes):
 *   order temperature -> top-k -> top-p on the top-k-renormalised mass;
 *   selection on raw logits, ties broken by lower token index; nucleus =
 *   smallest sorted prefix whose mass reaches top_p (at least one token);
 *   CDF walked in sorted order; top_k <= 0 means "no top-k"; top_k above the
 *   cap is clamped; T <= 0 or k_eff = 1 or top_p <= 0 is greedy; the draw is
 *   u = (x0 >> 40) * 2^-24 with x0 the first word of
 *   Philox4x64-10(counter = (step, codebook, 0, 0), key = (seed, request)).
 *
 *   Row errors (the row gets id -1, eos 0, no write-back, and a bit):
 *     bit 0 BAD_SHAPE    V <= 0, V > max_row_vocab, offset out of the
 *                        logits buffer, or row_stream out of [0, n_streams)
 *     bit 1 BAD_PARAM    temperature NaN or +-inf, or top_p NaN
 *     bit 2 NONFINITE    a NaN or +inf logit, or no finite logit at all
 *     bit 3 BAD_SLOT     feedback_slot >= feedback_len (slot < 0 = no write)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_ERR_BAD_SHAPE 1u
#define ORC_ERR_BAD_PARAM 2u
#define ORC_ERR_NONFINITE 4u
#define ORC_ERR_BAD_SLOT 8u

/* ------------------------------------------------------------------------ */
/* Philox4x64-10 [Philox]: two 64x64->128 multiplies per round, the round     */
/* key bumped by the Weyl increments (golden ratio and sqrt(3)-1 in Q0.64).    */
/* ------------------------------------------------------------------------ */
static void mul_64x64(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo) {
  /* schoolbook product on 32-bit halves, kept plain on purpose */
  uint64_t a_lo = a & 0xffffffffu, a_hi = a >> 32;
  uint64_t b_lo = b & 0xffffffffu, b_hi = b >> 32;
  uint64_t p0 = a_lo * b_lo;
  uint64_t p1 = a_lo * b_hi;
  uint64_t p2 = a_hi * b_lo;
  uint64_t p3 = a_hi * b_hi;
  uint64_t mid = (p0 >> 32) + (p1 & 0xffffffffu) + (p2 & 0xffffffffu);
  *lo = (mid << 32) | (p0 & 0xffffffffu);
  *hi = p3 + (p1 >> 32) + (p2 >> 32) + (mid >> 32);
}

void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2],
                          uint64_t out[4]) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
  uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t hi0, lo0, hi1, lo1;
    mul_64x64(M0, x0, &hi0, &lo0);
    mul_64x64(M1, x2, &hi1, &lo1);
    uint64_t y0 = hi1 ^ x1 ^ k0;
    uint64_t y1 = lo1;
    uint64_t y2 = hi0 ^ x3 ^ k1;
    uint64_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    k0 += W0;
    k1 += W1;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The 24-bit uniform integer behind u: u = u24 * 2^-24, u in [0, 1 - 2^-24]. */
uint32_t oracle_uniform24(uint64_t seed, uint64_t request, int64_t step,
                          int32_t codebook) {
  uint64_t ctr[4] = {(uint64_t)step, (uint64_t)(int64_t)codebook, 0, 0};
  uint64_t key[2] = {seed, request};
  uint64_t out[4];
  oracle_philox4x64_10(ctr, key, out);
  return (uint32_t)(out[0] >> 40);
}

/* [D3-limit]: 0 selects the default cap 64; otherwise a power of two in
 * [32, 4096].  Returns the effective cap, or -1 when the value is invalid. */
int oracle_cap(int requested) {
  if (requested == 0) return 64;
  if (requested < 32 || requested > 4096) return -1;
  if ((requested & (requested - 1)) != 0) return -1;
  return requested;
}

/* ------------------------------------------------------------------------ */
/* Row preparation: full sort, renormalisation and nucleus.                  */
/* ------------------------------------------------------------------------ */
typedef struct {
  double value;
  int32_t index;
} orc_entry;

static int cmp_desc_value_asc_index(const void *pa, const void *pb) {
  const orc_entry *a = (const orc_entry *)pa, *b = (const orc_entry *)pb;
  if (a->value > b->value) return -1;
  if (a->value < b->value) return 1;
  return (a->index < b->index) ? -1 : (a->index > b->index);
}

typedef struct {
  int32_t k_eff;    /* size of the top-k set */
  int32_t n_p;      /* size of the nucleus (1 <= n_p <= k_eff) */
  int greedy;       /* 1: the draw is the first sorted token */
  orc_entry *order; /* sorted row, first k_eff entries used */
  double *q;        /* kept-set probabilities, sorted order */
  double s_p;       /* sum of q over the nucleus */
  double margin_cut; /* distance of top_p from the nearest prefix mass */
} orc_row;

static double load_value(int dtype, const void *logits, int64_t pos) {
  if (dtype == 0) return (double)((const float *)logits)[pos];
  if (dtype == 2) return ((const double *)logits)[pos];
  uint16_t b = ((const uint16_t *)logits)[pos];
  uint32_t bits = (uint32_t)b << 16; /* bf16 widens exactly to fp32 */
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static int effective_k(int32_t top_k, int32_t vocab, int32_t cap) {
  int64_t k = top_k > 0 ? top_k : vocab;
  if (k > cap) k = cap;
  if (k > vocab) k = vocab;
  return (int)k;
}

/* bf16 round to nearest even of a float (finite or infinite). */
static float round_to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
  memcpy(&x, &u, sizeof x);
  return x;
}

/* The repetition penalty [CTRL] on one logit, in fp32, the result rounded to
 * the logits' type (bf16 for dtype 1): an in-place update of the row. */
static double penalised(int dtype, double v, float theta) {
  float f = (float)v; /* exact: v came from a bf16 or fp32 value */
  float pen = f > 0.0f ? f / theta : f * theta;
  if (dtype == 1) pen = round_to_bf16(pen);
  return (double)pen;
}

/* Returns error bits (0 = the row is valid and `row` is filled).  `hist`
 * lists the row's distinct previously generated tokens (n_hist of them, each
 * in [0, vocab)), whose logits get the repetition penalty theta first. */
static uint32_t prepare_row(int dtype, const void *logits, int64_t offset,
                            int32_t vocab, float temp, int32_t top_k,
                            float top_p, int32_t cap, orc_entry *scratch,
                            double *qbuf, orc_row *row, const int32_t *hist,
                            int n_hist, float theta) {
  uint32_t err = 0;
  if (isnan(temp) || isinf(temp) || isnan(top_p)) err |= ORC_ERR_BAD_PARAM;
  int any_finite = 0, bad_value = 0;
  for (int32_t i = 0; i < vocab; ++i) {
    double v = load_value(dtype, logits, offset + i);
    if (isnan(v) || v == INFINITY) bad_value = 1;
    if (isfinite(v)) any_finite = 1;
    scratch[i].value = v;
    scratch[i].index = i;
  }
  if (bad_value || !any_finite) err |= ORC_ERR_NONFINITE;
  if (err) return err;
  for (int j = 0; j < n_hist; ++j)
    scratch[hist[j]].value = penalised(dtype, scratch[hist[j]].value, theta);

  /* top-k by a full sort: value descending, lower index first on ties */
  qsort(scratch, (size_t)vocab, sizeof(orc_entry), cmp_desc_value_asc_index);
  int k_eff = effective_k(top_k, vocab, cap);
  row->k_eff = k_eff;
  row->order = scratch;
  row->q = qbuf;
  row->margin_cut = INFINITY;

  if (temp <= 0.0f || k_eff == 1) {
    /* greedy: a point mass on the first sorted token */
    row->greedy = 1;
    for (int j = 0; j < k_eff; ++j) qbuf[j] = (j == 0) ? 1.0 : 0.0;
    row->n_p = 1;
    row->s_p = 1.0;
    return 0;
  }
  row->greedy = 0;

  /* temperature-scaled softmax over the top-k set, renormalised explicitly */
  double m = scratch[0].value;
  double s_k = 0.0;
  for (int j = 0; j < k_eff; ++j) {
    qbuf[j] = exp((scratch[j].value - m) / (double)temp);
    s_k += qbuf[j];
  }
  for (int j = 0; j < k_eff; ++j) qbuf[j] /= s_k;

  /* nucleus: smallest sorted prefix whose mass reaches top_p */
  int n_p;
  if (top_p >= 1.0f) {
    n_p = k_eff;
  } else if (top_p <= 0.0f) {
    n_p = 1;
  } else {
    n_p = k_eff;
    double cum = 0.0;
    for (int n = 1; n <= k_eff; ++n) {
      cum += qbuf[n - 1];
      double d = fabs(cum - (double)top_p);
      if (d < row->margin_cut) row->margin_cut = d;
      if (cum >= (double)top_p) {
        n_p = n;
        break;
      }
    }
    /* the prefix after the stop can be the nearest one too */
    if (n_p < k_eff) {
      double d = fabs(cum + qbuf[n_p] - (double)top_p);
      if (d < row->margin_cut) row->margin_cut = d;
    }
  }
  row->n_p = n_p;
  double s_p = 0.0;
  for (int j = 0; j < n_p; ++j) s_p += qbuf[j];
  row->s_p = s_p;
  return 0;
}

/* Inverse-CDF draw over the nucleus in sorted order; returns the sorted
 * position and, optionally, the distance of u from the nearest CDF step. */
static int draw_row(const orc_row *row, uint32_t u24, double *margin_draw) {
  if (row->greedy) {
    if (margin_draw) *margin_draw = INFINITY;
    return 0;
  }
  double u = (double)u24 * (1.0 / 16777216.0);
  double cum = 0.0, best = INFINITY;
  int pick = -1, last_positive = 0;
  for (int j = 0; j < row->n_p; ++j) {
    cum += row->q[j];
    if (row->q[j] > 0.0) last_positive = j;
    double c = cum / row->s_p;
    double d = fabs(c - u);
    if (d < best) best = d;
    if (pick < 0 && c > u) pick = j;
  }
  if (pick < 0) pick = last_positive; /* rounding fall-through */
  if (margin_draw) *margin_draw = best;
  return pick;
}

/* ------------------------------------------------------------------------ */
/* Batched entry point.                                                      */
/* ------------------------------------------------------------------------ */
typedef struct {
  int64_t n_rows;
  int32_t dtype; /* 0 = fp32, 1 = bf16 (raw bits) */
  const void *logits;
  int64_t logits_len;
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
  int32_t *feedback_buf; /* may be NULL */
  const int32_t *feedback_slot;
  int64_t feedback_len;
  int32_t cap;
  int32_t max_row_vocab;
  const uint32_t *u24_override; /* may be NULL: else replaces the Philox draw */
  int32_t *out_ids;
  uint8_t *out_eos;
  uint32_t *out_err;
  /* optional diagnostics (each may be NULL) */
  int32_t max_keep;
  int32_t *kept_ids;   /* [n_rows, max_keep], sorted order */
  double *kept_probs;  /* [n_rows, max_keep] */
  int32_t *n_kept;     /* [n_rows] */
  int32_t *n_nucleus;  /* [n_rows] */
  double *margin;      /* [n_rows] min distance to a draw or cutoff boundary */
  uint32_t *u24_used;  /* [n_rows] */
  /* finished streams [QT-eos] (each may be NULL: off) */
  int64_t *stop_step;       /* [n_streams] step of the stream's EOS, < 0 = none */
  const int64_t *max_steps; /* [n_streams] length cap on the stream's step */
  uint8_t *finish_reason;   /* [n_streams] 0 running, 1 stop, 2 length */
  int32_t pad_id;           /* id of a finished stream's rows */
  uint8_t *row_finished;    /* [n_rows] scratch: the row's finish reason */
  /* repetition penalty over the frame history ([CTRL]; NULL ring: off):
   * the token of stream s at codebook q drawn at step t sits in
   * hist_ring[(s * hist_len + t % hist_len) * hist_codebooks + q] (< 0:
   * empty); a row penalises the distinct tokens of its column, then writes
   * its own draw into the slot of its step */
  int32_t *hist_ring;
  int32_t hist_len;
  int32_t hist_codebooks;
  const float *rep_penalty; /* [n_rows] theta (1: no penalty) */
} orc_batch;

/* The finish rule [QT-eos], read for a row of stream s at step t:
 * the stream stopped at an earlier step (its EOS was drawn at stop_step[s] <
 * t) -> 1 (stop); else t reached the stream's length cap -> 2 (length);
 * else 0 (the row is sampled).  A finished row draws nothing: it gets the
 * pad id, no EOS flag, and writes the pad id back. */
static int finish_rule(const orc_batch *b, int32_t stream, int64_t t) {
  if (b->stop_step && b->stop_step[stream] >= 0 && b->stop_step[stream] < t) return 1;
  if (b->max_steps && t >= b->max_steps[stream]) return 2;
  return 0;
}

typedef struct {
  const orc_batch *b;
  int64_t row_begin, row_end;
  int32_t width;
} orc_job;

static void run_rows(const orc_batch *b, int64_t r0, int64_t r1, int32_t width) {
  orc_entry *scratch = (orc_entry *)malloc(sizeof(orc_entry) * (size_t)(width > 0 ? width : 1));
  double *qbuf = (double *)malloc(sizeof(double) * (size_t)(width > 0 ? width : 1));
  for (int64_t r = r0; r < r1; ++r) {
    int32_t vocab = b->row_vocab[r];
    int64_t off = b->row_offsets[r];
    uint32_t err = 0;
    if (vocab <= 0 || vocab > b->max_row_vocab || off < 0 ||
        off > b->logits_len - (int64_t)vocab)
      err |= ORC_ERR_BAD_SHAPE;
    int32_t stream = b->row_stream[r];
    if (stream < 0 || stream >= b->n_streams) err |= ORC_ERR_BAD_SHAPE;
    int32_t slot = b->feedback_slot ? b->feedback_slot[r] : -1;
    if (b->feedback_buf && slot >= 0 && (int64_t)slot >= b->feedback_len)
      err |= ORC_ERR_BAD_SLOT;

    orc_row row;
    memset(&row, 0, sizeof row);
    if (b->n_kept) b->n_kept[r] = 0;
    if (b->n_nucleus) b->n_nucleus[r] = 0;
    if (b->margin) b->margin[r] = INFINITY;
    if (b->row_finished) b->row_finished[r] = 0;
    /* a finished stream's row: the pad id, no draw (shape and slot errors
     * still come first; its logits and parameters are not looked at) */
    if (!err) {
      int fin = finish_rule(b, stream, b->step[stream]);
      if (fin) {
        b->out_ids[r] = b->pad_id;
        b->out_eos[r] = 0;
        if (b->out_err) b->out_err[r] = 0;
        if (b->feedback_buf && slot >= 0) b->feedback_buf[slot] = b->pad_id;
        if (b->row_finished) b->row_finished[r] = (uint8_t)fin;
        continue;
      }
    }
    /* the row's distinct history tokens in [0, vocab) and its penalty */
    int32_t hist[64];
    int n_hist = 0;
    float theta = 1.0f;
    int64_t ring_col = -1;
    if (b->hist_ring && !(err & ORC_ERR_BAD_SHAPE)) {
      int32_t q = b->codebook[r];
      theta = b->rep_penalty[r];
      if (q < 0 || q >= b->hist_codebooks) err |= ORC_ERR_BAD_SHAPE;
      if (isnan(theta) || isinf(theta) || !(theta > 0.0f)) err |= ORC_ERR_BAD_PARAM;
      if (!err) {
        ring_col = (int64_t)stream * b->hist_len * b->hist_codebooks + q;
        for (int32_t j = 0; j < b->hist_len; ++j) {
          int32_t x = b->hist_ring[ring_col + (int64_t)j * b->hist_codebooks];
          if (x < 0 || x >= vocab) continue;
          int seen = 0;
          for (int i = 0; i < n_hist; ++i) seen |= hist[i] == x;
          if (!seen) hist[n_hist++] = x;
        }
      }
    }
    if (!(err & ORC_ERR_BAD_SHAPE))
      err |= prepare_row(b->dtype, b->logits, off, vocab, b->temp[r], b->top_k[r],
                         b->top_p[r], b->cap, scratch, qbuf, &row, hist, n_hist, theta);
    if (err) {
      b->out_ids[r] = -1;
      b->out_eos[r] = 0;
      if (b->out_err) b->out_err[r] = err;
      continue;
    }
    uint32_t u24 = b->u24_override
                       ? b->u24_override[r]
                       : oracle_uniform24(b->seed[r], b->request[r],
                                          b->step[stream], b->codebook[r]);
    double margin_draw;
    int pos = draw_row(&row, u24, &margin_draw);
    int32_t id = row.order[pos].index;
    b->out_ids[r] = id;
    b->out_eos[r] = (uint8_t)(b->eos_id[r] >= 0 && id == b->eos_id[r]);
    if (b->out_err) b->out_err[r] = 0;
    if (b->feedback_buf && slot >= 0) b->feedback_buf[slot] = id;
    if (ring_col >= 0) { /* this step's draw joins the column's history */
      int64_t t = b->step[stream];
      int64_t j = ((t % b->hist_len) + b->hist_len) % b->hist_len;
      b->hist_ring[ring_col + j * b->hist_codebooks] = id;
    }
    if (b->u24_used) b->u24_used[r] = u24;
    if (b->margin) b->margin[r] = fmin(margin_draw, row.margin_cut);
    if (b->n_kept) b->n_kept[r] = row.k_eff;
    if (b->n_nucleus) b->n_nucleus[r] = row.n_p;
    if (b->kept_ids && b->kept_probs) {
      int32_t n = row.k_eff < b->max_keep ? row.k_eff : b->max_keep;
      for (int32_t j = 0; j < n; ++j) {
        b->kept_ids[r * (int64_t)b->max_keep + j] = row.order[j].index;
        b->kept_probs[r * (int64_t)b->max_keep + j] = row.q[j];
      }
    }
  }
  free(scratch);
  free(qbuf);
}

static void *job_main(void *arg) {
  orc_job *job = (orc_job *)arg;
  run_rows(job->b, job->row_begin, job->row_end, job->width);
  return NULL;
}

/* Samples every row of the batch.  Rows are independent, so they may be
 * spread over n_threads plain threads (the arithmetic per row is unchanged).
 * Returns 0, or -1 for an invalid cap / dtype. */
static void apply_finish(const orc_batch *b);

int oracle_sample(const orc_batch *b, int n_threads) {
  if (b->dtype != 0 && b->dtype != 1) return -1;
  if (b->cap < 1) return -1;
  if (b->hist_ring && (b->hist_len < 1 || b->hist_len > 64 || b->hist_codebooks < 1 ||
                       !b->rep_penalty))
    return -1;
  if ((b->stop_step || b->max_steps) && !b->row_finished) return -1;
  int32_t width = 1;
  for (int64_t r = 0; r < b->n_rows; ++r)
    if (b->row_vocab[r] > width && b->row_vocab[r] <= b->max_row_vocab)
      width = b->row_vocab[r];
  if (n_threads <= 1 || b->n_rows < 2 * (int64_t)n_threads) {
    run_rows(b, 0, b->n_rows, width);
    apply_finish(b);
    return 0;
  }
  pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
  orc_job *jobs = (orc_job *)malloc(sizeof(orc_job) * (size_t)n_threads);
  for (int t = 0; t < n_threads; ++t) {
    jobs[t].b = b;
    jobs[t].row_begin = b->n_rows * t / n_threads;
    jobs[t].row_end = b->n_rows * (t + 1) / n_threads;
    jobs[t].width = width;
    pthread_create(&tids[t], NULL, job_main, &jobs[t]);
  }
  for (int t = 0; t < n_threads; ++t) pthread_join(tids[t], NULL);
  free(tids);
  free(jobs);
  apply_finish(b);
  return 0;
}

/* After every row of the call [QT-eos]: a stream whose EOS was drawn at this
 * step records the step (its later steps are finished, reason stop), and
 * finished rows report their reason for their stream.  Done after all rows,
 * so no row of the call sees another row's update. */
static void apply_finish(const orc_batch *b) {
  for (int64_t r = 0; r < b->n_rows; ++r) {
    int32_t stream = b->row_stream[r];
    if (stream < 0 || stream >= b->n_streams) continue;
    if (b->row_finished && b->row_finished[r]) {
      if (b->finish_reason) b->finish_reason[stream] = b->row_finished[r];
      continue;
    }
    if (b->out_ids[r] >= 0 && b->out_eos[r]) {
      if (b->stop_step) b->stop_step[stream] = b->step[stream];
      if (b->finish_reason) b->finish_reason[stream] = 1;
    }
  }
}

/* Exhaustive draw map of one row: counts[id] += 1 for every u24 in
 * [0, 2^24).  Used to check the inverse CDF against the exact interval
 * lengths.  `values` are the row's logits as doubles.
 * Returns 0, or the row's error bits. */
uint32_t oracle_draw_map(const double *values, int32_t vocab, float temp,
                         int32_t top_k, float top_p, int32_t cap,
                         uint64_t *counts) {
  orc_entry *scratch = (orc_entry *)malloc(sizeof(orc_entry) * (size_t)vocab);
  double *qbuf = (double *)malloc(sizeof(double) * (size_t)vocab);
  orc_row row;
  memset(&row, 0, sizeof row);
  uint32_t err = prepare_row(2, values, 0, vocab, temp, top_k, top_p, cap,
                             scratch, qbuf, &row, NULL, 0, 1.0f);
  if (!err) {
    for (int32_t i = 0; i < vocab; ++i) counts[i] = 0;
    for (uint32_t u24 = 0; u24 < (1u << 24); ++u24)
      counts[row.order[draw_row(&row, u24, NULL)].index] += 1;
  }
  free(scratch);
  free(qbuf);
  return err;
}

/* ------------------------------------------------------------------------ */
/* The LM head of a frame's rows, the step before sampling ([QT-topo]; one     */
/* forward per frame samples every codebook, [D3-run]).  Row r (stream        */
/* r / Q, codebook q = r mod Q) gets                                           */
/*   l_r[v] = sum_k h_r[k] * W_q[v][k]   for v < V_r,                           */
/* h_r = hidden[r D .. r D + D) and W_q[v] = weights[off_q + v D ..) as bf16   */
/* bits, every product and sum in fp64 (a bf16 product is exact there), the    */
/* sum rounded once to fp32.  A row whose head does not lie inside the        */
/* weights (off_q < 0, off_q not a multiple of 8 elements, or                  */
/* off_q + V_r D > weights_len) gets NaN logits, a NONFINITE row error once   */
/* sampled.  A row with a shape error (V_r <= 0, V_r > max_row_vocab, logits   */
/* outside the buffer) is left unwritten: sampling reports it.                  */
/* ------------------------------------------------------------------------ */
void oracle_lm_head(const uint16_t *hidden, const uint16_t *weights, int64_t weights_len,
                    const int64_t *head_offsets, int32_t n_heads, int32_t dim,
                    int64_t n_rows, const int32_t *row_vocab, const int64_t *row_offsets,
                    int32_t max_row_vocab, float *logits, int64_t logits_len) {
  for (int64_t r = 0; r < n_rows; ++r) {
    const int32_t vr = row_vocab[r];
    const int64_t off = row_offsets[r];
    if (vr <= 0 || vr > max_row_vocab || off < 0 || off > logits_len - vr) continue;
    const int64_t hoff = head_offsets[r % n_heads];
    const int head_ok = hoff >= 0 && hoff % 8 == 0 && hoff <= weights_len - (int64_t)vr * dim;
    const int64_t h0 = r * (int64_t)dim;
    for (int32_t v = 0; v < vr; ++v) {
      if (!head_ok) {
        logits[off + v] = NAN;
        continue;
      }
      const int64_t w0 = hoff + (int64_t)v * dim;
      double acc = 0.0;
      for (int32_t k = 0; k < dim; ++k)
        acc += load_value(1, hidden, h0 + k) * load_value(1, weights, w0 + k);
      logits[off + v] = (float)acc;
    }
  }
}
