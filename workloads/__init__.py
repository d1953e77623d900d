"""Seeded synthetic inputs for the token sampler: the five workload shapes.

This module only draws inputs (logits and per-row parameters) with numpy's
PCG64; it holds none of the sampler's arithmetic.  Tests, the benchmark and
the smoke check feed the same arrays to the CUDA library and to the CPU
oracle.  The shapes stand in for the model outputs of the pages' serving runs
(no model weights or evaluation data are used):

* tiny      4 rows x V=2048 fp32 ~ N(0,1) from seed 0, identical every step.
* qwen3tts  32 streams x 16 codebooks; codebook 0 V=3072 with EOS 2150,
            codebooks 1-15 V=2048 ("案例一：Qwen3-TTS", section "拓扑": 16
            code groups of size 2048, codec EOS 2150); bf16 N(0, 2.5^2) plus
            1-4 spiked tokens per row (+U[8, 12]).
* drama3    128 streams x 10 codebooks (Drama 3 article, sections "两阶段共享
            一张卡" and "测试口径": one main token plus 9 tower codebooks, 128
            concurrent streams); codebook 0 V=4096 with EOS 4095, codebooks
            1-9 V=1024; bf16 N(0, 2^2); 20% of the streams per step are in a
            near-silence state: one dominant token at +20 in every row and, in
            codebook 0, an EOS logit of 20 + ln(1e-14) so that p(EOS) ~ 1e-14
            (handbook section "一个真实问题：说完了却停不下来").
* mixed     256 rows x V=4096 bf16 Student-t(3); per-row top_k from
            {1, 32, 64, ..., 4096}, top_p ~ U[0.5, 1] (16 rows forced to 1),
            temperature ~ U[0.6, 1.4]; cap 4096.
* lm_head   (``make_lm_head``) the qwen3tts frame (32 streams x 16 codebooks,
            V = 3072 / 2048, EOS 2150) with its logits produced by an LM head:
            hidden states bf16 N(0, 1) of size 1024 (the talker's hidden size,
            "案例一：Qwen3-TTS", section "拓扑"), drawn anew each step, and one
            head per codebook with bf16 N(0, (2.5 / 32)^2) weights, fixed
            across steps, so that the logits are about N(0, 2.5^2); fp32
            logits; top_k 30, top_p 0.9, T 1.0, cap 64.
* stress    rows x V=151936 bf16, l_i = -1.1 ln(r_i) + 3 z_i with r a random
            permutation of 1..V (a Zipf(1.1)-shaped tail) and z ~ N(0,1);
            top_k 4096, top_p 0.9, cap 4096.

The serving parameters temperature 1.0 / top_p 0.9 / top_k 30 and the default
cap 64 follow the Drama 3 article (sections "测试口径" and "能跑通的命令，和文档
写明的边界").  Rows are stream-major (row = stream * Q + codebook), and the
frame write-back slot of a row is its row index.
"""
from __future__ import annotations

import numpy as np

CONFIGS = ("tiny", "qwen3tts", "drama3", "mixed", "stress")
STRESS_VOCAB = 151936
STRESS_ROWS = (1, 8, 32, 128, 512)
_CFG_ID = {name: i for i, name in enumerate(CONFIGS)}


def to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even); returns the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(name: str, *extra: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([_CFG_ID[name], *extra]))


def _frame_layout(n_streams: int, vocabs, eos_ids):
    """Stream-major rows, one per (stream, codebook)."""
    q = len(vocabs)
    n = n_streams * q
    codebook = np.tile(np.arange(q, dtype=np.int32), n_streams)
    row_stream = np.repeat(np.arange(n_streams, dtype=np.int32), q)
    row_vocab = np.asarray(vocabs, dtype=np.int32)[codebook]
    row_offsets = np.zeros(n, dtype=np.int64)
    row_offsets[1:] = np.cumsum(row_vocab[:-1], dtype=np.int64)
    eos_id = np.asarray(eos_ids, dtype=np.int32)[codebook]
    return n, codebook, row_stream, row_vocab, row_offsets, eos_id


def _params(n, temp, top_k, top_p):
    return (np.full(n, temp, np.float32), np.full(n, top_k, np.int32),
            np.full(n, top_p, np.float32))


def _batch(name, dtype, logits, n_streams, q, codebook, row_stream, row_vocab,
           row_offsets, eos_id, temp, top_k, top_p, cap, step, seed_base):
    n = row_vocab.size
    return {
        "name": name,
        "dtype": dtype,
        "logits": logits,
        "n_rows": n,
        "n_streams": n_streams,
        "n_codebooks": q,
        "row_vocab": row_vocab,
        "row_offsets": row_offsets,
        "max_row_vocab": int(row_vocab.max(initial=1)),
        "temp": temp,
        "top_k": top_k,
        "top_p": top_p,
        "seed": (np.uint64(seed_base) + row_stream.astype(np.uint64) * np.uint64(7919)),
        "request": row_stream.astype(np.uint64),
        "codebook": codebook,
        "row_stream": row_stream,
        "step": np.full(n_streams, step, np.int64),
        "eos_id": eos_id,
        "feedback_slot": np.arange(n, dtype=np.int32),
        "feedback_len": n_streams * q,
        "cap": cap,
    }


def logits_for(name: str, step: int = 0, rows: int | None = None) -> np.ndarray:
    """Only the packed logits of one step (bf16 bits, or float32 for tiny)."""
    return make(name, step, rows=rows)["logits"]


def make(name: str, step: int = 0, *, rows: int | None = None) -> dict:
    """One step of a workload: packed logits plus every per-row array."""
    if name == "tiny":
        n, cb, rs, rv, ro, eos = _frame_layout(4, [2048], [-1])
        # reading: four independent single-codebook streams
        logits = _rng(name).standard_normal(4 * 2048, dtype=np.float32)
        t, k, p = _params(n, 1.0, 30, 0.9)
        return _batch(name, "f32", logits, 4, 1, cb, rs, rv, ro, eos, t, k, p, 64,
                      step, 0)
    if name == "qwen3tts":
        vocabs = [3072] + [2048] * 15
        n, cb, rs, rv, ro, eos = _frame_layout(32, vocabs, [2150] + [-1] * 15)
        rng = _rng(name, step)
        x = (2.5 * rng.standard_normal(int(rv.sum()), dtype=np.float32))
        for r in range(n):
            n_spk = int(rng.integers(1, 5))
            ids = rng.choice(int(rv[r]), size=n_spk, replace=False)
            x[ro[r] + ids] += rng.uniform(8.0, 12.0, size=n_spk).astype(np.float32)
        t, k, p = _params(n, 1.0, 30, 0.9)
        return _batch(name, "bf16", to_bf16_bits(x), 32, 16, cb, rs, rv, ro, eos,
                      t, k, p, 64, step, 1000)
    if name == "drama3":
        vocabs = [4096] + [1024] * 9
        n_streams = 128
        n, cb, rs, rv, ro, eos = _frame_layout(n_streams, vocabs, [4095] + [-1] * 9)
        rng = _rng(name, step)
        x = 2.0 * rng.standard_normal(int(rv.sum()), dtype=np.float32)
        silent = rng.choice(n_streams, size=round(0.2 * n_streams), replace=False)
        for s in silent:
            for c in range(10):
                r = s * 10 + c
                x[ro[r] + int(rng.integers(0, rv[r]))] = 20.0
            x[ro[s * 10] + 4095] = np.float32(20.0 + np.log(1e-14))
        t, k, p = _params(n, 1.0, 30, 0.9)
        b = _batch(name, "bf16", to_bf16_bits(x), n_streams, 10, cb, rs, rv, ro, eos,
                   t, k, p, 64, step, 2000)
        b["silent_streams"] = np.sort(silent).astype(np.int32)
        return b
    if name == "mixed":
        n, cb, rs, rv, ro, eos = _frame_layout(256, [4096], [-1])
        rng = _rng(name, step)
        x = rng.standard_t(3.0, size=256 * 4096).astype(np.float32)
        prng = _rng(name, 1 << 30)  # per-row parameters, fixed across steps
        k_choices = np.array([1] + [1 << e for e in range(5, 13)], np.int32)
        top_k = k_choices[prng.integers(0, k_choices.size, size=n)]
        top_p = prng.uniform(0.5, 1.0, size=n).astype(np.float32)
        top_p[prng.choice(n, size=16, replace=False)] = 1.0
        temp = prng.uniform(0.6, 1.4, size=n).astype(np.float32)
        return _batch(name, "bf16", to_bf16_bits(x), 256, 1, cb, rs, rv, ro, eos,
                      temp, top_k, top_p, 4096, step, 3000)
    if name == "stress":
        rows = 8 if rows is None else int(rows)
        v = STRESS_VOCAB
        n, cb, rs, rv, ro, eos = _frame_layout(rows, [v], [-1])
        rng = _rng(name, step, rows)
        ranks = rng.permuted(np.broadcast_to(np.arange(1, v + 1, dtype=np.float32),
                                             (rows, v)), axis=1)
        z = rng.standard_normal((rows, v), dtype=np.float32)
        x = (-1.1 * np.log(ranks) + 3.0 * z).astype(np.float32).ravel()
        t, k, p = _params(n, 1.0, 4096, 0.9)
        return _batch(name, "bf16", to_bf16_bits(x), rows, 1, cb, rs, rv, ro, eos,
                      t, k, p, 4096, step, 4000)
    raise KeyError(f"unknown workload {name!r}; expected one of {CONFIGS}")


def logits_as_f32(batch: dict) -> np.ndarray:
    """The packed logits of a batch as float32 values (exact for bf16)."""
    if batch["dtype"] == "bf16":
        return bf16_bits_to_f32(batch["logits"])
    return np.asarray(batch["logits"], dtype=np.float32)


def logit_bytes(batch: dict) -> int:
    """Bytes of logits a step reads (sum of row widths times element size)."""
    es = 2 if batch["dtype"] == "bf16" else 4
    return int(np.asarray(batch["row_vocab"], np.int64).sum()) * es


def make_lm_head(step: int = 0, *, streams: int = 32, dim: int = 1024, vocabs=None,
                 eos_ids=None, weight_seed: int = 0) -> tuple[dict, dict]:
    """One frame for the LM head: the batch (fp32 logits buffer, zeroed, that
    the head fills) and the head inputs (``hidden``, ``weights``,
    ``head_offsets``, ``n_heads``, ``dim``); row r uses head r mod Q."""
    vocabs = [3072] + [2048] * 15 if vocabs is None else list(vocabs)
    q = len(vocabs)
    eos_ids = ([2150] + [-1] * (q - 1)) if eos_ids is None else list(eos_ids)
    n, cb, rs, rv, ro, eos = _frame_layout(streams, vocabs, eos_ids)
    t, k, p = _params(n, 1.0, 30, 0.9)
    batch = _batch("lm_head", "f32", np.zeros(int(rv.sum()), np.float32), streams, q, cb, rs,
                   rv, ro, eos, t, k, p, 64, step, 5000)
    rng = _rng("qwen3tts", 1 << 20, step, streams, dim)
    hidden = to_bf16_bits(rng.standard_normal(n * dim, dtype=np.float32))
    offs = np.zeros(q, np.int64)
    offs[1:] = np.cumsum(np.asarray(vocabs[:-1], np.int64) * dim)
    wrng = _rng("qwen3tts", 1 << 21, weight_seed, dim)
    sigma = np.float32(2.5 / np.sqrt(dim))
    weights = to_bf16_bits(sigma * wrng.standard_normal(int(sum(vocabs)) * dim, dtype=np.float32))
    head = {"hidden": hidden, "weights": weights, "head_offsets": offs, "n_heads": q, "dim": dim}
    return batch, head
