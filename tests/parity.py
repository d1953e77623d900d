"""Helpers for comparing the CUDA sampler with the CPU oracle.

Tolerances (derived in the design notes):
* the top-k set is integer logic: it must match exactly on every row;
* sampled ids must match bit-exactly on every row whose draw lies more than
  1e-5 (in renormalised mass) from a CDF step or from the top_p cutoff; on
  the other rows the GPU id must still be a member of the oracle's nucleus
  (widened by one token at the cutoff);
* kept-set probabilities: |p_gpu - p_ref| <= 1e-6 * p_ref + 2^-120 (fp32
  relative accuracy, with an absolute floor for weights in fp32's subnormal
  range, where relative precision is lost).
"""
from __future__ import annotations

import numpy as np

BOUNDARY = 1e-5
PROB_RTOL = 1e-6
PROB_ATOL = 2.0 ** -120


def run_gpu(sampler, host, *, debug_keep=0, feedback=True, stream=None):
    import codebook_token_sampling_gb300 as ts
    import torch
    batch = ts.DeviceBatch(host, "cuda", feedback=feedback)
    dbg = None
    if debug_keep:
        dbg = sampler.sample_debug(batch, debug_keep, stream)
    else:
        sampler.sample(batch, stream)
    torch.cuda.synchronize()
    out = {"ids": batch.ids(), "eos": batch.eos(), "status": sampler.read_status()}
    if feedback:
        out["feedback"] = batch.feedback.cpu().numpy()
    if dbg is not None:
        for k, v in dbg.items():
            out[k] = v.cpu().numpy()
    return out


def compare(host, gpu, ref, *, check_probs=True, label=""):
    """Asserts every parity rule; returns the number of off-boundary rows."""
    n = int(host["n_rows"])
    err = ref["err"]
    bad = err != 0
    want_status = int(np.bitwise_or.reduce(err)) if n else 0
    assert gpu["status"] == want_status, (label, gpu["status"], want_status)
    assert np.all(gpu["ids"][bad] == -1), label
    assert np.all(gpu["eos"][bad] == 0), label
    ok = ~bad
    if "n_kept" in gpu:
        assert np.array_equal(gpu["n_kept"][ok], ref["n_kept"][ok]), label
        for r in np.nonzero(ok)[0]:
            k = int(ref["n_kept"][r])
            g_ids = gpu["kept_ids"][r, :k]
            r_ids = ref["kept_ids"][r, :k]
            assert np.array_equal(np.sort(g_ids), np.sort(r_ids)), (label, "kept set", r)
            if check_probs:
                order = np.argsort(g_ids)
                g_p = gpu["kept_probs"][r, :k][order].astype(np.float64)
                r_p = ref["kept_probs"][r, :k][np.argsort(r_ids)]
                tol = PROB_RTOL * r_p + PROB_ATOL
                assert np.all(np.abs(g_p - r_p) <= tol), (
                    label, "probs", r, float(np.max(np.abs(g_p - r_p) / np.maximum(r_p, 1e-300))))
    margin = ref.get("margin")
    if margin is None:
        safe = ok.copy()
    else:
        safe = ok & (margin > BOUNDARY)
    mism = np.nonzero(gpu["ids"][safe] != ref["ids"][safe])[0]
    assert mism.size == 0, (label, "ids", np.nonzero(safe)[0][mism][:10])
    if "n_nucleus" in gpu and margin is not None:
        assert np.array_equal(gpu["n_nucleus"][safe], ref["n_nucleus"][safe]), label
    # boundary rows: the GPU id must be a valid nucleus member
    if "kept_ids" in ref:
        for r in np.nonzero(ok & ~safe)[0]:
            n_p = int(ref["n_nucleus"][r])
            allowed = set(ref["kept_ids"][r, : min(n_p + 1, int(ref["n_kept"][r]))].tolist())
            assert int(gpu["ids"][r]) in allowed, (label, "boundary row", r)
    eos_id = np.asarray(host["eos_id"])
    want_eos = (gpu["ids"] == eos_id) & (eos_id >= 0) & ok
    assert np.array_equal(gpu["eos"].astype(bool), want_eos), label
    if "feedback" in gpu:
        slots = np.asarray(host["feedback_slot"])
        wrote = ok & (slots >= 0)
        assert np.array_equal(gpu["feedback"][slots[wrote]], gpu["ids"][wrote]), label
    return int(safe.sum())


def sub_batch(host, rows):
    """The same rows (logits, parameters and step) as a smaller batch."""
    rows = np.asarray(rows)
    out = dict(host)
    vocab = np.asarray(host["row_vocab"])[rows]
    offs = np.asarray(host["row_offsets"])[rows]
    parts = [np.asarray(host["logits"])[o:o + v] for o, v in zip(offs, vocab)]
    out["logits"] = np.concatenate(parts) if parts else np.asarray(host["logits"])[:0]
    out["n_rows"] = rows.size
    out["row_vocab"] = vocab
    out["row_offsets"] = np.concatenate([[0], np.cumsum(vocab)[:-1]]).astype(np.int64)
    for name in ("temp", "top_k", "top_p", "seed", "request", "codebook", "eos_id"):
        out[name] = np.asarray(host[name])[rows]
    streams = np.asarray(host["row_stream"])[rows]
    out["step"] = np.asarray(host["step"])[streams]
    out["row_stream"] = np.arange(rows.size, dtype=np.int32)
    out["n_streams"] = rows.size
    out["feedback_slot"] = np.arange(rows.size, dtype=np.int32)
    out["feedback_len"] = rows.size
    return out
