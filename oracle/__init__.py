"""CPU oracle for the per-step multi-codebook token sampler.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` call this module; the product library never does,
and this module imports nothing from it.  The arithmetic lives in
``ts_oracle.c`` (plain C, fp64, full sort, explicit renormalisation,
inverse-CDF draw on a Philox4x64-10 stream written from the SC'11 paper; the
LM head that produces a frame's logits, in fp64 rounded once to fp32); this
file only marshals numpy arrays through ctypes.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
things other than itself: numpy's Philox generator, numpy ``argmax``, a
library softmax, exhaustive enumeration of all 2^24 draws on tiny rows, brute
force nucleus search, a chi-square test, and the EOS-starvation invariant of
the Qwen3-TTS handbook page (section "一个真实问题：说完了却停不下来").
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ts_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libts_oracle.so")

ERR_BAD_SHAPE = 1
ERR_BAD_PARAM = 2
ERR_NONFINITE = 4
ERR_BAD_SLOT = 8


def build(force: bool = False) -> str:
    """Compile ts_oracle.c with the host C compiler (no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC",
                           "-o", tmp, _SRC, "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Batch(ctypes.Structure):
    _fields_ = [
        ("n_rows", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("logits", ctypes.c_void_p),
        ("logits_len", ctypes.c_int64),
        ("row_vocab", ctypes.c_void_p),
        ("row_offsets", ctypes.c_void_p),
        ("temp", ctypes.c_void_p),
        ("top_k", ctypes.c_void_p),
        ("top_p", ctypes.c_void_p),
        ("seed", ctypes.c_void_p),
        ("request", ctypes.c_void_p),
        ("codebook", ctypes.c_void_p),
        ("row_stream", ctypes.c_void_p),
        ("step", ctypes.c_void_p),
        ("n_streams", ctypes.c_int32),
        ("eos_id", ctypes.c_void_p),
        ("feedback_buf", ctypes.c_void_p),
        ("feedback_slot", ctypes.c_void_p),
        ("feedback_len", ctypes.c_int64),
        ("cap", ctypes.c_int32),
        ("max_row_vocab", ctypes.c_int32),
        ("u24_override", ctypes.c_void_p),
        ("out_ids", ctypes.c_void_p),
        ("out_eos", ctypes.c_void_p),
        ("out_err", ctypes.c_void_p),
        ("max_keep", ctypes.c_int32),
        ("kept_ids", ctypes.c_void_p),
        ("kept_probs", ctypes.c_void_p),
        ("n_kept", ctypes.c_void_p),
        ("n_nucleus", ctypes.c_void_p),
        ("margin", ctypes.c_void_p),
        ("u24_used", ctypes.c_void_p),
        ("stop_step", ctypes.c_void_p),
        ("max_steps", ctypes.c_void_p),
        ("finish_reason", ctypes.c_void_p),
        ("pad_id", ctypes.c_int32),
        ("row_finished", ctypes.c_void_p),
        ("hist_ring", ctypes.c_void_p),
        ("hist_len", ctypes.c_int32),
        ("hist_codebooks", ctypes.c_int32),
        ("rep_penalty", ctypes.c_void_p),
    ]


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_philox4x64_10.argtypes = [ctypes.c_void_p] * 3
    lib.oracle_philox4x64_10.restype = None
    lib.oracle_uniform24.argtypes = [ctypes.c_uint64, ctypes.c_uint64,
                                     ctypes.c_int64, ctypes.c_int32]
    lib.oracle_uniform24.restype = ctypes.c_uint32
    lib.oracle_cap.argtypes = [ctypes.c_int]
    lib.oracle_cap.restype = ctypes.c_int
    lib.oracle_sample.argtypes = [ctypes.POINTER(_Batch), ctypes.c_int]
    lib.oracle_sample.restype = ctypes.c_int
    lib.oracle_draw_map.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                                    ctypes.c_int32, ctypes.c_float, ctypes.c_int32,
                                    ctypes.c_void_p]
    lib.oracle_draw_map.restype = ctypes.c_uint32
    lib.oracle_lm_head.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                   ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64]
    lib.oracle_lm_head.restype = None
    return lib


class Oracle:
    """The oracle's entry points, bound to one compiled ``ts_oracle.c``.

    The default instance (module-level functions below) uses the library that
    ``build()`` makes; the pin tests can bind a separately compiled copy.
    """

    def __init__(self, lib_path: str | None = None):
        self.lib = _bind(lib_path or build())

    def philox4x64_10(self, ctr, key):
        return _philox(self.lib, ctr, key)

    def uniform24(self, seed, request, step, codebook):
        return int(self.lib.oracle_uniform24(seed, request, step, codebook))

    def cap(self, requested):
        return int(self.lib.oracle_cap(requested))

    def sample(self, batch, **kw):
        return _sample(self.lib, batch, **kw)

    def draw_map(self, values, temp, top_k, top_p, cap_value):
        return _draw_map(self.lib, values, temp, top_k, top_p, cap_value)

    def lm_head(self, batch, head):
        return _lm_head(self.lib, batch, head)


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def _philox(lib, ctr, key):
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint64))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64))
    out = np.zeros(4, dtype=np.uint64)
    lib.oracle_philox4x64_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return tuple(int(v) for v in out)


def philox4x64_10(ctr, key):
    """One Philox4x64-10 block: 4 x uint64 counter, 2 x uint64 key."""
    return default().philox4x64_10(ctr, key)


def uniform24(seed: int, request: int, step: int, codebook: int) -> int:
    """The 24-bit integer u24 of a row's draw (u = u24 * 2^-24)."""
    return default().uniform24(seed, request, step, codebook)


def cap(requested: int) -> int:
    """Effective top-k cap for a requested value, or -1 if invalid."""
    return default().cap(requested)


def _arr(a, dtype):
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def sample(batch, **kw):
    """Sample every row of ``batch`` with the default oracle (see ``_sample``)."""
    return default().sample(batch, **kw)


def draw_map(values, temp: float, top_k: int, top_p: float, cap_value: int):
    """Counts of each token over all 2^24 values of u24 for one row."""
    return default().draw_map(values, temp, top_k, top_p, cap_value)


def lm_head(batch, head):
    """The LM head's fp32 logits for ``batch`` (see ``_lm_head``)."""
    return default().lm_head(batch, head)


def _lm_head(lib, batch, head):
    """The fp32 logits of every row of ``batch`` from its codebook's head.

    ``head`` holds ``hidden`` (bf16 bits, [n_rows, dim]), ``weights`` (bf16
    bits), ``head_offsets`` (int64 per head), ``n_heads`` and ``dim``; row r
    uses head r mod n_heads.  Returns a float32 array of the batch's logits length: the
    rows' logits at their offsets (NaN for a row whose head lies outside the
    weights), zeros elsewhere.  The batch's own ``logits`` are not read.
    """
    n = int(batch["n_rows"])
    hidden = _arr(head["hidden"], np.uint16)
    weights = _arr(head["weights"], np.uint16)
    offs = _arr(head["head_offsets"], np.int64)
    n_heads = int(head["n_heads"])
    dim = int(head["dim"])
    assert hidden.size == n * dim and offs.size == n_heads
    rv = _arr(batch["row_vocab"], np.int32)
    ro = _arr(batch["row_offsets"], np.int64)
    n_out = int(batch.get("logits_len", np.asarray(batch["logits"]).size))
    out = np.zeros(n_out, np.float32)
    mrv = int(batch.get("max_row_vocab", int(np.max(rv, initial=1))))
    lib.oracle_lm_head(hidden.ctypes.data, weights.ctypes.data, weights.size, offs.ctypes.data,
                       n_heads, dim, n, rv.ctypes.data, ro.ctypes.data, mrv,
                       out.ctypes.data, out.size)
    return out


def _sample(lib, batch, *, n_threads: int = 1, u24=None, max_keep: int = 0,
            feedback_buf=None, stop_step=None, max_steps=None, finish_reason=None,
            pad_id: int = -1, hist_ring=None, rep_penalty=None):
    """Sample every row of ``batch`` (a dict of numpy arrays, see ``workloads``).

    Returns a dict with ``ids`` (int32), ``eos`` (uint8), ``err`` (uint32 per-row
    error bits), ``u24`` (the draws used) and, when ``max_keep > 0``, the sorted
    kept set ``kept_ids`` / ``kept_probs`` (fp64), ``n_kept``, ``n_nucleus`` and
    ``margin`` (distance of the draw or of top_p from the nearest boundary).
    ``feedback_buf`` (int32, modified in place) receives the write-back.
    Finished streams (the handbook's EOS-starvation section): ``stop_step``
    (int64 per stream, < 0 = running; updated in place when a row draws its
    EOS) and ``max_steps`` (int64 per stream, the length cap on the stream's
    step) make a stream's rows draw nothing and return ``pad_id``;
    ``finish_reason`` (uint8 per stream, updated in place) gets 1 (stop) or 2
    (length).  The result then also holds ``finished`` (uint8 per row).
    Repetition penalty (CTRL, Keskar et al. 2019): ``hist_ring`` (int32,
    shape [n_streams, T, Q], updated in place with each row's draw at slot
    step mod T) and ``rep_penalty`` (float32 per row).
    """
    n = int(batch["n_rows"])
    keep = {}
    b = _Batch()
    b.n_rows = n
    b.dtype = 1 if batch["dtype"] == "bf16" else 0
    logits = _arr(batch["logits"], np.uint16 if b.dtype == 1 else np.float32)
    keep["logits"] = logits
    b.logits = logits.ctypes.data
    b.logits_len = logits.size
    spec = [("row_vocab", np.int32), ("row_offsets", np.int64), ("temp", np.float32),
            ("top_k", np.int32), ("top_p", np.float32), ("seed", np.uint64),
            ("request", np.uint64), ("codebook", np.int32), ("row_stream", np.int32),
            ("step", np.int64), ("eos_id", np.int32), ("feedback_slot", np.int32)]
    for name, dt in spec:
        a = _arr(batch[name], dt)
        keep[name] = a
        setattr(b, name, a.ctypes.data)
    b.n_streams = int(batch["n_streams"])
    if feedback_buf is not None:
        assert feedback_buf.dtype == np.int32 and feedback_buf.flags.c_contiguous
        b.feedback_buf = feedback_buf.ctypes.data
        b.feedback_len = feedback_buf.size
    b.cap = int(batch["cap"])
    b.max_row_vocab = int(batch.get("max_row_vocab", int(np.max(keep["row_vocab"], initial=1))))
    if hist_ring is not None:
        assert hist_ring.dtype == np.int32 and hist_ring.flags.c_contiguous and hist_ring.ndim == 3
        b.hist_ring = hist_ring.ctypes.data
        b.hist_len = hist_ring.shape[1]
        b.hist_codebooks = hist_ring.shape[2]
        rp = _arr(rep_penalty, np.float32)
        assert rp.size == n
        keep["rep_penalty"] = rp
        b.rep_penalty = rp.ctypes.data
    if u24 is not None:
        u = _arr(u24, np.uint32)
        assert u.size == n
        keep["u24"] = u
        b.u24_override = u.ctypes.data
    finished = None
    if stop_step is not None or max_steps is not None:
        finished = np.zeros(n, np.uint8)
        b.row_finished = finished.ctypes.data
        b.pad_id = int(pad_id)
        if stop_step is not None:
            assert stop_step.dtype == np.int64 and stop_step.flags.c_contiguous
            b.stop_step = stop_step.ctypes.data
        if max_steps is not None:
            ms = _arr(max_steps, np.int64)
            keep["max_steps"] = ms
            b.max_steps = ms.ctypes.data
        if finish_reason is not None:
            assert finish_reason.dtype == np.uint8 and finish_reason.flags.c_contiguous
            b.finish_reason = finish_reason.ctypes.data
    out = {"ids": np.zeros(n, np.int32), "eos": np.zeros(n, np.uint8),
           "err": np.zeros(n, np.uint32), "u24": np.zeros(n, np.uint32)}
    b.out_ids = out["ids"].ctypes.data
    b.out_eos = out["eos"].ctypes.data
    b.out_err = out["err"].ctypes.data
    b.u24_used = out["u24"].ctypes.data
    if max_keep > 0:
        out["kept_ids"] = np.full((n, max_keep), -1, np.int32)
        out["kept_probs"] = np.zeros((n, max_keep), np.float64)
        out["n_kept"] = np.zeros(n, np.int32)
        out["n_nucleus"] = np.zeros(n, np.int32)
        out["margin"] = np.zeros(n, np.float64)
        b.max_keep = max_keep
        b.kept_ids = out["kept_ids"].ctypes.data
        b.kept_probs = out["kept_probs"].ctypes.data
        b.n_kept = out["n_kept"].ctypes.data
        b.n_nucleus = out["n_nucleus"].ctypes.data
        b.margin = out["margin"].ctypes.data
    rc = lib.oracle_sample(ctypes.byref(b), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_sample rejected the batch (dtype or cap)")
    if finished is not None:
        out["finished"] = finished
    return out


def _draw_map(lib, values, temp, top_k, top_p, cap_value):
    v = _arr(values, np.float64)
    counts = np.zeros(v.size, np.uint64)
    err = lib.oracle_draw_map(v.ctypes.data, v.size, temp, top_k, top_p,
                                  cap_value, counts.ctypes.data)
    if err:
        raise ValueError(f"row error bits {err}")
    return counts
