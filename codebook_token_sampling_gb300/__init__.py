"""Python binding of the GB300 per-step multi-codebook token sampler.

Thin ctypes marshalling over the C ABI in ``include/ts_sampler.h``; every step
of sampling runs in the CUDA kernels of ``libts_sampler.so``.  PyTorch is used
only for device memory and streams.  The functions keep the C names:

    ts_create, ts_destroy, ts_max_top_k, ts_sample, ts_sample_debug,
    ts_sample_steps, ts_reserve, ts_sample_noalloc, ts_advance_steps,
    ts_read_status, ts_set_option, ts_plan, ts_status_string, ts_last_error,
    ts_lm_head_logits, ts_lm_head_sample, ts_sample_host

``Sampler`` wraps a handle; ``DeviceBatch`` holds one step's per-row arrays on
the GPU with a prebuilt ``ts_batch`` so that repeated calls marshal nothing;
``LmHead`` holds a frame's hidden states and output heads with a prebuilt
``ts_lm_head``.
Importing this module loads the compiled library and raises if it is missing;
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

TS_OK = 0
TS_ERR_INVALID_ARG = 1
TS_ERR_UNSUPPORTED = 2
TS_ERR_CUDA = 3
TS_ERR_NO_MEMORY = 4
TS_DTYPE_F32 = 0
TS_DTYPE_BF16 = 1
TS_ROW_BAD_SHAPE = 1
TS_ROW_BAD_PARAM = 2
TS_ROW_NONFINITE = 4
TS_ROW_BAD_SLOT = 8
TS_ROW_NOT_READY = 16
TS_OPT_PATH = 1
TS_OPT_CLUSTER = 2
TS_OPT_PDL = 3
TS_OPT_WIDE_EXACT = 4
TS_OPT_WARPS_PER_ROW = 5
TS_OPT_FAIL_LAUNCH = 6
TS_MAX_VOCAB_BF16 = 163840
TS_MAX_VOCAB_F32 = 81920
TS_NOALLOC_SCRATCH_BYTES = 4194304
TS_NOALLOC_MAX_ROWS = 64
TS_LM_HEAD_DIM_STEP = 64
TS_LM_HEAD_MAX_DIM = 16384

EXPORTED = ("ts_create", "ts_destroy", "ts_max_top_k", "ts_sample", "ts_sample_debug",
            "ts_sample_steps", "ts_reserve", "ts_sample_noalloc", "ts_advance_steps",
            "ts_read_status", "ts_set_option", "ts_plan", "ts_status_string", "ts_last_error",
            "ts_lm_head_logits", "ts_lm_head_sample", "ts_sample_host")


class TsBatch(ctypes.Structure):
    """Mirror of ``ts_batch``."""
    _fields_ = [
        ("logits", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("logits_len", ctypes.c_int64),
        ("n_rows", ctypes.c_int32),
        ("max_row_vocab", ctypes.c_int32),
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
        ("out_ids", ctypes.c_void_p),
        ("out_eos", ctypes.c_void_p),
        ("feedback_buf", ctypes.c_void_p),
        ("feedback_slot", ctypes.c_void_p),
        ("feedback_len", ctypes.c_int64),
        ("advance_steps", ctypes.c_int32),
        ("stop_step", ctypes.c_void_p),
        ("max_steps", ctypes.c_void_p),
        ("finish_reason", ctypes.c_void_p),
        ("pad_id", ctypes.c_int32),
        ("hist_ring", ctypes.c_void_p),
        ("hist_len", ctypes.c_int32),
        ("hist_codebooks", ctypes.c_int32),
        ("rep_penalty", ctypes.c_void_p),
        ("step_out", ctypes.c_void_p),
    ]


class TsSteps(ctypes.Structure):
    """Mirror of ``ts_steps``."""
    _fields_ = [
        ("n_steps", ctypes.c_int32),
        ("logits_step_stride", ctypes.c_int64),
        ("out_step_stride", ctypes.c_int64),
        ("feedback_step_stride", ctypes.c_int64),
        ("ready", ctypes.c_void_p),
        ("ready_timeout_ns", ctypes.c_uint64),
    ]


class TsLmHead(ctypes.Structure):
    """Mirror of ``ts_lm_head``."""
    _fields_ = [
        ("hidden", ctypes.c_void_p),
        ("weights", ctypes.c_void_p),
        ("weights_len", ctypes.c_int64),
        ("head_offsets", ctypes.c_void_p),
        ("dim", ctypes.c_int32),
        ("n_heads", ctypes.c_int32),
    ]


class SamplerError(RuntimeError):
    def __init__(self, status: int, what: str):
        detail = _lib.ts_last_error().decode() if status == TS_ERR_CUDA else ""
        msg = f"{what}: {_lib.ts_status_string(status).decode()}"
        super().__init__(msg + (f" ({detail})" if detail else ""))
        self.status = status


def _load(path: str):
    if not os.path.exists(path):
        raise ImportError(f"sampler library not built: {path} (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "ts_create": ([ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp)], ctypes.c_int),
        "ts_destroy": ([vp], ctypes.c_int),
        "ts_max_top_k": ([vp], i32),
        "ts_sample": ([vp, ctypes.POINTER(TsBatch), vp], ctypes.c_int),
        "ts_sample_debug": ([vp, ctypes.POINTER(TsBatch), i32, vp, vp, vp, vp, vp], ctypes.c_int),
        "ts_sample_steps": ([vp, ctypes.POINTER(TsBatch), ctypes.POINTER(TsSteps), vp],
                            ctypes.c_int),
        "ts_reserve": ([vp, i32, i32], ctypes.c_int),
        "ts_sample_noalloc": ([i32, ctypes.POINTER(TsBatch), vp, vp], ctypes.c_int),
        "ts_advance_steps": ([vp, i32, vp], ctypes.c_int),
        "ts_read_status": ([vp, ctypes.POINTER(ctypes.c_uint32), vp], ctypes.c_int),
        "ts_set_option": ([vp, i32, i32], ctypes.c_int),
        "ts_plan": ([vp, ctypes.POINTER(TsBatch)] + [ctypes.POINTER(i32)] * 5, ctypes.c_int),
        "ts_sample_host": ([vp, ctypes.POINTER(TsBatch), vp, vp, vp, vp], ctypes.c_int),
        "ts_lm_head_logits": ([vp, ctypes.POINTER(TsLmHead), ctypes.POINTER(TsBatch), vp],
                              ctypes.c_int),
        "ts_lm_head_sample": ([vp, ctypes.POINTER(TsLmHead), ctypes.POINTER(TsBatch), vp],
                              ctypes.c_int),
        "ts_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "ts_last_error": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    del i64
    return lib


LIB_PATH = _build.LIB_PATH
_lib = _load(LIB_PATH)


def library():
    """The loaded ctypes library (for symbol checks)."""
    return _lib


def _check(status: int, what: str):
    if status != TS_OK:
        raise SamplerError(status, what)


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


# --------------------------------------------------------------------------
# C-named functions
# --------------------------------------------------------------------------
def ts_create(device: int = 0, max_top_k: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(_lib.ts_create(device, max_top_k, ctypes.byref(h)), "ts_create")
    return h.value


def ts_destroy(handle: int) -> None:
    _check(_lib.ts_destroy(handle), "ts_destroy")


def ts_max_top_k(handle: int) -> int:
    return int(_lib.ts_max_top_k(handle))


def ts_sample(handle: int, batch: "DeviceBatch", stream=None) -> None:
    _check(_lib.ts_sample(handle, ctypes.byref(batch.c), _stream_ptr(stream)), "ts_sample")


def ts_sample_debug(handle: int, batch: "DeviceBatch", max_keep: int, kept_ids, kept_probs,
                    n_kept, n_nucleus, stream=None) -> None:
    _check(_lib.ts_sample_debug(handle, ctypes.byref(batch.c), max_keep, kept_ids.data_ptr(),
                                kept_probs.data_ptr(), n_kept.data_ptr(), n_nucleus.data_ptr(),
                                _stream_ptr(stream)), "ts_sample_debug")


def ts_sample_steps(handle: int, batch: "DeviceBatch", steps: TsSteps, stream=None) -> None:
    _check(_lib.ts_sample_steps(handle, ctypes.byref(batch.c), ctypes.byref(steps),
                                _stream_ptr(stream)), "ts_sample_steps")


def ts_reserve(handle: int, max_rows: int, max_row_vocab: int) -> None:
    _check(_lib.ts_reserve(handle, max_rows, max_row_vocab), "ts_reserve")


def ts_sample_noalloc(batch: "DeviceBatch", max_top_k: int = 0, status=None,
                      stream=None) -> None:
    """Samples ``batch`` without any allocation, for callers whose memory is
    all owned by their own pool (the workspace is the library's static scratch
    array).  ``status``: a one-element int32 device tensor that collects the
    row error bits, or None."""
    st = _lib.ts_sample_noalloc(max_top_k, ctypes.byref(batch.c),
                                status.data_ptr() if status is not None else None,
                                _stream_ptr(stream))
    if st == TS_ERR_UNSUPPORTED:
        raise SamplerError(st, f"ts_sample_noalloc ({ts_last_error()})")
    _check(st, "ts_sample_noalloc")


def ts_advance_steps(step, stream=None) -> None:
    _check(_lib.ts_advance_steps(step.data_ptr(), step.numel(), _stream_ptr(stream)),
           "ts_advance_steps")


def ts_read_status(handle: int, stream=None) -> int:
    bits = ctypes.c_uint32()
    _check(_lib.ts_read_status(handle, ctypes.byref(bits), _stream_ptr(stream)), "ts_read_status")
    return int(bits.value)


def ts_set_option(handle: int, option: int, value: int) -> None:
    _check(_lib.ts_set_option(handle, option, value), "ts_set_option")


def ts_plan(handle: int, batch: "DeviceBatch") -> dict:
    out = [ctypes.c_int32() for _ in range(5)]
    _check(_lib.ts_plan(handle, ctypes.byref(batch.c), *[ctypes.byref(o) for o in out]),
           "ts_plan")
    keys = ("path", "ctas_per_row", "threads", "smem_bytes", "grid")
    return {k: int(o.value) for k, o in zip(keys, out)}


def ts_sample_host(handle: int, batch: "DeviceBatch", host_logits, host_ids, host_eos,
                   stream=None) -> None:
    """Host logits in, host ids and EOS flags out (see the header).  The
    three host buffers are CPU tensors (pinned for asynchronous copies) or
    numpy arrays: logits in the batch's layout (int16 / uint16 bits for bf16,
    float32), int32 ids and uint8 flags of n_rows each."""
    def ptr(a):
        return a.data_ptr() if hasattr(a, "data_ptr") else a.ctypes.data
    _check(_lib.ts_sample_host(handle, ctypes.byref(batch.c), ptr(host_logits), ptr(host_ids),
                               ptr(host_eos), _stream_ptr(stream)), "ts_sample_host")


def ts_lm_head_logits(handle: int, head: "LmHead", batch: "DeviceBatch", stream=None) -> None:
    _check(_lib.ts_lm_head_logits(handle, ctypes.byref(head.c), ctypes.byref(batch.c),
                                  _stream_ptr(stream)), "ts_lm_head_logits")


def ts_lm_head_sample(handle: int, head: "LmHead", batch: "DeviceBatch", stream=None) -> None:
    _check(_lib.ts_lm_head_sample(handle, ctypes.byref(head.c), ctypes.byref(batch.c),
                                  _stream_ptr(stream)), "ts_lm_head_sample")


def ts_status_string(status: int) -> str:
    return _lib.ts_status_string(status).decode()


def ts_last_error() -> str:
    return _lib.ts_last_error().decode()


# --------------------------------------------------------------------------
# Convenience wrappers
# --------------------------------------------------------------------------
class Sampler:
    """Owns a ``ts_sampler`` handle on one device."""

    def __init__(self, device: int = 0, max_top_k: int = 0):
        self.handle = ts_create(device, max_top_k)
        self.device = device

    @property
    def cap(self) -> int:
        return ts_max_top_k(self.handle)

    def sample(self, batch: "DeviceBatch", stream=None) -> None:
        ts_sample(self.handle, batch, stream)

    def sample_debug(self, batch: "DeviceBatch", max_keep: int, stream=None) -> dict:
        import torch
        n = batch.n_rows
        dev = batch.out_ids.device
        kept_ids = torch.full((n, max_keep), -1, dtype=torch.int32, device=dev)
        kept_probs = torch.zeros((n, max_keep), dtype=torch.float32, device=dev)
        n_kept = torch.zeros(n, dtype=torch.int32, device=dev)
        n_nucleus = torch.zeros(n, dtype=torch.int32, device=dev)
        ts_sample_debug(self.handle, batch, max_keep, kept_ids, kept_probs, n_kept, n_nucleus,
                        stream)
        return {"kept_ids": kept_ids, "kept_probs": kept_probs, "n_kept": n_kept,
                "n_nucleus": n_nucleus}

    def sample_steps(self, batch: "DeviceBatch", n_steps: int, *, logits_step_stride: int,
                     out_step_stride: int, feedback_step_stride: int = 0, ready=None,
                     ready_timeout_ns: int = 0, stream=None) -> None:
        """``n_steps`` decode steps of ``batch`` in one launch (see ts_sample_steps);
        ``ready``: a uint32/int32 tensor of per-step flags the device can read, or None."""
        st = TsSteps()
        st.n_steps = n_steps
        st.logits_step_stride = logits_step_stride
        st.out_step_stride = out_step_stride
        st.feedback_step_stride = feedback_step_stride
        st.ready = ready.data_ptr() if ready is not None else None
        st.ready_timeout_ns = ready_timeout_ns
        ts_sample_steps(self.handle, batch, st, stream)

    def read_status(self, stream=None) -> int:
        return ts_read_status(self.handle, stream)

    def reserve(self, max_rows: int, max_row_vocab: int) -> None:
        ts_reserve(self.handle, max_rows, max_row_vocab)

    def set_option(self, option: int, value: int) -> None:
        ts_set_option(self.handle, option, value)

    def plan(self, batch: "DeviceBatch") -> dict:
        return ts_plan(self.handle, batch)

    def close(self) -> None:
        if getattr(self, "handle", None):
            ts_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_ARRAYS = (("row_vocab", np.int32), ("row_offsets", np.int64), ("temp", np.float32),
           ("top_k", np.int32), ("top_p", np.float32), ("seed", np.uint64),
           ("request", np.uint64), ("codebook", np.int32), ("row_stream", np.int32),
           ("eos_id", np.int32), ("feedback_slot", np.int32))


def _to_device(a, dtype, device):
    import torch
    arr = np.ascontiguousarray(np.asarray(a, dtype=dtype))
    if arr.dtype == np.uint64:
        arr = arr.view(np.int64)
    elif arr.dtype == np.uint16:
        arr = arr.view(np.int16)
    return torch.from_numpy(arr.copy()).to(device)


class DeviceBatch:
    """One step's inputs and outputs in device memory plus the ``ts_batch``.

    ``host`` is a workload dict (see ``workloads.make``): numpy arrays that
    are copied to ``device`` once.  ``logits`` may be replaced by any device
    tensor of the same layout (``set_logits``), e.g. to rotate step buffers.
    """

    def __init__(self, host: dict, device="cuda", feedback: bool = True,
                 advance_steps: bool = False, finish=None, history=None,
                 double_steps: bool = False):
        import torch
        self.device = torch.device(device)
        self.dtype = TS_DTYPE_BF16 if host["dtype"] == "bf16" else TS_DTYPE_F32
        self.n_rows = int(host["n_rows"])
        self.arrays = {}
        logits = np.asarray(host["logits"],
                            dtype=np.uint16 if self.dtype == TS_DTYPE_BF16 else np.float32)
        self.logits = _to_device(logits, logits.dtype, self.device)
        for name, dt in _ARRAYS:
            self.arrays[name] = _to_device(host[name], dt, self.device)
        self.step = _to_device(host["step"], np.int64, self.device)
        self.out_ids = torch.full((self.n_rows,), -2, dtype=torch.int32, device=self.device)
        self.out_eos = torch.zeros(self.n_rows, dtype=torch.uint8, device=self.device)
        self.feedback = None
        if feedback:
            self.feedback = torch.full((int(host["feedback_len"]),), -1, dtype=torch.int32,
                                       device=self.device)
        c = TsBatch()
        c.dtype = self.dtype
        c.n_rows = self.n_rows
        c.max_row_vocab = int(host.get("max_row_vocab",
                                       int(np.max(host["row_vocab"], initial=1))))
        for name, _ in _ARRAYS:
            setattr(c, name, self.arrays[name].data_ptr())
        c.step = self.step.data_ptr()
        c.n_streams = int(host["n_streams"])
        c.advance_steps = 1 if advance_steps else 0
        # double_steps: a second step array receives the advanced steps
        # (step_out); swap_steps() exchanges the two between calls
        self.step_next = None
        if double_steps:
            self.step_next = torch.empty_like(self.step)
            c.step_out = self.step_next.data_ptr()
        # finished streams: finish = {"max_steps": per-stream caps or None,
        # "pad_id": int}; stop_step starts at -1 and finish_reason at 0
        self.stop_step = self.max_steps = self.finish_reason = None
        if finish is not None:
            n_streams = int(host["n_streams"])
            self.stop_step = torch.full((n_streams,), -1, dtype=torch.int64, device=self.device)
            self.finish_reason = torch.zeros(n_streams, dtype=torch.uint8, device=self.device)
            c.stop_step = self.stop_step.data_ptr()
            c.finish_reason = self.finish_reason.data_ptr()
            if finish.get("max_steps") is not None:
                self.max_steps = _to_device(finish["max_steps"], np.int64, self.device)
                c.max_steps = self.max_steps.data_ptr()
            c.pad_id = int(finish.get("pad_id", -1))
        # repetition penalty: history = {"len": T, "codebooks": Q, "penalty":
        # per-row theta}; the ring [n_streams, T, Q] starts empty (-1)
        self.hist_ring = self.rep_penalty = None
        if history is not None:
            n_streams = int(host["n_streams"])
            self.hist_ring = torch.full((n_streams, int(history["len"]), int(history["codebooks"])),
                                        -1, dtype=torch.int32, device=self.device)
            self.rep_penalty = _to_device(history["penalty"], np.float32, self.device)
            c.hist_ring = self.hist_ring.data_ptr()
            c.hist_len = int(history["len"])
            c.hist_codebooks = int(history["codebooks"])
            c.rep_penalty = self.rep_penalty.data_ptr()
        c.out_ids = self.out_ids.data_ptr()
        c.out_eos = self.out_eos.data_ptr()
        if self.feedback is not None:
            c.feedback_buf = self.feedback.data_ptr()
            c.feedback_len = self.feedback.numel()
        else:
            c.feedback_buf = None
            c.feedback_slot = None
            c.feedback_len = 0
        self.c = c
        self.set_logits(self.logits)

    def swap_steps(self) -> None:
        """With double_steps: the array the last call wrote becomes the one the
        next call reads (host-side pointer swap; capture it between calls)."""
        if self.step_next is None:
            raise ValueError("the batch has no second step array")
        self.step, self.step_next = self.step_next, self.step
        self.c.step = self.step.data_ptr()
        self.c.step_out = self.step_next.data_ptr()

    def set_logits(self, t) -> None:
        """Point the batch at another device tensor of logits (same layout)."""
        self.logits = t
        self.c.logits = t.data_ptr()
        self.c.logits_len = t.numel()

    def ids(self) -> np.ndarray:
        return self.out_ids.cpu().numpy()

    def eos(self) -> np.ndarray:
        return self.out_eos.cpu().numpy()


class LmHead:
    """A frame's hidden states and output heads in device memory plus the
    ``ts_lm_head`` (see ``ts_lm_head_logits``).

    ``head`` is a dict of numpy arrays: ``hidden`` (bf16 bits, n_rows x dim),
    ``weights`` (bf16 bits), ``head_offsets`` (int64 per head), ``n_heads``
    and ``dim``; row r uses head r mod n_heads.  ``set_weights`` and
    ``set_hidden`` point the call at other device tensors of the same layout.
    """

    def __init__(self, head: dict, device="cuda"):
        import torch
        self.device = torch.device(device)
        self.hidden = _to_device(np.asarray(head["hidden"], np.uint16), np.uint16, self.device)
        self.weights = _to_device(np.asarray(head["weights"], np.uint16), np.uint16, self.device)
        self.head_offsets = _to_device(head["head_offsets"], np.int64, self.device)
        c = TsLmHead()
        c.head_offsets = self.head_offsets.data_ptr()
        c.dim = int(head["dim"])
        c.n_heads = int(head["n_heads"])
        self.c = c
        self.set_hidden(self.hidden)
        self.set_weights(self.weights)

    def set_hidden(self, t) -> None:
        self.hidden = t
        self.c.hidden = t.data_ptr()

    def set_weights(self, t) -> None:
        self.weights = t
        self.c.weights = t.data_ptr()
        self.c.weights_len = t.numel()
