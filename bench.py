"""Benchmark of the per-step multi-codebook token sampler.

One step = one full decode-step sample: one ts_sample call over every
(stream, codebook) row of the step with the fused step advance, replayed from
CUDA graphs (the decode loop of the Drama 3 article, section "两阶段共享一张卡",
replays decode steps as one graph with no host synchronisation).  The default
workload is the 128-stream x 10-codebook step (codebook 0 V=4096, codebooks
1-9 V=1024, bf16, temperature 1.0 / top_k 30 / top_p 0.9, cap 64).  Logits
rotate over distinct step buffers totalling more than twice the L2, so every
step reads from HBM.  The timed region is exactly --steps steps, run
--repeats times (at least 10); the median per-step time is reported with its
spread.  The line also carries the multi-step figure (ts_sample_steps: R
steps in one launch), an end-to-end figure through the public API with host
copies and a sync per step, and the same figures for every other workload
("configs").

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config drama3]
                    [--impl ours|reference]

Prints one JSON line (rank 0).  N > 1 runs N independent replicas, one per
GPU (the path has no exchange step), and reports the whole-job rate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "sampled rows/s and µs/step at 128 streams×10 codebooks; HBM GB/s vs roofline"
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (about 8 TB/s)
PARAM_BYTES_READ = 64   # per row: vocab, offset, temp, top_k, top_p, seed, request,
                        # codebook, stream, step, eos id, feedback slot
PARAM_BYTES_WRITTEN = 9  # per row: id, eos flag, feedback slot
DESCRIPTIONS = {
    "drama3": "drama3: 128 streams x 10 codebooks (cb0 V=4096 EOS 4095, cb1-9 V=1024), bf16 "
              "N(0,4) with 20% near-silence streams; T 1.0, top_k 30, top_p 0.9, cap 64",
    "qwen3tts": "qwen3tts: 32 streams x 16 codebooks (cb0 V=3072 EOS 2150, cb1-15 V=2048), bf16 "
                "N(0,6.25) + 1-4 spikes; T 1.0, top_k 30, top_p 0.9, cap 64",
    "tiny": "tiny: 4 rows x V=2048 fp32 N(0,1); T 1.0, top_k 30, top_p 0.9, cap 64",
    "mixed": "mixed: 256 rows x V=4096 bf16 Student-t(3); per-row top_k/top_p/T; cap 4096",
    "stress": "stress: {rows} rows x V=151936 bf16 Zipf(1.1)+N(0,9); top_k 4096, top_p 0.9, cap 4096",
}


def split_kernels(plan, num_sms: int, n_rows: int) -> int:
    """Kernels per ts_sample call on the split path: the threshold kernel is
    skipped when the streaming grid is small (its CTAs sample the row
    themselves)."""
    return 2 if n_rows * plan["ctas_per_row"] <= 2 * num_sms else 3


def kernel_source_hash(src: str | None = None) -> str:
    """Hash of the CUDA sources with comments and whitespace removed, to tell
    whether recorded ncu counters still describe the kernels that run."""
    import hashlib
    import re
    h = hashlib.sha256()
    src = src or os.path.join(ROOT, "codebook_token_sampling_gb300", "csrc")
    for name in sorted(os.listdir(src)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(src, name), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            text = " ".join(text.split())
            h.update(name.encode() + b"\0" + text.encode())
    return h.hexdigest()[:16]


def recorded_traffic(config: str, rows, path: str | None = None, src: str | None = None,
                     field: str = "dram_bytes_per_launch"):
    """DRAM bytes per launch from the committed ncu record of this workload,
    or None when there is none or the kernels changed since it was taken.
    ``field``: "dram_bytes_per_launch" (caches flushed before each profiled
    kernel, ncu's default) or "dram_bytes_per_launch_no_flush" (caches left as
    the previous kernel left them)."""
    path = path or os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    key = config if config != "stress" else f"stress{rows}"
    e = rec.get(key)
    if not e or e.get("source_hash") != kernel_source_hash(src):
        return None
    return e.get(field)


def concat_steps(hosts):
    """R steps' batches as one batch (R times the rows, streams and slots)."""
    out = dict(hosts[0])
    off, logits, streams = 0, [], 0
    for k in ("row_vocab", "temp", "top_k", "top_p", "seed", "request", "codebook", "eos_id"):
        out[k] = np.concatenate([np.asarray(h[k]) for h in hosts])
    offs, rs, slots, steps = [], [], [], []
    for h in hosts:
        lg = np.asarray(h["logits"])
        offs.append(np.asarray(h["row_offsets"]) + off)
        logits.append(lg)
        off += lg.size
        rs.append(np.asarray(h["row_stream"]) + streams)
        sl = np.asarray(h["feedback_slot"])
        before = sum(int(x["feedback_len"]) for x in hosts[:len(slots)])
        slots.append(np.where(sl >= 0, sl + before, sl).astype(sl.dtype))
        steps.append(np.asarray(h["step"]))
        streams += int(h["n_streams"])
    out.update(logits=np.concatenate(logits), row_offsets=np.concatenate(offs),
               row_stream=np.concatenate(rs), feedback_slot=np.concatenate(slots),
               step=np.concatenate(steps), n_rows=sum(int(h["n_rows"]) for h in hosts),
               n_streams=streams, feedback_len=sum(int(h["feedback_len"]) for h in hosts))
    return out


def algorithmic_bytes(host) -> int:
    n = int(host["n_rows"])
    return workloads.logit_bytes(host) + n * (PARAM_BYTES_READ + PARAM_BYTES_WRITTEN)


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.file = None
        self.device_index = device_index

    def start(self):
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            sel = str(self.device_index)
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file.read().splitlines() if ln.strip()]
        os.unlink(self.file.name)
        sm, sm_max, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1].split()[0]))
                sm_max = max(sm_max, float(r[2].split()[0]))
                for name, val in zip(names, r[5:9]):
                    if "Active" in val and "Not" not in val:
                        reasons.add(name)
            except Exception:
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": sm_max,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# the CPU oracle as a baseline (host cores)
# --------------------------------------------------------------------------
def oracle_rate(host_steps, budget_s: float, threads: int):
    import oracle
    oracle.build()
    n_rows = int(host_steps[0]["n_rows"])
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.sample(host_steps[done % len(host_steps)], n_threads=threads)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= 4 * len(host_steps) * 50:
            break
    return n_rows * done / el, el / done, done


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------
# distributed plumbing (replicas)
# --------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
def rotation_unit(host) -> int:
    """Elements of one stream's rows (one step for a single-row-stream
    workload): rotating a step's logits by whole units keeps every row's
    width, values and structure, only in another stream's place."""
    q = int(host["n_codebooks"])
    return int(np.asarray(host["row_vocab"][:q], np.int64).sum())


def step_buffers(name, rows, dev, l2, n_gen):
    """One step's host batch and device buffers for n_buf steps that total more
    than twice the L2 (so that every timed step reads HBM): n_gen freshly
    drawn steps, the rest the same steps with their streams rotated."""
    import torch
    hosts = [workloads.make(name, i, rows=rows) for i in range(n_gen)]
    host = hosts[0]
    np_dt = np.int16 if host["dtype"] == "bf16" else np.float32
    step_elems = int(np.asarray(host["logits"]).size)
    step_bytes = workloads.logit_bytes(host)
    n_buf = max(3, -(-(2 * l2 + step_bytes) // step_bytes))
    unit = rotation_unit(host)
    units = max(1, step_elems // unit)
    big = torch.empty(n_buf * step_elems, dtype=torch.int16 if np_dt == np.int16 else torch.float32,
                      device=dev)
    srcs = [torch.from_numpy(np.ascontiguousarray(h["logits"]).view(np_dt)).to(dev) for h in hosts]
    for j in range(n_buf):
        shift = ((j // n_gen) * 7 % units) * unit
        big[j * step_elems:(j + 1) * step_elems] = torch.roll(srcs[j % n_gen], shifts=shift)
    bufs = [big[j * step_elems:(j + 1) * step_elems] for j in range(n_buf)]
    return host, hosts, big, bufs


def time_steps(sampler, batch, bufs, k, w, repeats, stream):
    """Per-step times (s) of `repeats` timed runs of exactly k steps.  Each step
    is one ts_sample call (with the step advance inside it) on the next step
    buffer; the k-step runs are CUDA graphs over consecutive buffers, replayed
    in turn, so a buffer is read again only after the others.  A batch with two
    step arrays swaps them after every call (k even, so that a graph ends where
    it started)."""
    import torch
    double = batch.step_next is not None
    if double and k % 2:
        raise ValueError("double-buffered steps need an even step count per graph")
    n_buf = len(bufs)
    n_graph = -(-n_buf // k) if k < n_buf else 1
    graphs = []
    with torch.cuda.stream(stream):
        sampler.sample(batch, stream)  # first launch outside capture
    if double:
        batch.swap_steps()
    stream.synchronize()
    for gi in range(n_graph):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(k):
                batch.set_logits(bufs[(gi * k + i) % n_buf])
                sampler.sample(batch)
                if double:
                    batch.swap_steps()
        graphs.append(g)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        done = 0
        while done < max(w, k * n_graph):
            graphs[(done // k) % n_graph].replay()
            done += k
    stream.synchronize()
    times = []
    for r in range(repeats):
        with torch.cuda.stream(stream):
            e0.record(stream)
            graphs[r % n_graph].replay()
            e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3 / k)
    return times


def time_multi_step(sampler, host, big, bufs, n_steps, repeats, stream, dev, l2):
    """ts_sample_steps: n_steps steps' rows in one launch, the launches reading
    consecutive step buffers (more than twice the L2 apart).  Per-step times."""
    import torch
    import codebook_token_sampling_gb300 as ts
    n = int(host["n_rows"])
    step_elems = bufs[0].numel()
    step_bytes = bufs[0].numel() * bufs[0].element_size()
    n_buf = len(bufs)
    n_launch = max(2, -(-(2 * l2) // (n_steps * step_bytes)) + 1)
    if n_launch * n_steps > n_buf:  # not enough buffers: a larger pool of the same steps
        reps = -(-(n_launch * n_steps) // n_buf)
        big = torch.cat([torch.roll(big, shifts=i * rotation_unit(host)) for i in range(reps)])
    b = ts.DeviceBatch(host, dev, advance_steps=True)
    out_ids = torch.empty((n_steps, n), dtype=torch.int32, device=dev)
    out_eos = torch.empty((n_steps, n), dtype=torch.uint8, device=dev)
    fb_len = int(host["feedback_len"])
    frames = torch.empty((n_steps, fb_len), dtype=torch.int32, device=dev)
    b.c.out_ids = out_ids.data_ptr()
    b.c.out_eos = out_eos.data_ptr()
    b.c.feedback_buf = frames.data_ptr()
    views = [big[j * n_steps * step_elems:(j + 1) * n_steps * step_elems] for j in range(n_launch)]

    def launch(j):
        b.set_logits(views[j % n_launch])
        sampler.sample_steps(b, n_steps, logits_step_stride=step_elems, out_step_stride=n,
                             feedback_step_stride=fb_len, stream=stream)

    with torch.cuda.stream(stream):
        for j in range(2 * n_launch):
            launch(j)
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for r in range(repeats):
        with torch.cuda.stream(stream):
            e0.record(stream)
            launch(r)
            e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3 / n_steps)
    if sampler.read_status(stream) != 0:
        raise RuntimeError("row errors in the multi-step launch")
    return times


def level_batches(host, dev):
    """One DeviceBatch per codebook level of a frame: the rows of codebook q
    (one per stream) over the same step logits, their own write-back slots in
    the frame; the last level's call advances the steps (a frame shares one
    step).  The tower samples the levels one after another."""
    import codebook_token_sampling_gb300 as ts
    q = int(host["n_codebooks"])
    cb = np.asarray(host["codebook"])
    out = []
    for level in range(q):
        rows = np.nonzero(cb == level)[0]
        h = dict(host)
        for k in ("row_vocab", "row_offsets", "temp", "top_k", "top_p", "seed", "request",
                  "codebook", "row_stream", "eos_id", "feedback_slot"):
            h[k] = np.asarray(host[k])[rows]
        h["n_rows"] = rows.size
        h["max_row_vocab"] = int(np.max(h["row_vocab"]))
        out.append(ts.DeviceBatch(h, dev, advance_steps=level == q - 1))
    return out


def time_levels(sampler, host, bufs, dev, k, repeats, stream):
    """Per-level calls: each frame is one ts_sample call per codebook level (in
    order, all in one CUDA graph of k frames over the step buffers).  Returns
    per-frame times (s)."""
    import torch
    levels = level_batches(host, dev)
    frame = levels[0].feedback
    for b in levels[1:]:  # one frame buffer and one step counter for every level
        b.feedback = frame
        b.c.feedback_buf = frame.data_ptr()
        b.step = levels[0].step
        b.c.step = levels[0].step.data_ptr()
    n_buf = len(bufs)
    with torch.cuda.stream(stream):
        for b in levels:
            sampler.sample(b, stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(k):
            for b in levels:
                b.set_logits(bufs[i % n_buf])
                sampler.sample(b)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    times = []
    for _ in range(repeats):
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3 / k)
    return times, len(levels)


def lm_head_bytes(batch, head) -> int:
    """Algorithmic bytes of one LM-head call: every head row and hidden state
    read once (bf16), every fp32 logit written once."""
    return int(np.asarray(head["weights"]).size * 2 + np.asarray(head["hidden"]).size * 2 +
               int(np.asarray(batch["row_vocab"], np.int64).sum()) * 4)


def time_lm_head(sampler, dev, k, repeats, stream, peak):
    """The LM head in front of the sampler (qwen3tts frame: 32 streams x 16
    codebooks, hidden 1024, V 3072 / 2048; synthetic weights): k calls per
    CUDA graph over three weight sets and three frames of hidden states (3 x
    69 MB of weights, more than L2), 'repeats' timed replays, median.  Times
    ts_lm_head_logits alone (the head kernel's roofline) and
    ts_lm_head_sample (head and sampler in one call, the step advance into a
    second step array)."""
    import torch
    import codebook_token_sampling_gb300 as ts
    k = max(2, k - k % 2)
    sets = [workloads.make_lm_head(i, weight_seed=i) for i in range(3)]
    batch, head = sets[0]
    b = ts.DeviceBatch(batch, dev, advance_steps=True, double_steps=True)
    h = ts.LmHead(head, dev)
    weights = [h.weights] + [torch.from_numpy(np.asarray(hd["weights"]).view(np.int16)).to(dev)
                             for _, hd in sets[1:]]
    hidden = [h.hidden] + [torch.from_numpy(np.asarray(hd["hidden"]).view(np.int16)).to(dev)
                           for _, hd in sets[1:]]

    def graph_of(call):
        with torch.cuda.stream(stream):
            for i in range(4):
                h.set_weights(weights[i % 3])
                h.set_hidden(hidden[i % 3])
                call()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(k):
                h.set_weights(weights[i % 3])
                h.set_hidden(hidden[i % 3])
                call()
        return g

    def run(g):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        with torch.cuda.stream(stream):
            g.replay()
            stream.synchronize()
            for _ in range(repeats):
                e0.record(stream)
                g.replay()
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1) / 1e3 / k)
        return times

    def fused():
        ts.ts_lm_head_sample(sampler.handle, h, b, stream)
        b.swap_steps()

    t_logits = run(graph_of(lambda: ts.ts_lm_head_logits(sampler.handle, h, b, stream)))
    t_fused = run(graph_of(fused))
    del weights, hidden
    alg = lm_head_bytes(batch, head)
    tl = statistics.median(t_logits)
    tf = statistics.median(t_fused)
    n_rows, n_streams = int(batch["n_rows"]), int(batch["n_streams"])
    return {
        "workload": "qwen3tts frame through an LM head: 32 streams x 16 codebooks, hidden 1024, "
                    "V 3072 (codebook 0) / 2048, bf16 weights N(0, (2.5/32)^2) and hidden "
                    "states N(0, 1), fp32 logits; T 1.0, top_k 30, top_p 0.9, cap 64",
        "l2": "three weight sets of %.1f MB rotated (more than L2)" % (2 * np.asarray(head["weights"]).size / 1e6),
        "calls_per_graph": k, "repeats": repeats,
        "head": {"kernel": "lm_head_kernel", "us_per_call": 1e6 * tl,
                 "us_min": 1e6 * min(t_logits), "us_max": 1e6 * max(t_logits),
                 "algorithmic_bytes_per_launch": alg, "gb_per_s": alg / tl / 1e9,
                 "roofline": {"bound": "hbm", "achieved": alg / tl / 1e9, "peak": peak,
                              "unit": "GB/s", "frac": alg / tl / 1e9 / peak,
                              "traffic": recorded_traffic("lm_head", None),
                              "traffic_no_flush": recorded_traffic(
                                  "lm_head", None, field="dram_bytes_per_launch_no_flush")},
                 "tflops": 2.0 * n_rows / int(batch["n_codebooks"]) *
                           np.asarray(head["weights"]).size / tl / 1e12},
        "head_and_sample": {"us_per_frame": 1e6 * tf, "us_min": 1e6 * min(t_fused),
                            "us_max": 1e6 * max(t_fused), "frames_per_s": n_streams / tf,
                            "rows_per_s": n_rows / tf, "launches_per_call": 2},
    }


def summarize(times):
    t = sorted(times)
    return {"us_median": 1e6 * statistics.median(t), "us_min": 1e6 * t[0], "us_max": 1e6 * t[-1],
            "repeats": len(t)}


def measure_config(args, name, rows, dev, l2, peak, k, w, repeats, num_sms, multi=(8, 64),
                   in_place_too=False):
    """One workload's single-step and multi-step figures."""
    import torch
    import codebook_token_sampling_gb300 as ts
    n_gen = 1 if name == "stress" else 4
    host, hosts, big, bufs = step_buffers(name, rows, dev, l2, n_gen)
    n_rows = int(host["n_rows"])
    sampler = ts.Sampler(dev.index or 0, host["cap"])
    sampler.reserve(n_rows, int(host["max_row_vocab"]))  # the split path's workspace
    if args.path:
        sampler.set_option(ts.TS_OPT_PATH, args.path)
    if args.warps_per_row:
        sampler.set_option(ts.TS_OPT_WARPS_PER_ROW, args.warps_per_row)
    # the decode loop's two step arrays: each call reads one and writes the
    # advanced steps to the other (no ordering between the launch's blocks);
    # an odd step count (a graph that must end where it started) advances in place
    double = k % 2 == 0
    batch = ts.DeviceBatch(host, dev, advance_steps=True, double_steps=double)
    plan = sampler.plan(batch)
    stream = torch.cuda.Stream(device=dev)
    times = time_steps(sampler, batch, bufs, k, w, repeats, stream)
    if sampler.read_status(stream) != 0:
        raise RuntimeError(f"row errors in {name}")
    in_place = None
    if in_place_too and double:  # the same loop advancing one step array in place
        b1 = ts.DeviceBatch(host, dev, advance_steps=True)
        in_place = summarize(time_steps(sampler, b1, bufs, k, w, repeats, stream))
        del b1
    alg = algorithmic_bytes(host)
    sm = summarize(times)
    t = sm["us_median"] / 1e6
    launches = (split_kernels(plan, num_sms, n_rows) + 1 if plan["path"] == 4 else
                1 if plan["path"] == 1 else 2)
    out = {
        "workload": DESCRIPTIONS[name].format(rows=rows), "rows_per_step": n_rows,
        "streams": int(host["n_streams"]), "us_per_step": sm["us_median"],
        "us_per_step_min": sm["us_min"], "us_per_step_max": sm["us_max"], "repeats": repeats,
        "steps_per_repeat": k, "rows_per_s": n_rows / t, "frames_per_s": int(host["n_streams"]) / t,
        "gb_per_s": alg / t / 1e9, "algorithmic_bytes_per_step": alg,
        "frac": alg / t / 1e9 / peak, "frac_of_nominal": alg / t / 1e9 / NOMINAL_HBM_GBS,
        "kernel": plan, "launches_per_step": launches, "dtype": host["dtype"],
        "step_arrays": ("two, swapped every call (step_out)" if double
                        else "one, advanced in place"),
        "l2": f"{len(bufs)} step buffers ({len(bufs) * workloads.logit_bytes(host) / 2**20:.0f} MiB "
              f"> 2x L2 {l2 / 2**20:.0f} MiB)",
    }
    if in_place is not None:
        out["in_place_advance"] = {"us_per_step": in_place["us_median"],
                                   "us_per_step_min": in_place["us_min"],
                                   "rows_per_s": n_rows / (in_place["us_median"] / 1e6),
                                   "how": "the same loop with one step array advanced in place "
                                          "(a ticket between the launch's blocks)"}
    if plan["path"] == 1 and multi:
        ms = {}
        for r in multi:
            mt = summarize(time_multi_step(sampler, host, big, bufs, r, repeats, stream, dev, l2))
            tt = mt["us_median"] / 1e6
            ms[str(r)] = {"us_per_step": mt["us_median"], "us_per_launch": mt["us_median"] * r,
                          "rows_per_s": n_rows / tt, "gb_per_s": alg / tt / 1e9,
                          "frac": alg / tt / 1e9 / peak}
        out["multi_step"] = ms
        out["multi_step_how"] = ("ts_sample_steps: R steps' rows in one launch of a resident grid "
                                 "(fused step advance), launches over distinct buffers")
        if int(host["n_codebooks"]) > 1:
            lt, q = time_levels(sampler, host, bufs, dev, min(k, 200), repeats, stream)
            lm = summarize(lt)
            out["per_level"] = {"calls_per_frame": q, "us_per_frame": lm["us_median"],
                                "us_per_call": lm["us_median"] / q,
                                "rows_per_call": int(host["n_streams"]),
                                "how": "one ts_sample call per codebook level (the tower samples "
                                       "the levels in order), k frames in one CUDA graph, median"}
    res = {"summary": out, "host": host, "hosts": hosts, "bufs": bufs, "big": big,
           "sampler": sampler, "batch": batch, "stream": stream, "times": times, "plan": plan}
    return res


def e2e_host_calls(res, dev, k, world):
    """End to end through the public API: one ts_sample_host call per step,
    which copies the step's logits from pinned host memory to the device,
    samples them (fused step advance), copies the ids and EOS flags back to
    pinned host memory and waits for them.  Host wall clock over k steps (at
    least 200)."""
    import torch
    import codebook_token_sampling_gb300 as ts
    host, hosts = res["host"], res["hosts"]
    sampler, stream = res["sampler"], res["stream"]
    np_dt = np.int16 if host["dtype"] == "bf16" else np.float32
    pinned = [torch.from_numpy(np.ascontiguousarray(h["logits"]).view(np_dt)).pin_memory()
              for h in hosts]
    n_rows = int(host["n_rows"])
    dev_in = torch.empty_like(res["bufs"][0])
    batch = ts.DeviceBatch(host, dev, advance_steps=True)
    batch.set_logits(dev_in)
    ids_host = torch.empty(n_rows, dtype=torch.int32).pin_memory()
    eos_host = torch.empty(n_rows, dtype=torch.uint8).pin_memory()
    n = max(200, k)

    def step(i):
        ts.ts_sample_host(sampler.handle, batch, pinned[i % len(pinned)], ids_host, eos_host,
                          stream)

    for i in range(20):
        step(i)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(n):
        step(i)
    t = (time.perf_counter() - t0) / n
    t = max_over_ranks(t, world)
    return {"value": world * n_rows / t, "unit": "rows/s",
            "h2d_bytes_per_step": int(dev_in.numel() * dev_in.element_size()),
            "d2h_bytes_per_step": n_rows * 5, "us_per_step": 1e6 * t, "steps": n,
            "how": "host wall clock; per step one ts_sample_host call: pinned H2D copy of "
                   "the logits, sampling (fused step advance), D2H of ids and EOS flags, "
                   "stream wait"}


def profile_launches(args):
    """A few plain launches of one step, for a profiler to capture."""
    import torch
    import codebook_token_sampling_gb300 as ts
    if args.profile_lm_head:
        # the LM head's qwen3tts frame: ts_lm_head_sample calls (the head
        # kernel, then the sampler), weight sets rotated as the bench loop does
        sets = [workloads.make_lm_head(i, weight_seed=i) for i in range(3)]
        lb, lh = sets[0]
        sampler = ts.Sampler(0, lb["cap"])
        batch = ts.DeviceBatch(lb, "cuda", advance_steps=True, double_steps=True)
        head = ts.LmHead(lh, "cuda")
        weights = [head.weights] + [torch.from_numpy(np.asarray(h["weights"]).view(np.int16)).cuda()
                                    for _, h in sets[1:]]
        for i in range(args.profile):
            head.set_weights(weights[i % 3])
            ts.ts_lm_head_sample(sampler.handle, head, batch)
            batch.swap_steps()
        torch.cuda.synchronize()
        print(json.dumps({"profile": "lm_head", "rows": int(lb["n_rows"]), "launches": args.profile,
                          "plan": sampler.plan(batch), "status": sampler.read_status()}))
        return
    host = workloads.make(args.config, 0, rows=args.rows)
    sampler = ts.Sampler(0, host["cap"])
    sampler.reserve(int(host["n_rows"]), int(host["max_row_vocab"]))
    if args.path:
        sampler.set_option(ts.TS_OPT_PATH, args.path)
    if args.warps_per_row:
        sampler.set_option(ts.TS_OPT_WARPS_PER_ROW, args.warps_per_row)
    # as the step loop runs: two step arrays, swapped after every call
    batch = ts.DeviceBatch(host, "cuda", advance_steps=True, double_steps=True)
    if args.profile_steps > 1:
        hosts = [workloads.make(args.config, i, rows=args.rows) for i in range(args.profile_steps)]
        np_dt = np.int16 if host["dtype"] == "bf16" else np.float32
        flat = np.concatenate([np.ascontiguousarray(h["logits"]) for h in hosts]).view(np_dt)
        buf = torch.from_numpy(flat).cuda()
        per = int(np.asarray(host["logits"]).size)
        n = int(host["n_rows"])
        out = torch.empty((args.profile_steps, n), dtype=torch.int32, device="cuda")
        eos = torch.empty((args.profile_steps, n), dtype=torch.uint8, device="cuda")
        frames = torch.empty((args.profile_steps, int(host["feedback_len"])), dtype=torch.int32,
                             device="cuda")
        batch.set_logits(buf)
        batch.c.out_ids, batch.c.out_eos = out.data_ptr(), eos.data_ptr()
        batch.c.feedback_buf = frames.data_ptr()
        for _ in range(args.profile):
            sampler.sample_steps(batch, args.profile_steps, logits_step_stride=per,
                                 out_step_stride=n, feedback_step_stride=int(host["feedback_len"]))
    else:
        for _ in range(args.profile):
            sampler.sample(batch)
            batch.swap_steps()
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.config, "rows": int(host["n_rows"]), "launches": args.profile,
                      "steps_per_launch": args.profile_steps, "plan": sampler.plan(batch),
                      "status": sampler.read_status()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--repeats", type=int, default=10,
                    help="timed runs of exactly --steps steps (at least 10; the median is reported)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="drama3", choices=list(workloads.CONFIGS))
    ap.add_argument("--rows", type=int, default=None, help="rows of the stress config")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' figures (the configs object)")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-multi-step", action="store_true",
                    help="skip the multi-step batched figure (R steps' rows in one launch)")
    ap.add_argument("--no-lm-head", action="store_true",
                    help="skip the LM-head figure (the head kernel and head + sampler)")
    ap.add_argument("--path", type=int, default=0, choices=[0, 1, 2, 3, 4],
                    help="force the kernel family (0 = automatic, 1 = warp per row, 2 = CTA / "
                         "cluster per row, 3 = wide cluster, 4 = wide split)")
    ap.add_argument("--warps-per-row", type=int, default=0, choices=[0, 1, 2, 4],
                    help="the warp path's warps per row (0 = automatic)")
    ap.add_argument("--profile", type=int, default=0, metavar="N",
                    help="profiling mode: N plain launches of one step, no timing (for ncu)")
    ap.add_argument("--profile-lm-head", action="store_true",
                    help="profiling mode: the LM head's frame (ts_lm_head_sample) instead of --config")
    ap.add_argument("--profile-steps", type=int, default=1, metavar="R",
                    help="profiling mode: each launch samples R steps (ts_sample_steps)")
    args = ap.parse_args()
    if args.config == "stress" and args.rows is None:
        args.rows = 512
    world, rank, local = dist_env()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        profile_launches(args)
        return

    desc = DESCRIPTIONS[args.config].format(rows=args.rows)
    host0 = workloads.make(args.config, 0, rows=args.rows)
    n_rows = int(host0["n_rows"])
    n_streams = int(host0["n_streams"])

    if args.impl == "reference":
        if rank != 0:
            return
        threads = host_threads()
        steps_host = [workloads.make(args.config, i, rows=args.rows) for i in range(4)]
        budget = max(1.0, min(args.cpu_budget, 120.0))
        # warm-up steps, then the timed ones (a bounded sample of the workload)
        import oracle
        oracle.build()
        for i in range(min(args.warmup, 3)):
            oracle.sample(steps_host[i % 4], n_threads=threads)
        t0 = time.perf_counter()
        done = 0
        while done < args.steps:
            oracle.sample(steps_host[done % 4], n_threads=threads)
            done += 1
            if time.perf_counter() - t0 > budget:
                break
        el = time.perf_counter() - t0
        value = n_rows * done / el
        line = {
            "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": done, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / done, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": desc, "rows_per_step": n_rows, "streams": n_streams},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads, "kind": "oracle",
                             "sample": f"{done} full steps of {n_rows} rows (of {args.steps} asked, "
                                       f"bounded to {budget:.0f} s)"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20)) or 126 * 2**20
    num_sms = props.multi_processor_count
    peak, peak_kind = measured_peak_gbs()
    k, w, reps = args.steps, args.warmup, max(10, args.repeats)

    # the headline workload: clocks sampled while its timed runs go
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(world)
    head = measure_config(args, args.config, args.rows, dev, l2, peak, k, w, reps, num_sms,
                          multi=() if args.no_multi_step else (8, 64), in_place_too=True)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    summ = head["summary"]
    t_step = max_over_ranks(summ["us_per_step"] / 1e6, world)
    e2e = e2e_host_calls(head, dev, k, world)
    others = {}
    if rank == 0 and not args.no_configs:
        for name in [c for c in workloads.CONFIGS if c != args.config]:
            rows = 512 if name == "stress" else None
            res = measure_config(args, name, rows, dev, l2, peak, min(k, 200), min(w, 50), reps,
                                 num_sms, multi=() if args.no_multi_step else (64,))
            key = f"stress{rows}" if name == "stress" else name
            others[key] = res["summary"]
            res["summary"]["traffic"] = recorded_traffic(name, rows)
            res["summary"]["traffic_no_flush"] = recorded_traffic(
                name, rows, field="dram_bytes_per_launch_no_flush")
            del res
            torch.cuda.empty_cache()
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    lm = None
    if not args.no_lm_head:
        lm = time_lm_head(head["sampler"], dev, min(k, 60), reps, head["stream"], peak)
        torch.cuda.empty_cache()
    host = head["host"]
    n_rows = int(host["n_rows"])
    n_streams = int(host["n_streams"])
    alg = algorithmic_bytes(host)
    achieved = alg / t_step / 1e9
    plan = head["plan"]
    kname = {1: "row_sampler_kernel", 2: "cluster_sampler_kernel", 3: "wide_sampler_kernel",
             4: "split_stream_kernel"}[plan["path"]]
    cpu = None
    if not args.no_cpu_baseline and world == 1:  # the oracle baseline: rank 0 at N = 1 only
        threads = host_threads()
        steps_host = [workloads.make(args.config, i, rows=args.rows) for i in range(3)]
        rate, per_step, done = oracle_rate(steps_host, args.cpu_budget, threads)
        cpu = {"value": rate, "unit": "rows/s", "cores": threads, "kind": "oracle",
               "sample": f"{done} full steps of {n_rows} rows ({per_step * 1e3:.1f} ms/step), "
                         f"all {threads} host threads"}
    line = {
        "metric": METRIC, "value": world * n_rows / t_step, "unit": "rows/s", "n_gpus": world,
        "steps": k, "warmup": w, "ms_per_step": 1e3 * t_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if host["dtype"] == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": summ["workload"], "rows_per_step": n_rows, "streams": n_streams,
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": "inputs larger than L2: " + summ["l2"],
                   "graph": "each step = one ts_sample call with the step advance inside it, "
                            "two step arrays swapped every call; "
                            f"k-step CUDA graphs, {reps} timed runs of exactly k steps, median",
                   "kernel": plan},
        "us_per_step": 1e6 * t_step,
        "timing": {"us_per_step_median": summ["us_per_step"], "us_per_step_min":
                   summ["us_per_step_min"], "us_per_step_max": summ["us_per_step_max"],
                   "repeats": reps, "steps_per_repeat": k},
        "frames_per_s": world * n_streams / t_step,
        "gb_per_s": world * alg / t_step / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": recorded_traffic(args.config, args.rows),
                     "traffic_no_flush": recorded_traffic(args.config, args.rows,
                                                          field="dram_bytes_per_launch_no_flush"),
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
                     "kernel": kname, "launches_per_step": summ["launches_per_step"],
                     "algorithmic_bytes_per_launch": alg,
                     "us_per_launch": 1e6 * t_step,
                     "us_per_launch_measured_as": "median per-step time of the timed step loop "
                                                  "(CUDA events on the launching stream)"},
        "in_place_advance": summ.get("in_place_advance"),
        "multi_step": summ.get("multi_step"),
        "lm_head": lm,
        "e2e": e2e,
        "gpu_launches": summ["launches_per_step"] * k,
        "clocks": clk,
        "cpu_baseline": cpu,
        "configs": others,
    }
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
