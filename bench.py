"""Benchmark of the per-step multi-codebook token sampler.

One step = one full decode-step sample: ts_sample over every (stream,
codebook) row of the step, then ts_advance_steps, replayed from a CUDA graph
(the decode loop of the Drama 3 article, section "两阶段共享一张卡", replays
decode steps as one graph with no host synchronisation).  The default
workload is the 128-stream x 10-codebook step (codebook 0 V=4096, codebooks
1-9 V=1024, bf16, temperature 1.0 / top_k 30 / top_p 0.9, cap 64).  Logits
rotate over distinct step buffers totalling more than twice the L2, so every
step reads from HBM.

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


def recorded_traffic(config: str, rows, path: str | None = None, src: str | None = None):
    """DRAM bytes per launch from the committed ncu record of this workload,
    or None when there is none or the kernels changed since it was taken."""
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
    return e.get("dram_bytes_per_launch")


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


def multi_step(args, dev, l2, peak):
    """R steps' rows sampled by one launch (R = 1, 8, 64), to show the
    bandwidth bound of steps too small to fill the GPU on their own."""
    import torch
    import codebook_token_sampling_gb300 as ts
    res = {}
    for R in (1, 8, 64):
        host = concat_steps([workloads.make(args.config, i) for i in range(R)])
        n_rows = int(host["n_rows"])
        sbytes = workloads.logit_bytes(host)
        n_buf = max(2, min(64, -(-(2 * l2 + sbytes) // sbytes)))
        np_dt = np.int16 if host["dtype"] == "bf16" else np.float32
        base = torch.from_numpy(np.ascontiguousarray(host["logits"]).view(np_dt)).to(dev)
        # distinct buffers: the same rows' values rotated by a row-sized stride
        bufs = [torch.roll(base, shifts=int(i * 4099)) for i in range(n_buf)]
        sampler = ts.Sampler(dev.index or 0, host["cap"])
        batch = ts.DeviceBatch(host, dev)
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            sampler.sample(batch, stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_buf):
                batch.set_logits(bufs[i])
                sampler.sample(batch)
        reps = max(3, 2000 // (n_buf * R))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / (reps * n_buf)
        if sampler.read_status(stream) != 0:
            raise RuntimeError("row errors in the multi-step launch")
        gbs = algorithmic_bytes(host) / t / 1e9
        res[str(R)] = {"rows_per_launch": n_rows, "us_per_launch": 1e6 * t,
                       "us_per_step": 1e6 * t / R, "rows_per_s": n_rows / t,
                       "gb_per_s": gbs, "frac": gbs / peak}
        sampler.close()
        del bufs, base
    return res


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
def run_ours(args, world, rank, local):
    import torch
    import codebook_token_sampling_gb300 as ts

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20)) or 126 * 2**20
    host = workloads.make(args.config, 0, rows=args.rows)
    n_rows = int(host["n_rows"])
    step_bytes = workloads.logit_bytes(host)
    n_buf = max(2, min(args.max_buffers, -(-(2 * l2 + step_bytes) // step_bytes)))
    # distinct step buffers, each a freshly drawn step of the workload
    np_dt = np.int16 if host["dtype"] == "bf16" else np.float32
    base, bufs = [], []
    for i in range(n_buf):
        src = np.ascontiguousarray(workloads.make(args.config, i, rows=args.rows)["logits"])
        if i < 8:
            base.append(src)
        bufs.append(torch.from_numpy(src.view(np_dt)).to(dev))
    sampler = ts.Sampler(local, host["cap"])
    sampler.reserve(n_rows, int(host["max_row_vocab"]))  # workspace for the split wide path
    if args.path:
        sampler.set_option(ts.TS_OPT_PATH, args.path)
    batch = ts.DeviceBatch(host, dev)
    plan = sampler.plan(batch)
    stream = torch.cuda.Stream(device=dev)

    def capture(nsteps, with_advance=True, first=0):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            sampler.sample(batch, stream)  # warm-up launch outside capture
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsteps):
                batch.set_logits(bufs[(first + i) % n_buf])
                sampler.sample(batch)
                if with_advance:
                    ts.ts_advance_steps(batch.step)
        return g

    k, w = args.steps, args.warmup
    g_full = capture(n_buf)
    rem = k % n_buf
    g_rem = capture(rem) if rem else None

    def run_steps(nsteps):
        full, r = divmod(nsteps, n_buf)
        for _ in range(full):
            g_full.replay()
        if r:
            assert r == rem
            g_rem.replay()

    with torch.cuda.stream(stream):
        for _ in range(max(1, -(-w // n_buf))):
            g_full.replay()
    stream.synchronize()
    if sampler.read_status(stream) != 0:
        raise RuntimeError("row errors during warm-up")

    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_steps(k)
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_step = e0.elapsed_time(e1) / 1e3
    clk = clocks.stop() if clocks else None
    t_max = max_over_ranks(t_step, world)

    # kernel-only pass: the sampler launches alone (for the roofline)
    g_kern = capture(n_buf, with_advance=False)
    with torch.cuda.stream(stream):
        g_kern.replay()
        e0.record(stream)
        reps = max(1, k // n_buf)
        for _ in range(reps):
            g_kern.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t_launch = e0.elapsed_time(e1) / 1e3 / (reps * n_buf)

    # end to end through the C ABI from pinned host memory: per step the
    # step's logits go host->device, the frame's ids and EOS flags come back
    n_host = min(n_buf, 8)
    pinned = [torch.from_numpy(np.ascontiguousarray(base[i % len(base)]).view(np_dt)).pin_memory()
              for i in range(n_host)]
    dev_in = [torch.empty_like(bufs[0]) for _ in range(2)]
    ids_host = torch.empty((n_host, n_rows), dtype=torch.int32).pin_memory()
    eos_host = torch.empty((n_host, n_rows), dtype=torch.uint8).pin_memory()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        for i in range(n_host):
            d = dev_in[i % 2]
            d.copy_(pinned[i], non_blocking=True)
            batch.set_logits(d)
            sampler.sample(batch)
            ts.ts_advance_steps(batch.step)
            ids_host[i].copy_(batch.out_ids, non_blocking=True)
            eos_host[i].copy_(batch.out_eos, non_blocking=True)
    with torch.cuda.stream(stream):
        g_e2e.replay()
    torch.cuda.synchronize()
    e2e_reps = max(1, min(k, 20000) // n_host)
    barrier(world)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_reps):
            g_e2e.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3 / (e2e_reps * n_host), world)
    status = sampler.read_status(stream)
    if status != 0:
        raise RuntimeError(f"row errors during the run: {status}")

    return {
        "host": host, "n_rows": n_rows, "t_step": t_max / k, "t_launch": t_launch,
        "t_e2e": t_e2e, "clocks": clk, "plan": plan, "n_buf": n_buf, "l2": l2,
        "step_bytes": step_bytes,
        "split_kernels": split_kernels(plan, props.multi_processor_count, n_rows),
        "launches": (split_kernels(plan, props.multi_processor_count, n_rows)
                     if plan["path"] == 4 else 1) * k + k,
        "h2d": int(bufs[0].numel() * bufs[0].element_size()), "d2h": n_rows * 5,
    }


def profile_launches(args):
    """A few plain launches of one step, for a profiler to capture."""
    import torch
    import codebook_token_sampling_gb300 as ts
    host = workloads.make(args.config, 0, rows=args.rows)
    sampler = ts.Sampler(0, host["cap"])
    sampler.reserve(int(host["n_rows"]), int(host["max_row_vocab"]))
    if args.path:
        sampler.set_option(ts.TS_OPT_PATH, args.path)
    batch = ts.DeviceBatch(host, "cuda")
    for _ in range(args.profile):
        sampler.sample(batch)
        ts.ts_advance_steps(batch.step)
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.config, "rows": int(host["n_rows"]), "launches": args.profile,
                      "plan": sampler.plan(batch), "status": sampler.read_status()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="drama3", choices=list(workloads.CONFIGS))
    ap.add_argument("--rows", type=int, default=None, help="rows of the stress config")
    ap.add_argument("--max-buffers", type=int, default=160)
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-multi-step", action="store_true",
                    help="skip the multi-step batched figure (R steps' rows in one launch)")
    ap.add_argument("--path", type=int, default=0, choices=[0, 1, 2, 3, 4],
                    help="force the kernel family (0 = automatic, 1 = warp per row, 2 = CTA / "
                         "cluster per row, 3 = wide cluster, 4 = wide split)")
    ap.add_argument("--profile", type=int, default=0, metavar="N",
                    help="profiling mode: N plain launches of one step, no timing (for ncu)")
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
    r = run_ours(args, world, rank, local)
    peak, peak_kind = measured_peak_gbs()
    multi = None
    if args.config != "stress" and not args.no_multi_step and rank == 0:
        import torch
        multi = multi_step(args, torch.device("cuda", local), r["l2"], peak)
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    t = r["t_step"]
    value = world * n_rows / t
    alg = algorithmic_bytes(r["host"])
    # the sampler's launches timed inside the timed region: each step is one
    # ts_sample call plus the step-advance kernel, so this slightly
    # understates the sampler's own rate
    achieved = alg / t / 1e9
    split = r["plan"]["path"] == 4
    cpu = None
    if not args.no_cpu_baseline and world == 1:  # the oracle baseline: rank 0 at N = 1 only
        threads = host_threads()
        steps_host = [workloads.make(args.config, i, rows=args.rows) for i in range(3)]
        rate, per_step, done = oracle_rate(steps_host, args.cpu_budget, threads)
        cpu = {"value": rate, "unit": "rows/s", "cores": threads, "kind": "oracle",
               "sample": f"{done} full steps of {n_rows} rows ({per_step * 1e3:.1f} ms/step), "
                         f"all {threads} host threads"}
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if r["host"]["dtype"] == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": desc, "rows_per_step": n_rows, "streams": n_streams,
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": f"inputs rotate over {r['n_buf']} distinct step buffers "
                         f"({r['n_buf'] * r['step_bytes'] / 2**20:.0f} MiB > 2x L2 "
                         f"{r['l2'] / 2**20:.0f} MiB)",
                   "graph": "each step = ts_sample + ts_advance_steps, replayed from a CUDA graph",
                   "kernel": r["plan"]},
        "us_per_step": 1e6 * t,
        "frames_per_s": world * n_streams / t,
        "gb_per_s": world * alg / t / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(args.config, args.rows),
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "launch": ("one ts_sample call: split_stream_kernel (threshold inline) + "
                                "split_tail_kernel" if r["split_kernels"] == 2 else
                                "one ts_sample call: split_threshold_kernel + split_stream_kernel + "
                                "split_tail_kernel") if split else
                               "one ts_sample call: one kernel (" +
                               {1: "row_sampler_kernel", 2: "cluster_sampler_kernel",
                                3: "wide_sampler_kernel"}[r["plan"]["path"]] + ")",
                     "algorithmic_bytes_per_launch": alg,
                     "us_per_launch": 1e6 * t,
                     "us_per_launch_measured_as": "the timed step loop (ts_sample + step advance)",
                     "us_per_launch_back_to_back": 1e6 * r["t_launch"]},
        "multi_step": multi,
        "e2e": {"value": world * n_rows / r["t_e2e"], "unit": "rows/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "us_per_step": 1e6 * r["t_e2e"]},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
