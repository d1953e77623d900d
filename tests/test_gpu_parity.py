"""CUDA sampler vs the CPU oracle, element by element, through the C ABI.

Covers the five workload shapes (the 151,936-wide stress at 1/8/32 rows in
full and at 512 rows on sampled rows, in the launch configuration the
benchmark times), both kernel families, every cluster size, ragged and
misaligned rows, ties, non-finite values, degenerate parameters, row errors,
determinism, CUDA-graph capture and a 500-step graph loop with frame
write-back.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import compare, run_gpu, sub_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import codebook_token_sampling_gb300 as mod
    return mod


def make_sampler(ts, cap, path=0, cluster=0):
    s = ts.Sampler(0, cap)
    if path:
        s.set_option(ts.TS_OPT_PATH, path)
    if cluster:
        s.set_option(ts.TS_OPT_CLUSTER, cluster)
    return s


# ---------------------------------------------------------------------------
# the workload shapes
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", [0, 2])
@pytest.mark.parametrize("name", ["tiny", "qwen3tts", "drama3", "mixed"])
def test_workload_parity(ts, name, path):
    for step in (0, 7):
        host = workloads.make(name, step)
        keep = host["cap"]
        ref = oracle.sample(host, max_keep=keep, n_threads=8)
        s = make_sampler(ts, host["cap"], path)
        gpu = run_gpu(s, host, debug_keep=keep)
        n_safe = compare(host, gpu, ref, label=f"{name}/path{path}/step{step}")
        assert n_safe >= 0.98 * host["n_rows"]
        plain = run_gpu(s, host)
        assert np.array_equal(plain["ids"], gpu["ids"])
        s.close()


@pytest.mark.parametrize("rows", [1, 8, 32])
def test_stress_parity(ts, rows):
    host = workloads.make("stress", 1, rows=rows)
    ref = oracle.sample(host, max_keep=4096, n_threads=8)
    s = make_sampler(ts, 4096)
    gpu = run_gpu(s, host, debug_keep=4096)
    compare(host, gpu, ref, label=f"stress{rows}")
    s.close()


def test_stress_512_rows_sampled(ts):
    """Full-size stress step, launched as the benchmark launches it; the
    oracle checks 48 sampled rows one by one."""
    host = workloads.make("stress", 0, rows=512)
    s = make_sampler(ts, 4096)
    gpu = run_gpu(s, host)
    assert gpu["status"] == 0
    rows = np.random.default_rng(5).choice(512, size=48, replace=False)
    sub = sub_batch(host, rows)
    ref = oracle.sample(sub, max_keep=4096, n_threads=8)
    safe = ref["margin"] > 1e-5
    # a stress row's nucleus holds thousands of CDF steps, so about 11% of
    # rows lie within 1e-5 of a boundary; most must still be checked
    assert safe.sum() >= 0.75 * rows.size
    assert np.array_equal(gpu["ids"][rows][safe], ref["ids"][safe])
    assert np.array_equal(gpu["feedback"][rows], gpu["ids"][rows])
    s.close()


def test_drama3_full_step_bench_launch(ts):
    """The 128-stream x 10-codebook step exactly as the benchmark launches it."""
    host = workloads.make("drama3", 11)
    s = make_sampler(ts, host["cap"])
    gpu = run_gpu(s, host)
    ref = oracle.sample(host, max_keep=64)
    compare(host, gpu, ref, label="drama3 bench launch")
    s.close()


# ---------------------------------------------------------------------------
# geometry independence: warp path, CTA path and every cluster size agree
# ---------------------------------------------------------------------------
def test_geometry_independence(ts):
    rng = np.random.default_rng(3)
    v, rows = 20000, 6
    x = workloads.to_bf16_bits(rng.normal(0, 3, v * rows).astype(np.float32))
    host = workloads.make("mixed", 0)
    host = sub_batch(host, np.arange(rows))
    host.update(logits=x, row_vocab=np.full(rows, v, np.int32),
                row_offsets=np.arange(rows, dtype=np.int64) * v, max_row_vocab=v,
                top_k=np.array([1, 30, 64, 700, 4096, 0], np.int32))
    ref = oracle.sample(host, max_keep=4096)
    outs = []
    for g in (1, 2, 4, 8):
        s = make_sampler(ts, 4096, path=2, cluster=g)
        gpu = run_gpu(s, host, debug_keep=4096)
        compare(host, gpu, ref, label=f"cluster{g}")
        outs.append(gpu)
        s.close()
    for o in outs[1:]:
        assert np.array_equal(o["ids"], outs[0]["ids"])
        assert np.array_equal(o["n_nucleus"], outs[0]["n_nucleus"])
    d = workloads.make("drama3", 4)
    ids = []
    for path, pdl in ((1, 1), (2, 1), (1, 0), (2, 0)):
        s = make_sampler(ts, 64, path=path)
        s.set_option(ts.TS_OPT_PDL, pdl)
        ids.append(run_gpu(s, d)["ids"])
        s.close()
    for other in ids[1:]:
        assert np.array_equal(ids[0], other)


@pytest.mark.parametrize("name", ["tiny", "qwen3tts", "drama3"])
def test_warps_per_row(ts, name):
    """Rows shared by 1, 2 or 4 warps give the oracle's results, and the
    same ids as each other."""
    host = workloads.make(name, 3)
    ref = oracle.sample(host, max_keep=host["cap"], n_threads=8)
    ids = []
    for wpr in (1, 2, 4):
        s = make_sampler(ts, host["cap"], path=1)
        s.set_option(ts.TS_OPT_WARPS_PER_ROW, wpr)
        assert s.plan(ts.DeviceBatch(host, "cuda"))["ctas_per_row"] == wpr
        gpu = run_gpu(s, host, debug_keep=host["cap"])
        compare(host, gpu, ref, label=f"{name} wpr{wpr}")
        ids.append(gpu["ids"])
        s.close()
    assert np.array_equal(ids[0], ids[1]) and np.array_equal(ids[0], ids[2])


# ---------------------------------------------------------------------------
# edge cases: ragged / misaligned rows, ties, non-finite values, parameters
# ---------------------------------------------------------------------------
def _edge_batch(dtype, rng):
    rows = []  # (values, temp, top_k, top_p)
    nrm = lambda n, s=2.0: rng.normal(0, s, n).astype(np.float32)
    rows += [(nrm(1), 1.0, 30, 0.9), (nrm(5), 1.0, 30, 0.9), (nrm(13), 0.7, 4, 0.8),
             (nrm(1000), 1.0, 30, 0.9), (nrm(2045), 1.3, 64, 0.95)]
    rows += [(np.full(300, 1.5, np.float32), 1.0, 30, 0.9)]                # full ties
    rows += [(rng.choice([0.0, 0.5, 1.0], 777).astype(np.float32), 1.0, 30, 0.9)]
    y = np.full(200, -np.inf, np.float32)
    y[[7, 50, 199]] = [0.0, 1.0, 0.5]
    rows += [(y, 1.0, 30, 1.0)]                                            # -inf inside top-k
    rows += [(np.array([0.0, np.nan, 1.0] * 10, np.float32), 1.0, 30, 0.9)]
    rows += [(np.array([0.0, np.inf, 1.0] * 10, np.float32), 1.0, 30, 0.9)]
    rows += [(np.full(40, -np.inf, np.float32), 1.0, 30, 0.9)]
    base = nrm(500)
    for t, k, p in ((1.0, 900, 0.9), (1.0, 0, 0.9), (1.0, -5, 0.9), (1.0, 30, 0.0),
                    (1.0, 30, -1.0), (1.0, 30, 1.0), (1.0, 30, 2.0), (0.0, 30, 0.9),
                    (-1.0, 30, 0.9), (float("nan"), 30, 0.9), (1.0, 30, float("nan")),
                    (float("inf"), 30, 0.9), (0.05, 64, 0.99), (25.0, 64, 0.99)):
        rows.append((base, t, k, p))
    n = len(rows)
    gap = rng.integers(0, 7, n)  # misaligned starts
    offs, parts, pos = [], [], 0
    for (vals, *_), g in zip(rows, gap):
        parts.append(np.zeros(int(g), np.float32))
        pos += int(g)
        offs.append(pos)
        parts.append(vals)
        pos += vals.size
    flat = np.concatenate(parts)
    logits = workloads.to_bf16_bits(flat) if dtype == "bf16" else flat
    if dtype == "bf16":  # keep NaN / inf patterns exact
        nan = np.isnan(flat)
        logits[nan] = 0x7FC0
    host = {
        "dtype": dtype, "logits": logits, "n_rows": n, "n_streams": n, "n_codebooks": 1,
        "row_vocab": np.array([r[0].size for r in rows], np.int32),
        "row_offsets": np.array(offs, np.int64),
        "temp": np.array([r[1] for r in rows], np.float32),
        "top_k": np.array([r[2] for r in rows], np.int32),
        "top_p": np.array([r[3] for r in rows], np.float32),
        "seed": np.arange(n, dtype=np.uint64) * np.uint64(977), "request": np.arange(n, dtype=np.uint64),
        "codebook": np.zeros(n, np.int32), "row_stream": np.arange(n, dtype=np.int32),
        "step": np.full(n, 5, np.int64), "eos_id": np.full(n, 2, np.int32),
        "feedback_slot": np.arange(n, dtype=np.int32), "feedback_len": n, "cap": 64,
    }
    host["max_row_vocab"] = int(host["row_vocab"].max())
    return host


@pytest.mark.parametrize("path,wpr", [(1, 1), (1, 2), (1, 4), (2, 0)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_edge_rows(ts, dtype, path, wpr):
    rng = np.random.default_rng(21)
    host = _edge_batch(dtype, rng)
    ref = oracle.sample(host, max_keep=64)
    assert np.any(ref["err"] == 4) and np.any(ref["err"] == 2)
    s = make_sampler(ts, 64, path=path)
    if wpr:
        s.set_option(ts.TS_OPT_WARPS_PER_ROW, wpr)
    gpu = run_gpu(s, host, debug_keep=64)
    compare(host, gpu, ref, label=f"edge {dtype} path{path}")
    # full ties: the kept set is the 30 lowest indices
    r = 5
    assert sorted(gpu["kept_ids"][r, :30].tolist()) == list(range(30))
    s.close()


def _wide_f32_batch(rng):
    """fp32 rows of 2049 to 4096 logits (the warp path's two staged passes):
    gaussian, spiked, full ties (more candidates than the sorted set holds),
    a NaN or +inf in the second pass only, -inf everywhere but the second
    pass, and misaligned starts."""
    rows = []
    nrm = lambda n, sd=2.0: rng.normal(0, sd, n).astype(np.float32)
    rows += [(nrm(2049), 1.0, 30, 0.9), (nrm(3072), 1.0, 30, 0.9), (nrm(4096), 0.8, 64, 0.95),
             (nrm(3500, 0.3), 1.2, 1, 0.9), (nrm(4001), 1.0, 0, 1.0)]
    x = nrm(3072)
    x[rng.choice(3072, 4, replace=False)] += 12.0
    rows += [(x, 1.0, 30, 0.9)]
    rows += [(np.full(4096, 0.25, np.float32), 1.0, 30, 0.9)]             # full ties
    rows += [(rng.choice([0.0, 0.5, 1.0], 3333).astype(np.float32), 1.0, 64, 0.9)]
    y = nrm(3000)
    y[2900] = np.nan
    rows += [(y, 1.0, 30, 0.9)]
    y = nrm(4096)
    y[4095] = np.inf
    rows += [(y, 1.0, 30, 0.9)]
    y = np.full(3100, -np.inf, np.float32)
    y[[2100, 2500, 3099]] = [0.0, 1.0, 0.5]
    rows += [(y, 1.0, 30, 0.9)]
    rows += [(nrm(700), 1.0, 30, 0.9), (nrm(5), 1.0, 30, 0.9)]            # narrow rows beside them
    n = len(rows)
    gap = rng.integers(0, 4, n)
    offs, parts, pos = [], [], 0
    for (vals, *_), g in zip(rows, gap):
        parts.append(np.zeros(int(g), np.float32))
        pos += int(g)
        offs.append(pos)
        parts.append(vals)
        pos += vals.size
    host = {
        "dtype": "f32", "logits": np.concatenate(parts), "n_rows": n, "n_streams": n,
        "n_codebooks": 1, "row_vocab": np.array([r[0].size for r in rows], np.int32),
        "row_offsets": np.array(offs, np.int64),
        "temp": np.array([r[1] for r in rows], np.float32),
        "top_k": np.array([r[2] for r in rows], np.int32),
        "top_p": np.array([r[3] for r in rows], np.float32),
        "seed": np.arange(n, dtype=np.uint64) * np.uint64(131), "request": np.arange(n, dtype=np.uint64),
        "codebook": np.zeros(n, np.int32), "row_stream": np.arange(n, dtype=np.int32),
        "step": np.full(n, 9, np.int64), "eos_id": np.full(n, 3, np.int32),
        "feedback_slot": np.arange(n, dtype=np.int32), "feedback_len": n, "cap": 64,
    }
    host["max_row_vocab"] = int(host["row_vocab"].max())
    return host


@pytest.mark.parametrize("seed", [0, 1])
def test_wide_f32_rows_on_the_warp_path(ts, seed):
    """fp32 rows wider than 2048 stay on the warp path (one warp per row, 16
    of 32 chunk columns staged at a time) and match the oracle."""
    host = _wide_f32_batch(np.random.default_rng(40 + seed))
    ref = oracle.sample(host, max_keep=64)
    assert np.any(ref["err"] == 4)
    s = make_sampler(ts, 64)
    gpu = run_gpu(s, host, debug_keep=64)
    b = ts.DeviceBatch(host, "cuda")
    assert s.plan(b)["path"] == 1
    compare(host, gpu, ref, label=f"wide f32 {seed}")
    r = 6  # full ties: the kept set is the 30 lowest indices
    assert sorted(gpu["kept_ids"][r, :30].tolist()) == list(range(30))
    plain = run_gpu(s, host)
    assert np.array_equal(plain["ids"], gpu["ids"])
    s.close()


def test_shape_and_slot_errors(ts):
    host = workloads.make("tiny", 2)
    host["row_vocab"] = np.array([2048, 0, 2048, 2048], np.int32)
    host["row_offsets"] = np.array([0, 0, 4 * 2048 - 100, 0], np.int64)
    host["row_stream"] = np.array([0, 1, 2, 3], np.int32)
    host["feedback_slot"] = np.array([0, 1, 2, 9], np.int32)
    ref = oracle.sample(host, feedback_buf=np.full(4, -1, np.int32))
    assert list(ref["err"]) == [0, 1, 1, 8]
    s = make_sampler(ts, 64)
    gpu = run_gpu(s, host)
    compare(host, gpu, ref, label="shape errors")
    assert gpu["feedback"][0] == gpu["ids"][0] and np.all(gpu["feedback"][1:] == -1)
    s.close()


def test_zero_rows_and_host_errors(ts):
    host = workloads.make("tiny", 0)
    s = make_sampler(ts, 64)
    batch = ts.DeviceBatch(host, "cuda")
    batch.c.n_rows = 0
    s.sample(batch)
    torch.cuda.synchronize()
    assert np.all(batch.ids() == -2)  # untouched
    batch.c.n_rows = host["n_rows"]
    batch.c.dtype = 7
    with pytest.raises(ts.SamplerError):
        s.sample(batch)
    batch.c.dtype = ts.TS_DTYPE_F32
    batch.c.max_row_vocab = ts.TS_MAX_VOCAB_F32 + 1
    with pytest.raises(ts.SamplerError):
        s.sample(batch)
    with pytest.raises(ts.SamplerError):
        ts.Sampler(0, 100)
    s.close()


# ---------------------------------------------------------------------------
# EOS starvation on the device
# ---------------------------------------------------------------------------
def test_eos_never_sampled_in_near_silence(ts):
    s = make_sampler(ts, 64)
    seen = 0
    for step in range(20):
        host = workloads.make("drama3", step)
        gpu = run_gpu(s, host)
        cb0 = np.asarray(host["codebook"]) == 0
        silent = np.isin(np.asarray(host["row_stream"]), host["silent_streams"])
        assert not np.any(gpu["eos"][cb0 & silent])
        seen += int(np.sum(cb0 & silent))
    assert seen >= 20 * 25
    # positive control: an EOS inside the nucleus is drawn
    host = workloads.make("drama3", 0)
    x = workloads.logits_as_f32(host).copy()
    for st in host["silent_streams"]:
        r = int(st) * 10
        x[host["row_offsets"][r] + 4095] = 20.0
    host["logits"] = workloads.to_bf16_bits(x)
    gpu = run_gpu(s, host)
    ref = oracle.sample(host, max_keep=64)
    compare(host, gpu, ref, label="eos control")
    assert np.sum(gpu["eos"]) > 0
    s.close()


# ---------------------------------------------------------------------------
# determinism and CUDA graphs
# ---------------------------------------------------------------------------
def test_graph_capture_matches_eager(ts):
    host = workloads.make("drama3", 3)
    s = make_sampler(ts, 64)
    eager = run_gpu(s, host)
    again = run_gpu(s, host)
    assert np.array_equal(eager["ids"], again["ids"])
    batch = ts.DeviceBatch(host, "cuda")
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        s.sample(batch)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        s.sample(batch)
    batch.out_ids.fill_(-5)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(batch.ids(), eager["ids"])
    s.close()


def test_resume_from_a_step(ts):
    """The sampler keeps no state between steps: restarting at step k from
    (seed, request, step) alone reproduces the continuous run's ids, EOS flags
    and frames from step k on."""
    host = workloads.make("qwen3tts", 0)
    logits = [torch.from_numpy(np.ascontiguousarray(workloads.make("qwen3tts", i)["logits"])
                               .view(np.int16)).cuda() for i in range(4)]
    steps, k = 60, 30

    def run(first, count):
        h = dict(host)
        h["step"] = np.full(host["n_streams"], first, np.int64)
        s = make_sampler(ts, host["cap"])
        b = ts.DeviceBatch(h, "cuda")
        ids, eos, frames = [], [], []
        for i in range(count):
            b.set_logits(logits[(first + i) % 4])  # the logits of absolute step first + i
            s.sample(b)
            ts.ts_advance_steps(b.step)
            ids.append(b.out_ids.clone())
            eos.append(b.out_eos.clone())
            frames.append(b.feedback.clone())
        torch.cuda.synchronize()
        assert s.read_status() == 0
        s.close()
        return [torch.stack(x).cpu().numpy() for x in (ids, eos, frames)]

    full = run(0, steps)
    resumed = run(k, steps - k)
    for a, b in zip(full, resumed):
        assert np.array_equal(a[k:], b)


@pytest.mark.parametrize("name,steps", [("tiny", 500), ("qwen3tts", 40), ("drama3", 500)])
def test_graph_loop_with_feedback(ts, name, steps):
    """`steps` decode steps captured as one graph: ts_sample then
    ts_advance_steps per step; every step's ids checked against the oracle."""
    host = workloads.make(name, 0)
    n = host["n_rows"]
    s = make_sampler(ts, host["cap"])
    batch = ts.DeviceBatch(host, "cuda")
    logits = [torch.from_numpy(np.ascontiguousarray(
        workloads.make(name, i)["logits"]).view(np.int16 if host["dtype"] == "bf16" else np.float32)
    ).cuda() for i in range(min(steps, 4))]
    out = torch.full((steps, n), -3, dtype=torch.int32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(steps):
            batch.set_logits(logits[i % len(logits)])
            batch.c.out_ids = out[i].data_ptr()
            s.sample(batch)
            ts.ts_advance_steps(batch.step)
    g.replay()
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.all(batch.step.cpu().numpy() == steps)
    assert np.array_equal(batch.feedback.cpu().numpy(), got[-1])
    check = range(steps) if n * steps <= 4000 else range(0, steps, max(1, steps // 8))
    n_safe = n_checked = 0
    for i in check:
        h = workloads.make(name, i % len(logits))
        h["step"] = np.full(host["n_streams"], i, np.int64)
        ref = oracle.sample(h, max_keep=64, n_threads=8)
        safe = ref["margin"] > 1e-5
        assert np.array_equal(got[i][safe], ref["ids"][safe]), i
        n_safe += int(safe.sum())
        n_checked += n
    # the boundary rule must leave most rows checked
    assert n_safe >= 0.9 * n_checked, (n_safe, n_checked)
    assert s.read_status() == 0
    s.close()


def test_sample_host_matches_the_device_call(ts):
    """ts_sample_host (host logits in, host ids and EOS flags out, one call)
    gives the ids and flags of ts_sample on the same logits and steps, advances
    the steps the same way, and refuses a NULL host buffer before queueing
    anything."""
    import ctypes
    hosts = [workloads.make("drama3", i) for i in range(3)]
    host = hosts[0]
    n = int(host["n_rows"])
    s = make_sampler(ts, host["cap"])
    dev = ts.DeviceBatch(host, "cuda", advance_steps=True)
    hb = ts.DeviceBatch(host, "cuda", advance_steps=True)
    pinned = [torch.from_numpy(np.ascontiguousarray(h["logits"]).view(np.int16)).pin_memory()
              for h in hosts]
    ids = torch.empty(n, dtype=torch.int32).pin_memory()
    eos = torch.empty(n, dtype=torch.uint8).pin_memory()
    for i in range(3):
        dev.set_logits(pinned[i].cuda())
        s.sample(dev)
        torch.cuda.synchronize()
        ts.ts_sample_host(s.handle, hb, pinned[i], ids, eos)
        assert np.array_equal(ids.numpy(), dev.ids()), i
        assert np.array_equal(eos.numpy(), dev.eos()), i
        assert torch.equal(hb.logits.cpu(), pinned[i])
    assert np.array_equal(hb.step.cpu().numpy(), dev.step.cpu().numpy())
    assert s.read_status() == 0
    # numpy host buffers (pageable) work too
    ids_np = np.zeros(n, np.int32)
    eos_np = np.zeros(n, np.uint8)
    ts.ts_sample_host(s.handle, hb, pinned[0].numpy(), ids_np, eos_np)
    ref = oracle.sample(dict(host, step=np.asarray(host["step"]) + 3), max_keep=64, n_threads=8)
    safe = ref["margin"] > 1e-5
    assert safe.sum() >= 0.98 * n
    assert np.array_equal(ids_np[safe], ref["ids"][safe])
    st = ts.library().ts_sample_host(s.handle, ctypes.byref(hb.c), None, ids.data_ptr(),
                                     eos.data_ptr(), None)
    assert st == ts.TS_ERR_INVALID_ARG
    s.close()
