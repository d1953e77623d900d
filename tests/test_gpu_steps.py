"""The fused step advance, the multi-step launch (ts_sample_steps) and the
resident grid that walks several rows per row group, through the C ABI.

* ts_batch.advance_steps: the step counters grow by one per call, inside the
  warp path's own launch (its last block) or by one more launch on the other
  paths; ids equal those of ts_sample followed by ts_advance_steps.
* ts_batch.step_out: calls that read one step array and write the advanced
  steps to another, swapped after each call, equal in-place advancing.
* ts_sample_steps: R steps' logits in one buffer, sampled by one launch; every
  step's ids, EOS flags and frame equal R separate ts_sample calls and, on
  sampled steps, the oracle.
* ready flags: a flag that never comes gives the step's rows -1 and the
  TS_ROW_NOT_READY bit within the time limit; flags set by the host while the
  launch runs are waited for.  Nothing here makes a kernel wait on another
  kernel.
"""
import threading
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import codebook_token_sampling_gb300 as mod
    return mod


def _np_dtype(host):
    return np.int16 if host["dtype"] == "bf16" else np.float32


def _stacked(name, steps, first=0):
    """`steps` consecutive steps of a workload: the first step's host batch and
    one device buffer holding every step's logits back to back."""
    hosts = [workloads.make(name, first + i) for i in range(steps)]
    flat = np.concatenate([np.ascontiguousarray(h["logits"]) for h in hosts])
    buf = torch.from_numpy(flat.view(_np_dtype(hosts[0]))).cuda()
    return hosts, buf, int(np.asarray(hosts[0]["logits"]).size)


@pytest.mark.parametrize("path", [1, 2, 4])
def test_fused_advance_matches_separate(ts, path):
    """Ten steps with advance_steps set vs ts_sample + ts_advance_steps."""
    name = "drama3" if path == 1 else "mixed"
    host = workloads.make(name, 0)
    logits = [torch.from_numpy(np.ascontiguousarray(workloads.make(name, i)["logits"])
                               .view(_np_dtype(host))).cuda() for i in range(3)]
    outs = []
    for fused in (True, False):
        s = ts.Sampler(0, host["cap"])
        if path == 4:
            s.reserve(int(host["n_rows"]), int(host["max_row_vocab"]))
        s.set_option(ts.TS_OPT_PATH, path)
        b = ts.DeviceBatch(host, "cuda", advance_steps=fused)
        ids = []
        for i in range(10):
            b.set_logits(logits[i % 3])
            s.sample(b)
            if not fused:
                ts.ts_advance_steps(b.step)
            ids.append(b.out_ids.clone())
        torch.cuda.synchronize()
        assert s.read_status() == 0
        assert np.all(b.step.cpu().numpy() == np.asarray(host["step"]) + 10)
        outs.append(torch.stack(ids).cpu().numpy())
        s.close()
    assert np.array_equal(outs[0], outs[1])
    # step 7's rows against the oracle (step counters 7, logits of step 7 mod 3)
    h = workloads.make(name, 7 % 3)
    h["step"] = np.asarray(host["step"]) + 7
    ref = oracle.sample(h, max_keep=h["cap"], n_threads=8)
    safe = ref["margin"] > 1e-5
    assert safe.sum() >= 0.9 * h["n_rows"]
    assert np.array_equal(outs[0][7][safe], ref["ids"][safe])


@pytest.mark.parametrize("wpr", [0, 1, 2, 4])
@pytest.mark.parametrize("name,steps", [("drama3", 6), ("qwen3tts", 5), ("tiny", 9)])
def test_sample_steps_matches_single_steps(ts, name, steps, wpr):
    hosts, buf, per_step = _stacked(name, steps)
    host = hosts[0]
    n = int(host["n_rows"])
    s = ts.Sampler(0, host["cap"])
    if wpr:
        s.set_option(ts.TS_OPT_WARPS_PER_ROW, wpr)
    # separate calls, one per step
    single = ts.DeviceBatch(host, "cuda")
    want_ids, want_eos, want_fb = [], [], []
    for i in range(steps):
        single.set_logits(buf[i * per_step:(i + 1) * per_step])
        s.sample(single)
        ts.ts_advance_steps(single.step)
        want_ids.append(single.out_ids.clone())
        want_eos.append(single.out_eos.clone())
        want_fb.append(single.feedback.clone())
    # one launch over every step
    multi = ts.DeviceBatch(host, "cuda", advance_steps=True)
    multi.set_logits(buf)
    out_ids = torch.full((steps, n), -3, dtype=torch.int32, device="cuda")
    out_eos = torch.zeros((steps, n), dtype=torch.uint8, device="cuda")
    fb_len = int(host["feedback_len"])
    frames = torch.full((steps, fb_len), -3, dtype=torch.int32, device="cuda")
    multi.c.out_ids = out_ids.data_ptr()
    multi.c.out_eos = out_eos.data_ptr()
    multi.c.feedback_buf = frames.data_ptr()
    s.sample_steps(multi, steps, logits_step_stride=per_step, out_step_stride=n,
                   feedback_step_stride=fb_len)
    torch.cuda.synchronize()
    assert s.read_status() == 0
    assert np.array_equal(out_ids.cpu().numpy(), torch.stack(want_ids).cpu().numpy())
    assert np.array_equal(out_eos.cpu().numpy(), torch.stack(want_eos).cpu().numpy())
    assert np.array_equal(frames.cpu().numpy(), torch.stack(want_fb).cpu().numpy())
    assert np.all(multi.step.cpu().numpy() == np.asarray(host["step"]) + steps)
    # the last step against the oracle
    h = dict(hosts[-1])
    h["step"] = np.asarray(host["step"]) + steps - 1
    ref = oracle.sample(h, max_keep=h["cap"], n_threads=8)
    safe = ref["margin"] > 1e-5
    assert safe.sum() >= 0.9 * n
    assert np.array_equal(out_ids.cpu().numpy()[-1][safe], ref["ids"][safe])
    s.close()


def test_sample_steps_wide_f32(ts):
    """The qwen3tts frame with fp32 logits (rows of 3072 and 2048: the warp
    path's 32-column fp32 variant, two staged passes per 3072-wide row): one
    launch over five steps equals five separate calls and the oracle."""
    steps = 5
    hosts = []
    for i in range(steps):
        h = workloads.make("qwen3tts", i)
        h["logits"] = workloads.bf16_bits_to_f32(h["logits"])
        h["dtype"] = "f32"
        hosts.append(h)
    host = hosts[0]
    n, per_step = int(host["n_rows"]), int(host["logits"].size)
    buf = torch.from_numpy(np.concatenate([h["logits"] for h in hosts])).cuda()
    s = ts.Sampler(0, host["cap"])
    single = ts.DeviceBatch(host, "cuda")
    assert s.plan(single)["path"] == 1
    want = []
    for i in range(steps):
        single.set_logits(buf[i * per_step:(i + 1) * per_step])
        s.sample(single)
        ts.ts_advance_steps(single.step)
        want.append(single.out_ids.clone())
    multi = ts.DeviceBatch(host, "cuda", advance_steps=True)
    multi.set_logits(buf)
    out_ids = torch.full((steps, n), -3, dtype=torch.int32, device="cuda")
    out_eos = torch.zeros((steps, n), dtype=torch.uint8, device="cuda")
    multi.c.out_ids = out_ids.data_ptr()
    multi.c.out_eos = out_eos.data_ptr()
    multi.c.feedback_buf = None
    multi.c.feedback_slot = None
    multi.c.feedback_len = 0
    s.sample_steps(multi, steps, logits_step_stride=per_step, out_step_stride=n)
    torch.cuda.synchronize()
    assert s.read_status() == 0
    got = out_ids.cpu().numpy()
    assert np.array_equal(got, torch.stack(want).cpu().numpy())
    for i in (0, steps - 1):
        h = dict(hosts[i])
        h["step"] = np.asarray(host["step"]) + i
        ref = oracle.sample(h, max_keep=h["cap"], n_threads=8)
        safe = ref["margin"] > 1e-5
        assert safe.sum() >= 0.9 * n
        assert np.array_equal(got[i][safe], ref["ids"][safe])
    s.close()


def test_many_rows_per_group(ts):
    """One ts_sample call over 64 steps' rows (81,920 rows: a resident grid
    whose row groups walk many rows each) equals 64 separate calls."""
    steps = 64
    hosts, buf, per_step = _stacked("drama3", steps)
    host = hosts[0]
    n = int(host["n_rows"])
    s = ts.Sampler(0, host["cap"])
    # the 64 steps as one batch: rows r + i n read step i's logits
    big = {k: v for k, v in host.items()}
    big["logits"] = np.concatenate([np.asarray(h["logits"]) for h in hosts])
    for k in ("row_vocab", "temp", "top_k", "top_p", "seed", "request", "codebook", "eos_id"):
        big[k] = np.tile(np.asarray(host[k]), steps)
    big["row_offsets"] = np.concatenate([np.asarray(host["row_offsets"]) + i * per_step
                                         for i in range(steps)])
    big["row_stream"] = np.concatenate([np.asarray(host["row_stream"]) + i * host["n_streams"]
                                        for i in range(steps)]).astype(np.int32)
    big["step"] = np.concatenate([np.asarray(host["step"]) + i for i in range(steps)])
    big["n_streams"] = host["n_streams"] * steps
    big["n_rows"] = n * steps
    big["feedback_slot"] = np.arange(n * steps, dtype=np.int32)
    big["feedback_len"] = n * steps
    b = ts.DeviceBatch(big, "cuda")
    plan = s.plan(b)
    assert plan["path"] == 1 and plan["grid"] * (4 // plan["ctas_per_row"]) < n * steps
    s.sample(b)
    single = ts.DeviceBatch(host, "cuda")
    want = []
    for i in range(steps):
        single.set_logits(buf[i * per_step:(i + 1) * per_step])
        s.sample(single)
        ts.ts_advance_steps(single.step)
        want.append(single.out_ids.clone())
    torch.cuda.synchronize()
    assert s.read_status() == 0
    assert np.array_equal(b.ids(), torch.cat(want).cpu().numpy())
    s.close()


def test_ready_flag_that_never_comes(ts):
    """Steps 0, 1, 3 and 4 are ready, step 2 never is: step 2's rows get -1
    and TS_ROW_NOT_READY within about one limit; the others are sampled."""
    steps = 5
    hosts, buf, per_step = _stacked("drama3", steps)
    host = hosts[0]
    n = int(host["n_rows"])
    s = ts.Sampler(0, host["cap"])
    b = ts.DeviceBatch(host, "cuda", feedback=False)
    b.set_logits(buf)
    out_ids = torch.full((steps, n), -3, dtype=torch.int32, device="cuda")
    out_eos = torch.full((steps, n), 7, dtype=torch.uint8, device="cuda")
    b.c.out_ids = out_ids.data_ptr()
    b.c.out_eos = out_eos.data_ptr()
    ready = torch.tensor([1, 1, 0, 1, 1], dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    s.sample_steps(b, steps, logits_step_stride=per_step, out_step_stride=n, ready=ready,
                   ready_timeout_ns=2_000_000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0
    assert s.read_status() == ts.TS_ROW_NOT_READY
    got = out_ids.cpu().numpy()
    assert np.all(got[2] == -1) and np.all(out_eos.cpu().numpy()[2] == 0)
    assert np.all(got[[0, 1, 3, 4]] >= 0)
    for i in (0, 1, 3, 4):
        h = dict(hosts[i])
        h["step"] = np.asarray(host["step"]) + i
        ref = oracle.sample(h, max_keep=64, n_threads=8)
        safe = ref["margin"] > 1e-5
        assert np.array_equal(got[i][safe], ref["ids"][safe])
    s.close()


def test_ready_flags_set_by_the_host(ts):
    """The launch starts with no step ready; a host thread sets the flags one
    by one in pinned memory; every step is sampled as if it had been ready."""
    steps = 4
    hosts, buf, per_step = _stacked("qwen3tts", steps)
    host = hosts[0]
    n = int(host["n_rows"])
    s = ts.Sampler(0, host["cap"])
    b = ts.DeviceBatch(host, "cuda", feedback=False)
    b.set_logits(buf)
    out_ids = torch.full((steps, n), -3, dtype=torch.int32, device="cuda")
    b.c.out_ids = out_ids.data_ptr()
    eos = torch.zeros((steps, n), dtype=torch.uint8, device="cuda")
    b.c.out_eos = eos.data_ptr()
    flags = torch.zeros(steps, dtype=torch.int32).pin_memory()
    torch.cuda.synchronize()

    def producer():
        for i in range(steps):
            time.sleep(0.002)
            flags[i] = 1

    th = threading.Thread(target=producer)
    s.sample_steps(b, steps, logits_step_stride=per_step, out_step_stride=n, ready=flags,
                   ready_timeout_ns=2_000_000_000)
    th.start()
    torch.cuda.synchronize()
    th.join()
    assert s.read_status() == 0
    # the same launch with every flag already set
    ready = torch.ones(steps, dtype=torch.int32, device="cuda")
    want = torch.full((steps, n), -3, dtype=torch.int32, device="cuda")
    b.c.out_ids = want.data_ptr()
    s.sample_steps(b, steps, logits_step_stride=per_step, out_step_stride=n, ready=ready)
    torch.cuda.synchronize()
    assert np.array_equal(out_ids.cpu().numpy(), want.cpu().numpy())
    assert np.all(out_ids.cpu().numpy() >= 0)
    s.close()


def test_sample_steps_limits(ts):
    """Outside the warp path, or with bad strides: a status, nothing launched."""
    host = workloads.make("mixed", 0)  # cap 4096: not the warp path
    s = ts.Sampler(0, host["cap"])
    b = ts.DeviceBatch(host, "cuda")
    with pytest.raises(ts.SamplerError) as e:
        s.sample_steps(b, 2, logits_step_stride=0, out_step_stride=host["n_rows"],
                       feedback_step_stride=host["feedback_len"])
    assert e.value.status == ts.TS_ERR_UNSUPPORTED
    s.close()
    host = workloads.make("drama3", 0)
    s = ts.Sampler(0, host["cap"])
    b = ts.DeviceBatch(host, "cuda")
    for kw in ({"n_steps": 0, "out_step_stride": host["n_rows"]},
               {"n_steps": 2, "out_step_stride": host["n_rows"] - 1},
               {"n_steps": 2, "out_step_stride": host["n_rows"], "feedback_step_stride": 1}):
        n_steps = kw.pop("n_steps")
        with pytest.raises(ts.SamplerError) as e:
            s.sample_steps(b, n_steps, logits_step_stride=0, **kw)
        assert e.value.status == ts.TS_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert np.all(b.ids() == -2)
    s.close()


def _wide_edge_rows(n, seed):
    """n rows of 2,900 to 4,096 bf16 logits at misaligned offsets: gaussian
    rows with assorted parameters, huge ties (the slow path), -inf inside the
    top-k set, and a few NaN / +inf rows."""
    rng = np.random.default_rng(seed)
    vals, offs, vocab, pos = [], [], [], 0
    temp, top_k, top_p = [], [], []
    for r in range(n):
        v = int(rng.choice([4096, 4095, 4000, 2900]))
        kind = r % 50
        if kind == 7:
            x = np.full(v, 0.75, np.float32)                       # all tied
        elif kind == 13:
            x = rng.choice([0.0, 0.5], v).astype(np.float32)        # huge ties
        elif kind == 21:
            x = np.full(v, -np.inf, np.float32)
            x[rng.choice(v, 5, replace=False)] = rng.normal(0, 1, 5)
        elif kind == 29:
            x = rng.normal(0, 2, v).astype(np.float32)
            x[int(rng.integers(0, v))] = np.nan
        elif kind == 31:
            x = rng.normal(0, 2, v).astype(np.float32)
            x[int(rng.integers(0, v))] = np.inf
        else:
            x = rng.normal(0, 2, v).astype(np.float32)
        g = int(rng.integers(0, 7))
        vals.append(np.zeros(g, np.float32))
        pos += g
        offs.append(pos)
        vals.append(x)
        pos += v
        vocab.append(v)
        temp.append(float(rng.choice([1.0, 0.7, 0.0])))
        top_k.append(int(rng.choice([30, 64, 1, 0])))
        top_p.append(float(rng.choice([0.9, 1.0, 0.5])))
    flat = np.concatenate(vals)
    logits = workloads.to_bf16_bits(flat)
    logits[np.isnan(flat)] = 0x7FC0
    return {
        "dtype": "bf16", "logits": logits, "n_rows": n, "n_streams": n, "n_codebooks": 1,
        "row_vocab": np.array(vocab, np.int32), "row_offsets": np.array(offs, np.int64),
        "max_row_vocab": 4096, "temp": np.array(temp, np.float32),
        "top_k": np.array(top_k, np.int32), "top_p": np.array(top_p, np.float32),
        "seed": rng.integers(0, 2**63, n, dtype=np.uint64), "request": np.arange(n, dtype=np.uint64),
        "codebook": np.zeros(n, np.int32), "row_stream": np.arange(n, dtype=np.int32),
        "step": np.full(n, 4, np.int64), "eos_id": np.full(n, 3, np.int32),
        "feedback_slot": np.arange(n, dtype=np.int32), "feedback_len": n, "cap": 64,
    }


def test_segmented_stage_matches_unsegmented(ts):
    """A launch with more rows than the GPU holds at once stages 4096-wide rows
    in two segments (the second read again from L2; the slow path reads the
    row back from memory).  Its ids, EOS flags, frame and status equal those
    of the same rows sampled in slices small enough for the unsegmented
    kernel, and a sample of rows equals the oracle."""
    from parity import sub_batch
    n = 12000
    host = _wide_edge_rows(n, 77)
    s = ts.Sampler(0, 64)
    big = run_gpu(s, host)
    slices = []
    for a in range(0, n, 2000):
        h = sub_batch(host, np.arange(a, min(n, a + 2000)))
        h["step"] = np.full(h["n_rows"], 4, np.int64)
        h["max_row_vocab"] = 4096
        plan = s.plan(ts.DeviceBatch(h, "cuda"))
        assert plan["path"] == 1 and plan["grid"] * 4 // plan["ctas_per_row"] >= h["n_rows"]
        slices.append(run_gpu(s, h))
    assert np.array_equal(big["ids"], np.concatenate([x["ids"] for x in slices]))
    assert np.array_equal(big["eos"], np.concatenate([x["eos"] for x in slices]))
    assert big["status"] == (ts.TS_ROW_NONFINITE if big["status"] else 0)
    assert big["status"] == ts.TS_ROW_NONFINITE  # the NaN / +inf rows
    rows = np.concatenate([np.arange(0, 400), np.arange(n - 100, n)])
    sub = sub_batch(host, rows)
    sub["max_row_vocab"] = 4096
    ref = oracle.sample(sub, max_keep=64, n_threads=8)
    safe = ref["margin"] > 1e-5
    assert safe.sum() >= 0.9 * rows.size
    assert np.array_equal(big["ids"][rows][safe], ref["ids"][safe])
    assert np.all(big["ids"][rows][ref["err"] != 0] == -1)
    s.close()


@pytest.mark.parametrize("name", ["drama3", "qwen3tts"])
def test_per_level_calls_match_the_frame_call(ts, name):
    """A frame sampled level by level (one ts_sample call per codebook, as the
    tower samples them in order; the last call advances the steps) equals the
    one-call frame: ids, EOS flags and the frame, for three frames."""
    import bench
    hosts = [workloads.make(name, i) for i in range(3)]
    host = hosts[0]
    s = ts.Sampler(0, host["cap"])
    whole = ts.DeviceBatch(host, "cuda", advance_steps=True)
    levels = bench.level_batches(host, "cuda")
    frame = levels[0].feedback
    for b in levels[1:]:
        b.feedback, b.c.feedback_buf = frame, frame.data_ptr()
        b.step, b.c.step = levels[0].step, levels[0].step.data_ptr()
    n = int(host["n_rows"])
    cb = np.asarray(host["codebook"])
    for h in hosts:
        lg = torch.from_numpy(np.ascontiguousarray(h["logits"]).view(np.int16)).cuda()
        whole.set_logits(lg)
        s.sample(whole)
        got_ids = np.zeros(n, np.int32)
        got_eos = np.zeros(n, np.uint8)
        for q, b in enumerate(levels):
            b.set_logits(lg)
            s.sample(b)
        torch.cuda.synchronize()
        for q, b in enumerate(levels):
            got_ids[cb == q] = b.ids()
            got_eos[cb == q] = b.eos()
        assert np.array_equal(got_ids, whole.ids())
        assert np.array_equal(got_eos, whole.eos())
        assert np.array_equal(frame.cpu().numpy(), whole.feedback.cpu().numpy())
    assert np.array_equal(levels[0].step.cpu().numpy(), whole.step.cpu().numpy())
    assert s.read_status() == 0
    s.close()


def _with_idle_streams(host, extra):
    """The batch with `extra` more streams that no row belongs to (their steps
    must advance all the same)."""
    h = dict(host)
    n = int(h["n_streams"]) + extra
    h["n_streams"] = n
    h["step"] = np.concatenate([np.asarray(host["step"], np.int64),
                                np.arange(extra, dtype=np.int64) * 7 + 100])
    return h


@pytest.mark.parametrize("path", [1, 2])
def test_two_step_arrays_match_in_place(ts, path):
    """step_out: eight calls that read one step array and write the other,
    swapped after each call, give the ids, EOS flags and steps of eight calls
    advancing one array in place; streams without rows advance too."""
    name = "drama3" if path == 1 else "mixed"
    host = _with_idle_streams(workloads.make(name, 0), 37)
    logits = [torch.from_numpy(np.ascontiguousarray(workloads.make(name, i)["logits"])
                               .view(_np_dtype(host))).cuda() for i in range(3)]
    runs = []
    for double in (True, False):
        s = ts.Sampler(0, host["cap"])
        s.set_option(ts.TS_OPT_PATH, path)
        b = ts.DeviceBatch(host, "cuda", advance_steps=True, double_steps=double)
        ids, eos = [], []
        for i in range(8):
            b.set_logits(logits[i % 3])
            s.sample(b)
            if double:
                b.swap_steps()
            ids.append(b.out_ids.clone())
            eos.append(b.out_eos.clone())
        torch.cuda.synchronize()
        assert s.read_status() == 0
        runs.append((torch.stack(ids).cpu().numpy(), torch.stack(eos).cpu().numpy(),
                     b.step.cpu().numpy()))
        s.close()
    (ia, ea, sa), (ib, eb, sb) = runs
    assert np.array_equal(ia, ib) and np.array_equal(ea, eb)
    assert np.array_equal(sa, sb)
    assert np.array_equal(sa, np.asarray(host["step"]) + 8)


def test_two_step_arrays_with_several_steps_per_launch(ts):
    """ts_sample_steps with step_out: the launch reads step and writes
    step + R to the other array, leaving step as it was."""
    steps = 3
    hosts, buf, per_step = _stacked("qwen3tts", steps)
    host = _with_idle_streams(hosts[0], 5)
    n = int(host["n_rows"])
    s = ts.Sampler(0, host["cap"])
    b = ts.DeviceBatch(host, "cuda", feedback=False, advance_steps=True, double_steps=True)
    b.set_logits(buf)
    out = torch.full((steps, n), -3, dtype=torch.int32, device="cuda")
    eos = torch.zeros((steps, n), dtype=torch.uint8, device="cuda")
    b.c.out_ids, b.c.out_eos = out.data_ptr(), eos.data_ptr()
    before = b.step.cpu().numpy().copy()
    s.sample_steps(b, steps, logits_step_stride=per_step, out_step_stride=n)
    torch.cuda.synchronize()
    assert s.read_status() == 0
    assert np.array_equal(b.step.cpu().numpy(), before)
    assert np.array_equal(b.step_next.cpu().numpy(), before + steps)
    got = out.cpu().numpy()
    for i in range(steps):
        h = dict(hosts[i])
        h["step"] = np.asarray(hosts[0]["step"]) + i
        ref = oracle.sample(h, max_keep=64, n_threads=8)
        safe = ref["margin"] > 1e-5
        assert np.array_equal(got[i][safe], ref["ids"][safe])
    s.close()


def test_overlapping_step_arrays_are_refused(ts):
    host = workloads.make("drama3", 0)
    s = ts.Sampler(0, 64)
    b = ts.DeviceBatch(host, "cuda", advance_steps=True, double_steps=True)
    b.c.step_out = b.step.data_ptr() + 8  # one entry past step: overlaps it
    with pytest.raises(ts.SamplerError) as e:
        s.sample(b)
    assert e.value.status == ts.TS_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert np.all(b.ids() == -2)
    s.close()
