"""Finished streams on the GPU against the oracle, through the C ABI: a stream
whose EOS was drawn pads its rows from the next step on (reason stop), a
stream at its length cap pads (reason length), as the handbook's EOS-starvation
section asks of the serving side (section "一个真实问题：说完了却停不下来").
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle_pins import finish_workload
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import codebook_token_sampling_gb300 as mod
    return mod


@pytest.mark.parametrize("path", [1, 2])
def test_forced_eos_and_caps_step_by_step(ts, path):
    """The oracle pin's scenario (forced EOS events, caps, a stop before the cap,
    an EOS on the cap step), nine steps, every output and the finish state."""
    steps, pad = 9, -7
    forced = {2: (1,), 5: (3,), 6: (5,), 7: (1,)}
    max_steps = np.array([100, 5, 4, 100, 100, 6], np.int64)
    s = ts.Sampler(0, 64)
    s.set_option(ts.TS_OPT_PATH, path)
    h0 = finish_workload(0, forced)
    b = ts.DeviceBatch(h0, "cuda", advance_steps=True,
                       finish={"max_steps": max_steps, "pad_id": pad})
    stop = np.full(6, -1, np.int64)
    reason = np.zeros(6, np.uint8)
    for t in range(steps):
        h = finish_workload(t, forced)
        b.set_logits(torch.from_numpy(h["logits"]).cuda())
        s.sample(b)
        torch.cuda.synchronize()
        fb = np.full(18, -9, np.int32)
        ref = oracle.sample(h, stop_step=stop, max_steps=max_steps, finish_reason=reason,
                            pad_id=pad, feedback_buf=fb, max_keep=64)
        gpu = {"ids": b.ids(), "eos": b.eos(), "status": s.read_status(),
               "feedback": b.feedback.cpu().numpy()}
        compare(h, gpu, ref, check_probs=False, label=f"finish path{path} step{t}")
        assert np.array_equal(gpu["ids"][ref["finished"] > 0], np.full(int(np.sum(ref["finished"] > 0)), pad))
        assert np.array_equal(b.stop_step.cpu().numpy(), stop), t
        assert np.array_equal(b.finish_reason.cpu().numpy(), reason), t
    assert list(reason[[1, 2, 3, 5]]) == [1, 2, 1, 2]
    s.close()


def test_drama3_500_steps_with_caps(ts):
    """500 decode steps of the 128 x 10 shape as one CUDA graph (ts_sample with
    the fused step advance and the finish state), per-stream caps from 100 to
    500 steps.  Every step is checked against the oracle run from the finish
    state the GPU held before that step (so a draw at a boundary cannot carry
    into later steps), and the GPU's state after the step against the
    oracle's on every stream whose codebook-0 row is off-boundary."""
    steps, pad = 500, -1
    host = workloads.make("drama3", 0)
    n, n_streams = int(host["n_rows"]), int(host["n_streams"])
    rng = np.random.default_rng(3)
    caps = rng.integers(100, 500, n_streams).astype(np.int64)
    s = ts.Sampler(0, 64)
    b = ts.DeviceBatch(host, "cuda", advance_steps=True, finish={"max_steps": caps, "pad_id": pad})
    n_log = 6
    logits = [torch.from_numpy(np.ascontiguousarray(workloads.make("drama3", i)["logits"])
                               .view(np.int16)).cuda() for i in range(n_log)]
    ids = torch.full((steps, n), -3, dtype=torch.int32, device="cuda")
    stops = torch.zeros((steps, n_streams), dtype=torch.int64, device="cuda")
    reasons = torch.zeros((steps, n_streams), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        warm = ts.DeviceBatch(host, "cuda", advance_steps=True,
                              finish={"max_steps": caps, "pad_id": pad})
        s.sample(warm, side)
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(steps):
            b.set_logits(logits[i % n_log])
            b.c.out_ids = ids[i].data_ptr()
            s.sample(b)
            stops[i].copy_(b.stop_step)
            reasons[i].copy_(b.finish_reason)
    g.replay()
    torch.cuda.synchronize()
    assert s.read_status() == 0
    got, st, rs = ids.cpu().numpy(), stops.cpu().numpy(), reasons.cpu().numpy()
    n_safe = n_checked = 0
    for i in range(steps):
        h = workloads.make("drama3", i % n_log)
        h["step"] = np.full(n_streams, i, np.int64)
        stop = st[i - 1].copy() if i else np.full(n_streams, -1, np.int64)
        reason = rs[i - 1].copy() if i else np.zeros(n_streams, np.uint8)
        ref = oracle.sample(h, max_keep=64, n_threads=8, stop_step=stop, max_steps=caps,
                            finish_reason=reason, pad_id=pad)
        safe = ref["margin"] > 1e-5
        assert np.array_equal(got[i][safe], ref["ids"][safe]), i
        cb0_safe = safe[::10]
        assert np.array_equal(st[i][cb0_safe], stop[cb0_safe]), i
        assert np.array_equal(rs[i][cb0_safe], reason[cb0_safe]), i
        n_safe += int(safe.sum())
        n_checked += n
    assert n_safe >= 0.99 * n_checked
    # every stream ended one way or the other: length at its cap, or stop
    final = rs[-1]
    assert np.all(final > 0)
    assert np.all((final == 2) == (st[-1] < 0))
    assert np.sum(final == 1) >= 1 and np.sum(final == 2) >= 1
    s.close()


def test_finished_streams_on_the_split_path(ts):
    """Stress rows (the split path, three kernels): streams stopped earlier and
    streams at their cap pad; the others equal the run without the state."""
    host = workloads.make("stress", 5, rows=32)
    n = int(host["n_rows"])
    s = ts.Sampler(0, 4096)
    s.reserve(n, workloads.STRESS_VOCAB)
    plain = ts.DeviceBatch(host, "cuda")
    s.sample(plain)
    t = int(host["step"][0])
    caps = np.full(n, 10**9, np.int64)
    caps[[3, 4, 5]] = t          # at the cap: length
    b = ts.DeviceBatch(host, "cuda", finish={"max_steps": caps, "pad_id": 12345})
    b.stop_step.copy_(torch.full((n,), -1, dtype=torch.int64))
    b.stop_step[[0, 1, 3]] = t - 1   # stopped earlier (stream 3: stop before length)
    b.stop_step[2] = t               # stopped at this very step: not finished yet
    assert s.plan(b)["path"] == 4
    s.sample(b)
    torch.cuda.synchronize()
    assert s.read_status() == 0
    ids, want = b.ids(), plain.ids()
    fin = np.zeros(n, bool)
    fin[[0, 1, 3, 4, 5]] = True
    assert np.all(ids[fin] == 12345) and np.all(b.eos()[fin] == 0)
    assert np.array_equal(ids[~fin], want[~fin])
    assert np.array_equal(b.feedback.cpu().numpy()[fin], ids[fin])
    reason = b.finish_reason.cpu().numpy()
    assert list(reason[[0, 1, 3, 4, 5]]) == [1, 1, 1, 2, 2] and reason[2] == 0
    s.close()


def test_sample_steps_refuses_the_finish_state(ts):
    host = workloads.make("drama3", 0)
    s = ts.Sampler(0, 64)
    b = ts.DeviceBatch(host, "cuda", finish={"max_steps": None, "pad_id": -1})
    with pytest.raises(ts.SamplerError) as e:
        s.sample_steps(b, 2, logits_step_stride=0, out_step_stride=host["n_rows"],
                       feedback_step_stride=host["feedback_len"])
    assert e.value.status == ts.TS_ERR_UNSUPPORTED
    s.close()
