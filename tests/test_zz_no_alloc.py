"""ts_sample_noalloc, the entry point for callers that cannot allocate device
memory, against ts_sample through the C ABI.

Its workspace is the library's static scratch array, shared by every call and
left holding the previous call's contents, so each test makes two calls in a
row on one stream (the second over what the first left behind) and checks
both against ts_sample on a sampler of the same cap: ids, EOS flags, the
frame write-back and the row error bits must be identical.  The first call in
a process also does the per-device set-up.  This file is collected last, so
it runs both alone in a fresh process and after every other test.
"""
import numpy as np
import pytest

import workloads
from parity import sub_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import codebook_token_sampling_gb300 as mod
    return mod


def _existing(ts, host):
    """ids, eos, write-back and status bits of ts_sample (default plan)."""
    import torch
    s = ts.Sampler(0, int(host["cap"]))
    b = ts.DeviceBatch(host, "cuda")
    s.sample(b)
    torch.cuda.synchronize()
    out = {"ids": b.ids(), "eos": b.eos(), "feedback": b.feedback.cpu().numpy(),
           "status": s.read_status()}
    s.close()
    return out


def _noalloc_pair(ts, hosts):
    """Two ts_sample_noalloc calls in a row on one stream, then one sync."""
    import torch
    batches, stats = [], []
    for h in hosts:
        batches.append(ts.DeviceBatch(h, "cuda"))
        stats.append(torch.zeros(1, dtype=torch.int32, device="cuda"))
    for h, b, st in zip(hosts, batches, stats):
        ts.ts_sample_noalloc(b, int(h["cap"]), st)
    torch.cuda.synchronize()
    return [{"ids": b.ids(), "eos": b.eos(), "feedback": b.feedback.cpu().numpy(),
             "status": int(st.cpu().numpy()[0]) & 0xFFFFFFFF}
            for b, st in zip(batches, stats)]


def _assert_same(got, want, label):
    for key in ("ids", "eos", "feedback"):
        assert np.array_equal(got[key], want[key]), (label, key)
    assert got["status"] == want["status"], (label, got["status"], want["status"])


def _edge_batch(seed):
    """40 rows of 30,000 bf16 logits: ordinary rows plus a NaN row, a row
    with no finite logit, a +inf row and all-tied rows (status bits set)."""
    rng = np.random.default_rng(seed)
    n, v = 40, 30000
    vals = rng.normal(0, 3, (n, v)).astype(np.float32)
    vals[3, 1234] = np.nan
    vals[7, :] = -np.inf
    vals[11, 5] = np.inf
    vals[13, :] = 0.5
    flat = vals.reshape(-1)
    logits = workloads.to_bf16_bits(flat)
    logits[np.isnan(flat)] = 0x7FC0
    host = {
        "dtype": "bf16", "logits": logits, "n_rows": n, "n_streams": n, "n_codebooks": 1,
        "row_vocab": np.full(n, v, np.int32),
        "row_offsets": np.arange(n, dtype=np.int64) * v,
        "temp": rng.uniform(0.5, 1.5, n).astype(np.float32),
        "top_k": rng.choice([1, 30, 64, 500, 0], n).astype(np.int32),
        "top_p": rng.uniform(0.5, 1.0, n).astype(np.float32),
        "seed": rng.integers(0, 2**63, n, dtype=np.uint64),
        "request": np.arange(n, dtype=np.uint64),
        "codebook": np.zeros(n, np.int32), "row_stream": np.arange(n, dtype=np.int32),
        "step": np.full(n, 9, np.int64), "eos_id": np.full(n, 17, np.int32),
        "feedback_slot": np.arange(n, dtype=np.int32), "feedback_len": n, "cap": 512,
        "max_row_vocab": v,
    }
    return host


def test_noalloc_stress_then_tower_rows(ts):
    """24 rows of 151,936 logits, then 64 rows of the 4096-wide codebook rows."""
    first = workloads.make("stress", 11, rows=24)
    second = sub_batch(workloads.make("drama3", 4), np.arange(64))
    got = _noalloc_pair(ts, [first, second])
    _assert_same(got[0], _existing(ts, first), "stress 24 rows")
    _assert_same(got[1], _existing(ts, second), "64 tower rows")


def test_noalloc_small_then_large_stress(ts):
    """8 rows of 151,936 logits (few CTAs: the streaming CTAs sample the rows
    themselves, no threshold kernel), then 32 rows (the threshold kernel
    runs): the row counters left by the first call must not leak into the
    second."""
    first = workloads.make("stress", 21, rows=8)
    second = workloads.make("stress", 22, rows=32)
    got = _noalloc_pair(ts, [first, second])
    _assert_same(got[0], _existing(ts, first), "stress 8 rows")
    _assert_same(got[1], _existing(ts, second), "stress 32 rows")


def test_noalloc_one_row_then_eight_rows(ts):
    """1 row of 151,936 logits, then 8 rows: both calls small enough that the
    streaming CTAs sample the rows themselves (no threshold kernel zeroes the
    counters), and the second call uses rows the first did not.  Their
    counters must start at zero all the same."""
    import torch
    first = workloads.make("stress", 23, rows=1)
    second = workloads.make("stress", 24, rows=8)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for h in (first, second):  # the geometry that skips the threshold kernel
        s = ts.Sampler(0, int(h["cap"]))
        s.reserve(int(h["n_rows"]), int(h["max_row_vocab"]))
        plan = s.plan(ts.DeviceBatch(h, "cuda"))
        assert plan["path"] == 4 and h["n_rows"] * plan["ctas_per_row"] <= 2 * sms, plan
        s.close()
    got = _noalloc_pair(ts, [first, second])
    _assert_same(got[0], _existing(ts, first), "stress 1 row")
    _assert_same(got[1], _existing(ts, second), "stress 8 rows")


def test_noalloc_edge_rows_then_widest_rows(ts):
    """Rows with errors, then 64 rows of the widest bf16 vocabulary (the
    largest call the scratch takes)."""
    first = _edge_batch(5)
    rng = np.random.default_rng(6)
    v = ts.TS_MAX_VOCAB_BF16
    second = workloads.make("stress", 12, rows=64)
    second = dict(second)
    second["logits"] = workloads.to_bf16_bits(rng.normal(0, 2, 64 * v).astype(np.float32))
    second["row_vocab"] = np.full(64, v, np.int32)
    second["row_offsets"] = np.arange(64, dtype=np.int64) * v
    second["max_row_vocab"] = v
    got = _noalloc_pair(ts, [first, second])
    want0 = _existing(ts, first)
    assert want0["status"] != 0
    _assert_same(got[0], want0, "edge rows")
    _assert_same(got[1], _existing(ts, second), "64 rows of 163,840")


def test_noalloc_limits(ts):
    """Beyond the limits: a clear TS_ERR_UNSUPPORTED and nothing launched."""
    import torch
    host = sub_batch(workloads.make("drama3", 1), np.arange(65))
    b = ts.DeviceBatch(host, "cuda")
    with pytest.raises(ts.SamplerError) as e:
        ts.ts_sample_noalloc(b, 64)
    assert e.value.status == ts.TS_ERR_UNSUPPORTED and "64 rows" in str(e.value)
    f32 = dict(sub_batch(workloads.make("drama3", 1), np.arange(4)))
    f32["dtype"] = "f32"
    f32["logits"] = np.zeros(int(np.sum(f32["row_vocab"])), np.float32)
    bf = ts.DeviceBatch(f32, "cuda")
    with pytest.raises(ts.SamplerError) as e:
        ts.ts_sample_noalloc(bf, 64)
    assert e.value.status == ts.TS_ERR_UNSUPPORTED and "bf16" in str(e.value)
    torch.cuda.synchronize()
    assert np.all(b.ids() == -2) and np.all(bf.ids() == -2)
    empty = sub_batch(workloads.make("drama3", 1), np.arange(0))
    ts.ts_sample_noalloc(ts.DeviceBatch(empty, "cuda"), 64)  # set-up only
