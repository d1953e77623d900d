"""The wide-row paths vs the CPU oracle, through the C ABI: the cluster
kernel (path 3) and the split threshold + streaming kernels over a workspace
(path 4).

Covers the 151,936-wide stress rows on the sampled-threshold path and with
the exact re-reading path forced, every cluster size / unit count, rows whose
sample misleads the threshold (overflow, too few candidates), ties, signed
zeros, non-finite values, degenerate parameters, and the narrower workloads
forced onto the paths (all-candidates mode).  Results must also equal the
other kernel families' bit for bit.
"""
import numpy as np
import pytest

import oracle
import workloads
from parity import compare, run_gpu, sub_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import codebook_token_sampling_gb300 as mod
    return mod


def make_sampler(ts, cap, path=3, cluster=0, exact=0, host=None):
    s = ts.Sampler(0, cap)
    if path == 4:
        s.reserve(int(host["n_rows"]), int(host["max_row_vocab"]))
    s.set_option(ts.TS_OPT_PATH, path)
    if cluster:
        s.set_option(ts.TS_OPT_CLUSTER, cluster)
    if exact:
        s.set_option(ts.TS_OPT_WIDE_EXACT, 1)
    return s


def batch_from_rows(rows, *, cap, seed=0, gaps=True):
    """rows: list of (float32 values, temp, top_k, top_p); bf16 logits packed
    with random misaligned gaps."""
    rng = np.random.default_rng(seed)
    n = len(rows)
    offs, parts, pos = [], [], 0
    for vals, *_ in rows:
        g = int(rng.integers(0, 7)) if gaps else 0
        parts.append(np.zeros(g, np.float32))
        pos += g
        offs.append(pos)
        parts.append(vals)
        pos += vals.size
    flat = np.concatenate(parts)
    logits = workloads.to_bf16_bits(flat)
    logits[np.isnan(flat)] = 0x7FC0
    host = {
        "dtype": "bf16", "logits": logits, "n_rows": n, "n_streams": n, "n_codebooks": 1,
        "row_vocab": np.array([r[0].size for r in rows], np.int32),
        "row_offsets": np.array(offs, np.int64),
        "temp": np.array([r[1] for r in rows], np.float32),
        "top_k": np.array([r[2] for r in rows], np.int32),
        "top_p": np.array([r[3] for r in rows], np.float32),
        "seed": np.arange(n, dtype=np.uint64) * np.uint64(7919) + np.uint64(seed),
        "request": np.arange(n, dtype=np.uint64),
        "codebook": np.zeros(n, np.int32), "row_stream": np.arange(n, dtype=np.int32),
        "step": np.full(n, 3 + seed, np.int64), "eos_id": np.full(n, 5, np.int32),
        "feedback_slot": np.arange(n, dtype=np.int32), "feedback_len": n, "cap": cap,
    }
    host["max_row_vocab"] = int(host["row_vocab"].max())
    return host


# ---------------------------------------------------------------------------
# the stress shape: sampled threshold and forced exact path, all cluster sizes
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("exact", [0, 1])
@pytest.mark.parametrize("path,rows,cluster", [(3, 1, 0), (3, 8, 0), (3, 32, 4), (3, 6, 8),
                                               (4, 1, 0), (4, 8, 0), (4, 32, 0), (4, 6, 3),
                                               (4, 5, 16)])
def test_stress_wide(ts, path, rows, cluster, exact):
    host = workloads.make("stress", 2, rows=rows)
    ref = oracle.sample(host, max_keep=4096, n_threads=8)
    s = make_sampler(ts, 4096, path=path, cluster=cluster, exact=exact, host=host)
    gpu = run_gpu(s, host, debug_keep=4096)
    compare(host, gpu, ref, label=f"wide path{path} stress{rows} g{cluster} exact{exact}")
    s.close()


def test_stress_512_default_plans(ts):
    host = workloads.make("stress", 0, rows=512)
    s = ts.Sampler(0, 4096)
    batch = ts.DeviceBatch(host, "cuda")
    assert s.plan(batch)["path"] == 3  # no workspace: the cluster path
    s.reserve(512, workloads.STRESS_VOCAB)
    plan = s.plan(batch)
    assert plan["path"] == 4 and plan["grid"] == 512 * plan["ctas_per_row"]
    s.reserve(0, 0)
    assert s.plan(batch)["path"] == 3
    s.close()


def test_stress_512_rows_split_sampled(ts):
    """The full-size stress step on the split path, as the benchmark launches
    it; the oracle checks 48 sampled rows one by one."""
    host = workloads.make("stress", 3, rows=512)
    s = make_sampler(ts, 4096, path=4, host=host)
    gpu = run_gpu(s, host)
    assert gpu["status"] == 0
    rows = np.random.default_rng(9).choice(512, size=48, replace=False)
    ref = oracle.sample(sub_batch(host, rows), max_keep=4096, n_threads=8)
    safe = ref["margin"] > 1e-5
    # a stress row's nucleus holds thousands of CDF steps, so about 11% of
    # rows lie within 1e-5 of a boundary; most must still be checked
    assert safe.sum() >= 0.75 * rows.size
    assert np.array_equal(gpu["ids"][rows][safe], ref["ids"][safe])
    s.close()


@pytest.mark.parametrize("rows", [8, 64])
@pytest.mark.parametrize("which", [2, 3])
def test_split_refused_launch_leaves_clean_workspace(ts, rows, which):
    """A split-path call whose streaming (2) or tail (3) launch is refused on
    the host returns TS_ERR_CUDA; the next call on the same workspace is still
    oracle-exact.  The refusal is injected on the host (TS_OPT_FAIL_LAUNCH)
    before the launch is queued: nothing faults on the device.  With 8 rows
    the streaming CTAs sample the rows themselves (no threshold kernel clears
    the counters), with 64 the threshold kernel runs."""
    import torch
    first = workloads.make("stress", 31, rows=rows)
    s = make_sampler(ts, 4096, path=4, host=first)
    b = ts.DeviceBatch(first, "cuda")
    s.set_option(ts.TS_OPT_FAIL_LAUNCH, which)
    with pytest.raises(ts.SamplerError) as e:
        s.sample(b)
    assert e.value.status == ts.TS_ERR_CUDA
    torch.cuda.synchronize()
    assert np.all(b.ids() == -2)  # no tail ran: nothing was written
    second = workloads.make("stress", 32, rows=rows)
    ref = oracle.sample(second, max_keep=4096, n_threads=8)
    gpu = run_gpu(s, second, debug_keep=4096)
    n_safe = compare(second, gpu, ref, label=f"after refused launch {which}")
    assert n_safe >= 0.5 * rows  # about 89% of stress rows are off-boundary
    s.close()


# ---------------------------------------------------------------------------
# adversarial and degenerate wide rows
# ---------------------------------------------------------------------------
def _wide_rows(rng):
    V = 20000
    rows = []
    nrm = lambda n, sd=3.0: rng.normal(0, sd, n).astype(np.float32)
    for k, p, t in ((1, 0.9, 1.0), (30, 0.9, 1.0), (64, 0.5, 0.7), (700, 0.95, 1.3),
                    (4096, 0.9, 1.0), (0, 0.9, 1.0), (4096, 1.0, 1.0), (30, 0.0, 1.0),
                    (30, 0.9, 0.0), (30, 0.9, -2.0), (64, 0.99, 0.05), (64, 0.99, 25.0)):
        rows.append((nrm(V), t, k, p))
    rows.append((np.full(V, 1.5, np.float32), 1.0, 64, 0.9))                      # all tied
    rows.append((rng.choice([0.0, 0.5, 1.0], V).astype(np.float32), 1.0, 4096, 0.9))  # huge ties
    y = np.full(V, -np.inf, np.float32)
    y[[7, 5000, 19999]] = [0.0, 1.0, 0.5]
    rows.append((y, 1.0, 30, 1.0))                                                 # -inf in top-k
    z = nrm(V)
    z[12345] = np.nan
    rows.append((z, 1.0, 30, 0.9))                                                 # NaN
    z = nrm(V)
    z[3] = np.inf
    rows.append((z, 1.0, 30, 0.9))                                                 # +inf
    rows.append((np.full(V, -np.inf, np.float32), 1.0, 30, 0.9))                  # no finite
    sz = rng.choice([-0.0, 0.0], V).astype(np.float32)
    sz[rng.choice(V, 20, replace=False)] = 0.25
    rows.append((sz, 1.0, 64, 0.9))                                                # signed-zero ties
    rows.append((np.sort(nrm(V)), 1.0, 4096, 0.9))                                 # sorted row
    # the sample sees only the bulk: the top values sit between sampled chunks
    adv = nrm(V, 1.0)
    q = np.arange(V // 8)
    sampled = np.unique((np.arange(1024) * (V // 8) // 1024))
    free = np.setdiff1d(q, sampled)
    hot = rng.choice(free, 1000, replace=False)
    for c in hot:
        adv[8 * c: 8 * c + 8] += 20.0
    rows.append((adv, 1.0, 4096, 0.9))
    rows.append((adv, 1.0, 30, 0.9))
    # a sample that overestimates: the sampled chunks hold the largest values
    over = nrm(V, 1.0)
    for c in sampled:
        over[8 * c: 8 * c + 8] += 30.0
    rows.append((over, 1.0, 4096, 0.9))
    # the same two cases against the split path's sample: 64 runs of 8 chunks
    # at evenly spaced starts (8-element margins cover a misaligned row head)
    stride = (V // 8) // 64
    in_run = np.zeros(V, bool)
    for k in range(64):
        a = 8 * k * stride
        in_run[max(a - 8, 0):a + 72] = True
    adv2 = nrm(V, 1.0)
    adv2[rng.choice(np.nonzero(~in_run)[0], 8000, replace=False)] += 20.0
    rows.append((adv2, 1.0, 4096, 0.9))   # too many candidates: the exact path
    rows.append((adv2, 1.0, 30, 0.9))     # about 8,000 candidates, all gathered
    over2 = nrm(V, 1.0)
    over2[in_run] += 30.0
    rows.append((over2, 1.0, 4096, 0.9))  # too few candidates: the exact path
    # values crossing zero in the kept set (wide key range)
    rows.append((rng.standard_t(3, V).astype(np.float32), 1.0, 4096, 0.6))
    return rows


@pytest.mark.parametrize("exact", [0, 1])
@pytest.mark.parametrize("path,cluster", [(3, 1), (3, 2), (3, 4), (4, 0), (4, 2), (4, 7)])
def test_wide_edge_rows(ts, path, cluster, exact):
    rng = np.random.default_rng(41)
    host = batch_from_rows(_wide_rows(rng), cap=4096, seed=cluster)
    ref = oracle.sample(host, max_keep=4096, n_threads=8)
    assert np.any(ref["err"] == 4) and np.any(ref["err"] == 0)
    s = make_sampler(ts, 4096, path=path, cluster=cluster, exact=exact, host=host)
    gpu = run_gpu(s, host, debug_keep=4096)
    compare(host, gpu, ref, label=f"wide edge path{path} g{cluster} exact{exact}")
    s.close()


@pytest.mark.parametrize("path", [1, 2, 3, 4])
def test_signed_zero_ties_every_path(ts, path):
    """-0 and +0 are the same value: ties between them go by token index."""
    rng = np.random.default_rng(8)
    rows = []
    for v in (40, 777, 2000):
        x = rng.choice([-0.0, 0.0], v).astype(np.float32)
        x[rng.choice(v, 5, replace=False)] = rng.normal(0, 1, 5)
        rows.append((x, 1.0, 30, 0.9))
        rows.append((x, 0.0, 30, 0.9))
    host = batch_from_rows(rows, cap=64, seed=3)
    ref = oracle.sample(host, max_keep=64)
    s = make_sampler(ts, 64, path=path, host=host)
    gpu = run_gpu(s, host, debug_keep=64)
    compare(host, gpu, ref, label=f"signed zeros path{path}")
    s.close()


# ---------------------------------------------------------------------------
# narrower workloads forced onto the wide path (all-candidates mode)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", [3, 4])
@pytest.mark.parametrize("name", ["mixed", "drama3", "qwen3tts"])
def test_workloads_on_wide_path(ts, name, path):
    host = workloads.make(name, 5)
    cap = host["cap"]
    ref = oracle.sample(host, max_keep=cap, n_threads=8)
    s = make_sampler(ts, cap, path=path, host=host)
    gpu = run_gpu(s, host, debug_keep=cap)
    compare(host, gpu, ref, label=f"{name} wide")
    s.close()


def test_wide_matches_other_paths_bit_for_bit(ts):
    rng = np.random.default_rng(17)
    v, rows = 40000, 5
    x = workloads.to_bf16_bits(rng.normal(0, 3, v * rows).astype(np.float32))
    host = workloads.make("mixed", 0)
    host = sub_batch(host, np.arange(rows))
    host.update(logits=x, row_vocab=np.full(rows, v, np.int32),
                row_offsets=np.arange(rows, dtype=np.int64) * v, max_row_vocab=v,
                top_k=np.array([1, 30, 700, 4096, 0], np.int32))
    outs = []
    for path, g, exact in ((2, 0, 0), (3, 1, 0), (3, 2, 0), (3, 4, 0), (3, 8, 0), (3, 4, 1),
                           (4, 0, 0), (4, 3, 0), (4, 16, 0), (4, 2, 1)):
        s = make_sampler(ts, 4096, path=path, cluster=g, exact=exact, host=host)
        outs.append(run_gpu(s, host, debug_keep=4096))
        s.close()
    ref = oracle.sample(host, max_keep=4096)
    compare(host, outs[1], ref, label="wide g1")
    for o in outs[1:]:
        assert np.array_equal(o["ids"], outs[0]["ids"])
        assert np.array_equal(o["n_nucleus"], outs[0]["n_nucleus"])
