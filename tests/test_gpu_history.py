"""The repetition penalty over the fed-back frame history (Keskar et al. 2019,
CTRL; named among the sampling knobs by the Qwen3-TTS handbook page, section
"一个真实问题：说完了却停不下来") on the GPU against the oracle, through the C ABI.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import codebook_token_sampling_gb300 as mod
    return mod


def _np_dtype(host):
    return np.int16 if host["dtype"] == "bf16" else np.float32


@pytest.mark.parametrize("wpr", [0, 1, 2, 4])
@pytest.mark.parametrize("name", ["drama3", "qwen3tts"])
def test_history_ring_twenty_steps(ts, name, wpr):
    """Twenty steps with a ring of 8 frames and per-row penalties from 1 to 3:
    every step against the oracle run from the ring the GPU held before it,
    and the ring after it on every off-boundary row."""
    steps, t_len = 20, 8
    host = workloads.make(name, 0)
    n, n_streams, q = int(host["n_rows"]), int(host["n_streams"]), int(host["n_codebooks"])
    rng = np.random.default_rng(31)
    theta = rng.choice([1.0, 1.3, 2.0, 3.0], n).astype(np.float32)
    s = ts.Sampler(0, host["cap"])
    if wpr:
        s.set_option(ts.TS_OPT_WARPS_PER_ROW, wpr)
    b = ts.DeviceBatch(host, "cuda", advance_steps=True,
                       history={"len": t_len, "codebooks": q, "penalty": theta})
    n_safe = 0
    for t in range(steps):
        h = workloads.make(name, t % 5)
        h["step"] = np.full(n_streams, t, np.int64)
        b.set_logits(torch.from_numpy(np.ascontiguousarray(h["logits"]).view(_np_dtype(h))).cuda())
        ring = b.hist_ring.cpu().numpy().copy()
        s.sample(b)
        torch.cuda.synchronize()
        ref = oracle.sample(h, max_keep=64, n_threads=8, hist_ring=ring, rep_penalty=theta)
        gpu = {"ids": b.ids(), "eos": b.eos(), "status": s.read_status(),
               "feedback": b.feedback.cpu().numpy()}
        n_safe += compare(h, gpu, ref, check_probs=False, label=f"{name} history step {t}")
        safe = ref["margin"] > 1e-5
        got_ring = b.hist_ring.cpu().numpy()
        rows = np.nonzero(safe)[0]
        assert np.array_equal(got_ring[rows // q, t % t_len, rows % q],
                              ring[rows // q, t % t_len, rows % q]), t
    assert n_safe >= 0.98 * steps * n
    s.close()


@pytest.mark.parametrize("wpr", [1, 2, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_history_on_misaligned_rows(ts, dtype, wpr):
    """Rows at misaligned offsets whose history names their unaligned head and
    tail elements as well as body elements, with duplicates and out-of-range
    ids; the kept sets and probabilities too."""
    rng = np.random.default_rng(44)
    n, t_len = 48, 12
    vocab = rng.integers(20, 2000, n).astype(np.int32)
    gaps = rng.integers(0, 7, n)
    offs, parts, pos = [], [], 0
    for v, g in zip(vocab, gaps):
        parts.append(np.zeros(int(g), np.float32))
        pos += int(g)
        offs.append(pos)
        x = rng.normal(0, 2, int(v)).astype(np.float32)
        x[rng.choice(int(v), 3, replace=False)] += 5.0
        parts.append(x)
        pos += int(v)
    flat = np.concatenate(parts)
    logits = workloads.to_bf16_bits(flat) if dtype == "bf16" else flat
    host = {
        "dtype": dtype, "logits": logits, "n_rows": n, "n_streams": n, "n_codebooks": 1,
        "row_vocab": vocab, "row_offsets": np.array(offs, np.int64), "max_row_vocab": int(vocab.max()),
        "temp": rng.choice([1.0, 0.7], n).astype(np.float32),
        "top_k": rng.choice([30, 64, 5], n).astype(np.int32),
        "top_p": rng.choice([0.9, 1.0], n).astype(np.float32),
        "seed": np.arange(n, dtype=np.uint64) * np.uint64(31), "request": np.arange(n, dtype=np.uint64),
        "codebook": np.zeros(n, np.int32), "row_stream": np.arange(n, dtype=np.int32),
        "step": np.full(n, 3, np.int64), "eos_id": np.full(n, 1, np.int32),
        "feedback_slot": np.arange(n, dtype=np.int32), "feedback_len": n, "cap": 64,
    }
    theta = rng.choice([1.5, 4.0, 0.5], n).astype(np.float32)
    s = ts.Sampler(0, 64)
    s.set_option(ts.TS_OPT_PATH, 1)
    s.set_option(ts.TS_OPT_WARPS_PER_ROW, wpr)
    b = ts.DeviceBatch(host, "cuda", history={"len": t_len, "codebooks": 1, "penalty": theta})
    ring = np.full((n, t_len, 1), -1, np.int32)
    for r in range(n):
        v = int(vocab[r])
        # the top logits, the first and last elements (head / tail when the
        # row is misaligned), a duplicate, an id past the row, an empty slot
        top = np.argsort(-workloads.logits_as_f32(host)[offs[r]:offs[r] + v])[:4]
        cand = list(top) + [0, 1, v - 1, v - 2, int(top[0]), v + 5, -1, 2]
        ring[r, :, 0] = np.array(cand[:t_len], np.int32)
    b.hist_ring.copy_(torch.from_numpy(ring))
    kept = s.sample_debug(b, 64)
    torch.cuda.synchronize()
    ref = oracle.sample(host, max_keep=64, hist_ring=ring.copy(), rep_penalty=theta)
    gpu = {"ids": b.ids(), "eos": b.eos(), "status": s.read_status(),
           "feedback": b.feedback.cpu().numpy()}
    gpu.update({k: v.cpu().numpy() for k, v in kept.items()})
    compare(host, gpu, ref, label=f"history misaligned {dtype} wpr{wpr}")
    s.close()


def test_history_limits(ts):
    import ctypes
    host = workloads.make("mixed", 0)  # cap 4096: not the warp path
    s = ts.Sampler(0, host["cap"])
    b = ts.DeviceBatch(host, "cuda", history={"len": 4, "codebooks": 1,
                                              "penalty": np.ones(host["n_rows"], np.float32)})
    with pytest.raises(ts.SamplerError) as e:
        s.sample(b)
    assert e.value.status == ts.TS_ERR_UNSUPPORTED
    s.close()
    host = workloads.make("drama3", 0)
    s = ts.Sampler(0, 64)
    b = ts.DeviceBatch(host, "cuda", history={"len": 4, "codebooks": 10,
                                              "penalty": np.ones(host["n_rows"], np.float32)})
    with pytest.raises(ts.SamplerError) as e:
        s.sample_steps(b, 2, logits_step_stride=0, out_step_stride=host["n_rows"],
                       feedback_step_stride=host["feedback_len"])
    assert e.value.status == ts.TS_ERR_UNSUPPORTED
    b.c.hist_len = 33
    with pytest.raises(ts.SamplerError) as e:
        s.sample(b)
    assert e.value.status == ts.TS_ERR_INVALID_ARG
    # fp32 rows wider than 2048 go through the stage in two passes, and the
    # penalty edits the staged row in place: refused
    host = workloads.make("qwen3tts", 0)
    host["logits"] = workloads.bf16_bits_to_f32(host["logits"])
    host["dtype"] = "f32"
    b = ts.DeviceBatch(host, "cuda", history={"len": 4, "codebooks": 16,
                                              "penalty": np.ones(host["n_rows"], np.float32)})
    with pytest.raises(ts.SamplerError) as e:
        s.sample(b)
    assert e.value.status == ts.TS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert np.all(b.ids() == -2)
    s.close()
