"""The seeded input generators: shapes from the pages, determinism, bf16 rounding."""
import numpy as np
import pytest
import torch

import workloads
from oracle_pins import page_facts


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 3, 100000).astype(np.float32),
                        np.array([0.0, -0.0, 1e-40, 3.0e38, -2.5], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(workloads.to_bf16_bits(x), want)
    back = workloads.bf16_bits_to_f32(want)
    assert np.array_equal(back, torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("name", ["tiny", "qwen3tts", "drama3", "mixed"])
def test_workload_shapes_and_determinism(name):
    a = workloads.make(name, step=2)
    b = workloads.make(name, step=2)
    c = workloads.make(name, step=3)
    assert np.array_equal(a["logits"], b["logits"])
    if name != "tiny":
        assert not np.array_equal(a["logits"], c["logits"])
    else:
        assert np.array_equal(a["logits"], c["logits"])
    n = a["n_rows"]
    assert a["row_offsets"][-1] + a["row_vocab"][-1] == a["logits"].size
    assert n == a["n_streams"] * a["n_codebooks"]
    assert np.array_equal(a["feedback_slot"], np.arange(n))


def test_workloads_follow_the_pages():
    facts = page_facts()
    sp = facts["serving_params"]
    d = workloads.make("drama3")
    assert d["n_streams"] == facts["drama3_frame"]["concurrent_streams"]
    assert d["n_codebooks"] == facts["drama3_frame"]["codebooks_per_frame"]
    for b in (d, workloads.make("qwen3tts"), workloads.make("tiny")):
        assert np.all(b["temp"] == np.float32(sp["temperature"]))
        assert np.all(b["top_k"] == sp["top_k"])
        assert np.all(b["top_p"] == np.float32(sp["top_p"]))
        assert b["cap"] == facts["top_k_cap"]["default"]
    q = workloads.make("qwen3tts")
    qf = facts["qwen3tts_frame"]
    assert q["n_codebooks"] == qf["codebooks_per_frame"]
    assert np.all(q["row_vocab"][q["codebook"] > 0] == qf["codebook_size"])
    assert np.all(q["eos_id"][q["codebook"] == 0] == qf["codec_eos"])
    assert np.all(q["row_vocab"][q["codebook"] == 0] > qf["codec_eos"])


def test_drama3_near_silence_eos_probability():
    d = workloads.make("drama3", step=1)
    x = workloads.logits_as_f32(d).astype(np.float64)
    for s in d["silent_streams"][:5]:
        r = int(s) * 10
        row = x[d["row_offsets"][r]: d["row_offsets"][r] + d["row_vocab"][r]]
        lse = np.log(np.sum(np.exp(row - row.max()))) + row.max()
        p_eos = np.exp(row[4095] - lse)
        assert 1e-15 < p_eos < 1e-13
        assert np.sum(row > row[4095]) > 64  # far outside any top-k the cap allows


def test_stress_shape():
    s = workloads.make("stress", rows=2)
    assert s["row_vocab"].tolist() == [workloads.STRESS_VOCAB] * 2
    assert s["logits"].dtype == np.uint16 and s["logits"].size == 2 * workloads.STRESS_VOCAB
    assert np.all(s["top_k"] == 4096) and s["cap"] == 4096


def test_lm_head_frame_layout():
    """The LM head's frame: stream-major rows with head r mod Q, heads packed
    one after another (offsets multiples of the hidden size), fp32 logits
    buffer, hidden states that change with the step and weights that do not."""
    b0, h0 = workloads.make_lm_head(0)
    b1, h1 = workloads.make_lm_head(1)
    q, dim = h0["n_heads"], h0["dim"]
    assert (q, dim, b0["n_rows"], b0["dtype"]) == (16, 1024, 512, "f32")
    v = np.asarray(b0["row_vocab"])
    assert v[0] == 3072 and np.all(v[1:16] == 2048) and np.array_equal(v[:16], v[16:32])
    assert np.array_equal(np.asarray(b0["codebook"]), np.arange(512) % 16)
    offs = np.asarray(h0["head_offsets"])
    assert offs[0] == 0 and np.array_equal(np.diff(offs), v[:15].astype(np.int64) * dim)
    assert h0["weights"].size == int(v[:16].sum()) * dim and h0["hidden"].size == 512 * dim
    assert np.asarray(b0["logits"]).dtype == np.float32 and b0["logits"].size == int(v.sum())
    assert np.array_equal(h0["weights"], h1["weights"])
    assert not np.array_equal(h0["hidden"], h1["hidden"])
    w = workloads.bf16_bits_to_f32(h0["weights"][:1 << 20])
    assert abs(float(w.std()) - 2.5 / 32) < 0.002
