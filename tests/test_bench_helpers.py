"""The benchmark's host-side helpers (no GPU): the algorithmic byte count,
the multi-step batch, the split path's launch count and the check that
recorded ncu traffic still belongs to the kernels being measured."""
import json
import os
import shutil

import numpy as np

import bench
import workloads


def test_algorithmic_bytes_of_the_headline_step():
    # 128 x (4096 + 9 x 1024) bf16 logits, plus 64 B read and 9 B written per row
    host = workloads.make("drama3", 0)
    assert bench.algorithmic_bytes(host) == 128 * (4096 + 9 * 1024) * 2 + 1280 * (64 + 9)
    assert bench.algorithmic_bytes(host) == 3_501_312


def test_concat_steps_keeps_every_row():
    hosts = [workloads.make("qwen3tts", i) for i in range(3)]
    h = bench.concat_steps(hosts)
    n = int(hosts[0]["n_rows"])
    assert h["n_rows"] == 3 * n and h["n_streams"] == 3 * int(hosts[0]["n_streams"])
    assert h["feedback_len"] == 3 * int(hosts[0]["feedback_len"])
    for i, src in enumerate(hosts):
        for r in (0, n // 2, n - 1):
            rr = i * n + r
            o, v = int(h["row_offsets"][rr]), int(h["row_vocab"][rr])
            so = int(src["row_offsets"][r])
            assert np.array_equal(h["logits"][o:o + v], src["logits"][so:so + v])
            assert h["step"][h["row_stream"][rr]] == src["step"][src["row_stream"][r]]
            for k in ("temp", "top_k", "top_p", "seed", "request", "codebook", "eos_id"):
                assert h[k][rr] == src[k][r]
    slots = h["feedback_slot"][h["feedback_slot"] >= 0]
    assert len(np.unique(slots)) == slots.size and slots.max() < h["feedback_len"]


def test_split_launch_count_rule():
    # the threshold kernel is skipped when rows x CTAs per row <= 2 x SMs
    assert bench.split_kernels({"ctas_per_row": 16}, 152, 1) == 2
    assert bench.split_kernels({"ctas_per_row": 16}, 152, 19) == 2
    assert bench.split_kernels({"ctas_per_row": 10}, 152, 32) == 3
    assert bench.split_kernels({"ctas_per_row": 4}, 152, 512) == 3


def test_traffic_record_follows_the_kernel_sources(tmp_path):
    src = tmp_path / "csrc"
    shutil.copytree(os.path.join(bench.ROOT, "codebook_token_sampling_gb300", "csrc"), src,
                    ignore=shutil.ignore_patterns("*.so", "*.o"))
    h = bench.kernel_source_hash(str(src))
    rec = tmp_path / "traffic.json"
    rec.write_text(json.dumps({"drama3": {"dram_bytes_per_launch": 123.0, "source_hash": h}}))
    assert bench.recorded_traffic("drama3", None, str(rec), str(src)) == 123.0
    assert bench.recorded_traffic("mixed", None, str(rec), str(src)) is None
    # a comment does not change the kernels
    f = src / "ts_device.cuh"
    f.write_text(f.read_text() + "\n// a comment\n")
    assert bench.kernel_source_hash(str(src)) == h
    # code does
    f.write_text(f.read_text() + "\nconstexpr int kUnused = 1;\n")
    assert bench.kernel_source_hash(str(src)) != h
    assert bench.recorded_traffic("drama3", None, str(rec), str(src)) is None


def test_lm_head_bytes_of_the_qwen3tts_frame():
    """Weights (bf16), hidden states (bf16) and fp32 logits, once each:
    (3072 + 15 x 2048) x 1024 x 2 + 512 x 1024 x 2 + 32 x (3072 + 15 x 2048) x 4."""
    batch, head = workloads.make_lm_head(0)
    v = 3072 + 15 * 2048
    assert bench.lm_head_bytes(batch, head) == v * 1024 * 2 + 512 * 1024 * 2 + 32 * v * 4
