"""Pins of the CPU oracle against things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with:

* numpy's Philox generator (a library implementation of the SC'11 Philox);
* numpy ``argmax`` (greedy = first maximum);
* scipy's softmax (top_p = 1 with top_k = V is plain softmax sampling);
* brute force on tiny rows: the top-k set from pairwise ranks, the nucleus as
  the minimum-cardinality subset reaching top_p, and the exact draw map over
  all 2^24 values of the 24-bit uniform;
* a chi-square test of 10^6 draws against the truncated distribution;
* the EOS-starvation invariant of the Qwen3-TTS handbook page (section
  "一个真实问题：说完了却停不下来"): an EOS at p ~ 1e-14 outside the top-k
  set is never drawn;
* the cap rule of the Drama 3 article (section "能跑通的命令，和文档写明的边界"):
  default 64, else a power of two in [32, 4096], read from tests/golden.
* the LM head (Qwen3-TTS handbook page, section "拓扑": hidden size 1024, a
  head per codebook): exact rational dot products on tiny rows, one-hot heads
  that pick and scale hidden entries, and the documented rule for heads that
  lie outside the weights.

``PINS`` lists them cheapest first; the mutation test runs them against
deliberately broken copies of the oracle.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
from scipy import special, stats

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TWO24 = 1 << 24


def page_facts():
    with open(os.path.join(GOLDEN, "page_facts.json"), encoding="utf-8") as f:
        return json.load(f)


def shared_row_batch(values, *, dtype="f32", n_rows=1, temp=1.0, top_k=0, top_p=1.0,
                     cap=32, steps=None, seed=0, request=0, codebook=0, eos_id=-1):
    """n_rows rows that all read the same logits (offset 0), one stream each."""
    if dtype == "bf16":
        logits = np.asarray(values, dtype=np.uint16)
    else:
        logits = np.asarray(values, dtype=np.float32)
    v = logits.size
    steps = np.arange(n_rows, dtype=np.int64) if steps is None else np.asarray(steps, np.int64)

    def full(x, dt):
        a = np.asarray(x, dtype=dt)
        return np.broadcast_to(a, (n_rows,)).copy() if a.ndim == 0 else a.astype(dt)

    return {
        "dtype": dtype, "logits": logits, "n_rows": n_rows, "n_streams": n_rows,
        "row_vocab": np.full(n_rows, v, np.int32), "row_offsets": np.zeros(n_rows, np.int64),
        "max_row_vocab": max(v, 1),
        "temp": full(temp, np.float32), "top_k": full(top_k, np.int32),
        "top_p": full(top_p, np.float32), "seed": full(seed, np.uint64),
        "request": full(request, np.uint64), "codebook": full(codebook, np.int32),
        "row_stream": np.arange(n_rows, dtype=np.int32), "step": steps,
        "eos_id": full(eos_id, np.int32), "feedback_slot": np.full(n_rows, -1, np.int32),
        "cap": cap,
    }


# --------------------------------------------------------------------------
# brute-force reference pieces (no sorting routine of the oracle's kind)
# --------------------------------------------------------------------------
def brute_rank(values):
    """rank_i = number of tokens that beat i: larger value, or equal and lower index."""
    v = [float(x) for x in values]
    return [sum(1 for j in range(len(v)) if v[j] > v[i] or (v[j] == v[i] and j < i))
            for i in range(len(v))]


def brute_kept(values, top_k, cap):
    v = len(values)
    k = top_k if top_k > 0 else v
    k = min(k, cap, v)
    rank = brute_rank(values)
    return sorted((i for i in range(v) if rank[i] < k), key=lambda i: rank[i])


def brute_probs(values, kept, temp):
    m = max(float(values[i]) for i in kept)
    w = [math.exp((float(values[i]) - m) / temp) for i in kept]
    s = math.fsum(w)
    return [x / s for x in w]


def brute_nucleus_size(q, top_p):
    """Minimum cardinality of any subset of the kept set whose mass reaches top_p."""
    if top_p >= 1.0:
        return len(q)
    if top_p <= 0.0:
        return 1
    for size in range(1, len(q) + 1):
        for subset in itertools.combinations(range(len(q)), size):
            if math.fsum(q[i] for i in subset) >= top_p:
                return size
    return len(q)


def near_cutoff(q, top_p, eps=1e-9):
    acc = 0.0
    for x in q:
        acc += x
        if abs(acc - top_p) <= eps:
            return True
    return False


# --------------------------------------------------------------------------
# pins, cheapest first
# --------------------------------------------------------------------------
def pin_philox_matches_numpy(orc):
    rng = np.random.default_rng(11)
    cases = [([0, 0, 0, 0], [0, 0]), ([2**64 - 1] * 4, [2**64 - 1] * 2),
             ([1, 2, 3, 4], [5, 6])]
    for _ in range(300):
        cases.append(([int(x) for x in rng.integers(0, 2**64, 4, dtype=np.uint64)],
                      [int(x) for x in rng.integers(0, 2**64, 2, dtype=np.uint64)]))
    for ctr, key in cases:
        c = sum(int(x) << (64 * i) for i, x in enumerate(ctr))
        k = int(key[0]) | (int(key[1]) << 64)
        # numpy's Philox increments its 256-bit counter before each block
        ref = np.random.Philox(key=k, counter=(c - 1) % (1 << 256)).random_raw(4)
        assert orc.philox4x64_10(ctr, key) == tuple(int(x) for x in ref), (ctr, key)


def pin_uniform24_mapping(orc):
    """u24 = top 24 bits of word 0 of Philox(ctr=(step, codebook, 0, 0), key=(seed, request))."""
    rng = np.random.default_rng(12)
    for _ in range(300):
        seed = int(rng.integers(0, 2**64, dtype=np.uint64))
        request = int(rng.integers(0, 2**64, dtype=np.uint64))
        step = int(rng.integers(0, 2**40))
        cb = int(rng.integers(0, 16))
        c = step | (cb << 64)
        ref = np.random.Philox(key=seed | (request << 64), counter=(c - 1) % (1 << 256))
        assert orc.uniform24(seed, request, step, cb) == int(ref.random_raw(1)[0]) >> 40


def pin_cap_rule(orc):
    cap = page_facts()["top_k_cap"]
    allowed = {1 << e for e in range(13) if cap["allowed_min"] <= (1 << e) <= cap["allowed_max"]}
    assert orc.cap(0) == cap["default"]
    for req in range(-2, 5000):
        if req == 0:
            continue
        want = req if req in allowed else -1
        assert orc.cap(req) == want, req


def pin_greedy_is_argmax(orc):
    rng = np.random.default_rng(13)
    for v in (1, 2, 7, 64, 1000):
        for trial in range(6):
            # coarse values so that ties at the maximum are common
            x = np.round(rng.normal(0, 1, v) * 2) / 2
            bits = workloads.to_bf16_bits(x)
            for dtype, vals in (("f32", x.astype(np.float32)), ("bf16", bits)):
                for temp, top_k, top_p in ((1.0, 1, 0.9), (0.0, 30, 0.9), (-1.0, 0, 1.0),
                                           (0.7, 50, 0.0)):
                    b = shared_row_batch(vals, dtype=dtype, n_rows=3, temp=temp, top_k=top_k,
                                         top_p=top_p, cap=64)
                    o = orc.sample(b, max_keep=64)
                    assert np.all(o["err"] == 0)
                    assert np.all(o["ids"] == int(np.argmax(x))), (v, trial, temp, top_k, top_p)
                    if temp <= 0 or top_k == 1:
                        probs = o["kept_probs"][0, : o["n_kept"][0]]
                        assert probs[0] == 1.0 and np.all(probs[1:] == 0.0)


def pin_topk_set_bruteforce(orc):
    rng = np.random.default_rng(14)
    for v in (1, 3, 9, 16):
        x = np.round(rng.normal(0, 1, v) * 2) / 2
        for top_k in range(-1, v + 2):
            b = shared_row_batch(x, n_rows=1, temp=1.0, top_k=top_k, top_p=1.0, cap=32)
            o = orc.sample(b, max_keep=32)
            kept = brute_kept(x, top_k, 32)
            assert o["n_kept"][0] == len(kept)
            assert list(o["kept_ids"][0, : len(kept)]) == kept, (v, top_k)


def pin_softmax_special_case(orc):
    """top_p = 1, top_k = V <= cap: kept probabilities are the plain softmax."""
    rng = np.random.default_rng(15)
    for v, cap, dtype in ((32, 32, "f32"), (32, 32, "bf16"), (4096, 4096, "bf16"),
                          (20, 64, "f32")):
        x32 = rng.normal(0, 2, v).astype(np.float32)
        vals = workloads.to_bf16_bits(x32) if dtype == "bf16" else x32
        x = workloads.bf16_bits_to_f32(vals) if dtype == "bf16" else x32
        for temp in (1.0, 0.6, 1.7):
            b = shared_row_batch(vals, dtype=dtype, n_rows=64, temp=temp, top_k=v,
                                 top_p=1.0, cap=cap)
            o = orc.sample(b, max_keep=v)
            order = np.lexsort((np.arange(v), -x.astype(np.float64)))
            t = float(np.float32(temp))  # the row's temperature is an fp32 value
            p = special.softmax(x.astype(np.float64) / t)[order]
            assert np.array_equal(o["kept_ids"][0], order)
            assert np.allclose(o["kept_probs"][0], p, rtol=1e-12, atol=0)
            cdf = np.cumsum(p)
            u = o["u24"].astype(np.float64) / TWO24
            pick = np.searchsorted(cdf, u, side="right")
            ok = np.min(np.abs(cdf[None, :] - u[:, None]), axis=1) > 1e-12
            assert np.array_equal(o["ids"][ok], order[np.minimum(pick, v - 1)][ok])


def pin_nucleus_bruteforce(orc):
    rng = np.random.default_rng(16)
    rows = [np.array([0.0, 0.0]), np.array([0.0, 0.0, 0.0, 0.0]),
            np.array([1.0, 0.0, 0.5, 0.0, -1.0])]
    rows += [np.round(rng.normal(0, 1.5, v) * 4) / 4 for v in (6, 9, 12)]
    grid = [0.05, 0.25, 0.5, 0.75, 0.9, 0.97, 1.0]
    for x in rows:
        v = x.size
        for top_k in range(1, v + 1):
            for top_p in grid:
                for temp in (1.0, 0.5):
                    b = shared_row_batch(x, n_rows=1, temp=temp, top_k=top_k, top_p=top_p,
                                         cap=32)
                    o = orc.sample(b, max_keep=32)
                    kept = brute_kept(x, top_k, 32)
                    q = brute_probs(x, kept, temp)
                    # dyadic cases are exact; others skip a boundary within 1e-9
                    exact = all(float(t).is_integer() for t in (np.array(q) * 4))
                    if not exact and near_cutoff(q, top_p):
                        continue
                    want = 1 if top_k == 1 else brute_nucleus_size(q, top_p)
                    assert o["n_nucleus"][0] == want, (x, top_k, top_p, temp)
                    if top_k > 1:
                        assert np.allclose(o["kept_probs"][0, : len(q)], q, rtol=1e-12)
                        assert abs(o["kept_probs"][0, : len(q)].sum() - 1.0) < 1e-12


def brute_margin(values, top_k, top_p, temp, cap, u24):
    """Distance of a row's draw from the nearest decision boundary, from its
    definition: the smallest |prefix mass - top_p| over the sorted prefixes of
    the top-k set (when 0 < top_p < 1), and the smallest |C_j / S_p - u| over
    the nucleus, with C_j the inclusive sorted prefix masses (math.fsum) and
    S_p the nucleus mass.  Greedy rows have no boundary (inf)."""
    kept = brute_kept(values, top_k, cap)
    if temp <= 0.0 or len(kept) == 1:
        return math.inf
    q = brute_probs(values, kept, temp)
    m_cut = math.inf
    if 0.0 < top_p < 1.0:
        m_cut = min(abs(math.fsum(q[:n]) - top_p) for n in range(1, len(q) + 1))
    n_p = brute_nucleus_size(q, top_p)
    s_p = math.fsum(q[:n_p])
    u = u24 / TWO24
    m_draw = min(abs(math.fsum(q[:j + 1]) / s_p - u) for j in range(n_p))
    return min(m_cut, m_draw)


def pin_margin_bruteforce(orc):
    """The boundary margin that decides which rows must match bit for bit,
    against brute_margin on small rows with forced draws: random u and u set
    right at a CDF step (a tiny margin), top_p near and far from a prefix."""
    rng = np.random.default_rng(20)
    cases = []
    for v in (3, 6, 9, 16):
        for _ in range(6):
            x = np.round(rng.normal(0, 1.5, v) * 8) / 8
            top_k = int(rng.integers(0, v + 1))
            top_p = float(np.float32(rng.choice([rng.uniform(0.05, 0.99), 1.0, 0.5])))
            temp = float(np.float32(rng.choice([1.0, 0.7, 1.6])))
            cases.append((x, top_k, top_p, temp))
    for x, top_k, top_p, temp in cases:
        kept = brute_kept(x, top_k, 32)
        q = brute_probs(x, kept, temp) if len(kept) > 1 else [1.0]
        if near_cutoff(q, top_p, 1e-9):
            continue  # the nucleus size itself is a rounding call here
        n_p = brute_nucleus_size(q, top_p) if len(kept) > 1 else 1
        s_p = math.fsum(q[:n_p])
        us = [int(u) for u in rng.integers(0, TWO24, 6)]
        # draws on a CDF step: the margin is below 2^-24
        us += [min(TWO24 - 1, int(math.floor(math.fsum(q[:j + 1]) / s_p * TWO24)))
               for j in range(n_p)]
        b = shared_row_batch(x, n_rows=len(us), temp=temp, top_k=top_k, top_p=top_p, cap=32)
        o = orc.sample(b, u24=us, max_keep=32)
        assert np.all(o["err"] == 0)
        for i, u in enumerate(us):
            want = brute_margin(x, top_k, top_p, temp, 32, u)
            got = float(o["margin"][i])
            if math.isinf(want):
                assert math.isinf(got), (x, top_k, top_p, temp, u, got)
            else:
                assert abs(got - want) <= 1e-12, (x, top_k, top_p, temp, u, got, want)


def pin_draw_map_exact(orc):
    """All 2^24 draws: each nucleus token's count equals its interval on the grid."""
    cases = [
        (np.array([0.0, 0.0]), 1.0, 2, 1.0),            # exactly 1/2, 1/2
        (np.array([0.0, 0.0, 0.0, 0.0]), 1.0, 4, 0.6),  # 1/4 each, nucleus of 3
        (np.array([2.0, -1.0, 0.5, 0.5, 1.25, -3.0, 0.0]), 1.0, 5, 0.9),
        (np.array([0.3, 1.1, -0.4, 2.2, 0.9, 0.0, -2.0, 1.7, 0.2]), 0.8, 0, 0.95),
    ]
    for x, temp, top_k, top_p in cases:
        counts = orc.draw_map(x, temp, top_k, top_p, 32).astype(np.int64)
        assert counts.sum() == TWO24
        kept = brute_kept(x, top_k, 32)
        q = brute_probs(x, kept, float(np.float32(temp)))
        n_p = brute_nucleus_size(q, float(np.float32(top_p)))
        s_p = math.fsum(q[:n_p])
        nucleus = kept[:n_p]
        # the sorted-order CDF on the grid: count_j = ceil(2^24 C_j) - ceil(2^24 C_{j-1})
        acc = 0.0
        for j, tok in enumerate(nucleus):
            lo = acc
            acc += q[j] / s_p
            want = math.ceil(TWO24 * acc - 1e-9) - math.ceil(TWO24 * lo - 1e-9)
            if j == n_p - 1:
                want = TWO24 - sum(int(counts[t]) for t in nucleus[:-1])
            dyadic = (TWO24 * acc).is_integer() and (TWO24 * lo).is_integer()
            assert abs(int(counts[tok]) - want) <= (0 if dyadic else 1), \
                (x, tok, counts[tok], want)
        for tok in range(x.size):
            if tok not in nucleus:
                assert counts[tok] == 0


def pin_eos_never_drawn(orc):
    """Near-silence: EOS at p ~ 1e-14, ranked outside the top-k set, is never drawn.

    Checked for every one of the 2^24 values of the uniform (a superset of any
    10^6 draws), then through the Philox path on 20,000 steps.
    """
    facts = page_facts()["eos_starvation"]
    rng = np.random.default_rng(17)
    v, eos = 4096, 4095
    x = 2.0 * rng.standard_normal(v).astype(np.float32)
    x[int(rng.integers(0, v - 1))] = 20.0
    x[eos] = np.float32(20.0 + np.log(facts["eos_probability"]))
    bits = workloads.to_bf16_bits(x)
    xf = workloads.bf16_bits_to_f32(bits).astype(np.float64)
    counts = orc.draw_map(xf, 1.0, 30, 0.9, 64)
    assert counts.sum() == TWO24 and counts[eos] == 0
    n = 20000
    b = shared_row_batch(bits, dtype="bf16", n_rows=n, temp=1.0, top_k=30, top_p=0.9,
                         cap=64, eos_id=eos)
    o = orc.sample(b, n_threads=4)
    assert np.all(o["err"] == 0)
    assert not np.any(o["ids"] == eos) and not np.any(o["eos"])
    # the largest u takes the last nucleus token, still not EOS
    last = shared_row_batch(bits, dtype="bf16", n_rows=1, temp=1.0, top_k=30, top_p=0.9,
                            cap=64, eos_id=eos)
    o1 = orc.sample(last, u24=[TWO24 - 1], max_keep=64)
    assert o1["ids"][0] == o1["kept_ids"][0, o1["n_nucleus"][0] - 1] != eos
    # positive control: an EOS inside the nucleus is drawn and flagged
    y = x.copy()
    y[eos] = 20.0
    b2 = shared_row_batch(workloads.to_bf16_bits(y), dtype="bf16", n_rows=4000, temp=1.0,
                          top_k=30, top_p=0.9, cap=64, eos_id=eos)
    o2 = orc.sample(b2, n_threads=4)
    frac = float(np.mean(o2["ids"] == eos))
    assert 0.4 < frac < 0.6 and np.array_equal(o2["eos"].astype(bool), o2["ids"] == eos)


def pin_chi_square(orc):
    rng = np.random.default_rng(18)
    x = workloads.to_bf16_bits(rng.normal(0, 2, 64).astype(np.float32))
    xf = workloads.bf16_bits_to_f32(x).astype(np.float64)
    n = 1_000_000
    b = shared_row_batch(x, dtype="bf16", n_rows=n, temp=1.0, top_k=30, top_p=0.9, cap=64,
                         seed=7, request=3)
    o = orc.sample(b, n_threads=4)
    kept = brute_kept(xf, 30, 64)
    q = brute_probs(xf, kept, 1.0)
    n_p = brute_nucleus_size(q, 0.9)
    p = np.array(q[:n_p]) / math.fsum(q[:n_p])
    counts = np.array([np.sum(o["ids"] == t) for t in kept[:n_p]])
    assert counts.sum() == n
    exp_counts = p * n
    big = exp_counts >= 5
    obs = np.append(counts[big], counts[~big].sum())
    exp = np.append(exp_counts[big], exp_counts[~big].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    assert stats.chisquare(obs, exp).pvalue > 0.001


def pin_error_rows(orc):
    nan = np.float32("nan")
    rows = {
        "nan": ([0.0, nan, 1.0], 4), "pinf": ([0.0, np.inf, 1.0], 4),
        "all_ninf": ([-np.inf, -np.inf], 4), "ok": ([0.5, -np.inf, 2.0], 0),
    }
    for name, (vals, bit) in rows.items():
        b = shared_row_batch(np.array(vals, np.float32), n_rows=2, temp=1.0, top_k=30,
                             top_p=0.9, cap=64)
        o = orc.sample(b)
        assert np.all(o["err"] == bit), name
        assert np.all(o["ids"] == (-1 if bit else 2)), name
    x = np.array([0.0, 1.0, 2.0], np.float32)
    for temp, top_p, bit in ((float("nan"), 0.9, 2), (float("inf"), 0.9, 2),
                             (1.0, float("nan"), 2), (1.0, 0.9, 0)):
        o = orc.sample(shared_row_batch(x, temp=temp, top_p=top_p, top_k=30, cap=64))
        assert o["err"][0] == bit and (o["ids"][0] == -1) == bool(bit)
    # shape errors: V <= 0, V > max_row_vocab, offset beyond the buffer, bad stream
    b = shared_row_batch(x, n_rows=4, top_k=30, cap=64)
    b["row_vocab"] = np.array([0, 3, 3, 3], np.int32)
    b["row_offsets"] = np.array([0, 0, 1, 0], np.int64)
    b["row_stream"] = np.array([0, 1, 2, 7], np.int32)
    b["max_row_vocab"] = 3
    o = orc.sample(b)
    assert list(o["err"]) == [1, 0, 1, 1] and list(o["ids"][[0, 2, 3]]) == [-1, -1, -1]
    # -inf tokens are never drawn even when they enter the top-k set
    y = np.full(40, -np.inf, np.float32)
    y[[3, 17]] = [0.0, 0.0]
    o = orc.sample(shared_row_batch(y, n_rows=5000, top_k=30, top_p=1.0, cap=64))
    assert set(np.unique(o["ids"])) == {3, 17}


def pin_k_clamp(orc):
    rng = np.random.default_rng(19)
    x = rng.normal(0, 1, 100).astype(np.float32)
    for top_k, cap, want in ((500, 64, 64), (0, 64, 64), (-3, 32, 32), (0, 4096, 100),
                             (64, 64, 64), (10, 64, 10)):
        o = orc.sample(shared_row_batch(x, n_rows=50, top_k=top_k, top_p=1.0, cap=cap),
                       max_keep=128)
        assert np.all(o["n_kept"] == want), (top_k, cap)
        ref = orc.sample(shared_row_batch(x, n_rows=50, top_k=want, top_p=1.0, cap=cap))
        assert np.array_equal(o["ids"], ref["ids"])


def pin_writeback_and_frame(orc):
    b = workloads.make("drama3", step=3)
    fb = np.full(b["feedback_len"], -7, np.int32)
    b["feedback_slot"] = b["feedback_slot"].copy()
    b["feedback_slot"][5] = -1
    o = orc.sample(b, feedback_buf=fb)
    assert np.all(o["err"] == 0)
    mask = np.ones(b["n_rows"], bool)
    mask[5] = False
    assert np.array_equal(fb[b["feedback_slot"][mask]], o["ids"][mask]) and fb[5] == -7
    frame = fb.reshape(b["n_streams"], b["n_codebooks"])
    assert frame.shape == (128, page_facts()["drama3_frame"]["codebooks_per_frame"])
    b["feedback_slot"][6] = b["feedback_len"]
    o = orc.sample(b, feedback_buf=fb)
    assert o["err"][6] == 8 and o["ids"][6] == -1
    o4 = orc.sample(workloads.make("drama3", step=3), n_threads=4)
    o1 = orc.sample(workloads.make("drama3", step=3), n_threads=1)
    assert np.array_equal(o4["ids"], o1["ids"])


def finish_workload(step, forced_eos):
    """A small frame batch: 6 streams x 3 codebooks (codebook 0 of 64 tokens
    with EOS 63, codebooks 1-2 of 32 tokens), gaussian logits; streams in
    forced_eos[step] get a dominant EOS logit at this step."""
    rng = np.random.default_rng(500 + step)
    n_streams, q = 6, 3
    vocab = [64, 32, 32]
    rows = n_streams * q
    rv = np.array([vocab[r % q] for r in range(rows)], np.int32)
    ro = np.concatenate([[0], np.cumsum(rv[:-1])]).astype(np.int64)
    x = rng.normal(0, 1.5, int(rv.sum())).astype(np.float32)
    for s in forced_eos.get(step, ()):
        x[ro[s * q] + 63] = 30.0
    return {
        "dtype": "f32", "logits": x, "n_rows": rows, "n_streams": n_streams,
        "row_vocab": rv, "row_offsets": ro, "max_row_vocab": 64,
        "temp": np.full(rows, 1.0, np.float32), "top_k": np.full(rows, 30, np.int32),
        "top_p": np.full(rows, 0.9, np.float32),
        "seed": np.repeat(np.arange(n_streams, dtype=np.uint64) + np.uint64(9), q),
        "request": np.repeat(np.arange(n_streams, dtype=np.uint64), q),
        "codebook": np.tile(np.arange(q, dtype=np.int32), n_streams),
        "row_stream": np.repeat(np.arange(n_streams, dtype=np.int32), q),
        "step": np.full(n_streams, step, np.int64),
        "eos_id": np.tile(np.array([63, -1, -1], np.int32), n_streams),
        "feedback_slot": np.arange(rows, dtype=np.int32), "feedback_len": rows, "cap": 64,
    }


def pin_finish_rule(orc):
    """The finished-stream rule of the handbook's EOS-starvation section, against
    its restatement on plain sampling: a stream whose EOS is drawn at step s
    pads every row from step s + 1 (reason stop); a stream at or past its
    length cap pads (reason length), unless it stopped earlier; a padded row
    draws nothing, so every other row equals the plain run."""
    steps, pad = 9, -7
    forced = {2: (1,), 5: (3,), 6: (5,), 7: (1,)}
    max_steps = np.array([100, 5, 4, 100, 100, 6], np.int64)
    plain = [orc.sample(finish_workload(t, forced)) for t in range(steps)]
    stop = np.full(6, -1, np.int64)
    reason = np.zeros(6, np.uint8)
    got = []
    for t in range(steps):
        fb = np.full(18, -9, np.int32)
        got.append(orc.sample(finish_workload(t, forced), stop_step=stop, max_steps=max_steps,
                              finish_reason=reason, pad_id=pad, feedback_buf=fb))
        assert np.array_equal(fb, got[-1]["ids"]), t
    # the restatement
    want_stop = np.full(6, -1, np.int64)
    want_reason = np.zeros(6, np.uint8)
    for t in range(steps):
        ids, eos = plain[t]["ids"].copy(), plain[t]["eos"].astype(bool)
        for s in range(6):
            rows = slice(3 * s, 3 * s + 3)
            if 0 <= want_stop[s] < t:
                fin = 1
            elif t >= max_steps[s]:
                fin = 2
            else:
                fin = 0
            if fin:
                assert np.all(got[t]["ids"][rows] == pad) and not np.any(got[t]["eos"][rows]), (t, s)
                assert np.all(got[t]["finished"][rows] == fin), (t, s)
                want_reason[s] = fin
                continue
            assert np.array_equal(got[t]["ids"][rows], ids[rows]), (t, s)
            assert np.array_equal(got[t]["eos"][rows].astype(bool), eos[rows]), (t, s)
            if np.any(eos[rows]):
                want_stop[s] = t
                want_reason[s] = 1
    assert np.array_equal(stop, want_stop) and np.array_equal(reason, want_reason)
    # the forced events happened as planned: stream 1 stops at step 2 (and
    # stays stopped past its cap 5; its forced EOS at step 7 is never drawn),
    # stream 3 stops at step 5, stream 2 runs out at step 4, and stream 5
    # reaches its cap (6) at the step of its EOS
    assert want_stop[1] == 2 and want_stop[3] == 5 and want_stop[5] < 0
    assert list(want_reason[[1, 2, 3, 5]]) == [1, 2, 1, 2]


def pin_repetition_penalty(orc):
    """The repetition penalty (CTRL, Keskar et al. 2019) over the frame history,
    against its restatement: the penalised logits computed here with numpy
    (fp32 division or product, then bf16 round to nearest even for bf16 rows,
    once per distinct token of the row's history column) and sampled without
    the penalty.  theta = 1 changes nothing; the draw joins the ring at slot
    step mod T and no other slot changes."""
    rng = np.random.default_rng(21)
    t_len, q = 5, 3
    for dtype in ("f32", "bf16"):
        for step in (0, 7):
            h = finish_workload(step, {1: (0,)})
            n, n_streams = h["n_rows"], h["n_streams"]
            x32 = rng.normal(0, 2, h["logits"].size).astype(np.float32)
            x32[rng.choice(x32.size, 30, replace=False)] += 6.0
            if dtype == "bf16":
                h["dtype"] = "bf16"
                h["logits"] = workloads.to_bf16_bits(x32)
                xs = workloads.bf16_bits_to_f32(h["logits"])
            else:
                h["logits"] = x32
                xs = x32
            ring = rng.integers(-2, 70, (n_streams, t_len, q)).astype(np.int32)
            ring[:, 1, :] = ring[:, 0, :]          # duplicates in every column
            theta = rng.choice([1.0, 1.3, 2.5, 0.7], n).astype(np.float32)
            before = ring.copy()
            got = orc.sample(h, max_keep=64, hist_ring=ring, rep_penalty=theta)
            # restatement
            y = np.array(xs, np.float32).copy()
            for r in range(n):
                s_, c = r // q, r % q
                v, o = int(h["row_vocab"][r]), int(h["row_offsets"][r])
                for tok in set(int(t) for t in before[s_, :, c]):
                    if 0 <= tok < v:
                        f = np.float32(y[o + tok])
                        pen = np.float32(f / theta[r]) if f > 0 else np.float32(f * theta[r])
                        if dtype == "bf16":
                            pen = workloads.bf16_bits_to_f32(workloads.to_bf16_bits(
                                np.array([pen], np.float32)))[0]
                        y[o + tok] = pen
            h2 = dict(h)
            h2["logits"] = workloads.to_bf16_bits(y) if dtype == "bf16" else y
            if dtype == "bf16":
                assert np.array_equal(workloads.bf16_bits_to_f32(h2["logits"]), y)
            want = orc.sample(h2, max_keep=64)
            for key in ("ids", "eos", "n_kept", "n_nucleus", "kept_ids", "kept_probs", "margin"):
                assert np.array_equal(got[key], want[key]), (dtype, step, key)
            # theta = 1 rows equal the run without any penalty
            plain = orc.sample(h, max_keep=64)
            one = theta == 1.0
            assert np.array_equal(got["ids"][one], plain["ids"][one])
            # the ring: each row's draw at slot step mod T, nothing else moved
            after = before.copy()
            for r in range(n):
                after[r // q, step % t_len, r % q] = got["ids"][r]
            assert np.array_equal(ring, after), (dtype, step)


def lm_head_case(rng, n_heads, n_streams, dim, vocabs, *, lo=-6, hi=3):
    """A frame of n_streams x n_heads rows (row = stream * Q + q) with packed
    logits, bf16 hidden states and one head per codebook, heads packed one
    after another at offsets that are multiples of 8 elements.  Values are
    +-m 2^e with an 8-bit m and e in [lo, hi], so that every dot product of a
    few dozen terms is exact in fp64."""
    def bf16(shape):
        m = rng.integers(128, 256, shape).astype(np.float64)
        e = rng.integers(lo, hi + 1, shape)
        sgn = rng.choice([-1.0, 1.0], shape)
        x = (sgn * m * np.exp2(e - 7)).astype(np.float32)
        bits = workloads.to_bf16_bits(x)
        assert np.array_equal(workloads.bf16_bits_to_f32(bits), x)
        return bits
    n = n_streams * n_heads
    rv = np.array([vocabs[r % n_heads] for r in range(n)], np.int32)
    ro = np.concatenate([[0], np.cumsum(rv)[:-1]]).astype(np.int64)
    offs, cur = [], 0
    for q in range(n_heads):
        offs.append(cur)
        cur += -(-vocabs[q] * dim // 8) * 8
    batch = {"n_rows": n, "row_vocab": rv, "row_offsets": ro, "logits_len": int(rv.sum()),
             "logits": np.zeros(int(rv.sum()), np.float32), "max_row_vocab": int(max(vocabs))}
    head = {"hidden": bf16(n * dim), "weights": bf16(cur), "head_offsets": np.array(offs, np.int64),
            "n_heads": n_heads, "dim": dim}
    return batch, head


def pin_lm_head_exact(orc):
    """Every logit of tiny rows equals the exact rational dot product of the
    row's hidden state with its codebook's head row (head r mod Q), rounded
    once to fp32; rows with a head outside the weights or misaligned are NaN,
    rows with a shape error are left unwritten."""
    from fractions import Fraction
    rng = np.random.default_rng(31)
    for n_heads, n_streams, dim, vocabs in ((3, 2, 16, (5, 7, 3)), (1, 3, 24, (9,)),
                                            (4, 1, 8, (2, 6, 1, 4))):
        batch, head = lm_head_case(rng, n_heads, n_streams, dim, vocabs)
        got = orc.lm_head(batch, head)
        hv = workloads.bf16_bits_to_f32(head["hidden"]).astype(np.float64)
        wv = workloads.bf16_bits_to_f32(head["weights"]).astype(np.float64)
        for r in range(batch["n_rows"]):
            q, v_r, o = r % n_heads, int(batch["row_vocab"][r]), int(batch["row_offsets"][r])
            w0 = int(head["head_offsets"][q])
            for v in range(v_r):
                exact = sum(Fraction(float(hv[r * dim + k])) * Fraction(float(wv[w0 + v * dim + k]))
                            for k in range(dim))
                assert Fraction(float(exact)) == exact  # no rounding before the fp32 one
                want = np.float32(float(exact))
                assert got[o + v].view(np.uint32) == want.view(np.uint32), (n_heads, r, v)
    # heads outside the weights: negative, misaligned, one row past the end
    batch, head = lm_head_case(rng, 3, 2, 16, (5, 7, 3))
    w_len = head["weights"].size
    # a view into a longer buffer: an oracle that reads past weights_len
    # reads zeros, not unmapped memory
    head["weights"] = np.concatenate([head["weights"], np.zeros(64, np.uint16)])[:w_len]
    base = orc.lm_head(batch, head)
    for q, bad in ((0, -8), (1, int(head["head_offsets"][1]) + 4), (2, w_len - 3 * 16 + 8)):
        h2 = dict(head)
        h2["head_offsets"] = head["head_offsets"].copy()
        h2["head_offsets"][q] = bad
        got = orc.lm_head(batch, h2)
        for r in range(batch["n_rows"]):
            o, v_r = int(batch["row_offsets"][r]), int(batch["row_vocab"][r])
            seg = got[o:o + v_r]
            if r % 3 == q:
                assert np.all(np.isnan(seg)), (q, bad, r)
            else:
                assert np.array_equal(seg.view(np.uint32), base[o:o + v_r].view(np.uint32))
    # the last head ending exactly at the end of the weights is inside them
    h2 = dict(head)
    h2["weights"] = head["weights"][:int(head["head_offsets"][2]) + 3 * 16]
    got = orc.lm_head(batch, h2)
    assert not np.any(np.isnan(got)) and np.array_equal(got.view(np.uint32), base.view(np.uint32))
    # a shape error (V = 0 or V above max_row_vocab) leaves the row unwritten
    b2 = dict(batch)
    b2["row_vocab"] = batch["row_vocab"].copy()
    b2["row_vocab"][1] = 0
    b2["max_row_vocab"] = 6
    got = orc.lm_head(b2, head)
    o1, o4 = int(batch["row_offsets"][1]), int(batch["row_offsets"][4])
    assert not np.any(got[o1:o1 + 7]) and not np.any(got[o4:o4 + 7])  # row 4 is 7 wide
    o0 = int(batch["row_offsets"][0])
    assert np.array_equal(got[o0:o0 + 5].view(np.uint32), base[o0:o0 + 5].view(np.uint32))


def pin_lm_head_one_hot(orc):
    """One-hot heads: head q's row v is 2^q at column pi_q(v), so row r's logit
    v is exactly 2^q h_r[pi_q(v)] (q = r mod Q): a transposed head, a wrong
    head or a wrong hidden row changes these values."""
    rng = np.random.default_rng(32)
    n_heads, n_streams, dim, vocab = 4, 3, 64, 24
    batch, head = lm_head_case(rng, n_heads, n_streams, dim, (vocab,) * n_heads)
    w = np.zeros(head["weights"].size, np.float32)
    perms = [rng.permutation(dim)[:vocab] for _ in range(n_heads)]
    for q in range(n_heads):
        w0 = int(head["head_offsets"][q])
        for v in range(vocab):
            w[w0 + v * dim + perms[q][v]] = 2.0 ** q
    head["weights"] = workloads.to_bf16_bits(w)
    got = orc.lm_head(batch, head)
    hv = workloads.bf16_bits_to_f32(head["hidden"]).reshape(-1, dim)
    for r in range(batch["n_rows"]):
        q, o = r % n_heads, int(batch["row_offsets"][r])
        want = (hv[r, perms[q]] * np.float32(2.0 ** q)).astype(np.float32)
        assert np.array_equal(got[o:o + vocab].view(np.uint32), want.view(np.uint32)), r


PINS = [
    pin_philox_matches_numpy,
    pin_uniform24_mapping,
    pin_cap_rule,
    pin_lm_head_one_hot,
    pin_lm_head_exact,
    pin_greedy_is_argmax,
    pin_topk_set_bruteforce,
    pin_softmax_special_case,
    pin_k_clamp,
    pin_error_rows,
    pin_writeback_and_frame,
    pin_finish_rule,
    pin_repetition_penalty,
    pin_nucleus_bruteforce,
    pin_margin_bruteforce,
    pin_draw_map_exact,
    pin_eos_never_drawn,
    pin_chi_square,
]
