"""The LM head (ts_lm_head_logits / ts_lm_head_sample) against the CPU oracle.

The logits: the kernel accumulates bf16 products in fp32 in its own order, the
oracle sums them in fp64 and rounds once to fp32.  Recursive summation of n
terms in fp32 is off the exact sum by at most about n u sum_k |h_k w_k|
(u = 2^-24; Higham, "Accuracy and Stability of Numerical Algorithms", 2nd ed.,
section 4.2), so every GPU logit must lie within
    2 * dim * 2^-24 * sum_k |h_k w_k| + 2^-24 |l|
of the oracle's (twice the bound, for the tensor cores' own adder order,
plus the oracle's final rounding).

The draws: a logit that moves by at most d moves every renormalised
probability by a factor within exp(+-2 d / T), so a prefix mass moves by at
most exp(4 d / T) - 1.  A row's id must match the oracle's when its draw and
its top_p cutoff lie farther than that (plus 1e-6) from a boundary and its
k_eff-th and (k_eff+1)-th largest logits are more than 2 d apart, with d the
row's largest logit difference; the other rows' ids must be members of the
oracle's nucleus widened by one token.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import codebook_token_sampling_gb300 as mod
    return mod


def abs_dot_bound(batch, head):
    """Per logit, sum_k |h_k w_k| (fp64), packed like the logits."""
    dim, q = int(head["dim"]), int(head["n_heads"])
    hv = np.abs(workloads.bf16_bits_to_f32(head["hidden"]).astype(np.float64)).reshape(-1, dim)
    wv = np.abs(workloads.bf16_bits_to_f32(head["weights"]).astype(np.float64))
    out = np.zeros(int(np.asarray(batch["logits"]).size), np.float64)
    for r in range(int(batch["n_rows"])):
        v, o = int(batch["row_vocab"][r]), int(batch["row_offsets"][r])
        w0 = int(head["head_offsets"][r % q])
        out[o:o + v] = wv[w0:w0 + v * dim].reshape(v, dim) @ hv[r]
    return out


def gpu_logits(ts, sampler, batch, head):
    b = ts.DeviceBatch(batch, "cuda", feedback=False)
    h = ts.LmHead(head, "cuda")
    ts.ts_lm_head_logits(sampler.handle, h, b)
    torch.cuda.synchronize()
    return b.logits.cpu().numpy()


def check_logits(batch, head, got, want):
    dim = int(head["dim"])
    bound = abs_dot_bound(batch, head)
    tol = 2.0 * dim * 2.0 ** -24 * bound + 2.0 ** -24 * np.abs(want.astype(np.float64))
    diff = np.abs(got.astype(np.float64) - want.astype(np.float64))
    written = np.zeros(got.size, bool)
    for r in range(int(batch["n_rows"])):
        o, v = int(batch["row_offsets"][r]), int(batch["row_vocab"][r])
        written[o:o + v] = True
    assert np.all(np.isfinite(got[written]))
    bad = np.nonzero(diff[written] > tol[written])[0]
    assert bad.size == 0, (bad[:5], diff[written][bad[:5]], tol[written][bad[:5]])
    return diff


@pytest.mark.parametrize("streams,vocabs,dim", [
    (40, (300, 257, 128), 1024),   # two stream tiles (32 + 8), ragged vocab tiles
    (5, (129, 1, 64), 192),        # fewer K stages than the ring holds
    (33, (2048,), 64),             # one K stage, one codebook
    (32, (3072,) + (2048,) * 15, 1024),  # the qwen3tts frame
])
def test_lm_head_logits_match_oracle(ts, streams, vocabs, dim):
    batch, head = workloads.make_lm_head(3, streams=streams, dim=dim, vocabs=vocabs,
                                         eos_ids=[-1] * len(vocabs))
    s = ts.Sampler(0, 64)
    got = gpu_logits(ts, s, batch, head)
    want = oracle.lm_head(batch, head)
    diff = check_logits(batch, head, got, want)
    # fp32 accumulation, not bf16: the typical difference is far below a
    # bf16 rounding step (2^-9 relative)
    assert np.median(diff) <= 2.0 ** -14 * np.median(np.abs(want))


def robust_rows(batch, ref_logits, got_logits, ref):
    """Rows whose id must match exactly (see the module docstring)."""
    n = int(batch["n_rows"])
    safe = np.zeros(n, bool)
    for r in range(n):
        o, v = int(batch["row_offsets"][r]), int(batch["row_vocab"][r])
        d = float(np.max(np.abs(got_logits[o:o + v].astype(np.float64) -
                                ref_logits[o:o + v].astype(np.float64))))
        k = int(ref["n_kept"][r])
        srt = np.sort(ref_logits[o:o + v].astype(np.float64))[::-1]
        gap = srt[k - 1] - srt[k] if k < v else np.inf
        eps = np.expm1(4.0 * d / float(batch["temp"][r])) + 1e-6
        safe[r] = ref["err"][r] == 0 and ref["margin"][r] > eps and gap > 2.0 * d
    return safe


@pytest.mark.parametrize("step", [0, 11])
def test_lm_head_sample_matches_oracle(ts, step):
    """The qwen3tts frame through ts_lm_head_sample (the benchmark's call):
    ids, EOS flags and the frame write-back against the oracle sampling the
    oracle's own logits."""
    batch, head = workloads.make_lm_head(step)
    s = ts.Sampler(0, 64)
    b = ts.DeviceBatch(batch, "cuda")
    h = ts.LmHead(head, "cuda")
    ts.ts_lm_head_sample(s.handle, h, b)
    torch.cuda.synchronize()
    ids, eos, frame = b.ids(), b.eos(), b.feedback.cpu().numpy()
    assert s.read_status() == 0
    got_logits = b.logits.cpu().numpy()
    ref_logits = oracle.lm_head(batch, head)
    check_logits(batch, head, got_logits, ref_logits)
    rb = dict(batch)
    rb["logits"] = ref_logits
    ref = oracle.sample(rb, max_keep=64, n_threads=8)
    safe = robust_rows(batch, ref_logits, got_logits, ref)
    assert safe.sum() >= 0.95 * batch["n_rows"], int(safe.sum())
    mism = np.nonzero(ids[safe] != ref["ids"][safe])[0]
    assert mism.size == 0, np.nonzero(safe)[0][mism][:10]
    for r in np.nonzero(~safe)[0]:
        n_p = int(ref["n_nucleus"][r])
        allowed = set(ref["kept_ids"][r, :min(n_p + 1, int(ref["n_kept"][r]))].tolist())
        assert int(ids[r]) in allowed, r
    want_eos = (ids == batch["eos_id"]) & (batch["eos_id"] >= 0)
    assert np.array_equal(eos.astype(bool), want_eos)
    assert np.array_equal(frame[batch["feedback_slot"]], ids)


def test_lm_head_rows_outside_the_weights(ts):
    """A head with a negative, misaligned or too-short extent gives its rows
    NaN logits (TS_ROW_NONFINITE, id -1); a row of width 0 is a shape error
    and is not written; the other rows are untouched by either."""
    batch, head = workloads.make_lm_head(1, streams=6, dim=128, vocabs=(200, 160, 96, 64),
                                         eos_ids=[-1] * 4)
    offs = head["head_offsets"].copy()
    offs[1] = -8
    offs[2] = offs[2] + 4                            # not a multiple of 8
    head["head_offsets"] = offs
    head["weights"] = head["weights"][:int(offs[3]) + 63 * 128]  # head 3 one row short
    batch["row_vocab"] = batch["row_vocab"].copy()
    batch["row_vocab"][4] = 0                        # stream 1, head 0
    s = ts.Sampler(0, 64)
    b = ts.DeviceBatch(batch, "cuda")
    h = ts.LmHead(head, "cuda")
    sentinel = torch.full_like(b.logits, 7.0)
    b.set_logits(sentinel)
    ts.ts_lm_head_sample(s.handle, h, b)
    torch.cuda.synchronize()
    got = b.logits.cpu().numpy()
    want = oracle.lm_head(batch, head)
    ids = b.ids()
    status = s.read_status()
    assert status == ts.TS_ROW_NONFINITE | ts.TS_ROW_BAD_SHAPE
    for r in range(batch["n_rows"]):
        o, v = int(batch["row_offsets"][r]), int(batch["row_vocab"][r])
        if r == 4:
            assert ids[r] == -1
            assert np.all(got[o:o + 200] == 7.0)    # nothing written
        elif r % 4 in (1, 2, 3):
            assert ids[r] == -1
            assert np.all(np.isnan(got[o:o + v])) and np.all(np.isnan(want[o:o + v]))
        else:
            assert ids[r] >= 0
            assert np.all(np.abs(got[o:o + v] - want[o:o + v]) <= 1e-3)


def test_lm_head_host_checks(ts):
    """Refusals on the host: nothing is launched and nothing is written."""
    batch, head = workloads.make_lm_head(0, streams=4, dim=128, vocabs=(256, 128),
                                         eos_ids=[-1, -1])
    s = ts.Sampler(0, 64)
    b = ts.DeviceBatch(batch, "cuda")
    h = ts.LmHead(head, "cuda")
    b.set_logits(torch.full_like(b.logits, 7.0))

    def refused(expect, fn=ts.ts_lm_head_sample):
        with pytest.raises(ts.SamplerError) as e:
            fn(s.handle, h, b)
        assert e.value.status == expect

    h.c.dim = 96                                   # not a multiple of 64
    refused(ts.TS_ERR_INVALID_ARG)
    h.c.dim = 128
    h.c.n_heads = 3                                # 8 rows are not whole frames of 3
    refused(ts.TS_ERR_INVALID_ARG)
    h.c.n_heads = 2
    h.c.hidden = h.hidden.data_ptr() + 2           # misaligned hidden states
    refused(ts.TS_ERR_INVALID_ARG, ts.ts_lm_head_logits)
    h.c.hidden = h.hidden.data_ptr()
    b.c.dtype = ts.TS_DTYPE_BF16                   # the head writes fp32 logits
    refused(ts.TS_ERR_INVALID_ARG)
    b.c.dtype = ts.TS_DTYPE_F32
    torch.cuda.synchronize()
    assert torch.all(b.logits == 7.0)
    ts.ts_lm_head_sample(s.handle, h, b)           # and the restored call runs
    torch.cuda.synchronize()
    assert np.all(b.ids() >= 0)


def test_lm_head_sample_in_a_graph(ts):
    """Captured in a CUDA graph with the fused step advance: replays of one
    graph over three frames' hidden states give the ids of three plain calls."""
    frames = [workloads.make_lm_head(t, streams=8, dim=256, vocabs=(512, 384), eos_ids=[-1, -1])
              for t in range(3)]
    batch, head = frames[0]
    s = ts.Sampler(0, 64)
    plain = []
    b = ts.DeviceBatch(batch, "cuda", advance_steps=True)
    h = ts.LmHead(head, "cuda")
    for _, hd in frames:
        h.set_hidden(torch.from_numpy(hd["hidden"].view(np.int16)).cuda())
        ts.ts_lm_head_sample(s.handle, h, b)
        torch.cuda.synchronize()
        plain.append(b.ids())
    b2 = ts.DeviceBatch(batch, "cuda", advance_steps=True)
    hid = torch.empty_like(h.hidden)
    h.set_hidden(hid)
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        ts.ts_lm_head_sample(s.handle, h, b2, st)  # warm-up outside the capture
        st.synchronize()
        b2.step.copy_(torch.from_numpy(batch["step"]).cuda())
        st.synchronize()
        with torch.cuda.graph(g, stream=st):
            ts.ts_lm_head_sample(s.handle, h, b2, st)
    for i, (_, hd) in enumerate(frames):
        hid.copy_(torch.from_numpy(hd["hidden"].view(np.int16)).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(b2.ids(), plain[i]), i


def test_lm_head_sample_refusal_comes_before_the_head(ts):
    """A refusal of the sampler (the repetition penalty on fp32 rows wider
    than 2048) is returned before the head runs: the logits are untouched.
    The head alone still runs."""
    batch, head = workloads.make_lm_head(0, streams=4, dim=128, vocabs=(3072, 2048),
                                         eos_ids=[-1, -1])
    s = ts.Sampler(0, 64)
    b = ts.DeviceBatch(batch, "cuda", history={"len": 4, "codebooks": 2,
                                               "penalty": np.ones(batch["n_rows"], np.float32)})
    h = ts.LmHead(head, "cuda")
    b.set_logits(torch.full_like(b.logits, 7.0))
    with pytest.raises(ts.SamplerError) as e:
        ts.ts_lm_head_sample(s.handle, h, b)
    assert e.value.status == ts.TS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(b.logits == 7.0)
    ts.ts_lm_head_logits(s.handle, h, b)
    torch.cuda.synchronize()
    got = b.logits.cpu().numpy()
    want = oracle.lm_head(batch, head)
    check_logits(batch, head, got, want)
