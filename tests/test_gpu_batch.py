"""Batched decode (lf_batch_begin / lf_batch_step / lf_batch_generate) and its
tensor-core GEMV (lf_gemv_f16) against the oracle.

Each sample of a batch continues the engine's sequence on its own tokens and
must match an oracle that ran the same prompt and then that sample's tokens
(teacher forced), at the same gates as the single-sequence decode.  The GEMV
is checked against an fp64 product of the same FP16 operands, and for
determinism (the split reduction is summed in a fixed order)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import REL_L2, assert_gates, note, rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,k,batch", [(1000, 256, 1), (4096, 4096, 8), (8192, 4096, 16), (300, 128, 3),
                                       (64, 64, 16), (32000, 4096, 5), (4096, 7168, 2), (200, 4096, 7)])
def test_gemv_against_fp64(n, k, batch):
    import torch
    from decode_persistent_sm_gb300 import gemv_f16
    g = np.random.default_rng(n + k + batch)
    w = (0.02 * g.standard_normal((n, k))).astype(np.float16)
    x = g.standard_normal((batch, k)).astype(np.float16)
    wd, xd = torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda()
    ys = []
    for _ in range(2):
        y = torch.full((batch, n), float("nan"), dtype=torch.float32, device="cuda")
        gemv_f16(wd.data_ptr(), xd.data_ptr(), y.data_ptr(), n, k, batch)
        ys.append(y.cpu().numpy())
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    scale = np.sqrt(k) * 0.02
    assert np.all(np.isfinite(ys[0]))
    assert np.abs(ys[0] - ref).max() <= 1e-4 * scale + 1e-5 * np.abs(ref).max()
    assert np.array_equal(ys[0], ys[1]), "the split reduction must be deterministic"


def test_gemv_rejections():
    import torch
    from decode_persistent_sm_gb300 import LaneformerError, gemv_f16
    w = torch.zeros((128, 128), dtype=torch.float16, device="cuda")
    y = torch.zeros((17, 128), dtype=torch.float32, device="cuda")
    for n, k, b in [(128, 100, 1), (128, 128, 0), (128, 128, 17), (0, 128, 1)]:
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            gemv_f16(w.data_ptr(), w.data_ptr(), y.data_ptr(), n, k, b)


def run_batch(shape, seed, n_prompt, n_steps, B, gain_std=0.1, kv_fill=0):
    """Prompt (decode steps, or a KV fill), then a batch of B samples, sample
    b fed its own tokens; per step and sample the logits against an oracle
    that saw the same prompt and that sample's tokens."""
    from decode_persistent_sm_gb300 import Engine
    blob = synth.make_weights(shape, seed, gain_std=gain_std)
    prompt = synth.make_tokens(seed, n_prompt, shape.vocab)
    steps = [synth.make_tokens(seed * 100 + b, n_steps, shape.vocab) for b in range(B)]
    kv = synth.make_kv(shape, seed, kv_fill) if kv_fill else None
    orcs = []
    for b in range(B):
        o = oracle.Oracle(shape, blob)
        if kv_fill:
            o.load_kv(kv, kv_fill)
        for t in prompt:
            o.step(int(t))
        orcs.append(o)
    rels, agree = [], []
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        if kv_fill:
            eng.load_kv(kv, kv_fill)
        for t in prompt:
            eng.decode_step(int(t))
        eng.batch_begin(B)
        assert eng.batch_info() == (B, kv_fill + n_prompt)
        for i in range(n_steps):
            toks = [int(steps[b][i]) for b in range(B)]
            got, am = eng.batch_step(toks)
            for b in range(B):
                ref = orcs[b].step(toks[b])
                rels.append(note(got[b], ref, am[b]))
                agree.append(am[b] == oracle.argmax(ref))
        assert eng.batch_info() == (B, kv_fill + n_prompt + n_steps)
    return np.array(rels), np.array(agree)


def test_tiny_batch_of_five():
    rels, agree = run_batch(synth.TINY, 3, 20, 10, 5)
    assert_gates(rels, agree, "tiny, batch of 5")


@pytest.mark.parametrize("lanes,delay", [(8, 0), (8, 1), (1, 2), (4, 3)])
def test_tiny_lanes_and_delays(lanes, delay):
    shape = synth.TINY.replace(n_lanes=lanes, dtp_delay=delay)
    rels, agree = run_batch(shape, 4, 9, 6, 3)
    assert_gates(rels, agree, f"batch, lanes={lanes} delay={delay}")


def test_six_layers_windows_crossed():
    # 70-token prompt: the 64-, 16- and 8-key windows are all crossed
    shape = synth.TINY.replace(n_layers=6, swa_window=(64, 0, 16, 0, 8, 0))
    rels, agree = run_batch(shape, 5, 70, 6, 4)
    assert_gates(rels, agree, "batch, 6 layers")


@pytest.mark.parametrize("B", [1, 16])
def test_batch_sizes(B):
    rels, agree = run_batch(synth.TINY, 6, 12, 5, B)
    assert_gates(rels, agree, f"batch of {B}")


def test_batch_from_an_empty_sequence():
    rels, agree = run_batch(synth.TINY, 7, 0, 8, 2)
    assert_gates(rels, agree, "batch from position 0")


def test_engine_sequence_untouched_by_the_batch():
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY
    blob = synth.make_weights(shape, 8, gain_std=0.1)
    toks = synth.make_tokens(8, 30, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        for t in toks[:20]:
            eng.decode_step(int(t))
            orc.step(int(t))
        eng.batch_begin(3)
        for i in range(5):
            eng.batch_step([int(toks[(i + 7 * b) % 30]) for b in range(3)])
        for t in toks[20:]:
            got, _ = eng.decode_step(int(t))
            assert note(got, orc.step(int(t))) <= REL_L2
        eng.batch_end()
        assert eng.batch_info() == (0, 0)


def test_rejections():
    from decode_persistent_sm_gb300 import Engine, LaneformerError
    shape = synth.TINY
    with Engine.from_shape(shape) as eng:
        with pytest.raises(LaneformerError, match="NOT_LOADED"):
            eng.batch_begin(2)
        eng.load_weights(synth.make_weights(shape, 1))
        with pytest.raises(LaneformerError, match="NOT_LOADED"):
            eng.batch_step([1, 2])
        for bad in (0, 17):
            with pytest.raises(LaneformerError, match="INVALID_ARG"):
                eng.batch_begin(bad)
        eng.prefill(synth.make_tokens(1, shape.ctx_cap - 2, shape.vocab), logits=False)
        eng.batch_begin(2)
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.batch_step([1, shape.vocab])
        eng.batch_step([1, 2])
        eng.batch_step([3, 4])
        with pytest.raises(LaneformerError, match="CTX_OVERFLOW"):
            eng.batch_step([5, 6])
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.batch_generate([1, 2], 1, -1.0, 0.9, 0)
    with Engine.from_shape(shape.replace(own_lane_immediate=1)) as eng:
        eng.load_weights(synth.make_weights(shape, 1))
        with pytest.raises(LaneformerError, match="UNSUPPORTED"):
            eng.batch_begin(2)


def valid_draw(z, tok, temperature, top_p, u, slack):
    z = np.asarray(z, dtype=np.float64)
    p = np.exp((z - z.max()) / temperature)
    s = np.sort(p)[::-1]
    tau = s[np.searchsorted(np.cumsum(s), top_p * p.sum() * (1 - slack))]
    keep = p >= tau * (1 - slack)
    if not keep[tok]:
        return False
    kept = p[keep].sum()
    before = p[:tok][keep[:tok]].sum()
    t = u * kept
    return before <= t + slack * kept and before + p[tok] >= t - slack * kept


def test_sampled_batch_against_the_oracle_and_repeatable():
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY
    blob = synth.make_weights(shape, 21, gain_std=0.1)
    prompt = synth.make_tokens(21, 16, shape.vocab)
    T, top_p, seed, B, n = 0.8, 0.9, 77, 4, 30
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.prefill(prompt[:-1], logits=False)
        eng.batch_begin(B)
        toks = eng.batch_generate([int(prompt[-1])] * B, n, T, top_p, seed)
        assert eng.batch_info() == (B, 15 + n)
        eng.batch_begin(B)
        again = eng.batch_generate([int(prompt[-1])] * B, n, T, top_p, seed)
    assert np.array_equal(toks, again)
    assert len({tuple(r) for r in toks}) == B  # independent streams per sample
    same = 0
    for b in range(B):
        orc = oracle.Oracle(shape, blob)
        for t in prompt[:-1]:
            orc.step(int(t))
        feed = [int(prompt[-1])] + [int(t) for t in toks[b][:-1]]
        for i, (t, got) in enumerate(zip(feed, toks[b])):
            z = orc.step(t)
            ref, u, _ = oracle.sample(z, T, top_p, seed, 15 + i, b)
            if ref == got:
                same += 1
            else:  # the logits differ from the oracle's at the 1e-3 level
                assert valid_draw(z, int(got), T, top_p, u, 5e-3), (b, i, got, ref)
    assert same >= B * n - 3


def test_greedy_batch_generate_is_the_argmax_chain():
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY
    blob = synth.make_weights(shape, 22, gain_std=0.1)
    prompt = synth.make_tokens(22, 10, shape.vocab)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.prefill(prompt, logits=False)
        eng.batch_begin(2)
        toks = eng.batch_generate([3, 9], 12, 0.0, 1.0, 0)
        eng.batch_begin(2)
        feed = [3, 9]
        for i in range(12):
            _, am = eng.batch_step(feed)
            assert list(am) == list(toks[:, i])
            feed = [int(a) for a in am]


@pytest.mark.slow
def test_full_shape_batch_against_the_oracle():
    rels, agree = run_batch(synth.FULL, 1, 0, 2, 3, gain_std=0.0, kv_fill=300)
    assert_gates(rels, agree, "full shape, batch of 3")


@pytest.mark.slow
def test_full_shape_batch_matches_the_single_sequence_decode():
    # both GPU paths, many steps: each sample fed the single-sequence decode's tokens
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL
    blob = synth.make_weights(shape, 2)
    kv = synth.make_kv(shape, 2, 700)
    toks = synth.make_tokens(2, 24, shape.vocab)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.load_kv(kv, 700)
        eng.batch_begin(2)
        for t in toks:
            single, am1 = eng.decode_step(int(t))
            got, am = eng.batch_step([int(t), int(t)])
            for b in range(2):
                assert rel_l2(got[b], single) <= REL_L2
            assert np.array_equal(got[0], got[1])
