"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a library routine, a closed form, an
invariant or a special case that reduces to a textbook model, chosen so that a
plausible mistake (a dropped gain, a wrong RoPE pairing, a GQA head mapping,
an off-by-one in the delay or the window, a missing FP16 rounding) fails one
of them.
"""
import numpy as np
import pytest

import oracle
import synth
from dense_reference import closed_form_all_read_embedding, delayed_lanes, standard_transformer

RTOL = 1e-9  # fp64 on both sides; only the summation order differs


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / np.linalg.norm(np.asarray(b)))


def tiny(**kw):
    return synth.TINY.replace(**kw)


def run_oracle(shape, blob, tokens, **kw):
    return oracle.Oracle(shape, blob, **kw).run(tokens)


# ------------------------------------------------------------------ binary16

def test_half_decode_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_half_round_matches_numpy():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        # exact ties between neighbouring halves, subnormals, overflow edge
        (np.arange(0, 2048, dtype=np.float64) + 0.5) * 2.0 ** -24,
        (1024 + np.arange(0, 1024) + 0.5) * 2.0 ** -10,
        [0.0, -0.0, 65504.0, 65519.999, 65520.0, -65520.0, 6.1e-5, 2.0 ** -14, 2.0 ** -25,
         2.0 ** -25 * 1.0000001, 1e-30, 1e30],
    ])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref), vals[got != ref][:5]


def test_argmax_lowest_index_on_ties():
    x = np.zeros(100)
    x[[7, 30, 99]] = 3.0
    assert oracle.argmax(x) == 7
    x[2] = 3.0
    assert oracle.argmax(x) == 2
    assert oracle.argmax(np.full(5, -1.0)) == 0


# --------------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal(128)
    assert np.array_equal(oracle.rope(x, 0, 1e4), x)


def test_rope_matches_complex_rotation_and_keeps_norm():
    rng = np.random.default_rng(2)
    for dh in (32, 128):
        x = rng.standard_normal(dh)
        for p in (1, 17, 4095):
            y = oracle.rope(x, p, 1e4)
            half = dh // 2
            z = (x[:half] + 1j * x[half:]) * np.exp(1j * p * 1e4 ** (-2.0 * np.arange(half) / dh))
            assert np.allclose(y, np.concatenate([z.real, z.imag]), rtol=1e-12, atol=1e-12)
            assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-11


def test_rope_dot_depends_only_on_offset():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    ref = oracle.rope(q, 40, 1e4) @ oracle.rope(k, 33, 1e4)
    for shift in (1, 100, 3000):
        got = oracle.rope(q, 40 + shift, 1e4) @ oracle.rope(k, 33 + shift, 1e4)
        assert abs(got - ref) < 1e-9 * max(1.0, abs(ref))


# ------------------------------------------------------- whole-model pins

@pytest.fixture(scope="module")
def tiny_blob():
    # random RMSNorm gains so that a gain that is dropped or misplaced shows
    return synth.make_weights(synth.TINY, 0, gain_std=0.1)


@pytest.fixture(scope="module")
def tiny_tokens():
    return synth.make_tokens(0, 40, synth.TINY.vocab)


@pytest.mark.parametrize("lanes", [1, 8])
@pytest.mark.parametrize("round_kv", [True, False])
def test_delay0_equals_standard_transformer(tiny_blob, tiny_tokens, lanes, round_kv):
    shape = tiny(dtp_delay=0, n_lanes=lanes)
    got = run_oracle(shape, tiny_blob, tiny_tokens, round_kv_fp16=round_kv)
    ref = standard_transformer(shape, tiny_blob, tiny_tokens, round_kv=round_kv)
    assert rel(got, ref) < RTOL


def test_fp16_kv_rounding_matters(tiny_blob, tiny_tokens):
    # the two settings differ, so the pins above do test the rounding
    shape = tiny(dtp_delay=0)
    a = run_oracle(shape, tiny_blob, tiny_tokens[:8], round_kv_fp16=True)
    b = run_oracle(shape, tiny_blob, tiny_tokens[:8], round_kv_fp16=False)
    assert rel(a, b) > 1e-6


def test_delay0_mha_special_case(tiny_tokens):
    shape = tiny(dtp_delay=0, n_kv_heads=8)
    blob = synth.make_weights(shape, 5, gain_std=0.1)
    assert rel(run_oracle(shape, blob, tiny_tokens[:20]),
               standard_transformer(shape, blob, tiny_tokens[:20])) < RTOL


def test_lanes_are_exact_tensor_parallelism_at_delay0(tiny_blob, tiny_tokens):
    a = run_oracle(tiny(dtp_delay=0, n_lanes=8), tiny_blob, tiny_tokens)
    b = run_oracle(tiny(dtp_delay=0, n_lanes=1), tiny_blob, tiny_tokens)
    assert rel(a, b) < 1e-12


def test_lane_order_is_irrelevant(tiny_blob, tiny_tokens):
    shape = tiny(n_layers=6, swa_window=(64, 0, 16, 0, 64, 0), dtp_delay=1)
    blob = synth.make_weights(shape, 7, gain_std=0.1)
    a = run_oracle(shape, blob, tiny_tokens[:24])
    b = run_oracle(shape, blob, tiny_tokens[:24], lane_order=[5, 2, 7, 0, 3, 6, 1, 4])
    assert rel(a, b) < 1e-12


def test_window_at_least_context_equals_full(tiny_blob, tiny_tokens):
    a = run_oracle(tiny(swa_window=(0, 0)), tiny_blob, tiny_tokens)
    b = run_oracle(tiny(swa_window=(40, 128)), tiny_blob, tiny_tokens)
    assert rel(a, b) < 1e-13
    c = run_oracle(tiny(swa_window=(39, 0)), tiny_blob, tiny_tokens)  # one key short at the end
    assert rel(a[:-1], c[:-1]) < 1e-13 and rel(a[-1], c[-1]) > 1e-8


@pytest.mark.parametrize("window", [1, 5, 16])
def test_sliding_window_matches_masked_sdpa(tiny_blob, tiny_tokens, window):
    shape = tiny(dtp_delay=0, swa_window=(window, window))
    assert rel(run_oracle(shape, tiny_blob, tiny_tokens),
               standard_transformer(shape, tiny_blob, tiny_tokens)) < RTOL


def test_window_one_attends_to_current_value_only(tiny_tokens):
    # With W = 1 every head attends to its current key alone, so its output is
    # the current V whatever the scores are: scaling Wk (which changes only the
    # scores) must leave the logits unchanged.
    shape = tiny(dtp_delay=0, swa_window=(1, 1))
    blob = synth.make_weights(shape, 9, gain_std=0.1)
    views = synth.weight_views(shape, blob)
    blob2 = blob.copy()
    v2 = synth.weight_views(shape, blob2)
    for l in range(shape.n_layers):
        v2[f"Wk.{l}"][...] = (views[f"Wk.{l}"].astype(np.float64) * 3.0).astype(np.float16)
    a = run_oracle(shape, blob, tiny_tokens[:12])
    b = run_oracle(shape, blob2, tiny_tokens[:12])
    assert rel(a, b) < 1e-13


def test_equal_scores_give_mean_of_values(tiny_tokens):
    # Wq = 0 gives q = 0, every score 0, attention = mean of the window's V.
    shape = tiny(dtp_delay=0, swa_window=(7, 0))
    blob = synth.make_weights(shape, 11, gain_std=0.1)
    v = synth.weight_views(shape, blob)
    for l in range(shape.n_layers):
        v[f"Wq.{l}"][...] = 0
    got = run_oracle(shape, blob, tiny_tokens[:20])
    assert rel(got, standard_transformer(shape, blob, tiny_tokens[:20])) < RTOL


@pytest.mark.parametrize("n_layers,delay", [(2, 2), (3, 3), (1, 1)])
def test_long_delay_closed_form(tiny_tokens, n_layers, delay):
    # 2d + 1 >= 2L: every sub-block reads the embedding alone.
    shape = tiny(n_layers=n_layers, dtp_delay=delay, swa_window=(64, 0, 0)[:n_layers])
    blob = synth.make_weights(shape, 13, gain_std=0.1)
    got = run_oracle(shape, blob, tiny_tokens[:24])
    assert rel(got, closed_form_all_read_embedding(shape, blob, tiny_tokens[:24])) < RTOL


def test_delay_just_below_closed_form_differs(tiny_tokens):
    # L = 3, d = 2: 2d + 1 = 5 < 6, so the last sub-block sees sub-block 0.
    shape = tiny(n_layers=3, dtp_delay=2, swa_window=(64, 0, 0))
    blob = synth.make_weights(shape, 13, gain_std=0.1)
    got = run_oracle(shape, blob, tiny_tokens[:8])
    assert rel(got, closed_form_all_read_embedding(shape, blob, tiny_tokens[:8])) > 1e-6


@pytest.mark.parametrize("delay", [1, 2])
@pytest.mark.parametrize("own", [0, 1])
def test_delayed_lanes_match_prefill_evaluation(tiny_tokens, delay, own):
    shape = tiny(n_layers=6, dtp_delay=delay, own_lane_immediate=own,
                 swa_window=(64, 0, 16, 0, 64, 0))
    blob = synth.make_weights(shape, 17, gain_std=0.1)
    got = run_oracle(shape, blob, tiny_tokens[:24])
    assert rel(got, delayed_lanes(shape, blob, tiny_tokens[:24])) < RTOL


def test_own_lane_immediate_with_one_lane_is_dense(tiny_blob, tiny_tokens):
    shape = tiny(n_lanes=1, dtp_delay=2, own_lane_immediate=1)
    got = run_oracle(shape, tiny_blob, tiny_tokens)
    assert rel(got, standard_transformer(shape, tiny_blob, tiny_tokens)) < RTOL


def test_delay_changes_the_function(tiny_tokens):
    shape = tiny(n_layers=6, swa_window=(64, 0, 16, 0, 64, 0))
    blob = synth.make_weights(shape, 17, gain_std=0.1)
    outs = [run_oracle(shape.replace(dtp_delay=d), blob, tiny_tokens[:8]) for d in (0, 1, 2)]
    assert rel(outs[0], outs[1]) > 1e-6 and rel(outs[1], outs[2]) > 1e-6


def test_kv_prefill_matches_reference_prefix(tiny_tokens):
    # a cache pre-filled with random values (as in the single-step workload)
    shape = tiny(dtp_delay=0, ctx_cap=128)
    blob = synth.make_weights(shape, 19, gain_std=0.1)
    n0 = 50
    kv = synth.make_kv(shape, 19, n0)
    o = oracle.Oracle(shape, blob)
    o.load_kv(kv, n0)
    assert o.pos == n0
    got = o.run(tiny_tokens[:6])
    ref = standard_transformer(shape, blob, tiny_tokens[:6], kv_prefix=kv, n_prefix=n0)
    assert rel(got, ref) < RTOL


def test_context_cap_and_bad_token(tiny_blob):
    shape = tiny(ctx_cap=4)
    o = oracle.Oracle(shape, tiny_blob)
    for t in (1, 2, 3, 4):
        o.step(t)
    with pytest.raises(ValueError, match="context full"):
        o.step(5)
    o.set_pos(0)
    with pytest.raises(ValueError, match="token"):
        o.step(shape.vocab)
