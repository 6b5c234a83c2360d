"""GPU parity on the tiny lane model (and variants) through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import assert_gates, note, rel_l2, teacher_forced

pytestmark = pytest.mark.gpu


def engine_for(shape):
    from decode_persistent_sm_gb300 import Engine
    return Engine.from_shape(shape)


def run_case(shape, seed=0, n=48, gain_std=0.0):
    blob = synth.make_weights(shape, seed, gain_std=gain_std)
    tokens = synth.make_tokens(seed, n, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    with engine_for(shape) as eng:
        eng.load_weights(blob)
        return teacher_forced(eng, orc, tokens)


def test_tiny_workload_prompt16_greedy32():
    # prompt of 16 ids, then 32 more steps (teacher forced), context cap 128
    rels, agree, _, _ = run_case(synth.TINY, seed=0, n=48)
    assert_gates(rels, agree, "tiny")
    assert agree.all()


@pytest.mark.parametrize("lanes,delay", [(8, 0), (8, 1), (8, 2), (1, 0), (1, 2), (2, 1), (4, 2)])
def test_tiny_lanes_and_delays(lanes, delay):
    shape = synth.TINY.replace(n_lanes=lanes, dtp_delay=delay)
    rels, agree, _, _ = run_case(shape, seed=3, n=40, gain_std=0.1)
    assert_gates(rels, agree, f"lanes={lanes} delay={delay}")


@pytest.mark.parametrize("delay", [0, 1, 2])
def test_six_layers_exercise_the_delayed_sum(delay):
    shape = synth.TINY.replace(n_layers=6, dtp_delay=delay, swa_window=(64, 0, 16, 0, 5, 0))
    rels, agree, _, _ = run_case(shape, seed=7, n=40, gain_std=0.1)
    assert_gates(rels, agree, f"L=6 delay={delay}")


def test_windows_at_boundaries():
    # windows 1 and 3 and a window equal to the run length
    shape = synth.TINY.replace(swa_window=(1, 3))
    rels, agree, _, _ = run_case(shape, seed=9, n=24, gain_std=0.1)
    assert_gates(rels, agree, "windows 1/3")


def test_kv_append_matches_oracle():
    shape = synth.TINY
    blob = synth.make_weights(shape, 11, gain_std=0.1)
    tokens = synth.make_tokens(11, 10, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    with engine_for(shape) as eng:
        eng.load_weights(blob)
        teacher_forced(eng, orc, tokens)
        for layer in range(shape.n_layers):
            for kvh in range(shape.n_kv_heads):
                lane = kvh * (shape.n_q_heads // shape.n_kv_heads) // (shape.n_q_heads // shape.n_lanes)
                for pos in (0, 5, 9):
                    k, v = eng.read_kv(layer, kvh, pos)
                    rk, rv = orc.kv(lane, layer, 0, pos)
                    # both sides round K and V to FP16; allow one FP16 ulp
                    assert np.allclose(k, rk, rtol=2e-3, atol=1e-4)
                    assert np.allclose(v, rv, rtol=2e-3, atol=1e-4)


def test_prefill_equals_steps_and_reset():
    shape = synth.TINY
    blob = synth.make_weights(shape, 13)
    tokens = synth.make_tokens(13, 20, shape.vocab)
    with engine_for(shape) as eng:
        eng.load_weights(blob)
        lg1, am1 = eng.prefill(tokens)
        assert eng.position == 20
        eng.reset()
        assert eng.position == 0
        for t in tokens[:-1]:
            eng.decode_step(int(t), logits=False)
        lg2, am2 = eng.decode_step(int(tokens[-1]))
        assert am1 == am2
        assert np.array_equal(lg1, lg2)  # same kernels, same order: bitwise


def test_repeated_step_is_deterministic():
    shape = synth.TINY
    blob = synth.make_weights(shape, 15)
    tokens = synth.make_tokens(15, 12, shape.vocab)
    with engine_for(shape) as eng:
        eng.load_weights(blob)
        eng.prefill(tokens[:-1], logits=False)
        a, _ = eng.decode_step(int(tokens[-1]))
        eng.set_position(11)
        b, _ = eng.decode_step(int(tokens[-1]))
        assert np.array_equal(a, b)


def test_error_paths():
    from decode_persistent_sm_gb300 import LaneformerError
    shape = synth.TINY.replace(ctx_cap=8)
    with engine_for(shape) as eng:
        with pytest.raises(LaneformerError, match="NOT_LOADED"):
            eng.decode_step(1)
        eng.load_weights(synth.make_weights(shape, 1))
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.decode_step(shape.vocab)
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.decode_step(-1)
        with pytest.raises(LaneformerError, match="CTX_OVERFLOW"):
            eng.prefill(list(range(9)))
        eng.prefill(list(range(8)), logits=False)
        with pytest.raises(LaneformerError, match="CTX_OVERFLOW"):
            eng.decode_step(0)
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.set_position(9)
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.load_weights(np.zeros(10, dtype=np.uint16))
        eng.set_position(0)
        eng.decode_step(3)


def test_async_steps_then_synchronous_step():
    shape = synth.TINY
    blob = synth.make_weights(shape, 17)
    tokens = synth.make_tokens(17, 8, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    with engine_for(shape) as eng:
        eng.load_weights(blob)
        for t in tokens[:-1]:
            eng.decode_step_async(int(t))  # enqueued only
            orc.step(int(t))
        eng.synchronize()
        got, am = eng.decode_step(int(tokens[-1]))
        ref = orc.step(int(tokens[-1]))
        assert note(got, ref, am) < 1e-2 and am == oracle.argmax(ref)
        assert eng.logits_device_ptr() != 0 and eng.argmax_device_ptr() != 0
