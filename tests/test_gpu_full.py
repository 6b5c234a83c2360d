"""GPU parity at the full 2.3B lane-model shape (one engine for the module).

Covers the single-step microbench (cache pre-filled with N(0,1) values to
position 512), a teacher-forced run from an empty cache, the long-context end
of the cache (positions up to 4095) and the delay / lane variants."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import REL_L2, assert_gates, note, rel_l2, teacher_forced

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SEED = 1


@pytest.fixture(scope="module")
def full_blob():
    return synth.make_weights(synth.FULL, SEED)


@pytest.fixture(scope="module")
def engine(full_blob):
    from decode_persistent_sm_gb300 import Engine
    eng = Engine.from_shape(synth.FULL)
    eng.load_weights(full_blob)
    yield eng
    eng.close()


def test_microbench_step_at_512(engine, full_blob):
    shape = synth.FULL
    kv = synth.make_kv(shape, SEED, 512)
    tok = int(synth.make_tokens(SEED, 1, shape.vocab)[0])
    orc = oracle.Oracle(shape, full_blob)
    orc.load_kv(kv, 512)
    engine.reset()
    engine.load_kv(kv, 512)
    ref = orc.step(tok)
    got, am = engine.decode_step(tok)
    assert note(got, ref, am) <= REL_L2
    assert am == oracle.argmax(ref)
    # same step again at the same position: bitwise identical
    engine.set_position(512)
    got2, am2 = engine.decode_step(tok)
    assert np.array_equal(got, got2) and am2 == am


def test_teacher_forced_from_empty_cache(engine, full_blob):
    shape = synth.FULL
    tokens = synth.make_tokens(SEED, 12, shape.vocab)
    orc = oracle.Oracle(shape, full_blob)
    engine.reset()
    rels, agree, _, _ = teacher_forced(engine, orc, tokens)
    assert_gates(rels, agree, "full shape, positions 0..11")


def test_long_context_end(engine, full_blob):
    # cache pre-filled to 4090; steps at 4090..4095 cross the full layers'
    # whole-cache reads and end at the context cap
    shape = synth.FULL
    n0 = 4090
    kv = synth.make_kv(shape, SEED + 5, n0)
    tokens = synth.make_tokens(SEED + 5, 6, shape.vocab)
    orc = oracle.Oracle(shape, full_blob)
    orc.load_kv(kv, n0)
    engine.reset()
    engine.load_kv(kv, n0)
    rels, agree, _, _ = teacher_forced(engine, orc, tokens)
    assert_gates(rels, agree, "positions 4090..4095")
    assert engine.position == 4096
    from decode_persistent_sm_gb300 import LaneformerError
    with pytest.raises(LaneformerError, match="CTX_OVERFLOW"):
        engine.decode_step(0)


@pytest.mark.parametrize("pos", [0, 1, 1023, 1024, 1025, 2047])
def test_window_edges_single_step(engine, full_blob, pos):
    # positions around the 1024-key window of the SWA layers
    shape = synth.FULL
    kv = synth.make_kv(shape, SEED + 11, max(pos, 1))
    tok = int(synth.make_tokens(SEED + pos, 1, shape.vocab)[0])
    orc = oracle.Oracle(shape, full_blob)
    engine.reset()
    if pos > 0:
        orc.load_kv(kv, pos)
        engine.load_kv(kv, pos)
    ref = orc.step(tok)
    got, am = engine.decode_step(tok)
    assert note(got, ref, am) <= REL_L2
    assert am == oracle.argmax(ref)


@pytest.mark.parametrize("lanes,delay", [(8, 0), (8, 1), (1, 0), (1, 2)])
def test_delay_lane_variants(full_blob, lanes, delay):
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL.replace(n_lanes=lanes, dtp_delay=delay)
    kv = synth.make_kv(shape, SEED + 21, 300)
    tokens = synth.make_tokens(SEED + 21, 3, shape.vocab)
    orc = oracle.Oracle(shape, full_blob)
    orc.load_kv(kv, 300)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(full_blob)
        eng.load_kv(kv, 300)
        rels, agree, _, _ = teacher_forced(eng, orc, tokens)
    assert_gates(rels, agree, f"lanes={lanes} delay={delay}")
