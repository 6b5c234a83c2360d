"""The own-lane-immediate reading of the delayed lane sum on the GPU: each lane
adds its own partial of a sub-block at once and the other lanes' share 2d
sub-blocks later.  Teacher-forced against the oracle run with the same
reading; the two readings give different functions whenever lanes > 1 and the
delay is > 0, and the GPU must follow the one it was asked for."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import REL_L2, assert_gates, note, rel_l2, teacher_forced

pytestmark = pytest.mark.gpu


def run(shape, seed, n, kv_fill=0):
    from decode_persistent_sm_gb300 import Engine
    blob = synth.make_weights(shape, seed, gain_std=0.1 if shape.d_model < 4096 else 0.0)
    tokens = synth.make_tokens(seed, n, shape.vocab)
    orc_b = oracle.Oracle(shape, blob)
    orc_a = oracle.Oracle(shape.replace(own_lane_immediate=0), blob)
    kv = synth.make_kv(shape, seed, kv_fill) if kv_fill else None
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        if kv_fill:
            eng.load_kv(kv, kv_fill)
            orc_b.load_kv(kv, kv_fill)
            orc_a.load_kv(kv, kv_fill)
        rels, agree, gaps = [], [], []
        for t in tokens:
            got, am = eng.decode_step(int(t))
            rb, ra = orc_b.step(int(t)), orc_a.step(int(t))
            rels.append(note(got, rb, am))
            agree.append(am == oracle.argmax(rb))
            gaps.append(rel_l2(ra, rb))
    return np.array(rels), np.array(agree), np.array(gaps)


@pytest.mark.parametrize("lanes,delay", [(8, 1), (8, 2), (4, 3), (2, 2)])
def test_tiny_own_lane(lanes, delay):
    shape = synth.TINY.replace(n_lanes=lanes, dtp_delay=delay, own_lane_immediate=1)
    rels, agree, gaps = run(shape, 13, 40)
    assert_gates(rels, agree, f"own lane, lanes={lanes} delay={delay}")
    # the readings differ by far more than the GPU's error against its own one
    assert gaps.max() > 5 * rels.max()


def test_tiny_own_lane_six_layers():
    shape = synth.TINY.replace(n_layers=6, swa_window=(64, 0, 16, 0, 8, 0), dtp_delay=2, own_lane_immediate=1)
    rels, agree, gaps = run(shape, 14, 30)
    assert_gates(rels, agree, "own lane, 6 layers")


def test_one_lane_own_reading():
    # with one lane, "own" is everything: the sum is never delayed
    shape = synth.TINY.replace(n_lanes=1, dtp_delay=2, own_lane_immediate=1)
    rels, agree, _ = run(shape, 15, 20)
    assert_gates(rels, agree, "own lane, 1 lane")


@pytest.mark.slow
@pytest.mark.parametrize("delay", [1, 2])
def test_full_shape_own_lane(delay):
    shape = synth.FULL.replace(dtp_delay=delay, own_lane_immediate=1)
    rels, agree, gaps = run(shape, 1, 3, kv_fill=300)
    assert_gates(rels, agree, f"full shape, own lane, delay {delay}")
