"""GPU parity of the decode attention over the head layouts the planner
accepts: q heads per KV head (the group: 1, 2 or 4 per lane), one or two
lane-local KV heads per attention chunk (odd counts take one head at a time),
several chunks per lane, and lanes sharing a KV head.  The tiny model's
cache is filled deep enough that one CTA's share of the keys spans several
32-key tiles, then steps are teacher-forced against the oracle."""
import pytest

import oracle
import synth
from gpu_helpers import REL_L2, assert_gates, teacher_forced

pytestmark = pytest.mark.gpu


# (q heads, KV heads, lanes, KV fill): per lane q heads HQ_L = q / lanes,
# group = q / KV, lane-local KV heads HQ_L / group (1 when lanes share one)
CASES = [
    (8, 2, 1, 2000),   # group 4, two KV heads per lane: one chunk of two
    (8, 2, 2, 3000),   # group 4, one KV head per lane; 2 tiles per CTA
    (8, 2, 4, 2000),   # two lanes share a KV head (group 2 per lane)
    (16, 4, 2, 3000),  # group 4, two KV heads per lane; 2 tiles per CTA
    (8, 8, 2, 3000),   # group 1, four KV heads per lane: two chunks
    (8, 8, 8, 2000),   # group 1, one KV head per lane; 4 tiles per CTA
    (6, 3, 1, 2000),   # three KV heads per lane: three chunks of one
    (12, 3, 1, 2000),  # group 4, three KV heads per lane
]


@pytest.mark.parametrize("nq,nkv,lanes,fill", CASES)
def test_head_layout_against_oracle(nq, nkv, lanes, fill):
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY.replace(n_q_heads=nq, n_kv_heads=nkv, n_lanes=lanes, ctx_cap=4096, swa_window=(100, 0))
    seed = 31 + nq + nkv + lanes
    blob = synth.make_weights(shape, seed, gain_std=0.1)
    kv = synth.make_kv(shape, seed, fill)
    tokens = synth.make_tokens(seed, 6, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    orc.load_kv(kv, fill)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.load_kv(kv, fill)
        rels, agree, _, _ = teacher_forced(eng, orc, tokens)
    assert_gates(rels, agree, f"q {nq} / KV {nkv}, lanes {lanes}, fill {fill}")
    assert rels.max() <= REL_L2
