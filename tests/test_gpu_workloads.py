"""Parity on the end-to-end, long-context and sweep workloads at the full
2.3B lane-model shape (all synthetic, seed 1).

- End to end: a 128-token prompt, then 512 greedy steps chained on the device
  (positions 127..638 decoded).  The generated tokens are replayed
  teacher-forced through lf_decode_step (same tokens, same logits bit for
  bit) and every one of the 512 steps is compared with the oracle.
- Long context: cache filled to 3584, the first 8 decode steps there (the
  end of the cache, 4090..4095, is covered by test_gpu_full).
- Sweep: cache filled to 2048, 3 steps for each delay in {0, 1, 2} and lane
  count in {1, 8}, each against the oracle of its own variant.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import assert_gates, teacher_forced

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SEED = 1


@pytest.fixture(scope="module")
def full_blob():
    return synth.make_weights(synth.FULL, SEED)


def test_end_to_end_prompt_128_greedy_512(full_blob):
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL
    prompt = synth.make_tokens(SEED, 128, shape.vocab)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(full_blob)
        eng.prefill(prompt[:-1], logits=False)
        gen, _ = eng.generate(int(prompt[-1]), 512)
        assert eng.position == 639
        feed = np.concatenate([prompt[-1:], gen[:-1]]).astype(np.int32)
        # replay teacher-forced: the chain must be reproduced exactly
        eng.reset()
        eng.prefill(prompt[:-1], logits=False)
        orc = oracle.Oracle(shape, full_blob)
        for t in prompt[:-1]:
            orc.step(int(t))
        rels, agree, _, _ = teacher_forced(eng, orc, feed)
        eng.set_position(127)
        replay = [eng.decode_step(int(t), logits=False)[1] for t in feed]
    assert replay == gen.tolist()
    assert_gates(rels, agree, "prompt 128 + 512 greedy steps")


def test_long_context_from_3584(full_blob):
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL
    n0 = 3584
    kv = synth.make_kv(shape, SEED + 7, n0)
    tokens = synth.make_tokens(SEED + 7, 8, shape.vocab)
    orc = oracle.Oracle(shape, full_blob)
    orc.load_kv(kv, n0)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(full_blob)
        eng.load_kv(kv, n0)
        rels, agree, _, _ = teacher_forced(eng, orc, tokens)
    assert_gates(rels, agree, "positions 3584..3591")


@pytest.mark.parametrize("delay", [0, 1, 2])
@pytest.mark.parametrize("lanes", [1, 8])
def test_sweep_context_2048(full_blob, delay, lanes):
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL.replace(n_lanes=lanes, dtp_delay=delay)
    kv = synth.make_kv(shape, SEED + 13, 2048)
    tokens = synth.make_tokens(SEED + 13, 3, shape.vocab)
    orc = oracle.Oracle(shape, full_blob)
    orc.load_kv(kv, 2048)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(full_blob)
        eng.load_kv(kv, 2048)
        rels, agree, _, _ = teacher_forced(eng, orc, tokens)
    assert_gates(rels, agree, f"context 2048, lanes={lanes} delay={delay}")
