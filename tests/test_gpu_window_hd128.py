"""Sliding-window attention at the model's real head size (head_dim 128)
against the oracle, for the attention kernels that the single-step decode
tests do not reach: the tensor-core and the CUDA-core prefill attentions, and
the batched-decode attention.

The sliding window is the edge case the model is built around (Blog,
"Designing the architecture": sliding-window attention in 10 of the 15
layers).  The models here have the full width (d_model 4096, 32 query and 16
KV heads of 128, 8 lanes) and fewer layers, a narrower FFN and a smaller
vocabulary, so that the oracle can step through thousands of positions:

- small windows (100 and 40 keys next to a full layer) crossed by a
  300-position prompt: several 128-query and 128-key tiles on each side of
  every window edge;
- the real 1024-key window, crossed by a 1300-position prompt, continued by a
  second prefill to 3584 positions (the long workload's prompt length) and by
  decode steps;
- prefills that start after decode steps;
- batched decode with KV fills past the 1024-key window and past the point
  where the key splits reach their cap (2048 keys).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import REL_L2, assert_gates, note, teacher_forced

pytestmark = pytest.mark.gpu

# full width, three layers: full attention, a 100-key and a 40-key window
SMALL_WIN = synth.FULL.replace(n_layers=3, ffn_dim=1024, vocab=2048, swa_window=(0, 100, 40), ctx_cap=2048)
# full width, two layers: full attention and the model's 1024-key window
REAL_WIN = synth.FULL.replace(n_layers=2, ffn_dim=1024, vocab=2048, swa_window=(0, 1024), ctx_cap=4096)


def prefill_against_oracle(shape, seed, lead, n_prompt, n_steps, tensor_cores):
    """`lead` decode steps, one batched prefill of n_prompt ids, n_steps
    teacher-forced decode steps; every logits vector against the oracle."""
    from decode_persistent_sm_gb300 import Engine
    blob = synth.make_weights(shape, seed, gain_std=0.1)
    tokens = synth.make_tokens(seed, lead + n_prompt + n_steps, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.set_prefill_attention(tensor_cores)
        for t in tokens[:lead]:
            got, am = eng.decode_step(int(t))
            assert note(got, orc.step(int(t)), am) <= REL_L2
        got, am = eng.prefill_batched(tokens[lead:lead + n_prompt])
        for t in tokens[lead:lead + n_prompt]:
            ref = orc.step(int(t))
        assert eng.position == lead + n_prompt
        assert note(got, ref, am) <= REL_L2 and am == oracle.argmax(ref)
        rels, agree, _, _ = teacher_forced(eng, orc, tokens[lead + n_prompt:])
        assert_gates(rels, agree, f"after a {n_prompt}-id prefill from position {lead}")


@pytest.mark.parametrize("tensor_cores", [True, False], ids=["tcgen05", "cuda_cores"])
def test_prefill_small_windows_crossed(tensor_cores):
    prefill_against_oracle(SMALL_WIN, 31, 0, 300, 4, tensor_cores)


@pytest.mark.parametrize("tensor_cores", [True, False], ids=["tcgen05", "cuda_cores"])
def test_prefill_after_decode_steps_small_windows(tensor_cores):
    # the prefill starts at position 37; the 40-key window of its first query
    # reaches back into the positions the decode steps wrote
    prefill_against_oracle(SMALL_WIN, 32, 37, 150, 3, tensor_cores)


@pytest.mark.slow
def test_prefill_past_the_1024_window_to_3584_ids():
    """One oracle pass over 3584 + 2 ids; each prefill attention then runs a
    1300-id prefill (window crossed by 276 keys), a second prefill from 1300
    to 3584 and two decode steps."""
    from decode_persistent_sm_gb300 import Engine
    shape = REAL_WIN
    blob = synth.make_weights(shape, 33, gain_std=0.1)
    tokens = synth.make_tokens(33, 3586, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    want = {}
    for i, t in enumerate(tokens):
        z = orc.step(int(t))
        if i in (1299, 3583, 3584, 3585):
            want[i] = z
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        for tc in (True, False):
            eng.reset()
            eng.set_prefill_attention(tc)
            got, am = eng.prefill_batched(tokens[:1300])
            assert note(got, want[1299], am) <= REL_L2 and am == oracle.argmax(want[1299]), tc
            got, am = eng.prefill_batched(tokens[1300:3584])
            assert note(got, want[3583], am) <= REL_L2 and am == oracle.argmax(want[3583]), tc
            for i in (3584, 3585):
                got, am = eng.decode_step(int(tokens[i]))
                assert note(got, want[i], am) <= REL_L2 and am == oracle.argmax(want[i]), (tc, i)


def batch_against_oracle(shape, seed, kv_fill, n_steps, B):
    from decode_persistent_sm_gb300 import Engine
    blob = synth.make_weights(shape, seed, gain_std=0.1)
    kv = synth.make_kv(shape, seed, kv_fill)
    steps = [synth.make_tokens(seed * 100 + b, n_steps, shape.vocab) for b in range(B)]
    orcs = []
    for b in range(B):
        o = oracle.Oracle(shape, blob)
        o.load_kv(kv, kv_fill)
        orcs.append(o)
    rels, agree = [], []
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.load_kv(kv, kv_fill)
        eng.batch_begin(B)
        for i in range(n_steps):
            toks = [int(steps[b][i]) for b in range(B)]
            got, am = eng.batch_step(toks)
            for b in range(B):
                ref = orcs[b].step(toks[b])
                rels.append(note(got[b], ref, am[b]))
                agree.append(am[b] == oracle.argmax(ref))
    assert_gates(np.array(rels), np.array(agree), f"batch of {B} from a KV fill of {kv_fill}")


def test_batch_decode_small_windows_crossed():
    batch_against_oracle(SMALL_WIN, 34, 300, 4, 3)


@pytest.mark.parametrize("kv_fill", [1030, 2100])
def test_batch_decode_past_the_1024_window_and_the_split_cap(kv_fill):
    # 1030: the window starts inside the first 128-key split; 2100: the full
    # layer's keys need more than 16 splits of 128, so the splits grow
    batch_against_oracle(REAL_WIN, 35, kv_fill, 3, 2)
