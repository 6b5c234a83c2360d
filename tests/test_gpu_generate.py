"""Greedy generation chained on the device (lf_generate, lf_decode_step_chained).

Each chained step reads its token from the previous step's argmax in device
memory.  Checked here: the chain gives exactly the tokens and logits of a host
loop that feeds each argmax back through lf_decode_step (same kernel, fixed
summation order); the oracle, teacher-forced with the generated tokens, picks
the same next token at every step; bad arguments are refused on the host and
a token outside the vocabulary found on the device ends in an error status.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import REL_L2, note, rel_l2

pytestmark = pytest.mark.gpu


def host_loop(eng, first, n):
    toks, t = [], int(first)
    logits = None
    for _ in range(n):
        logits, t = eng.decode_step(t)
        toks.append(t)
    return np.array(toks, dtype=np.int32), logits


def oracle_agreement(orc, first, gen):
    """Teacher-forces the oracle with [first, gen[:-1]]; fraction of steps whose
    oracle argmax is the generated token."""
    feed = [int(first)] + [int(t) for t in gen[:-1]]
    hits = [oracle.argmax(orc.step(t)) == int(g) for t, g in zip(feed, gen)]
    return float(np.mean(hits))


def test_tiny_generate_equals_host_loop_and_oracle():
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY
    blob = synth.make_weights(shape, 0, gain_std=0.1)
    prompt = synth.make_tokens(0, 16, shape.vocab)
    with Engine.from_shape(shape) as a, Engine.from_shape(shape) as b:
        a.load_weights(blob)
        b.load_weights(blob)
        a.prefill(prompt[:-1], logits=False)
        b.prefill(prompt[:-1], logits=False)
        gen, last = a.generate(int(prompt[-1]), 32, logits=True)
        ref, ref_last = host_loop(b, prompt[-1], 32)
        assert np.array_equal(gen, ref)
        assert np.array_equal(last, ref_last)
        assert a.position == b.position == 15 + 32
    orc = oracle.Oracle(shape, blob)
    for t in prompt[:-1]:
        orc.step(int(t))
    assert oracle_agreement(orc, prompt[-1], gen) >= 31 / 32


def test_full_generate_from_filled_cache():
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL
    blob = synth.make_weights(shape, 1)
    kv = synth.make_kv(shape, 1, 512)
    first = int(synth.make_tokens(41, 1, shape.vocab)[0])
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.load_kv(kv, 512)
        gen, last = eng.generate(first, 8, logits=True)
        eng.set_position(512)
        ref, ref_last = host_loop(eng, first, 8)
    assert np.array_equal(gen, ref) and np.array_equal(last, ref_last)
    orc = oracle.Oracle(shape, blob)
    orc.load_kv(kv, 512)
    assert oracle_agreement(orc, first, gen) >= 7 / 8


def test_chained_steps_on_torch_buffers():
    import torch
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY
    blob = synth.make_weights(shape, 3)
    tokens = synth.make_tokens(3, 4, shape.vocab)
    with Engine.from_shape(shape) as a, Engine.from_shape(shape) as b:
        a.load_weights(blob)
        b.load_weights(blob)
        buf = torch.tensor([int(tokens[0]), -1, -1, -1], dtype=torch.int32, device="cuda")
        for i in range(3):  # token from buf[i], argmax into buf[i + 1]
            a.decode_step_chained(buf[i:].data_ptr(), buf[i + 1:].data_ptr())
        a.synchronize()
        ref, _ = host_loop(b, tokens[0], 3)
        assert buf[1:].cpu().numpy().tolist() == ref.tolist()
        # the same word as input and output
        one = torch.tensor([int(tokens[1])], dtype=torch.int32, device="cuda")
        a.decode_step_chained(one.data_ptr(), one.data_ptr())
        a.synchronize()
        _, am = b.decode_step(int(tokens[1]))
        assert int(one.item()) == am


def test_bad_arguments_are_refused_on_the_host():
    from decode_persistent_sm_gb300 import Engine, LaneformerError
    shape = synth.TINY
    with Engine.from_shape(shape) as eng:
        eng.load_weights(synth.make_weights(shape, 4))
        host = np.zeros(2, dtype=np.int32)  # pageable host memory: not readable by the GPU
        assert eng.raw_call("lf_decode_step_chained", ctypes.c_void_p(host.ctypes.data),
                            ctypes.c_void_p(host.ctypes.data + 4)) == 1
        assert eng.raw_call("lf_decode_step_chained", None, None) == 1
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.generate(shape.vocab, 2)
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.generate(0, 0)
        eng.set_position(shape.ctx_cap - 2)
        with pytest.raises(LaneformerError, match="CTX_OVERFLOW"):
            eng.generate(0, 3)
        assert eng.position == shape.ctx_cap - 2
        toks, _ = eng.generate(0, 2)
        assert toks.shape == (2,) and eng.position == shape.ctx_cap


def test_out_of_vocabulary_device_token_poisons_until_reset():
    import torch
    from decode_persistent_sm_gb300 import Engine, LaneformerError
    shape = synth.TINY
    blob = synth.make_weights(shape, 5)
    tokens = synth.make_tokens(5, 3, shape.vocab)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        bad = torch.tensor([shape.vocab + 5, -1], dtype=torch.int32, device="cuda")
        eng.decode_step_chained(bad.data_ptr(), bad[1:].data_ptr())
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.synchronize()
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.decode_step(int(tokens[0]))
        eng.reset()
        orc = oracle.Oracle(shape, blob)
        for t in tokens:
            got, am = eng.decode_step(int(t))
            ref = orc.step(int(t))
            assert note(got, ref, am) <= REL_L2
            assert am == oracle.argmax(ref)


@pytest.mark.parametrize("lanes,delay,own", [(8, 0, 0), (8, 1, 0), (1, 2, 0), (4, 3, 0), (8, 2, 1), (2, 1, 1)])
def test_generate_in_one_launch_equals_separate_steps(lanes, delay, own):
    # lf_generate runs all steps in one launch of the persistent kernel; the
    # tokens and the last logits must be those of one launch per step
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY.replace(n_layers=6, swa_window=(64, 0, 16, 0, 8, 0), n_lanes=lanes, dtp_delay=delay,
                               own_lane_immediate=own)
    blob = synth.make_weights(shape, 60 + lanes + delay, gain_std=0.1)
    prompt = synth.make_tokens(60, 10, shape.vocab)
    with Engine.from_shape(shape) as a, Engine.from_shape(shape) as b:
        a.load_weights(blob)
        b.load_weights(blob)
        a.prefill(prompt[:-1], logits=False)
        b.prefill(prompt[:-1], logits=False)
        gen, last = a.generate(int(prompt[-1]), 40, logits=True)
        ref, ref_last = host_loop(b, prompt[-1], 40)
        assert np.array_equal(gen, ref) and np.array_equal(last, ref_last)
        stamps = a.generate_stamps(40).astype(np.int64)
        assert np.all(np.diff(stamps) > 0)
        # and the next call continues the same sequence
        gen2, _ = a.generate(int(gen[-1]), 5)
        ref2, _ = host_loop(b, gen[-1], 5)
        assert np.array_equal(gen2, ref2)


@pytest.mark.slow
def test_full_generate_in_one_launch_across_the_window():
    # 40 tokens from position 1000: the sliding-window layers cross their
    # 1024-key window inside the launch, and each step's attention reads the
    # keys the launch's earlier steps appended
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL
    blob = synth.make_weights(shape, 1)
    kv = synth.make_kv(shape, 1, 1000)
    first = int(synth.make_tokens(42, 1, shape.vocab)[0])
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.load_kv(kv, 1000)
        gen, last = eng.generate(first, 40, logits=True)
        stamps = eng.generate_stamps(40).astype(np.int64)
        eng.set_position(1000)
        ref, ref_last = host_loop(eng, first, 40)
    assert np.array_equal(gen, ref) and np.array_equal(last, ref_last)
    per_token_ms = np.diff(stamps) / 1e6
    assert 0.2 < np.median(per_token_ms) < 5.0
    orc = oracle.Oracle(shape, blob)
    orc.load_kv(kv, 1000)
    assert oracle_agreement(orc, first, gen) >= 39 / 40
