"""The batched prefill (lf_prefill_batched: tensor-core GEMMs, one pass per
sub-block over all prompt positions) against the oracle, which computes the
prompt one position at a time.

Checked: the last position's logits and argmax, the KV cache the pass leaves
behind (through the decode steps that follow it, teacher forced, and read
back directly), prompts spanning several 64-position blocks and crossing the
sliding window, every delay / lane variant of the tiny model, a prefill that
starts after earlier decode steps, and the full 2.3B shape."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import REL_L2, assert_gates, note, rel_l2, teacher_forced

pytestmark = pytest.mark.gpu


def prefill_then_steps(shape, seed, n_prompt, n_steps, gain_std=0.1, lead=0):
    """Optional `lead` decode steps, a batched prefill of n_prompt tokens, then
    n_steps teacher-forced steps; every result against the oracle."""
    from decode_persistent_sm_gb300 import Engine
    blob = synth.make_weights(shape, seed, gain_std=gain_std)
    tokens = synth.make_tokens(seed, lead + n_prompt + n_steps, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        for t in tokens[:lead]:
            got, am = eng.decode_step(int(t))
            ref = orc.step(int(t))
            assert note(got, ref, am) <= REL_L2
        prompt = tokens[lead:lead + n_prompt]
        got, am = eng.prefill_batched(prompt)
        for t in prompt:
            ref = orc.step(int(t))
        assert eng.position == lead + n_prompt
        pre_rel, pre_agree = note(got, ref, am), am == oracle.argmax(ref)
        rels, agree, _, _ = teacher_forced(eng, orc, tokens[lead + n_prompt:])
        return eng, orc, pre_rel, pre_agree, rels, agree


def test_tiny_prompt_spanning_blocks_and_window():
    # 100 positions: two 64-query blocks; layer 0's 64-key window is crossed
    shape = synth.TINY
    _, _, pre_rel, pre_agree, rels, agree = prefill_then_steps(shape, 2, 100, 12)
    assert pre_rel <= REL_L2 and pre_agree
    assert_gates(rels, agree, "tiny after a 100-token batched prefill")


@pytest.mark.parametrize("lanes,delay", [(8, 0), (8, 1), (8, 2), (1, 0), (1, 2), (4, 3)])
def test_tiny_lanes_and_delays(lanes, delay):
    shape = synth.TINY.replace(n_lanes=lanes, dtp_delay=delay)
    _, _, pre_rel, pre_agree, rels, agree = prefill_then_steps(shape, 5, 70, 6)
    assert pre_rel <= REL_L2 and pre_agree
    assert_gates(rels, agree, f"lanes={lanes} delay={delay}")


def test_six_layers_and_single_token_prompt():
    shape = synth.TINY.replace(n_layers=6, swa_window=(64, 0, 16, 0, 8, 0))
    _, _, pre_rel, pre_agree, rels, agree = prefill_then_steps(shape, 7, 1, 4)
    assert pre_rel <= REL_L2 and pre_agree
    _, _, pre_rel, pre_agree, rels, agree = prefill_then_steps(shape, 8, 90, 4)
    assert pre_rel <= REL_L2 and pre_agree
    assert_gates(rels, agree, "6 layers")


def test_ffn_width_not_a_multiple_of_128():
    # the gate/up GEMM fuses SwiGLU into its epilogue only when F is a
    # multiple of 128; F = 320 takes the separate SwiGLU pass
    shape = synth.TINY.replace(ffn_dim=320)
    _, _, pre_rel, pre_agree, rels, agree = prefill_then_steps(shape, 6, 75, 4)
    assert pre_rel <= REL_L2 and pre_agree
    assert_gates(rels, agree, "F = 320")


def test_prefill_after_decode_steps_and_kv_contents():
    shape = synth.TINY
    eng, orc, pre_rel, pre_agree, rels, agree = prefill_then_steps(shape, 9, 40, 3, lead=21)
    assert pre_rel <= REL_L2 and pre_agree
    assert_gates(rels, agree, "prefill from position 21")


def test_kv_written_by_the_batched_prefill():
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY
    blob = synth.make_weights(shape, 11, gain_std=0.1)
    tokens = synth.make_tokens(11, 70, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    orc.run(tokens)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.prefill_batched(tokens, logits=False)
        for layer in range(shape.n_layers):
            for kvh in range(shape.n_kv_heads):
                lane = kvh * (shape.n_q_heads // shape.n_kv_heads) // (shape.n_q_heads // shape.n_lanes)
                for pos in (0, 33, 64, 69):
                    k, v = eng.read_kv(layer, kvh, pos)
                    rk, rv = orc.kv(lane, layer, 0, pos)
                    assert np.allclose(k, rk, rtol=4e-3, atol=2e-4)
                    assert np.allclose(v, rv, rtol=4e-3, atol=2e-4)


def test_rejections():
    from decode_persistent_sm_gb300 import Engine, LaneformerError
    shape = synth.TINY
    with Engine.from_shape(shape) as eng:
        with pytest.raises(LaneformerError, match="NOT_LOADED"):
            eng.prefill_batched([1, 2])
        eng.load_weights(synth.make_weights(shape, 1))
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.prefill_batched([1, shape.vocab])
        with pytest.raises(LaneformerError, match="CTX_OVERFLOW"):
            eng.prefill_batched([1] * (shape.ctx_cap + 1))
        assert eng.position == 0


@pytest.mark.slow
def test_full_shape_prompt_128():
    shape = synth.FULL
    _, _, pre_rel, pre_agree, rels, agree = prefill_then_steps(shape, 1, 128, 2, gain_std=0.0)
    assert pre_rel <= REL_L2 and pre_agree
    assert_gates(rels, agree, "full shape after a 128-token batched prefill")


@pytest.mark.slow
def test_full_shape_prompt_260_tensor_core_attention():
    # three 128-query tiles and three 128-key tiles on the tensor-core path
    shape = synth.FULL
    _, _, pre_rel, pre_agree, rels, agree = prefill_then_steps(shape, 3, 260, 2, gain_std=0.0)
    assert pre_rel <= REL_L2 and pre_agree
    assert_gates(rels, agree, "full shape after a 260-token batched prefill")


@pytest.mark.slow
def test_tensor_core_and_cuda_core_attention_agree_past_the_window():
    # 1500 positions: the sliding-window layers' 1024-key window is crossed;
    # both prefill attentions must give the same function (the oracle checks
    # each of them on shorter prompts)
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL
    blob = synth.make_weights(shape, 4)
    tokens = synth.make_tokens(4, 1503, shape.vocab)
    out = {}
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        for tc in (True, False):
            eng.reset()
            eng.set_prefill_attention(tc)
            got, am = eng.prefill_batched(tokens[:1500])
            steps = [eng.decode_step(int(t)) for t in tokens[1500:]]
            out[tc] = (got, am, steps)
    (g1, a1, s1), (g0, a0, s0) = out[True], out[False]
    assert rel_l2(g1, g0) <= REL_L2 and a1 == a0
    for (l1, m1), (l0, m0) in zip(s1, s0):
        assert rel_l2(l1, l0) <= REL_L2 and m1 == m0


@pytest.mark.slow
def test_tensor_core_attention_after_decode_steps():
    # a prefill that starts at position 37, after decode steps: the tensor-core
    # attention reads the earlier positions' V through the transposed copy, the
    # CUDA-core attention from the cache itself; both must give the same function
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL
    blob = synth.make_weights(shape, 6)
    tokens = synth.make_tokens(6, 37 + 150 + 3, shape.vocab)
    out = {}
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        for tc in (True, False):
            eng.reset()
            eng.set_prefill_attention(tc)
            for t in tokens[:37]:
                eng.decode_step(int(t))
            got, am = eng.prefill_batched(tokens[37:187])
            steps = [eng.decode_step(int(t)) for t in tokens[187:]]
            out[tc] = (got, am, steps)
    (g1, a1, s1), (g0, a0, s0) = out[True], out[False]
    assert rel_l2(g1, g0) <= REL_L2 and a1 == a0
    for (l1, m1), (l0, m0) in zip(s1, s0):
        assert rel_l2(l1, l0) <= REL_L2 and m1 == m0


def _small_hd128(delay):
    # full width and head size (the tensor-core attention), 3 layers, small FFN and vocabulary
    return synth.FULL.replace(n_layers=3, ffn_dim=1024, vocab=2048, dtp_delay=delay, swa_window=(0, 100, 40),
                              ctx_cap=512)


@pytest.mark.parametrize("shape_name,delay", [("tiny", 0), ("tiny", 2), ("hd128", 2)])
def test_prefill_on_a_callers_stream_is_bitwise_the_default_streams(shape_name, delay):
    # the pass runs its odd sub-blocks on a second stream that the engine's
    # stream waits for: on a caller's stream it must give bit for bit what it
    # gives on the default stream (same kernels, same fp32 summation order),
    # the KV cache it leaves and the steps after it included
    import torch
    from decode_persistent_sm_gb300 import Engine
    if shape_name == "tiny":
        shape = synth.TINY.replace(dtp_delay=delay, n_layers=4, swa_window=(64, 0, 16, 0), ctx_cap=256)
    else:
        shape = _small_hd128(delay)
    seed = 71 + delay
    blob = synth.make_weights(shape, seed, gain_std=0.1)
    tokens = synth.make_tokens(seed, 203, shape.vocab)
    side = torch.cuda.Stream()
    out = []
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        for stream in (None, side.cuda_stream):
            eng.reset()
            eng.set_stream(stream)
            got, am = eng.prefill_batched(tokens[:200])
            kv = [eng.read_kv(l, h, p) for l in range(shape.n_layers) for h in range(shape.n_kv_heads)
                  for p in (0, 99, 199)]
            steps = [eng.decode_step(int(t)) for t in tokens[200:]]
            out.append((got, am, kv, steps))
        eng.set_stream(None)
    (g0, a0, kv0, s0), (g1, a1, kv1, s1) = out
    assert np.array_equal(g0, g1) and a0 == a1
    for (k0, v0), (k1, v1) in zip(kv0, kv1):
        assert np.array_equal(k0, k1) and np.array_equal(v0, v1)
    for (l0, m0), (l1, m1) in zip(s0, s1):
        assert np.array_equal(l0, l1) and m0 == m1
