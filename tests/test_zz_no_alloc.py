"""The decode step that allocates nothing (lf_decode_step_static_scratch).

That call serves callers that may not call the CUDA allocator while they
decode (a host that owns a fixed device-memory budget, or a serving loop that
cannot afford cudaMalloc's device-wide synchronisation): its working memory is
a fixed array inside the library.  These tests call it through the C ABI and
check that two calls in a row give the same results as lf_decode_step, within
the tolerance the other parity tests use.  They run alone in a fresh process
as well as after the rest of the suite, so the array may hold anything when
they start.
"""
import ctypes

import numpy as np
import pytest

import synth
from gpu_helpers import REL_L2, rel_l2

pytestmark = pytest.mark.gpu


def static_step(eng, token, logits_dev, argmax_dev) -> int:
    return eng.raw_call("lf_decode_step_static_scratch", ctypes.c_int32(int(token)),
                        ctypes.c_void_p(logits_dev.data_ptr()),
                        ctypes.c_void_p(argmax_dev.data_ptr()))


def compare_two_calls(eng_ref, eng_static, tokens):
    import torch
    refs = [eng_ref.decode_step(int(t)) for t in tokens[:2]]
    logits_dev = torch.full((eng_static.vocab,), float("nan"), dtype=torch.float32, device="cuda")
    argmax_dev = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for (ref_logits, ref_am), t in zip(refs, tokens[:2]):
        assert static_step(eng_static, t, logits_dev, argmax_dev) == 0
        got = logits_dev.cpu().numpy()
        assert rel_l2(got, ref_logits) <= REL_L2
        assert int(argmax_dev.item()) == ref_am


def test_tiny_two_calls_match_decode_step():
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY
    blob = synth.make_weights(shape, 23, gain_std=0.1)
    tokens = synth.make_tokens(23, 12, shape.vocab)
    with Engine.from_shape(shape) as ref, Engine.from_shape(shape) as st:
        ref.load_weights(blob)
        st.load_weights(blob)
        ref.prefill(tokens[:10], logits=False)
        st.prefill(tokens[:10], logits=False)
        compare_two_calls(ref, st, tokens[10:])
        assert st.position == 12


def test_full_model_two_calls_match_decode_step():
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL
    blob = synth.make_weights(shape, 1)
    kv = synth.make_kv(shape, 1, 512)
    tokens = synth.make_tokens(29, 2, shape.vocab)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.load_kv(kv, 512)
        refs = [eng.decode_step(int(t)) for t in tokens]
        eng.set_position(512)  # the same two steps again, through the static array
        import torch
        logits_dev = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        argmax_dev = torch.empty(1, dtype=torch.int32, device="cuda")
        for (ref_logits, ref_am), t in zip(refs, tokens):
            assert static_step(eng, t, logits_dev, argmax_dev) == 0
            assert rel_l2(logits_dev.cpu().numpy(), ref_logits) <= REL_L2
            assert int(argmax_dev.item()) == ref_am


def test_rejects_working_set_beyond_the_array_and_null_outputs():
    import torch
    from decode_persistent_sm_gb300 import Engine
    # 24 layers with delay 10: 24 slots of lane-sum partials (~60 MB) > the array
    big = synth.FULL.replace(n_layers=24, swa_window=synth.FULL.swa_window + (0,) * 9, ctx_cap=64,
                             dtp_delay=10)
    logits_dev = torch.empty(big.vocab, dtype=torch.float32, device="cuda")
    argmax_dev = torch.empty(1, dtype=torch.int32, device="cuda")
    with Engine.from_shape(big) as eng:
        assert static_step(eng, 0, logits_dev, argmax_dev) == 7  # LF_ERR_UNSUPPORTED
        rc = eng.raw_call("lf_decode_step_static_scratch", ctypes.c_int32(0), None,
                          ctypes.c_void_p(argmax_dev.data_ptr()))
        assert rc == 1  # LF_ERR_INVALID_ARG
