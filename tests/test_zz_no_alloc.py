"""The decode step that allocates nothing (lf_decode_step_static_scratch).

That call serves callers that may not call the CUDA allocator while they
decode (a host that owns a fixed device-memory budget, or a serving loop that
cannot afford cudaMalloc's device-wide synchronisation): its working memory is
a fixed array inside the library.  These tests call it through the C ABI,
two calls in a row, and check that

- it gives bit for bit the results of lf_decode_step (the same kernel with the
  same fixed summation order, only the working memory moved);
- it matches the oracle at the gates of the other parity tests;
- neither the engine's device-memory count nor the device's free memory moves
  across a call;
- it refuses output pointers the GPU cannot write (host memory, misaligned).

They run alone in a fresh process as well as after the rest of the suite, so
the array may hold anything when they start.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import REL_L2, note, rel_l2

pytestmark = pytest.mark.gpu

LF_ERR_INVALID_ARG = 1
LF_ERR_UNSUPPORTED = 7


def static_step(eng, token, logits_ptr, argmax_ptr) -> int:
    return eng.raw_call("lf_decode_step_static_scratch", ctypes.c_int32(int(token)),
                        ctypes.c_void_p(logits_ptr), ctypes.c_void_p(argmax_ptr))


def device_bytes(eng) -> int:
    info = (ctypes.c_int64 * 8)()
    assert eng.raw_call("lf_engine_info", info) == 0
    return int(info[2])


def test_tiny_two_calls_bitwise_equal_to_decode_step_and_match_the_oracle():
    import torch
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY
    blob = synth.make_weights(shape, 23, gain_std=0.1)
    tokens = synth.make_tokens(23, 12, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    for t in tokens[:10]:
        orc.step(int(t))
    with Engine.from_shape(shape) as ref, Engine.from_shape(shape) as st:
        ref.load_weights(blob)
        st.load_weights(blob)
        ref.prefill(tokens[:10], logits=False)
        st.prefill(tokens[:10], logits=False)
        logits_dev = torch.full((shape.vocab,), float("nan"), dtype=torch.float32, device="cuda")
        argmax_dev = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        for t in tokens[10:12]:
            want, want_am = ref.decode_step(int(t))
            assert static_step(st, t, logits_dev.data_ptr(), argmax_dev.data_ptr()) == 0
            got, got_am = logits_dev.cpu().numpy(), int(argmax_dev.item())
            assert np.array_equal(got, want), "static-scratch step differs from lf_decode_step"
            assert got_am == want_am
            z = orc.step(int(t))
            assert note(got, z, got_am) <= REL_L2 and got_am == oracle.argmax(z)
        assert st.position == 12


def test_full_model_two_calls_bitwise_and_nothing_allocated():
    import torch
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
        logits_dev = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        argmax_dev = torch.empty(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        owned = device_bytes(eng)
        for i, ((ref_logits, ref_am), t) in enumerate(zip(refs, tokens)):
            # the first call in a process may load the library's array onto the
            # device; from then on a call must leave the free memory as it was
            free_before = torch.cuda.mem_get_info()[0]
            assert static_step(eng, t, logits_dev.data_ptr(), argmax_dev.data_ptr()) == 0
            torch.cuda.synchronize()
            free_after = torch.cuda.mem_get_info()[0]
            if i > 0:
                assert free_after == free_before, f"device free memory moved by {free_before - free_after} B"
            assert device_bytes(eng) == owned
            assert np.array_equal(logits_dev.cpu().numpy(), ref_logits)
            assert int(argmax_dev.item()) == ref_am
        assert eng.position == 514


def test_rejects_bad_outputs_and_a_working_set_beyond_the_array():
    import torch
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY
    logits_dev = torch.empty(shape.vocab + 4, dtype=torch.float32, device="cuda")
    argmax_dev = torch.empty(4, dtype=torch.int32, device="cuda")
    host_logits = np.empty(shape.vocab, dtype=np.float32)
    host_argmax = np.empty(1, dtype=np.int32)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(synth.make_weights(shape, 3))
        bad = [(0, argmax_dev.data_ptr()),
               (logits_dev.data_ptr(), 0),
               (host_logits.ctypes.data, argmax_dev.data_ptr()),
               (logits_dev.data_ptr(), host_argmax.ctypes.data),
               (logits_dev.data_ptr() + 2, argmax_dev.data_ptr()),
               (logits_dev.data_ptr(), argmax_dev.data_ptr() + 1)]
        for lp, ap in bad:
            assert static_step(eng, 0, lp, ap) == LF_ERR_INVALID_ARG
        assert eng.position == 0  # nothing ran
        assert static_step(eng, 0, logits_dev.data_ptr(), argmax_dev.data_ptr()) == 0
        assert eng.position == 1
    # 24 layers with delay 10: 24 slots of lane-sum partials (~60 MB) > the array
    big = synth.FULL.replace(n_layers=24, swa_window=synth.FULL.swa_window + (0,) * 9, ctx_cap=64,
                             dtp_delay=10)
    logits_big = torch.empty(big.vocab, dtype=torch.float32, device="cuda")
    with Engine.from_shape(big) as eng:
        assert static_step(eng, 0, logits_big.data_ptr(), argmax_dev.data_ptr()) == LF_ERR_UNSUPPORTED
