"""The debug build (liblaneformer_debug.so, compiled with LF_DEBUG): the
decode kernel checks every weight-tile, KV, q/k/v, partial, lane-sum,
attention-partial and logit index before it uses it, and every engine buffer
sits between canary regions that the host checks after each step.

A clean run on the tiny model and on one full-shape step must match the
oracle at the usual gates with every check silent; a canary that the host
overwrites itself must make the next check report LF_ERR_BOUNDS and poison
the engine.  (A device-side bounds check is never provoked on purpose: a
check missed by mistake would let the access through and fault a shared
GPU.)"""
import ctypes

import pytest

import oracle
import synth
from gpu_helpers import assert_gates, note, teacher_forced

pytestmark = pytest.mark.gpu

LF_OK, LF_ERR_BOUNDS, LF_ERR_UNSUPPORTED = 0, 8, 7


def canaries(eng):
    n = ctypes.c_int(-1)
    rc = eng.raw_call("lf_debug_canaries", ctypes.byref(n))
    return rc, n.value


def test_tiny_clean_run_with_every_check_on():
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY.replace(n_layers=6, swa_window=(64, 0, 16, 0, 8, 0))
    blob = synth.make_weights(shape, 51, gain_std=0.1)
    tokens = synth.make_tokens(51, 90, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    with Engine.from_shape(shape, debug=True) as eng:
        eng.load_weights(blob)
        rels, agree, _, _ = teacher_forced(eng, orc, tokens)
        assert_gates(rels, agree, "debug build, 6 layers, windows crossed")
        rc, n = canaries(eng)
        assert rc == LF_OK and n >= 20


def test_canary_written_by_the_host_is_caught():
    from decode_persistent_sm_gb300 import Engine, LaneformerError
    shape = synth.TINY
    blob = synth.make_weights(shape, 52)
    for which, back in ((0, 0), (5, 1), (-1, 1)):
        with Engine.from_shape(shape, debug=True) as eng:
            eng.load_weights(blob)
            eng.decode_step(3)
            rc, n = canaries(eng)
            assert rc == LF_OK
            i = which % n
            assert eng.raw_call("lf_debug_corrupt_canary", ctypes.c_int(i), ctypes.c_int(back)) == LF_OK
            assert canaries(eng)[0] == LF_ERR_BOUNDS
            with pytest.raises(LaneformerError, match="BOUNDS"):
                eng.decode_step(4)  # poisoned until lf_reset
        with Engine.from_shape(shape, debug=True) as eng:  # a fresh engine is clean again
            eng.load_weights(blob)
            eng.decode_step(3)
            assert canaries(eng)[0] == LF_OK


def test_release_library_refuses_the_debug_calls():
    from decode_persistent_sm_gb300 import Engine
    with Engine.from_shape(synth.TINY) as eng:
        assert canaries(eng)[0] == LF_ERR_UNSUPPORTED
        assert eng.raw_call("lf_debug_corrupt_canary", ctypes.c_int(0), ctypes.c_int(0)) == LF_ERR_UNSUPPORTED


@pytest.mark.slow
@pytest.mark.parametrize("fill", [1030, 4000])
def test_full_shape_step_with_every_check_on(fill):
    # past the 1024-key window, every lane and op of the real plan; at 4000
    # a CTA's share of a full-attention layer spans seven 32-key tiles
    from decode_persistent_sm_gb300 import Engine
    shape = synth.FULL
    blob = synth.make_weights(shape, 1)
    kv = synth.make_kv(shape, 1, fill)
    toks = synth.make_tokens(53, 2, shape.vocab)
    orc = oracle.Oracle(shape, blob)
    orc.load_kv(kv, fill)
    with Engine.from_shape(shape, debug=True) as eng:
        eng.load_weights(blob)
        eng.load_kv(kv, fill)
        for t in toks:
            got, am = eng.decode_step(int(t))
            ref = orc.step(int(t))
            assert note(got, ref, am) <= 1e-2 and am == oracle.argmax(ref)
        assert canaries(eng)[0] == LF_OK
