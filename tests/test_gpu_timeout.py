"""Failure detection on the GPU without a fault: a lane barrier that never
completes (one CTA skips its arrival) must end the step with LF_ERR_TIMEOUT
after the configured limit, poison the engine until lf_reset, and leave the
CUDA context usable (the next steps are checked against the oracle)."""
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import REL_L2, note, rel_l2

pytestmark = pytest.mark.gpu


def test_skipped_arrival_times_out_and_reset_recovers():
    from decode_persistent_sm_gb300 import Engine, LaneformerError
    shape = synth.TINY
    blob = synth.make_weights(shape, 31)
    tokens = synth.make_tokens(31, 6, shape.vocab)
    with Engine.from_shape(shape) as eng:
        eng.load_weights(blob)
        eng.set_timeout_ns(20_000_000)  # 20 ms
        eng.debug_skip_arrival(5)
        t0 = time.time()
        with pytest.raises(LaneformerError, match="TIMEOUT"):
            eng.decode_step(int(tokens[0]))
        assert time.time() - t0 < 10.0
        # poisoned until reset
        with pytest.raises(LaneformerError, match="TIMEOUT"):
            eng.decode_step(int(tokens[0]))
        eng.reset()
        eng.set_timeout_ns(2_000_000_000)
        orc = oracle.Oracle(shape, blob)
        for t in tokens:
            got, am = eng.decode_step(int(t))
            ref = orc.step(int(t))
            assert note(got, ref, am) <= REL_L2
            assert am == oracle.argmax(ref)


def test_timeout_setting_is_validated():
    from decode_persistent_sm_gb300 import Engine, LaneformerError
    with Engine.from_shape(synth.TINY) as eng:
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.set_timeout_ns(0)
        with pytest.raises(LaneformerError, match="INVALID_ARG"):
            eng.debug_skip_arrival(10_000)
