"""GPU checks of the per-op trace (lf_debug_trace / lf_debug_read_trace): a
single step fills every streaming op's slot in op-list order on every CTA,
and a launch of several steps (lf_generate) leaves its last step's record,
checked against the steps' completion stamps (the same global timer)."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

# ops whose slot the streaming warps write on every CTA (the attention warps
# write ATTN, the lane-sum warps REDUCE / LREDUCE on the CTAs that sum)
STREAM_OPS = {0, 1, 2, 3, 4, 5, 7, 9, 11}
ATTN, EMBED, LMHEAD = 6, 0, 9
SLACK_NS = 2000


def check_record(tr, ops):
    tr = tr.astype(np.int64)
    kinds = [int(o) & 0xFF for o in ops]
    idx = [j for j, k in enumerate(kinds) if k in STREAM_OPS]
    assert idx and kinds[0] == EMBED and kinds[-1] == LMHEAD
    st, en = tr[:, idx, 0], tr[:, idx, 1]
    assert (st > 0).all() and (en >= st).all()
    assert (st[:, 1:] >= en[:, :-1]).all(), "a CTA's streaming ops out of list order"
    a = [j for j, k in enumerate(kinds) if k == ATTN]
    assert (tr[:, a, 0] > 0).all() and (tr[:, a, 1] >= tr[:, a, 0]).all()
    # blocked times fit inside their op
    assert (tr[:, idx, 2] <= en - st + SLACK_NS).all() and (tr[:, idx, 3] <= en - st + SLACK_NS).all()
    return tr, kinds


def make_engine(shape, blob):
    from decode_persistent_sm_gb300 import Engine
    eng = Engine.from_shape(shape)
    eng.load_weights(blob)
    return eng


def test_single_step_record():
    shape = synth.TINY
    blob = synth.make_weights(shape, 41)
    tokens = synth.make_tokens(41, 8, shape.vocab)
    with make_engine(shape, blob) as eng:
        for t in tokens[:4]:
            eng.decode_step(int(t))
        eng.trace(True)
        eng.decode_step(int(tokens[4]))
        tr, ops = eng.read_trace()
        eng.trace(False)
        assert tr.shape == (eng.info()["n_sm"], eng.info()["n_ops"], 6)
        check_record(tr, ops)


def test_generate_leaves_the_last_steps_record():
    shape = synth.TINY
    blob = synth.make_weights(shape, 43)
    n = 6
    with make_engine(shape, blob) as eng:
        eng.generate(5, 4)  # warm
        eng.reset()
        eng.trace(True)
        eng.generate(7, n)
        tr, ops = eng.read_trace()
        eng.trace(False)
        stamps = eng.generate_stamps(n).astype(np.int64)
    tr, kinds = check_record(tr, ops)
    assert (np.diff(stamps) > 0).all()
    emb, lm = kinds.index(EMBED), len(kinds) - 1
    # the last step embeds the previous step's argmax: no CTA can finish its
    # embedding before that step is complete; its LM head ends by its own stamp
    assert tr[:, emb, 1].min() >= stamps[n - 2] - SLACK_NS
    assert tr[:, lm, 1].max() <= stamps[n - 1] + SLACK_NS
