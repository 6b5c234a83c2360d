"""The argmax rule on the GPU: the lowest index among equal maxima (greedy
decoding, News (asector), "Training and data specialisation"; the tie rule is
this library's reading, stated in include/laneformer.h).

Random weights never produce two equal logits, so the tests plant them.  An
LM-head row with a single non-zero weight c in column j has the logit
c * h_j, with h the normed final hidden state: every product but one is an
exact zero, so the fp32 result is the same whatever the summation order, and
two such rows tie bit for bit on every path (the decode kernel's per-CTA
slices and cross-CTA merge, the batched decode's split GEMV, the batched
prefill's LM head).  With c = 2048 the planted logits dominate the random
ones (standard deviation about 1.3).  h does not depend on the LM head, so
planting rows moves nothing else.

- Tiny model: every row in turn is planted as the lower row of a tie with the
  next row, so each row is found as a maximum and each adjacent pair, the
  pairs that straddle two CTAs' slices included, resolves to the lower index;
  far pairs tie across CTAs; the last row is planted alone.
- Full width with the real 32000-entry vocabulary: ties between the first
  and last rows of CTA slices, three-way ties, on the single-step decode, the
  chained greedy generation, the sampled generation at temperature 0, the
  batched decode and batched generation, and the batched prefill; the
  expected index comes from the oracle (fp64, where the planted logits tie
  exactly and its argmax takes the lowest index).
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

C = 2048.0  # planted weight; exact in FP16


def lm_head(shape, blob):
    return synth.weight_views(shape, blob)["W_lm"]


def plant(w_lm, rows, j, value):
    for r in rows:
        w_lm[r, :] = 0
        w_lm[r, j] = value


def n_ctas(eng) -> int:
    info = (ctypes.c_int64 * 8)()
    assert eng.raw_call("lf_engine_info", info) == 0
    return int(info[0])


def lm_slices(vocab, n):
    """First row of each CTA's LM-head slice: vocab rows split into n near-equal
    contiguous parts, the first vocab % n parts one row longer."""
    base, rem = divmod(vocab, n)
    return [k * base + min(k, rem) for k in range(n)] + [vocab]


def test_tiny_every_row_and_every_adjacent_tie():
    from decode_persistent_sm_gb300 import Engine
    shape = synth.TINY
    blob = synth.make_weights(shape, 41, gain_std=0.1)
    tok = int(synth.make_tokens(41, 1, shape.vocab)[0])
    V, d = shape.vocab, shape.d_model
    # h of the step, read off an oracle whose LM head is the identity on rows 0..d-1
    probe = blob.copy()
    w = lm_head(shape, probe)
    w[:d, :] = np.eye(d, dtype=np.float16)
    h = oracle.Oracle(shape, probe).step(tok)[:d]
    j = int(np.argmax(np.abs(h)))
    val = np.float16(C if h[j] > 0 else -C)
    assert abs(h[j]) * C > 100.0

    w = lm_head(shape, blob)
    keep = w.copy()
    cases = [((r, r + 1), r) for r in range(V - 1)]
    cases += [((r, V - 1 - r), r) for r in range(0, V // 2, 7)]
    cases += [((V - 1,), V - 1), ((3, 500, V - 2), 3)]
    with Engine.from_shape(shape) as eng:
        for rows, want in cases:
            plant(w, rows, j, val)
            eng.load_weights(blob)
            eng.reset()
            z, am = eng.decode_step(tok)
            assert am == want, (rows, am)
            assert len({z[r].tobytes() for r in rows}) == 1, (rows, [z[r] for r in rows])
            w[list(rows), :] = keep[list(rows), :]


def planted_full_width(cases):
    """Full-width two-layer model with the real vocabulary; `cases` maps a
    value sign to the rows planted with it."""
    shape = synth.FULL.replace(n_layers=2, ffn_dim=1024, swa_window=(0, 1024), ctx_cap=512)
    blob = synth.make_weights(shape, 42, gain_std=0.1)
    w = lm_head(shape, blob)
    for sign, rows in cases.items():
        plant(w, rows, 7, np.float16(sign * C))
    return shape, blob


def check_against_oracle(z_gpu, am_gpu, z_ref, planted, what):
    """The GPU's argmax must be the oracle's, and planted rows that tie in
    the oracle must tie bit for bit on the GPU; returns True when a planted
    row held the maximum."""
    top = z_ref.max()
    winners = [r for r in planted if z_ref[r] == top]
    if winners:
        assert am_gpu == min(winners) == oracle.argmax(z_ref), (what, am_gpu, winners)
        if z_gpu is not None:
            assert len({z_gpu[r].tobytes() for r in winners}) == 1, (what, [z_gpu[r] for r in winners])
        return True
    s = np.sort(z_ref)
    if s[-1] - s[-2] > 1e-2:  # planted rows lost (h_j near 0): an ordinary step
        assert am_gpu == oracle.argmax(z_ref), (what, am_gpu)
    return False


@pytest.mark.slow
def test_full_width_ties_on_every_argmax_path():
    from decode_persistent_sm_gb300 import Engine
    probe_shape = synth.FULL.replace(n_layers=2, ffn_dim=1024, swa_window=(0, 1024), ctx_cap=512)
    with Engine.from_shape(probe_shape) as eng:
        first = lm_slices(probe_shape.vocab, n_ctas(eng))
    n = len(first) - 1
    last = [first[k + 1] - 1 for k in range(n)]
    layouts = [
        # first row of the first slice with the last row of the last slice; the
        # last row of one slice with the first row of the next
        {+1: (first[0], last[n - 1]), -1: (last[0], first[1])},
        # three-way ties over three slices; a pair inside one slice
        {+1: (last[n // 2], first[n // 3], last[n - 2]), -1: (first[n // 2] + 1, first[n // 2] + 2)},
    ]
    for layout in layouts:
        shape, blob = planted_full_width(layout)
        planted = sorted(r for rows in layout.values() for r in rows)
        tokens = synth.make_tokens(43, 24, shape.vocab)
        wins = 0
        with Engine.from_shape(shape) as eng:
            eng.load_weights(blob)
            # single steps, teacher forced
            orc = oracle.Oracle(shape, blob)
            for t in tokens[:8]:
                z, am = eng.decode_step(int(t))
                wins += check_against_oracle(z, am, orc.step(int(t)), planted, "decode_step")
            # chained greedy generation, and the sampler at temperature 0
            for greedy in ("generate", "generate_sampled"):
                eng.set_position(8)
                orc.set_pos(8)
                if greedy == "generate":
                    chain, _ = eng.generate(int(tokens[8]), 6)
                else:
                    chain, _ = eng.generate_sampled(int(tokens[8]), 6, 0.0, 1.0, seed=1)
                feed = [int(tokens[8])] + [int(c) for c in chain[:-1]]
                for f, c in zip(feed, chain):
                    wins += check_against_oracle(None, int(c), orc.step(f), planted, greedy)
            # batched prefill: its argmax comes from its own LM head and argmax kernels
            eng.reset()
            z, am = eng.prefill_batched(tokens[:12])
            orc.set_pos(0)
            for t in tokens[:12]:
                ref = orc.step(int(t))
            wins += check_against_oracle(z, am, ref, planted, "prefill_batched")
            # batched decode of two samples from position 12, then batched greedy generation
            eng.batch_begin(2)
            orcs = [oracle.Oracle(shape, blob) for _ in range(2)]
            for o in orcs:
                for t in tokens[:12]:
                    o.step(int(t))
            for i in range(3):
                toks = [int(tokens[12 + i]), int(tokens[20 + i])]
                zb, amb = eng.batch_step(toks)
                for b in range(2):
                    wins += check_against_oracle(zb[b], int(amb[b]), orcs[b].step(toks[b]), planted, "batch_step")
            eng.batch_begin(2)
            for o in orcs:
                o.set_pos(12)
            firsts = [int(tokens[15]), int(tokens[16])]
            chains = eng.batch_generate(firsts, 4, 0.0, 1.0, 0)
            for b in range(2):
                feed = [firsts[b]] + [int(c) for c in chains[b][:-1]]
                for f, c in zip(feed, chains[b]):
                    wins += check_against_oracle(None, int(c), orcs[b].step(f), planted, "batch_generate")
        # 8 + 12 + 1 + 6 + 8 checks per layout; nearly all must be planted wins
        assert wins >= 30, wins
