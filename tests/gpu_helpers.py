"""Shared pieces of the GPU parity tests: tolerances and teacher forcing."""
import numpy as np

import oracle

# Gates: per-step logits rel-L2 <= 1e-2 and argmax agreement >= 99% under
# teacher forcing (the GPU is fed the same tokens as the oracle).
REL_L2 = 1e-2
ARGMAX_MIN = 0.99


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def top2_margin(ref) -> float:
    s = np.sort(np.asarray(ref))
    return float(s[-1] - s[-2])


def teacher_forced(engine, orc, tokens):
    """Feeds `tokens` to both; returns (rel errors, argmax agree flags, margins, max abs err)."""
    rels, agree, margins, abserr = [], [], [], []
    for t in tokens:
        ref = orc.step(int(t))
        got, am = engine.decode_step(int(t))
        rels.append(rel_l2(got, ref))
        agree.append(am == oracle.argmax(ref))
        margins.append(top2_margin(ref))
        abserr.append(float(np.max(np.abs(got - ref))))
    return np.array(rels), np.array(agree), np.array(margins), np.array(abserr)


def assert_gates(rels, agree, what=""):
    assert rels.max() <= REL_L2, f"{what}: worst logits rel-L2 {rels.max():.3e}"
    assert agree.mean() >= ARGMAX_MIN, f"{what}: argmax agreement {agree.mean():.3f}"
