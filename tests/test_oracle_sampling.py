"""Pins of the oracle's sampler (stochastic decoding for pass@N) to facts
outside itself: the Philox4x32-10 known-answer vectors published with the
generator (Random123 distribution, kat_vectors, philox4x32 with 10 rounds),
closed-form draws on hand-made distributions, special cases that reduce to
greedy or uniform choice, and the sampling frequencies of a softmax."""
import numpy as np
import pytest

import oracle

KAT = [  # (counter, key, output) of Philox4x32-10
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,out", KAT)
def test_philox_known_answers(ctr, key, out):
    assert oracle.philox(ctr, key) == out


def draws(n, seed=7):
    return np.array([oracle.sample(np.zeros(2), 1.0, 1.0, seed, p, 0)[1] for p in range(n)])


def test_uniform_draws_are_uniform_and_24_bit():
    u = draws(20000)
    assert np.all((u >= 0) & (u < 1))
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))
    hist, _ = np.histogram(u, bins=16, range=(0, 1))
    chi2 = np.sum((hist - 1250.0) ** 2 / 1250.0)
    assert chi2 < 45  # 15 degrees of freedom, far in the tail
    assert abs(u.mean() - 0.5) < 0.01


def test_streams_differ_by_seed_position_and_sample():
    base = oracle.sample(np.zeros(4), 1.0, 1.0, 1, 10, 0)[1]
    assert oracle.sample(np.zeros(4), 1.0, 1.0, 2, 10, 0)[1] != base
    assert oracle.sample(np.zeros(4), 1.0, 1.0, 1, 11, 0)[1] != base
    assert oracle.sample(np.zeros(4), 1.0, 1.0, 1, 10, 1)[1] != base


def test_two_tokens_with_odds_one_to_three():
    # p = (1/4, 3/4): token 1 exactly when u >= 1/4
    for p in range(200):
        tok, u, _ = oracle.sample(np.array([0.0, np.log(3.0)]), 1.0, 1.0, 3, p, 0)
        assert tok == (1 if u >= 0.25 else 0)


def test_equal_logits_give_floor_u_times_vocab():
    for p in range(200):
        tok, u, _ = oracle.sample(np.full(1000, 0.7), 1.0, 1.0, 9, p, 2)
        assert tok == int(np.floor(u * 1000))


def test_nucleus_keeps_the_smallest_top_set():
    logits = np.log(np.array([0.2, 0.5, 0.3]))
    for p in range(200):
        tok, u, tau = oracle.sample(logits, 1.0, 0.8, 4, p, 0)   # kept {1, 2}: mass 0.8
        assert tau == pytest.approx(0.3 / 0.5)
        assert tok == (1 if u * 0.8 < 0.5 else 2)
        tok, u, _ = oracle.sample(logits, 1.0, 0.5, 4, p, 0)     # kept {1}
        assert tok == 1


def test_ties_at_the_threshold_are_all_kept():
    logits = np.array([1.0, 1.0, 0.0, 1.0])
    seen = {oracle.sample(logits, 1.0, 0.1, 5, p, 0)[0] for p in range(300)}
    assert seen == {0, 1, 3}


def test_zero_temperature_and_tiny_top_p_are_greedy():
    g = np.random.default_rng(1)
    for p in range(50):
        z = g.standard_normal(500)
        assert oracle.sample(z, 0.0, 0.9, 1, p, 0)[0] == oracle.argmax(z)
        assert oracle.sample(z, 1.0, 1e-12, 1, p, 0)[0] == oracle.argmax(z)


def test_temperature_divides_the_logits():
    g = np.random.default_rng(2)
    z = g.standard_normal(300)
    for p in range(100):
        assert oracle.sample(z, 2.0, 0.9, 8, p, 1)[0] == oracle.sample(z / 2.0, 1.0, 0.9, 8, p, 1)[0]


def test_frequencies_follow_the_softmax():
    z = np.array([0.0, 1.0, 2.0, -1.0])
    pr = np.exp(z) / np.exp(z).sum()
    n = 20000
    counts = np.bincount([oracle.sample(z, 1.0, 1.0, 11, p, 0)[0] for p in range(n)], minlength=4)
    sigma = np.sqrt(n * pr * (1 - pr))
    assert np.all(np.abs(counts - n * pr) < 4.5 * sigma)
