"""Pins of the oracle's sampled choice (oracle/sampling.py) on the CPU.

Philox4x32-10 against the published known-answer vectors; the choice against
closed forms (greedy limits, equal logits, a two-token nucleus) and, over many
draws, against the exact probabilities of a small vocabulary.
"""
import math
import os

import numpy as np
import pytest

from oracle import sampling as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_philox_known_answers():
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        assert S.philox4x32_10(v[:4], v[4:6]) == tuple(v[6:])


def test_uniform_range_and_layout():
    us = [S.uniform(42, s, p) for s in range(3) for p in range(200)]
    assert all(0.0 <= u < 1.0 for u in us)
    assert len(set(us)) == len(us)  # distinct counters, distinct draws
    x0 = S.philox4x32_10((7, 1, 0, 0), (42, 0))[0]
    assert S.uniform(42, 1, 7) == (x0 >> 8) / 2.0 ** 24
    assert S.uniform(42 + (5 << 32), 1, 7) != S.uniform(42, 1, 7)  # the seed's high word is the second key word


def test_greedy_limits():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal(500).astype(np.float32)
    lg[17] = lg[123] = lg.max() + 1.0  # a tie for the maximum: top-k 1 and a nucleus of one take the lower id
    for u in (0.0, 0.37, 0.999):
        assert S.sample(lg, 1.0, 1, 1.0, u)[0] == 17
        assert S.sample(lg, 1.0, 40, 1e-9, u)[0] == 17
    lg[123] -= 0.5  # a unique maximum: temperature -> 0 is greedy
    for u in (0.0, 0.37, 0.999):
        assert S.sample(lg, 1e-4, 40, 0.95, u)[0] == 17
    lg[123] += 0.5  # an exact tie at temperature -> 0: each of the two with probability 1/2
    assert S.sample(lg, 1e-4, 40, 1.0, 0.49)[0] == 17 and S.sample(lg, 1e-4, 40, 1.0, 0.51)[0] == 123


@pytest.mark.parametrize("k", [1, 5, 40, 64])
def test_equal_logits_pick_by_u(k):
    lg = np.zeros(100, np.float32)
    for u in np.linspace(0.0, 0.999, 37):
        tok, info = S.sample(lg, 0.7, k, 1.0, float(u))
        assert info["ids"] == list(range(k))  # ties: lower ids first
        assert tok == min(int(math.floor(u * k + 1e-12)), k - 1)


def test_two_token_nucleus():
    lg = np.log(np.array([0.7, 0.3, 1e-30], np.float64)).astype(np.float32)
    assert all(S.sample(lg, 1.0, 2, 0.6, u)[0] == 0 for u in (0.0, 0.5, 0.99))
    assert S.sample(lg, 1.0, 2, 0.8, 0.69)[0] == 0
    assert S.sample(lg, 1.0, 2, 0.8, 0.71)[0] == 1
    # temperature 2 flattens: p = softmax(log p / 2) = (0.6046, 0.3954)
    assert S.sample(lg, 2.0, 2, 1.0, 0.60)[0] == 0 and S.sample(lg, 2.0, 2, 1.0, 0.61)[0] == 1


def test_draws_follow_the_truncated_distribution():
    rng = np.random.default_rng(5)
    lg = (rng.standard_normal(12) * 1.5).astype(np.float32)
    T, k, p = 0.8, 6, 0.9
    # exact truncated distribution, brute force
    ids = sorted(range(12), key=lambda i: (-lg[i], i))[:k]
    e = np.exp((lg[ids].astype(np.float64) - lg[ids[0]]) / T)
    q = e / e.sum()
    n = int(np.argmax(np.cumsum(q) >= p)) + 1
    q = q[:n] / q[:n].sum()
    N = 20000
    counts = np.zeros(12)
    for pos in range(N):
        counts[S.sample(lg, T, k, p, S.uniform(1234, 0, pos))[0]] += 1
    for j, tok in enumerate(ids[:n]):
        sd = math.sqrt(N * q[j] * (1 - q[j]))
        assert abs(counts[tok] - N * q[j]) <= 5 * sd + 1
    assert counts.sum() == counts[ids[:n]].sum()  # nothing outside the nucleus
