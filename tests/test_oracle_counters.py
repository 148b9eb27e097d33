"""Pins of oracle.acceptance_counters (per-position acceptance statistics).

The counters follow from the accepted lengths alone: a hand-worked batch,
the chain identity accepted[i] == tested[i + 1] (the rows accepted at
position i are exactly the rows tested at i + 1), the totals sum(accepted) =
sum(n) and tokens = sum(n + 1), and the lesson's expected-acceptance closed
form E[n + 1] = (1 - a^(K+1)) / (1 - a) when every test passes with
probability a.
"""
import numpy as np

import oracle


def test_hand_batch():
    # K = 4, rows with n = 0, 2, 4 and one error row (-1, not counted)
    c = oracle.acceptance_counters([0, 2, 4, -1], 4)
    # tested: i=0 all three rows; i=1 rows n>=1 (2); i=2 (2); i=3 rows n>=3 (1)
    # accepted: i=0 rows n>0 (2); i=1 (2); i=2 rows n>2 (1); i=3 (1)
    assert c.tolist() == [3, 2, 2, 1, 2, 2, 1, 1, 3, 9]


def test_chain_identity_and_totals():
    rng = np.random.default_rng(3)
    for K in (1, 2, 5, 31):
        n = rng.integers(-1, K + 1, size=500)
        c = oracle.acceptance_counters(n, K)
        tested, acc = c[:K], c[K:2 * K]
        assert np.all(acc[:-1] == tested[1:])
        valid = n[n >= 0]
        assert tested[0] == c[2 * K] == valid.size
        assert acc.sum() == valid.sum()
        assert c[2 * K + 1] == valid.sum() + valid.size


def test_mean_acceptance_length_closed_form():
    # iid tests passing with probability a: mean tokens per row -> (1 - a^(K+1)) / (1 - a)
    rng = np.random.default_rng(11)
    a, K, rows = 0.8, 4, 200_000
    passes = rng.random((rows, K)) < a
    n = np.where(passes.all(1), K, np.argmin(passes, axis=1))
    c = oracle.acceptance_counters(n, K)
    mean = c[2 * K + 1] / c[2 * K]
    expect = (1 - a ** (K + 1)) / (1 - a)
    sd = 1.603  # per-row standard deviation of n + 1 at a = 0.8, K = 4
    assert abs(mean - expect) < 4 * sd / np.sqrt(rows)
    # per-position acceptance rate a_i = accepted / tested is a at every position
    rate = c[K:2 * K] / c[:K]
    assert np.all(np.abs(rate - a) < 0.01)
