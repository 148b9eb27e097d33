"""Pins for the fp64 oracle of the accept/reject step (CPU only).

Each test ties the oracle to something other than itself: hand-worked examples
(tests/golden/hand_examples.json), closed forms from the pages (expected
accepted tokens per verifier call), the losslessness theorem checked by brute
force, and special cases that reduce to library routines (argmax, softmax of
log-probabilities). `test_oracle_mutations.py` plants plausible mistakes in
the oracle and checks that these pins catch them.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def _logits_from_probs(probs, T):
    with np.errstate(divide="ignore"):
        return T * np.log(np.asarray(probs, np.float64))


# ---------------------------------------------------------------- hand examples
@pytest.mark.parametrize("T", [1.0, 0.5, 2.0])
def test_hand_sample_cases(golden, T):
    for case in golden["sample_cases"]:
        q = np.asarray(case["q"])
        p = np.asarray(case["p"])
        zt = _logits_from_probs(q, T)[None]
        zd = _logits_from_probs(p, T)[None]
        tok = np.asarray(case["draft_tokens"])[None]
        u = np.asarray(case["uniforms"], np.float64)[None]
        r = oracle.verify_sample(zt, zd, tok, u, T)
        assert r["out_tokens"][0].tolist() == case["out_tokens"], case["name"]
        assert int(r["num_accepted"][0]) == case["num_accepted"], case["name"]
        # probabilities of the draft tokens come back as given
        K = tok.shape[1]
        np.testing.assert_allclose(r["q_at_d"][0], q[np.arange(K), tok[0]], rtol=1e-12)
        np.testing.assert_allclose(r["p_at_d"][0], p[np.arange(K), tok[0]], rtol=1e-12)


def test_hand_probability_cases(golden):
    for case in golden["probability_cases"]:
        w = oracle.residual(case["q"], case["p"])
        for u, want in case["draws"]:
            idx, _ = oracle.inverse_cdf(w[None], np.array([u]))
            assert int(idx[0]) == want, (case["name"], u)


def test_hand_greedy_cases(golden):
    for case in golden["greedy_cases"]:
        zt = np.asarray(case["target_logits"], np.float64)[None]
        tok = np.asarray(case["draft_tokens"])[None]
        r = oracle.verify_greedy(zt, tok)
        assert r["out_tokens"][0].tolist() == case["out_tokens"], case["name"]
        assert int(r["num_accepted"][0]) == case["num_accepted"], case["name"]
        # T == 0 routes the sampling entry to greedy
        r0 = oracle.verify_step(zt, None, tok, np.zeros((1, tok.shape[1] + 1)), 0.0)
        assert r0["out_tokens"][0].tolist() == case["out_tokens"]


# ---------------------------------------------------------------- accept rule edge cases
def test_accept_rule_edges():
    # p(d) <= 0 accepts whatever q and u are
    assert oracle.accept_test(-np.inf, -np.inf, 0.999)
    assert oracle.accept_test(np.log(0.1), -np.inf, 0.999)
    # q(d) = 0 with p(d) > 0 always rejects, even at u = 0 (strict <)
    assert not oracle.accept_test(-np.inf, np.log(0.3), 0.0)
    # u = 0 accepts when q(d) > 0
    assert oracle.accept_test(np.log(1e-30), np.log(0.9), 0.0)
    # strict comparison at the ratio itself (dyadic: ratio exactly 0.5)
    assert not oracle.accept_test(np.log(0.25), np.log(0.5), 0.5)
    assert oracle.accept_test(np.log(0.25), np.log(0.5), np.nextafter(0.5, 0))
    # ratio above 1 clips to 1: any u in [0, 1) accepts
    assert oracle.accept_test(np.log(0.9), np.log(0.1), np.nextafter(1.0, 0))


def test_inverse_cdf_skips_zero_weights_and_reports_margin():
    w = np.array([[0.0, 0.5, 0.0, 0.5]])
    idx, dist = oracle.inverse_cdf(w, np.array([0.0]))
    assert idx[0] == 1 and dist[0] == 0.0
    idx, dist = oracle.inverse_cdf(w, np.array([0.75]))
    assert idx[0] == 3 and abs(dist[0] - 0.25) < 1e-15


# ---------------------------------------------------------------- softmax closed form
@pytest.mark.parametrize("T", [1.0, 0.6, 1.7])
def test_softmax_of_scaled_log_probs(T):
    rng = np.random.default_rng(3)
    p = rng.dirichlet(np.ones(50), size=4)
    T64 = oracle.temperature64(T)
    z = T64 * np.log(p) + rng.normal(0, 5, size=(4, 1))   # shift invariance
    np.testing.assert_allclose(oracle.softmax(z, T64), p, rtol=1e-12)
    np.testing.assert_allclose(oracle.log_softmax(z, T64), np.log(p), atol=1e-12)
    assert oracle.temperature64(0.6) == float(np.float32(0.6)) != 0.6


def test_masked_logits_have_zero_probability():
    z = np.array([[0.0, -np.inf, 1.0]])
    q = oracle.softmax(z, 1.0)
    assert q[0, 1] == 0.0
    np.testing.assert_allclose(q[0, [0, 2]], np.array([1, math.e]) / (1 + math.e), rtol=1e-15)


# ---------------------------------------------------------------- losslessness (theorem)
# q0 puts its excess on two tokens and p0 puts most mass on a third, so every
# rejection draws from a residual split evenly over two tokens
SKEWED_Q = np.array([[0.4, 0.4, 0.2], [0.2, 0.3, 0.5]])
SKEWED_P = np.array([[0.1, 0.1, 0.8]])


def _lossless_run(V, K, N, seed, q=None, p=None):
    """N independent steps with fixed q_0..q_K, p_0..p_{K-1}; d_i ~ p_i drawn by
    the library sampler; returns the oracle outputs and the distributions."""
    rng = np.random.default_rng(seed)
    if q is None:
        q = rng.dirichlet(np.full(V, 0.8), size=K + 1)
        p = rng.dirichlet(np.full(V, 0.8), size=K)
    tok = np.stack([rng.choice(V, size=N, p=p[i]) for i in range(K)], axis=1)
    u = rng.random((N, K + 1))
    zt = np.broadcast_to(np.log(q), (N, K + 1, V))
    zd = np.broadcast_to(np.log(p), (N, K, V))
    r = oracle.verify_sample(zt, zd, tok, u, 1.0, row_chunk=N)
    return r, q, p


@pytest.mark.slow
@pytest.mark.parametrize("V,K,skewed", [(3, 1, True), (3, 1, False), (5, 2, False),
                                        (16, 2, False)])
def test_losslessness_brute_force(V, K, skewed):
    """The emitted token at index i, over the steps that reach index i, is
    distributed as q_i (total variation < 0.005 over 10^6 steps). The
    acceptance rate at position 0 is sum_v min(p_0(v), q_0(v))."""
    N = 1_000_000
    if skewed:
        r, q, p = _lossless_run(V, K, N, seed=7, q=SKEWED_Q, p=SKEWED_P)
    else:
        r, q, p = _lossless_run(V, K, N, seed=11 + V)
    out, n = r["out_tokens"], r["num_accepted"]
    for i in range(K + 1):
        reached = n >= i
        emp = np.bincount(out[reached, i], minlength=V) / reached.sum()
        tv = 0.5 * np.abs(emp - q[i]).sum()
        assert tv < 0.005, (i, tv)
    alpha0 = np.minimum(p[0], q[0]).sum()
    acc0 = (n >= 1).mean()
    assert abs(acc0 - alpha0) < 4 * math.sqrt(alpha0 * (1 - alpha0) / N)


# ---------------------------------------------------------------- planted alpha (closed form)
def _accepted_pmf(alpha, K):
    """pmf of n = leading successes of K iid Bernoulli(alpha) trials."""
    pmf = [alpha ** k * (1 - alpha) for k in range(K)] + [alpha ** K]
    return np.array(pmf)


@pytest.mark.parametrize("alpha,K", [(0.5, 2), (0.8, 4), (0.95, 8)])
def test_planted_alpha_greedy_mean(alpha, K):
    """E[n + 1] = (1 - alpha^{K+1}) / (1 - alpha) ("What decides the speed-up")."""
    c = synth.greedy_case(4000, K, 64, alpha=alpha, dtype=synth.F32, seed=5)
    r = oracle.verify_greedy(c.target_values(), c.tokens)
    m = r["num_accepted"] + 1
    closed = (1 - alpha ** (K + 1)) / (1 - alpha)
    pmf = _accepted_pmf(alpha, K)
    var = (pmf * (np.arange(K + 1) + 1.0) ** 2).sum() - closed ** 2
    z = (m.mean() - closed) / math.sqrt(var / m.size)
    assert abs(z) < 4, (m.mean(), closed, z)
    # the planted argmax is what greedy reports
    assert np.array_equal(r["argmax"], c.recipe["planted"])


@pytest.mark.parametrize("alpha,K", [(0.6, 3), (0.9, 5)])
def test_planted_alpha_sampling_mean(alpha, K):
    """Sampling mode with sum_v min(p(v), q(v)) = alpha at every position: each
    test accepts with probability alpha independently, so E[n + 1] follows the
    same closed form. V = 2, p = (1/2, 1/2), q = (1/2 + d, 1/2 - d), d = 1 - alpha."""
    N = 20000
    rng = np.random.default_rng(17)
    d = 1 - alpha
    q = np.array([0.5 + d, 0.5 - d])
    p = np.array([0.5, 0.5])
    zt = np.broadcast_to(np.log(q), (N, K + 1, 2))
    zd = np.broadcast_to(np.log(p), (N, K, 2))
    tok = rng.integers(0, 2, size=(N, K))
    u = rng.random((N, K + 1))
    r = oracle.verify_sample(zt, zd, tok, u, 1.0, row_chunk=N)
    m = r["num_accepted"] + 1
    closed = (1 - alpha ** (K + 1)) / (1 - alpha)
    pmf = _accepted_pmf(alpha, K)
    var = (pmf * (np.arange(K + 1) + 1.0) ** 2).sum() - closed ** 2
    z = (m.mean() - closed) / math.sqrt(var / N)
    assert abs(z) < 4, (m.mean(), closed, z)


# ---------------------------------------------------------------- greedy = target-only decode
def test_greedy_emits_target_argmax_everywhere():
    """Every emitted token equals the target's own argmax at its position
    (np.argmax: first maximum), so greedy output matches the target alone."""
    rng = np.random.default_rng(9)
    B, K, V = 300, 5, 40
    zt = rng.integers(-3, 4, size=(B, K + 1, V)).astype(np.float64)   # many ties
    g = np.argmax(zt, axis=-1)
    tok = np.where(rng.random((B, K)) < 0.7, g[:, :K], rng.integers(0, V, size=(B, K)))
    r = oracle.verify_greedy(zt, tok)
    for b in range(B):
        n = r["num_accepted"][b]
        assert r["out_tokens"][b, : n + 1].tolist() == g[b, : n + 1].tolist()
        assert (r["out_tokens"][b, n + 1:] == -1).all()
        assert n == K or tok[b, n] != g[b, n]


def test_sampling_prefix_is_accepted_drafts():
    c = synth.sampling_case(6, 4, 257, temperature=0.8, target_std=2.0, draft_noise_std=0.7,
                            dtype=synth.F32, seed=1)
    r = oracle.verify_sample(c.target_values(), c.draft_values(), c.tokens, c.uniforms, 0.8)
    for b in range(c.B):
        n = r["num_accepted"][b]
        assert r["out_tokens"][b, :n].tolist() == c.tokens[b, :n].tolist()
        assert 0 <= r["out_tokens"][b, n] < c.V
        assert (r["out_tokens"][b, n + 1:] == -1).all()


def test_greedy_unusable_rows_by_hand():
    """Greedy with a NaN row or a bad draft token, worked by hand: a NaN row
    has no argmax; it makes the batch row an error only when the step uses it
    (the first position not accepted, or row K after K acceptances); a draft
    token outside [0, V) is always an error. Rows of equal values (-inf
    included) have argmax 0."""
    nan, inf = np.nan, np.inf
    V = 4
    good = [0.0, 3.0, 1.0, 2.0]                  # argmax 1
    cases = [
        # (rows 0..K, draft tokens, expected out, expected n)
        ([[0, nan, 1, 2], good, good], [1, 1], [-1, -1, -1], -1),   # row 0 used, NaN
        ([good, [0, 1, nan, 2], good], [1, 1], [-1, -1, -1], -1),   # row 1 is the first mismatch
        ([good, good, [nan] * 4], [1, 1], [-1, -1, -1], -1),        # all accepted, bonus row NaN
        ([good, good, [nan] * 4], [1, 3], [1, 1, -1], 1),           # row 2 never used
        ([good, [2, 9, 9, 0], [nan] * 4], [2, 1], [1, -1, -1], 0),  # mismatch at 0
        ([good, good, good], [1, 4], [-1, -1, -1], -1),             # token out of range
        ([good, good, good], [-1, 1], [-1, -1, -1], -1),            # negative token
        ([[-inf] * 4, good, good], [0, 1], [0, 1, 1], 2),           # all -inf: argmax 0
        ([[5, 5, 5, 5], good, good], [1, 1], [0, -1, -1], 0),       # tie: lowest index
    ]
    for rows, tok, exp_out, exp_n in cases:
        z = np.array([rows], np.float64)
        r = oracle.verify_greedy(z, np.array([tok]))
        assert r["out_tokens"][0].tolist() == exp_out, (rows, tok)
        assert int(r["num_accepted"][0]) == exp_n, (rows, tok)
