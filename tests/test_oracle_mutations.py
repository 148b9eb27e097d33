"""Planted mistakes in the oracle (CPU only).

Each test swaps one oracle function for a plausible wrong version and checks
that at least one pin from test_oracle_verify.py / test_oracle_kv.py fails on
it. This shows the pins can tell a right oracle from a wrong one; the mistakes
live only here, in the CPU copy under test.
"""
import numpy as np
import pytest

import oracle
from oracle import kv as okv
from oracle import verify as ov
from tests import test_oracle_verify as tv


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def test_swapped_residual_is_caught(golden, monkeypatch):
    monkeypatch.setattr(ov, "residual", lambda q, p: np.maximum(np.asarray(p) - np.asarray(q), 0.0))
    monkeypatch.setattr(oracle, "residual", ov.residual)
    assert _fails(tv.test_hand_sample_cases, golden, 1.0)


def test_non_strict_accept_is_caught(monkeypatch):
    def wrong(lq, lp, u):
        lq, lp, u = (np.asarray(x, np.float64) for x in (lq, lp, u))
        return np.isneginf(lp) | (u <= np.minimum(1.0, np.exp(lq - lp)))
    monkeypatch.setattr(ov, "accept_test", wrong)
    monkeypatch.setattr(oracle, "accept_test", wrong)
    assert _fails(tv.test_accept_rule_edges)


def test_non_strict_inverse_cdf_is_caught(golden, monkeypatch):
    def wrong(w, u):
        w = np.asarray(w, np.float64)
        c = np.cumsum(w, axis=-1)
        t = np.asarray(u, np.float64) * c[..., -1]
        return np.argmax(t[..., None] <= c, axis=-1), np.zeros(np.shape(u))
    monkeypatch.setattr(ov, "inverse_cdf", wrong)
    monkeypatch.setattr(oracle, "inverse_cdf", wrong)
    assert _fails(tv.test_hand_probability_cases, golden)


def test_bonus_from_wrong_row_is_caught(golden, monkeypatch):
    real_softmax = ov.softmax

    def verify_sample_wrong_bonus(target, draft, tokens, uniforms, temperature, **kw):
        # bonus drawn from q_{K-1} instead of q_K
        t = np.array(target, np.float64, copy=True)
        t[:, -1] = t[:, -2]
        return ov.__dict__["_real_verify_sample"](t, draft, tokens, uniforms, temperature, **kw)

    ov.__dict__["_real_verify_sample"] = ov.verify_sample
    monkeypatch.setattr(oracle, "verify_sample", verify_sample_wrong_bonus)
    try:
        assert _fails(tv.test_hand_sample_cases, golden, 1.0)
    finally:
        del ov.__dict__["_real_verify_sample"]
    assert ov.softmax is real_softmax


def test_reused_accept_uniform_is_caught(monkeypatch):
    """Drawing the correction with u_j (the uniform of the failed test) instead of
    u_K biases the correction; the brute-force losslessness pin detects it."""
    real = ov.verify_sample

    def wrong(target, draft, tokens, uniforms, temperature, **kw):
        u = np.array(uniforms, np.float64, copy=True)
        r0 = real(target, draft, tokens, u, temperature, **kw)
        n = r0["num_accepted"]
        K = u.shape[1] - 1
        rows = np.arange(u.shape[0])
        u[rows, K] = np.where(n < K, u[rows, np.minimum(n, K - 1)], u[rows, K])
        return real(target, draft, tokens, u, temperature, **kw)

    monkeypatch.setattr(oracle, "verify_sample", wrong)
    assert _fails(tv.test_losslessness_brute_force, 3, 1, True)


def test_missing_temperature_on_draft_is_caught(golden, monkeypatch):
    real = ov.verify_sample

    def wrong(target, draft, tokens, uniforms, temperature, **kw):
        # draft logits left at T = 1 while the target uses T
        T = oracle.temperature64(temperature)
        return real(target, np.asarray(draft) / T, tokens, uniforms, temperature, **kw)

    monkeypatch.setattr(oracle, "verify_sample", wrong)
    assert _fails(tv.test_hand_sample_cases, golden, 0.5)


def test_greedy_highest_index_tie_is_caught(golden, monkeypatch):
    def wrong(target, tokens):
        t = np.asarray(target, np.float64)[..., ::-1]
        V = t.shape[-1]
        g = V - 1 - np.argmax(t, axis=-1)
        tok = np.asarray(tokens)
        K = tok.shape[1]
        n = ov._leading_true(tok == g[:, :K])
        out = np.full((tok.shape[0], K + 1), -1)
        for b in range(tok.shape[0]):
            out[b, :n[b]] = tok[b, :n[b]]
            out[b, n[b]] = g[b, n[b]]
        return dict(out_tokens=out, num_accepted=n, argmax=g)

    monkeypatch.setattr(oracle, "verify_greedy", wrong)
    assert _fails(tv.test_hand_greedy_cases, golden)


def test_kv_push_before_pop_is_caught(monkeypatch):
    """Freeing provisional blocks before allocating lets a row receive a block it
    is copying from; the brute-force logical read-back fails."""
    from oracle import kv as okv
    from tests import test_oracle_kv as tk
    real = okv.kv_commit

    def wrong(block_table, seq_lens, num_accepted, prov_blocks, free_stack, free_top, **kw):
        fs = np.array(free_stack, np.int64, copy=True)
        top = int(free_top)
        pb = np.asarray(prov_blocks)
        for b in range(pb.shape[0]):
            for x in pb[b]:
                if x >= 0:
                    fs[top] = x
                    top += 1
        r = real(block_table, seq_lens, num_accepted, prov_blocks, fs, top, **kw)
        return r

    monkeypatch.setattr(oracle, "kv_commit", wrong)
    assert _fails(tk.test_two_sequences_exercise) or _fails(tk.test_every_rejection_pattern, 4, 16)


# ---------------------------------------------------------------- draft trees
from tests import test_oracle_tree as tt  # noqa: E402


def _tree_pins_fail():
    failed = False
    for case in tt._fixture()["cases"]:
        failed |= _fails(tt.test_hand_tree_cases, case)
    for distinct in (True, False):
        failed |= _fails(tt.test_brute_force_random_trees, 0, distinct)
    return failed


def test_tree_own_row_instead_of_parent_row_is_caught(monkeypatch):
    def wrong(g, bad_row, par, tok):
        N = len(par)
        alive = np.zeros(N, bool)
        depth = np.zeros(N, np.int64)
        for i in range(N):
            p = int(par[i])
            alive[i] = (p < 0 or alive[p]) and tok[i] == g[i + 1]   # the node's own row
            depth[i] = 1 if p < 0 else depth[p] + 1
        return alive, depth
    monkeypatch.setattr(ov, "tree_survivors", wrong)
    assert _tree_pins_fail()


def test_tree_first_survivor_instead_of_longest_is_caught(monkeypatch):
    def wrong(alive, depth):
        # the lowest-index survivor, not the end of the longest surviving path
        hits = np.flatnonzero(alive)
        return int(hits[0]) if hits.size else -1
    monkeypatch.setattr(ov, "tree_kept_node", wrong)
    assert _tree_pins_fail()


def test_tree_ancestor_not_required_is_caught(monkeypatch):
    def wrong(g, bad_row, par, tok):
        N = len(par)
        alive = np.zeros(N, bool)
        depth = np.zeros(N, np.int64)
        for i in range(N):
            p = int(par[i])
            alive[i] = tok[i] == g[p + 1]                           # parent's survival dropped
            depth[i] = 1 if p < 0 else depth[p] + 1
        return alive, depth
    monkeypatch.setattr(ov, "tree_survivors", wrong)
    assert _tree_pins_fail()


def test_tree_highest_index_among_equals_is_caught(monkeypatch):
    def wrong(alive, depth):
        best = -1
        for i in range(len(alive)):
            if alive[i] and (best < 0 or depth[i] >= depth[best]):
                best = i
        return best
    monkeypatch.setattr(ov, "tree_kept_node", wrong)
    assert _fails(tt.test_hand_tree_cases, tt._fixture()["cases"][2])


# ---------------------------------------------------------------- top-k / top-p
from oracle import filters as ofl  # noqa: E402
from tests import test_oracle_filters as tf  # noqa: E402


def test_top_p_ignoring_top_k_is_caught(monkeypatch):
    real = ofl.filter_threshold

    def wrong(z, temperature, top_k=0, top_p=1.0):
        # top-p over the whole row instead of the renormalised top-k set
        return max(real(z, temperature, top_k, 1.0), real(z, temperature, 0, top_p))
    monkeypatch.setattr(ofl, "filter_threshold", wrong)
    monkeypatch.setattr(oracle, "filter_threshold", wrong)
    assert _fails(tf.test_top_p_hand_rows) or _fails(tf.test_brute_force, 0)


def test_top_p_without_temperature_is_caught(monkeypatch):
    real = ofl.filter_threshold

    def wrong(z, temperature, top_k=0, top_p=1.0):
        return real(z, 1.0, top_k, top_p)
    monkeypatch.setattr(ofl, "filter_threshold", wrong)
    monkeypatch.setattr(oracle, "filter_threshold", wrong)
    assert _fails(tf.test_brute_force, 1) or _fails(tf.test_parameter_limits)


def test_always_true_pool_checker_is_caught(monkeypatch):
    """A pool checker that accepts everything fails the checker's own pins."""
    from tests import test_oracle_kv as tk
    monkeypatch.setattr(okv, "pool_invariant_ok", lambda *a, **k: True)
    monkeypatch.setattr(oracle, "pool_invariant_ok", lambda *a, **k: True)
    assert _fails(tk.test_pool_checker_rejects_a_leaked_block)
    assert _fails(tk.test_pool_checker_rejects_a_block_in_a_table_and_on_the_stack)


def test_stack_counted_past_top_is_caught(monkeypatch):
    """A checker that counts every stack entry, live or dead."""
    from tests import test_oracle_kv as tk

    def wrong(block_table, prov_blocks, free_stack, free_top, num_blocks):
        fs = np.asarray(free_stack)
        return okv.__dict__["_real_pool_ok"](block_table, prov_blocks, fs, fs.size, num_blocks)

    okv.__dict__["_real_pool_ok"] = okv.pool_invariant_ok
    monkeypatch.setattr(oracle, "pool_invariant_ok", wrong)
    assert _fails(tk.test_pool_checker_ignores_dead_stack_entries_only)
