"""Pins of the greedy tree-verification oracle (CPU only).

The oracle keeps the deepest surviving node (lowest index among equals) and
walks its parents. The pins check it against what the pages and the
mathematics fix, by other routes:
  * hand-worked trees (tests/golden/tree_examples.json, cited there);
  * a chain tree is the linear draft, so the result equals oracle
    verify_greedy (pinned on its own in test_oracle_verify.py);
  * brute force over every root-to-node path, checked token by token;
  * with distinct sibling tokens the kept path is target-only greedy
    decoding followed down the tree (the losslessness of greedy
    verification), computed by a forward walk;
  * error rows: invalid trees, bad tokens, NaN rows that the result uses.
"""
import json
import pathlib

import numpy as np
import pytest

import oracle
import synth

GOLDEN = pathlib.Path(__file__).parent / "golden" / "tree_examples.json"


def _fixture():
    return json.loads(GOLDEN.read_text())


def _logits_from_argmax(row_argmax, V, extra_max=()):
    z = np.zeros((1, len(row_argmax), V), np.float64)
    for r, g in enumerate(row_argmax):
        z[0, r, g] = 1.0
    for r, v in extra_max:
        z[0, r, v] = 1.0
    return z


@pytest.mark.parametrize("case", _fixture()["cases"], ids=lambda c: c["name"])
def test_hand_tree_cases(case):
    V = _fixture()["V"]
    z = _logits_from_argmax(case["row_argmax"], V, case.get("extra_max", ()))
    r = oracle.verify_tree_greedy(z, [case["parents"]], [case["tokens"]])
    assert r["out_tokens"][0].tolist() == case["out_tokens"]
    assert int(r["num_accepted"][0]) == case["num_accepted"]
    assert r["slots"][0].tolist() == case["slots"]


@pytest.mark.parametrize("seed", range(4))
def test_chain_tree_equals_linear_greedy(seed):
    c = synth.greedy_case(16, 6, 300, alpha=0.8, seed=seed, dtype=synth.F32)
    chain = np.tile(np.arange(-1, c.K - 1, dtype=np.int32), (c.B, 1))
    r = oracle.verify_tree_greedy(c.target_values(), chain, c.tokens)
    g = oracle.verify_greedy(c.target_values(), c.tokens)
    assert np.array_equal(r["out_tokens"], g["out_tokens"])
    assert np.array_equal(r["num_accepted"], g["num_accepted"])
    n = g["num_accepted"]
    for b in range(c.B):
        assert r["slots"][b, :n[b] + 1].tolist() == list(range(n[b] + 1))
        assert (r["slots"][b, n[b] + 1:] == -1).all()


def _brute_force(z, par, tok):
    """Every node's root path, checked position by position; longest kept,
    lowest end node among equals. Rows are compared by their maximum value
    and first index, written out with Python max()."""
    N = len(par)

    def arg(r):
        row = list(z[r])
        m = max(row)
        return row.index(m)

    best_path = []
    for i in range(N):
        path, j = [], i
        while j >= 0:
            path.append(j)
            j = int(par[j])
        path = path[::-1]
        ok = all(int(tok[node]) == arg(0 if k == 0 else path[k - 1] + 1)
                 for k, node in enumerate(path))
        if ok and len(path) > len(best_path):
            best_path = path
    last_row = 0 if not best_path else best_path[-1] + 1
    return [int(tok[x]) for x in best_path] + [arg(last_row)], best_path


@pytest.mark.parametrize("distinct", [True, False])
@pytest.mark.parametrize("seed", range(3))
def test_brute_force_random_trees(seed, distinct):
    c = synth.tree_case(12, 40, N=9, alpha=0.8, distinct=distinct, seed=seed, dtype=synth.F32)
    z = c.target_values().astype(np.float64)
    r = oracle.verify_tree_greedy(z, c.parents, c.tokens)
    for b in range(c.B):
        toks, path = _brute_force(z[b], c.parents[b], c.tokens[b])
        n = len(path)
        assert int(r["num_accepted"][b]) == n
        assert r["out_tokens"][b, :n + 1].tolist() == toks
        assert (r["out_tokens"][b, n + 1:] == -1).all()
        assert r["slots"][b, :n + 1].tolist() == [0] + [p + 1 for p in path]


@pytest.mark.parametrize("branching", [(2, 2, 2), (4, 2), (1, 1, 1, 1), (3, 3, 3)])
def test_distinct_siblings_follow_target_decoding(branching):
    """Walk forward: emit the target's argmax of the current row, move to the
    child carrying it, stop when none does. With distinct siblings this is
    the unique surviving path and equals the oracle's result."""
    c = synth.tree_case(24, 64, branching=branching, alpha=0.75, seed=len(branching),
                        dtype=synth.F32)
    z = c.target_values().astype(np.float64)
    r = oracle.verify_tree_greedy(z, c.parents, c.tokens)
    planted = c.recipe["planted"]
    for b in range(c.B):
        emitted, row = [], 0
        while True:
            g = int(planted[b, row])           # the planted maximum is the argmax
            emitted.append(g)
            kids = [i for i in range(c.N) if c.parents[b, i] == row - 1 and c.tokens[b, i] == g]
            if not kids:
                break
            row = kids[0] + 1
        n = len(emitted) - 1
        assert int(r["num_accepted"][b]) == n
        assert r["out_tokens"][b, :n + 1].tolist() == emitted


def test_invalid_tree_and_tokens_are_errors():
    z = np.zeros((1, 4, 10))
    z[0, :, 3] = 1.0
    for par, tok in [([-1, 1, 0], [3, 3, 3]),      # parent not before the node
                     ([-1, -2, 0], [3, 3, 3]),     # parent below -1
                     ([-1, 0, 1], [3, 10, 3]),     # token out of range
                     ([-1, 0, 1], [-1, 3, 3])]:
        r = oracle.verify_tree_greedy(z, [par], [tok])
        assert int(r["num_accepted"][0]) == -1
        assert (r["out_tokens"] == -1).all() and (r["slots"] == -1).all()


def test_nan_rows_only_matter_when_used():
    z = np.zeros((1, 4, 10))
    z[0, :, 3] = 1.0
    par, tok = [-1, -1, 0], [3, 5, 3]     # node 0 and node 2 survive; node 1 does not
    zn = z.copy()
    zn[0, 2, 4] = np.nan                  # row of node 1 (not a survivor)
    r = oracle.verify_tree_greedy(zn, [par], [tok])
    assert int(r["num_accepted"][0]) == 2
    assert r["out_tokens"][0].tolist() == [3, 3, 3, -1]
    for row in (0, 1, 3):                 # root row, rows of survivors 0 and 2
        zn = z.copy()
        zn[0, row, 7] = np.nan
        assert int(oracle.verify_tree_greedy(zn, [par], [tok])["num_accepted"][0]) == -1
    zi = z.copy()
    zi[0, 1, :] = -np.inf                 # all equal: argmax 0 by the lowest-index rule
    r = oracle.verify_tree_greedy(zi, [par], [tok])
    assert int(r["num_accepted"][0]) == 1 and r["out_tokens"][0].tolist() == [3, 0, -1, -1]


def test_empty_tree():
    z = np.zeros((2, 1, 7))
    z[0, 0, 4] = 2.0
    z[1, 0, 6] = 2.0
    r = oracle.verify_tree_greedy(z, np.zeros((2, 0), np.int32), np.zeros((2, 0), np.int32))
    assert r["out_tokens"].tolist() == [[4], [6]]
    assert r["num_accepted"].tolist() == [0, 0]
    assert r["slots"].tolist() == [[0], [0]]
