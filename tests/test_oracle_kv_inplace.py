"""Pins of oracle.kv_truncate_inplace (in-place KV commit and eviction).

A hand-worked table; the round trip append-then-evict restores the table and
the set of free blocks exactly; after a commit the lengths are those of the
copying commit (L + n + 1) and each row keeps exactly ceil(len / bs) blocks;
no block is leaked or freed twice; invalid calls change nothing.
"""
import numpy as np
import pytest

import oracle
from oracle.kv import ERR_BAD_ACCEPT, ERR_BAD_BLOCK, ERR_BAD_LENGTH


def _cdiv(a, b):
    return -(-a // b)


def test_hand_table():
    # bs = 4, K = 3; the row's prefix L = 6 occupies blocks 10, 11; the provisional
    # positions 6..9 reach block index 2 (block 12)
    bt = np.array([[10, 11, 12, -1]])
    fs = np.array([20, 21, -1, -1, -1])
    kw = dict(block_size=4, K=3, num_blocks=25)
    r = oracle.kv_truncate_inplace(bt, [6], [1], fs, 2, **kw)    # new length 8: block 12 free
    assert r["err"] == 0 and r["seq_lens"].tolist() == [8]
    assert r["block_table"].tolist() == [[10, 11, -1, -1]]
    assert r["free_stack"][:r["free_top"]].tolist() == [20, 21, 12]
    r = oracle.kv_truncate_inplace(bt, [6], [2], fs, 2, **kw)    # new length 9: keeps block 12
    assert r["block_table"].tolist() == [[10, 11, 12, -1]] and r["free_top"] == 2
    r = oracle.kv_truncate_inplace(bt, [6], None, fs, 2, evict=True, **kw)  # back to 6
    assert r["seq_lens"].tolist() == [6] and r["block_table"].tolist() == [[10, 11, -1, -1]]


def _state(rng, B, K, bs, nb, max_blocks):
    """Prefix tables (rows ascending from a shuffled pool), then the append of the
    K+1 provisional slots (new blocks popped from the free stack)."""
    ids = rng.permutation(nb)
    L = rng.integers(0, (max_blocks - 2) * bs - K, size=B)
    bt = -np.ones((B, max_blocks), np.int64)
    k = 0
    for b in range(B):
        for j in range(_cdiv(int(L[b]), bs)):
            bt[b, j] = ids[k]
            k += 1
    fs = -np.ones(nb, np.int64)
    rest = ids[k:]
    fs[:rest.size] = rest
    top = rest.size
    before = dict(bt=bt.copy(), fs=fs.copy(), top=top)
    for b in range(B):
        for j in range(_cdiv(int(L[b]), bs), _cdiv(int(L[b]) + K + 1, bs)):
            top -= 1
            bt[b, j] = fs[top]
            fs[top] = -1
    return L, bt, fs, top, before


@pytest.mark.parametrize("bs", [1, 4, 16])
def test_append_then_evict_restores(bs):
    rng = np.random.default_rng(bs)
    B, K, nb, mb = 12, 5, 600, 40
    L, bt, fs, top, before = _state(rng, B, K, bs, nb, mb)
    r = oracle.kv_truncate_inplace(bt, L, None, fs, top, block_size=bs, K=K, num_blocks=nb,
                                   evict=True)
    assert r["err"] == 0
    assert np.array_equal(r["block_table"], before["bt"])
    assert r["free_top"] == before["top"]
    assert sorted(r["free_stack"][:r["free_top"]].tolist()) == \
        sorted(before["fs"][:before["top"]].tolist())
    assert np.array_equal(r["seq_lens"], L)


@pytest.mark.parametrize("bs", [1, 4, 16])
def test_commit_lengths_blocks_and_invariant(bs):
    rng = np.random.default_rng(100 + bs)
    B, K, nb, mb = 12, 5, 600, 40
    L, bt, fs, top, _ = _state(rng, B, K, bs, nb, mb)
    n = rng.integers(0, K + 1, size=B)
    r = oracle.kv_truncate_inplace(bt, L, n, fs, top, block_size=bs, K=K, num_blocks=nb)
    assert r["err"] == 0
    assert np.array_equal(r["seq_lens"], L + n + 1)
    for b in range(B):
        live = int(np.sum(r["block_table"][b] >= 0))
        assert live == _cdiv(int(L[b] + n[b] + 1), bs)
        assert np.all(r["block_table"][b, :live] >= 0)
        assert np.all(r["block_table"][b, :live] == bt[b, :live])  # kept blocks unchanged
    assert oracle.pool_invariant_ok(r["block_table"], np.zeros((0,)), r["free_stack"],
                                    r["free_top"], nb)


def test_errors_change_nothing():
    rng = np.random.default_rng(7)
    B, K, bs, nb, mb = 6, 3, 4, 200, 20
    L, bt, fs, top, _ = _state(rng, B, K, bs, nb, mb)
    n = rng.integers(0, K + 1, size=B)
    cases = []
    bad_n = n.copy(); bad_n[2] = K + 1
    cases.append((bt, L, bad_n, fs, top, ERR_BAD_ACCEPT))
    bad_L = L.copy(); bad_L[1] = -1
    cases.append((bt, bad_L, n, fs, top, ERR_BAD_LENGTH))
    bad_bt = bt.copy(); bad_bt[3, int(L[3]) // bs] = nb
    cases.append((bad_bt, L, n, fs, top, ERR_BAD_BLOCK))
    cases.append((bt, L, n, fs, nb, ERR_BAD_BLOCK))  # pushes would overflow the stack
    for t_bt, t_L, t_n, t_fs, t_top, bit in cases:
        r = oracle.kv_truncate_inplace(t_bt, t_L, t_n, t_fs, t_top, block_size=bs, K=K,
                                       num_blocks=nb)
        assert r["err"] & bit
        assert np.array_equal(r["block_table"], t_bt) and np.array_equal(r["seq_lens"], t_L)
        assert r["free_top"] == t_top and np.array_equal(r["free_stack"], t_fs)
