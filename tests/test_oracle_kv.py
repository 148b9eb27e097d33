"""Pins for the KV commit/rollback oracle (CPU only).

The oracle works on block tables and returns a copy list. These tests check it
against a brute-force model that never looks at block tables the way the
oracle does: a dict from (block, offset) to the token-slot label it holds,
walked through each row's logical positions after the commit. Sources: the
lesson's exercise of two sequences (one accepts everything, one rejects at
position 2) and "Step 4: KV rollback accounting"; the sglang_spec_decode README
requirement that no block is leaked or freed twice across all rejection
patterns.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import kv as okv
import synth


def _apply_and_read(case, res):
    """Brute force: label every slot, apply the copy list, read logical sequences."""
    bs = case.block_size
    mem = {}
    for b in range(case.B):
        for pos in range(int(case.seq_lens[b])):
            blk = int(case.block_table[b, pos // bs])
            mem[(blk, pos % bs)] = ("prefix", b, pos)
        for s in range(case.K + 1):
            blk = int(case.prov_blocks[b, s // bs])
            mem[(blk, s % bs)] = ("prov", b, s)
    snapshot = dict(mem)
    for (b, s, sb, so, db, do) in res["copies"]:
        mem[(db, do)] = snapshot[(sb, so)]
    seqs = []
    for b in range(case.B):
        L = int(res["seq_lens"][b])
        seqs.append([mem.get((int(res["block_table"][b, p // bs]), p % bs)) for p in range(L)])
    return seqs


def _commit(case):
    return oracle.kv_commit(case.block_table, case.seq_lens, case.num_accepted, case.prov_blocks,
                            case.free_stack, case.free_top, block_size=case.block_size, K=case.K,
                            num_blocks=case.num_blocks)


def _expected_seq(case, b):
    L, n = int(case.seq_lens[b]), int(case.num_accepted[b])
    return [("prefix", b, p) for p in range(L)] + [("prov", b, s) for s in range(n + 1)]


def test_two_sequences_exercise():
    """Row A accepts all K = 4 drafts, row B rejects at position 2 (n = 2):
    new lengths prefix + 5 and prefix + 3."""
    c = synth.kv_case(2, 4, seq_lens=np.array([37, 64]), num_accepted=np.array([4, 2]), seed=1)
    res = _commit(c)
    assert res["err"] == 0
    assert res["seq_lens"].tolist() == [37 + 5, 64 + 3]
    seqs = _apply_and_read(c, res)
    for b in range(2):
        assert seqs[b] == _expected_seq(c, b)
    assert oracle.pool_invariant_ok(res["block_table"], res["prov_blocks"], res["free_stack"],
                                    res["free_top"], c.num_blocks)


@pytest.mark.parametrize("K,bs", [(4, 16), (7, 16), (15, 16), (5, 4), (9, 8)])
def test_every_rejection_pattern(K, bs):
    """Every n in 0..K at prefix lengths straddling block boundaries."""
    lens = [bs * 3 - 1, bs * 3, bs * 3 + 1, bs * 4 - K, bs * 4 - K - 1, 0, 1]
    rows = list(itertools.product(lens, range(K + 1)))
    sl = np.array([r[0] for r in rows])
    na = np.array([r[1] for r in rows])
    c = synth.kv_case(len(rows), K, block_size=bs, seq_lens=sl, num_accepted=na, seed=K * 31 + bs)
    res = _commit(c)
    assert res["err"] == 0
    seqs = _apply_and_read(c, res)
    for b in range(c.B):
        assert seqs[b] == _expected_seq(c, b), b
        assert res["seq_lens"][b] == sl[b] + na[b] + 1
    assert oracle.pool_invariant_ok(res["block_table"], res["prov_blocks"], res["free_stack"],
                                    res["free_top"], c.num_blocks)
    assert oracle.pool_invariant_ok(c.block_table, c.prov_blocks, c.free_stack, c.free_top,
                                    c.num_blocks)
    # exactly the blocks the new lengths need are in use, and no provisional block remains
    used = sum(-(-int(L) // bs) for L in res["seq_lens"])
    assert (res["block_table"] >= 0).sum() == used
    assert (res["prov_blocks"] == -1).all()


def test_allocation_order_is_rows_ascending_pop_before_push():
    c = synth.kv_case(3, 4, seq_lens=np.array([16, 15, 32]), num_accepted=np.array([0, 4, 1]),
                      seed=2)
    top0 = c.free_top
    stack0 = c.free_stack.copy()
    res = _commit(c)
    # row 0 (16 -> 17) needs a block, row 1 (15 -> 20) needs one, row 2 (32 -> 34) needs one
    assert res["block_table"][0, 1] == stack0[top0 - 1]
    assert res["block_table"][1, 1] == stack0[top0 - 2]
    assert res["block_table"][2, 2] == stack0[top0 - 3]
    # then the three provisional blocks are pushed in row order
    assert res["free_top"] == top0 - 3 + 3
    assert res["free_stack"][top0 - 3: top0].tolist() == c.prov_blocks[:, 0].tolist()


@pytest.mark.parametrize("mutate,bit", [
    ("accept_high", okv.ERR_BAD_ACCEPT),
    ("accept_neg", okv.ERR_BAD_ACCEPT),
    ("len_neg", okv.ERR_BAD_LENGTH),
    ("table_small", okv.ERR_BAD_LENGTH),
    ("no_space", okv.ERR_NO_SPACE),
    ("bad_table_block", okv.ERR_BAD_BLOCK),
    ("bad_prov_block", okv.ERR_BAD_BLOCK),
    ("slot_taken", okv.ERR_BAD_BLOCK),
    ("top_too_big", okv.ERR_NO_SPACE),
    ("bad_free_entry", okv.ERR_BAD_BLOCK),
    ("prov_out_of_range", okv.ERR_BAD_BLOCK),
])
def test_errors_leave_state_unchanged(mutate, bit):
    c = synth.kv_case(4, 4, seq_lens=np.array([16, 20, 31, 47]), num_accepted=np.array([1, 2, 4, 0]),
                      seed=4)
    if mutate == "accept_high":
        c.num_accepted[2] = 5
    elif mutate == "accept_neg":
        c.num_accepted[1] = -1
    elif mutate == "len_neg":
        c.seq_lens[0] = -3
    elif mutate == "table_small":
        c.block_table = c.block_table[:, :2].copy()
    elif mutate == "no_space":
        c.free_top = 1
    elif mutate == "bad_table_block":
        c.block_table[3, 2] = c.num_blocks       # row 3 (L = 47) has its tail in block 2
    elif mutate == "bad_prov_block":
        c.prov_blocks[1, 0] = -1
    elif mutate == "slot_taken":
        c.block_table[0, 1] = c.free_stack[0]
    elif mutate == "top_too_big":
        c.free_top = c.num_blocks + 1
    elif mutate == "bad_free_entry":
        c.free_stack[c.free_top - 1] = -5
    elif mutate == "prov_out_of_range":
        c.prov_blocks[2, 0] = c.num_blocks + 3
    res = _commit(c)
    assert res["err"] & bit
    assert res["copies"] == []
    assert np.array_equal(res["block_table"], c.block_table)
    assert np.array_equal(res["seq_lens"], c.seq_lens)
    assert np.array_equal(res["prov_blocks"], c.prov_blocks)
    assert res["free_top"] == c.free_top


# ------------------------------------------------------------- tree slot maps
def test_identity_slot_map_is_the_linear_commit():
    c = synth.kv_case(6, 5, block_size=4, seed=9)
    ident = np.tile(np.arange(6, dtype=np.int32), (6, 1))
    a = _commit(c)
    b = oracle.kv_commit(c.block_table, c.seq_lens, c.num_accepted, c.prov_blocks, c.free_stack,
                         c.free_top, block_size=c.block_size, K=c.K, num_blocks=c.num_blocks,
                         slot_map=ident)
    for k in ("block_table", "seq_lens", "prov_blocks", "free_stack"):
        assert np.array_equal(a[k], b[k])
    assert a["free_top"] == b["free_top"] and a["copies"] == b["copies"] and b["err"] == 0


@pytest.mark.parametrize("bs", [4, 16])
@pytest.mark.parametrize("branching", [(2, 2, 2), (3, 2)])
def test_tree_commit_keeps_the_surviving_path(bs, branching):
    """Greedy tree verification, then the commit with its slot map: each row's
    sequence becomes prefix + the KV of the last committed token + the KV of
    the kept nodes, in path order (brute-force slot labels)."""
    t = synth.tree_case(10, 50, branching=branching, alpha=0.9, seed=bs, dtype=synth.F32)
    r = oracle.verify_tree_greedy(t.target_values(), t.parents, t.tokens)
    N = t.N
    c = synth.kv_case(t.B, N, block_size=bs, prefix_lo=0, prefix_hi=3 * bs,
                      num_accepted=r["num_accepted"].astype(np.int32), seed=bs + N)
    slot_map = np.where(r["slots"] < 0, 0, r["slots"]).astype(np.int32)
    res = oracle.kv_commit(c.block_table, c.seq_lens, c.num_accepted, c.prov_blocks, c.free_stack,
                           c.free_top, block_size=bs, K=N, num_blocks=c.num_blocks,
                           slot_map=slot_map)
    assert res["err"] == 0
    seqs = _apply_and_read(c, res)
    assert any(int(n) >= 2 for n in r["num_accepted"])
    for b in range(c.B):
        L, n = int(c.seq_lens[b]), int(r["num_accepted"][b])
        kept = [0] + [1 + int(x) for x in oracle.tree_path(
            t.parents[b], int(r["slots"][b, n]) - 1 if n else -1)]
        assert kept == r["slots"][b, :n + 1].tolist()
        assert seqs[b] == [("prefix", b, p) for p in range(L)] + [("prov", b, s) for s in kept]
    assert oracle.pool_invariant_ok(res["block_table"], res["prov_blocks"], res["free_stack"],
                                    res["free_top"], c.num_blocks)


@pytest.mark.parametrize("bad", [-1, 5])
def test_bad_slot_map_entry_leaves_state_unchanged(bad):
    c = synth.kv_case(3, 4, seq_lens=np.array([5, 9, 16]), num_accepted=np.array([2, 4, 0]),
                      seed=5)
    sm = np.tile(np.arange(5, dtype=np.int32), (3, 1))
    sm[0, 4] = bad                      # beyond row 0's kept positions: ignored
    ok = oracle.kv_commit(c.block_table, c.seq_lens, c.num_accepted, c.prov_blocks, c.free_stack,
                          c.free_top, block_size=c.block_size, K=4, num_blocks=c.num_blocks,
                          slot_map=sm)
    assert ok["err"] == 0
    sm[1, 3] = bad                      # a kept position of row 1
    res = oracle.kv_commit(c.block_table, c.seq_lens, c.num_accepted, c.prov_blocks, c.free_stack,
                           c.free_top, block_size=c.block_size, K=4, num_blocks=c.num_blocks,
                           slot_map=sm)
    assert res["err"] == okv.ERR_BAD_SLOT
    assert np.array_equal(res["block_table"], c.block_table) and res["copies"] == []
    assert np.array_equal(res["seq_lens"], c.seq_lens) and res["free_top"] == c.free_top


# ------------------------------------------------------- the pool checker itself
def _pool(case):
    return dict(block_table=case.block_table.copy(), prov_blocks=case.prov_blocks.copy(),
                free_stack=case.free_stack.copy(), free_top=int(case.free_top),
                num_blocks=case.num_blocks)


def _sound_pool():
    c = synth.kv_case(3, 4, seq_lens=np.array([20, 33, 16]), num_accepted=np.array([1, 4, 0]),
                      spare_blocks=5, seed=11)
    st = _pool(c)
    assert oracle.pool_invariant_ok(**st)
    return st


def test_pool_checker_rejects_a_leaked_block():
    """A block that no table, provisional entry or live stack entry holds."""
    st = _sound_pool()
    st["block_table"][1, 0] = -1
    assert not oracle.pool_invariant_ok(**st)
    st = _sound_pool()
    st["free_top"] -= 1                     # the top stack entry becomes dead
    assert not oracle.pool_invariant_ok(**st)


def test_pool_checker_rejects_a_block_in_two_tables():
    st = _sound_pool()
    leaked = int(st["block_table"][1, 0])
    st["block_table"][1, 0] = st["block_table"][0, 0]      # double allocation
    assert not oracle.pool_invariant_ok(**st)
    # even when the count of live entries is restored by freeing the lost id
    st["free_stack"][st["free_top"]] = leaked
    st["free_top"] += 1
    st["block_table"][2, 0] = -1
    assert not oracle.pool_invariant_ok(**st)


def test_pool_checker_rejects_a_block_in_a_table_and_on_the_stack():
    st = _sound_pool()
    top = st["free_top"]
    st["free_stack"][top - 1] = st["block_table"][0, 1]    # double free
    assert not oracle.pool_invariant_ok(**st)


def test_pool_checker_rejects_a_provisional_block_also_free():
    st = _sound_pool()
    st["free_stack"][st["free_top"]] = st["prov_blocks"][2, 0]
    st["free_top"] += 1
    assert not oracle.pool_invariant_ok(**st)


@pytest.mark.parametrize("where", ["table", "prov", "stack"])
@pytest.mark.parametrize("bad", ["num_blocks", "minus_two"])
def test_pool_checker_rejects_an_out_of_range_id(where, bad):
    st = _sound_pool()
    v = st["num_blocks"] if bad == "num_blocks" else -2
    if where == "table":
        st["block_table"][0, 0] = v
    elif where == "prov":
        st["prov_blocks"][1, 0] = v
    else:
        st["free_stack"][0] = v
    assert not oracle.pool_invariant_ok(**st)


def test_pool_checker_ignores_dead_stack_entries_only():
    """Entries at or above free_top are dead: a stale copy there of a block in a
    table is fine, but a block whose only copy is there is leaked."""
    st = _sound_pool()
    top = st["free_top"]
    st["free_stack"][top] = st["block_table"][2, 0]        # stale, dead entry
    assert oracle.pool_invariant_ok(**st)
    st = _sound_pool()
    top = st["free_top"]
    st["free_stack"][top], st["free_stack"][top - 1] = st["free_stack"][top - 1], -1
    st["free_top"] = top - 1                               # the only copy is now dead
    assert not oracle.pool_invariant_ok(**st)


def test_pool_checker_rejects_a_top_outside_the_stack():
    st = _sound_pool()
    st["free_top"] = -1
    assert not oracle.pool_invariant_ok(**st)
    st = _sound_pool()
    st["free_top"] = st["free_stack"].size + 1
    assert not oracle.pool_invariant_ok(**st)
