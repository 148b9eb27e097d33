"""Paged KV-cache commit/rollback, restated on block tables (test infrastructure only).

Sources: "aiengineeringfromscratch.com - Speculative decoding and EAGLE-3",
sections "Rolling back the KV cache" (write drafts to a scratch area and commit
on accept; the rollback cost is bytes per layer per head) and "Step 4: KV
rollback accounting" (the logical length after a step is prefix + j + 1);
"sglang_spec_decode" README, provisional-layer section (provisional blocks are
committed or freed at once; no block may be leaked or freed twice).

Reading used here: each row holds K+1 provisional slots whose KV covers
[last committed token, d_0 .. d_{K-1}]. With n accepted drafts, slots 0..n are
copied to logical positions seq_len .. seq_len + n of the row's own paged
cache, new blocks are taken from the top of the free stack (rows in ascending
order, all pops before any push), then every provisional block is pushed back
in row order and the row's length becomes seq_len + n + 1.

With a slot map (tree drafts: thakicloud.com's "Speculative decoding: when it
loses", section "Grading every branch in one pass", keeps one
root-to-node path of the flattened tree, whose nodes need not sit in
consecutive provisional slots), kept position s = 0..n takes its KV from
provisional slot slot_map[b, s] instead of slot s; the identity map is the
linear case.

The whole call is all-or-nothing: if any row is invalid, or the free stack
cannot cover every row, nothing changes and error bits are returned.
"""
from __future__ import annotations

import numpy as np

# error bits shared in meaning (not in code) with the library's device error word
ERR_BAD_ACCEPT = 1 << 2     # num_accepted outside [0, K]
ERR_BAD_LENGTH = 1 << 3     # negative seq_len, or the row outgrows its block table
ERR_NO_SPACE = 1 << 4       # the free stack cannot supply every new block
ERR_BAD_BLOCK = 1 << 5      # a block id outside [0, num_blocks) where one is needed
ERR_BAD_SLOT = 1 << 7       # a slot_map entry outside [0, K] for a kept position


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def kv_commit(block_table, seq_lens, num_accepted, prov_blocks, free_stack, free_top: int,
              *, block_size: int, K: int, num_blocks: int, slot_map=None) -> dict:
    """One commit/rollback of every row. Returns the new state, the copy list and error bits.

    copies: list of (row, s, src_block, src_offset, dst_block, dst_offset); each
    entry moves one token's KV (all layers, K and V) into kept position s, from
    provisional slot slot_map[row, s] (slot s without a map).
    """
    bt = np.array(block_table, np.int64, copy=True)
    sl = np.array(seq_lens, np.int64, copy=True)
    na = np.asarray(num_accepted, np.int64)
    pb = np.array(prov_blocks, np.int64, copy=True)
    fs = np.array(free_stack, np.int64, copy=True)
    top = int(free_top)
    B, max_blocks = bt.shape
    P = pb.shape[1]
    err = 0
    if slot_map is None:
        sm = np.tile(np.arange(K + 1, dtype=np.int64), (B, 1))
    else:
        sm = np.asarray(slot_map, np.int64).reshape(B, K + 1)

    def ok_block(x):
        return 0 <= x < num_blocks

    # validation of every row before anything changes
    need = np.zeros(B, np.int64)
    push_total = 0
    for b in range(B):
        for k in range(P):                      # every provisional block goes back on the stack
            x = int(pb[b, k])
            if x >= 0:
                push_total += 1
                if x >= num_blocks:
                    err |= ERR_BAD_BLOCK
        n, L = int(na[b]), int(sl[b])
        if not 0 <= n <= K:
            err |= ERR_BAD_ACCEPT
            continue
        if L < 0 or _cdiv(L + n + 1, block_size) > max_blocks:
            err |= ERR_BAD_LENGTH
            continue
        have = _cdiv(L, block_size)
        total = _cdiv(L + n + 1, block_size)
        for j in range(L // block_size, total):  # the blocks the commit writes into
            x = int(bt[b, j])
            if j < have:
                if not ok_block(x):
                    err |= ERR_BAD_BLOCK        # the partly filled tail block
            elif x != -1:
                err |= ERR_BAD_BLOCK            # a slot the commit must fill is already taken
        kept = [int(sm[b, s]) for s in range(n + 1)]   # provisional slots kept
        if any(not 0 <= x <= K for x in kept):
            err |= ERR_BAD_SLOT
        elif any(x // block_size >= P or not ok_block(int(pb[b, x // block_size])) for x in kept):
            err |= ERR_BAD_BLOCK
        need[b] = total - have
    need_total = int(need.sum())
    if err == 0 and (top < 0 or top > num_blocks or need_total > top):
        err |= ERR_NO_SPACE
    if err == 0 and top - need_total + push_total > num_blocks:
        err |= ERR_BAD_BLOCK                    # the pushes would overflow the stack
    if err == 0 and not all(ok_block(int(x)) for x in fs[top - need_total: top]):
        err |= ERR_BAD_BLOCK                    # a block about to be popped is not a valid id
    if err:
        return dict(block_table=np.asarray(block_table, np.int64).copy(),
                    seq_lens=np.asarray(seq_lens, np.int64).copy(),
                    prov_blocks=np.asarray(prov_blocks, np.int64).copy(),
                    free_stack=np.asarray(free_stack, np.int64).copy(), free_top=int(free_top),
                    copies=[], err=err)

    # 1. allocation: pop from the top of the stack, rows ascending
    for b in range(B):
        have = _cdiv(int(sl[b]), block_size)
        for k in range(int(need[b])):
            top -= 1
            bt[b, have + k] = fs[top]
            fs[top] = -1
    # 2. copies of the accepted slots 0..n into logical positions L..L+n
    copies = []
    for b in range(B):
        L, n = int(sl[b]), int(na[b])
        for s in range(n + 1):
            x = int(sm[b, s])
            src_b, src_o = int(pb[b, x // block_size]), x % block_size
            p = L + s
            dst_b, dst_o = int(bt[b, p // block_size]), p % block_size
            copies.append((b, s, src_b, src_o, dst_b, dst_o))
    # 3. every provisional block goes back on the stack, rows ascending
    for b in range(B):
        for k in range(P):
            if pb[b, k] >= 0:
                fs[top] = pb[b, k]
                top += 1
                pb[b, k] = -1
    # 4. new logical lengths: prefix + n + 1
    sl = sl + na + 1
    return dict(block_table=bt, seq_lens=sl, prov_blocks=pb, free_stack=fs, free_top=top,
                copies=copies, err=0)


def pool_invariant_ok(block_table, prov_blocks, free_stack, free_top: int, num_blocks: int) -> bool:
    """No leak, no double free (sglang_spec_decode README, provisional layer:
    no block may be leaked or freed twice across all rejection patterns).

    The live holders of a block are the block-table entries, the provisional
    entries and the free-stack entries below free_top; -1 marks an unused
    table or provisional entry, and stack entries at or above free_top are
    dead. The pool is sound when every id 0..num_blocks-1 has exactly one
    live holder and no live entry holds anything else (an id out of range,
    or a negative value other than -1).
    """
    bt = np.asarray(block_table, np.int64).ravel()
    pb = np.asarray(prov_blocks, np.int64).ravel()
    stack = np.asarray(free_stack, np.int64).ravel()
    top = int(free_top)
    if top < 0 or top > stack.size:
        return False
    live = np.concatenate([bt[bt != -1], pb[pb != -1], stack[:top]])
    if np.any((live < 0) | (live >= num_blocks)):
        return False
    holders = np.bincount(live, minlength=num_blocks)
    return bool(np.all(holders == 1))


def kv_truncate_inplace(block_table, seq_lens, num_accepted, free_stack, free_top: int, *,
                        block_size: int, K: int, num_blocks: int, evict: bool = False) -> dict:
    """The in-place variant: provisional slots live in the row's own blocks.

    Source: the lesson's "Rolling back the KV cache" gives, besides the scratch
    buffer, the design that keeps the physical KV cache and truncates a logical
    length; the sglang_spec_decode README adds eviction of a row's provisional
    KV on preemption. Reading used here: before the verify step the caller
    appended the K+1 provisional slots at logical positions L .. L+K of each row
    (blocks allocated as needed). A commit truncates the row to L + n + 1
    (`evict`: back to L) and frees every block that then holds no position
    below the new length: block indices ceil(new/bs) .. ceil((L+K+1)/bs) - 1,
    pushed onto the free stack rows ascending, indices ascending, and set to -1.
    No KV byte moves. All-or-nothing, with the same error bits as kv_commit.
    """
    bt = np.array(block_table, np.int64, copy=True)
    sl = np.array(seq_lens, np.int64, copy=True)
    fs = np.array(free_stack, np.int64, copy=True)
    top = int(free_top)
    B, max_blocks = bt.shape
    na = np.zeros(B, np.int64) if evict else np.asarray(num_accepted, np.int64)
    err = 0
    new_len = np.zeros(B, np.int64)
    frees = []
    for b in range(B):
        n, L = int(na[b]), int(sl[b])
        if not evict and not 0 <= n <= K:
            err |= ERR_BAD_ACCEPT
            continue
        end = _cdiv(L + K + 1, block_size)          # blocks holding prefix + provisional slots
        if L < 0 or end > max_blocks:
            err |= ERR_BAD_LENGTH
            continue
        for j in range(L // block_size, end):
            if not 0 <= int(bt[b, j]) < num_blocks:
                err |= ERR_BAD_BLOCK
        new_len[b] = L if evict else L + n + 1
        frees.append((b, _cdiv(int(new_len[b]), block_size), end))
    n_push = sum(e - s for _, s, e in frees)
    if err == 0 and (top < 0 or top + n_push > num_blocks):
        err |= ERR_BAD_BLOCK                        # the pushes would overflow the stack
    if err:
        return dict(block_table=np.asarray(block_table, np.int64).copy(),
                    seq_lens=np.asarray(seq_lens, np.int64).copy(),
                    free_stack=np.asarray(free_stack, np.int64).copy(), free_top=int(free_top),
                    err=err)
    for b, s, e in frees:
        for j in range(s, e):
            fs[top] = bt[b, j]
            top += 1
            bt[b, j] = -1
    return dict(block_table=bt, seq_lens=new_len, free_stack=fs, free_top=top, err=0)
