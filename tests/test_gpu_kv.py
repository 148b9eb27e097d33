"""GPU parity of kv_commit_rollback against the block-table oracle.

Tables (block table, lengths, provisional entries, free stack) must match the
oracle bit for bit; the KV pool after the call must equal the pre-call pool
with exactly the oracle's copies applied (every byte), and the pool invariant
(no block leaked or freed twice) must hold.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return gh.gpu_lib()


def _dev(case):
    import torch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()  # noqa: E731
    return dict(bt=t(case.block_table), sl=t(case.seq_lens), na=t(case.num_accepted),
                pb=t(case.prov_blocks), fs=t(case.free_stack), ft=t([case.free_top]),
                st=t([-99]))


def _run(sv, case, pool, d=None):
    import torch
    d = d or _dev(case)
    sv.kv_commit_rollback(d["bt"], d["sl"], d["na"], d["pb"], pool, d["fs"], d["ft"], d["st"],
                          K=case.K, block_size=case.block_size)
    torch.cuda.synchronize()
    return d


def _oracle(case):
    return oracle.kv_commit(case.block_table, case.seq_lens, case.num_accepted, case.prov_blocks,
                            case.free_stack, case.free_top, block_size=case.block_size, K=case.K,
                            num_blocks=case.num_blocks)


def _check_tables(case, d, o):
    assert int(d["st"].item()) == o["err"]
    assert np.array_equal(d["bt"].cpu().numpy(), o["block_table"])
    assert np.array_equal(d["sl"].cpu().numpy(), o["seq_lens"])
    assert np.array_equal(d["pb"].cpu().numpy(), o["prov_blocks"])
    top = int(d["ft"].item())
    assert top == o["free_top"]
    assert np.array_equal(d["fs"].cpu().numpy()[:top], o["free_stack"][:top])


def _small_pool(case, NL=2, H=2, D=8, seed=0):
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    raw = torch.randint(-32768, 32767, (case.num_blocks, NL, 2, case.block_size, H, D),
                        dtype=torch.int16, device="cuda", generator=g)
    return raw.view(torch.bfloat16)


def _expected_pool(before: np.ndarray, copies):
    exp = before.copy()
    for (b, s, sb, so, db, do) in copies:
        exp[db, :, :, do] = before[sb, :, :, so]
    return exp


@pytest.mark.parametrize("K,bs", [(4, 16), (7, 16), (15, 16), (5, 4), (9, 8), (31, 16)])
def test_every_rejection_pattern(sv, K, bs):
    import itertools
    lens = [bs * 3 - 1, bs * 3, bs * 3 + 1, bs * 4 - K, bs * 4 - K - 1, 0, 1]
    rows = list(itertools.product(lens, range(K + 1)))
    c = synth.kv_case(len(rows), K, block_size=bs, seq_lens=np.array([r[0] for r in rows]),
                      num_accepted=np.array([r[1] for r in rows]), seed=K + bs)
    import torch
    pool = _small_pool(c, seed=K)
    before = pool.cpu().view(torch.int16).numpy()
    d = _run(sv, c, pool)
    o = _oracle(c)
    assert o["err"] == 0
    _check_tables(c, d, o)
    after = pool.cpu().view(torch.int16).numpy()
    assert np.array_equal(after, _expected_pool(before, o["copies"]))
    assert oracle.pool_invariant_ok(d["bt"].cpu().numpy(), d["pb"].cpu().numpy(),
                                    d["fs"].cpu().numpy(), int(d["ft"].item()), c.num_blocks)


@pytest.mark.parametrize("mutate", ["accept_high", "accept_neg", "len_neg", "table_small",
                                    "no_space", "bad_table_block", "bad_prov_block",
                                    "slot_taken", "top_too_big", "bad_free_entry"])
def test_errors_leave_state_unchanged(sv, mutate):
    import torch
    c = synth.kv_case(4, 4, seq_lens=np.array([16, 20, 31, 47]),
                      num_accepted=np.array([1, 2, 4, 0]), seed=4)
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
        c.block_table[3, 2] = c.num_blocks
    elif mutate == "bad_prov_block":
        c.prov_blocks[1, 0] = -1
    elif mutate == "slot_taken":
        c.block_table[0, 1] = c.free_stack[0]
    elif mutate == "top_too_big":
        c.free_top = c.num_blocks + 1
    elif mutate == "bad_free_entry":
        c.free_stack[c.free_top - 1] = -5
    pool = _small_pool(c)
    before = pool.cpu().view(torch.int16).numpy()
    d = _run(sv, c, pool)
    o = _oracle(c)
    assert o["err"] != 0
    _check_tables(c, d, o)
    assert np.array_equal(pool.cpu().view(torch.int16).numpy(), before)


def test_verify_then_commit_full_size(sv):
    """Sampling + KV rollback workload: B=256, K=4, V=128256 bf16, T=1.0, sigma=0.5;
    paged pool of 32 layers x 8 KV heads x head_dim 128 bf16, block 16, prefix
    lengths ~ U[512, 4096]. num_accepted comes from the verify call on the same
    stream; the provisional slots hold random bf16."""
    import torch
    B, K, V = 256, 4, 128256
    vc = synth.sampling_case(B, K, V, temperature=1.0, target_std=3.0, draft_noise_std=0.5,
                             seed=404, uniform_seed=4)
    dv = gh.dev_case(vc)
    out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((B,), dtype=torch.int32, device="cuda")
    sv.spec_verify_sample(dv["target"], dv["draft"], dv["tokens"], dv["uniforms"], 1.0, out, n)
    torch.cuda.synchronize()
    na = n.cpu().numpy()
    assert (na >= 0).all()
    c = synth.kv_case(B, K, block_size=16, prefix_lo=512, prefix_hi=4096, num_accepted=na,
                      seed=44)
    NL, H, D = 32, 8, 128
    pool = torch.empty((c.num_blocks, NL, 2, 16, H, D), dtype=torch.bfloat16, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(1)
    touched = set(int(x) for x in c.prov_blocks.ravel())
    touched |= set(int(c.block_table[b, c.seq_lens[b] // 16]) for b in range(B)
                   if c.seq_lens[b] % 16)
    for blk in sorted(touched):
        pool[blk].view(torch.int16).copy_(torch.randint(-32768, 32767, pool[blk].shape,
                                                        dtype=torch.int16, device="cuda",
                                                        generator=g))
    src = {(b, s): pool[int(c.prov_blocks[b, s // 16]), :, :, s % 16].clone()
           for b in range(B) for s in range(int(na[b]) + 1)}
    tails = {b: pool[int(c.block_table[b, c.seq_lens[b] // 16])].clone()
             for b in range(B) if c.seq_lens[b] % 16}
    # fingerprint of blocks no row touches
    rng = np.random.default_rng(3)
    others = [int(x) for x in rng.choice(c.num_blocks, 64, replace=False) if int(x) not in touched]
    fp_before = {x: pool[x].view(torch.int16).to(torch.int64).sum().item() for x in others}
    d = _run(sv, c, pool, _dev(c))
    o = _oracle(c)
    assert o["err"] == 0
    _check_tables(c, d, o)
    bits = lambda x: x.view(torch.int16)  # noqa: E731  (compare bit patterns: NaN codes too)
    for (b, s, sb, so, db, do) in o["copies"]:
        assert torch.equal(bits(pool[db, :, :, do]), bits(src[(b, s)])), (b, s)
    for b, t in tails.items():
        L = int(c.seq_lens[b])
        blk = int(c.block_table[b, L // 16])
        assert torch.equal(bits(pool[blk, :, :, : L % 16]), bits(t[:, :, : L % 16])), b
    for x, v in fp_before.items():
        if x in set(int(y) for y in o["block_table"].ravel()):
            continue  # newly allocated blocks receive copies
        assert pool[x].view(torch.int16).to(torch.int64).sum().item() == v
    assert oracle.pool_invariant_ok(d["bt"].cpu().numpy(), d["pb"].cpu().numpy(),
                                    d["fs"].cpu().numpy(), int(d["ft"].item()), c.num_blocks)
