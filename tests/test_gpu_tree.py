"""GPU parity of spec_verify_tree_greedy and of the slot-mapped KV commit.

Every output (kept tokens, accepted count, KV slots) is integer work and must
equal the oracle exactly, row by row: hand-worked trees, the [2, 2, 2] tree of
the lesson's exercise, random topologies up to 31 nodes with and without
duplicate siblings, several vocabulary sizes (several ring stages per row and
a ragged tail), bf16 and float32, the full-size batch, the error rows, and a
tree commit of the KV pool through kv_commit_rollback's slot map.
"""
import json
import pathlib

import numpy as np
import pytest

import oracle
import synth
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

GOLDEN = pathlib.Path(__file__).parent / "golden" / "tree_examples.json"


@pytest.fixture(scope="module")
def sv():
    return gh.gpu_lib()


def _run(sv, target, parents, tokens, dtype, slots=True):
    import torch
    B, N1, V = target.shape
    dt = gh.to_dev_logits(target, dtype)
    par = torch.from_numpy(np.ascontiguousarray(parents, np.int32)).cuda()
    tok = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).cuda()
    out = torch.full((B, N1), -7, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    sl = torch.full((B, N1), -7, dtype=torch.int32, device="cuda") if slots else None
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    sv.spec_verify_tree_greedy(dt, par, tok, out, n, out_slots=sl, err_flag=err)
    torch.cuda.synchronize()
    return dict(out_tokens=out.cpu().numpy(), num_accepted=n.cpu().numpy(),
                slots=None if sl is None else sl.cpu().numpy(), err=int(err.item()))


def _oracle(case: synth.TreeCase, rows_per_call: int = 16):
    z = case.target_values()
    outs = [oracle.verify_tree_greedy(z[b0:b0 + rows_per_call], case.parents[b0:b0 + rows_per_call],
                                      case.tokens[b0:b0 + rows_per_call])
            for b0 in range(0, case.B, rows_per_call)]
    return {k: np.concatenate([o[k] for o in outs]) for k in ("out_tokens", "num_accepted", "slots")}


def _same(g, o):
    assert np.array_equal(g["num_accepted"], o["num_accepted"])
    assert np.array_equal(g["out_tokens"], o["out_tokens"])
    if g["slots"] is not None:
        assert np.array_equal(g["slots"], o["slots"])


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_hand_cases(sv, dtype):
    fx = json.loads(GOLDEN.read_text())
    V = fx["V"]
    for case in fx["cases"]:
        z = np.zeros((1, len(case["row_argmax"]), V), np.float32)
        for r, gmax in enumerate(case["row_argmax"]):
            z[0, r, gmax] = 1.0
        for r, v in case.get("extra_max", ()):
            z[0, r, v] = 1.0
        stored = synth.f32_to_bf16_bits(z) if dtype == synth.BF16 else z
        g = _run(sv, stored, [case["parents"]], [case["tokens"]], dtype)
        assert g["out_tokens"][0].tolist() == case["out_tokens"], case["name"]
        assert int(g["num_accepted"][0]) == case["num_accepted"], case["name"]
        assert g["slots"][0].tolist() == case["slots"], case["name"]
        assert g["err"] == 0


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
@pytest.mark.parametrize("V", [8, 1000, 4096 + 8, 70000])
def test_exercise_tree_parity(sv, V, dtype):
    c = synth.tree_case(24, V, branching=(2, 2, 2), alpha=0.8, dtype=dtype, seed=V)
    g = _run(sv, c.target, c.parents, c.tokens, dtype)
    _same(g, _oracle(c))
    assert g["err"] == 0


@pytest.mark.parametrize("distinct", [True, False])
@pytest.mark.parametrize("N", [1, 5, 17, 31])
def test_random_topology_parity(sv, N, distinct):
    c = synth.tree_case(40, 3000, N=N, alpha=0.85, distinct=distinct, seed=N * 7 + distinct)
    g = _run(sv, c.target, c.parents, c.tokens, c.dtype)
    _same(g, _oracle(c))
    assert g["err"] == 0


def test_random_logits_without_planting(sv):
    """Unplanted N(0, 1) logits in bf16: exact ties inside a row are common,
    so the lowest-index rule decides; trees whose tokens copy some row's
    argmax get accepted often enough to reach depth."""
    rng = np.random.default_rng(5)
    B, V = 64, 2048
    par = np.tile(synth.tree_parents((3, 2, 2)), (B, 1))
    N = par.shape[1]
    z = rng.normal(0, 1, size=(B, N + 1, V)).astype(np.float32)
    stored = synth.f32_to_bf16_bits(z)
    zv = synth.bf16_bits_to_f32(stored)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    # half the nodes copy a maximum (possibly one of several tied) of their parent's row
    for b in range(B):
        for i in range(N):
            if rng.random() < 0.5:
                row = zv[b, par[b, i] + 1]
                tok[b, i] = int(rng.choice(np.flatnonzero(row == row.max())))
    g = _run(sv, stored, par, tok, synth.BF16)
    o = oracle.verify_tree_greedy(zv, par, tok)
    _same(g, o)


def test_chain_tree_equals_linear_greedy(sv):
    import torch
    c = synth.greedy_case(48, 6, 5000, alpha=0.8, seed=3)
    chain = np.tile(np.arange(-1, c.K - 1, dtype=np.int32), (c.B, 1))
    g = _run(sv, c.target, chain, c.tokens, c.dtype)
    d = gh.dev_case(c)
    out = torch.full((c.B, c.K + 1), -7, dtype=torch.int32, device="cuda")
    n = torch.full((c.B,), -7, dtype=torch.int32, device="cuda")
    sv.spec_verify_greedy(d["target"], d["tokens"], out, n)
    torch.cuda.synchronize()
    assert np.array_equal(g["out_tokens"], out.cpu().numpy())
    assert np.array_equal(g["num_accepted"], n.cpu().numpy())


def test_without_slots_output(sv):
    c = synth.tree_case(8, 512, branching=(2, 2), seed=2)
    g = _run(sv, c.target, c.parents, c.tokens, c.dtype, slots=False)
    o = _oracle(c)
    assert np.array_equal(g["out_tokens"], o["out_tokens"])
    assert np.array_equal(g["num_accepted"], o["num_accepted"])


def test_error_rows(sv):
    c = synth.tree_case(6, 1024, branching=(2, 2), alpha=1.0, dtype=synth.F32, seed=11)
    par, tok = c.parents.copy(), c.tokens.copy()
    z = c.target.copy()
    par[1, 3] = 3                          # a node as its own parent
    tok[2, 0] = 1024                       # token out of range
    z[3, 0, 17] = np.nan                   # NaN in row 0
    # row 4: NaN in the row of a node that does not survive (no error)
    o_clean = oracle.verify_tree_greedy(c.target_values(), c.parents, c.tokens)
    dead = [i for i in range(c.N) if i not in set(o_clean["slots"][4, 1:] - 1)]
    z[4, 1 + dead[0], 5] = np.nan
    # row 5: NaN in the row of the deepest kept node
    n5 = int(o_clean["num_accepted"][5])
    assert n5 >= 1
    z[5, int(o_clean["slots"][5, n5]), 9] = np.nan
    g = _run(sv, z, par, tok, synth.F32)
    o = oracle.verify_tree_greedy(z, par, tok)
    _same(g, o)
    assert g["num_accepted"].tolist()[1:4] == [-1, -1, -1] and g["num_accepted"][5] == -1
    assert g["num_accepted"][4] >= 0 and g["num_accepted"][0] >= 0
    assert g["err"] == (sv.SPEC_DERR_TOKEN | sv.SPEC_DERR_LOGITS)


def test_host_validation(sv):
    import torch
    c = synth.tree_case(2, 64, branching=(2,), seed=0)
    d = gh.to_dev_logits(c.target, c.dtype)
    par = torch.from_numpy(c.parents).cuda()
    tok = torch.from_numpy(c.tokens).cuda()
    out = torch.zeros((2, 3), dtype=torch.int32, device="cuda")
    n = torch.zeros((2,), dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        bad = torch.zeros((2, 3, 60), dtype=torch.bfloat16, device="cuda")  # 120-byte rows
        sv.spec_verify_tree_greedy(bad, par, tok, out, n)
    assert e.value.status == sv.SPEC_ENOTSUP
    big = synth.tree_case(1, 64, N=32, seed=0)
    with pytest.raises(sv.SpecError) as e:
        sv.spec_verify_tree_greedy(gh.to_dev_logits(big.target, big.dtype),
                                   torch.from_numpy(big.parents).cuda(),
                                   torch.from_numpy(big.tokens).cuda(),
                                   torch.zeros((1, 33), dtype=torch.int32, device="cuda"),
                                   torch.zeros((1,), dtype=torch.int32, device="cuda"))
    assert e.value.status == sv.SPEC_EINVAL


def test_full_size_exercise_tree(sv):
    """B = 256, V = 151936 bf16, the [2, 2, 2] tree (15 target rows per batch
    row): every row against the oracle."""
    c = synth.tree_case(256, 151936, branching=(2, 2, 2), alpha=0.8, seed=99)
    g = _run(sv, c.target, c.parents, c.tokens, c.dtype)
    _same(g, _oracle(c))
    assert g["err"] == 0
    assert g["num_accepted"].max() == 3


# ----------------------------------------------------------- tree KV commit
def test_tree_kv_commit_through_slot_map(sv):
    """Verify a [2, 2, 2] tree, then commit its kept path with the slot map:
    tables and every pool byte against the oracle's copies."""
    import torch
    from tests import test_gpu_kv as tk
    t = synth.tree_case(64, 512, branching=(2, 2, 2), alpha=0.9, seed=21)
    g = _run(sv, t.target, t.parents, t.tokens, t.dtype)
    N = t.N
    c = synth.kv_case(t.B, N, block_size=4, prefix_lo=0, prefix_hi=40,
                      num_accepted=g["num_accepted"], seed=8)
    smap = np.where(g["slots"] < 0, 0, g["slots"]).astype(np.int32)
    pool = tk._small_pool(c, seed=3)
    before = pool.cpu().view(torch.int16).numpy()
    d = tk._dev(c)
    sv.kv_commit_rollback(d["bt"], d["sl"], d["na"], d["pb"], pool, d["fs"], d["ft"], d["st"],
                          K=N, block_size=c.block_size, slot_map=torch.from_numpy(smap).cuda())
    torch.cuda.synchronize()
    o = oracle.kv_commit(c.block_table, c.seq_lens, c.num_accepted, c.prov_blocks, c.free_stack,
                         c.free_top, block_size=c.block_size, K=N, num_blocks=c.num_blocks,
                         slot_map=smap)
    assert o["err"] == 0
    tk._check_tables(c, d, o)
    after = pool.cpu().view(torch.int16).numpy()
    assert np.array_equal(after, tk._expected_pool(before, o["copies"]))
    assert any(s != k for (b, k, sb, so, db, do) in o["copies"]
               for s in [int(smap[b, k])])   # some kept slot is not its position


def test_bad_slot_map_is_rejected_on_device(sv):
    import torch
    from tests import test_gpu_kv as tk
    c = synth.kv_case(4, 6, block_size=4, num_accepted=np.array([6, 2, 0, 3]), seed=4)
    smap = np.tile(np.arange(7, dtype=np.int32), (4, 1))
    smap[3, 2] = 7
    pool = tk._small_pool(c, seed=1)
    before = pool.cpu().view(torch.int16).numpy()
    d = tk._dev(c)
    sv.kv_commit_rollback(d["bt"], d["sl"], d["na"], d["pb"], pool, d["fs"], d["ft"], d["st"],
                          K=6, block_size=4, slot_map=torch.from_numpy(smap).cuda())
    torch.cuda.synchronize()
    o = oracle.kv_commit(c.block_table, c.seq_lens, c.num_accepted, c.prov_blocks, c.free_stack,
                         c.free_top, block_size=4, K=6, num_blocks=c.num_blocks, slot_map=smap)
    assert o["err"] == sv.SPEC_DERR_BAD_SLOT
    tk._check_tables(c, d, o)
    assert np.array_equal(pool.cpu().view(torch.int16).numpy(), before)
