"""GPU parity of spec_verify_sample / spec_verify_greedy against the fp64 oracle.

Inputs are the seeded synthetic workloads of `synth` (shapes and distributions
of the pages' workloads). Greedy tokens and accepted lengths are compared bit
for bit; sampled tokens must equal the oracle's except where the uniform lies
within 1e-5 of the decision boundary in the oracle's fp64 arithmetic, and such
rows must stay below 1e-4 of the draws; the probabilities of the draft tokens
must agree within 1e-5.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return gh.gpu_lib()


def oracle_sample(case, rows=None):
    t = case.target_values()
    d = case.draft_values()
    tok, u = case.tokens, case.uniforms
    if rows is not None:
        t, d, tok, u = t[rows], d[rows], tok[rows], u[rows]
    return oracle.verify_sample(t, d, tok, u, case.temperature)


def oracle_greedy(case, rows=None):
    t = case.target_values()
    tok = case.tokens
    if rows is not None:
        t, tok = t[rows], tok[rows]
    return oracle.verify_greedy(t, tok)


# ------------------------------------------------------------------ hardware exp2 bound
@pytest.mark.parametrize("lo,hi", [(-126.0, 1.0), (1.0, 127.0)])
def test_ex2_error_bound_holds(sv, lo, hi):
    """The fp32 certification assumes the max rel. error of ex2.approx over the
    arguments it meets stays below kEx2RelErrBound: [-126, 1] for normalised
    terms, up to 100 for the raw bonus draw's guessed offset. Measure every
    fp32 argument of [-126, 127] exhaustively on this GPU."""
    worst = sv.spec_selftest_ex2(lo, hi)
    bound = gh.ex2_bound_constant()
    print(f"ex2.approx max relative error on [{lo}, {hi}]: {worst:.4e} (bound {bound:.1e})")
    assert 0.0 < worst < bound


# ------------------------------------------------------------------ hand examples
def _pad_probs(rows, Vp):
    out = np.full((len(rows), Vp), -np.inf)
    for i, r in enumerate(rows):
        out[i, :len(r)] = np.log(np.asarray(r, np.float64))
    return out


@pytest.mark.parametrize("T", [1.0, 0.5, 2.0])
def test_hand_sample_cases(sv, golden, T):
    import torch
    for case in golden["sample_cases"]:
        V = len(case["q"][0])
        Vp = -(-V // 4) * 4  # fp32 rows must be a multiple of 16 bytes: pad with -inf
        zt = (T * _pad_probs(case["q"], Vp)).astype(np.float32)[None]
        zd = (T * _pad_probs(case["p"], Vp)).astype(np.float32)[None]
        c = synth.VerifyCase(zt, zd, np.asarray([case["draft_tokens"]], np.int32),
                             np.asarray([case["uniforms"]], np.float32), T, synth.F32)
        g = gh.run_sample(sv, c)
        assert g["out_tokens"][0].tolist() == case["out_tokens"], (case["name"], g)
        assert g["num_accepted"][0] == case["num_accepted"]
        assert g["err"] == 0


def test_hand_greedy_cases(sv, golden):
    for case in golden["greedy_cases"]:
        zt = np.asarray(case["target_logits"], np.float32)[None]
        c = synth.VerifyCase(zt, None, np.asarray([case["draft_tokens"]], np.int32),
                             np.zeros((1, zt.shape[1]), np.float32), 0.0, synth.F32)
        g = gh.run_greedy(sv, c)
        assert g["out_tokens"][0].tolist() == case["out_tokens"], case["name"]
        assert g["num_accepted"][0] == case["num_accepted"]
        # T == 0 through the sampling entry point is greedy
        s = gh.run_sample(sv, c, temperature=0.0)
        assert s["out_tokens"][0].tolist() == case["out_tokens"]


# ------------------------------------------------------------------ greedy workloads
@pytest.mark.parametrize("B", [1, 8])
@pytest.mark.parametrize("K", [2, 4, 6, 8])
def test_greedy_parity_config(sv, B, K):
    """Greedy mode, V = 151936 bf16 logits ~ N(0, 3^2), planted acceptance alpha."""
    for alpha in (0.5, 0.8, 0.95):
        c = synth.greedy_case(B, K, 151936, alpha=alpha, seed=100 * K + B + int(alpha * 100))
        g = gh.run_greedy(sv, c)
        o = oracle_greedy(c)
        assert np.array_equal(g["num_accepted"], o["num_accepted"])
        assert np.array_equal(g["out_tokens"], o["out_tokens"])
        assert g["err"] == 0


@pytest.mark.parametrize("B", [1, 8])
@pytest.mark.parametrize("K", [2, 4, 6, 8])
def test_greedy_parity_unaltered_rows(sv, B, K):
    """Greedy mode on unaltered N(0, 3^2) bf16 rows of V = 151936 (nothing
    clipped or planted), where the largest values of a row often round to the
    same bf16 value. Draft token i is the oracle's own argmax of row i with
    probability alpha (input generation), else a uniform other id. On top of
    the natural ties, every other target row gets a copy of its maximum half a
    row away, below or above the first maximum, so that a tie between two
    vocabulary slices occurs in every batch (any slicing into two or more
    slices separates positions V/2 apart); the lowest index must win."""
    V = 151936
    for alpha in (0.5, 0.8, 0.95):
        seed = 500 + 100 * K + B + int(alpha * 100)
        tgt = synth.normal_target(B, K, V, seed=seed)
        z = synth.logits_values(tgt, synth.BF16)
        rng = np.random.default_rng(seed)
        g0 = oracle.verify_greedy(z, np.zeros((B, K), np.int64))["argmax"]
        planted = 0
        for b in range(B):
            for i in range(K + 1):
                if (b * (K + 1) + i) % 2 == 0:
                    at = (int(g0[b, i]) + V // 2) % V
                    tgt[b, i, at] = tgt[b, i, g0[b, i]]
                    planted += 1
        z = synth.logits_values(tgt, synth.BF16)
        g = oracle.verify_greedy(z, np.zeros((B, K), np.int64))["argmax"]
        other = (g[:, :K] + 1 + rng.integers(0, V - 1, size=(B, K))) % V
        tok = np.where(rng.random((B, K)) < alpha, g[:, :K], other).astype(np.int32)
        c = synth.VerifyCase(tgt, None, tok, np.zeros((B, K + 1), np.float32), 0.0, synth.BF16)
        gg = gh.run_greedy(sv, c)
        o = oracle.verify_greedy(z, tok)
        assert np.array_equal(gg["num_accepted"], o["num_accepted"]), alpha
        assert np.array_equal(gg["out_tokens"], o["out_tokens"]), alpha
        assert gg["err"] == 0
        # the ties are there: rows whose maximum occurs at least twice
        ties = sum(int(np.count_nonzero(z[b, i] == z[b, i].max()) >= 2)
                   for b in range(B) for i in range(K + 1))
        assert ties >= planted >= 1


@pytest.mark.parametrize("alpha", [0.5, 0.8, 0.95])
@pytest.mark.parametrize("K", [2, 4, 6, 8])
def test_greedy_planted_alpha_mean(sv, alpha, K):
    """2000 steps per cell: the mean accepted count matches (1 - a^(K+1)) / (1 - a),
    and every output equals the planted argmax decode."""
    import torch
    steps, B, V = 250, 8, 151936
    gen = torch.Generator(device="cuda").manual_seed(K * 1000 + int(alpha * 100))
    total = []
    for s in range(steps):
        z = torch.clamp(torch.randn((B, K + 1, V), device="cuda", generator=gen) * 3.0,
                        -synth.CLIP, synth.CLIP)
        g = torch.randint(0, V, (B, K + 1), device="cuda", generator=gen)
        z.scatter_(2, g[..., None], synth.PLANT_VALUE)
        hit = torch.rand((B, K), device="cuda", generator=gen) < alpha
        other = (g[:, :K] + 1 + torch.randint(0, V - 1, (B, K), device="cuda", generator=gen)) % V
        tok = torch.where(hit, g[:, :K], other).to(torch.int32).contiguous()
        zt = z.to(torch.bfloat16).contiguous()
        out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
        n = torch.empty((B,), dtype=torch.int32, device="cuda")
        sv.spec_verify_greedy(zt, tok, out, n)
        # expected: the planted decode
        gg, tt = g.cpu().numpy(), tok.cpu().numpy()
        nn = n.cpu().numpy()
        oo = out.cpu().numpy()
        for b in range(B):
            m = 0
            while m < K and tt[b, m] == gg[b, m]:
                m += 1
            assert nn[b] == m
            assert oo[b, : m + 1].tolist() == gg[b, : m + 1].tolist()
        total.append(nn + 1)
    m = np.concatenate(total).astype(np.float64)
    closed = (1 - alpha ** (K + 1)) / (1 - alpha)
    pmf = np.array([alpha ** k * (1 - alpha) for k in range(K)] + [alpha ** K])
    var = (pmf * (np.arange(K + 1) + 1.0) ** 2).sum() - closed ** 2
    z = (m.mean() - closed) / math.sqrt(var / m.size)
    assert abs(z) < 4, (m.mean(), closed, z)


# ------------------------------------------------------------------ sampling workloads
def test_sample_pr1_thousand_steps(sv):
    """B=1, K=4, V=32000 fp32, T=1.0: 1000 independent steps."""
    stats = dict(mism=0, refined=0, window=0)
    for step in range(1000):
        c = synth.pr1_case(step)
        g = gh.run_sample(sv, c)
        o = oracle_sample(c)
        r = gh.compare_sample(g, o)
        assert r["outside"] == [], (step, r)
        assert r["max_dq"] <= gh.PROB_TOL and r["max_dp"] <= gh.PROB_TOL, (step, r)
        stats["mism"] += r["mismatches"]
        stats["window"] += r["window_draws"]
        stats["refined"] += int(g["row_info"][0] != 0)
        assert g["err"] == 0
    print("PR1:", stats)
    assert stats["mism"] <= gh.MAX_RATE * 1000


@pytest.mark.parametrize("sigma", [0.25, 1.0])
def test_sample_config_b64_k7(sv, sigma):
    """B=64, K=7, V=151936 bf16, T=0.6, draft = target + N(0, sigma^2), Philox seed 1."""
    c = synth.sampling_case(64, 7, 151936, temperature=0.6, target_std=3.0,
                            draft_noise_std=sigma, seed=31 + int(sigma * 4), uniform_seed=1)
    g = gh.run_sample(sv, c)
    o = oracle_sample(c)
    r = gh.assert_sample_parity(g, o, label=f"sigma={sigma}")
    print(f"B64 K7 sigma={sigma}:", r, "refined rows:", int(np.sum(g["row_info"] != 0)))
    assert g["err"] == 0


def test_sample_config_b256_k4_v128256(sv):
    """B=256, K=4, V=128256 bf16, T=1.0, sigma=0.5 (the verify half of the KV workload)."""
    c = synth.sampling_case(256, 4, 128256, temperature=1.0, target_std=3.0,
                            draft_noise_std=0.5, seed=404, uniform_seed=4)
    g = gh.run_sample(sv, c)
    o = oracle_sample(c)
    r = gh.assert_sample_parity(g, o, label="b256")
    print("B256 K4 V128256:", r, "refined rows:", int(np.sum(g["row_info"] != 0)))


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_sample_full_size_sampled_rows(sv, T):
    """B=256, K=4, V=151936 bf16 (the benchmark workload), all rows on the GPU,
    48 rows re-derived by the oracle."""
    c = synth.sampling_case(256, 4, 151936, temperature=T, target_std=3.0, draft_noise_std=0.5,
                            seed=77, uniform_seed=5)
    g = gh.run_sample(sv, c)
    rows = np.random.default_rng(0).choice(256, size=48, replace=False)
    o = oracle_sample(c, rows)
    r = gh.assert_sample_parity(g, o, rows=rows, label=f"full T={T}")
    assert (g["num_accepted"] >= 0).all() and g["err"] == 0
    print(f"full size T={T}:", r, "refined rows:", int(np.sum(g["row_info"] != 0)))


@pytest.mark.parametrize("B,K,T", [(1024, 8, 1.0), (1, 8, 0.6), (8, 2, 1.0)])
def test_sweep_extremes(sv, B, K, T):
    """Corners of the B x K grid of the sweep at V = 151936 bf16: the largest
    batch (5.3 GB of logits; 24 rows re-derived by the oracle) and single or
    few rows (all rows), greedy on the same inputs."""
    c = synth.sampling_case(B, K, 151936, temperature=T, target_std=3.0, draft_noise_std=0.5,
                            seed=B + 10 * K, uniform_seed=3)
    dev = gh.dev_case(c)
    g = gh.run_sample(sv, c, dev)
    gg = gh.run_greedy(sv, c, dev)
    del dev
    rows = np.sort(np.random.default_rng(1).choice(B, size=min(B, 24), replace=False))
    t = synth.logits_values(c.target[rows], c.dtype).astype(np.float64)
    d = synth.logits_values(c.draft[rows], c.dtype).astype(np.float64)
    o = oracle.verify_sample(t, d, c.tokens[rows], c.uniforms[rows], c.temperature)
    r = gh.assert_sample_parity(g, o, rows=rows, label=f"B={B} K={K}")
    assert (g["num_accepted"] >= 0).all() and g["err"] == 0
    og = oracle.verify_greedy(t, c.tokens[rows])
    assert np.array_equal(gg["out_tokens"][rows], og["out_tokens"])
    print(f"B={B} K={K} T={T}:", r)


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("B,K,V,dtype", [
    (3, 1, 64, synth.BF16),          # K = 1
    (2, 31, 256, synth.F32),         # K = 31 (maximum), tiny V
    (5, 3, 8, synth.BF16),           # V = one 16-byte vector: one slice per row
    (4, 5, 32008, synth.BF16),       # ragged V: slices of unequal length
    (3, 4, 1000, synth.F32),         # fp32, V not a multiple of the slice split
    (7, 2, 4, synth.F32),            # V = 4
])
def test_sample_shapes(sv, B, K, V, dtype):
    c = synth.sampling_case(B, K, V, temperature=0.9, target_std=2.0, draft_noise_std=0.8,
                            dtype=dtype, seed=B * 7 + K * 13 + V)
    g = gh.run_sample(sv, c)
    gh.assert_sample_parity(g, oracle_sample(c), label=str((B, K, V, dtype)))
    og = oracle_greedy(c)
    gg = gh.run_greedy(sv, c)
    assert np.array_equal(gg["out_tokens"], og["out_tokens"])


@pytest.mark.parametrize("grid", ["1", "3", "37", "151"])
def test_grid_sizes_agree(sv, monkeypatch, grid):
    """The persistent grid capped at fewer CTAs (one CTA runs every task of
    the launch) gives the same rows: no task depends on which or how many
    CTAs run it."""
    monkeypatch.setenv("SPECVERIFY_GRID", grid)
    c = synth.sampling_case(6, 3, 20000, temperature=0.7, target_std=3.0, draft_noise_std=0.5,
                            seed=5)
    g = gh.run_sample(sv, c)
    gh.assert_sample_parity(g, oracle_sample(c), label=grid)
    gg = gh.run_greedy(sv, c)
    assert np.array_equal(gg["out_tokens"], oracle_greedy(c)["out_tokens"])


@pytest.mark.parametrize("shift,T", [(0.0, 0.05), (20000.0, 0.5), (1.5e5, 1.0), (-1.5e5, 1.0)])
def test_large_exponent_offsets(sv, shift, T):
    """Rows whose offset max * log2(e)/T is large in magnitude (a low
    temperature, or fp32 logits shifted by a constant, which leaves every
    distribution unchanged; up to 2^17.7 here, the range ends at 2^18): the
    double-float refinements keep their bound, parity with the oracle."""
    c = synth.sampling_case(32, 4, 20000, temperature=T, target_std=3.0, draft_noise_std=0.5,
                            dtype=synth.F32, seed=int(abs(shift)) % 997 + 11)
    c.target = (c.target + np.float32(shift)).astype(np.float32)
    c.draft = (c.draft + np.float32(shift)).astype(np.float32)
    g = gh.run_sample(sv, c)
    o = oracle_sample(c)
    gh.assert_sample_parity(g, o, label=f"shift={shift} T={T}")
    assert g["err"] == 0
    print(f"shift={shift} T={T}: refined rows", int(np.sum(g["row_info"] != 0)))


def test_offset_beyond_range_is_a_logits_error(sv):
    """max * log2(e)/T at or beyond 2^18 in magnitude: the exponent offset is
    out of range, every row reports SPEC_DERR_LOGITS with outputs -1."""
    c = synth.sampling_case(4, 3, 512, temperature=1.0, target_std=2.0, draft_noise_std=0.5,
                            dtype=synth.F32, seed=4)
    c.target = (c.target + np.float32(2.0e5)).astype(np.float32)
    c.draft = (c.draft + np.float32(2.0e5)).astype(np.float32)
    g = gh.run_sample(sv, c)
    assert g["err"] & sv.SPEC_DERR_LOGITS
    assert (g["num_accepted"] == -1).all() and (g["out_tokens"] == -1).all()


@pytest.mark.parametrize("shift", [-1000.0, -30.0, 40.0, 110.0, 300.0])
def test_bonus_row_offset_guess(sv, shift):
    """Every draft accepted (draft rows = target rows), target row K shifted
    against rows 0..K-1: the bonus draw's offset, guessed from rows 0..K-1, is
    then far too high (-1000: every term flushed, the statistics stage takes
    the row), somewhat high (-30), low (+40: terms up to 2^58, still drawn
    raw), too low for the raw draw (+110: totals above 2^100 go to the
    statistics stage) or far too low (+300: the sums overflow, the statistics
    stage takes the row). The draws match the oracle in every case."""
    c = synth.sampling_case(16, 4, 4096, temperature=1.0, target_std=3.0, draft_noise_std=0.0,
                            dtype=synth.F32, seed=17)
    t = c.target.copy()
    t[:, 4, :] += np.float32(shift)
    c.target = t
    c.draft = t[:, :4].copy()
    g = gh.run_sample(sv, c)
    o = oracle_sample(c)
    assert (o["num_accepted"] == 4).all()
    gh.assert_sample_parity(g, o, label=f"shift={shift}")
    assert g["err"] == 0


def test_bonus_row_nan(sv):
    """A NaN in target row K of a row that accepts every draft: the raw bonus
    draw's total is NaN, the statistics stage takes the row and reports it."""
    import speculative_decoding_verification_sample_gb300 as m
    c = synth.sampling_case(6, 4, 4096, temperature=1.0, target_std=3.0, draft_noise_std=0.0,
                            dtype=synth.F32, seed=23)
    t = c.target.copy()
    t[2, 4, 100] = np.nan
    c.target = t
    c.draft = t[:, :4].copy()
    g = gh.run_sample(sv, c)
    assert g["num_accepted"][2] == -1 and (g["out_tokens"][2] == -1).all()
    assert g["err"] & m.SPEC_DERR_LOGITS
    good = np.array([0, 1, 3, 4, 5])
    gh.assert_sample_parity(g, oracle_sample(c, good), rows=good)


def test_identical_draft_accepts_everything(sv):
    c = synth.sampling_case(8, 4, 4096, temperature=1.0, target_std=3.0, draft_noise_std=0.0,
                            seed=3)
    c.draft = c.target[:, :4].copy()
    g = gh.run_sample(sv, c)
    o = oracle_sample(c)
    assert (o["num_accepted"] == 4).all()
    gh.assert_sample_parity(g, o)


def test_masked_logits(sv):
    """-inf logits: probability 0. A draft token the draft model gives p = 0 is
    accepted; a token the target gives q = 0 is rejected."""
    c = synth.sampling_case(4, 3, 512, temperature=1.0, target_std=2.0, draft_noise_std=0.5,
                            dtype=synth.F32, seed=8)
    t, d = c.target.copy(), c.draft.copy()
    t[:, :, 100:200] = -np.inf
    d[:, :, 300:400] = -np.inf
    c.tokens[0, 0] = 350           # p = 0 -> accepted
    c.tokens[1, 0] = 150           # q = 0 -> rejected
    c.target, c.draft = t, d
    g = gh.run_sample(sv, c)
    o = oracle_sample(c)
    assert o["num_accepted"][1] == 0 and o["num_accepted"][0] >= 1
    gh.assert_sample_parity(g, o)


def test_bad_token_and_nan_rows(sv):
    import speculative_decoding_verification_sample_gb300 as m
    c = synth.sampling_case(4, 3, 512, temperature=1.0, target_std=2.0, draft_noise_std=0.5,
                            dtype=synth.F32, seed=9)
    c.tokens[1, 2] = 512            # out of range
    t = c.target.copy()
    t[2, 0, 17] = np.nan            # NaN in a row every step needs
    c.target = t
    g = gh.run_sample(sv, c)
    assert g["num_accepted"][1] == -1 and (g["out_tokens"][1] == -1).all()
    assert g["num_accepted"][2] == -1 and (g["out_tokens"][2] == -1).all()
    assert g["err"] & m.SPEC_DERR_TOKEN and g["err"] & m.SPEC_DERR_LOGITS
    good = [0, 3]
    o = oracle_sample(c, good)
    gh.assert_sample_parity(dict((k, v) for k, v in g.items()), o, rows=np.array(good))


def test_host_validation(sv):
    import torch
    import speculative_decoding_verification_sample_gb300 as m
    c = synth.sampling_case(2, 2, 64, temperature=1.0, target_std=1.0, draft_noise_std=0.5,
                            seed=1)
    dv = gh.dev_case(c)
    out = torch.empty((2, 3), dtype=torch.int32, device="cuda")
    n = torch.empty((2,), dtype=torch.int32, device="cuda")
    for T in (-1.0, float("nan"), float("inf")):
        with pytest.raises(m.SpecError) as e:
            m.spec_verify_sample(dv["target"], dv["draft"], dv["tokens"], dv["uniforms"], T, out, n)
        assert e.value.status == m.SPEC_EINVAL
    # V * 2 bytes not a multiple of 16
    bad = torch.zeros((2, 3, 63), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.SpecError) as e:
        m.spec_verify_greedy(bad, dv["tokens"], out, n)
    assert e.value.status == m.SPEC_ENOTSUP
    # misaligned base
    buf = torch.zeros((2 * 3 * 64 + 1,), dtype=torch.bfloat16, device="cuda")
    mis = buf[1:].view(2, 3, 64)
    ws = m.workspace_for(2, 2, 64, m.SPEC_BF16, "cuda")
    st = m.lib().spec_verify_greedy(mis.data_ptr(), dv["tokens"].data_ptr(), 2, 2, 64,
                                    out.data_ptr(), n.data_ptr(), None, m.SPEC_BF16, None,
                                    ws.data_ptr(), ws.numel(), None)
    assert st == m.SPEC_EINVAL
    # workspace too small
    import ctypes
    st = m.lib().spec_verify_greedy(dv["target"].data_ptr(), dv["tokens"].data_ptr(), 2, 2, 64,
                                    out.data_ptr(), n.data_ptr(), None, m.SPEC_BF16, None,
                                    ws.data_ptr(), ctypes.c_size_t(16), None)
    assert st == m.SPEC_EINVAL


def test_deterministic(sv):
    c = synth.sampling_case(32, 4, 50000, temperature=0.8, target_std=3.0, draft_noise_std=0.5,
                            seed=12)
    dv = gh.dev_case(c)
    a = gh.run_sample(sv, c, dv)
    b = gh.run_sample(sv, c, dv)
    for k in ("out_tokens", "num_accepted", "row_info", "q_at_d", "p_at_d"):
        assert np.array_equal(a[k], b[k]), k
