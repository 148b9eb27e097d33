"""The small-batch dispatch forced both ways (-m gpu).

Sampling batches of at most 48 rows (greedy: 64) take a different work
split (one first-stage task per persistent CTA, per-position first-stage
tasks for one row) and, from 4 rows, start residual draws with the accurate
refinement pass instead of the fp32 sweep. The test knob SPECVERIFY_SMALL_BATCH forces those choices off (0)
or on (1) whatever the batch size. Every case here runs three times on the
same inputs (default, off, on): each run must match the oracle, and the three
runs must agree exactly, since every decision is certified (a row flagged
SPEC_ROW_UNCERTIFIED would be exempt; none occurs).
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


def _runs(sv, monkeypatch, run):
    res = {}
    for knob in (None, "0", "1"):
        if knob is None:
            monkeypatch.delenv("SPECVERIFY_SMALL_BATCH", raising=False)
        else:
            monkeypatch.setenv("SPECVERIFY_SMALL_BATCH", knob)
        res[knob] = run()
    monkeypatch.delenv("SPECVERIFY_SMALL_BATCH", raising=False)
    return res


@pytest.mark.parametrize("B,K,V,T", [(1, 4, 32000, 1.0), (3, 4, 32000, 1.0), (8, 4, 32000, 1.0),
                                     (8, 8, 151936, 0.6), (24, 4, 32000, 1.0),
                                     (16, 2, 151936, 1.0), (40, 4, 32000, 1.0),
                                     (64, 4, 32000, 0.6)])
def test_sampling_both_dispatches(sv, monkeypatch, B, K, V, T):
    c = synth.sampling_case(B, K, V, temperature=T, target_std=3.0, draft_noise_std=0.5,
                            seed=700 + 10 * B + K)
    o = oracle.verify_sample(c.target_values(), c.draft_values(), c.tokens, c.uniforms, T)
    dev = gh.dev_case(c)
    res = _runs(sv, monkeypatch, lambda: gh.run_sample(sv, c, dev))
    for knob, g in res.items():
        assert g["err"] == 0, knob
        assert not (g["row_info"] & sv.SPEC_ROW_UNCERTIFIED).any(), knob
        gh.assert_sample_parity(g, o, label=f"B={B} K={K} V={V} T={T} knob={knob}")
    for knob in ("0", "1"):
        assert np.array_equal(res[knob]["out_tokens"], res[None]["out_tokens"]), knob
        assert np.array_equal(res[knob]["num_accepted"], res[None]["num_accepted"]), knob


@pytest.mark.parametrize("B,K", [(1, 4), (8, 4), (24, 2), (48, 4), (96, 4)])
def test_greedy_both_dispatches(sv, monkeypatch, B, K):
    c = synth.greedy_case(B, K, 151936, alpha=0.8, seed=800 + 10 * B + K)
    o = oracle.verify_greedy(c.target_values(), c.tokens)
    dev = gh.dev_case(c)
    res = _runs(sv, monkeypatch, lambda: gh.run_greedy(sv, c, dev))
    for knob, g in res.items():
        assert g["err"] == 0, knob
        assert np.array_equal(g["num_accepted"], o["num_accepted"]), knob
        assert np.array_equal(g["out_tokens"], o["out_tokens"]), knob


@pytest.mark.parametrize("B,K,V,T,k,p", [(1, 4, 4096, 1.0, 50, 0.9), (8, 4, 4096, 0.7, 20, 1.0),
                                         (8, 4, 32000, 1.0, 0, 0.8)])
def test_filtered_both_dispatches(sv, monkeypatch, B, K, V, T, k, p):
    """Top-k / top-p thresholds (tokens below a row's threshold are -inf in
    every stage) on small batches, whose first stage runs per position (B = 1)
    and whose residual draws start at the refinement pass (B = 8)."""
    import torch
    c = synth.sampling_case(B, K, V, temperature=T, target_std=3.0, draft_noise_std=0.8,
                            seed=900 + 10 * B + k)
    dev = gh.dev_case(c)
    tt = torch.empty((B, K + 1), dtype=torch.float32, device="cuda")
    td = torch.empty((B, K), dtype=torch.float32, device="cuda")
    sv.spec_filter_thresholds(dev["target"], T, k, p, tt)
    sv.spec_filter_thresholds(dev["draft"], T, k, p, td)
    torch.cuda.synchronize()
    pf = float(np.float32(p))
    zt = c.target_values().astype(np.float64)
    zd = c.draft_values().astype(np.float64)
    ot, od = oracle.filter_thresholds(zt, T, k, pf), oracle.filter_thresholds(zd, T, k, pf)
    assert np.array_equal(tt.cpu().numpy(), ot) and np.array_equal(td.cpu().numpy(), od)
    o = oracle.verify_sample(oracle.apply_threshold(zt, ot), oracle.apply_threshold(zd, od),
                             c.tokens, c.uniforms, T)
    res = _runs(sv, monkeypatch,
                lambda: gh.run_sample(sv, c, dev, target_threshold=tt, draft_threshold=td))
    for knob, g in res.items():
        assert g["err"] == 0, knob
        gh.assert_sample_parity(g, o, label=f"filtered B={B} k={k} p={p} knob={knob}")
    for knob in ("0", "1"):
        assert np.array_equal(res[knob]["out_tokens"], res[None]["out_tokens"]), knob
