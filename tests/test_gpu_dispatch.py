"""The small-batch dispatch forced both ways (-m gpu).

Batches of at most 16 rows take a different work split (one first-stage task
per persistent CTA, per-position first-stage tasks for one row) and, from 4
rows, start residual draws with the accurate refinement pass instead of the
fp32 sweep. The test knob SPECVERIFY_SMALL_BATCH forces those choices off (0)
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
                                     (16, 2, 151936, 1.0)])
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


@pytest.mark.parametrize("B,K", [(1, 4), (8, 4), (24, 2)])
def test_greedy_both_dispatches(sv, monkeypatch, B, K):
    c = synth.greedy_case(B, K, 151936, alpha=0.8, seed=800 + 10 * B + K)
    o = oracle.verify_greedy(c.target_values(), c.tokens)
    dev = gh.dev_case(c)
    res = _runs(sv, monkeypatch, lambda: gh.run_greedy(sv, c, dev))
    for knob, g in res.items():
        assert g["err"] == 0, knob
        assert np.array_equal(g["num_accepted"], o["num_accepted"]), knob
        assert np.array_equal(g["out_tokens"], o["out_tokens"]), knob
