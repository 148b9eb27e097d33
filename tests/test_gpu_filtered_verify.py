"""GPU parity of sampling verification on top-k / top-p filtered rows.

The GPU path: spec_filter_thresholds on the target and draft tensors, then
spec_verify_sample with those thresholds. The oracle path: the oracle's own
thresholds, the logits below them set to -inf, then the oracle verification.
Draft tokens come from the unfiltered draft model, so some of them fall
outside the filtered draft support (p(d) = 0: accepted) or outside the
filtered target support (q(d) = 0: rejected); both are exercised.
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


def _thresholds(sv, dev_logits, T, k, p):
    import torch
    shp = dev_logits.shape[:-1]
    out = torch.empty(shp, dtype=torch.float32, device="cuda")
    sv.spec_filter_thresholds(dev_logits, T, k, p, out)
    return out


def _check(sv, c, k, p, rows=None):
    import torch
    T = c.temperature
    dev = gh.dev_case(c)
    tt = _thresholds(sv, dev["target"], T, k, p)
    td = _thresholds(sv, dev["draft"], T, k, p)
    g = gh.run_sample(sv, c, dev, target_threshold=tt, draft_threshold=td)
    torch.cuda.synchronize()
    pf = float(np.float32(p))
    sel = np.arange(c.B) if rows is None else np.asarray(rows)
    zt = c.target_values()[sel].astype(np.float64)
    zd = c.draft_values()[sel].astype(np.float64)
    ot = oracle.filter_thresholds(zt, T, k, pf)
    od = oracle.filter_thresholds(zd, T, k, pf)
    assert np.array_equal(tt.cpu().numpy()[sel], ot) and np.array_equal(td.cpu().numpy()[sel], od)
    o = oracle.verify_sample(oracle.apply_threshold(zt, ot), oracle.apply_threshold(zd, od),
                             c.tokens[sel], c.uniforms[sel], T)
    r = gh.assert_sample_parity(g, o, rows=None if rows is None else sel, label=f"k={k} p={p}")
    assert g["err"] == 0
    return g, o, r


@pytest.mark.parametrize("k,p", [(20, 1.0), (0, 0.9), (50, 0.8), (5, 0.5), (1, 1.0)])
@pytest.mark.parametrize("T", [0.7, 1.0])
def test_filtered_parity(sv, k, p, T):
    c = synth.sampling_case(48, 4, 4096, temperature=T, target_std=3.0, draft_noise_std=0.8,
                            seed=k * 10 + int(p * 10) + int(T * 100))
    g, o, _ = _check(sv, c, k, p)
    assert np.array_equal(g["num_accepted"], o["num_accepted"])


def test_filtering_changes_the_outcome(sv):
    """A narrow filter must change acceptance compared with no filter."""
    c = synth.sampling_case(64, 4, 2048, temperature=1.0, target_std=2.0, draft_noise_std=1.0,
                            seed=77)
    g0 = gh.run_sample(sv, c)
    g1, _, _ = _check(sv, c, 3, 1.0)
    assert not np.array_equal(g0["num_accepted"], g1["num_accepted"])


def test_full_size_sampled_rows(sv):
    c = synth.sampling_case(256, 4, 151936, temperature=1.0, target_std=3.0, draft_noise_std=0.5,
                            seed=8)
    rows = np.random.default_rng(1).choice(256, 12, replace=False)
    _check(sv, c, 50, 0.95, rows=rows)
