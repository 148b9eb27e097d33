"""Pins of the top-k / top-p filter oracle (CPU only).

The oracle takes the k-th largest logit for top-k and, for top-p, the first
position of the descending sort whose cumulative mass reaches p. The pins
check it against hand-worked rows, a brute force that tries every logit of the row
as a candidate threshold, the defining properties of the kept set, the
limits of the parameters, and the losslessness of verification on the
filtered distributions (the emitted token follows the filtered target).
"""
import numpy as np
import pytest

import oracle
from oracle import filters as of


def test_top_k_hand_rows():
    z = [1.0, 3.0, 3.0, 2.0]
    assert oracle.filter_threshold(z, 1.0, top_k=1) == 3.0   # both tied maxima kept
    assert oracle.filter_threshold(z, 1.0, top_k=2) == 3.0
    assert oracle.filter_threshold(z, 1.0, top_k=3) == 2.0
    assert oracle.filter_threshold(z, 1.0, top_k=4) == -np.inf  # k >= V: no filter
    assert oracle.filter_threshold(z, 1.0, top_k=0) == -np.inf


def test_top_p_hand_rows():
    probs = np.array([0.5, 0.25, 0.125, 0.125])
    z = np.log(probs)
    assert oracle.filter_threshold(z, 1.0, top_p=0.4) == z[0]
    assert oracle.filter_threshold(z, 1.0, top_p=0.6) == z[1]
    assert oracle.filter_threshold(z, 1.0, top_p=0.8) == z[2]    # both 0.125 tokens kept
    assert oracle.filter_threshold(z, 1.0, top_p=1.0) == -np.inf
    # top-p on the renormalised top-k distribution: top-2 leaves (2/3, 1/3)
    assert oracle.filter_threshold(z, 1.0, top_k=2, top_p=0.6) == z[0]
    assert oracle.filter_threshold(z, 1.0, top_k=2, top_p=0.7) == z[1]


def _brute(z, T, k, p):
    """Every logit as a candidate threshold; the largest that qualifies."""
    z = np.asarray(z, np.float64)
    tk = -np.inf
    if 0 < k < z.size:
        tk = max(t for t in z if np.count_nonzero(z >= t) >= k)
    if p >= 1.0:
        return tk
    kept = z[z >= tk]
    w = np.exp((kept - kept.max()) / float(np.float32(T)))
    Z = w.sum()
    tp = max(t for t in kept if w[kept >= t].sum() >= p * Z)
    return max(tk, tp)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force(seed):
    rng = np.random.default_rng(seed)
    V = 40
    z = np.round(rng.normal(0, 2, V), 1)        # rounded: many ties
    for T in (0.5, 1.0, 1.7):
        for k in (0, 1, 3, 17, 39, 40):
            for p in (0.05, 0.5, 0.9, 0.999, 1.0):
                assert oracle.filter_threshold(z, T, k, p) == _brute(z, T, k, p), (T, k, p)


@pytest.mark.parametrize("seed", range(4))
def test_kept_set_properties(seed):
    rng = np.random.default_rng(100 + seed)
    z = rng.normal(0, 3, 500)
    T = 0.8
    for p in (0.3, 0.9, 0.99):
        t = oracle.filter_threshold(z, T, top_p=p)
        w = np.exp((z - z.max()) / float(np.float32(T)))
        kept = w[z >= t].sum() / w.sum()
        assert kept >= p
        smaller = z[z >= t].min()
        above = w[z > smaller].sum() / w.sum()
        assert above < p              # the smallest kept value is needed
    for k in (1, 10, 250):
        t = oracle.filter_threshold(z, T, top_k=k)
        assert np.count_nonzero(z >= t) >= k
        assert np.count_nonzero(z > t) < k


def test_parameter_limits():
    rng = np.random.default_rng(3)
    z = rng.normal(0, 2, 200)
    assert oracle.filter_threshold(z, 1.0, top_p=1e-9) == z.max()
    assert oracle.filter_threshold(z, 1.0, top_k=1) == z.max()
    # top-k does not depend on the temperature; top-p keeps more at higher T
    assert oracle.filter_threshold(z, 0.3, top_k=20) == oracle.filter_threshold(z, 3.0, top_k=20)
    kept = [np.count_nonzero(z >= oracle.filter_threshold(z, T, top_p=0.9)) for T in (0.3, 1, 3)]
    assert kept[0] <= kept[1] <= kept[2]
    # -inf logits: never above a finite threshold, and ignored by top-p
    zi = z.copy()
    zi[:50] = -np.inf
    t = oracle.filter_threshold(zi, 1.0, top_p=0.5)
    assert np.isfinite(t) and t == _brute(zi[50:], 1.0, 0, 0.5)
    with pytest.raises(ValueError):
        oracle.filter_threshold([0.0, np.nan], 1.0, top_k=1)


def test_apply_threshold():
    z = np.array([[1.0, 3.0, 3.0, 2.0]])
    out = oracle.apply_threshold(z, [3.0])
    assert out.tolist() == [[-np.inf, 3.0, 3.0, -np.inf]]


def test_filtered_verification_is_lossless():
    """Drafts drawn from the filtered draft row, verified against the
    filtered target row: the emitted first token follows the filtered
    target distribution (total variation within sampling noise)."""
    rng = np.random.default_rng(11)
    V, T, k, p = 7, 0.9, 5, 0.8
    zt = rng.normal(0, 1.5, (1, 2, V))
    zd = zt[:, :1] + rng.normal(0, 0.7, (1, 1, V))
    tt = of.filter_thresholds(zt, T, k, p)
    td = of.filter_thresholds(zd, T, k, p)
    ft = of.apply_threshold(zt, tt)
    fd = of.apply_threshold(zd, td)
    q0 = oracle.softmax(ft[0, 0], float(np.float32(T)))
    p0 = oracle.softmax(fd[0, 0], float(np.float32(T)))
    n = 40000
    toks = rng.choice(V, size=n, p=p0)
    u = rng.random((n, 2))
    counts = np.zeros(V)
    B = 2000
    for b0 in range(0, n, B):
        nb = min(B, n - b0)
        r = oracle.verify_sample(np.repeat(ft, nb, 0), np.repeat(fd, nb, 0),
                                 toks[b0:b0 + nb, None], u[b0:b0 + nb], T)
        np.add.at(counts, r["out_tokens"][:, 0], 1)
    tv = 0.5 * np.abs(counts / n - q0).sum()
    assert tv < 0.012, tv
    assert counts[q0 == 0].sum() == 0        # filtered-out target tokens never emitted
