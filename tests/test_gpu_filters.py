"""GPU parity of spec_filter_thresholds against the filter oracle.

A threshold is one of the row's logit values (or -inf / +inf), so the GPU and
the oracle must agree exactly: bf16 and fp32 rows, several vocabulary sizes,
heavy ties, top-k alone, top-p alone and both, the edge values of k and p,
NaN and all -inf rows, top-p values placed on a cumulative-mass boundary (the
fp32 pass cannot certify them and the double-float pass decides), and sampled
rows of the full-size batch.
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


def _run(sv, stored, dtype, T, k, p):
    import torch
    x = gh.to_dev_logits(stored, dtype)
    R = int(np.prod(stored.shape[:-1]))
    out = torch.full((R,), 12345.0, dtype=torch.float32, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    sv.spec_filter_thresholds(x, T, k, p, out, err_flag=err)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), int(err.item())


def _oracle(values, T, k, p):
    flat = values.reshape(-1, values.shape[-1])
    return np.array([oracle.filter_threshold(r, T, k, p) for r in flat])


def _rows(R, V, dtype, seed, std=3.0, round_to=None):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, std, (R, V)).astype(np.float32)
    if round_to is not None:
        z = np.round(z / round_to) * round_to
    stored = synth.f32_to_bf16_bits(z) if dtype == synth.BF16 else z
    return stored, synth.logits_values(stored, dtype).astype(np.float64)


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
@pytest.mark.parametrize("V", [64, 1000, 4104])
def test_parity_grid(sv, dtype, V):
    stored, vals = _rows(12, V, dtype, seed=V)
    for T in (0.6, 1.0, 2.0):
        for k, p in ((0, 0.9), (20, 1.0), (20, 0.5), (1, 0.3), (V - 1, 0.99), (5, 0.05)):
            g, err = _run(sv, stored, dtype, T, k, p)
            o = _oracle(vals, T, k, float(np.float32(p)))
            assert err == 0
            assert np.array_equal(g, o), (T, k, p, g[g != o][:4], o[g != o][:4])


def test_heavy_ties(sv):
    stored, vals = _rows(16, 2048, synth.BF16, seed=5, std=2.0, round_to=0.5)
    for k, p in ((3, 1.0), (100, 1.0), (0, 0.7), (50, 0.8)):
        g, _ = _run(sv, stored, synth.BF16, 1.0, k, p)
        assert np.array_equal(g, _oracle(vals, 1.0, k, float(np.float32(p))))


def test_edges(sv):
    stored, vals = _rows(4, 512, synth.F32, seed=9)
    vals = vals.copy()
    stored = stored.copy()
    stored[1, :] = -np.inf
    stored[2, 7] = np.nan
    stored[3, :300] = -np.inf
    vals = stored.astype(np.float64)
    for k, p in ((0, 1.0), (512, 1.0), (600, 1.0), (10, 0.5), (0, 0.2)):
        g, err = _run(sv, stored, synth.F32, 1.0, k, p)
        assert g[2] == np.inf and err == sv.SPEC_DERR_LOGITS
        for r in (0, 1, 3):
            assert g[r] == oracle.filter_threshold(vals[r], 1.0, k, float(np.float32(p))), (r, k, p)


def test_bf16_edges(sv):
    """bf16 rows through the two-pass top-k kernel and its fallback: a NaN
    row, an all -inf row, a mostly -inf row, a maximum of zero with both
    signed zeros present, a +inf maximum (top-k only), and k beyond the 256
    keys below the maximum (the general kernel takes the row)."""
    rng = np.random.default_rng(13)
    V = 1024
    z = rng.normal(0, 2, (6, V)).astype(np.float32)
    z[1, :] = -np.inf
    z[2, :1000] = -np.inf
    z[3] = -np.abs(z[3])
    z[3, 5] = 0.0
    z[3, 9] = -0.0
    z[4, 17] = np.inf
    stored = synth.f32_to_bf16_bits(z)
    stored[0, 33] = 0x7FC0                     # NaN
    vals = synth.logits_values(stored, synth.BF16).astype(np.float64)
    for k, p in ((1, 1.0), (7, 1.0), (30, 0.6), (900, 1.0), (1000, 0.9)):
        g, err = _run(sv, stored, synth.BF16, 1.0, k, p)
        assert g[0] == np.inf and err & sv.SPEC_DERR_LOGITS
        rows = (1, 2, 3, 5) if p < 1.0 else (1, 2, 3, 4, 5)
        for r in rows:
            assert g[r] == oracle.filter_threshold(vals[r], 1.0, k, float(np.float32(p))), (r, k, p)
    g, _ = _run(sv, stored[3:4], synth.BF16, 1.0, 2, 1.0)
    assert g[0] == 0.0                         # both zeros kept


def test_boundary_p_uses_the_accurate_pass(sv):
    """p set to the cumulative mass of a prefix (rounded to float32): the
    comparison with p lies within the fp32 pass's error bound, so the
    double-float pass must take it, and agree with the oracle."""
    stored, vals = _rows(8, 3000, synth.BF16, seed=21)
    T = 1.0
    for r in range(8):
        z = vals[r]
        zs = np.sort(z)[::-1]
        w = np.exp((zs - zs[0]) / T)
        cs = np.cumsum(w)
        for i in (3, 40, 400):
            # end of the tie group at position i
            j = i
            while j + 1 < zs.size and zs[j + 1] == zs[i]:
                j += 1
            p = float(np.float32(cs[j] / cs[-1]))
            g, _ = _run(sv, stored[r:r + 1], synth.BF16, T, 0, p)
            assert g[0] == oracle.filter_threshold(z, T, 0, p), (r, i, p)


@pytest.mark.parametrize("shift,T", [(20000.0, 0.5), (1.5e5, 1.0)])
def test_large_offsets(sv, shift, T):
    """fp32 rows shifted by a constant (the distributions do not change), row
    offsets up to 2^17.7 (the range ends at 2^18): p on cumulative-mass
    boundaries forces the double-float pass, which keeps its bound."""
    stored, vals = _rows(4, 3000, synth.F32, seed=31)
    stored = (stored + np.float32(shift)).astype(np.float32)
    vals = stored.astype(np.float64)
    for r in range(4):
        z = vals[r]
        zs = np.sort(z)[::-1]
        cs = np.cumsum(np.exp((zs - zs[0]) / float(np.float32(T))))
        for i in (5, 200):
            j = i
            while j + 1 < zs.size and zs[j + 1] == zs[i]:
                j += 1
            p = float(np.float32(cs[j] / cs[-1]))
            g, err = _run(sv, stored[r:r + 1], synth.F32, T, 0, p)
            assert err == 0
            assert g[0] == oracle.filter_threshold(z, T, 0, p), (r, i, p)
    g, _ = _run(sv, stored, synth.F32, T, 40, 0.9)
    assert np.array_equal(g, _oracle(vals, T, 40, float(np.float32(0.9))))


def test_top_p_offset_beyond_range(sv):
    """With top-p, a maximum logit whose offset reaches 2^18 is out of range:
    +inf and SPEC_DERR_LOGITS. Top-k alone needs no exponentials."""
    stored, vals = _rows(2, 256, synth.F32, seed=2)
    stored = (stored + np.float32(2.0e5)).astype(np.float32)
    g, err = _run(sv, stored, synth.F32, 1.0, 0, 0.9)
    assert (g == np.inf).all() and err == sv.SPEC_DERR_LOGITS
    g, err = _run(sv, stored, synth.F32, 1.0, 10, 1.0)
    assert err == 0
    assert np.array_equal(g, _oracle(stored.astype(np.float64), 1.0, 10, 1.0))


def test_input_validation(sv):
    import torch
    x = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((2,), dtype=torch.float32, device="cuda")
    for T, k, p in ((0.0, 1, 0.5), (1.0, -1, 0.5), (1.0, 1, 0.0), (1.0, 1, 1.5)):
        with pytest.raises(sv.SpecError) as e:
            sv.spec_filter_thresholds(x, T, k, p, out)
        assert e.value.status == sv.SPEC_EINVAL
    bad = torch.zeros((2, 60), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_filter_thresholds(bad, 1.0, 5, 0.9, out)
    assert e.value.status == sv.SPEC_ENOTSUP


def test_full_size_sampled_rows(sv):
    """The bench batch's shape: B = 256 rows of K + 1 = 5 target rows,
    V = 151936 bf16 (1280 rows); 24 sampled rows against the oracle."""
    c = synth.sampling_case(256, 4, 151936, temperature=1.0, target_std=3.0,
                            draft_noise_std=0.5, seed=3)
    vals = c.target_values().reshape(-1, c.V)
    rng = np.random.default_rng(0)
    pick = rng.choice(vals.shape[0], 24, replace=False)
    for k, p in ((50, 0.95), (0, 0.9), (1000, 1.0)):
        g, err = _run(sv, c.target, c.dtype, 1.0, k, p)
        assert err == 0
        for r in pick:
            assert g[r] == oracle.filter_threshold(vals[r], 1.0, k, float(np.float32(p))), (r, k, p)
