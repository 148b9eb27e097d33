"""The bench's byte accounting (CPU): algorithmic bytes of a verify launch, the
secondary 'sequential' figure, greedy bytes and KV bytes, on hand-counted
batches."""
import numpy as np

import bench

V, E = 1000, 2


def test_sampling_bytes_hand_count():
    K = 3
    na = np.array([0, 3, 1])                      # rejected at 0, all accepted, rejected at 1
    meta = 3 * (4 * K + 4 * (K + 1) + 4 * (K + 1) + 4)
    # every row streams its 2K rows; only the fully accepted row adds row K
    assert bench.algorithmic_verify_bytes(na, K, V) == 3 * 2 * K * V * E + 1 * V * E + meta
    # positions up to the first rejection: 2 rows, 2K + 1 rows, 4 rows
    assert bench.sequential_verify_bytes(na, K, V) == (2 + 7 + 4) * V * E + meta


def test_sequential_never_exceeds_algorithmic():
    rng = np.random.default_rng(0)
    for K in (1, 4, 8):
        na = rng.integers(0, K + 1, size=64)
        assert bench.sequential_verify_bytes(na, K, V) <= bench.algorithmic_verify_bytes(na, K, V)
    na = np.full(16, 4)                           # all accepted: both figures agree
    assert bench.sequential_verify_bytes(na, 4, V) == bench.algorithmic_verify_bytes(na, 4, V)


def test_greedy_and_kv_bytes():
    K = 4
    na = np.array([4, 0, 2])
    assert bench.greedy_verify_bytes(na, K, V) == (3 * K + 1) * V * E + 3 * (4 * K + 4 * (K + 1) + 4)
    w = dict(kv_layers=32, kv_heads=8, head_dim=128)
    slot = 32 * 2 * 8 * 128 * 2                   # one token's K and V over all layers, bf16
    assert bench.kv_bytes(na, w) == (5 + 1 + 3) * slot * 2


def test_job_rate_counts_every_rank():
    assert bench.job_rate(4, 256, 4, 0.5) == 4 * bench.job_rate(1, 256, 4, 0.5)


def test_profiling_options(monkeypatch):
    """The small-footprint options the committed ncu summaries were taken with:
    short KV prefixes are named in the workload string, and the filter-only
    mode and the no-extras switch parse."""
    import sys
    monkeypatch.setattr(sys, "argv", ["bench.py", "--kv-prefix", "16,64", "--no-extras", "--steps", "3"])
    a = bench.parse()
    assert a.kv_prefix == "16,64" and a.no_extras and a.mode == "step"
    assert "prefix U[16, 64]" in bench.workload_name(1.0, (16, 64))
    assert "prefix U[512, 4096]" in bench.workload_name(1.0)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--mode", "filter"])
    assert bench.parse().mode == "filter"

