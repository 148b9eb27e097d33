"""Fused acceptance counters of the verify kernels against the oracle.

Both verify calls accumulate, per draft position, how many rows tested and
accepted it, plus rows and tokens emitted. The counts are integers, so the
comparison with oracle.acceptance_counters (computed from the oracle's own
accepted lengths on the same inputs) is exact; two calls in a row must
double them (the counters accumulate).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import dev_case, gpu_lib

pytestmark = pytest.mark.gpu


def _counters(torch, K):
    return torch.zeros(2 * K + 2, dtype=torch.int64, device="cuda")


@pytest.mark.parametrize("B,K,V,T,dtype", [(16, 4, 32000, 1.0, synth.F32),
                                           (32, 7, 151936, 0.6, synth.BF16)])
def test_sample_counters(B, K, V, T, dtype):
    import torch
    sv = gpu_lib()
    c = synth.sampling_case(B, K, V, temperature=T, target_std=3.0, draft_noise_std=0.5,
                            dtype=dtype, seed=900 + K, uniform_seed=901 + K)
    ref = oracle.verify_step(c.target_values(), c.draft_values(), c.tokens, c.uniforms, T)
    want = oracle.acceptance_counters(ref["num_accepted"], K)
    d = dev_case(c)
    cnt = _counters(torch, K)
    out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((B,), dtype=torch.int32, device="cuda")
    for rep in (1, 2):
        sv.spec_verify_sample(d["target"], d["draft"], d["tokens"], d["uniforms"], T, out, n,
                              accept_counters=cnt)
        torch.cuda.synchronize()
        assert np.array_equal(n.cpu().numpy(), ref["num_accepted"])
        assert np.array_equal(cnt.cpu().numpy(), rep * want)


def test_greedy_counters_and_temperature_zero():
    import torch
    sv = gpu_lib()
    B, K = 8, 6
    c = synth.greedy_case(B, K, 151936, alpha=0.8, seed=77)
    ref = oracle.verify_greedy(c.target_values(), c.tokens)
    want = oracle.acceptance_counters(ref["num_accepted"], K)
    d = dev_case(c)
    out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((B,), dtype=torch.int32, device="cuda")
    cnt = _counters(torch, K)
    sv.spec_verify_greedy(d["target"], d["tokens"], out, n, accept_counters=cnt)
    torch.cuda.synchronize()
    assert np.array_equal(cnt.cpu().numpy(), want)
    # T = 0 through the sampling entry point takes the greedy path, counters included
    cnt0 = _counters(torch, K)
    sv.spec_verify_sample(d["target"], None, d["tokens"], None, 0.0, out, n, accept_counters=cnt0)
    torch.cuda.synchronize()
    assert np.array_equal(cnt0.cpu().numpy(), want)


def test_counters_skip_error_rows():
    import torch
    sv = gpu_lib()
    B, K = 4, 3
    c = synth.greedy_case(B, K, 4096, alpha=0.95, seed=5)
    tokens = c.tokens.copy()
    tokens[1, 0] = 4096  # out of range: row 1 is an error row
    d = dev_case(c)
    d["tokens"] = torch.from_numpy(tokens.astype(np.int32)).cuda()
    out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((B,), dtype=torch.int32, device="cuda")
    cnt = _counters(torch, K)
    sv.spec_verify_greedy(d["target"], d["tokens"], out, n, accept_counters=cnt)
    torch.cuda.synchronize()
    got_n = n.cpu().numpy()
    assert got_n[1] == -1
    assert np.array_equal(cnt.cpu().numpy(), oracle.acceptance_counters(got_n, K))
    assert cnt[2 * K].item() == B - 1
