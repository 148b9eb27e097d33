"""Failure detection on the GPU: a wait that runs out (-m gpu).

Every wait of the verification kernels is bounded; when one gives up the
launch aborts, drains and reports SPEC_DERR_TIMEOUT through the error word,
and the context stays usable. To make a wait run out without faulting
anything, the library's test knob SPECVERIFY_STALL_ROW withholds every stage
arrival of one batch row (a flag that nothing sets): that row never
completes, the producers' idle wait (shortened with SPECVERIFY_IDLE_NS) runs
out, and the launch returns. The stalled row's outputs stay unwritten; every
other row is finished and matches the oracle; the next launch without the
knob is normal.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

STALL = 3
IDLE_NS = "5000000"  # 5 ms


@pytest.fixture(scope="module")
def sv():
    return gh.gpu_lib()


def test_sampling_wait_runs_out(sv, monkeypatch):
    c = synth.sampling_case(8, 4, 4096, temperature=1.0, target_std=3.0, draft_noise_std=0.5,
                            seed=31)
    o = oracle.verify_sample(c.target_values(), c.draft_values(), c.tokens, c.uniforms, 1.0)
    monkeypatch.setenv("SPECVERIFY_STALL_ROW", str(STALL))
    monkeypatch.setenv("SPECVERIFY_IDLE_NS", IDLE_NS)
    g = gh.run_sample(sv, c)
    assert g["err"] & sv.SPEC_DERR_TIMEOUT
    assert g["num_accepted"][STALL] == -7 and (g["out_tokens"][STALL] == -7).all()
    rest = np.array([b for b in range(c.B) if b != STALL])
    assert (g["num_accepted"][rest] >= 0).all()
    assert np.array_equal(g["out_tokens"][rest], o["out_tokens"][rest])
    assert np.array_equal(g["num_accepted"][rest], o["num_accepted"][rest])
    monkeypatch.delenv("SPECVERIFY_STALL_ROW")
    monkeypatch.delenv("SPECVERIFY_IDLE_NS")
    again = gh.run_sample(sv, c)
    assert again["err"] == 0
    gh.assert_sample_parity(again, o)


def test_greedy_wait_runs_out(sv, monkeypatch):
    c = synth.greedy_case(8, 4, 4096, alpha=0.8, seed=32)
    o = oracle.verify_greedy(c.target_values(), c.tokens)
    monkeypatch.setenv("SPECVERIFY_STALL_ROW", str(STALL))
    monkeypatch.setenv("SPECVERIFY_IDLE_NS", IDLE_NS)
    g = gh.run_greedy(sv, c)
    assert g["err"] & sv.SPEC_DERR_TIMEOUT
    assert g["num_accepted"][STALL] == -7 and (g["out_tokens"][STALL] == -7).all()
    rest = np.array([b for b in range(c.B) if b != STALL])
    assert np.array_equal(g["out_tokens"][rest], o["out_tokens"][rest])
    assert np.array_equal(g["num_accepted"][rest], o["num_accepted"][rest])
    monkeypatch.delenv("SPECVERIFY_STALL_ROW")
    monkeypatch.delenv("SPECVERIFY_IDLE_NS")
    again = gh.run_greedy(sv, c)
    assert again["err"] == 0
    assert np.array_equal(again["out_tokens"], o["out_tokens"])
