"""GPU check of the host-buffer path (HostVerifier): row chunks copied on a copy
stream and verified as they land must give the same rows as one
spec_verify_sample call on the whole device batch, and match the oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return gh.gpu_lib()


@pytest.mark.parametrize("chunks", [1, 3, 8])
def test_host_verifier_matches_device_call(sv, chunks):
    import torch
    c = synth.sampling_case(40, 4, 4096, temperature=0.9, target_std=3.0, draft_noise_std=0.5,
                            seed=chunks)
    d = gh.dev_case(c)
    ref = gh.run_sample(sv, c, d)
    host = {k: v.cpu().pin_memory() for k, v in d.items()}
    hv = sv.HostVerifier(c.B, c.K, c.V, chunks=chunks)
    out, n = hv(host["target"], host["draft"], host["tokens"], host["uniforms"], c.temperature)
    out_h = torch.empty((c.B, c.K + 1), dtype=torch.int32).pin_memory()
    n_h = torch.empty((c.B,), dtype=torch.int32).pin_memory()
    hv.to_host(out_h, n_h)
    torch.cuda.synchronize()
    assert np.array_equal(out_h.numpy(), ref["out_tokens"])
    assert np.array_equal(n_h.numpy(), ref["num_accepted"])
    o = oracle.verify_sample(c.target_values(), c.draft_values(), c.tokens, c.uniforms,
                             c.temperature)
    assert np.array_equal(n_h.numpy(), o["num_accepted"])
