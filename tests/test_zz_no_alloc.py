"""spec_verify_greedy_noalloc: the allocation-free greedy entry point (collected last).

Some callers cannot give the library a device allocation of their own: code
whose device memory belongs to another framework's pool, or plain C callers
with no device allocator at hand. For them spec_verify_greedy_noalloc runs the
same greedy kernel on the library's built-in 4 MiB device scratch. Its
outputs must equal those of the workspace entry point exactly (greedy
verification is integer work) and the fp64 oracle's, on two calls in a row
(the scratch keeps the previous call's contents, so nothing may carry over),
and a step too large for the built-in scratch is refused on the host.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _run(sv, torch, case, noalloc):
    dev = "cuda"
    tgt = torch.from_numpy(case.target.view(np.int16)).to(dev).view(torch.bfloat16)
    tok = torch.from_numpy(case.tokens.astype(np.int32)).to(dev)
    B, K = case.tokens.shape
    out = torch.full((B, K + 1), -7, dtype=torch.int32, device=dev)
    n = torch.full((B,), -7, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if noalloc:
        sv.spec_verify_greedy_noalloc(tgt, tok, out, n, err_flag=err)
    else:
        sv.spec_verify_greedy(tgt, tok, out, n, err_flag=err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), n.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("B,K,alpha", [(8, 4, 0.8), (64, 8, 0.95), (256, 4, 0.5)])
def test_noalloc_matches_workspace_entry_point_and_oracle(B, K, alpha):
    torch = pytest.importorskip("torch")
    sv = gh.gpu_lib()
    case = synth.greedy_case(B, K, 151936, alpha=alpha, seed=7000 + B + K)
    orc = oracle.verify_greedy(case.target_values(), case.tokens)
    ref = _run(sv, torch, case, noalloc=False)
    first = _run(sv, torch, case, noalloc=True)
    second = _run(sv, torch, case, noalloc=True)
    for got in (first, second):
        assert np.array_equal(got[0], ref[0])
        assert np.array_equal(got[1], ref[1])
        assert got[2] == ref[2] == 0
        assert np.array_equal(got[0], orc["out_tokens"])
        assert np.array_equal(got[1], orc["num_accepted"])
    assert (ref[1] >= 0).all()


def test_noalloc_refuses_oversize_step():
    pytest.importorskip("torch")
    sv = gh.gpu_lib()
    cap = sv.spec_verify_greedy_noalloc_max_bytes()
    assert cap == 4 << 20
    B, K, V = 16384, 31, 151936
    assert sv.spec_verify_workspace_bytes(B, K, V, sv.SPEC_BF16) > cap
    st = sv.lib().spec_verify_greedy_noalloc(1 << 20, 1 << 20, B, K, V, 1 << 20, 1 << 20, None,
                                             sv.SPEC_BF16, None)
    assert st == sv.SPEC_ENOTSUP
