"""kv_commit_inplace / kv_evict_provisional against the oracle (exact)."""
import numpy as np
import pytest

import oracle
from gpu_helpers import gpu_lib
from test_oracle_kv_inplace import _state

pytestmark = pytest.mark.gpu


def _dev(torch, x):
    return torch.from_numpy(np.ascontiguousarray(x, np.int32)).cuda()


def _run(sv, torch, bt, L, n, fs, top, *, bs, K, nb, evict=False):
    d_bt, d_sl, d_fs = _dev(torch, bt), _dev(torch, L), _dev(torch, fs)
    d_top, d_st = _dev(torch, [top]), _dev(torch, [-7])
    if evict:
        sv.kv_evict_provisional(d_bt, d_sl, d_fs, d_top, d_st, K=K, block_size=bs, num_blocks=nb)
    else:
        sv.kv_commit_inplace(d_bt, d_sl, _dev(torch, n), d_fs, d_top, d_st, K=K, block_size=bs,
                             num_blocks=nb)
    torch.cuda.synchronize()
    return dict(block_table=d_bt.cpu().numpy(), seq_lens=d_sl.cpu().numpy(),
                free_stack=d_fs.cpu().numpy(), free_top=int(d_top.item()),
                status=int(d_st.item()))


def _same(got, want):
    assert got["status"] == want["err"]
    assert np.array_equal(got["block_table"], want["block_table"])
    assert np.array_equal(got["seq_lens"], want["seq_lens"])
    assert got["free_top"] == want["free_top"]
    assert np.array_equal(got["free_stack"], want["free_stack"])


@pytest.mark.parametrize("bs,K", [(1, 3), (4, 4), (16, 7), (16, 0)])
def test_commit_and_evict_match_oracle(bs, K):
    import torch
    sv = gpu_lib()
    rng = np.random.default_rng(31 * bs + K)
    B, mb = 2000, 64
    nb = B * mb + 1000  # room for every prefix and its provisional blocks
    L, bt, fs, top, _ = _state(rng, B, K, bs, nb, mb)
    n = np.arange(B) % (K + 1)  # every acceptance pattern
    kw = dict(block_size=bs, K=K, num_blocks=nb)
    _same(_run(sv, torch, bt, L, n, fs, top, bs=bs, K=K, nb=nb),
          oracle.kv_truncate_inplace(bt, L, n, fs, top, **kw))
    _same(_run(sv, torch, bt, L, None, fs, top, bs=bs, K=K, nb=nb, evict=True),
          oracle.kv_truncate_inplace(bt, L, None, fs, top, evict=True, **kw))


def test_errors_leave_state_unchanged():
    import torch
    sv = gpu_lib()
    rng = np.random.default_rng(5)
    B, K, bs, nb, mb = 64, 3, 4, 2000, 20
    L, bt, fs, top, _ = _state(rng, B, K, bs, nb, mb)
    n = rng.integers(0, K + 1, size=B)
    bad_n = n.copy(); bad_n[9] = -1
    bad_bt = bt.copy(); bad_bt[4, int(L[4]) // bs] = -1
    cases = [(bt, L, bad_n, top), (bad_bt, L, n, top), (bt, L, n, nb)]
    for c_bt, c_L, c_n, c_top in cases:
        want = oracle.kv_truncate_inplace(c_bt, c_L, c_n, fs, c_top, block_size=bs, K=K,
                                          num_blocks=nb)
        assert want["err"] != 0
        _same(_run(sv, torch, c_bt, c_L, c_n, fs, c_top, bs=bs, K=K, nb=nb), want)
