"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every
function that include/*.h declares (no compute calls here)."""
import ctypes
import glob
import os
import re

from tests.gpu_helpers import ROOT


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text,
                             flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol():
    from speculative_decoding_verification_sample_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    declared = _declared()
    assert {"spec_verify_sample", "spec_verify_greedy", "kv_commit_rollback"} <= declared
    for name in sorted(declared):
        assert hasattr(lib, name), name
    import speculative_decoding_verification_sample_gb300 as sv
    assert set(sv.EXPORTED) == declared
    assert sv.lib().spec_version() == 100
    assert sv.lib().spec_status_string(-1) == b"invalid argument"


def test_binding_refuses_cpu_tensors():
    import pytest
    import torch
    import speculative_decoding_verification_sample_gb300 as sv
    t = torch.zeros((1, 2, 8), dtype=torch.bfloat16)
    tok = torch.zeros((1, 1), dtype=torch.int32)
    with pytest.raises(ValueError):
        sv.spec_verify_greedy(t, tok, torch.zeros((1, 2), dtype=torch.int32),
                              torch.zeros((1,), dtype=torch.int32))


def test_small_batch_knob_changes_the_split(monkeypatch):
    """SPECVERIFY_SMALL_BATCH (host logic, no GPU needed): the workspace size
    follows the work split, so forcing the small-batch dispatch off for B = 8
    (38 slices a row by default, 64 without) or on for B = 64 (10 and 19
    slices a row by default for sampling and greedy, 4 with) changes it; any
    value but 0 or 1 leaves the default."""
    import speculative_decoding_verification_sample_gb300 as sv
    ws = lambda B: sv.spec_verify_workspace_bytes(B, 4, 151936, sv.SPEC_BF16)  # noqa: E731
    monkeypatch.delenv("SPECVERIFY_SMALL_BATCH", raising=False)
    d8, d64 = ws(8), ws(64)
    monkeypatch.setenv("SPECVERIFY_SMALL_BATCH", "0")
    assert ws(8) > d8 and ws(64) == d64
    monkeypatch.setenv("SPECVERIFY_SMALL_BATCH", "1")
    assert ws(8) == d8 and ws(64) < d64
    monkeypatch.setenv("SPECVERIFY_SMALL_BATCH", "2")
    assert ws(8) == d8 and ws(64) == d64
