"""Helpers for the GPU tests: build/load the library, move synthetic cases to the
device, run the C-ABI calls through the binding, and compare with the oracle."""
from __future__ import annotations

import os

import numpy as np

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def gpu_lib():
    """Builds (if needed) and loads the library; a GPU test without a GPU fails."""
    import torch
    from speculative_decoding_verification_sample_gb300 import build
    build.build()
    import speculative_decoding_verification_sample_gb300 as sv
    assert torch.cuda.is_available(), "GPU test run without a CUDA device"
    sv.lib()
    return sv


def ex2_bound_constant() -> float:
    path = os.path.join(ROOT, "speculative_decoding_verification_sample_gb300", "csrc",
                        "launch.h")
    for line in open(path):
        if "kEx2RelErrBound" in line and "=" in line:
            return float(line.split("=")[1].strip().rstrip(";"))
    raise AssertionError("kEx2RelErrBound not found")


def to_dev_logits(arr: np.ndarray, dtype: str):
    import torch
    if dtype == synth.BF16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()


def dev_case(case: synth.VerifyCase) -> dict:
    import torch
    d = dict(target=to_dev_logits(case.target, case.dtype),
             tokens=torch.from_numpy(case.tokens.astype(np.int32)).cuda(),
             uniforms=torch.from_numpy(case.uniforms.astype(np.float32)).cuda())
    d["draft"] = to_dev_logits(case.draft, case.dtype) if case.draft is not None else None
    return d


def run_sample(sv, case: synth.VerifyCase, dev: dict | None = None, temperature=None,
               **kw) -> dict:
    import torch
    dev = dev or dev_case(case)
    B, K = case.B, case.K
    T = case.temperature if temperature is None else temperature
    out = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    info = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    qd = torch.zeros((B, K), dtype=torch.float32, device="cuda")
    pd = torch.zeros((B, K), dtype=torch.float32, device="cuda")
    sv.spec_verify_sample(dev["target"], dev["draft"], dev["tokens"], dev["uniforms"], T, out, n,
                          err_flag=err, row_info=info, q_at_d=qd, p_at_d=pd, **kw)
    torch.cuda.synchronize()
    return dict(out_tokens=out.cpu().numpy(), num_accepted=n.cpu().numpy(),
                row_info=info.cpu().numpy(), err=int(err.item()), q_at_d=qd.cpu().numpy(),
                p_at_d=pd.cpu().numpy())


def run_greedy(sv, case: synth.VerifyCase, dev: dict | None = None) -> dict:
    import torch
    dev = dev or dev_case(case)
    B, K = case.B, case.K
    out = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    sv.spec_verify_greedy(dev["target"], dev["tokens"], out, n, err_flag=err)
    torch.cuda.synchronize()
    return dict(out_tokens=out.cpu().numpy(), num_accepted=n.cpu().numpy(), err=int(err.item()))


WINDOW = 1e-5      # a uniform this close to a decision boundary (oracle fp64) may differ
MAX_RATE = 1e-4    # ... and such differences must stay below this fraction of draws
PROB_TOL = 1e-5    # softmax probabilities of the draft tokens, absolute


def compare_sample(gpu: dict, orc: dict, rows=None) -> dict:
    """Row-by-row comparison. Returns counts; a row may differ from the oracle only
    if the decision that differs was within WINDOW of its boundary."""
    go, gn = gpu["out_tokens"], gpu["num_accepted"]
    oo, on = orc["out_tokens"], orc["num_accepted"]
    if rows is not None:
        go, gn = go[rows], gn[rows]
    B, K1 = oo.shape
    K = K1 - 1
    mism, outside = 0, []
    for b in range(B):
        if gn[b] == on[b] and np.array_equal(go[b], oo[b]):
            continue
        mism += 1
        nmin = min(int(gn[b]), int(on[b]))
        if gn[b] != on[b]:
            margin = orc["accept_margin"][b, nmin] if nmin < K else 0.0
        else:
            margin = orc["sample_margin"][b]
        if not (margin < WINDOW):
            outside.append((b, int(gn[b]), int(on[b]), float(margin)))
    qd = gpu["q_at_d"] if rows is None else gpu["q_at_d"][rows]
    pd = gpu["p_at_d"] if rows is None else gpu["p_at_d"][rows]
    dq = float(np.max(np.abs(qd - orc["q_at_d"]))) if qd.size else 0.0
    dp = float(np.max(np.abs(pd - orc["p_at_d"]))) if pd.size else 0.0
    window = int(np.sum(orc["sample_margin"] < WINDOW))
    return dict(rows=B, mismatches=mism, outside=outside, max_dq=dq, max_dp=dp,
                window_draws=window)


def assert_sample_parity(gpu: dict, orc: dict, rows=None, label=""):
    r = compare_sample(gpu, orc, rows)
    assert r["outside"] == [], (label, r)
    assert r["mismatches"] <= MAX_RATE * r["rows"], (label, r)
    assert r["max_dq"] <= PROB_TOL and r["max_dp"] <= PROB_TOL, (label, r)
    return r
