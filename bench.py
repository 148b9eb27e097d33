"""Benchmark of the speculative-decoding verification step on GB300.

One step = one pass of the whole hot path over one batch:
  spec_verify_sample  (accept/reject, first rejection, residual or bonus draw)
  kv_commit_rollback  (commit of the accepted slots in the paged KV cache)
on B=256 rows, K=4 drafts, V=151936 bf16 logits, T=1.0, draft = target + N(0, 0.5^2),
paged KV of 32 layers x 8 KV heads x head_dim 128 bf16, block 16, prefixes U[512, 4096].

Metric: verified draft positions per second (B*K per step), whole job over all ranks.
Inputs rotate over 3 pre-generated batches (3 x 622 MB of logits, larger than the
129 MB L2) so no step finds its logits in L2. Each step also restores the small KV
tables (so every step commits the same rows); that copy is inside the timed region.

Prints one JSON line (rank 0). `--impl reference` times the fp64 CPU oracle on the
same workload instead (a bounded sample of rows per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified draft positions/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "positions/s"
WORKLOAD = dict(B=256, K=4, V=151936, T=1.0, sigma=0.5, target_std=3.0, logits="bf16",
                kv_layers=32, kv_heads=8, head_dim=128, kv_dtype="bf16", block_size=16,
                prefix_lo=512, prefix_hi=4096)
PROFILES = {  # committed ncu summaries of the timed kernel, per mode
    "sample": os.path.join(ROOT, "profiles", "verify_sample_kernel_b256_k4_v151936.md"),
    "greedy": os.path.join(ROOT, "profiles", "verify_greedy_kernel_b256_k4_v151936.md"),
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--temperature", type=float, default=WORKLOAD["T"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--mode", default="step", choices=["step", "verify", "greedy", "filter"],
                   help="step: verify + KV commit (the benchmark); verify / greedy: that kernel "
                        "alone on the same logits, no KV pool (small footprint, for profiling); "
                        "filter: the top-k / top-p thresholds of one batch alone")
    p.add_argument("--kv-prefix", default=None,
                   help="LO,HI: committed prefix lengths U[LO, HI] of the KV case (default: the "
                        "workload's); short prefixes shrink the paged pool (profiling)")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the extra measurements after the timed step (profiling)")
    p.add_argument("--batches", type=int, default=3, help="input batches to rotate over")
    p.add_argument("--sweep", action="store_true",
                   help="time the verify launch over the B x K x V x T grid (one JSON line per cell)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_name(T, prefix=None):
    w = WORKLOAD
    lo, hi = prefix or (w["prefix_lo"], w["prefix_hi"])
    return (f"sampling verify + paged-KV commit: B={w['B']}, K={w['K']}, V={w['V']} bf16 logits, "
            f"T={T}, draft = target + N(0, {w['sigma']}^2), target ~ N(0, {w['target_std']}^2); "
            f"KV {w['kv_layers']}L x {w['kv_heads']}H x {w['head_dim']}D bf16, block "
            f"{w['block_size']}, prefix U[{lo}, {hi}]")


# ------------------------------------------------------------------ inputs
def gen_batch(torch, seed, T, B=None, K=None, V=None):
    """Synthetic verifier inputs on the GPU (the draft token is the draft model's
    own Gumbel-max sample; the verifier never sees how it was drawn). Shape
    defaults to the bench workload."""
    import numpy as np
    import synth
    w = WORKLOAD
    B, K, V = B or w["B"], K or w["K"], V or w["V"]
    g = torch.Generator(device="cuda").manual_seed(seed)
    zt = (torch.randn((B, K + 1, V), device="cuda", generator=g) * w["target_std"]).to(torch.bfloat16)
    zd = (zt[:, :K].float() + torch.randn((B, K, V), device="cuda", generator=g) * w["sigma"]
          ).to(torch.bfloat16)
    gum = -torch.log(-torch.log(torch.rand((B, K, V), device="cuda", generator=g)
                                .clamp_(1e-20, 1.0 - 1e-7)))
    tok = torch.argmax(zd.float() / float(np.float32(T)) + gum, dim=-1).to(torch.int32)
    del gum
    u = torch.from_numpy(synth.philox_uniforms((B, K + 1), seed)).cuda()
    return dict(target=zt.contiguous(), draft=zd.contiguous(), tokens=tok.contiguous(), uniforms=u)


def kv_state(torch, na, prefix=None):
    import numpy as np
    import synth
    w = WORKLOAD
    lo, hi = prefix or (w["prefix_lo"], w["prefix_hi"])
    c = synth.kv_case(w["B"], w["K"], block_size=w["block_size"], prefix_lo=lo,
                      prefix_hi=hi, num_accepted=na, seed=44)
    # the tables a commit changes live in one buffer, restored by one copy per step
    host = dict(bt=c.block_table, sl=c.seq_lens, pb=c.prov_blocks, fs=c.free_stack,
                ft=[c.free_top])
    host = {k: np.ascontiguousarray(v, np.int32) for k, v in host.items()}
    buf = torch.from_numpy(np.concatenate([v.ravel() for v in host.values()])).cuda()
    d, o = {}, 0
    for k, v in host.items():
        d[k] = buf[o:o + v.size].view(v.shape)
        o += v.size
    d["st"] = torch.zeros(1, dtype=torch.int32, device="cuda")
    saved = (buf, buf.clone())
    pool = torch.empty((c.num_blocks, w["kv_layers"], 2, w["block_size"], w["kv_heads"],
                        w["head_dim"]), dtype=torch.bfloat16, device="cuda")
    return c, d, saved, pool


def inplace_kv_us(torch, sv, na, reps=200):
    """Mean device time (us) of kv_commit_inplace on the bench's batch: prefix lengths
    U[prefix_lo, prefix_hi], the K+1 provisional slots appended in each row's own
    blocks, the accepted counts of the verify step. State restored between calls."""
    import numpy as np
    w = WORKLOAD
    B, K, bs = w["B"], w["K"], w["block_size"]
    rng = np.random.default_rng(45)
    L = rng.integers(w["prefix_lo"], w["prefix_hi"] + 1, size=B)
    mb = -(-(w["prefix_hi"] + K + 1) // bs)
    nb = B * mb + 64
    ids = rng.permutation(nb)
    bt = -np.ones((B, mb), np.int32)
    k = 0
    for b in range(B):
        for j in range(-(-int(L[b] + K + 1) // bs)):
            bt[b, j] = ids[k]
            k += 1
    fs = -np.ones(nb, np.int32)
    fs[:nb - k] = ids[k:]
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.int32)).cuda()  # noqa: E731
    saved = dict(bt=dev(bt), sl=dev(L), fs=dev(fs), ft=dev([nb - k]))
    cur = {key: v.clone() for key, v in saved.items()}
    st, n = dev([0]), dev(na)
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for i in range(reps + 3):
        for key in cur:
            cur[key].copy_(saved[key], non_blocking=True)
        if i >= 3:
            evs[i - 3][0].record(stream)
        sv.kv_commit_inplace(cur["bt"], cur["sl"], n, cur["fs"], cur["ft"], st, K=K,
                             block_size=bs, num_blocks=nb)
        if i >= 3:
            evs[i - 3][1].record(stream)
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"kv_commit_inplace status {int(st.item())}")
    return 1e3 * statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)


def tree_greedy_stats(torch, sv, peak, reps=50):
    """spec_verify_tree_greedy on the lesson's [2, 2, 2] draft tree (14 nodes, 15
    target rows per batch row) at B=256, V=151936 bf16: mean device time of one
    launch, its algorithmic HBM bytes (every target row read once) and the
    fraction of the measured copy peak. Planted argmaxes (target ~ N(0, 3^2)
    clipped, one logit per row raised to 16); each sibling group carries its
    row's argmax with probability 0.8. One 1.17 GB input (> L2)."""
    import numpy as np
    import synth
    w = WORKLOAD
    B, V = w["B"], w["V"]
    par = synth.tree_parents((2, 2, 2))
    N = len(par)
    rng = np.random.default_rng(46)
    g = rng.integers(0, V, size=(B, N + 1))
    tok = (g[:, par + 1] + 1 + rng.integers(0, V - 1, size=(B, N))) % V
    for r in range(N + 1):
        kids = np.flatnonzero(par == r - 1)
        if kids.size == 0:
            continue
        hit = rng.random(B) < 0.8
        pick = kids[rng.integers(0, kids.size, size=B)]
        tok[hit, pick[hit]] = g[hit, r]
    gen = torch.Generator(device="cuda").manual_seed(46)
    z = (torch.randn((B, N + 1, V), device="cuda", generator=gen) * w["target_std"]).clamp_(
        -synth.CLIP, synth.CLIP)
    gt = torch.from_numpy(g).cuda()
    z.scatter_(2, gt.unsqueeze(-1), synth.PLANT_VALUE)
    target = z.to(torch.bfloat16).contiguous()
    del z
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.int32)).cuda()  # noqa: E731
    pt, tt = dev(np.tile(par, (B, 1))), dev(tok)
    out = torch.empty((B, N + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((B,), dtype=torch.int32, device="cuda")
    slots = torch.empty((B, N + 1), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for i in range(reps + 3):
        if i >= 3:
            evs[i - 3][0].record(stream)
        sv.spec_verify_tree_greedy(target, pt, tt, out, n, out_slots=slots)
        if i >= 3:
            evs[i - 3][1].record(stream)
    torch.cuda.synchronize()
    us = 1e3 * statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    alg = B * (N + 1) * V * 2 + B * N * 8
    gbs = alg / (us / 1e6) / 1e9
    return {"tree": "[2, 2, 2] (14 nodes)", "us": us, "algorithmic_bytes": alg, "gbs": gbs,
            "frac_of_measured_peak": gbs / peak,
            "mean_accepted": float(n.float().mean().item())}


def filter_stats(torch, sv, bt, T, peak, reps=10, top_k=50, top_p=0.95):
    """spec_filter_thresholds (top-k 50, top-p 0.95) on one bench batch: the
    target [B, K+1, V] and draft [B, K, V] bf16 tensors (700 MB of logits per
    read), then spec_verify_sample with those thresholds. Mean device
    times; algorithmic bytes of the filter = every logit read once."""
    w = WORKLOAD
    B, K, V = w["B"], w["K"], w["V"]
    tt = torch.empty((B, K + 1), dtype=torch.float32, device="cuda")
    td = torch.empty((B, K), dtype=torch.float32, device="cuda")
    out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((B,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def filt():
        sv.spec_filter_thresholds(bt["target"], T, top_k, top_p, tt)
        sv.spec_filter_thresholds(bt["draft"], T, top_k, top_p, td)

    def ver():
        sv.spec_verify_sample(bt["target"], bt["draft"], bt["tokens"], bt["uniforms"], T, out, n,
                              target_threshold=tt, draft_threshold=td)

    res = {}
    for name, fn in (("filter", filt), ("verify_filtered", ver)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name + "_us"] = 1e3 * e0.elapsed_time(e1) / reps
    alg = B * (2 * K + 1) * V * 2
    res["filter_algorithmic_bytes"] = alg
    res["filter_gbs"] = alg / (res["filter_us"] / 1e6) / 1e9
    res["filter_frac_of_measured_peak"] = res["filter_gbs"] / peak
    res["top_k"], res["top_p"] = top_k, top_p
    return res


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.p = None
        self.gpu = gpu_index
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ helpers
def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_sample_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kind):
    """DRAM bytes (read + write) per launch from the committed ncu summary of the
    kernel, if it was taken on the current kernel sources (else None)."""
    fields = {}
    try:
        with open(PROFILES[kind]) as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip() in ("source_hash", "dram_bytes_per_launch") and v.strip():
                    fields[k.strip()] = v.strip()
    except OSError:
        return None
    if fields.get("source_hash") != source_hash():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def algorithmic_verify_bytes(na, K, V, e=2):
    """Bytes the verify launch must move: all 2K logit rows of every batch row, the
    bonus row of fully accepted rows, and the per-row inputs/outputs."""
    import numpy as np
    B = len(na)
    full = int(np.sum(np.asarray(na) == K))
    meta = B * (4 * K + 4 * (K + 1) + 4 * (K + 1) + 4)
    return B * 2 * K * V * e + full * V * e + meta


def sequential_verify_bytes(na, K, V, e=2):
    """Secondary figure: the bytes a verifier that reads only the positions it
    needs would move (target and draft rows 0..n of a row rejected at n, all 2K
    rows plus the bonus row of a fully accepted one), plus the per-row I/O."""
    import numpy as np
    na = np.asarray(na)
    rows = np.where(na < K, 2 * (na + 1), 2 * K + 1)
    meta = len(na) * (4 * K + 4 * (K + 1) + 4 * (K + 1) + 4)
    return int(np.sum(rows)) * V * e + meta


def greedy_verify_bytes(na, K, V, e=2):
    """Bytes the greedy launch must move: target rows 0..K-1 of every row, row K of
    the rows that accept everything, and the per-row I/O."""
    import numpy as np
    B = len(na)
    full = int(np.sum(np.asarray(na) == K))
    return B * K * V * e + full * V * e + B * (4 * K + 4 * (K + 1) + 4)


def kv_bytes(na, w):
    import numpy as np
    slot = w["kv_layers"] * 2 * w["kv_heads"] * w["head_dim"] * 2  # bytes of one token's KV
    return int(np.sum(np.asarray(na) + 1)) * slot * 2              # read + write


# ------------------------------------------------------------------ CPU oracle baseline
def _oracle_worker(job):
    """One host process: the fp64 oracle (verify + KV bookkeeping) on `rows` rows
    of the workload, repeated until `budget_s` seconds; returns (positions, s)."""
    rows, T, budget_s, seed = job
    import oracle
    import synth
    w = WORKLOAD
    c = synth.sampling_case(rows, w["K"], w["V"], temperature=T, target_std=w["target_std"],
                            draft_noise_std=w["sigma"], seed=seed, uniform_seed=seed)
    t_vals, d_vals = c.target_values(), c.draft_values()
    kc = synth.kv_case(rows, w["K"], block_size=w["block_size"], prefix_lo=w["prefix_lo"],
                       prefix_hi=w["prefix_hi"], seed=seed)
    done, t0 = 0, time.perf_counter()
    while True:
        r = oracle.verify_sample(t_vals, d_vals, c.tokens, c.uniforms, T)
        oracle.kv_commit(kc.block_table, kc.seq_lens, r["num_accepted"], kc.prov_blocks,
                         kc.free_stack, kc.free_top, block_size=w["block_size"], K=w["K"],
                         num_blocks=kc.num_blocks)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return done * rows * w["K"], el


def oracle_rate(T: float, budget_s: float, procs: int | None = None):
    """The fp64 oracle on the host cores, rows split over `procs` processes (all
    cores by default; started with `spawn`, so no process inherits a CUDA
    context), one batch row each, each repeating its row for `budget_s`
    seconds. Returns (positions/s over all processes, processes, description)."""
    import multiprocessing as mp
    procs = procs or os.cpu_count() or 1
    jobs = [(1, T, budget_s, 99 + i) for i in range(procs)]
    if procs == 1:
        res = [_oracle_worker(jobs[0])]
    else:
        with mp.get_context("spawn").Pool(procs) as pool:
            res = pool.map(_oracle_worker, jobs)
    positions = sum(r[0] for r in res)
    el = max(r[1] for r in res)
    rate = positions / el
    desc = (f"{procs} host processes (os.cpu_count() = {os.cpu_count()}), one batch row of the "
            f"workload each (K={WORKLOAD['K']}, V={WORKLOAD['V']}, T={T}), verify + KV "
            f"bookkeeping repeated for {el:.1f} s; rate = positions of all processes / the "
            f"longest process time; NumPy fp64")
    return rate, procs, desc


# ------------------------------------------------------------------ main
SWEEP = dict(B=(1, 8, 64, 256, 1024), K=(2, 4, 8), V=(32000, 128256, 151936), T=(0.0, 0.6, 1.0))


def sweep_cell(torch, sv, B, K, V, T, reps, flush, peak, peak_kind):
    """One cell of the sweep: 3 warm-up launches, then `reps` launches timed with
    CUDA events around each one and a write of `flush` (larger than L2) between
    them; the median launch with its algorithmic bytes against the peak. Small
    batches rotate over several input batches (a single row's draw path, and so
    its time, depends on its draws)."""
    import numpy as np
    nb = 8 if B <= 8 else 4 if B <= 64 else 1
    bts = [gen_batch(torch, 7 + B + K + 1000 * i, T if T > 0 else 1.0, B=B, K=K, V=V)
           for i in range(nb)]
    out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((B,), dtype=torch.int32, device="cuda")
    if T > 0:
        def call(bt):
            sv.spec_verify_sample(bt["target"], bt["draft"], bt["tokens"], bt["uniforms"], T,
                                  out, n)
    else:
        def call(bt):
            sv.spec_verify_greedy(bt["target"], bt["tokens"], out, n)
    nas = []
    for bt in bts:
        call(bt)
        torch.cuda.synchronize()
        nas.append(n.cpu().numpy().copy())
    ts = []
    for r in range(reps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        call(bts[r % nb])
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = float(np.median(ts))
    na = np.concatenate(nas)
    bpb = (algorithmic_verify_bytes if T > 0 else greedy_verify_bytes)
    alg = float(np.mean([bpb(x, K, V) for x in nas]))
    gbs = alg / (ms / 1e3) / 1e9
    cell = {"sweep": {"B": B, "K": K, "V": V, "T": T, "mode": "sample" if T > 0 else "greedy"},
            "us": ms * 1e3, "positions_per_s": B * K / (ms / 1e3), "algorithmic_bytes": alg,
            "gbs": gbs, "frac": gbs / peak, "peak_kind": peak_kind,
            "mean_accepted": float(na.mean())}
    if T > 0:
        seq = float(np.mean([sequential_verify_bytes(x, K, V) for x in nas]))
        cell["sequential_frac"] = seq / (ms / 1e3) / 1e9 / peak
    del bts
    torch.cuda.empty_cache()
    return cell


def run_sweep(a):
    """Verify-launch times over the grid of batch sizes, draft lengths, vocabularies
    and temperatures (T = 0: greedy), bf16 logits generated like the bench
    workload (target N(0, 3^2), draft = target + N(0, 0.5^2)); one JSON line
    per cell (sweep_cell, at most 20 timed launches)."""
    import torch
    import speculative_decoding_verification_sample_gb300 as sv
    from speculative_decoding_verification_sample_gb300 import build
    build.build()
    sv.lib()
    peak, peak_kind = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    reps = max(5, min(20, a.steps))
    for V in SWEEP["V"]:
        for K in SWEEP["K"]:
            for B in SWEEP["B"]:
                for T in SWEEP["T"]:
                    cell = sweep_cell(torch, sv, B, K, V, T, reps, flush, peak, peak_kind)
                    print(json.dumps(cell), flush=True)


SWEEP_SMALL = dict(B=(1, 8, 1024), K=4, V=151936, T=(0.0, 1.0))


def sweep_small(torch, sv, peak, peak_kind, reps=20):
    """The sweep cells B in {1, 8, 1024} x T in {0 (greedy), 1} at K=4, V=151936."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    cells = []
    for B in SWEEP_SMALL["B"]:
        for T in SWEEP_SMALL["T"]:
            c = sweep_cell(torch, sv, B, SWEEP_SMALL["K"], SWEEP_SMALL["V"], T, reps, flush,
                           peak, peak_kind)
            cells.append({k: c[k] for k in ("sweep", "us", "positions_per_s", "gbs", "frac",
                                            "mean_accepted")})
    del flush
    torch.cuda.empty_cache()
    return cells


def greedy_stats(torch, sv, batches, peak, reps=100):
    """verify_greedy_kernel on the bench's rotating batches (B=256, K=4,
    V=151936 bf16): mean device time per launch (CUDA events around each
    launch), algorithmic bytes = target rows 0..K-1 of every row + row K of
    the rows the greedy rule accepts in full + per-row I/O, and the fraction
    of the measured HBM peak."""
    import numpy as np
    w = WORKLOAD
    B, K, V = w["B"], w["K"], w["V"]
    out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((B,), dtype=torch.int32, device="cuda")
    nas = []
    for bt in batches:
        sv.spec_verify_greedy(bt["target"], bt["tokens"], out, n)
        torch.cuda.synchronize()
        nas.append(n.cpu().numpy().copy())
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    nb = len(batches)
    for i in range(reps + 3):
        bt = batches[i % nb]
        if i >= 3:
            evs[i - 3][0].record(stream)
        sv.spec_verify_greedy(bt["target"], bt["tokens"], out, n)
        if i >= 3:
            evs[i - 3][1].record(stream)
    torch.cuda.synchronize()
    us = 1e3 * statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    alg = statistics.mean(greedy_verify_bytes(x, K, V) for x in nas)
    gbs = alg / (us / 1e6) / 1e9
    return {"kernel": "verify_greedy_kernel<bf16>", "us": us, "algorithmic_bytes": alg,
            "gbs": gbs, "frac_of_measured_peak": gbs / peak,
            "mean_accepted": float(np.mean([x.mean() for x in nas])),
            "positions_per_s": B * K / (us / 1e6)}


def main():
    a = parse()
    if a.sweep:
        return run_sweep(a)
    rank, world, local = dist_env()
    T = a.temperature
    if a.impl == "reference":
        return run_reference(a, rank, world, T)
    import numpy as np
    import torch
    import speculative_decoding_verification_sample_gb300 as sv
    from speculative_decoding_verification_sample_gb300 import build
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    build.build()
    sv.lib()
    w = WORKLOAD
    B, K, V = w["B"], w["K"], w["V"]
    stream = torch.cuda.current_stream()
    nb = max(1, a.batches)
    batches = [gen_batch(torch, 1000 * rank + i, T) for i in range(nb)]
    if a.mode == "filter":
        if rank == 0:
            r = filter_stats(torch, sv, batches[0], T, peaks()[0], reps=max(1, a.steps))
            print(json.dumps({"mode": "filter", "config": {"workload": workload_name(T)}, **r}))
        return
    prefix = tuple(int(x) for x in a.kv_prefix.split(",")) if a.kv_prefix else None
    out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((B,), dtype=torch.int32, device="cuda")
    info = torch.empty((B,), dtype=torch.int32, device="cuda")
    # accepted counts of each batch (fixed for the run) to build the KV state and byte counts
    na_list = []
    for bt in batches:
        sv.spec_verify_sample(bt["target"], bt["draft"], bt["tokens"], bt["uniforms"], T, out, n,
                              row_info=info)
        torch.cuda.synchronize()
        na_list.append((n.cpu().numpy().copy(), info.cpu().numpy().copy()))
    if a.mode == "step":
        kc, kd, saved, pool = kv_state(torch, np.max([x[0] for x in na_list], axis=0), prefix)

    def step(i, ev=None):
        bt = batches[i % nb]
        if a.mode == "step":
            saved[0].copy_(saved[1], non_blocking=True)
        if ev is not None:
            ev[0].record(stream)
        if a.mode == "greedy":
            sv.spec_verify_greedy(bt["target"], bt["tokens"], out, n)
        else:
            sv.spec_verify_sample(bt["target"], bt["draft"], bt["tokens"], bt["uniforms"], T,
                                  out, n)
        if ev is not None:
            ev[1].record(stream)
        if a.mode == "step":
            sv.kv_commit_rollback(kd["bt"], kd["sl"], n, kd["pb"], pool, kd["fs"], kd["ft"],
                                  kd["st"], K=K, block_size=w["block_size"])

    for i in range(max(3, a.warmup)):
        step(i)
    torch.cuda.synchronize()
    if a.mode == "step" and int(kd["st"].item()) != 0:
        raise RuntimeError(f"kv commit status {int(kd['st'].item())}")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(a.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    time.sleep(0.2)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(a.steps):
        step(i, evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    verify_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    if world > 1:
        total_ms = max_over_ranks(total_ms, "cuda")
    ms_per_step = total_ms / a.steps
    value = job_rate(world, B, K, ms_per_step)

    # roofline of the dominant kernel (spec_verify_sample), live CUDA-event durations
    if a.mode == "greedy":
        # greedy reads target rows 0..K-1, plus row K for rows that accept everything
        gna = []
        for bt in batches:
            sv.spec_verify_greedy(bt["target"], bt["tokens"], out, n)
            torch.cuda.synchronize()
            gna.append(n.cpu().numpy().copy())
        alg = statistics.mean(greedy_verify_bytes(x, K, V) for x in gna)
    else:
        alg = statistics.mean(algorithmic_verify_bytes(x[0], K, V) for x in na_list)
    v_ms = statistics.mean(verify_ms)
    peak, peak_kind = peaks()
    achieved = alg / (v_ms / 1e3) / 1e9
    refined = float(np.mean([np.mean(x[1] != 0) for x in na_list]))
    seqb = statistics.mean(sequential_verify_bytes(x[0], K, V) for x in na_list)
    kvb = statistics.mean(kv_bytes(x[0], w) for x in na_list)

    # end-to-end through the public API with host buffers
    e2e = None
    if a.e2e_steps > 0 and a.mode == "step" and nb >= 2:
        host = [{k: v.cpu().pin_memory() for k, v in bt.items()} for bt in batches]
        h2d = sum(v.numel() * v.element_size() for v in host[0].values())
        d2h = out.numel() * 4 + n.numel() * 4
        out_h = torch.empty_like(out, device="cpu").pin_memory()
        n_h = torch.empty_like(n, device="cpu").pin_memory()

        # HostVerifier: the rows are copied in chunks on a copy stream and each
        # chunk is verified as soon as it lands, hiding the verification
        # behind the host-to-device transfer
        hv = sv.HostVerifier(B, K, batches[0]["target"].shape[-1], dtype=batches[0]["target"].dtype,
                             chunks=8)

        def e2e_step(i):
            hb = host[i % nb]
            saved[0].copy_(saved[1], non_blocking=True)
            _, nd = hv(hb["target"], hb["draft"], hb["tokens"], hb["uniforms"], T)
            sv.kv_commit_rollback(kd["bt"], kd["sl"], nd, kd["pb"], pool, kd["fs"], kd["ft"],
                                  kd["st"], K=K, block_size=w["block_size"])
            hv.to_host(out_h, n_h)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(a.e2e_steps):
            e2e_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / a.e2e_steps
        if world > 1:
            e2e_ms = max_over_ranks(e2e_ms, "cuda")
        e2e = {"value": job_rate(world, B, K, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline and a.mode == "step":
        rate, procs, desc = oracle_rate(T, 10.0)
        cpu = {"value": rate, "unit": UNIT, "cores": procs, "nproc": os.cpu_count(),
               "kind": "oracle", "rows_split_over_processes": procs > 1, "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": max(3, a.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_name(T, prefix), "global_batch": world * B,
                       "B_per_gpu": B,
                       "K": K, "V": V, "logits_dtype": "bf16", "temperature": T,
                       "parallelism": f"replicas x{world} (batch rows sharded, no collective)",
                       "mode": a.mode,
                       "l2": f"inputs rotate over {nb} batch(es) of 622 MB logits (> 129 MB L2)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": profiled_traffic("greedy" if a.mode == "greedy" else "sample"),
                         "kernel": ("verify_greedy_kernel<bf16>" if a.mode == "greedy"
                                    else "verify_sample_kernel<bf16>"), "peak_kind": peak_kind,
                         "algorithmic_bytes_per_launch": alg, "avg_launch_ms": v_ms},
            "cpu_baseline": cpu,
            "e2e": e2e,
            # workspace zeroing + verify (+ kv plan, copy, finish) per step
            "gpu_launches": (5 if a.mode == "step" else 2) * a.steps,
            "clocks": clk,
            "extra": {"verify_ms": v_ms, "kv_commit_and_table_restore_ms": ms_per_step - v_ms,
                      **extras(a, torch, sv, batches, na_list, T, peak, peak_kind),
                      "kv_bytes_per_step": kvb, "refined_row_fraction": refined,
                      "mean_accepted": float(np.mean([x[0].mean() for x in na_list])),
                      "hbm_frac_of_nominal_8TBs": achieved / 8000.0,
                      "sequential_bytes_per_launch": (seqb if a.mode != "greedy" else None),
                      "sequential_frac_of_measured_peak": (
                          seqb / (v_ms / 1e3) / 1e9 / peak if a.mode != "greedy" else None)},
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def extras(a, torch, sv, batches, na_list, T, peak, peak_kind):
    """The extra measurements after the timed step (step mode)."""
    if a.mode != "step" or a.no_extras:
        return {}
    return {"kv_commit_inplace_us": inplace_kv_us(torch, sv, na_list[0][0]),
            "tree_greedy": tree_greedy_stats(torch, sv, peak),
            "top_k_top_p": filter_stats(torch, sv, batches[0], T, peak),
            "greedy": greedy_stats(torch, sv, batches, peak),
            "sweep_small": sweep_small(torch, sv, peak, peak_kind)}


def max_over_ranks(x, device=None):
    """The maximum of a per-rank float over the process group (x itself when
    no group is initialised). Tensors live on `device` (CUDA under NCCL, CPU
    under gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, B, K, ms_per_step):
    """Whole-job verified positions per second: every rank verifies B rows of
    K draft positions per step (weak scaling, replicas)."""
    return world * B * K / (ms_per_step / 1e3)


_REF_CASES = {}


def _reference_init(rows, T):
    """Pool initializer: every process generates all `rows` batch rows once, so
    whichever row a step hands it is ready."""
    import synth
    w = WORKLOAD
    for i in range(rows):
        c = synth.sampling_case(1, w["K"], w["V"], temperature=T, target_std=w["target_std"],
                                draft_noise_std=w["sigma"], seed=99 + i, uniform_seed=99 + i)
        kc = synth.kv_case(1, w["K"], block_size=w["block_size"], prefix_lo=w["prefix_lo"],
                           prefix_hi=w["prefix_hi"], seed=99 + i)
        _REF_CASES[i] = (c, c.target_values(), c.draft_values(), kc)


def _reference_row(job):
    """One row of the reference arm in a host process: the fp64 oracle's verify +
    KV bookkeeping on batch row `i` of the workload."""
    i, T = job
    import oracle
    w = WORKLOAD
    c, tv, dv, kc = _REF_CASES[i]
    t0 = time.perf_counter()
    r = oracle.verify_sample(tv, dv, c.tokens, c.uniforms, T)
    oracle.kv_commit(kc.block_table, kc.seq_lens, r["num_accepted"], kc.prov_blocks,
                     kc.free_stack, kc.free_top, block_size=w["block_size"], K=w["K"],
                     num_blocks=kc.num_blocks)
    return time.perf_counter() - t0


def run_reference(a, rank, world, T):
    """Reference arm: the fp64 CPU oracle on a bounded sample of the same workload.
    Each step verifies one batch row per host core, the rows split over a pool of
    `spawn`ed processes (one row per process, generated once); the step time is
    the wall time of that parallel map."""
    if rank != 0:
        return
    import multiprocessing as mp
    w = WORKLOAD
    procs = os.cpu_count() or 1
    jobs = [(i, T) for i in range(procs)]
    with mp.get_context("spawn").Pool(procs, initializer=_reference_init,
                                      initargs=(procs, T)) as pool:
        for _ in range(max(3, a.warmup)):
            pool.map(_reference_row, jobs)
        t0 = time.perf_counter()
        for _ in range(a.steps):
            pool.map(_reference_row, jobs)
        el = time.perf_counter() - t0
    ms = el * 1e3 / a.steps
    value = procs * w["K"] / (el / a.steps)
    sample = (f"{procs} batch rows per step (one per host process, os.cpu_count() = "
              f"{os.cpu_count()}), verify + KV bookkeeping, NumPy fp64")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": a.steps, "warmup": max(3, a.warmup), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload_name(T) + f" (oracle: {procs} rows per step)",
                       "global_batch": procs, "K": w["K"], "V": w["V"]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": procs,
                             "nproc": os.cpu_count(), "kind": "oracle",
                             "rows_split_over_processes": procs > 1, "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
