"""GB300 speculative-decoding verification (sm_103a).

Thin ctypes binding of the in-tree C-ABI library `libspecverify.so`: argument
marshalling only. Every step of the verification runs in the library's CUDA
kernels; PyTorch supplies device memory and the current stream. There is no
CPU fallback: without the built library (or without a GPU) these calls raise.

The entry points carry the C names:
  spec_verify_sample(...)   accept/reject with temperature softmax, residual or bonus draw
  spec_verify_greedy(...)   argmax-match verification
  spec_verify_tree_greedy(...)  argmax-match verification of a draft tree
  kv_commit_rollback(...)   commit accepted provisional KV slots, free provisional blocks
See include/specverify.h for layouts, ownership and error behaviour.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SPEC_OK, SPEC_EINVAL, SPEC_ECUDA, SPEC_ENOTSUP = 0, -1, -2, -3
SPEC_BF16, SPEC_F32 = 0, 1
SPEC_DERR_TOKEN, SPEC_DERR_LOGITS = 1, 2
SPEC_DERR_BAD_ACCEPT, SPEC_DERR_BAD_LENGTH, SPEC_DERR_NO_SPACE, SPEC_DERR_BAD_BLOCK = 4, 8, 16, 32
SPEC_DERR_TIMEOUT = 64
SPEC_DERR_BAD_SLOT = 128
SPEC_ROW_ACCEPT_REFINED, SPEC_ROW_SAMPLE_REFINED = 1, 2
SPEC_ROW_UNCERTIFIED, SPEC_ROW_ZERO_RESIDUAL = 4, 8

EXPORTED = ("spec_verify_sample", "spec_verify_greedy", "spec_verify_workspace_bytes",
            "kv_commit_rollback", "spec_selftest_ex2", "spec_status_string", "spec_version",
            "spec_verify_greedy_noalloc", "spec_verify_greedy_noalloc_max_bytes",
            "kv_commit_inplace", "kv_evict_provisional", "spec_verify_tree_greedy",
            "spec_filter_thresholds")

_lib = None


class SpecError(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, fn: str, status: int):
        msg = lib().spec_status_string(status).decode() if _lib else str(status)
        super().__init__(f"{fn}: status {status} ({msg})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libspecverify.so (built by `build.build()`); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run "
                               "speculative_decoding_verification_sample_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        Z = ctypes.c_size_t
        L.spec_verify_sample.argtypes = [P, P, P, P, F, I, I, I, P, P, P, I, P, P, P, P, P, Z, P,
                                         P, P]
        L.spec_verify_sample.restype = I
        L.spec_verify_greedy.argtypes = [P, P, I, I, I, P, P, P, I, P, P, Z, P]
        L.spec_verify_greedy.restype = I
        L.spec_verify_tree_greedy.argtypes = [P, P, P, I, I, I, P, P, P, P, I, P, P, Z]
        L.spec_verify_tree_greedy.restype = I
        L.spec_filter_thresholds.argtypes = [P, I, I, I, F, I, F, P, P, P]
        L.spec_filter_thresholds.restype = I
        L.spec_verify_greedy_noalloc.argtypes = [P, P, I, I, I, P, P, P, I, P]
        L.spec_verify_greedy_noalloc.restype = I
        L.kv_commit_inplace.argtypes = [P, P, P, I, I, I, I, I, P, P, P, P]
        L.kv_commit_inplace.restype = I
        L.kv_evict_provisional.argtypes = [P, P, I, I, I, I, I, P, P, P, P]
        L.kv_evict_provisional.restype = I
        L.spec_verify_greedy_noalloc_max_bytes.argtypes = []
        L.spec_verify_greedy_noalloc_max_bytes.restype = Z
        L.spec_verify_workspace_bytes.argtypes = [I, I, I, I]
        L.spec_verify_workspace_bytes.restype = Z
        L.kv_commit_rollback.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, P, P, P, P,
                                         P]
        L.kv_commit_rollback.restype = I
        L.spec_selftest_ex2.argtypes = [F, F, P, P]
        L.spec_selftest_ex2.restype = I
        L.spec_status_string.argtypes = [I]
        L.spec_status_string.restype = ctypes.c_char_p
        L.spec_version.argtypes = []
        L.spec_version.restype = I
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _check(t, name, ndim=None, dtype=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


_workspaces = {}


def spec_verify_workspace_bytes(B: int, K: int, V: int, dtype_code: int) -> int:
    """Device workspace bytes the verify calls need for (B, K, V, dtype)."""
    return int(lib().spec_verify_workspace_bytes(B, K, V, dtype_code))


def workspace_for(B: int, K: int, V: int, dtype_code: int, device):
    """A cached device workspace (uint8 tensor) large enough for (B, K, V, dtype)
    on `device`. Calls sharing it must be ordered on the device."""
    import torch
    need = spec_verify_workspace_bytes(B, K, V, dtype_code)
    if need == 0:
        raise SpecError("spec_verify_workspace_bytes", SPEC_EINVAL)
    dev = torch.device(device)
    key = (dev.type, dev.index if dev.index is not None else torch.cuda.current_device())
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.empty(need + 256, dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def _ws_args(ws, B, K, V, code, device):
    if ws is None:
        if spec_verify_workspace_bytes(B, K, V, code) == 0:
            # unsupported shape: the library call itself reports why
            return ctypes.c_void_p(0), ctypes.c_size_t(0)
        ws = workspace_for(B, K, V, code, device)
    off = (-ws.data_ptr()) % 256
    return ctypes.c_void_p(ws.data_ptr() + off), ctypes.c_size_t(ws.numel() - off)


def _counters(t, K):
    """Pointer of an optional [2K+2] 64-bit integer device tensor of counters."""
    if t is None:
        return None
    import torch
    if not t.is_cuda or t.dtype not in (torch.int64, torch.uint64) or t.numel() != 2 * K + 2 \
            or not t.is_contiguous():
        raise ValueError(f"accept_counters must be a contiguous 64-bit integer CUDA tensor "
                         f"of {2 * K + 2} elements")
    return _ptr(t)


def _thr(t, B, n):
    """Pointer of an optional [B, n] float32 CUDA tensor of row thresholds."""
    if t is None:
        return None
    import torch
    if not t.is_cuda or t.dtype != torch.float32 or t.numel() != B * n or not t.is_contiguous():
        raise ValueError(f"thresholds must be a contiguous float32 CUDA tensor of {B * n} values")
    return _ptr(t)


def spec_verify_sample(target_logits, draft_logits, draft_tokens, uniforms, temperature: float,
                       out_tokens, out_num_accepted, *, stream=None, err_flag=None,
                       row_info=None, q_at_d=None, p_at_d=None, workspace=None,
                       accept_counters=None, target_threshold=None,
                       draft_threshold=None) -> None:
    """Sampling-mode verification; shapes [B,K+1,V], [B,K,V], [B,K], [B,K+1] -> [B,K+1], [B].
    accept_counters: optional int64/uint64 [2K+2] device tensor, accumulated (see the header).
    target_threshold [B,K+1] / draft_threshold [B,K]: optional float32 logit thresholds
    (spec_filter_thresholds) for top-k / top-p filtering."""
    import torch
    _check(target_logits, "target_logits", 3)
    B, K1, V = target_logits.shape
    K = K1 - 1
    if float(temperature) != 0.0:
        _check(draft_logits, "draft_logits", 3, target_logits.dtype)
        _check(uniforms, "uniforms", 2, torch.float32)
    _check(draft_tokens, "draft_tokens", 2, torch.int32)
    _check(out_tokens, "out_tokens", 2, torch.int32)
    _check(out_num_accepted, "out_num_accepted", 1, torch.int32)
    code = _dtype_code(target_logits)
    wsp, wsn = _ws_args(workspace, B, K, V, code, target_logits.device)
    st = lib().spec_verify_sample(
        _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(uniforms),
        ctypes.c_float(temperature), B, K, V, _ptr(out_tokens), _ptr(out_num_accepted),
        _stream(stream), code, _ptr(err_flag), _ptr(row_info),
        _ptr(q_at_d), _ptr(p_at_d), wsp, wsn, _counters(accept_counters, K),
        _thr(target_threshold, B, K + 1), _thr(draft_threshold, B, K))
    if st != SPEC_OK:
        raise SpecError("spec_verify_sample", st)


def spec_verify_greedy(target_logits, draft_tokens, out_tokens, out_num_accepted, *,
                       stream=None, err_flag=None, workspace=None, accept_counters=None) -> None:
    """Greedy verification; target [B,K+1,V], tokens [B,K] -> [B,K+1], [B]."""
    import torch
    _check(target_logits, "target_logits", 3)
    _check(draft_tokens, "draft_tokens", 2, torch.int32)
    _check(out_tokens, "out_tokens", 2, torch.int32)
    _check(out_num_accepted, "out_num_accepted", 1, torch.int32)
    B, K1, V = target_logits.shape
    code = _dtype_code(target_logits)
    wsp, wsn = _ws_args(workspace, B, K1 - 1, V, code, target_logits.device)
    st = lib().spec_verify_greedy(_ptr(target_logits), _ptr(draft_tokens), B, K1 - 1, V,
                                  _ptr(out_tokens), _ptr(out_num_accepted), _stream(stream),
                                  code, _ptr(err_flag), wsp, wsn,
                                  _counters(accept_counters, K1 - 1))
    if st != SPEC_OK:
        raise SpecError("spec_verify_greedy", st)


def spec_verify_tree_greedy(target_logits, tree_parents, tree_tokens, out_tokens,
                            out_num_accepted, *, out_slots=None, stream=None, err_flag=None,
                            workspace=None) -> None:
    """Greedy verification of a draft tree; target [B,N+1,V], parents and tokens [B,N]
    -> tokens [B,N+1], accepted [B], optional KV slots [B,N+1]."""
    import torch
    _check(target_logits, "target_logits", 3)
    _check(tree_parents, "tree_parents", 2, torch.int32)
    _check(tree_tokens, "tree_tokens", 2, torch.int32)
    _check(out_tokens, "out_tokens", 2, torch.int32)
    _check(out_num_accepted, "out_num_accepted", 1, torch.int32)
    if out_slots is not None:
        _check(out_slots, "out_slots", 2, torch.int32)
    B, N1, V = target_logits.shape
    code = _dtype_code(target_logits)
    wsp, wsn = _ws_args(workspace, B, N1 - 1, V, code, target_logits.device)
    st = lib().spec_verify_tree_greedy(_ptr(target_logits), _ptr(tree_parents),
                                       _ptr(tree_tokens), B, N1 - 1, V, _ptr(out_tokens),
                                       _ptr(out_num_accepted), _ptr(out_slots), _stream(stream),
                                       code, _ptr(err_flag), wsp, wsn)
    if st != SPEC_OK:
        raise SpecError("spec_verify_tree_greedy", st)


def spec_filter_thresholds(logits, temperature: float, top_k: int, top_p: float, out_threshold,
                           *, stream=None, err_flag=None) -> None:
    """Top-k / top-p logit threshold of every row of logits [..., V] -> out_threshold [...]
    (float32; keep tokens with logit >= threshold)."""
    import torch
    _check(logits, "logits")
    _check(out_threshold, "out_threshold", None, torch.float32)
    V = logits.shape[-1]
    R = logits.numel() // V
    if out_threshold.numel() != R:
        raise ValueError(f"out_threshold must hold {R} values")
    st = lib().spec_filter_thresholds(_ptr(logits), R, V, _dtype_code(logits),
                                      ctypes.c_float(temperature), int(top_k),
                                      ctypes.c_float(top_p), _ptr(out_threshold),
                                      _stream(stream), _ptr(err_flag))
    if st != SPEC_OK:
        raise SpecError("spec_filter_thresholds", st)


def spec_verify_greedy_noalloc(target_logits, draft_tokens, out_tokens, out_num_accepted, *,
                               stream=None, err_flag=None) -> None:
    """Greedy verification on the library's built-in device scratch (no workspace
    argument, nothing allocated). Calls on one device must not overlap."""
    import torch
    _check(target_logits, "target_logits", 3)
    _check(draft_tokens, "draft_tokens", 2, torch.int32)
    _check(out_tokens, "out_tokens", 2, torch.int32)
    _check(out_num_accepted, "out_num_accepted", 1, torch.int32)
    B, K1, V = target_logits.shape
    st = lib().spec_verify_greedy_noalloc(_ptr(target_logits), _ptr(draft_tokens), B, K1 - 1, V,
                                          _ptr(out_tokens), _ptr(out_num_accepted),
                                          _stream(stream), _dtype_code(target_logits),
                                          _ptr(err_flag))
    if st != SPEC_OK:
        raise SpecError("spec_verify_greedy_noalloc", st)


def spec_verify_greedy_noalloc_max_bytes() -> int:
    """Size of the built-in scratch used by spec_verify_greedy_noalloc."""
    return int(lib().spec_verify_greedy_noalloc_max_bytes())


def kv_commit_inplace(block_table, seq_lens, num_accepted, free_stack, free_top, status, *,
                      K: int, block_size: int, num_blocks: int, stream=None) -> None:
    """In-place KV commit: truncate each row to L + n + 1 and free the blocks past it."""
    import torch
    _check(block_table, "block_table", 2, torch.int32)
    for t, n in ((seq_lens, "seq_lens"), (num_accepted, "num_accepted"),
                 (free_stack, "free_stack"), (free_top, "free_top"), (status, "status")):
        _check(t, n, 1, torch.int32)
    B, MB = block_table.shape
    st = lib().kv_commit_inplace(_ptr(block_table), _ptr(seq_lens), _ptr(num_accepted),
                                 num_blocks, block_size, B, K, MB, _ptr(free_stack),
                                 _ptr(free_top), _ptr(status), _stream(stream))
    if st != SPEC_OK:
        raise SpecError("kv_commit_inplace", st)


def kv_evict_provisional(block_table, seq_lens, free_stack, free_top, status, *, K: int,
                         block_size: int, num_blocks: int, stream=None) -> None:
    """In-place layout: discard every row's K+1 provisional slots (preemption)."""
    import torch
    _check(block_table, "block_table", 2, torch.int32)
    for t, n in ((seq_lens, "seq_lens"), (free_stack, "free_stack"), (free_top, "free_top"),
                 (status, "status")):
        _check(t, n, 1, torch.int32)
    B, MB = block_table.shape
    st = lib().kv_evict_provisional(_ptr(block_table), _ptr(seq_lens), num_blocks, block_size, B,
                                    K, MB, _ptr(free_stack), _ptr(free_top), _ptr(status),
                                    _stream(stream))
    if st != SPEC_OK:
        raise SpecError("kv_evict_provisional", st)


def kv_commit_rollback(block_table, seq_lens, num_accepted, prov_blocks, kv_pool, free_stack,
                       free_top, status, *, K: int, block_size: int, stream=None,
                       slot_map=None) -> None:
    """Commit the accepted provisional slots. kv_pool: [num_blocks, layers, 2, block_size,
    heads, head_dim] (any element type); tables int32 as in include/specverify.h.
    slot_map: optional [B, K+1] int32 (a tree draft's kept slots)."""
    import torch
    if slot_map is not None:
        _check(slot_map, "slot_map", 2, torch.int32)
    for t, n in ((block_table, "block_table"), (prov_blocks, "prov_blocks")):
        _check(t, n, 2, torch.int32)
    for t, n in ((seq_lens, "seq_lens"), (num_accepted, "num_accepted"),
                 (free_stack, "free_stack"), (free_top, "free_top"), (status, "status")):
        _check(t, n, 1, torch.int32)
    _check(kv_pool, "kv_pool", 6)
    NB, NL, two, bs, H, D = kv_pool.shape
    if two != 2 or bs != block_size:
        raise ValueError("kv_pool must be [num_blocks, layers, 2, block_size, heads, head_dim]")
    B, MB = block_table.shape
    P = prov_blocks.shape[1]
    st = lib().kv_commit_rollback(
        _ptr(block_table), _ptr(seq_lens), _ptr(num_accepted), _ptr(prov_blocks), _ptr(kv_pool),
        NB, NL, H, D, kv_pool.element_size(), block_size, B, K, MB, P, _ptr(free_stack),
        _ptr(free_top), _ptr(status), _stream(stream), _ptr(slot_map))
    if st != SPEC_OK:
        raise SpecError("kv_commit_rollback", st)


def spec_selftest_ex2(lo: float, hi: float, *, stream=None) -> float:
    """Maximum relative error of the hardware exp2 over all fp32 arguments in [lo, hi]."""
    import torch
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    st = lib().spec_selftest_ex2(ctypes.c_float(lo), ctypes.c_float(hi), _ptr(out),
                                 _stream(stream))
    if st != SPEC_OK:
        raise SpecError("spec_selftest_ex2", st)
    return float(out.item())


# ------------------------------------------------------------------ conveniences
def verify(target_logits, draft_logits, draft_tokens, uniforms, temperature: float, *,
           stream=None, with_info: bool = False):
    """Allocates the outputs on the logits' device and runs spec_verify_sample.
    Returns (out_tokens [B,K+1], num_accepted [B]) (+ (row_info, err) if with_info)."""
    import torch
    B, K1, _ = target_logits.shape
    dev = target_logits.device
    out = torch.empty((B, K1), dtype=torch.int32, device=dev)
    n = torch.empty((B,), dtype=torch.int32, device=dev)
    info = torch.empty((B,), dtype=torch.int32, device=dev) if with_info else None
    err = torch.zeros((1,), dtype=torch.int32, device=dev) if with_info else None
    spec_verify_sample(target_logits, draft_logits, draft_tokens, uniforms, temperature, out, n,
                       stream=stream, err_flag=err, row_info=info)
    return (out, n, info, err) if with_info else (out, n)


def verify_host(target_logits, draft_logits, draft_tokens, uniforms, temperature: float, *,
                device="cuda", stream=None):
    """End-to-end call on HOST (CPU, ideally pinned) tensors: copies the inputs to the
    device, verifies, and copies (out_tokens, num_accepted) back to the host."""
    import torch
    s = stream or torch.cuda.current_stream()
    with torch.cuda.stream(s):
        t = target_logits.to(device, non_blocking=True)
        d = draft_logits.to(device, non_blocking=True) if draft_logits is not None else None
        k = draft_tokens.to(device, non_blocking=True)
        u = uniforms.to(device, non_blocking=True)
        out, n = verify(t, d, k, u, temperature, stream=s)
        out_h = out.to("cpu", non_blocking=False)
        n_h = n.to("cpu", non_blocking=False)
    return out_h, n_h


class HostVerifier:
    """End-to-end sampling verification of batches held in HOST memory (pinned).

    The batch rows are copied to preallocated device buffers in `chunks` row
    chunks on a copy stream; chunk c is verified (spec_verify_sample on its
    rows) as soon as its copy lands, while the next chunk is still in flight,
    so the verification hides behind the transfer. Outputs stay on the device
    (`out_tokens`, `num_accepted`); `to_host` copies them into pinned host
    tensors on the same stream.
    """

    def __init__(self, B: int, K: int, V: int, *, dtype=None, chunks: int = 8, device="cuda"):
        import torch
        dtype = dtype or torch.bfloat16
        self.B, self.K, self.V = B, K, V
        self.chunks = max(1, min(chunks, B))
        d = torch.device(device)
        self.target = torch.empty((B, K + 1, V), dtype=dtype, device=d)
        self.draft = torch.empty((B, K, V), dtype=dtype, device=d)
        self.tokens = torch.empty((B, K), dtype=torch.int32, device=d)
        self.uniforms = torch.empty((B, K + 1), dtype=torch.float32, device=d)
        self.out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=d)
        self.num_accepted = torch.empty((B,), dtype=torch.int32, device=d)
        self.copy_stream = torch.cuda.Stream(device=d)
        self.events = [torch.cuda.Event() for _ in range(self.chunks)]
        step = -(-B // self.chunks)
        self.bounds = [(r0, min(B, r0 + step)) for r0 in range(0, B, step)]

    def __call__(self, target_h, draft_h, tokens_h, uniforms_h, temperature: float, *,
                 stream=None):
        import torch
        main = stream or torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(main)                      # earlier work on the buffers is ordered first
        cs = self.copy_stream
        cs.wait_event(start)
        with torch.cuda.stream(cs):
            for (r0, r1), ev in zip(self.bounds, self.events):
                self.target[r0:r1].copy_(target_h[r0:r1], non_blocking=True)
                self.draft[r0:r1].copy_(draft_h[r0:r1], non_blocking=True)
                self.tokens[r0:r1].copy_(tokens_h[r0:r1], non_blocking=True)
                self.uniforms[r0:r1].copy_(uniforms_h[r0:r1], non_blocking=True)
                ev.record(cs)
        for (r0, r1), ev in zip(self.bounds, self.events):
            main.wait_event(ev)
            spec_verify_sample(self.target[r0:r1], self.draft[r0:r1], self.tokens[r0:r1],
                               self.uniforms[r0:r1], temperature, self.out_tokens[r0:r1],
                               self.num_accepted[r0:r1], stream=main)
        return self.out_tokens, self.num_accepted

    def to_host(self, out_h, n_h, *, stream=None):
        """Copies the outputs into host tensors (pinned for an asynchronous copy)."""
        import torch
        main = stream or torch.cuda.current_stream()
        with torch.cuda.stream(main):
            out_h.copy_(self.out_tokens, non_blocking=True)
            n_h.copy_(self.num_accepted, non_blocking=True)

