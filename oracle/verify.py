"""fp64 restatement of the verifier's accept/reject step (test infrastructure only).

Notation follows "aiengineeringfromscratch.com - Speculative decoding and
EAGLE-3", section "Variant: Leviathan rejection sampling": q is the verifier
(target) distribution, p the draft distribution, d ~ p the draft token.
The verifier returns q_1..q_{N+1}; here positions are 0-based, so the K draft
positions are 0..K-1 and the bonus distribution is target row K.

All arithmetic is float64. Logits arrive as float32 values (bf16 and float32
both widen exactly); the temperature is the float32 the library receives,
widened exactly (`temperature64`).
"""
from __future__ import annotations

import numpy as np


def temperature64(T) -> float:
    """The temperature as the library sees it: a float32, widened exactly."""
    return float(np.float32(T))


def log_softmax(z, T64: float) -> np.ndarray:
    """log softmax(z / T) over the last axis.

    Max subtraction, then log of the sum of exponentials. A logit of -inf has
    probability 0 (log -inf). Temperature scales both target and draft logits
    (one T for both).
    """
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    with np.errstate(invalid="ignore"):
        a = (z - m) / T64
    s = np.sum(np.exp(a), axis=-1, keepdims=True)
    return a - np.log(s)


def softmax(z, T64: float) -> np.ndarray:
    """softmax(z / T) over the last axis: exp((z - max)/T) / sum."""
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    with np.errstate(invalid="ignore"):
        e = np.exp((z - m) / T64)
    return e / np.sum(e, axis=-1, keepdims=True)


def accept_test(log_q_d, log_p_d, u) -> np.ndarray:
    """The rejection rule (lesson, "Step 1: the rejection rule").

    If p(d) <= 0 the draft token is accepted. Otherwise it is accepted iff
    u < min(1, q(d)/p(d)), with a strict comparison. The ratio is formed from
    log-probabilities, exp(log q(d) - log p(d)), so neither factor underflows.
    """
    log_q_d = np.asarray(log_q_d, np.float64)
    log_p_d = np.asarray(log_p_d, np.float64)
    u = np.asarray(u, np.float64)
    p_zero = np.isneginf(log_p_d)
    with np.errstate(invalid="ignore", over="ignore"):
        ratio = np.exp(np.where(p_zero, 0.0, log_q_d - log_p_d))
    return p_zero | (u < np.minimum(1.0, ratio))


def residual(q, p) -> np.ndarray:
    """Residual distribution (lesson, "Step 2: residual distribution"), unnormalised.

    r = max(0, q - p) elementwise. If the residual mass sum(r) is exactly 0 the
    lesson returns q itself, and so does this. Normalisation by sum(r) is left to
    `inverse_cdf`, which compares u * sum(r) with the cumulative sum.
    """
    q = np.asarray(q, np.float64)
    p = np.asarray(p, np.float64)
    r = np.maximum(q - p, 0.0)
    s = np.sum(r, axis=-1, keepdims=True)
    return np.where(s == 0.0, q, r)


def inverse_cdf(w, u) -> tuple[np.ndarray, np.ndarray]:
    """Draw one index per row from the unnormalised weights w with one uniform u.

    The drawn index is the smallest v with u * sum(w) < sum_{x <= v} w_x (token-
    index order, strict <). If rounding leaves no such v, the last index with
    positive weight is taken. Also returns the distance from u to the nearest
    boundary of the normalised CDF, which is the nearer of the drawn index's two
    boundaries.
    """
    w = np.asarray(w, np.float64)
    u = np.asarray(u, np.float64)
    c = np.cumsum(w, axis=-1)
    total = c[..., -1]
    t = u * total
    hit = t[..., None] < c
    any_hit = hit.any(axis=-1)
    first = np.argmax(hit, axis=-1)
    last_pos = w.shape[-1] - 1 - np.argmax((w > 0)[..., ::-1], axis=-1)
    idx = np.where(any_hit, first, last_pos)
    hi = np.take_along_axis(c, idx[..., None], axis=-1)[..., 0]
    lo = hi - np.take_along_axis(w, idx[..., None], axis=-1)[..., 0]
    with np.errstate(invalid="ignore", divide="ignore"):
        dist = np.minimum(np.abs(u - lo / total), np.abs(hi / total - u))
    return idx.astype(np.int64), dist


def _leading_true(mask: np.ndarray) -> np.ndarray:
    """Number of leading True values per row (the first rejection index j)."""
    K = mask.shape[1]
    return np.where(mask.all(axis=1), K, np.argmin(mask, axis=1)).astype(np.int64)


def verify_sample(target, draft, tokens, uniforms, temperature, *, row_chunk: int = 8) -> dict:
    """Sampling-mode verification of one batch (lesson, "Step 3: one full speculative step").

    For each row: test positions 0..K-1 in order with u[i]; at the first
    rejection j draw the correction from residual(q_j, p_j) with u[K]; if all
    K are accepted draw the bonus token from q_K with u[K]. Outputs:
      out_tokens [B, K+1]: d_0..d_{n-1}, then the correction or bonus token, then -1;
      num_accepted [B]: n.
    Diagnostics: q_at_d / p_at_d [B, K] (probabilities of the draft tokens),
    accept_margin [B, K] = |u_i - min(1, ratio_i)| for the tests performed
    (NaN after the first rejection), sample_margin [B] = distance of u[K] from the
    nearest boundary of the final draw's CDF.
    """
    T64 = temperature64(temperature)
    if T64 == 0.0:
        return verify_greedy(target, tokens)
    target = np.asarray(target)
    draft = np.asarray(draft)
    tokens = np.asarray(tokens, np.int64)
    uniforms = np.asarray(uniforms, np.float64)
    B, K1, V = target.shape
    K = K1 - 1
    out = np.full((B, K1), -1, np.int64)
    n_out = np.zeros(B, np.int64)
    q_at_d = np.zeros((B, K))
    p_at_d = np.zeros((B, K))
    a_margin = np.full((B, K), np.nan)
    s_margin = np.zeros(B)
    pos = np.arange(K)
    for b0 in range(0, B, row_chunk):
        b1 = min(B, b0 + row_chunk)
        rows = np.arange(b1 - b0)
        zt = target[b0:b1]
        zd = draft[b0:b1]
        tok = tokens[b0:b1]
        u = uniforms[b0:b1]
        lq = log_softmax(zt[:, :K], T64)
        lp = log_softmax(zd, T64)
        lq_d = lq[rows[:, None], pos[None, :], tok]
        lp_d = lp[rows[:, None], pos[None, :], tok]
        del lq, lp
        acc = accept_test(lq_d, lp_d, u[:, :K])
        n = _leading_true(acc)
        # distribution of the final draw
        j = np.minimum(n, K - 1)
        r = residual(softmax(zt[rows, j], T64), softmax(zd[rows, j], T64))
        bonus = softmax(zt[:, K], T64)
        w = np.where((n < K)[:, None], r, bonus)
        tok_final, dist = inverse_cdf(w, u[:, K])
        out[b0:b1, :K] = np.where(pos[None, :] < n[:, None], tok, -1)
        out[b0 + rows, n] = tok_final
        n_out[b0:b1] = n
        q_at_d[b0:b1] = np.exp(lq_d)
        p_at_d[b0:b1] = np.exp(lp_d)
        with np.errstate(invalid="ignore", over="ignore"):
            ratio = np.minimum(1.0, np.exp(lq_d - lp_d))
        performed = pos[None, :] <= np.minimum(n, K - 1)[:, None]
        a_margin[b0:b1] = np.where(performed, np.abs(u[:, :K] - ratio), np.nan)
        s_margin[b0:b1] = dist
    return dict(out_tokens=out, num_accepted=n_out, q_at_d=q_at_d, p_at_d=p_at_d,
                accept_margin=a_margin, sample_margin=s_margin)


def verify_greedy(target, tokens) -> dict:
    """Greedy verification ("devpost.com - phoenix", section "What it does").

    g_i = argmax of target row i over raw logits, ties to the lowest index
    (temperature does not change an argmax). n = number of leading positions
    with d_i == g_i; the emitted tokens are d_0..d_{n-1}, g_n, then -1.

    Unusable input (the pages are silent; same reading as verify_tree_greedy):
    a row with a NaN has no argmax and never matches a draft token; if the
    step uses it (row n, the first position not accepted, or row K after K
    acceptances) the batch row is an error. A draft token outside [0, V) is an
    error too. An error row has out_tokens all -1 and num_accepted -1. A row of
    equal values (all -inf included) has argmax 0 by the lowest-index rule.
    """
    target = np.asarray(target)
    tokens = np.asarray(tokens, np.int64)
    B, K1, V = target.shape
    K = K1 - 1
    rows = np.arange(B)
    bad_row = np.isnan(target).any(axis=-1)
    g = np.argmax(target.astype(np.float64), axis=-1)
    n = _leading_true((tokens == g[:, :K]) & ~bad_row[:, :K])
    error = bad_row[rows, n] | ((tokens < 0) | (tokens >= V)).any(axis=1)
    out = np.full((B, K1), -1, np.int64)
    out[:, :K] = np.where(np.arange(K)[None, :] < n[:, None], tokens, -1)
    out[rows, n] = g[rows, n]
    out[error] = -1
    n = np.where(error, -1, n)
    return dict(out_tokens=out, num_accepted=n, argmax=g)


def tree_survivors(g, bad_row, par, tok):
    """Survival and depth of every node of one tree, parents first.

    Node i is consistent when its token equals g of its parent's row (row
    p + 1, row 0 for a root child) and that row is usable; it survives when it
    and every ancestor are consistent. Depth 1 for a root child.
    """
    N = len(par)
    alive = np.zeros(N, bool)
    depth = np.zeros(N, np.int64)
    for i in range(N):
        p = int(par[i])
        up_ok = p < 0 or alive[p]
        alive[i] = up_ok and not bad_row[p + 1] and tok[i] == g[p + 1]
        depth[i] = 1 if p < 0 else depth[p] + 1
    return alive, depth


def tree_kept_node(alive, depth) -> int:
    """End of the kept path: the deepest survivor, lowest index among equally
    deep ones; -1 when nothing survives."""
    best = -1
    for i in range(len(alive)):
        if alive[i] and (best < 0 or depth[i] > depth[best]):
            best = i
    return best


def tree_path(par, node) -> list:
    """Nodes from the root's child down to `node` (empty for -1)."""
    path = []
    while node >= 0:
        path.append(node)
        node = int(par[node])
    return path[::-1]


def verify_tree_greedy(target, parents, tokens) -> dict:
    """Greedy verification of a draft tree, one verifier pass over all nodes.

    Sources: "thakicloud.com - Speculative decoding: when it loses", section
    "Grading every branch in one pass": the drafter's branches are flattened into one
    sequence under an ancestor-only mask, the target grades every node in one
    forward pass, and the longest surviving path is kept; the lesson's
    "EAGLE-2" entry and its tree exercise (a [2, 2, 2] tree, one verifier
    run, the surviving path wins); "devpost.com - phoenix", "What it does"
    for the greedy acceptance of one token.

    Layout (reading): N nodes in topological order, parents[b, i] in
    [-1, i) (-1: a child of the last committed token); target row 0 is the
    distribution after the committed prefix and row 1 + i the one after
    node i. Node i is consistent when its token equals the argmax of its
    parent's row (row 0 for the root's children); it survives when it and all
    its ancestors are consistent. The kept path ends at the deepest survivor,
    the lowest node index among equally deep ones (depth 0: no survivor), and
    the step emits the path's tokens and then the argmax of the last kept
    node's row. slots[p] is the provisional KV slot of kept position p: 0 for
    the last committed token, 1 + node for the node at depth p.

    An invalid tree or token, or a row with a NaN whose argmax the result
    uses (row 0 and the rows of survivors), makes the row an error: outputs
    -1 and num_accepted -1. As in verify_greedy, a row of equal values (all
    -inf included) has argmax 0 by the lowest-index rule.
    """
    target = np.asarray(target, np.float64)
    parents = np.asarray(parents, np.int64)
    tokens = np.asarray(tokens, np.int64)
    B, N1, V = target.shape
    N = N1 - 1
    out = np.full((B, N1), -1, np.int64)
    slots = np.full((B, N1), -1, np.int64)
    n_out = np.full(B, -1, np.int64)
    for b in range(B):
        rows = target[b]
        bad_row = np.isnan(rows).any(axis=1)
        g = np.argmax(np.where(bad_row[:, None], 0.0, rows), axis=1)
        par, tok = parents[b], tokens[b]
        if any(not (0 <= tok[i] < V and -1 <= par[i] < i) for i in range(N)):
            continue
        alive, depth = tree_survivors(g, bad_row, par, tok)
        if bad_row[0] or any(alive[i] and bad_row[i + 1] for i in range(N)):
            continue
        path = tree_path(par, tree_kept_node(alive, depth))
        n = len(path)
        out[b, :n] = tok[path]
        out[b, n] = g[0] if n == 0 else g[path[-1] + 1]
        slots[b, 0] = 0
        slots[b, 1:n + 1] = np.asarray(path, np.int64) + 1
        n_out[b] = n
    return dict(out_tokens=out, num_accepted=n_out, slots=slots)


def verify_step(target, draft, tokens, uniforms, temperature, **kw) -> dict:
    """T == 0 selects greedy mode (the pages list temperature 0.0 as greedy)."""
    if temperature64(temperature) == 0.0:
        return verify_greedy(target, tokens)
    return verify_sample(target, draft, tokens, uniforms, temperature, **kw)


def acceptance_counters(num_accepted, K: int) -> np.ndarray:
    """Per-position acceptance statistics of a batch of verified rows.

    The quickscale.ai page ("Quand et pourquoi utiliser le speculative
    decoding") defines the per-position acceptance rate a_i and the mean
    acceptance length; the lesson's expected-acceptance formula counts the
    tokens one step emits (accepted drafts plus the correction or bonus).
    For a row with n accepted drafts (n = -1: a row with an error, not
    counted): draft position i is tested iff i <= n (and i < K) and accepted
    iff i < n; the step emits n + 1 tokens.

    Returns int64 [2K + 2]: tested[0..K), accepted[0..K), rows, tokens emitted.
    """
    n = np.asarray(num_accepted, np.int64).ravel()
    n = n[n >= 0]
    out = np.zeros(2 * K + 2, np.int64)
    for i in range(K):
        out[i] = int(np.sum(n >= i))
        out[K + i] = int(np.sum(n > i))
    out[2 * K] = n.size
    out[2 * K + 1] = int(np.sum(n + 1))
    return out

