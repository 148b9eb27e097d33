"""Top-k / top-p filtering of a logit row before verification (test infrastructure only).

Source: "quickscale.ai - Quand et pourquoi utiliser le speculative decoding",
section "Influence du sampling": temperature, top-p and top-k are the
generation parameters that shape the distributions being verified (wider
settings lower the acceptance). The page does not define the filters; the
reading used here is the common one:

* temperature first (softmax(z / T)), then top-k, then top-p on the
  renormalised top-k distribution;
* top-k keeps every token whose logit is at least the k-th largest logit
  (ties at that value are all kept); k = 0 or k >= V disables it;
* top-p keeps every token whose logit is at least t*, the largest logit value
  t for which the probability of the tokens with logit >= t reaches p
  (again ties at t* are all kept); p >= 1 disables it;
* the filter is one logit threshold per row: tokens below it get logit -inf,
  i.e. probability 0, and the verification runs unchanged on the filtered
  target and draft rows (the same k and p for both).

All arithmetic is float64.
"""
from __future__ import annotations

import numpy as np


def filter_threshold(z, temperature: float, top_k: int = 0, top_p: float = 1.0) -> float:
    """The logit threshold of one row: keep tokens with z >= threshold.

    Returns -inf when nothing is filtered. Raises ValueError on NaN logits.
    """
    z = np.asarray(z, dtype=np.float64)
    if np.isnan(z).any():
        raise ValueError("NaN logit")
    V = z.size
    tau = -np.inf
    # top-k: the k-th largest logit value
    if 0 < top_k < V:
        tau = float(np.sort(z)[::-1][top_k - 1])
    # top-p on the renormalised top-k distribution
    if top_p < 1.0:
        T = float(np.float32(temperature))
        kept = z[z >= tau]
        m = float(np.max(kept))
        if np.isfinite(m):
            zs = np.sort(kept)[::-1]                    # descending
            cs = np.cumsum(np.exp((zs - m) / T))
            # the first sorted position whose cumulative mass reaches p; every
            # earlier tie group ends before it, so its value is t*
            i = int(np.argmax(cs >= float(np.float32(top_p)) * cs[-1]))
            tau = max(tau, float(zs[i]))
    return tau


def filter_thresholds(logits, temperature: float, top_k: int = 0, top_p: float = 1.0):
    """filter_threshold of every row of a [..., V] array (float64 thresholds)."""
    a = np.asarray(logits, dtype=np.float64)
    flat = a.reshape(-1, a.shape[-1])
    out = np.array([filter_threshold(r, temperature, top_k, top_p) for r in flat])
    return out.reshape(a.shape[:-1])


def apply_threshold(logits, thresholds):
    """Logits with every token below its row's threshold set to -inf."""
    a = np.asarray(logits, dtype=np.float64)
    t = np.asarray(thresholds, dtype=np.float64)[..., None]
    return np.where(a >= t, a, -np.inf)
