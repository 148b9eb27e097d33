"""Plain fp64 CPU oracle for speculative-decoding verification.

TEST INFRASTRUCTURE ONLY. Only the tests, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline leg import this package. The CUDA library never calls
it and shares no code, header, table or constant with it; the two meet only on
the seeded inputs made by `synth`.

Every function restates the method as the pages give it, step by step, in
float64 NumPy (library routines: exp, log, cumsum, argmax). Sources:

* "aiengineeringfromscratch.com - Speculative decoding and EAGLE-3"
  (machine-translated lesson), sections "Variant: Leviathan rejection sampling"
  (accept with probability min(1, q(d)/p(d)), residual (q - p)+ / ||(q - p)+||_1,
  bonus token from q_{N+1}), "Step 1: the rejection rule" (p <= 0 accepts,
  strict u < min(1, q/p)), "Step 2: residual distribution" (zero residual
  mass falls back to q), "Step 4: KV rollback accounting" (logical length
  becomes prefix + j + 1), and "What decides the speed-up" (E[accepted]).
* "devpost.com - phoenix", section "What it does": greedy verification keeps
  tokens up to the first disagreement with the target's argmax and emits the
  target's token there; output identical to the target alone.
* "sglang_spec_decode" README, section on the provisional KV layer:
  provisional slots are committed or freed, with no block leaked or freed twice.

Readings where the pages are silent (each listed in the design notes):
q = target, p = draft; one temperature for both; T == 0 selects greedy; ties
in argmax go to the lowest index; K+1 uniforms per row, u[i] for test i and
u[K] for the single final draw; the final draw is an inverse CDF in token-index
order with a strict comparison against the unnormalised cumulative sum.

Parity status: every function here is pinned by tests in `tests/test_oracle_*.py`
against hand-worked examples, closed forms, the losslessness theorem, or
library special cases.
"""
from .verify import (  # noqa: F401
    temperature64,
    log_softmax,
    softmax,
    accept_test,
    residual,
    inverse_cdf,
    verify_sample,
    verify_greedy,
    verify_tree_greedy,
    tree_survivors,
    tree_kept_node,
    tree_path,
    verify_step,
    acceptance_counters,
)
from .kv import kv_commit, kv_truncate_inplace, pool_invariant_ok  # noqa: F401
from .filters import filter_threshold, filter_thresholds, apply_threshold  # noqa: F401
