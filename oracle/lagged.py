"""Commit the previous step, then verify the next one (CPU oracle).

TEST INFRASTRUCTURE, like the rest of this package: only `tests/`,
`__graft_entry__.smoke()` and the CPU baseline leg of `bench.py` use it.

In an engine the accepted lengths of a step are known only after all its
layers have verified, so a layer's commit of step n - 1 can run just before
its verify of step n.  ReplaySSM rolls back by keeping the accepted prefix of
the drafts on top of the checkpoint (OCRia write-up, section "Make
speculative verification cheaper"); here that prefix is folded into the
checkpoint at the start of the next step, and the next drafts are verified
from the result:

  commit_verify(prev, prob, pool):
      after = pool with, for every request r with prev.accepted[r] > 0, its
              slot replaced by the state after the first prev.accepted[r]
              rows of the previous step (replayed from the slot's checkpoint);
      o     = the outputs of prob's drafts from the slots of `after`.

`prev` is the previous step's problem (same requests: batch, heads, slot ids)
or None for the first step, which commits nothing.  The recurrence is the C
oracle's (`run_units`), applied twice; nothing here does arithmetic.

Parity unpinned: none.  Pinned by `tests/test_lagged_oracle.py` against one
uninterrupted run of the recurrence over the concatenated accepted rows.
"""
from __future__ import annotations

import numpy as np


def commit_verify(prev, prob, pool: np.ndarray, threads: int = 1):
    """Returns (pool_after, o): float64 [slots][H][dk][dv] and [N_tok][H][dv]."""
    from . import commit, gather_s0, run_units, scatter_outputs

    if prev is not None:
        if (prev.batch != prob.batch or prev.heads != prob.heads
                or not np.array_equal(prev.slot_ids, prob.slot_ids)):
            raise ValueError("the previous step must have the same requests")
        after = commit(prev, pool, threads=threads)
    else:
        after = np.array(pool, dtype=np.float64, copy=True)
    units = np.arange(prob.batch * prob.heads)
    s0 = gather_s0(after, prob.slot_ids, prob.heads)
    o_units, _ = run_units(prob, s0=s0, want_o=True, want_state=False, threads=threads)
    return after, scatter_outputs(prob, units, o_units)
