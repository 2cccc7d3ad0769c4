"""Accepted length of each request by greedy prefix match (CPU oracle).

TEST INFRASTRUCTURE, like the rest of this package: only `tests/`,
`__graft_entry__.smoke()` and the CPU baseline leg of `bench.py` use it.

Speculative decoding keeps the draft tokens that agree with the target model
and rolls the state back to the accepted prefix (OCRia write-up, sections
"Generate more tokens per target pass: speculative decoding" and "Make
speculative verification cheaper").  With greedy verification a position
agrees when the draft token equals the target model's own choice there, and
the accepted length is the number of agreeing positions before the first
disagreement.  The caller lines up both id arrays so that position t of
request r holds the draft token and the target's choice for that same token
(a position that is always kept is passed with equal ids).

Parity unpinned: none.  Pinned by `tests/test_accept_oracle.py`.
"""
from __future__ import annotations

import numpy as np


def accept_prefix(draft_ids, target_ids, cu_seqlens) -> np.ndarray:
    """accepted[r] = the largest a <= T_r with draft[c_r + t] == target[c_r + t]
    for every t < a, where c_r = cu_seqlens[r] and T_r = cu_seqlens[r+1] - c_r."""
    draft = [int(x) for x in np.asarray(draft_ids).ravel()]
    target = [int(x) for x in np.asarray(target_ids).ravel()]
    cu = [int(x) for x in np.asarray(cu_seqlens).ravel()]
    out = []
    for r in range(len(cu) - 1):
        a = 0
        for t in range(cu[r + 1] - cu[r]):
            if draft[cu[r] + t] != target[cu[r] + t]:
                break
            a += 1
        out.append(a)
    return np.array(out, dtype=np.int32)
