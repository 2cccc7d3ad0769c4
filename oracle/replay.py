"""ReplaySSM buffer: outputs and commits from a checkpoint plus buffered rows
(CPU oracle).

TEST INFRASTRUCTURE, like the rest of this package: only `tests/`,
`__graft_entry__.smoke()` and the CPU baseline leg of `bench.py` use it.

ReplaySSM keeps a checkpoint of the recurrent state next to a small buffer of
recent inputs, computes outputs from the checkpoint and the buffered inputs,
writes the full checkpoint only at periodic flushes, and rolls a rejection
back by moving the buffer pointer so that it keeps the accepted prefix (OCRia
write-up, section "Make speculative verification cheaper").

Here each pool slot s has a buffer of C rows (k, v, alpha, beta, with the
layout of the token arrays) and a length n_s: the rows accepted since the
slot's last flush.  The step's draft rows of request r sit at buffer rows
n_s + [0, T_r) of its slot; its q rows are the usual q rows cu[r] + [0, T_r).

  verify:  o_t of the draft rows = the recurrence from the checkpoint over
           buffer rows [0, n_s + T_r), outputs of its last T_r rows.
  commit:  keep = n_s + a_r.  When keep + max_T > C (a full next draft would
           not fit) the slot is flushed: checkpoint <- the state after buffer
           rows [0, keep), n_s <- 0.  Otherwise only n_s <- keep (rejected
           rows are overwritten by the next step's drafts).
The flush rule is this oracle's reading of "periodic"; the recurrence itself
is the C oracle's, run over the replayed rows.

Parity unpinned: none.  Pinned by `tests/test_replay_oracle.py`.
"""
from __future__ import annotations

import numpy as np


class _Seq:
    """A problem whose request r is the replayed row sequence of one request."""

    def __init__(self, prob, ks, vs, als, bes, qs, accepted, s0):
        self.heads, self.dk, self.dv = prob.heads, prob.dk, prob.dv
        self.gate = getattr(prob, "gate", "alpha")
        self.batch = len(ks)
        lens = np.array([len(x) for x in ks], dtype=np.int64)
        self.cu_seqlens = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        self.max_T = int(lens.max()) if len(lens) else 0
        cat = (lambda xs, tail: np.concatenate(xs) if xs else np.zeros((0,) + tail))
        self.k = cat(ks, (prob.heads, prob.dk))
        self.v = cat(vs, (prob.heads, prob.dv))
        self.alpha = cat(als, (prob.heads,))
        self.beta = cat(bes, (prob.heads,))
        self.q = cat(qs, (prob.heads, prob.dk))
        self.accepted = np.asarray(accepted, dtype=np.int64)
        self.s0 = s0


def _slot_rows(buf, slot, n):
    C = int(buf["capacity"])
    lo = slot * C
    return (buf["k"][lo:lo + n], buf["v"][lo:lo + n], buf["alpha"][lo:lo + n],
            buf["beta"][lo:lo + n])


def _lengths(prob, buf):
    return np.array([int(buf["len_in"][int(s)]) for s in prob.slot_ids], dtype=np.int64)


def replay_verify(prob, buf, pool, threads: int = 1) -> np.ndarray:
    """o of every draft row, float64 [N_tok][H][dv].  `pool` holds the checkpoints
    ([slots][H][dk][dv]); `buf` has capacity, k, v, alpha, beta ([slots*C][H][...])
    and len_in ([slots])."""
    from . import gather_s0, run_units
    n = _lengths(prob, buf)
    T = prob.lengths.astype(np.int64)
    if np.any(n + T > int(buf["capacity"])) or np.any(n < 0):
        raise ValueError("buffered rows plus drafts exceed the capacity")
    ks, vs, als, bes, qs = [], [], [], [], []
    for r in range(prob.batch):
        k, v, a, b = _slot_rows(buf, int(prob.slot_ids[r]), int(n[r] + T[r]))
        c0 = int(prob.cu_seqlens[r])
        q = np.concatenate([np.zeros((int(n[r]), prob.heads, prob.dk)),
                            prob.q[c0:c0 + int(T[r])]])
        ks.append(k), vs.append(v), als.append(a), bes.append(b), qs.append(q)
    s0 = gather_s0(pool, prob.slot_ids, prob.heads)
    seq = _Seq(prob, ks, vs, als, bes, qs, n + T, s0)
    o_seq, _ = run_units(seq, want_o=True, want_state=False, threads=threads)
    out = np.zeros((prob.n_tok, prob.heads, prob.dv))
    for u in range(prob.batch * prob.heads):
        r, h = divmod(u, prob.heads)
        c0 = int(prob.cu_seqlens[r])
        out[c0:c0 + int(T[r]), h] = o_seq[u, int(n[r]):int(n[r] + T[r])]
    return out


def replay_commit(prob, buf, pool, threads: int = 1):
    """(pool after, len_out, flushed): the commit step of every request.  len_out
    is len_in with the named slots updated; `flushed` is the boolean [B] flush
    decision.  Slots that are not flushed are left bit-identical."""
    from . import gather_s0, run_units
    C = int(buf["capacity"])
    n = _lengths(prob, buf)
    keep = n + prob.accepted.astype(np.int64)
    if np.any(keep > C) or np.any(n < 0):
        raise ValueError("kept rows exceed the capacity")
    flushed = keep + int(prob.max_T) > C
    out = np.array(pool, copy=True)
    len_out = np.array(buf["len_in"], dtype=np.int32, copy=True)
    for r in range(prob.batch):
        len_out[int(prob.slot_ids[r])] = 0 if flushed[r] else int(keep[r])
    rs = np.flatnonzero(flushed & (keep > 0))
    if rs.size:
        ks, vs, als, bes, qs = [], [], [], [], []
        for r in rs:
            k, v, a, b = _slot_rows(buf, int(prob.slot_ids[r]), int(keep[r]))
            ks.append(k), vs.append(v), als.append(a), bes.append(b)
            qs.append(np.zeros((int(keep[r]), prob.heads, prob.dk)))
        all_s0 = gather_s0(pool, prob.slot_ids, prob.heads).reshape(prob.batch, prob.heads,
                                                                   prob.dk, prob.dv)
        seq = _Seq(prob, ks, vs, als, bes, qs, keep[rs],
                   all_s0[rs].reshape(-1, prob.dk, prob.dv))
        _, s_acc = run_units(seq, want_o=False, want_state=True, threads=threads)
        for i, r in enumerate(rs):
            for h in range(prob.heads):
                out[int(prob.slot_ids[r]), h] = s_acc[i * prob.heads + h]
    return out, len_out, flushed
