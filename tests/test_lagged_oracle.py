"""Pins of oracle.commit_verify (commit the previous step, verify the next),
without a GPU.

The step is tied to one uninterrupted run of the recurrence over the
concatenated accepted rows, a route that shares none of its bookkeeping (no
pool, no slot gather or scatter, no split of the sequence): the states after
a chain of steps and every step's outputs must agree bit for bit, since both
routes apply the same float64 operations to every token in the same order.
"""
import numpy as np
import pytest

import oracle
from speculative_decode_gated_gb300 import inputs


def step(seed, layer, lengths, accepted):
    """One step of the same requests (slot ids come from the seed's metadata
    stream; the tokens differ with `layer`)."""
    return inputs.make_custom(batch=len(lengths), heads=2, dk=16, dv=8, lengths=lengths,
                              pool_slots=7, qkv_dtype="fp32", seed=seed, layer=layer,
                              accepted=np.asarray(accepted, np.int32), name=f"step{layer}")


class Concat:
    """Request r's rows: the accepted prefixes of `done` steps, then (optionally)
    the drafts of `last`; one problem run from the original checkpoints."""

    def __init__(self, done, last, s0):
        p0 = done[0] if done else last
        self.heads, self.dk, self.dv, self.gate = p0.heads, p0.dk, p0.dv, "alpha"
        self.batch = p0.batch
        rows = {name: [] for name in ("q", "k", "v", "alpha", "beta")}
        lens, acc = [], []
        for r in range(self.batch):
            n = 0
            for p in done:
                c0, a = int(p.cu_seqlens[r]), int(p.accepted[r])
                for name in ("k", "v", "alpha", "beta"):
                    rows[name].append(getattr(p, name)[c0:c0 + a])
                rows["q"].append(np.zeros_like(p.q[c0:c0 + a]))
                n += a
            acc.append(n)
            if last is not None:
                c0, T = int(last.cu_seqlens[r]), int(last.lengths[r])
                for name in ("q", "k", "v", "alpha", "beta"):
                    rows[name].append(getattr(last, name)[c0:c0 + T])
                n += T
            lens.append(n)
        for name, xs in rows.items():
            setattr(self, name, np.concatenate(xs))
        self.cu_seqlens = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        self.lengths = np.asarray(lens)
        self.max_T = max(max(lens), 1)
        self.accepted = np.asarray(acc, np.int64)
        self.s0 = s0


SHORT = ([[5, 1, 4], [3, 6, 2], [4, 4, 6]], [[2, 0, 4], [3, 1, 0], [0, 4, 6]])
# drafts longer than one 16-row chunk: commit points inside a chunk, on a
# chunk boundary (16, 32) and at the full length
LONG = ([[40, 17, 33], [16, 35, 20], [32, 9, 48]], [[37, 0, 16], [16, 35, 3], [32, 9, 0]])


def chain(seed=3, lens_accs=SHORT):
    lens, accs = lens_accs
    steps = [step(seed, i, l, a) for i, (l, a) in enumerate(zip(lens, accs))]
    rng = np.random.default_rng(11)
    p0 = steps[0]
    pool = rng.standard_normal((p0.pool_slots, p0.heads, p0.dk, p0.dv)) * 0.1
    return steps, pool


@pytest.mark.parametrize("lens_accs", [SHORT, LONG], ids=["short", "multichunk"])
def test_chain_equals_one_run_over_the_accepted_rows(lens_accs):
    steps, pool0 = chain(lens_accs=lens_accs)
    p0 = steps[0]
    s0 = oracle.gather_s0(pool0, p0.slot_ids, p0.heads).reshape(p0.batch, p0.heads, p0.dk, p0.dv)
    pool, prev = pool0, None
    for k, p in enumerate(steps):
        pool, o = oracle.commit_verify(prev, p, pool)
        # outputs: the accepted rows of the earlier steps, then this step's drafts
        ref = Concat(steps[:k], p, s0)
        o_ref, _ = oracle.run_units(ref, want_state=False)
        for r in range(p.batch):
            c0, T, n = int(p.cu_seqlens[r]), int(p.lengths[r]), int(ref.accepted[r])
            for h in range(p.heads):
                assert np.array_equal(o[c0:c0 + T, h], o_ref[r * p.heads + h, n:n + T])
        prev = p
    pool = oracle.commit(prev, pool)  # the last step's prefix
    ref = Concat(steps, None, s0)
    _, s_ref = oracle.run_units(ref, want_o=False)
    for r in range(p0.batch):
        slot = int(p0.slot_ids[r])
        for h in range(p0.heads):
            want = s_ref[r * p0.heads + h] if ref.accepted[r] > 0 else pool0[slot, h]
            assert np.array_equal(pool[slot, h], want)


def test_first_step_commits_nothing():
    steps, pool = chain(seed=5)
    p = steps[0]
    after, o = oracle.commit_verify(None, p, pool)
    assert np.array_equal(after, pool)
    s0 = oracle.gather_s0(pool, p.slot_ids, p.heads)
    o_units, _ = oracle.run_units(p, s0=s0, want_state=False)
    assert np.array_equal(o, oracle.scatter_outputs(p, np.arange(p.batch * p.heads), o_units))


def test_nothing_accepted_is_a_plain_verify():
    steps, pool = chain(seed=6)
    prev = step(6, 0, [5, 1, 4], [0, 0, 0])
    after, o = oracle.commit_verify(prev, steps[1], pool)
    assert np.array_equal(after, pool)
    _, o_first = oracle.commit_verify(None, steps[1], pool)
    assert np.array_equal(o, o_first)


def test_other_requests_are_rejected():
    steps, pool = chain()
    other = inputs.make_custom(batch=3, heads=2, dk=16, dv=8, lengths=[2, 2, 2], pool_slots=7,
                               qkv_dtype="fp32", seed=99, name="other")
    with pytest.raises(ValueError):
        oracle.commit_verify(other, steps[1], pool)
