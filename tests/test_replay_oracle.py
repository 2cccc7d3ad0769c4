"""Pins of the ReplaySSM buffer oracle (oracle.replay_verify / replay_commit),
without a GPU.

The replay is tied to the plain oracle (itself pinned) by routes that do not
share its row bookkeeping: with empty buffers it is the plain verify and
commit, bit for bit; over a sequence of steps it gives the outputs and the
final states of committing every step (flush each step) to float64 rounding;
rows past the drafts never matter and buffered rows always do; and the flush
bookkeeping follows its rule exactly.
"""
import numpy as np
import pytest

import oracle
from speculative_decode_gated_gb300 import inputs


def pool_with(prob, extra_slots_fill=0.5):
    rng = np.random.default_rng(7)
    pool = rng.standard_normal((prob.pool_slots, prob.heads, prob.dk, prob.dv)) * extra_slots_fill
    for r in range(prob.batch):
        pool[int(prob.slot_ids[r])] = prob.s0[r]
    return pool


def small(seed=1, **kw):
    spec = dict(batch=3, heads=2, dk=16, dv=8, T=5, pool_slots=5, qkv_dtype="fp32",
                accept="uniform", seed=seed)
    spec.update(kw)
    return inputs.make_custom(**spec)


def test_empty_buffers_are_the_plain_calls():
    prob = small()
    pool = pool_with(prob)
    # capacity large enough that nothing flushes
    buf = inputs.make_replay(prob, capacity=40, seed=3, len_in=np.zeros(prob.pool_slots))
    o = oracle.replay_verify(prob, buf, pool)
    assert np.array_equal(o, oracle.verify(prob))
    after, len_out, flushed = oracle.replay_commit(prob, buf, pool)
    assert not flushed.any()
    assert np.array_equal(after, pool)
    for r in range(prob.batch):
        assert len_out[prob.slot_ids[r]] == prob.accepted[r]
    # capacity = max_T: every slot that keeps a row flushes, which is the plain commit
    buf = inputs.make_replay(prob, capacity=prob.max_T, seed=3, len_in=np.zeros(prob.pool_slots))
    after, len_out, flushed = oracle.replay_commit(prob, buf, pool)
    assert np.array_equal(flushed, prob.accepted > 0)
    assert np.array_equal(after, oracle.commit(prob, pool))
    assert not len_out[prob.slot_ids].any()


def place_drafts(buf, prob):
    C = buf["capacity"]
    for r in range(prob.batch):
        s, c0, T = int(prob.slot_ids[r]), int(prob.cu_seqlens[r]), int(prob.lengths[r])
        lo = s * C + int(buf["len_in"][s])
        buf["k"][lo:lo + T] = prob.k[c0:c0 + T]
        buf["v"][lo:lo + T] = prob.v[c0:c0 + T]
        buf["alpha"][lo:lo + T] = prob.alpha[c0:c0 + T]
        buf["beta"][lo:lo + T] = prob.beta[c0:c0 + T]


@pytest.mark.parametrize("capacity", [7, 12, 23])
def test_steps_equal_committing_every_step(capacity):
    slots = np.array([3, 0, 4], dtype=np.int32)
    first = small(seed=50, slot_ids=slots)
    pool_a = pool_with(first)
    pool_b = pool_a.copy()
    H = first.heads
    buf = dict(capacity=capacity, len_in=np.zeros(first.pool_slots, np.int32),
               k=np.zeros((first.pool_slots * capacity, H, first.dk)),
               v=np.zeros((first.pool_slots * capacity, H, first.dv)),
               alpha=np.ones((first.pool_slots * capacity, H)),
               beta=np.zeros((first.pool_slots * capacity, H)))
    n_flush = n_keep = 0
    for step in range(8):
        prob = small(seed=60 + step, slot_ids=slots)
        units = np.arange(prob.units)
        # committing every step: verify and commit from the slots of pool_a
        s0 = oracle.gather_s0(pool_a, prob.slot_ids, H)
        o_seq, s_acc = oracle.run_units(prob, units, s0=s0)
        o_a = oracle.scatter_outputs(prob, units, o_seq)
        pool_a = oracle.commit_pool(pool_a, prob.slot_ids, prob.accepted, s_acc, H)
        # the buffer: drafts placed after the buffered rows, replayed from pool_b
        place_drafts(buf, prob)
        o_b = oracle.replay_verify(prob, buf, pool_b)
        scale = np.abs(o_a).max()
        assert np.abs(o_a - o_b).max() <= 1e-12 * scale
        pool_b, len_out, flushed = oracle.replay_commit(prob, buf, pool_b)
        n_flush += int(flushed.sum())
        n_keep += int((~flushed).sum())
        buf["len_in"] = len_out
    assert n_flush and n_keep, "the sequence must exercise both branches"
    # flush whatever is still buffered and compare the states
    final = small(seed=99, slot_ids=slots, T=capacity, accept="zero")
    pool_b, _, _ = oracle.replay_commit(final, buf, pool_b)
    for s in slots:
        assert np.abs(pool_a[s] - pool_b[s]).max() <= 1e-12 * np.abs(pool_a[s]).max()


def test_rows_past_the_drafts_never_matter_and_buffered_rows_do():
    prob = small(seed=5, accept="full")
    pool = pool_with(prob)
    buf = inputs.make_replay(prob, capacity=16, seed=8)
    o = oracle.replay_verify(prob, buf, pool)
    C = buf["capacity"]
    past = {key: np.array(buf[key], copy=True) for key in ("k", "v", "alpha", "beta")}
    for r in range(prob.batch):
        s = int(prob.slot_ids[r])
        lo = s * C + int(buf["len_in"][s]) + int(prob.lengths[r])
        past["k"][lo:(s + 1) * C] += 3.0
        past["beta"][lo:(s + 1) * C] = 0.7
    assert np.array_equal(oracle.replay_verify(prob, dict(buf, **past), pool), o)
    r = int(np.argmax(buf["len_in"][prob.slot_ids]))
    s = int(prob.slot_ids[r])
    assert buf["len_in"][s] > 0
    changed = {key: np.array(buf[key], copy=True) for key in ("k", "v", "alpha", "beta")}
    changed["v"][s * C] += 1.0
    o2 = oracle.replay_verify(prob, dict(buf, **changed), pool)
    c0 = int(prob.cu_seqlens[r])
    assert not np.allclose(o2[c0:c0 + int(prob.lengths[r])], o[c0:c0 + int(prob.lengths[r])])


def test_flush_bookkeeping():
    prob = small(seed=9, batch=4, pool_slots=7)
    pool = pool_with(prob)
    buf = inputs.make_replay(prob, capacity=11, seed=10)
    after, len_out, flushed = oracle.replay_commit(prob, buf, pool)
    named = set(int(s) for s in prob.slot_ids)
    for s in range(prob.pool_slots):
        if s not in named:
            assert len_out[s] == buf["len_in"][s]
            assert np.array_equal(after[s], pool[s])
    for r in range(prob.batch):
        s = int(prob.slot_ids[r])
        keep = int(buf["len_in"][s]) + int(prob.accepted[r])
        assert flushed[r] == (keep + prob.max_T > buf["capacity"])
        assert len_out[s] == (0 if flushed[r] else keep)
        if not flushed[r] or keep == 0:
            assert np.array_equal(after[s], pool[s])
        else:
            assert not np.array_equal(after[s], pool[s])


def test_rejects_overfull_buffers():
    prob = small(seed=11)
    pool = pool_with(prob)
    buf = inputs.make_replay(prob, capacity=8, seed=12)
    bad = dict(buf, len_in=np.full(prob.pool_slots, 4, np.int32))  # 4 + 5 > 8
    with pytest.raises(ValueError):
        oracle.replay_verify(prob, bad, pool)
