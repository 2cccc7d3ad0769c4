"""GPU parity of the ReplaySSM buffer calls (gdn_replay_verify / gdn_replay_commit)
against the float64 oracle: single steps with buffered lengths from empty to
full and buffers of many chunks, then a run of steps in which the GPU's own
buffer lengths and pool carry from one step to the next (each step compared
with the oracle fed the GPU's state), and bad lengths."""
import os
import numpy as np
import pytest
import torch

import oracle
from parity import TOL, rel_err
from speculative_decode_gated_gb300 import binding, inputs, staging

pytestmark = pytest.mark.gpu

CASES = {
    "b3_h4_t16_c40": (dict(batch=3, heads=4, dk=128, dv=128, T=16, pool_slots=7,
                           accept="binom", seed=41), 40),
    "ragged_b5_h2_c32": (dict(batch=5, heads=2, dk=128, dv=128, lengths=[1, 16, 9, 4, 13],
                              pool_slots=9, accept="uniform", seed=42), 32),
    "b2_h2_t8_c200": (dict(batch=2, heads=2, dk=128, dv=128, T=8, pool_slots=3,
                           accept="full", seed=43), 200),
    "b4_h2_t16_c16": (dict(batch=4, heads=2, dk=128, dv=128, T=16, pool_slots=4,
                           accept="uniform", seed=44), 16),   # every buffer empty, capacity = T
}


def setup(name, len_in=None):
    spec, cap = CASES[name]
    prob = inputs.make_custom(name=name, qkv_dtype="bf16", **spec)
    buf = inputs.make_replay(prob, cap, seed=5, len_in=len_in)
    d = staging.DeviceProblem(prob, "cuda")
    r = staging.DeviceReplay(buf, prob.qkv_dtype)
    return prob, buf, d, r


@pytest.mark.parametrize("name", list(CASES))
def test_replay_verify_single_step(name):
    prob, buf, d, r = setup(name)
    pool = d.pool.double().cpu().numpy()
    want = oracle.replay_verify(prob, buf, pool)
    before = d.pool.view(torch.int32).clone()
    kbefore = r.k.clone()
    d.o.fill_(float("nan"))
    binding.gdn_replay_verify(d.c, r.c, d.o)
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(d.c) == 0
    assert torch.equal(d.pool.view(torch.int32), before)
    assert torch.equal(r.k, kbefore)
    err = rel_err(d.o.cpu().numpy(), want)
    assert err <= TOL, f"o: {err:.3e}"


@pytest.mark.parametrize("name", list(CASES))
def test_replay_commit_single_step(name):
    prob, buf, d, r = setup(name)
    pool = d.pool.double().cpu().numpy()
    want_pool, want_len, flushed = oracle.replay_commit(prob, buf, pool)
    before = d.pool.cpu().numpy()
    binding.gdn_replay_commit(d.c, r.c, d.accepted)
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(d.c) == 0
    assert np.array_equal(r.len_out.cpu().numpy(), want_len)
    after = d.pool.cpu().numpy()
    flushed_slots = {int(prob.slot_ids[i]) for i in np.flatnonzero(flushed)}
    for s in range(prob.pool_slots):
        if s in flushed_slots:
            err = rel_err(after[s], want_pool[s])
            assert err <= TOL, f"slot {s}: {err:.3e}"
        else:
            assert np.array_equal(after[s].view(np.int32), before[s].view(np.int32))


def test_replay_steps_carry_state():
    """Seven steps of one request set: drafts placed in the buffer on the device,
    verify, commit, swap.  Each step is checked against the oracle fed the
    GPU's pool and lengths of that step; both branches of the flush rule occur."""
    spec, cap = dict(batch=4, heads=2, dk=128, dv=128, T=16, pool_slots=6, accept="binom"), 48
    slots = np.array([5, 1, 3, 0], dtype=np.int32)
    first = inputs.make_custom(name="steps", qkv_dtype="bf16", seed=70, slot_ids=slots, **spec)
    buf0 = inputs.make_replay(first, cap, seed=6, len_in=np.zeros(6, np.int32))
    r = staging.DeviceReplay(buf0, "bf16")
    pool = staging.new_pool(6, 2, 128, 128, "cuda", fill="zero")
    staging.place_checkpoints(pool, first)
    n_flush = n_keep = 0
    for step in range(7):
        prob = inputs.make_custom(name="steps", qkv_dtype="bf16", seed=71 + step, slot_ids=slots,
                                  **spec)
        d = staging.DeviceProblem(prob, "cuda", pool=pool, place_s0=False)
        r.place_drafts(d)
        torch.cuda.synchronize()
        host_buf = r.host()
        host_pool = pool.double().cpu().numpy()
        want_o = oracle.replay_verify(prob, host_buf, host_pool)
        want_pool, want_len, flushed = oracle.replay_commit(prob, host_buf, host_pool)
        d.o.fill_(float("nan"))
        binding.gdn_replay_verify(d.c, r.c, d.o)
        binding.gdn_replay_commit(d.c, r.c, d.accepted)
        torch.cuda.synchronize()
        assert binding.gdn_read_device_error(d.c) == 0
        assert rel_err(d.o.cpu().numpy(), want_o) <= TOL
        assert np.array_equal(r.len_out.cpu().numpy()[slots], want_len[slots])
        for i, s in enumerate(slots):
            if flushed[i]:
                assert rel_err(pool[s].cpu().numpy(), want_pool[s]) <= TOL
            else:
                assert np.array_equal(pool[s].cpu().numpy(), host_pool[s].astype(np.float32))
        n_flush += int(flushed.sum())
        n_keep += int((~flushed).sum())
        r.swap()
    assert n_flush and n_keep


def test_replay_bad_length_is_flagged_and_skipped():
    prob, buf, d, r = setup("b3_h4_t16_c40")
    lens = r.len_in.clone()
    s0 = int(prob.slot_ids[0])
    lens[s0] = 40 - 16 + 1  # buffered plus drafts exceed the capacity
    r.len_in.copy_(lens)
    d.o.fill_(float("nan"))
    binding.gdn_replay_verify(d.c, r.c, d.o)
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(d.c) == binding.GDN_DEVERR_REPLAY
    o = d.o.cpu().numpy()
    c0 = int(prob.cu_seqlens[0])
    assert np.isnan(o[c0:c0 + 16]).all()          # request 0: nothing written
    assert not np.isnan(o[int(prob.cu_seqlens[1]):]).any()


@pytest.mark.parametrize("cap", [32, 64])
def test_replay_full_size(cap):
    """The 24-layer workload's batch, heads and draft length (2048 units, the
    benchmark's grid and rounds; a 64-slot pool keeps the oracle's copy small)
    with C buffered rows per slot: every unit's outputs and every flushed
    slot against the oracle, untouched slots bit for bit, the new lengths
    exactly."""
    prob = inputs.make_custom(name="replay_full", batch=64, heads=32, dk=128, dv=128, T=16,
                              qkv_dtype="bf16", pool_slots=64, accept="binom", seed=1003)
    buf = inputs.make_replay(prob, cap, seed=9)
    d = staging.DeviceProblem(prob, "cuda")
    r = staging.DeviceReplay(buf, prob.qkv_dtype)
    pool = d.pool.double().cpu().numpy()
    want_o = oracle.replay_verify(prob, buf, pool, threads=os.cpu_count() or 1)
    want_pool, want_len, flushed = oracle.replay_commit(prob, buf, pool,
                                                        threads=os.cpu_count() or 1)
    before = d.pool.cpu().numpy()
    d.o.fill_(float("nan"))
    binding.gdn_replay_verify(d.c, r.c, d.o)
    binding.gdn_replay_commit(d.c, r.c, d.accepted)
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(d.c) == 0
    err = rel_err(d.o.cpu().numpy(), want_o)
    assert err <= TOL, f"o: {err:.3e}"
    assert np.array_equal(r.len_out.cpu().numpy(), want_len)
    after = d.pool.cpu().numpy()
    flushed_slots = {int(prob.slot_ids[i]) for i in np.flatnonzero(flushed)}
    assert flushed_slots  # the flush branch is exercised
    for s in range(prob.pool_slots):
        if s in flushed_slots:
            e = rel_err(after[s], want_pool[s])
            assert e <= TOL, f"slot {s}: {e:.3e}"
        else:
            assert np.array_equal(after[s].view(np.int32), before[s].view(np.int32))
