"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare it with the float64 oracle on the same seeded inputs.

Tolerance: every output tensor and every written state slot must satisfy
max|gpu - oracle| <= 2e-3 * max|oracle|.  Slot bookkeeping is compared bitwise.
"""
import os

import numpy as np
import torch

import oracle
from speculative_decode_gated_gb300 import binding, staging

TOL = 2e-3
THREADS = os.cpu_count() or 1


def rel_err(got, want) -> float:
    want = np.asarray(want, np.float64)
    got = np.asarray(got, np.float64)
    if want.size == 0:
        return 0.0
    scale = float(np.abs(want).max())
    diff = float(np.abs(got - want).max())
    if not np.isfinite(diff):
        return float("inf")
    return diff / scale if scale > 0 else diff


def pick_units(prob, n_sample):
    """All units, or a spread sample that always contains the first and last unit,
    requests with a_r = 0, with a_r = T_r and the shortest ragged request."""
    U = prob.units
    if n_sample is None or n_sample >= U:
        return np.arange(U)
    rng = np.random.default_rng(12345)
    lens = prob.lengths
    special_r = {0, prob.batch - 1, int(np.argmin(lens)), int(np.argmax(lens))}
    special_r.update(np.flatnonzero(prob.accepted == 0)[:2].tolist())
    special_r.update(np.flatnonzero(prob.accepted == lens)[:2].tolist())
    units = {r * prob.heads + int(rng.integers(prob.heads)) for r in special_r}
    units.update({0, U - 1})
    while len(units) < n_sample:
        units.add(int(rng.integers(U)))
    return np.array(sorted(units))


def oracle_units(prob, units):
    return oracle.run_units(prob, units, threads=THREADS)


def gather_outputs(prob, units, o_dev: np.ndarray, like: np.ndarray) -> np.ndarray:
    """GPU outputs of the listed units in the oracle's [n][max_T][dv] layout."""
    got = np.zeros_like(like)
    for n, u in enumerate(units):
        r, h = divmod(int(u), prob.heads)
        c0, L = int(prob.cu_seqlens[r]), int(prob.lengths[r])
        got[n, :L] = o_dev[c0:c0 + L, h]
    return got


def check_verify(d: staging.DeviceProblem, units, o_ref):
    prob = d.host
    pool_before = d.pool.view(torch.int32).clone()
    d.o.fill_(float("nan"))
    d.verify()
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(d.c) == 0
    assert torch.equal(d.pool.view(torch.int32), pool_before), "verify changed the pool"
    err = rel_err(gather_outputs(prob, units, d.o.cpu().numpy(), o_ref), o_ref)
    assert err <= TOL, f"verify: max rel err {err:.3e}"
    return err


def check_state_update(d: staging.DeviceProblem, units, s_ref, run):
    """Runs `run` (commit or fused) and checks written slots and bookkeeping."""
    prob = d.host
    before = d.pool.cpu().numpy()
    run()
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(d.c) == 0
    after = d.pool.cpu().numpy()
    touched = {int(prob.slot_ids[r]) for r in range(prob.batch) if prob.accepted[r] > 0}
    b32, a32 = before.view(np.int32), after.view(np.int32)
    unchanged = [s for s in range(prob.pool_slots) if s not in touched]
    assert np.array_equal(a32[unchanged], b32[unchanged]), \
        "a slot with a_r = 0 or a slot no request names changed"
    worst = 0.0
    by_slot = {}
    for n, u in enumerate(units):
        r, h = divmod(int(u), prob.heads)
        if prob.accepted[r] == 0:
            continue
        by_slot.setdefault(int(prob.slot_ids[r]), []).append((h, s_ref[n]))
    for slot, items in by_slot.items():
        got = np.stack([after[slot, h] for h, _ in items])
        want = np.stack([s for _, s in items])
        err = rel_err(got, want)
        worst = max(worst, err)
        assert err <= TOL, f"state of slot {slot}: max rel err {err:.3e}"
    return worst
