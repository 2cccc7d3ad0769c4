"""A seeded sweep of random small problems through the C ABI against the
float64 oracle: batch 1-12, 1-7 heads (odd counts included), uniform or ragged
drafts (empty requests, lengths across 16-token chunk boundaries), random
accepted lengths and slot ids, on every kernel that applies.  Every unit is
compared; slot bookkeeping is compared bitwise over the whole pool."""
import ctypes

import numpy as np
import pytest

from parity import TOL, check_state_update, check_verify, gather_outputs, oracle_units, rel_err
from speculative_decode_gated_gb300 import binding, inputs, staging

pytestmark = pytest.mark.gpu

ALGOS = (binding.GDN_ALGO_AUTO, binding.GDN_ALGO_RECURRENT, binding.GDN_ALGO_CHUNK_TC)


def random_problem(seed):
    rng = np.random.default_rng(seed)
    batch = int(rng.integers(1, 13))
    heads = int(rng.integers(1, 8))
    long = rng.random() < 0.3  # drafts over several 16-token chunks
    max_len = 48 if long else 16
    if rng.random() < 0.5:
        spec = dict(T=int(rng.integers(1, max_len + 1)))
    else:
        lens = rng.integers(0, max_len + 1, size=batch)
        lens[rng.random(batch) < 0.15] = 0  # empty requests
        if lens.max() == 0:
            lens[0] = 1
        spec = dict(lengths=lens.tolist())
    return inputs.make_custom(name=f"sweep{seed}", batch=batch, heads=heads, dk=128, dv=128,
                              qkv_dtype="bf16", pool_slots=batch + int(rng.integers(0, 9)),
                              accept=["uniform", "full", "zero", "binom"][seed % 4],
                              seed=5000 + seed, **spec)


def applies(prob, algo):
    d = binding.gdn_problem()
    d.batch, d.heads, d.dk, d.dv, d.max_T = prob.batch, prob.heads, prob.dk, prob.dv, prob.max_T
    d.qkv_dtype = binding.GDN_BF16
    d.algo = algo
    return binding.lib().gdn_select_algo(ctypes.byref(d)) >= 0


@pytest.mark.parametrize("seed", range(24))
def test_random_problem(seed):
    prob = random_problem(seed)
    units = np.arange(prob.units)
    o_ref, s_ref = oracle_units(prob, units)
    for algo in ALGOS:
        if not applies(prob, algo):
            continue
        d = staging.DeviceProblem(prob, "cuda", algo=algo)
        check_verify(d, units, o_ref)
        check_state_update(d, units, s_ref, d.commit)
        f = staging.DeviceProblem(prob, "cuda", algo=algo)
        f.o.fill_(float("nan"))
        check_state_update(f, units, s_ref, f.fused)
        err = rel_err(gather_outputs(prob, units, f.o.cpu().numpy(), o_ref), o_ref)
        assert err <= TOL, f"algo {algo} fused o: {err:.3e}"
