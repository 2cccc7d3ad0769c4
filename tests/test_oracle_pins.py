"""The float64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(lib, pin):
    pin(lib)


# ---------------------------------------------------------------- log-space gates

def test_log_gate_decay_closed_form():
    """beta = 0 with log-space gates g_t: S_T = exp(sum_t g_t) S_0, a closed form
    that sums the logs instead of multiplying decays token by token."""
    from speculative_decode_gated_gb300 import inputs
    prob = inputs.make_custom(batch=2, heads=2, dk=8, dv=4, T=6, qkv_dtype="fp32",
                              accept="full", seed=21, gate="log")
    prob.beta = np.zeros_like(prob.beta)
    _, s_acc = oracle.run_units(prob)
    for u in range(prob.units):
        r, h = divmod(u, prob.heads)
        c0, c1 = int(prob.cu_seqlens[r]), int(prob.cu_seqlens[r + 1])
        scale = np.exp(np.sum(prob.alpha[c0:c1, h].astype(np.float64)))
        want = scale * prob.s0[r, h].astype(np.float64)
        assert np.abs(s_acc[u] - want).max() <= 1e-12 * max(np.abs(want).max(), 1e-300)


def test_log_gate_zero_is_no_decay():
    """g = 0 means alpha = exp(0) = 1 exactly: the same result, bit for bit, as
    the problem with alpha = 1 given directly."""
    from speculative_decode_gated_gb300 import inputs
    prob = inputs.make_custom(batch=2, heads=2, dk=8, dv=4, T=5, qkv_dtype="fp32",
                              accept="uniform", seed=22, gate="log")
    prob.alpha = np.zeros_like(prob.alpha)
    o1, s1 = oracle.run_units(prob)
    prob.gate = "alpha"
    prob.alpha = np.ones_like(prob.alpha)
    o2, s2 = oracle.run_units(prob)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)
