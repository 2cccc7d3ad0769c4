"""Failure detection on the GPU, without a fault: the kernels' bounded wait,
run to its expiry on a barrier that nothing completes, reports
GDN_DEVERR_TIMEOUT through the caller's error word after about two seconds,
and the same CUDA context then computes correct results again."""
import time

import pytest
import torch

from parity import check_state_update, check_verify, oracle_units, pick_units
from speculative_decode_gated_gb300 import binding, inputs, staging

pytestmark = pytest.mark.gpu


def test_wait_expiry_reports_timeout_and_the_context_survives():
    dev = torch.device("cuda:0")
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    binding.gdn_selftest_wait_timeout(err)
    torch.cuda.synchronize()  # raises if the kernel had faulted
    dt = time.perf_counter() - t0
    assert int(err.item()) == binding.GDN_DEVERR_TIMEOUT
    assert 1.5 < dt < 30.0, f"the wait gave up after {dt:.2f} s"

    # The context is intact: the chunk kernel still matches the oracle.
    prob = inputs.make_problem("b8_h16_d128_t8")
    units = pick_units(prob, None)
    o_ref, s_ref = oracle_units(prob, units)
    d = staging.DeviceProblem(prob, "cuda", algo=binding.GDN_ALGO_CHUNK)
    check_verify(d, units, o_ref)
    check_state_update(d, units, s_ref, d.commit)


def test_wait_expiry_keeps_other_bits_and_repeats():
    # The timeout bit is ORed in: bits already set stay, and a second expiry
    # on the same word leaves it unchanged.
    err = torch.full((1,), binding.GDN_DEVERR_SLOT, dtype=torch.int32, device="cuda:0")
    binding.gdn_selftest_wait_timeout(err)
    binding.gdn_selftest_wait_timeout(err)
    torch.cuda.synchronize()
    assert int(err.item()) == binding.GDN_DEVERR_SLOT | binding.GDN_DEVERR_TIMEOUT
