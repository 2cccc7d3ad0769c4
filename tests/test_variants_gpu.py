"""GPU checks of the precision and layout variants (gdn_problem.flags).

* bf16 o (GDN_FLAG_O_BF16): the output must be, bit for bit, the round to
  nearest even of the float32 output of the same call, and, on its own,
  within the float32 tolerance plus one bfloat16 rounding of the float64
  oracle: |bf16(o) - o_ref| <= |bf16(o) - o| + |o - o_ref|
  <= 2^-9 |o| + TOL max|o_ref| <= (TOL + 2^-9 (1 + TOL)) max|o_ref|.
* log-space gates (GDN_FLAG_LOG_GATE): alpha holds g and the kernels use
  alpha = expf(g); compared with the oracle, which takes alpha = exp(g).
"""
import numpy as np
import pytest
import torch

import oracle

from parity import TOL, check_state_update, check_verify, gather_outputs, oracle_units, rel_err
from speculative_decode_gated_gb300 import binding, inputs, staging

pytestmark = pytest.mark.gpu

REC = binding.GDN_ALGO_RECURRENT

SHAPES = {
    "chunk_b3_h4_t16": dict(batch=3, heads=4, dk=128, dv=128, T=16, pool_slots=7, seed=81),
    "chunk_ragged_b5": dict(batch=5, heads=2, dk=128, dv=128, lengths=[1, 16, 9, 4, 13],
                            pool_slots=9, seed=82),
    "chunk_multi_b2_t40": dict(batch=2, heads=2, dk=128, dv=128, T=40, pool_slots=3, seed=83),
    "rec_fp32_dk64_dv96": dict(batch=3, heads=2, dk=64, dv=96, T=5, qkv_dtype="fp32",
                               pool_slots=4, seed=84),
    "rec_dk256_dv64": dict(batch=2, heads=2, dk=256, dv=64, T=6, pool_slots=3, seed=85),
}


def problem(name, gate="alpha"):
    spec = dict(SHAPES[name])
    spec.setdefault("qkv_dtype", "bf16")
    return inputs.make_custom(name=name, accept="uniform", gate=gate, **spec)


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("mode", ["verify", "fused"])
def test_bf16_output_is_the_rounded_fp32_output(name, mode):
    prob = problem(name)
    d32 = staging.DeviceProblem(prob, "cuda")
    d16 = staging.DeviceProblem(prob, "cuda", o_bf16=True)
    for d in (d32, d16):
        d.o.fill_(float("nan"))
        (d.verify if mode == "verify" else d.fused)()
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(d16.c) == 0
    assert torch.equal(d16.o.view(torch.int16), d32.o.to(torch.bfloat16).view(torch.int16))
    if mode == "fused":
        assert torch.equal(d16.pool.view(torch.int32), d32.pool.view(torch.int32))


# The bf16-output bound against the oracle (round to nearest even: relative
# error at most 2^-9 per element).
TOL_BF16 = TOL + 2.0 ** -9 * (1.0 + TOL)


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("mode", ["verify", "fused"])
def test_bf16_output_against_the_oracle(name, mode):
    prob = problem(name)
    units = np.arange(prob.units)
    o_ref, s_ref = oracle_units(prob, units)
    d = staging.DeviceProblem(prob, "cuda", algo=REC if name.startswith("rec") else 0,
                              o_bf16=True)
    d.o.fill_(float("nan"))
    if mode == "verify":
        d.verify()
    else:
        check_state_update(d, units, s_ref, d.fused)  # the state stays float32: TOL
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(d.c) == 0
    got = gather_outputs(prob, units, d.o.float().cpu().numpy(), o_ref)
    err = rel_err(got, o_ref)
    assert err <= TOL_BF16, f"bf16 o: max rel err {err:.3e}"


def test_bf16_output_replay_verify_against_the_oracle():
    prob = problem("chunk_b3_h4_t16")
    buf = inputs.make_replay(prob, 40, seed=3)
    d = staging.DeviceProblem(prob, "cuda", o_bf16=True)
    r = staging.DeviceReplay(buf, prob.qkv_dtype)
    o_ref = oracle.replay_verify(prob, buf, d.pool.double().cpu().numpy())
    d.o.fill_(float("nan"))
    binding.gdn_replay_verify(d.c, r.c, d.o)
    torch.cuda.synchronize()
    got = d.o.float().cpu().numpy()
    err = rel_err(got, o_ref)
    assert err <= TOL_BF16, f"replay bf16 o: max rel err {err:.3e}"


def test_bf16_output_replay_verify():
    prob = problem("chunk_b3_h4_t16")
    buf = inputs.make_replay(prob, 40, seed=3)
    outs = []
    for o_bf16 in (False, True):
        d = staging.DeviceProblem(prob, "cuda", o_bf16=o_bf16)
        r = staging.DeviceReplay(buf, prob.qkv_dtype)
        binding.gdn_replay_verify(d.c, r.c, d.o)
        torch.cuda.synchronize()
        outs.append(d.o)
    assert torch.equal(outs[1].view(torch.int16), outs[0].to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("mode", ["verify", "commit", "fused"])
def test_log_gate_parity(name, mode):
    prob = problem(name, gate="log")
    assert prob.gate == "log" and np.all(prob.alpha <= 0)
    units = np.arange(prob.units)
    o_ref, s_ref = oracle_units(prob, units)
    d = staging.DeviceProblem(prob, "cuda", algo=REC if name.startswith("rec") else 0)
    assert d.flags & binding.GDN_FLAG_LOG_GATE
    if mode == "verify":
        check_verify(d, units, o_ref)
    elif mode == "commit":
        check_state_update(d, units, s_ref, d.commit)
    else:
        d.o.fill_(float("nan"))
        check_state_update(d, units, s_ref, d.fused)
        assert rel_err(gather_outputs(prob, units, d.o.cpu().numpy(), o_ref), o_ref) <= TOL
