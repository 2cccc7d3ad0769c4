"""The fused call against verify followed by commit, on the same kernel path:
the same outputs and the same pool, bit for bit.  The fused pass reads each
checkpoint once, but it does the same arithmetic for o and for the state
after a_r tokens as the two separate calls."""
import ctypes

import pytest
import torch

from speculative_decode_gated_gb300 import binding, inputs, staging

pytestmark = pytest.mark.gpu

REC, CHUNK, TC = binding.GDN_ALGO_RECURRENT, binding.GDN_ALGO_CHUNK, binding.GDN_ALGO_CHUNK_TC


def custom(name, **kw):
    kw.setdefault("qkv_dtype", "bf16")
    kw.setdefault("accept", "uniform")
    return lambda: inputs.make_custom(name=name, **kw)


CASES = {
    "b3_h4_d128_t16": custom("b3_h4_d128_t16", batch=3, heads=4, dk=128, dv=128, T=16,
                             pool_slots=9, accept="binom", seed=31),
    "ragged_b6_d128": custom("ragged_b6_d128", batch=6, heads=3, dk=128, dv=128,
                             lengths=[1, 16, 7, 3, 12, 16], pool_slots=40, seed=32),
    "ragged_multichunk_b7_d128": custom("ragged_multichunk_b7_d128", batch=7, heads=2, dk=128,
                                        dv=128, lengths=[1, 16, 17, 33, 48, 31, 64],
                                        pool_slots=9, seed=33),
    "b4_h2_d64_t8": custom("b4_h2_d64_t8", batch=4, heads=2, dk=64, dv=64, T=8, pool_slots=6,
                           seed=34),
    "fp32_dk32_dv96_t5": custom("fp32_dk32_dv96_t5", batch=3, heads=2, dk=32, dv=96, T=5,
                                qkv_dtype="fp32", pool_slots=3, seed=35),
}


def applies(prob, algo):
    d = binding.gdn_problem()
    d.batch, d.heads, d.dk, d.dv, d.max_T = prob.batch, prob.heads, prob.dk, prob.dv, prob.max_T
    d.qkv_dtype = binding.GDN_BF16 if prob.qkv_dtype == "bf16" else binding.GDN_FP32
    d.algo = algo
    return binding.lib().gdn_select_algo(ctypes.byref(d)) >= 0


def run_both(prob, algo):
    sep = staging.DeviceProblem(prob, "cuda", algo=algo)
    fus = staging.DeviceProblem(prob, "cuda", algo=algo)
    sep.verify()
    sep.commit()
    fus.fused()
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(sep.c) == 0
    assert binding.gdn_read_device_error(fus.c) == 0
    return sep, fus


@pytest.mark.parametrize("algo", [REC, CHUNK, TC], ids=["rec", "chunk", "tc"])
@pytest.mark.parametrize("name", list(CASES))
def test_fused_is_bitwise_verify_then_commit(name, algo):
    prob = CASES[name]()
    if not applies(prob, algo):
        pytest.skip("algo does not apply to this shape")
    sep, fus = run_both(prob, algo)
    assert torch.equal(sep.o.view(torch.int32), fus.o.view(torch.int32)), "outputs differ"
    assert torch.equal(sep.pool.view(torch.int32), fus.pool.view(torch.int32)), "pools differ"
