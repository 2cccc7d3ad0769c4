"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Every unit is compared, small problems and the full-size workloads alike (the
b32 and b128 ragged workloads, and the first and last layer of the 24-layer
one), in the same launch configuration the benchmark times.  Bookkeeping
(which pool slots change) is compared bitwise over the whole pool in every
case.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle_pins import load_golden, problem_from_arrays
from parity import (TOL, check_state_update, check_verify, gather_outputs, oracle_units,
                    pick_units, rel_err)
from speculative_decode_gated_gb300 import binding, inputs, staging

pytestmark = pytest.mark.gpu

AUTO, REC, CHUNK, TC = (binding.GDN_ALGO_AUTO, binding.GDN_ALGO_RECURRENT, binding.GDN_ALGO_CHUNK,
                         binding.GDN_ALGO_CHUNK_TC)


def custom(name, **kw):
    kw.setdefault("qkv_dtype", "bf16")
    kw.setdefault("accept", "uniform")
    return lambda: inputs.make_custom(name=name, **kw)


SMALL = {
    "tiny_b1_h2_d32_t4": lambda: inputs.make_problem("tiny_b1_h2_d32_t4"),
    "b8_h16_d128_t8": lambda: inputs.make_problem("b8_h16_d128_t8"),
    "b3_h4_d128_t16": custom("b3_h4_d128_t16", batch=3, heads=4, dk=128, dv=128, T=16,
                             pool_slots=9, accept="binom", seed=11),
    "ragged_b6_d128": custom("ragged_b6_d128", batch=6, heads=3, dk=128, dv=128,
                             lengths=[1, 16, 7, 3, 12, 16], pool_slots=40, seed=12),
    "b4_h2_d64_t8": custom("b4_h2_d64_t8", batch=4, heads=2, dk=64, dv=64, T=8,
                           pool_slots=6, seed=13),
    "fp32_dk32_dv96_t5": custom("fp32_dk32_dv96_t5", batch=3, heads=2, dk=32, dv=96, T=5,
                                qkv_dtype="fp32", pool_slots=3, seed=14),
    "b2_h2_dk128_dv256_t6": custom("b2_h2_dk128_dv256_t6", batch=2, heads=2, dk=128, dv=256,
                                   T=6, pool_slots=4, seed=15),
    "b3_h2_dk64_dv32_t3": custom("b3_h2_dk64_dv32_t3", batch=3, heads=2, dk=64, dv=32, T=3,
                                 pool_slots=3, seed=16),
    "b2_h2_d128_t40": custom("b2_h2_d128_t40", batch=2, heads=2, dk=128, dv=128, T=40,
                             pool_slots=5, seed=17),
    "b4_h4_d128_t1": custom("b4_h4_d128_t1", batch=4, heads=4, dk=128, dv=128, T=1,
                            pool_slots=4, seed=18),
    "fp32_b2_h2_d128_t8": custom("fp32_b2_h2_d128_t8", batch=2, heads=2, dk=128, dv=128, T=8,
                                 qkv_dtype="fp32", pool_slots=2, seed=19),
    "accept_zero_b4_d128_t16": custom("accept_zero_b4_d128_t16", batch=4, heads=2, dk=128,
                                      dv=128, T=16, pool_slots=8, accept="zero", seed=20),
    "accept_full_b4_d128_t16": custom("accept_full_b4_d128_t16", batch=4, heads=2, dk=128,
                                      dv=128, T=16, pool_slots=8, accept="full", seed=21),
    # several 16-token chunks per unit: lengths across chunk boundaries, commit
    # points in every chunk and on a boundary
    "ragged_multichunk_b7_d128": custom("ragged_multichunk_b7_d128", batch=7, heads=2, dk=128,
                                        dv=128, lengths=[1, 16, 17, 33, 48, 31, 64],
                                        pool_slots=9, seed=22),
    "b3_h2_d128_t64_full": custom("b3_h2_d128_t64_full", batch=3, heads=2, dk=128, dv=128,
                                  T=64, pool_slots=3, accept="full", seed=23),
    "b2_h2_d128_t200": custom("b2_h2_d128_t200", batch=2, heads=2, dk=128, dv=128, T=200,
                              pool_slots=2, seed=24),
    # ragged batches with empty requests (no rows: nothing to verify, a_r = 0),
    # in the middle and at the end
    "ragged_empty_b6_d128": custom("ragged_empty_b6_d128", batch=6, heads=2, dk=128, dv=128,
                                   lengths=[3, 0, 16, 0, 5, 0], pool_slots=8, seed=27),
    # the longest draft the ABI accepts (64 chained chunks)
    "b1_h1_d128_t1024": custom("b1_h1_d128_t1024", batch=1, heads=1, dk=128, dv=128, T=1024,
                               pool_slots=2, accept="full", seed=28),
    # dk = 256 (recurrent kernel, four threads per value column)
    "b2_h2_dk256_dv64_t6": custom("b2_h2_dk256_dv64_t6", batch=2, heads=2, dk=256, dv=64, T=6,
                                  pool_slots=3, seed=25),
    "fp32_b2_h2_dk256_dv256_t5": custom("fp32_b2_h2_dk256_dv256_t5", batch=2, heads=2, dk=256,
                                        dv=256, T=5, qkv_dtype="fp32", pool_slots=2, seed=26),
}

_cache = {}


def small(name):
    if name not in _cache:
        prob = SMALL[name]()
        units = np.arange(prob.units)
        _cache[name] = (prob, units, *oracle_units(prob, units))
    return _cache[name]


def algo_applies(prob, algo):
    d = binding.gdn_problem()
    d.batch, d.heads, d.dk, d.dv, d.max_T = prob.batch, prob.heads, prob.dk, prob.dv, prob.max_T
    d.qkv_dtype = binding.GDN_BF16 if prob.qkv_dtype == "bf16" else binding.GDN_FP32
    d.algo = algo
    return binding.lib().gdn_select_algo(ctypes.byref(d)) >= 0


def _params():
    for name in SMALL:
        for algo in (AUTO, REC, CHUNK, TC):
            for mode in ("verify", "commit", "fused"):
                yield pytest.param(name, algo, mode,
                                   id=f"{name}-{['auto', 'rec', 'chunk', 'tc'][algo]}-{mode}")


@pytest.mark.parametrize("name,algo,mode", list(_params()))
def test_small_parity(name, algo, mode):
    prob, units, o_ref, s_ref = small(name)
    if not algo_applies(prob, algo):
        pytest.skip("algo does not apply to this shape")
    d = staging.DeviceProblem(prob, "cuda", algo=algo)
    if mode == "verify":
        check_verify(d, units, o_ref)
    elif mode == "commit":
        check_state_update(d, units, s_ref, d.commit)
    else:
        d.o.fill_(float("nan"))
        check_state_update(d, units, s_ref, d.fused)
        assert rel_err(gather_outputs(prob, units, d.o.cpu().numpy(), o_ref), o_ref) <= TOL


FULL = ["b32_h32_d128_t16", "b64_h32_d128_t16_x24", "b128_h32_d128_ragged16"]


FULL_LAYERS = [(n, l) for n in FULL for l in ([0, 23] if n.endswith("x24") else [0])]


@pytest.mark.parametrize("name,layer", FULL_LAYERS, ids=[f"{n}-layer{l}" for n, l in FULL_LAYERS])
def test_full_size_every_unit(name, layer):
    """All units of the workload (of the named layer), against one oracle run:
    verify then commit, and fused, on the default kernel and on the tcgen05 one.
    Per-unit or per-round faults of the persistent kernel (its last, partly
    filled round of units) would show here."""
    prob = inputs.make_problem(name, layer=layer)
    units = np.arange(prob.units)
    o_ref, s_ref = oracle_units(prob, units)
    for algo in (AUTO, TC):
        for mode in ("separate", "fused"):
            d = staging.DeviceProblem(prob, "cuda", algo=algo)
            if mode == "separate":
                check_verify(d, units, o_ref)
                check_state_update(d, units, s_ref, d.commit)
            else:
                d.o.fill_(float("nan"))
                check_state_update(d, units, s_ref, d.fused)
                err = rel_err(gather_outputs(prob, units, d.o.cpu().numpy(), o_ref), o_ref)
                assert err <= TOL, f"fused o: max rel err {err:.3e}"
            del d
            torch.cuda.empty_cache()


@pytest.mark.parametrize("golden", ["hand_2x2_t2.txt", "hand_dk3_dv2_t2.txt"])
def test_hand_cases_exact_on_fp32_path(golden):
    """The hand-worked fixtures hold exact binary fractions; the fp32 recurrent
    path reproduces them exactly.  dk and dv are padded with zeros to the
    smallest supported shape (zero rows/columns do not interact)."""
    g = load_golden(golden)
    dk, dv, T = int(g["dk"][0]), int(g["dv"][0]), int(g["T"][0])
    DK, DV = 32, 32
    s0 = np.zeros((DK, DV))
    s0[:dk, :dv] = g["s0"].reshape(dk, dv)
    pad = lambda x, d, Dp: np.pad(x.reshape(T, d), ((0, 0), (0, Dp - d)))
    for a in range(T + 1):
        prob = problem_from_arrays(s0, g["alpha"], g["beta"], pad(g["k"], dk, DK),
                                   pad(g["v"], dv, DV), pad(g["q"], dk, DK), accepted=a)
        d = staging.DeviceProblem(prob, "cuda", algo=REC)
        d.fused()
        torch.cuda.synchronize()
        o = d.o.cpu().numpy()[:, 0, :dv]
        assert np.array_equal(o, g["o"].reshape(T, dv).astype(np.float32))
        st = d.pool.cpu().numpy()[0, 0, :dk, :dv]
        assert np.array_equal(st, g[f"state_{a}"].reshape(dk, dv).astype(np.float32))


def _with_bad(name, tweak, ragged_max_T=None, algo=AUTO):
    lens = {"lengths": [10, 4, 6, 3]} if ragged_max_T else {"T": 8}
    prob = inputs.make_custom(batch=4, heads=2, dk=128, dv=128, qkv_dtype="bf16",
                              pool_slots=6, accept="uniform", seed=30, name=name, **lens)
    d = staging.DeviceProblem(prob, "cuda", algo=algo)
    if ragged_max_T is not None:
        d.c.c.max_T = ragged_max_T
    tweak(d, prob)
    return prob, d


@pytest.mark.parametrize("algo", [AUTO, REC])
@pytest.mark.parametrize("kind", ["slot", "accepted", "seqlen"])
def test_device_side_argument_errors(kind, algo):
    """A bad slot id, accepted length or ragged length sets its error bit and the
    unit is skipped: nothing is written for that request; the others are right."""
    bad_r = 0
    if kind == "slot":
        prob, d = _with_bad("bad_slot", lambda d, p: d.slot_ids.__setitem__(bad_r, p.pool_slots + 3),
                            algo=algo)
        bit = binding.GDN_DEVERR_SLOT
    elif kind == "accepted":
        prob, d = _with_bad("bad_acc", lambda d, p: d.accepted.__setitem__(bad_r, 99), algo=algo)
        bit = binding.GDN_DEVERR_ACCEPTED
    else:
        # request 0 has 10 tokens; the problem claims at most 8
        prob, d = _with_bad("bad_len", lambda d, p: None, ragged_max_T=8, algo=algo)
        bit = binding.GDN_DEVERR_SEQLEN
    pool0 = d.pool.clone()
    d.o.fill_(float("nan"))
    d.fused()
    code = binding.gdn_read_device_error(d.c)
    assert code & bit
    o = d.o.cpu().numpy()
    rows = slice(int(prob.cu_seqlens[bad_r]), int(prob.cu_seqlens[bad_r + 1]))
    assert np.isnan(o[rows]).all(), "skipped request's outputs were written"
    slot = int(prob.slot_ids[bad_r])
    assert torch.equal(d.pool[slot].view(torch.int32), pool0[slot].view(torch.int32))
    good = [r for r in range(prob.batch) if r != bad_r]
    units = np.array([r * prob.heads + hh for r in good for hh in range(prob.heads)])
    o_ref, _ = oracle_units(prob, units)
    assert rel_err(gather_outputs(prob, units, o, o_ref), o_ref) <= TOL


@pytest.mark.parametrize("algo", [AUTO, REC, TC], ids=["auto", "rec", "tc"])
def test_extreme_gates(algo):
    """Gates at their limits in one batch: alpha in {0, 1e-30, 1e-6, 1} (the decay
    products of the chunk form underflow to zero or stay exactly 1) and beta in
    {0, 1}; the outputs and committed states still match the oracle."""
    prob = inputs.make_custom(batch=4, heads=2, dk=128, dv=128, lengths=[16, 9, 16, 5],
                              qkv_dtype="bf16", pool_slots=6, accept="uniform", seed=61,
                              name="extreme_gates")
    rng = np.random.default_rng(62)
    prob.alpha = rng.choice(np.array([0.0, 1e-30, 1e-6, 1.0], np.float32),
                            size=prob.alpha.shape).astype(np.float32)
    prob.beta = rng.choice(np.array([0.0, 1.0], np.float32), size=prob.beta.shape).astype(np.float32)
    units = np.arange(prob.units)
    o_ref, s_ref = oracle_units(prob, units)
    d = staging.DeviceProblem(prob, "cuda", algo=algo)
    check_verify(d, units, o_ref)
    check_state_update(d, units, s_ref, d.commit)


@pytest.mark.parametrize("algo", [AUTO, REC], ids=["auto", "rec"])
def test_commit_without_q(algo):
    """The commit calls read no q: a problem given none (q = NULL) commits the
    same bits as one given q."""
    prob = inputs.make_custom(batch=5, heads=3, dk=128, dv=128, lengths=[16, 3, 0, 9, 12],
                              qkv_dtype="bf16", pool_slots=8, accept="uniform", seed=91,
                              name="commit_no_q")
    with_q = staging.DeviceProblem(prob, "cuda", algo=algo)
    no_q = staging.DeviceProblem(prob, "cuda", algo=algo)
    c = binding.make_problem(q=None, k=no_q.k, v=no_q.v, alpha=no_q.alpha, beta=no_q.beta,
                             pool=no_q.pool, slot_ids=no_q.slot_ids, max_T=prob.max_T,
                             cu_seqlens=no_q.cu_seqlens, dev_err=no_q.dev_err, algo=algo)
    with_q.commit()
    binding.gdn_commit(c, no_q.accepted)
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(c) == 0
    assert torch.equal(with_q.pool.view(torch.int32), no_q.pool.view(torch.int32))
    with pytest.raises(binding.GdnError):  # verify needs q
        binding.gdn_verify(c, no_q.o)


def test_full_size_long_drafts():
    """32-token drafts on the 24-layer workload's shape (two 16-token chunks per
    unit, the multi-chunk kernel over 2048 units): every unit against the
    oracle, verify then commit and fused."""
    prob = inputs.make_problem("b64_h32_d128_t16_x24", layer=0, draft=32)
    units = np.arange(prob.units)
    o_ref, s_ref = oracle_units(prob, units)
    d = staging.DeviceProblem(prob, "cuda")
    check_verify(d, units, o_ref)
    check_state_update(d, units, s_ref, d.commit)
    f = staging.DeviceProblem(prob, "cuda")
    f.o.fill_(float("nan"))
    check_state_update(f, units, s_ref, f.fused)
    assert rel_err(gather_outputs(prob, units, f.o.cpu().numpy(), o_ref), o_ref) <= TOL


@pytest.mark.parametrize("o_bf16,gate", [(False, "log"), (True, "alpha"), (True, "log")],
                         ids=["log_gate", "bf16_o", "both"])
def test_full_size_variants(o_bf16, gate):
    """The precision variants on one layer of the 24-layer workload (their own
    single-chunk instantiations): every unit against the oracle; bf16 o within
    the float32 tolerance plus one bfloat16 rounding."""
    prob = inputs.make_problem("b64_h32_d128_t16_x24", layer=0, gate=gate)
    units = np.arange(prob.units)
    o_ref, s_ref = oracle_units(prob, units)
    tol_o = TOL + 2.0 ** -9 * (1.0 + TOL) if o_bf16 else TOL
    d = staging.DeviceProblem(prob, "cuda", o_bf16=o_bf16)
    d.o.fill_(float("nan"))
    d.verify()
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(d.c) == 0
    err = rel_err(gather_outputs(prob, units, d.o.float().cpu().numpy(), o_ref), o_ref)
    assert err <= tol_o, f"verify o: {err:.3e}"
    check_state_update(d, units, s_ref, d.commit)
    f = staging.DeviceProblem(prob, "cuda", o_bf16=o_bf16)
    f.o.fill_(float("nan"))
    check_state_update(f, units, s_ref, f.fused)
    err = rel_err(gather_outputs(prob, units, f.o.float().cpu().numpy(), o_ref), o_ref)
    assert err <= tol_o, f"fused o: {err:.3e}"
