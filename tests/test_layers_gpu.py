"""GPU parity of the layer-batch calls (gdn_*_layers): several layers of one step
in as few launches as possible.

Each layer is checked against the float64 oracle on every unit, with the same
tolerance and bitwise bookkeeping as the single-problem calls, and the results
must be bit-identical to calling the single-problem function once per layer
(the per-unit arithmetic does not depend on how units are batched).
"""
import numpy as np
import pytest
import torch

from parity import TOL, gather_outputs, oracle_units, rel_err
from speculative_decode_gated_gb300 import binding, inputs, staging

pytestmark = pytest.mark.gpu

AUTO, REC, TC = binding.GDN_ALGO_AUTO, binding.GDN_ALGO_RECURRENT, binding.GDN_ALGO_CHUNK_TC

CASES = {
    # chunked kernel, uniform drafts, one launch
    "b3_h4_d128_t16_x3": dict(batch=3, heads=4, dk=128, dv=128, T=16, pool_slots=9,
                              accept="binom", seed=31, layers=3),
    # chunked kernel, ragged drafts (with a length-1 and a full request)
    "ragged_b5_h2_d128_x4": dict(batch=5, heads=2, dk=128, dv=128, lengths=[1, 16, 9, 4, 13],
                                 pool_slots=12, accept="uniform", seed=32, layers=4),
    # 35 layers: more than one launch's worth (32 + 3)
    "b2_h2_d128_t4_x35": dict(batch=2, heads=2, dk=128, dv=128, T=4, pool_slots=3,
                              accept="uniform", seed=33, layers=35),
    # recurrent kernel (fp32 q/k/v), one launch per layer
    "fp32_b3_h2_d64_t5_x3": dict(batch=3, heads=2, dk=64, dv=64, T=5, qkv_dtype="fp32",
                                 pool_slots=4, accept="uniform", seed=34, layers=3),
}

_cache = {}


def case(name):
    if name not in _cache:
        spec = dict(CASES[name])
        n_layers = spec.pop("layers")
        spec.setdefault("qkv_dtype", "bf16")
        probs = [inputs.make_custom(name=name, layer=l, **spec) for l in range(n_layers)]
        refs = []
        for pr in probs:
            units = np.arange(pr.units)
            refs.append((units, *oracle_units(pr, units)))
        _cache[name] = (probs, refs)
    return _cache[name]


def stage(probs, algo=AUTO):
    """One [L, slots, H, dk, dv] pool; layer l's problem points at pool[l]."""
    p0 = probs[0]
    pool = staging.new_pool(p0.pool_slots, p0.heads, p0.dk, p0.dv, "cuda", fill="sentinel",
                            layers=len(probs))
    dps = [staging.DeviceProblem(pr, "cuda", pool=pool[l], algo=algo) for l, pr in enumerate(probs)]
    # request-level arrays must be the same device arrays in every layer
    for d in dps[1:]:
        d.slot_ids, d.accepted, d.cu_seqlens = dps[0].slot_ids, dps[0].accepted, dps[0].cu_seqlens
        d.c = binding.make_problem(q=d.q, k=d.k, v=d.v, alpha=d.alpha, beta=d.beta, pool=d.pool,
                                   slot_ids=d.slot_ids, max_T=d.host.max_T,
                                   cu_seqlens=d.cu_seqlens, dev_err=d.dev_err, algo=algo)
    return pool, dps, binding.ProblemArray([d.c for d in dps])


def check_layer_state(prob, before, after, units, s_ref):
    touched = {int(prob.slot_ids[r]) for r in range(prob.batch) if prob.accepted[r] > 0}
    unchanged = [s for s in range(prob.pool_slots) if s not in touched]
    assert np.array_equal(after.view(np.int32)[unchanged], before.view(np.int32)[unchanged])
    for n, u in enumerate(units):
        r, h = divmod(int(u), prob.heads)
        if prob.accepted[r] == 0:
            continue
        err = rel_err(after[int(prob.slot_ids[r]), h], s_ref[n])
        assert err <= TOL, f"layer state unit {u}: {err:.3e}"


def _layer_params():
    for name in CASES:
        for mode in ("verify", "commit", "fused"):
            yield pytest.param(name, mode, None, id=f"{name}-{mode}")
    # the tcgen05 kernel: layer batches run as one launch per layer
    for mode in ("verify", "commit", "fused"):
        yield pytest.param("ragged_b5_h2_d128_x4", mode, TC, id=f"ragged_b5_h2_d128_x4-{mode}-tc")


@pytest.mark.parametrize("name,mode,algo", list(_layer_params()))
def test_layers_parity_and_equal_to_single_calls(name, mode, algo):
    probs, refs = case(name)
    if algo is None:
        algo = REC if probs[0].qkv_dtype == "fp32" else AUTO
    pool, dps, arr = stage(probs, algo)
    pool_single = pool.clone()
    for d in dps:
        d.o.fill_(float("nan"))
    before = pool.cpu().numpy()
    acc = dps[0].accepted
    if mode == "verify":
        binding.gdn_verify_layers(arr, [d.o for d in dps])
    elif mode == "commit":
        binding.gdn_commit_layers(arr, acc)
    else:
        binding.gdn_verify_commit_fused_layers(arr, acc, [d.o for d in dps])
    torch.cuda.synchronize()
    after = pool.cpu().numpy()
    outs = [d.o.clone() for d in dps]
    for l, (pr, d, (units, o_ref, s_ref)) in enumerate(zip(probs, dps, refs)):
        assert binding.gdn_read_device_error(d.c) == 0
        if mode != "commit":
            err = rel_err(gather_outputs(pr, units, outs[l].cpu().numpy(), o_ref), o_ref)
            assert err <= TOL, f"layer {l} o: {err:.3e}"
        if mode == "verify":
            assert np.array_equal(after[l].view(np.int32), before[l].view(np.int32))
        else:
            check_layer_state(pr, before[l], after[l], units, s_ref)

    # The same layers through the single-problem calls, on a copy of the pool.
    pool.copy_(pool_single)
    for d in dps:
        d.o.fill_(float("nan"))
        {"verify": d.verify, "commit": d.commit, "fused": d.fused}[mode]()
    torch.cuda.synchronize()
    assert torch.equal(pool.view(torch.int32).cpu(), torch.from_numpy(after.view(np.int32)))
    if mode != "commit":
        for l, d in enumerate(dps):
            assert torch.equal(d.o.view(torch.int32), outs[l].view(torch.int32)), f"layer {l}"


def test_layers_device_errors_reach_every_layer():
    probs, _ = case("b3_h4_d128_t16_x3")
    _, dps, arr = stage(probs)
    dps[0].accepted[1] = probs[0].max_T + 1  # shared by all layers
    binding.gdn_commit_layers(arr, dps[0].accepted)
    torch.cuda.synchronize()
    for d in dps:
        assert binding.gdn_read_device_error(d.c) == binding.GDN_DEVERR_ACCEPTED


def test_layers_mismatch_rejected_before_launch():
    probs, _ = case("b3_h4_d128_t16_x3")
    _, dps, _ = stage(probs)
    other = binding.make_problem(q=dps[1].q, k=dps[1].k, v=dps[1].v, alpha=dps[1].alpha,
                                 beta=dps[1].beta, pool=dps[1].pool,
                                 slot_ids=dps[1].slot_ids.clone(), max_T=probs[1].max_T)
    arr = binding.ProblemArray([dps[0].c, other])
    with pytest.raises(binding.GdnError) as e:
        binding.gdn_commit_layers(arr, dps[0].accepted)
    assert e.value.status == binding.GDN_ERR_LAYER_MISMATCH


@pytest.mark.parametrize("mode", ["verify", "commit", "fused"])
def test_full_size_layer_batch(mode):
    """The 24-layer workload in one layer-batch launch: 24 x 2048 units, about
    160 rounds of the persistent grid.  Bit for bit equal to the 24 single
    calls, and the last layer (whose units come last in the launch) against
    the oracle on every unit."""
    probs = inputs.make_layers("b64_h32_d128_t16_x24")
    pool, dps, arr = stage(probs)
    pool_single = pool.clone()
    for d in dps:
        d.o.fill_(float("nan"))
    acc = dps[0].accepted
    if mode == "verify":
        binding.gdn_verify_layers(arr, [d.o for d in dps])
    elif mode == "commit":
        binding.gdn_commit_layers(arr, acc)
    else:
        binding.gdn_verify_commit_fused_layers(arr, acc, [d.o for d in dps])
    torch.cuda.synchronize()
    for d in dps:
        assert binding.gdn_read_device_error(d.c) == 0
    outs = [d.o.clone() for d in dps] if mode != "commit" else None
    batched = pool.clone()
    # the last layer against the oracle
    last = probs[-1]
    units = np.arange(last.units)
    o_ref, s_ref = oracle_units(last, units)
    if mode != "commit":
        err = rel_err(gather_outputs(last, units, outs[-1].cpu().numpy(), o_ref), o_ref)
        assert err <= TOL, f"last layer o: {err:.3e}"
    if mode != "verify":
        check_layer_state(last, pool_single[-1].cpu().numpy(), batched[-1].cpu().numpy(),
                          units, s_ref)
    # the single-problem calls on a copy of the pool
    pool.copy_(pool_single)
    for d in dps:
        d.o.fill_(float("nan"))
        {"verify": d.verify, "commit": d.commit, "fused": d.fused}[mode]()
    torch.cuda.synchronize()
    assert torch.equal(pool.view(torch.int32), batched.view(torch.int32))
    if outs is not None:
        for l, d in enumerate(dps):
            assert torch.equal(d.o.view(torch.int32), outs[l].view(torch.int32)), f"layer {l}"
    del pool, pool_single, batched, dps, arr
    torch.cuda.empty_cache()
