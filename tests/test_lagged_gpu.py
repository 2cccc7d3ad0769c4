"""GPU parity of gdn_commit_verify (commit the previous step, verify the next)
against the float64 oracle (oracle.commit_verify), over chains of steps that
carry the GPU's own pool and W from one call to the next.

Per step: every output within the tolerance, every slot a request commits
within the tolerance of the oracle's state, every other slot bit for bit
unchanged (unnamed slots hold NaN sentinels).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL, rel_err
from speculative_decode_gated_gb300 import binding, inputs, staging

pytestmark = pytest.mark.gpu


def steps(kind, seed=41, n=3, gate="alpha"):
    """n steps of the same requests (slot ids from the seed's metadata stream)."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        if kind == "uniform":
            spec = dict(batch=5, heads=3, T=16)
            T = np.full(5, 16)
        else:
            T = rng.integers(0, 17, size=6)
            T[1] = 0  # an empty request
            spec = dict(batch=6, heads=3, lengths=T.tolist())
        acc = np.array([rng.integers(0, t + 1) for t in T], np.int32)
        acc[0] = T[0]  # a fully accepted draft
        if len(acc) > 2:
            acc[2] = 0  # nothing accepted
        out.append(inputs.make_custom(dk=128, dv=128, pool_slots=11, qkv_dtype="bf16", seed=seed,
                                      layer=i, accepted=acc, name=f"{kind}{i}", gate=gate, **spec))
    return out


def run_chain(probs, bad=None):
    """GPU and oracle side by side, one step at a time; returns per-step errors."""
    p0 = probs[0]
    pool = staging.new_pool(p0.pool_slots, p0.heads, p0.dk, p0.dv, "cuda")
    staging.place_checkpoints(pool, p0)
    pool_ref = pool.cpu().numpy().astype(np.float64)
    prev_d, prev_w, prev_host = None, None, None
    for i, prob in enumerate(probs):
        d = staging.DeviceProblem(prob, "cuda", pool=pool, place_s0=False)
        w = torch.full((prob.n_tok, prob.heads, prob.dv), float("nan"), device="cuda")
        prev = None
        if prev_d is not None:
            acc = prev_d.accepted
            if bad is not None and i == 1:
                acc = acc.clone()
                acc[bad] = int(prev_host.lengths[bad]) + 1
            prev = binding.make_prev_step(k=prev_d.k, alpha=prev_d.alpha, w=prev_w, accepted=acc,
                                          max_T=prev_host.max_T, cu_seqlens=prev_d.cu_seqlens)
        before = pool.cpu().numpy()
        d.o.fill_(float("nan"))
        binding.gdn_commit_verify(d.c, prev, d.o, w)
        torch.cuda.synchronize()
        code = binding.gdn_read_device_error(d.c)
        after = pool.cpu().numpy()
        ref_after, o_ref = oracle.commit_verify(prev_host, prob, pool_ref)
        yield i, prob, prev_host, code, before, after, ref_after, d.o.cpu().numpy(), o_ref
        pool_ref = ref_after
        prev_d, prev_w, prev_host = d, w, prob


@pytest.mark.parametrize("kind,gate", [("uniform", "alpha"), ("ragged", "alpha"), ("ragged", "log")])
def test_chain_matches_the_oracle(kind, gate):
    """gate = "log": alpha holds g for both steps; the kernel applies expf to the
    previous step's gates too."""
    for i, prob, prev, code, before, after, ref_after, o, o_ref in run_chain(steps(kind, gate=gate)):
        assert code == 0
        # outputs of every draft row
        rows = np.concatenate([np.arange(prob.cu_seqlens[r], prob.cu_seqlens[r + 1])
                               for r in range(prob.batch)]).astype(int)
        err = rel_err(o[rows], o_ref[rows])
        assert err <= TOL, f"step {i}: outputs, max rel err {err:.3e}"
        # slots: committed ones against the oracle, every other one untouched
        touched = set()
        if prev is not None:
            touched = {int(prev.slot_ids[r]) for r in range(prev.batch) if prev.accepted[r] > 0}
        for s in range(prob.pool_slots):
            if s in touched:
                err = rel_err(after[s], ref_after[s])
                assert err <= TOL, f"step {i}: slot {s}, max rel err {err:.3e}"
            else:
                assert np.array_equal(after[s].view(np.int32), before[s].view(np.int32)), \
                    f"step {i}: slot {s} changed"


def test_first_step_is_a_verify():
    prob = steps("uniform", seed=43, n=1)[0]
    d = staging.DeviceProblem(prob, "cuda")
    w = torch.zeros((prob.n_tok, prob.heads, prob.dv), device="cuda")
    pool0 = d.pool.clone()
    binding.gdn_commit_verify(d.c, None, d.o, w)
    o_cv = d.o.clone()
    d.verify()
    torch.cuda.synchronize()
    assert torch.equal(d.pool.view(torch.int32), pool0.view(torch.int32))
    assert torch.equal(o_cv, d.o)  # the same arithmetic as gdn_verify, bit for bit


def test_bad_previous_length_is_flagged_and_skipped():
    bad = 3
    for i, prob, prev, code, before, after, ref_after, o, o_ref in run_chain(
            steps("uniform", seed=44, n=2), bad=bad):
        if i == 0:
            continue
        assert code & binding.GDN_DEVERR_ACCEPTED
        slot = int(prob.slot_ids[bad])
        assert np.array_equal(after[slot].view(np.int32), before[slot].view(np.int32))
        c0, c1 = int(prob.cu_seqlens[bad]), int(prob.cu_seqlens[bad + 1])
        assert np.isnan(o[c0:c1]).all(), "the skipped request's outputs were written"
        good = [r for r in range(prob.batch) if r != bad]
        rows = np.concatenate([np.arange(prob.cu_seqlens[r], prob.cu_seqlens[r + 1])
                               for r in good]).astype(int)
        assert rel_err(o[rows], o_ref[rows]) <= TOL


@pytest.mark.parametrize("name", ["b32_h32_d128_t16", "b64_h32_d128_t16_x24",
                                  "b128_h32_d128_ragged16"])
def test_full_size_every_unit(name):
    """The benchmark's workloads at full size, in the launch the benchmark times
    (the previous step is the same problem, as in bench.py --order lagged):
    every unit against the oracle (commit the previous step's prefix, then
    verify), every committed state within the tolerance."""
    prob = inputs.make_problem(name)
    units = np.arange(prob.units)
    # oracle: the state after a_prev rows of the previous step (or the checkpoint), then verify
    _, s_acc = oracle.run_units(prob, units, want_o=False)
    s0 = prob.s0.reshape(prob.units, prob.dk, prob.dv)[units].astype(np.float64)
    acc_u = np.array([prob.accepted[int(u) // prob.heads] for u in units])
    s_mid = np.where(acc_u[:, None, None] > 0, s_acc, s0)
    o_ref, _ = oracle.run_units(prob, units, s0=s_mid, want_state=False)
    d = staging.DeviceProblem(prob, "cuda")
    w_prev = torch.zeros((prob.n_tok, prob.heads, prob.dv), device="cuda")
    w = torch.zeros_like(w_prev)
    # the previous step's W: what its own call (from the same checkpoints) writes
    binding.gdn_commit_verify(d.c, None, d.o, w_prev)
    prev = binding.make_prev_step(k=d.k, alpha=d.alpha, w=w_prev, accepted=d.accepted,
                                  max_T=prob.max_T, cu_seqlens=d.cu_seqlens)
    d.o.fill_(float("nan"))
    binding.gdn_commit_verify(d.c, prev, d.o, w)
    torch.cuda.synchronize()
    assert binding.gdn_read_device_error(d.c) == 0
    o = d.o.cpu().numpy()
    pool = d.pool.cpu().numpy()
    got = np.zeros_like(o_ref)
    for n, u in enumerate(units):
        r, h = divmod(int(u), prob.heads)
        c0, L = int(prob.cu_seqlens[r]), int(prob.lengths[r])
        got[n, :L] = o[c0:c0 + L, h]
        if prob.accepted[r] > 0:
            assert rel_err(pool[int(prob.slot_ids[r]), h], s_acc[n]) <= TOL, f"unit {u} state"
    assert rel_err(got, o_ref) <= TOL
    del d
    torch.cuda.empty_cache()
