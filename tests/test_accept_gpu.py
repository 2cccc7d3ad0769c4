"""GPU parity of the greedy accept-length kernel (gdn_accept_prefix) against the
oracle, bit for bit: on the token ids of every workload (where it must also
give back the workload's own accepted lengths), on long and ragged blocks
(several 32-row windows, empty requests) and on bad ragged offsets."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decode_gated_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def run(draft, target, batch, max_T, cu=None, sentinel=-7):
    dev = torch.device("cuda")
    d = torch.from_numpy(np.ascontiguousarray(draft, np.int32)).to(dev)
    t = torch.from_numpy(np.ascontiguousarray(target, np.int32)).to(dev)
    c = None if cu is None else torch.from_numpy(np.ascontiguousarray(cu, np.int32)).to(dev)
    acc = torch.full((batch,), sentinel, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding.gdn_accept_prefix(d, t, acc, max_T, cu_seqlens=c, dev_err=err)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("name", sorted(inputs.WORKLOADS))
def test_workload_ids_give_back_accepted(name):
    prob = inputs.make_problem(name)
    draft, target = inputs.make_token_ids(prob, seed=5)
    want = oracle.accept_prefix(draft, target, prob.cu_seqlens)
    assert np.array_equal(want, prob.accepted)
    for cu in ((prob.cu_seqlens if prob.ragged else None), prob.cu_seqlens):
        got, err = run(draft, target, prob.batch, prob.max_T, cu)
        assert err == 0
        assert np.array_equal(got, want)


@pytest.mark.parametrize("seed,batch,max_T,p", [
    (1, 300, 1024, 0.002),   # long blocks: many 32-row windows before the first difference
    (2, 3000, 16, 0.2),      # many requests, several warps per block and blocks
    (3, 257, 100, 0.05),
    (4, 64, 33, 0.0),        # no difference anywhere: accepted = T_r
    (5, 64, 31, 1.0),        # difference everywhere: accepted = 0
])
def test_random_blocks(seed, batch, max_T, p):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, max_T + 1, size=batch)
    lens[:3] = [0, max_T, 1]
    cu, draft, target = inputs.random_token_ids(lens, seed, p_differ=p)
    want = oracle.accept_prefix(draft, target, cu)
    got, err = run(draft, target, batch, max_T, cu)
    assert err == 0
    assert np.array_equal(got, want)


def test_uniform_rows():
    batch, T = 50, 24
    cu, draft, target = inputs.random_token_ids([T] * batch, 9, p_differ=0.08)
    got, err = run(draft, target, batch, T, None)
    assert err == 0
    assert np.array_equal(got, oracle.accept_prefix(draft, target, cu))


def test_bad_ragged_offsets_flag_and_skip():
    _, draft, target = inputs.random_token_ids([4, 6, 3, 5], 11, p_differ=0.3)
    # request 1 is longer than max_T = 6, request 2 has a negative length,
    # request 4 runs past n_tok = 18; requests 0 and 3 are well formed
    bad = np.array([0, 4, 11, 10, 13, 19], dtype=np.int32)
    got, err = run(draft, target, 5, 6, bad)
    assert err == binding.GDN_DEVERR_SEQLEN
    assert got[1] == -7 and got[2] == -7 and got[4] == -7   # skipped: not written
    assert got[0] == oracle.accept_prefix(draft, target, [0, 4])[0]
    assert got[3] == oracle.accept_prefix(draft, target, [10, 13])[0]


def test_empty_batch():
    got, err = run(np.zeros(1), np.zeros(1), 0, 4, None)
    assert got.size == 0 and err == 0
