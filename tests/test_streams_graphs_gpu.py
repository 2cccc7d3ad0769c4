"""Use of the C ABI the way an engine drives it: calls captured in a CUDA graph
and replayed, and independent problems issued concurrently on two streams.
The kernels launch with programmatic dependent launch and keep no state
between calls, so both must reproduce the plain stream-ordered results bit
for bit."""
import numpy as np
import pytest
import torch

from parity import TOL, oracle_units, rel_err
from speculative_decode_gated_gb300 import binding, inputs, staging

pytestmark = pytest.mark.gpu


def _problems(n, seed):
    return [inputs.make_custom(name=f"graph{i}", batch=6, heads=4, dk=128, dv=128,
                               lengths=[16, 9, 1, 16, 12, 5], qkv_dtype="bf16", pool_slots=11,
                               accept="uniform", seed=seed, layer=i) for i in range(n)]


def _device(probs):
    return [staging.DeviceProblem(p, "cuda") for p in probs]


def _step(ds, stream):
    for d in ds:
        binding.gdn_verify(d.c, d.o, stream)
        binding.gdn_commit(d.c, d.accepted, stream)


def test_graph_replay_matches_stream_order():
    probs = _problems(3, 71)
    eager, captured = _device(probs), _device(probs)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _step(eager, s)
    torch.cuda.synchronize()
    # the first calls (set-up of the library's per-device state) run before capture
    warm = _device(probs)
    with torch.cuda.stream(s):
        _step(warm, s)
    torch.cuda.synchronize()
    pools0 = [d.pool.clone() for d in captured]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _step(captured, s)
    # capture records the launches without running them
    for d, p0 in zip(captured, pools0):
        assert torch.equal(d.pool.view(torch.int32), p0.view(torch.int32))
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, captured):
        assert binding.gdn_read_device_error(b.c) == 0
        assert torch.equal(a.o.view(torch.int32), b.o.view(torch.int32))
        assert torch.equal(a.pool.view(torch.int32), b.pool.view(torch.int32))
    # a second replay commits again from the committed states: it equals a
    # second eager step
    with torch.cuda.stream(s):
        _step(eager, s)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, captured):
        assert torch.equal(a.pool.view(torch.int32), b.pool.view(torch.int32))


def test_two_streams_concurrently():
    probs = _problems(4, 72)
    ref, conc = _device(probs), _device(probs)
    _step(ref, torch.cuda.current_stream())
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for i, d in enumerate(conc):
        s = streams[i % 2]
        with torch.cuda.stream(s):
            _step([d], s)
    torch.cuda.synchronize()
    for a, b, p in zip(ref, conc, probs):
        assert torch.equal(a.o.view(torch.int32), b.o.view(torch.int32))
        assert torch.equal(a.pool.view(torch.int32), b.pool.view(torch.int32))
    # and one of them against the oracle
    units = np.arange(probs[0].units)
    o_ref, _ = oracle_units(probs[0], units)
    got = np.zeros_like(o_ref)
    o = conc[0].o.cpu().numpy()
    for n, u in enumerate(units):
        r, h = divmod(int(u), probs[0].heads)
        c0, L = int(probs[0].cu_seqlens[r]), int(probs[0].lengths[r])
        got[n, :L] = o[c0:c0 + L, h]
    assert rel_err(got, o_ref) <= TOL
