"""The seeded input generator (shared by the CUDA path and the oracle) against
its stated recipe: bf16 rounding, value distributions, slot ids, accepted
lengths, ragged lengths, determinism and the layer-shared metadata."""
import numpy as np
import pytest
import torch

from speculative_decode_gated_gb300 import inputs


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-8, 8, 20000),
        # exact ties: halfway between two bf16 values, both parities of the kept bit
        (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        -(np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, np.float32(3.4e38), np.float32(1e-40)], np.float32),
    ]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = inputs.round_to_bf16(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_bf16_bits_rejects_unrounded_values():
    assert inputs.bf16_bits(np.array([1.0, -2.5], np.float32)).tolist() == [0x3F80, 0xC020]
    with pytest.raises(ValueError):
        inputs.bf16_bits(np.array([1.0 + 2.0 ** -10], np.float32))


@pytest.fixture(scope="module")
def b32():
    return inputs.make_problem("b32_h32_d128_t16")


def test_recipe_values(b32):
    p = b32
    for x in (p.q, p.k):
        assert np.array_equal(x, inputs.round_to_bf16(x))  # stored as bf16
        nrm = np.linalg.norm(x.astype(np.float64), axis=-1)
        assert np.all(np.abs(nrm - 1.0) < 2e-2)  # unit rows, up to bf16 rounding
    assert np.array_equal(p.v, inputs.round_to_bf16(p.v))
    assert abs(float(p.v.std()) - 1.0) < 0.02
    assert np.all((p.alpha > 0) & (p.alpha < 1)) and np.all((p.beta > 0) & (p.beta < 1))
    # alpha = 1 / (1 + e^x) and beta = sigmoid(y) with x, y ~ N(0, 1): both have mean 1/2
    assert abs(float(p.alpha.mean()) - 0.5) < 0.01 and abs(float(p.beta.mean()) - 0.5) < 0.01
    assert abs(float(p.s0.std()) - 0.1) < 0.002 and abs(float(p.s0.mean())) < 0.002
    assert p.q.shape == (32 * 16, 32, 128) and p.s0.shape == (32, 32, 128, 128)


def test_recipe_metadata(b32):
    p = b32
    assert len(set(p.slot_ids.tolist())) == p.batch
    assert np.all((p.slot_ids >= 0) & (p.slot_ids < p.pool_slots))
    assert not np.array_equal(np.sort(p.slot_ids), np.arange(p.batch))  # not the first slots
    assert np.all((p.accepted >= 0) & (p.accepted <= p.lengths))
    assert 10.0 < float(p.accepted.mean()) < 14.0  # Binomial(16, 0.75): mean 12
    assert np.array_equal(p.cu_seqlens, np.arange(p.batch + 1) * 16)


def test_ragged_workload():
    p = inputs.make_problem("b128_h32_d128_ragged16")
    assert p.ragged and p.batch == 128 and p.pool_slots == 1024
    assert np.all((p.lengths >= 1) & (p.lengths <= 16)) and p.max_T == int(p.lengths.max())
    assert p.n_tok == int(p.lengths.sum()) == p.q.shape[0]
    assert np.all((p.accepted >= 0) & (p.accepted <= p.lengths))


def test_determinism_and_layer_sharing():
    kw = dict(batch=5, heads=2, dk=32, dv=32, T=6, pool_slots=11, accept="uniform", seed=77)
    a0 = inputs.make_custom(layer=0, **kw)
    a0b = inputs.make_custom(layer=0, **kw)
    a1 = inputs.make_custom(layer=1, **kw)
    for f in ("q", "k", "v", "alpha", "beta", "s0", "slot_ids", "accepted"):
        assert np.array_equal(getattr(a0, f), getattr(a0b, f)), f
    # one request keeps its slot and accepted length in every layer
    assert np.array_equal(a0.slot_ids, a1.slot_ids) and np.array_equal(a0.accepted, a1.accepted)
    assert not np.array_equal(a0.q, a1.q) and not np.array_equal(a0.s0, a1.s0)


def test_log_gate_is_the_same_draw_in_log_space():
    kw = dict(batch=3, heads=2, dk=32, dv=32, T=5, accept="uniform", seed=5)
    a = inputs.make_custom(**kw)
    g = inputs.make_custom(gate="log", **kw)
    assert g.gate == "log" and np.all(g.alpha < 0)
    assert np.allclose(np.exp(g.alpha.astype(np.float64)), a.alpha, rtol=1e-6, atol=0)
    assert np.array_equal(a.q, g.q) and np.array_equal(a.beta, g.beta)


def test_token_ids_reproduce_accepted_lengths():
    p = inputs.make_problem("b128_h32_d128_ragged16")
    draft, target = inputs.make_token_ids(p, seed=5)
    for r in range(p.batch):
        c0, T = int(p.cu_seqlens[r]), int(p.lengths[r])
        a = 0
        while a < T and draft[c0 + a] == target[c0 + a]:
            a += 1
        assert a == p.accepted[r]


def test_batch_override_keeps_the_recipe():
    """`batch` replaces only the number of requests of a uniform workload."""
    from speculative_decode_gated_gb300 import inputs
    base = inputs.make_problem("b32_h32_d128_t16")
    p = inputs.make_problem("b32_h32_d128_t16", batch=19)
    assert p.batch == 19 and p.units == 19 * 32
    assert (p.heads, p.dk, p.dv, p.max_T, p.pool_slots) == \
        (base.heads, base.dk, base.dv, base.max_T, base.pool_slots)
    assert len(set(p.slot_ids.tolist())) == 19
    for bad in (0, base.pool_slots + 1):
        with pytest.raises(ValueError):
            inputs.make_problem("b32_h32_d128_t16", batch=bad)
    with pytest.raises(ValueError):
        inputs.make_problem("b128_h32_d128_ragged16", batch=64)
