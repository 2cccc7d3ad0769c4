"""Pins of the float64 oracle: checks against things other than the oracle itself.

Each pin takes the oracle library handle, so the same checks run against the
real oracle (tests/test_oracle_pins.py) and against copies with a planted
mistake (tests/test_oracle_mutants.py), which must fail at least one of them.

What pins what (the recurrence is the gated delta rule that the OCRia write-up
"OCRia 推理栈：单卡 B200 提速近 10 倍" has ReplaySSM replay over a Gated DeltaNet
state, section "Make speculative verification cheaper"):
  * hand cases    - two hand-worked fixtures under tests/golden/ (exact fractions)
  * identity      - beta = 0, alpha = 1: o_t = S_0 q_t, a plain matrix-vector product
  * decay only    - beta = 0: S_t = (prod alpha) S_0, closed form
  * forget        - alpha_t = 0: S_t = beta_t v_t k_t^T, closed form
  * retrieval     - beta = 1, |k| = 1: S_t k_t = v_t; alpha = 1 and orthonormal
                    keys keep every earlier association: S_T k_s = v_s
  * chunk form    - the WY / chunked closed form (a different algorithm, numpy
                    linear solve) gives the same outputs and states
  * equivariance  - rotating key space or mapping value space moves the outputs
                    and states as the algebra says (dk != dv catches transposes)
  * linearity     - outputs and states are linear in (S_0, V) jointly
  * commit/verify - the state after a accepted tokens equals what verification's
                    outputs reveal about it (probe tokens), for every a in [0, T]
  * rollback      - a = 0 leaves the slot bit-identical; unnamed slots never change
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import oracle
from speculative_decode_gated_gb300.inputs import Problem, make_custom

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def problem_from_arrays(s0_tile, alpha, beta, k, v, q, accepted=None, name="explicit"):
    """One request, one head, T tokens, from explicit float arrays."""
    s0_tile = np.asarray(s0_tile, np.float64)
    dk, dv = s0_tile.shape
    T = len(alpha)
    f32 = lambda x, d: np.asarray(x, np.float64).reshape(T, 1, d)
    return Problem(name=name, batch=1, heads=1, dk=dk, dv=dv, max_T=T, ragged=False,
                   qkv_dtype="fp32", cu_seqlens=np.array([0, T], np.int32),
                   q=f32(q, dk), k=f32(k, dk), v=f32(v, dv),
                   alpha=np.asarray(alpha, np.float64).reshape(T, 1),
                   beta=np.asarray(beta, np.float64).reshape(T, 1),
                   pool_slots=1, slot_ids=np.zeros(1, np.int32),
                   accepted=np.array([T if accepted is None else accepted], np.int32),
                   s0=s0_tile.reshape(1, 1, dk, dv))


def load_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            vals[key] = np.array([float(Fraction(x)) for x in rest])
    return vals


def _states_at(lib, prob, accepted_values):
    out = []
    for a in accepted_values:
        _, s = oracle.run_units(prob, accepted=np.array([a]), want_o=False, lib=lib)
        out.append(s[0])
    return out


# --------------------------------------------------------------------------- pins

def pin_hand_cases(lib):
    for name in ("hand_2x2_t2.txt", "hand_dk3_dv2_t2.txt"):
        g = load_golden(name)
        dk, dv, T = int(g["dk"][0]), int(g["dv"][0]), int(g["T"][0])
        prob = problem_from_arrays(g["s0"].reshape(dk, dv), g["alpha"], g["beta"],
                                   g["k"], g["v"], g["q"])
        o, _ = oracle.run_units(prob, want_state=False, lib=lib)
        assert np.array_equal(o[0], g["o"].reshape(T, dv)), (name, o[0])
        for a, s in enumerate(_states_at(lib, prob, range(T + 1))):
            assert np.array_equal(s, g[f"state_{a}"].reshape(dk, dv)), (name, a, s)


def _random_unit(seed, dk, dv, T, **over):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((T, dk))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    arrs = dict(s0_tile=0.1 * rng.standard_normal((dk, dv)),
                alpha=1.0 / (1.0 + np.exp(rng.standard_normal(T))),
                beta=1.0 / (1.0 + np.exp(-rng.standard_normal(T))),
                k=k, v=rng.standard_normal((T, dv)), q=q)
    arrs.update(over)
    return arrs


def pin_identity_is_gemv(lib):
    a = _random_unit(1, 7, 5, 6, alpha=np.ones(6), beta=np.zeros(6))
    o, s = oracle.run_units(problem_from_arrays(**a), lib=lib)
    expect = a["q"] @ a["s0_tile"]            # o_t[j] = sum_i q_t[i] tile[i][j]
    assert np.allclose(o[0], expect, rtol=0, atol=1e-15)
    assert np.array_equal(s[0], a["s0_tile"])


def pin_decay_only(lib):
    a = _random_unit(2, 6, 9, 5, beta=np.zeros(5))
    o, s = oracle.run_units(problem_from_arrays(**a), lib=lib)
    gam = np.cumprod(a["alpha"])
    expect = gam[:, None] * (a["q"] @ a["s0_tile"])
    assert np.allclose(o[0], expect, rtol=1e-14, atol=1e-16)
    assert np.allclose(s[0], gam[-1] * a["s0_tile"], rtol=1e-14, atol=1e-18)


def pin_full_forget(lib):
    a = _random_unit(3, 6, 4, 3, alpha=np.array([0.3, 0.0, 0.7]))
    prob = problem_from_arrays(**a, accepted=2)
    _, s = oracle.run_units(prob, lib=lib)
    # alpha_2 = 0 erases the past: S_2 = beta_2 v_2 k_2^T, tile = beta_2 k_2 v_2^T
    expect = a["beta"][1] * np.outer(a["k"][1], a["v"][1])
    assert np.allclose(s[0], expect, rtol=1e-14, atol=1e-16)


def pin_delta_retrieval(lib):
    dk, dv, T = 8, 5, 6
    a = _random_unit(4, dk, dv, T, beta=np.ones(T))
    # beta = 1 and |k_t| = 1: the newest key retrieves its value exactly,
    # whatever alpha is.  Probe with q_t = k_t.
    b = dict(a, q=a["k"])
    o, _ = oracle.run_units(problem_from_arrays(**b), lib=lib, want_state=False)
    assert np.allclose(o[0], a["v"], rtol=0, atol=1e-13)
    # alpha = 1 and orthonormal keys: every stored association survives.
    rng = np.random.default_rng(5)
    keys = np.linalg.qr(rng.standard_normal((dk, dk)))[0].T[:T]
    c = dict(a, k=keys, q=keys, alpha=np.ones(T))
    _, s = oracle.run_units(problem_from_arrays(**c), lib=lib)
    tile = s[0]
    for t in range(T):
        assert np.allclose(keys[t] @ tile, a["v"][t], rtol=0, atol=1e-13)


def chunk_form(s0_tile, alpha, beta, k, v, q):
    """WY / chunked closed form of the same recurrence, numpy, tile orientation.

    gamma_t = prod_{r<=t} alpha_r,  D[t, s] = prod_{s<r<=t} alpha_r,
    (I + A) W = diag(beta) (V - diag(gamma) K H_0),  A[t, s] = beta_t D[t, s] k_t.k_s  (s < t),
    O = diag(gamma) Q H_0 + (D * Q K^T, lower incl. diagonal) W,
    H_a = gamma_{a-1} H_0 + sum_{s<a} D[a-1, s] k_s w_s^T.
    """
    T = len(alpha)
    D = np.zeros((T, T))
    for t in range(T):
        for s in range(t + 1):
            D[t, s] = np.prod(alpha[s + 1:t + 1])
    gam = np.cumprod(alpha)
    A = np.tril(beta[:, None] * D * (k @ k.T), -1)
    W = np.linalg.solve(np.eye(T) + A, beta[:, None] * (v - gam[:, None] * (k @ s0_tile)))
    O = gam[:, None] * (q @ s0_tile) + (np.tril(D) * (q @ k.T)) @ W
    states = [s0_tile.copy()]
    for a in range(1, T + 1):
        states.append(gam[a - 1] * s0_tile + (k[:a].T * D[a - 1, :a]) @ W[:a])
    return O, states


def pin_chunk_form(lib):
    for seed, (dk, dv, T) in enumerate([(16, 12, 9), (32, 32, 16), (5, 7, 3)]):
        a = _random_unit(10 + seed, dk, dv, T)
        prob = problem_from_arrays(**a)
        o, _ = oracle.run_units(prob, lib=lib, want_state=False)
        O, states = chunk_form(**a)
        scale = np.abs(O).max()
        assert np.abs(o[0] - O).max() <= 1e-12 * scale
        for a_len, s in enumerate(_states_at(lib, prob, range(T + 1))):
            assert np.abs(s - states[a_len]).max() <= 1e-12 * np.abs(states[a_len]).max()


def pin_equivariance(lib):
    dk, dv, T = 6, 4, 5
    a = _random_unit(20, dk, dv, T)
    o, s = oracle.run_units(problem_from_arrays(**a), lib=lib)
    rng = np.random.default_rng(21)
    R = np.linalg.qr(rng.standard_normal((dk, dk)))[0]          # key-space rotation
    P = rng.standard_normal((dv, dv))                            # any value-space map
    b = dict(a, k=a["k"] @ R.T, q=a["q"] @ R.T, s0_tile=R @ a["s0_tile"])
    o2, s2 = oracle.run_units(problem_from_arrays(**b), lib=lib)
    assert np.allclose(o2[0], o[0], rtol=0, atol=1e-13)          # outputs unchanged
    assert np.allclose(s2[0], R @ s[0], rtol=0, atol=1e-13)      # state rotates with keys
    c = dict(a, v=a["v"] @ P.T, s0_tile=a["s0_tile"] @ P.T)
    o3, s3 = oracle.run_units(problem_from_arrays(**c), lib=lib)
    assert np.allclose(o3[0], o[0] @ P.T, rtol=0, atol=1e-12)    # outputs mapped by P
    assert np.allclose(s3[0], s[0] @ P.T, rtol=0, atol=1e-12)


def pin_linearity(lib):
    a = _random_unit(30, 9, 7, 6)
    b = _random_unit(31, 9, 7, 6)
    sum_ = dict(a, s0_tile=a["s0_tile"] + b["s0_tile"], v=a["v"] + b["v"])
    b = dict(a, s0_tile=b["s0_tile"], v=b["v"])
    oa, sa = oracle.run_units(problem_from_arrays(**a), lib=lib)
    ob, sb = oracle.run_units(problem_from_arrays(**b), lib=lib)
    os_, ss = oracle.run_units(problem_from_arrays(**sum_), lib=lib)
    assert np.allclose(os_, oa + ob, rtol=0, atol=1e-13)
    assert np.allclose(ss, sa + sb, rtol=0, atol=1e-13)


def pin_commit_matches_verify(lib):
    """The committed state after a tokens is what verification's own outputs
    reveal: replay a tokens, then dk probe tokens with alpha = 1, beta = 0,
    q = e_i; probe i outputs S_a e_i, which is row i of the stored tile."""
    dk, dv, T = 6, 5, 7
    a = _random_unit(40, dk, dv, T)
    prob = problem_from_arrays(**a)
    eye = np.eye(dk)
    for a_len, s in enumerate(_states_at(lib, prob, range(T + 1))):
        n = a_len + dk
        probe = problem_from_arrays(
            a["s0_tile"],
            np.concatenate([a["alpha"][:a_len], np.ones(dk)]),
            np.concatenate([a["beta"][:a_len], np.zeros(dk)]),
            np.concatenate([a["k"][:a_len], eye]),
            np.concatenate([a["v"][:a_len], np.zeros((dk, dv))]),
            np.concatenate([a["q"][:a_len], eye]))
        o, _ = oracle.run_units(probe, lib=lib, want_state=False)
        assert np.array_equal(o[0][a_len:n], s), a_len


def pin_composition(lib):
    """Verifying T tokens equals committing t of them and verifying the rest."""
    dk, dv, T, t = 8, 6, 9, 4
    a = _random_unit(50, dk, dv, T)
    o, _ = oracle.run_units(problem_from_arrays(**a), lib=lib, want_state=False)
    _, s = oracle.run_units(problem_from_arrays(**a, accepted=t), lib=lib)
    rest = {key: (val[t:] if key != "s0_tile" else s[0]) for key, val in a.items()}
    o2, _ = oracle.run_units(problem_from_arrays(**rest), lib=lib, want_state=False)
    assert np.allclose(o[0][t:], o2[0], rtol=0, atol=1e-13)


def pin_rollback_bookkeeping(lib):
    prob = make_custom(batch=6, heads=3, dk=8, dv=4, T=5, qkv_dtype="fp32",
                       pool_slots=20, accept="uniform", seed=60)
    prob.accepted[:] = [0, 5, 2, 0, 1, 3]
    pool = np.full((20, 3, 8, 4), np.nan)
    pool.view(np.uint64)[...] = 0x7FF8DEADBEEF0001  # NaN with a payload
    for r, slot in enumerate(prob.slot_ids):
        pool[slot] = prob.s0[r]
    new = oracle.commit(prob, pool, lib=lib)
    touched = {int(prob.slot_ids[r]) for r in range(6) if prob.accepted[r] > 0}
    for slot in range(20):
        same = np.array_equal(new[slot].view(np.uint64), pool[slot].view(np.uint64))
        assert same == (slot not in touched), slot
    # The written slots hold the state after a_r tokens, which the oracle's
    # replay of exactly a_r tokens (a request cut to a_r tokens) reproduces.
    for r in range(6):
        a_r = int(prob.accepted[r])
        if a_r == 0:
            continue
        for h in range(3):
            rows = slice(int(prob.cu_seqlens[r]), int(prob.cu_seqlens[r]) + a_r)
            cut = problem_from_arrays(prob.s0[r, h], prob.alpha[rows, h], prob.beta[rows, h],
                                      prob.k[rows, h], prob.v[rows, h], prob.q[rows, h])
            _, s = oracle.run_units(cut, lib=lib)
            assert np.array_equal(new[int(prob.slot_ids[r]), h], s[0])


ALL_PINS = [pin_hand_cases, pin_identity_is_gemv, pin_decay_only, pin_full_forget,
            pin_delta_retrieval, pin_chunk_form, pin_equivariance, pin_linearity,
            pin_commit_matches_verify, pin_composition, pin_rollback_bookkeeping]
