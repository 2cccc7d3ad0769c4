"""Seeded synthetic inputs for the Gated DeltaNet speculative verify/commit path.

This module only draws random tensors with the shapes and value distributions of
the workloads and rounds them to their storage types.  It holds none of the
method's arithmetic, so both the CUDA path and the float64 oracle can be fed from
it without sharing any computation.

Value recipe (every workload):
  * q, k  ~ N(0, 1) per element, L2-normalised per (token, head) in float32, then
            rounded to bfloat16 (round to nearest even) unless the workload keeps
            float32.  The rounded values are the inputs; nothing renormalises them.
  * v     ~ N(0, 1), rounded the same way.
  * alpha = exp(-softplus(x)) = 1 / (1 + exp(x)),  x ~ N(0, 1), float32; with
            gate="log" the same draw is given in log space, g = -softplus(x),
            float32 (the kernel and the oracle then take alpha = exp(g)).
  * beta  = sigmoid(y) = 1 / (1 + exp(-y)),        y ~ N(0, 1), float32.
  * S0    = 0.1 * N(0, 1) per element, float32 (the standard deviation is 0.1).
  * slot ids: the first B entries of a random permutation of the pool slots
    (distinct and non-contiguous).
  * accepted length a_r: uniform on {0..T_r} or Binomial(T, 0.75), per workload.

The state tile of one (request, head) is stored key-index-major: element (i, j)
with i the key index (0..dk-1) and j the value index (0..dv-1), value index
contiguous.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

__all__ = [
    "Problem",
    "WORKLOADS",
    "round_to_bf16",
    "bf16_bits",
    "make_problem",
    "make_custom",
    "make_layers",
    "make_token_ids",
    "make_replay",
    "random_token_ids",
    "POOL_SENTINEL_BITS",
]

# Bit pattern (a quiet NaN with a payload) written into pool slots that no
# request names, so a stray write by any implementation shows up bitwise.
POOL_SENTINEL_BITS = 0x7FC0BEEF


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); float32 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bfloat16 encodings of float32 values that are already bf16-exact."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("bf16_bits: values are not bfloat16-representable")
    return (u >> 16).astype(np.uint16)


@dataclasses.dataclass
class Problem:
    """One layer-call's inputs, host side (numpy)."""

    name: str
    batch: int
    heads: int
    dk: int
    dv: int
    max_T: int
    ragged: bool
    qkv_dtype: str  # "bf16" or "fp32": how q, k, v are stored for the kernels
    cu_seqlens: np.ndarray  # int32 [B+1], token rows of request r are [cu[r], cu[r+1])
    q: np.ndarray  # float32 [N_tok][H][dk]
    k: np.ndarray  # float32 [N_tok][H][dk]
    v: np.ndarray  # float32 [N_tok][H][dv]
    alpha: np.ndarray  # float32 [N_tok][H]
    beta: np.ndarray  # float32 [N_tok][H]
    pool_slots: int
    slot_ids: np.ndarray  # int32 [B]
    accepted: np.ndarray  # int32 [B]
    s0: np.ndarray  # float32 [B][H][dk][dv], the state held in slot slot_ids[r]
    gate: str = "alpha"  # what `alpha` holds: the decay alpha, or "log": g = log(alpha)

    @property
    def n_tok(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def lengths(self) -> np.ndarray:
        return np.diff(self.cu_seqlens).astype(np.int32)

    @property
    def units(self) -> int:
        return self.batch * self.heads


def _draw_tokens(rng: np.random.Generator, n_tok: int, heads: int, dk: int, dv: int,
                 qkv_dtype: str, gate: str = "alpha"):
    def unit_rows(d):
        x = rng.standard_normal((n_tok, heads, d), dtype=np.float32)
        nrm = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
        return (x / np.maximum(nrm, np.float32(1e-30))).astype(np.float32)

    q = unit_rows(dk)
    k = unit_rows(dk)
    v = rng.standard_normal((n_tok, heads, dv), dtype=np.float32)
    if qkv_dtype == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    elif qkv_dtype != "fp32":
        raise ValueError(qkv_dtype)
    x = rng.standard_normal((n_tok, heads), dtype=np.float32).astype(np.float64)
    y = rng.standard_normal((n_tok, heads), dtype=np.float32).astype(np.float64)
    if gate == "log":  # the same decay drawn in log space: g = -softplus(x)
        alpha = (-np.log1p(np.exp(x))).astype(np.float32)
    elif gate == "alpha":
        alpha = (1.0 / (1.0 + np.exp(x))).astype(np.float32)
    else:
        raise ValueError(gate)
    beta = (1.0 / (1.0 + np.exp(-y))).astype(np.float32)
    return q, k, v, alpha, beta


def _draw_accepted(rng: np.random.Generator, lengths: np.ndarray, dist: str) -> np.ndarray:
    if dist == "uniform":
        return np.array([rng.integers(0, int(L) + 1) for L in lengths], dtype=np.int32)
    if dist == "binom":
        a = rng.binomial(int(lengths.max()), 0.75, size=len(lengths))
        return np.minimum(a, lengths).astype(np.int32)
    if dist == "full":
        return lengths.astype(np.int32).copy()
    if dist == "zero":
        return np.zeros(len(lengths), dtype=np.int32)
    raise ValueError(dist)


def make_custom(*, batch: int, heads: int, dk: int, dv: int,
                T: Optional[int] = None, lengths: Optional[Sequence[int]] = None,
                qkv_dtype: str = "bf16", pool_slots: Optional[int] = None,
                accept: str = "uniform", seed: int = 0, layer: int = 0,
                slot_ids: Optional[np.ndarray] = None,
                accepted: Optional[np.ndarray] = None,
                name: str = "custom", gate: str = "alpha") -> Problem:
    """Draw one problem.  Give either a uniform draft length T or per-request lengths.

    Slot ids and accepted lengths come from a stream that does not depend on
    `layer`, so the layers of one multi-layer step share them (one request keeps
    its slot index and its accepted length in every layer).
    """
    if (T is None) == (lengths is None):
        raise ValueError("give exactly one of T or lengths")
    ragged = lengths is not None
    lens = np.full(batch, T, dtype=np.int32) if T is not None else np.asarray(lengths, np.int32)
    if lens.shape != (batch,) or np.any(lens < 0):
        raise ValueError("bad lengths")
    cu = np.zeros(batch + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    pool_slots = batch if pool_slots is None else pool_slots
    meta = np.random.default_rng(np.random.SeedSequence([seed, 0]))
    data = np.random.default_rng(np.random.SeedSequence([seed, 1 + layer]))
    if slot_ids is None:
        slot_ids = meta.permutation(pool_slots)[:batch].astype(np.int32)
    if accepted is None:
        accepted = _draw_accepted(meta, lens, accept)
    q, k, v, alpha, beta = _draw_tokens(data, int(cu[-1]), heads, dk, dv, qkv_dtype, gate)
    s0 = (np.float32(0.1) * data.standard_normal((batch, heads, dk, dv), dtype=np.float32))
    return Problem(name=name, batch=batch, heads=heads, dk=dk, dv=dv,
                   max_T=int(lens.max()) if batch else 0, ragged=ragged,
                   qkv_dtype=qkv_dtype, cu_seqlens=cu, q=q, k=k, v=v, alpha=alpha,
                   beta=beta, pool_slots=pool_slots,
                   slot_ids=np.asarray(slot_ids, np.int32),
                   accepted=np.asarray(accepted, np.int32), s0=s0.astype(np.float32), gate=gate)


# The five workloads: (name, recipe).  Seeds are 1000 + workload index.
WORKLOADS = {
    # batch 1, 2 heads, dk = dv = 32, 4 draft tokens, everything float32.
    "tiny_b1_h2_d32_t4": dict(batch=1, heads=2, dk=32, dv=32, T=4, qkv_dtype="fp32",
                              pool_slots=1, accept="uniform", seed=1000),
    # batch 8, 16 heads, dk = dv = 128, 8 draft tokens, 64-slot pool.
    "b8_h16_d128_t8": dict(batch=8, heads=16, dk=128, dv=128, T=8, qkv_dtype="bf16",
                           pool_slots=64, accept="uniform", seed=1001),
    # batch 32, 32 heads, 16 draft tokens, 256-slot pool, ~12 accepted tokens.
    "b32_h32_d128_t16": dict(batch=32, heads=32, dk=128, dv=128, T=16, qkv_dtype="bf16",
                             pool_slots=256, accept="binom", seed=1002),
    # batch 64, 32 heads, 16 draft tokens, 24 layers, 512 slots per layer.
    "b64_h32_d128_t16_x24": dict(batch=64, heads=32, dk=128, dv=128, T=16, qkv_dtype="bf16",
                                 pool_slots=512, accept="binom", seed=1003, layers=24),
    # batch 128 ragged (draft length uniform in 1..16), 32 heads, 1024-slot pool.
    "b128_h32_d128_ragged16": dict(batch=128, heads=32, dk=128, dv=128, lengths="u1_16",
                                   qkv_dtype="bf16", pool_slots=1024, accept="uniform",
                                   seed=1004),
}


def _recipe_kwargs(name: str) -> dict:
    spec = dict(WORKLOADS[name])
    spec.pop("layers", None)
    if spec.get("lengths") == "u1_16":
        rng = np.random.default_rng(np.random.SeedSequence([spec["seed"], 999]))
        spec["lengths"] = rng.integers(1, 17, size=spec["batch"]).astype(np.int32)
    return spec


def make_problem(name: str, layer: int = 0, draft: Optional[int] = None,
                 gate: str = "alpha", batch: Optional[int] = None) -> Problem:
    """The named workload (one layer of it for the multi-layer one).  `draft`
    replaces the draft length of a uniform workload (accepted lengths keep
    their distribution, over the new length); `batch` replaces its number of
    requests (at most its pool's slots); gate="log" draws the same decay in
    log space (the log-gate variant)."""
    kw = _recipe_kwargs(name)
    if draft is not None:
        if "T" not in kw:
            raise ValueError(f"{name} has ragged drafts")
        kw["T"] = int(draft)
    if batch is not None:
        if "T" not in kw:
            raise ValueError(f"{name} has ragged drafts")
        if not 1 <= int(batch) <= kw["pool_slots"]:
            raise ValueError(f"batch {batch} outside 1..{kw['pool_slots']}")
        kw["batch"] = int(batch)
    return make_custom(name=name, layer=layer, gate=gate, **kw)


def make_layers(name: str) -> List[Problem]:
    """Every layer of a workload (one element for single-layer workloads)."""
    n = WORKLOADS[name].get("layers", 1)
    return [make_problem(name, layer=l) for l in range(n)]


def make_token_ids(prob: Problem, seed: int = 0, vocab: int = 151936):
    """Draft and target token ids (int32 [N_tok] each) whose greedy prefix match
    gives back the problem's accepted lengths: in request r the ids agree at
    rows t < a_r, differ at row a_r (when a_r < T_r) and are drawn
    independently after it (so they may agree again there)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 77]))
    n = prob.n_tok
    draft = rng.integers(0, vocab, size=n).astype(np.int64)
    target = rng.integers(0, vocab, size=n).astype(np.int64)
    for r in range(prob.batch):
        c0, T, a = int(prob.cu_seqlens[r]), int(prob.lengths[r]), int(prob.accepted[r])
        target[c0:c0 + a] = draft[c0:c0 + a]
        if a < T:
            target[c0 + a] = (draft[c0 + a] + 1 + rng.integers(0, vocab - 1)) % vocab
    return draft.astype(np.int32), target.astype(np.int32)


def random_token_ids(lengths: Sequence[int], seed: int, p_differ: float = 0.1, vocab: int = 50):
    """cu_seqlens and draft/target ids where each row's target differs from the
    draft with probability p_differ (independently per row)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 78]))
    lens = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    n = int(cu[-1])
    draft = rng.integers(0, vocab, size=n)
    differ = rng.random(n) < p_differ
    target = np.where(differ, (draft + 1 + rng.integers(0, vocab - 1, size=n)) % vocab, draft)
    return cu, draft.astype(np.int32), target.astype(np.int32)


def make_replay(prob: Problem, capacity: int, seed: int = 0,
                len_in: Optional[np.ndarray] = None, dense: bool = True) -> dict:
    """A ReplaySSM buffer for `prob`: `capacity` rows per pool slot in the token
    layout (k [slots*C][H][dk], v [slots*C][H][dv], alpha/beta [slots*C][H]),
    and len_in[slot], the rows already buffered.  For a named slot len_in is
    uniform on [0, C - T_r] (room for the drafts) unless given; its rows are
    drawn like the workload's tokens, and request r's drafts are copied to
    rows slot*C + len_in + [0, T_r).  Rows of unnamed slots are zero (alpha 1).
    dense=False returns only the named slots' rows ("slots": their ids in
    order, k/v/alpha/beta with len(slots) * C rows), for large pools."""
    C = int(capacity)
    if prob.batch and C < prob.max_T:
        raise ValueError("capacity below the draft length")
    rng = np.random.default_rng(np.random.SeedSequence([seed, 90]))
    S, H = prob.pool_slots, prob.heads
    named = [int(s) for s in prob.slot_ids]
    where = {s: i for i, s in enumerate(named)}
    R = S if dense else len(named)
    k = np.zeros((R * C, H, prob.dk), np.float32)
    v = np.zeros((R * C, H, prob.dv), np.float32)
    alpha = np.full((R * C, H), 0.0 if prob.gate == "log" else 1.0, np.float32)  # decay 1
    beta = np.zeros((R * C, H), np.float32)
    lens = np.zeros(S, np.int32) if len_in is None else np.array(len_in, np.int32, copy=True)
    for r in range(prob.batch):
        s, T, c0 = int(prob.slot_ids[r]), int(prob.lengths[r]), int(prob.cu_seqlens[r])
        if len_in is None:
            lens[s] = rng.integers(0, C - T + 1)
        _, ks, vs, al, be = _draw_tokens(rng, C, H, prob.dk, prob.dv, prob.qkv_dtype, prob.gate)
        n = int(lens[s])
        if n + T > C:
            raise ValueError("buffered rows plus drafts exceed the capacity")
        ks[n:n + T], vs[n:n + T] = prob.k[c0:c0 + T], prob.v[c0:c0 + T]
        al[n:n + T], be[n:n + T] = prob.alpha[c0:c0 + T], prob.beta[c0:c0 + T]
        i = s if dense else where[s]
        k[i * C:(i + 1) * C], v[i * C:(i + 1) * C] = ks, vs
        alpha[i * C:(i + 1) * C], beta[i * C:(i + 1) * C] = al, be
    out = dict(capacity=C, k=k, v=v, alpha=alpha, beta=beta, len_in=lens)
    if not dense:
        out["slots"] = np.array(named, np.int64)
        out["pool_slots"] = S
    return out
