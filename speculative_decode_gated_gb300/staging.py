"""Host problem (inputs.Problem, numpy) -> device tensors and a C problem.

Plain data movement: dtype casts of already-rounded values, copies, and the
placement of each request's checkpoint into its pool slot.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import binding
from .inputs import POOL_SENTINEL_BITS, Problem, bf16_bits


def qkv_tensor(x: np.ndarray, qkv_dtype: str, device) -> torch.Tensor:
    if qkv_dtype == "bf16":
        return torch.from_numpy(bf16_bits(x).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)


def new_pool(slots: int, heads: int, dk: int, dv: int, device, fill: str = "sentinel",
             layers: Optional[int] = None) -> torch.Tensor:
    shape = (slots, heads, dk, dv) if layers is None else (layers, slots, heads, dk, dv)
    pool = torch.empty(shape, dtype=torch.float32, device=device)
    if fill == "sentinel":
        pool.view(torch.int32).fill_(POOL_SENTINEL_BITS)
    elif fill == "zero":
        pool.zero_()
    elif fill != "none":
        raise ValueError(fill)
    return pool


def place_checkpoints(pool: torch.Tensor, prob: Problem) -> None:
    """pool[slot_ids[r]] <- the request's checkpoint tiles (all heads)."""
    idx = torch.from_numpy(prob.slot_ids.astype(np.int64)).to(pool.device)
    src = torch.from_numpy(np.ascontiguousarray(prob.s0, np.float32)).to(pool.device)
    pool.index_copy_(0, idx, src)


class DeviceProblem:
    """Device copies of one layer-call's inputs and the matching C problem."""

    def __init__(self, prob: Problem, device="cuda", pool: Optional[torch.Tensor] = None,
                 pool_fill: str = "sentinel", algo: int = binding.GDN_ALGO_AUTO,
                 with_dev_err: bool = True, place_s0: bool = True, o_bf16: bool = False):
        self.host = prob
        dev = torch.device(device)
        self.q = qkv_tensor(prob.q, prob.qkv_dtype, dev)
        self.k = qkv_tensor(prob.k, prob.qkv_dtype, dev)
        self.v = qkv_tensor(prob.v, prob.qkv_dtype, dev)
        self.alpha = torch.from_numpy(np.ascontiguousarray(prob.alpha, np.float32)).to(dev)
        self.beta = torch.from_numpy(np.ascontiguousarray(prob.beta, np.float32)).to(dev)
        self.slot_ids = torch.from_numpy(prob.slot_ids.astype(np.int32)).to(dev)
        self.accepted = torch.from_numpy(prob.accepted.astype(np.int32)).to(dev)
        self.cu_seqlens = (torch.from_numpy(prob.cu_seqlens.astype(np.int32)).to(dev)
                           if prob.ragged else None)
        if pool is None:
            pool = new_pool(prob.pool_slots, prob.heads, prob.dk, prob.dv, dev, pool_fill)
        self.pool = pool
        if place_s0:  # else the pool already holds the states (a later step)
            place_checkpoints(self.pool, prob)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev) if with_dev_err else None
        self.o = torch.zeros((prob.n_tok, prob.heads, prob.dv),
                             dtype=torch.bfloat16 if o_bf16 else torch.float32, device=dev)
        self.algo = algo
        # alpha holds g = log(alpha) for a log-space problem: the kernels apply expf
        self.flags = ((binding.GDN_FLAG_O_BF16 if o_bf16 else 0)
                      | (binding.GDN_FLAG_LOG_GATE if prob.gate == "log" else 0))
        self.c = self._make_c()

    def _make_c(self) -> binding.Problem:
        return binding.make_problem(q=self.q, k=self.k, v=self.v, alpha=self.alpha,
                                    beta=self.beta, pool=self.pool, slot_ids=self.slot_ids,
                                    max_T=self.host.max_T, cu_seqlens=self.cu_seqlens,
                                    dev_err=self.dev_err, algo=self.algo, flags=self.flags)

    def verify(self, stream=None):
        binding.gdn_verify(self.c, self.o, stream)

    def commit(self, stream=None):
        binding.gdn_commit(self.c, self.accepted, stream)

    def fused(self, stream=None):
        binding.gdn_verify_commit_fused(self.c, self.accepted, self.o, stream)

    def launcher(self, mode: str, stream):
        """A zero-argument callable issuing one call on `stream` with every
        argument marshalled in advance (for timing loops and graph capture)."""
        lib = binding.lib()
        ref = self.c.ref
        s = binding._stream(stream)
        o, acc = self.o.data_ptr(), self.accepted.data_ptr()
        fn = {"verify": lambda: lib.gdn_verify(ref, o, s),
              "commit": lambda: lib.gdn_commit(ref, acc, s),
              "fused": lambda: lib.gdn_verify_commit_fused(ref, acc, o, s)}[mode]

        def call():
            st = fn()
            if st != binding.GDN_OK:
                raise binding.GdnError(st, f"gdn {mode}")
        # The raw addresses above stay valid only while their tensors (and the
        # C problem) do: the callable keeps this object alive.
        call.keep = (self, self.c)
        return call


def share_request_arrays(dps) -> None:
    """Point every layer at the first layer's slot_ids, accepted and cu_seqlens
    device arrays (one step's requests are the same in every layer), as the
    layer-batch calls require.  The values must already be equal."""
    d0 = dps[0]
    for d in dps[1:]:
        for name in ("slot_ids", "accepted"):
            if not torch.equal(getattr(d, name), getattr(d0, name)):
                raise ValueError(f"layers disagree on {name}")
        d.slot_ids, d.accepted, d.cu_seqlens = d0.slot_ids, d0.accepted, d0.cu_seqlens
        d.c = d._make_c()


def layers_launcher(dps, mode: str, stream):
    """A zero-argument callable issuing one layer-batch call (verify, commit or
    fused) over all of `dps` on `stream`, every argument marshalled in advance."""
    lib = binding.lib()
    arr = binding.ProblemArray([d.c for d in dps])
    o = binding._ptr_array([d.o for d in dps])
    s = binding._stream(stream)
    acc = dps[0].accepted.data_ptr()
    fn = {"verify": lambda: lib.gdn_verify_layers(arr.ref, arr.n, o, s),
          "commit": lambda: lib.gdn_commit_layers(arr.ref, arr.n, acc, s),
          "fused": lambda: lib.gdn_verify_commit_fused_layers(arr.ref, arr.n, acc, o, s)}[mode]

    def call():
        st = fn()
        if st != binding.GDN_OK:
            raise binding.GdnError(st, f"gdn {mode} layers")
    call.keep = (list(dps), arr, o)  # the owners of the raw addresses above
    return call


class DeviceReplay:
    """Device copies of a ReplaySSM buffer (inputs.make_replay) and its C struct.
    len_out starts as a copy of len_in."""

    def __init__(self, buf: dict, qkv_dtype: str, device="cuda"):
        dev = torch.device(device)
        self.capacity = C = int(buf["capacity"])
        k = qkv_tensor(buf["k"], qkv_dtype, dev)
        v = qkv_tensor(buf["v"], qkv_dtype, dev)
        alpha = torch.from_numpy(np.ascontiguousarray(buf["alpha"], np.float32)).to(dev)
        beta = torch.from_numpy(np.ascontiguousarray(buf["beta"], np.float32)).to(dev)
        if "slots" in buf:  # compact: only the named slots' rows; scatter into the full buffer
            S = int(buf["pool_slots"])
            rows = (torch.from_numpy(buf["slots"]).to(dev)[:, None] * C
                    + torch.arange(C, device=dev)[None, :]).reshape(-1)
            full = []
            for x, fill in ((k, 0.0), (v, 0.0), (alpha, 1.0), (beta, 0.0)):
                f = torch.full((S * C,) + tuple(x.shape[1:]), fill, dtype=x.dtype, device=dev)
                f[rows] = x
                full.append(f)
            k, v, alpha, beta = full
        self.k, self.v, self.alpha, self.beta = k, v, alpha, beta
        self.len_in = torch.from_numpy(np.ascontiguousarray(buf["len_in"], np.int32)).to(dev)
        self.len_out = self.len_in.clone()
        self.c = binding.make_replay(capacity=self.capacity, k=self.k, v=self.v, alpha=self.alpha,
                                     beta=self.beta, len_in=self.len_in, len_out=self.len_out)

    def swap(self) -> None:
        """The lengths written by the last commit become the next step's input."""
        self.len_in, self.len_out = self.len_out, self.len_in
        self.c.swap_lengths()

    def place_drafts(self, d: "DeviceProblem") -> None:
        """Copy the step's draft rows (k, v, alpha, beta of `d`) to buffer rows
        slot * C + len_in[slot] + [0, T_r): what an engine's projection
        kernels would write there."""
        prob = d.host
        lens = torch.from_numpy(prob.lengths.astype(np.int64)).to(self.k.device)
        cu = torch.from_numpy(prob.cu_seqlens[:-1].astype(np.int64)).to(self.k.device)
        slots = d.slot_ids.long()
        req = torch.repeat_interleave(torch.arange(prob.batch, device=self.k.device), lens)
        t = torch.arange(int(lens.sum()), device=self.k.device) - cu[req]
        dst = slots[req] * self.capacity + self.len_in.long()[slots[req]] + t
        src = cu[req] + t
        for buf, x in ((self.k, d.k), (self.v, d.v), (self.alpha, d.alpha), (self.beta, d.beta)):
            buf[dst] = x[src]

    def host(self) -> dict:
        """The buffer as inputs.make_replay lays it out (float32 numpy)."""
        return dict(capacity=self.capacity, k=self.k.float().cpu().numpy(),
                    v=self.v.float().cpu().numpy(), alpha=self.alpha.cpu().numpy(),
                    beta=self.beta.cpu().numpy(), len_in=self.len_in.cpu().numpy())


def replay_launcher(d: DeviceProblem, r: DeviceReplay, mode: str, stream):
    """A zero-argument callable issuing one ReplaySSM call on `stream`, every
    argument marshalled in advance."""
    lib = binding.lib()
    s = binding._stream(stream)
    o, acc = d.o.data_ptr(), d.accepted.data_ptr()
    pref, rref = d.c.ref, r.c.ref
    fn = {"verify": lambda: lib.gdn_replay_verify(pref, rref, o, s),
          "commit": lambda: lib.gdn_replay_commit(pref, rref, acc, s)}[mode]

    def call():
        st = fn()
        if st != binding.GDN_OK:
            raise binding.GdnError(st, f"gdn replay {mode}")
    call.keep = (d, d.c, r, r.c)  # the owners of the raw addresses above
    return call


def commit_verify_launcher(d: DeviceProblem, prevs, ws, stream):
    """A zero-argument callable issuing gdn_commit_verify for `d` on `stream`,
    alternating between two previous-step descriptors (prevs[j] reads ws[j]) and
    writing the other W buffer: call n reads ws[n % 2] and writes ws[1 - n % 2]."""
    lib = binding.lib()
    ref = d.c.ref
    s = binding._stream(stream)
    o = d.o.data_ptr()
    args = [(prevs[j].ref, ws[1 - j].data_ptr()) for j in range(2)]
    state = {"n": 0}

    def call():
        pref, w = args[state["n"] & 1]
        state["n"] += 1
        st = lib.gdn_commit_verify(ref, pref, o, w, s)
        if st != binding.GDN_OK:
            raise binding.GdnError(st, "gdn_commit_verify")
    call.keep = (d, d.c, prevs, ws)  # the owners of the raw addresses above
    return call
