"""Float64 CPU oracle of the Gated DeltaNet speculative verify/commit path.

TEST INFRASTRUCTURE.  Only `tests/`, `__graft_entry__.smoke()` and the CPU
baseline leg of `bench.py` may import this package.  The product path (the CUDA
library and its Python binding) never imports, links or calls it, and this
package imports nothing from the product path.

The arithmetic lives in `gdn_oracle.c` (plain loops in float64, the update
written as the definition).  This module compiles it with gcc, marshals numpy
arrays into it and applies the slot bookkeeping of the commit step in plain
numpy: a request with accepted length a_r > 0 overwrites its slot with the
state after a_r tokens; a request with a_r = 0 leaves its slot untouched
(ReplaySSM keeps the accepted prefix and rolls the rest back, OCRia write-up,
section "Make speculative verification cheaper").

The greedy accept-length rule lives in `accept.py` (pure Python loops); the
ReplaySSM buffer (checkpoint plus buffered rows, periodic flush) in `replay.py`,
which runs this recurrence over the replayed rows; the step that commits the
previous step's accepted prefix and then verifies the next drafts in
`lagged.py`.

Parity unpinned: none.  Every function here is pinned by `tests/test_oracle_pins.py`,
`tests/test_accept_oracle.py`, `tests/test_replay_oracle.py` and
`tests/test_lagged_oracle.py`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np

from .accept import accept_prefix  # noqa: F401  (greedy accept length)
from .replay import replay_commit, replay_verify  # noqa: F401  (ReplaySSM buffer)
from .lagged import commit_verify  # noqa: F401  (commit the previous step, verify the next)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIB_DIR, "libgdn_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_loaded = {}


def build(src: str = _SRC, out: str = _LIB, cc: str = "gcc") -> str:
    """Compile the oracle into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run([cc, *CFLAGS, "-I", os.path.dirname(src), src, "-o", tmp], check=True)
    os.replace(tmp, out)
    return out


def _stale(path: str) -> bool:
    return (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(_SRC)


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building first if missing or older than the source) the oracle library."""
    with _lock:
        if path is None:
            path = _LIB
            if _stale(path):
                build()
        if path not in _loaded:
            lib = ctypes.CDLL(path)
            f = lib.gdn_oracle_run_units
            P = ctypes.c_void_p
            f.argtypes = [ctypes.c_int64] * 4 + [P] * 6 + [ctypes.c_int64] + [P] * 5
            f.restype = ctypes.c_int
            _loaded[path] = lib
        return _loaded[path]


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def run_units(prob, unit_ids: Optional[Sequence[int]] = None, *, s0: Optional[np.ndarray] = None,
              accepted: Optional[np.ndarray] = None, want_o: bool = True,
              want_state: bool = True, threads: int = 1, lib: Optional[ctypes.CDLL] = None):
    """Run the recurrence for the listed units (default: all) of an inputs.Problem.

    Returns (o, s_acc): o is float64 [n][max_T][dv] (rows t >= T_r are zero) or
    None; s_acc is float64 [n][dk][dv], the state after accepted[r] tokens, or None.
    `s0` overrides the checkpoint tiles ([n][dk][dv]); by default they are the
    problem's own.  `accepted` overrides the problem's accepted lengths.
    """
    lib = lib or load()
    H, dk, dv, T = prob.heads, prob.dk, prob.dv, max(int(prob.max_T), 1)
    if unit_ids is None:
        unit_ids = np.arange(prob.batch * H)
    units = np.ascontiguousarray(unit_ids, dtype=np.int64)
    n = len(units)
    if s0 is None:
        s0 = prob.s0.reshape(prob.batch * H, dk, dv)[units]
    s0 = _f64(s0).reshape(n, dk, dv)
    acc = np.ascontiguousarray(prob.accepted if accepted is None else accepted, dtype=np.int64)
    cu = np.ascontiguousarray(prob.cu_seqlens, dtype=np.int64)
    q, k, v = _f64(prob.q), _f64(prob.k), _f64(prob.v)
    al, be = _f64(prob.alpha), _f64(prob.beta)
    if getattr(prob, "gate", "alpha") == "log":
        # The log-space gate variant: the input is g and the decay is alpha = exp(g).
        al = np.exp(al)
    o = np.zeros((n, T, dv)) if want_o else None
    s_acc = np.zeros((n, dk, dv)) if want_state else None

    def work(lo: int, hi: int) -> int:
        return lib.gdn_oracle_run_units(
            H, dk, dv, T, _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(al), _ptr(be),
            hi - lo, _ptr(units[lo:hi]), _ptr(s0[lo:hi]),
            _ptr(acc) if want_state else None,
            None if o is None else o[lo:hi].ctypes.data_as(ctypes.c_void_p),
            None if s_acc is None else s_acc[lo:hi].ctypes.data_as(ctypes.c_void_p))

    if threads <= 1 or n <= 1:
        rcs = [work(0, n)]
    else:
        bounds = np.linspace(0, n, min(threads, n) + 1).astype(int)
        with ThreadPoolExecutor(max_workers=len(bounds) - 1) as ex:
            rcs = list(ex.map(lambda i: work(bounds[i], bounds[i + 1]), range(len(bounds) - 1)))
    if any(rc != 0 for rc in rcs):
        raise ValueError(f"oracle rejected the inputs (status {max(rcs)})")
    return o, s_acc


def verify(prob, threads: int = 1, lib=None) -> np.ndarray:
    """Outputs of every draft token: float64 [N_tok][H][dv].  S_0 is not changed."""
    o, _ = run_units(prob, want_o=True, want_state=False, threads=threads, lib=lib)
    return scatter_outputs(prob, np.arange(prob.batch * prob.heads), o)


def scatter_outputs(prob, unit_ids, o_units: np.ndarray) -> np.ndarray:
    """Place per-unit outputs [n][max_T][dv] at their token rows: [N_tok][H][dv]."""
    out = np.zeros((prob.n_tok, prob.heads, prob.dv))
    lens = prob.lengths
    for n, u in enumerate(np.asarray(unit_ids)):
        r, h = divmod(int(u), prob.heads)
        c0 = int(prob.cu_seqlens[r])
        out[c0:c0 + lens[r], h, :] = o_units[n, :lens[r], :]
    return out


def commit_pool(pool: np.ndarray, slot_ids, accepted, s_acc_units: np.ndarray,
                heads: int, unit_ids=None) -> np.ndarray:
    """Slot bookkeeping of the commit step on a copy of `pool` ([slots][H][dk][dv]).

    Unit n = (r, h) writes s_acc_units[n] into pool[slot_ids[r]][h] when
    accepted[r] > 0; when accepted[r] == 0 the slot is left as it was.
    """
    out = np.array(pool, copy=True)
    if unit_ids is None:
        unit_ids = np.arange(len(slot_ids) * heads)
    for n, u in enumerate(np.asarray(unit_ids)):
        r, h = divmod(int(u), heads)
        if int(accepted[r]) > 0:
            out[int(slot_ids[r]), h] = s_acc_units[n]
    return out


def gather_s0(pool: np.ndarray, slot_ids, heads: int, unit_ids=None) -> np.ndarray:
    """Checkpoint tiles of the listed units read from their slots: [n][dk][dv]."""
    if unit_ids is None:
        unit_ids = np.arange(len(slot_ids) * heads)
    return np.stack([pool[int(slot_ids[int(u) // heads]), int(u) % heads]
                     for u in np.asarray(unit_ids)])


def commit(prob, pool: np.ndarray, threads: int = 1, lib=None) -> np.ndarray:
    """The pool after the commit step of every request of `prob`; S_0 is read
    from the slots of `pool` (slot gather), the result written back (scatter)."""
    s0 = gather_s0(pool, prob.slot_ids, prob.heads)
    _, s_acc = run_units(prob, s0=s0, want_o=False, want_state=True, threads=threads, lib=lib)
    return commit_pool(pool, prob.slot_ids, prob.accepted, s_acc, prob.heads)
