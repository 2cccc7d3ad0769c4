"""Python binding of libgdn.so: argument marshalling only.

Every function here has the name of the C entry point it calls (include/gdn.h)
and only turns torch tensors into device pointers and sizes; all computation
runs in the CUDA kernels.  If the library has not been built this module raises
on first use: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libgdn.so")

GDN_OK = 0
GDN_ERR_DEVICE_ARG = 5
GDN_ERR_ALIAS, GDN_ERR_LAYER_MISMATCH = 8, 9
GDN_FP32, GDN_BF16 = 0, 1
GDN_FLAG_O_BF16, GDN_FLAG_LOG_GATE = 1, 2
GDN_ALGO_AUTO, GDN_ALGO_RECURRENT, GDN_ALGO_CHUNK, GDN_ALGO_CHUNK_TC = 0, 1, 2, 3
GDN_DEVERR_SLOT, GDN_DEVERR_ACCEPTED, GDN_DEVERR_SEQLEN = 1, 2, 4
GDN_DEVERR_TIMEOUT, GDN_DEVERR_REPLAY = 8, 16
GDN_MAX_T = 1024

# Every symbol include/gdn.h declares.
EXPORTED = (
    "gdn_verify", "gdn_commit", "gdn_verify_commit_fused",
    "gdn_verify_layers", "gdn_commit_layers", "gdn_verify_commit_fused_layers",
    "gdn_accept_prefix", "gdn_replay_verify", "gdn_replay_commit", "gdn_commit_verify",
    "gdn_read_device_error", "gdn_selftest_wait_timeout",
    "gdn_select_algo", "gdn_status_string", "gdn_last_error_string", "gdn_version",
)


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {gdn_status_string(status)} (status {status})"
        if status == 6:
            msg += f": {gdn_last_error_string()}"
        super().__init__(msg)


class gdn_problem(ctypes.Structure):
    """Mirror of the C struct gdn_problem (include/gdn.h), field for field."""

    _fields_ = [
        ("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("dk", ctypes.c_int32),
        ("dv", ctypes.c_int32), ("max_T", ctypes.c_int32), ("qkv_dtype", ctypes.c_int32),
        ("algo", ctypes.c_int32), ("flags", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p), ("q", ctypes.c_void_p), ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p), ("alpha", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("pool", ctypes.c_void_p), ("pool_slots", ctypes.c_int64),
        ("slot_ids", ctypes.c_void_p), ("dev_err", ctypes.c_void_p), ("n_tok", ctypes.c_int64),
    ]


class gdn_replay(ctypes.Structure):
    """Mirror of the C struct gdn_replay (include/gdn.h), field for field."""

    _fields_ = [
        ("capacity", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("alpha", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("len_in", ctypes.c_void_p), ("len_out", ctypes.c_void_p),
    ]


class gdn_prev_step(ctypes.Structure):
    """Mirror of the C struct gdn_prev_step (include/gdn.h), field for field."""

    _fields_ = [
        ("cu_seqlens", ctypes.c_void_p), ("max_T", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("n_tok", ctypes.c_int64), ("k", ctypes.c_void_p), ("alpha", ctypes.c_void_p),
        ("w", ctypes.c_void_p), ("accepted", ctypes.c_void_p),
    ]


_lib_handle: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it was never built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with speculative_decode_gated_gb300.build() "
                "(there is no CPU or PyTorch fallback)")
        h = ctypes.CDLL(LIB_PATH)
        P, S = ctypes.POINTER(gdn_problem), ctypes.c_void_p
        h.gdn_verify.argtypes = [P, S, S]
        h.gdn_commit.argtypes = [P, S, S]
        h.gdn_verify_commit_fused.argtypes = [P, S, S, S]
        I32 = ctypes.c_int32
        h.gdn_verify_layers.argtypes = [P, I32, S, S]
        h.gdn_commit_layers.argtypes = [P, I32, S, S]
        h.gdn_verify_commit_fused_layers.argtypes = [P, I32, S, S, S]
        h.gdn_accept_prefix.argtypes = [I32, I32, S, ctypes.c_int64, S, S, S, S, S]
        R = ctypes.POINTER(gdn_replay)
        h.gdn_replay_verify.argtypes = [P, R, S, S]
        h.gdn_replay_commit.argtypes = [P, R, S, S]
        h.gdn_commit_verify.argtypes = [P, ctypes.POINTER(gdn_prev_step), S, S, S]
        h.gdn_read_device_error.argtypes = [P, S, ctypes.POINTER(ctypes.c_int32)]
        h.gdn_selftest_wait_timeout.argtypes = [S, S]
        h.gdn_select_algo.argtypes = [P]
        h.gdn_status_string.argtypes = [ctypes.c_int]
        for name in ("gdn_verify", "gdn_commit", "gdn_verify_commit_fused",
                     "gdn_verify_layers", "gdn_commit_layers", "gdn_verify_commit_fused_layers",
                     "gdn_accept_prefix", "gdn_replay_verify", "gdn_replay_commit",
                     "gdn_commit_verify", "gdn_read_device_error", "gdn_selftest_wait_timeout",
                     "gdn_select_algo"):
            getattr(h, name).restype = ctypes.c_int
        for name in ("gdn_status_string", "gdn_last_error_string", "gdn_version"):
            getattr(h, name).restype = ctypes.c_char_p
        _lib_handle = h
    return _lib_handle


class Problem:
    """A gdn_problem plus references to the tensors it points into."""

    def __init__(self, c: gdn_problem, refs: tuple):
        self.c = c
        self.refs = refs

    @property
    def ref(self):
        return ctypes.byref(self.c)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t: Optional[torch.Tensor], name: str, dtypes, device) -> None:
    if t is None:
        return
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def make_problem(*, q: Optional[torch.Tensor], k: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor,
                 beta: torch.Tensor, pool: torch.Tensor, slot_ids: torch.Tensor,
                 max_T: int, cu_seqlens: Optional[torch.Tensor] = None,
                 dev_err: Optional[torch.Tensor] = None, algo: int = GDN_ALGO_AUTO,
                 flags: int = 0) -> Problem:
    """Builds the C problem from device tensors (shapes as in include/gdn.h).

    q, k: [N_tok, H, dk]; v: [N_tok, H, dv] (bf16 or fp32, same dtype);
    alpha, beta: [N_tok, H] fp32; pool: [slots, H, dk, dv] fp32; slot_ids: [B] int32;
    cu_seqlens: [B+1] int32 or None (uniform length max_T); dev_err: [1] int32 or None.
    flags: GDN_FLAG_* bits (bf16 o, log-space alpha).  q may be None for a problem
    that only commits (the commit calls read no q).
    """
    dev = pool.device
    if k.dtype not in (torch.bfloat16, torch.float32) or v.dtype != k.dtype or \
            (q is not None and q.dtype != k.dtype):
        raise TypeError("q, k, v must all be bf16 or all fp32")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, (k.dtype,), dev)
    _check(alpha, "alpha", (torch.float32,), dev)
    _check(beta, "beta", (torch.float32,), dev)
    _check(pool, "pool", (torch.float32,), dev)
    _check(slot_ids, "slot_ids", (torch.int32,), dev)
    _check(cu_seqlens, "cu_seqlens", (torch.int32,), dev)
    _check(dev_err, "dev_err", (torch.int32,), dev)
    if pool.dim() != 4:
        raise ValueError("pool must be [slots, heads, dk, dv]")
    slots, H, dk, dv = pool.shape
    c = gdn_problem()
    c.batch = slot_ids.numel()
    c.heads, c.dk, c.dv = H, dk, dv
    c.max_T = int(max_T)
    c.qkv_dtype = GDN_BF16 if k.dtype == torch.bfloat16 else GDN_FP32
    c.algo = int(algo)
    c.flags = int(flags)
    c.cu_seqlens = _ptr(cu_seqlens)
    c.q, c.k, c.v = _ptr(q), _ptr(k), _ptr(v)
    c.alpha, c.beta = _ptr(alpha), _ptr(beta)
    c.pool = _ptr(pool)
    c.pool_slots = slots
    c.slot_ids = _ptr(slot_ids)
    c.dev_err = _ptr(dev_err)
    c.n_tok = k.shape[0]
    return Problem(c, (q, k, v, alpha, beta, pool, slot_ids, cu_seqlens, dev_err))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _raise(status: int, where: str) -> None:
    if status != GDN_OK:
        raise GdnError(status, where)


def _o_dtype(prob: Problem):
    return torch.bfloat16 if prob.c.flags & GDN_FLAG_O_BF16 else torch.float32


def gdn_verify(prob: Problem, o: torch.Tensor, stream=None) -> None:
    _check(o, "o", (_o_dtype(prob),), None)
    _raise(lib().gdn_verify(prob.ref, _ptr(o), _stream(stream)), "gdn_verify")


def gdn_commit(prob: Problem, accepted: torch.Tensor, stream=None) -> None:
    _check(accepted, "accepted", (torch.int32,), None)
    _raise(lib().gdn_commit(prob.ref, _ptr(accepted), _stream(stream)), "gdn_commit")


def gdn_verify_commit_fused(prob: Problem, accepted: torch.Tensor, o: torch.Tensor,
                            stream=None) -> None:
    _check(accepted, "accepted", (torch.int32,), None)
    _check(o, "o", (_o_dtype(prob),), None)
    _raise(lib().gdn_verify_commit_fused(prob.ref, _ptr(accepted), _ptr(o), _stream(stream)),
           "gdn_verify_commit_fused")


class ProblemArray:
    """A host array of gdn_problem (one per layer) for the layer-batch calls."""

    def __init__(self, problems):
        self.problems = list(problems)
        n = len(self.problems)
        self.c = (gdn_problem * max(n, 1))()
        for i, p in enumerate(self.problems):
            self.c[i] = p.c
        self.n = n

    @property
    def ref(self):
        return ctypes.cast(self.c, ctypes.POINTER(gdn_problem))


def _ptr_array(tensors) -> ctypes.Array:
    arr = (ctypes.c_void_p * max(len(tensors), 1))()
    for i, t in enumerate(tensors):
        _check(t, f"o[{i}]", (torch.float32, torch.bfloat16), None)
        arr[i] = _ptr(t)
    return arr


def gdn_verify_layers(probs: ProblemArray, o, stream=None) -> None:
    """o: one fp32 output tensor per layer."""
    arr = _ptr_array(o)
    _raise(lib().gdn_verify_layers(probs.ref, probs.n, arr, _stream(stream)), "gdn_verify_layers")


def gdn_commit_layers(probs: ProblemArray, accepted: torch.Tensor, stream=None) -> None:
    _check(accepted, "accepted", (torch.int32,), None)
    _raise(lib().gdn_commit_layers(probs.ref, probs.n, _ptr(accepted), _stream(stream)),
           "gdn_commit_layers")


def gdn_verify_commit_fused_layers(probs: ProblemArray, accepted: torch.Tensor, o,
                                   stream=None) -> None:
    _check(accepted, "accepted", (torch.int32,), None)
    arr = _ptr_array(o)
    _raise(lib().gdn_verify_commit_fused_layers(probs.ref, probs.n, _ptr(accepted), arr,
                                                _stream(stream)),
           "gdn_verify_commit_fused_layers")


def gdn_accept_prefix(draft_ids: torch.Tensor, target_ids: torch.Tensor, accepted: torch.Tensor,
                      max_T: int, cu_seqlens: Optional[torch.Tensor] = None,
                      dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """accepted[r] <- greedy accepted length of request r (int32 tensors on one device;
    draft_ids/target_ids [N_tok], accepted [B], cu_seqlens [B+1] or None)."""
    dev = accepted.device
    for t, n in ((draft_ids, "draft_ids"), (target_ids, "target_ids"), (accepted, "accepted"),
                 (cu_seqlens, "cu_seqlens"), (dev_err, "dev_err")):
        _check(t, n, (torch.int32,), dev)
    batch = accepted.numel()
    st = lib().gdn_accept_prefix(batch, int(max_T), _ptr(cu_seqlens), draft_ids.numel(),
                                 _ptr(draft_ids), _ptr(target_ids), _ptr(accepted), _ptr(dev_err),
                                 _stream(stream))
    _raise(st, "gdn_accept_prefix")


def gdn_selftest_wait_timeout(dev_err: torch.Tensor, stream=None) -> None:
    """Runs the kernels' bounded wait on a barrier nothing completes: about two
    seconds later GDN_DEVERR_TIMEOUT is ORed into dev_err (int32, one element)."""
    _check(dev_err, "dev_err", (torch.int32,), dev_err.device)
    st = lib().gdn_selftest_wait_timeout(_ptr(dev_err), _stream(stream))
    _raise(st, "gdn_selftest_wait_timeout")


class Replay:
    """A gdn_replay plus references to the tensors it points into."""

    def __init__(self, c: gdn_replay, refs: tuple):
        self.c = c
        self.refs = refs

    @property
    def ref(self):
        return ctypes.byref(self.c)

    def swap_lengths(self) -> None:
        """len_in <-> len_out, for the next step."""
        self.c.len_in, self.c.len_out = self.c.len_out, self.c.len_in
        self.refs = self.refs[:4] + (self.refs[5], self.refs[4])


def make_replay(*, capacity: int, k: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor,
                beta: torch.Tensor, len_in: torch.Tensor, len_out: torch.Tensor) -> Replay:
    """k: [slots*capacity, H, dk], v: [slots*capacity, H, dv] (the q/k/v dtype);
    alpha, beta: [slots*capacity, H] fp32; len_in, len_out: [slots] int32."""
    dev = len_in.device
    _check(k, "k", (torch.bfloat16, torch.float32), dev)
    _check(v, "v", (k.dtype,), dev)
    for t, n in ((alpha, "alpha"), (beta, "beta")):
        _check(t, n, (torch.float32,), dev)
    for t, n in ((len_in, "len_in"), (len_out, "len_out")):
        _check(t, n, (torch.int32,), dev)
    c = gdn_replay()
    c.capacity, c.reserved = int(capacity), 0
    c.k, c.v, c.alpha, c.beta = _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta)
    c.len_in, c.len_out = _ptr(len_in), _ptr(len_out)
    return Replay(c, (k, v, alpha, beta, len_in, len_out))


def gdn_replay_verify(prob: Problem, rb: Replay, o: torch.Tensor, stream=None) -> None:
    _check(o, "o", (_o_dtype(prob),), None)
    _raise(lib().gdn_replay_verify(prob.ref, rb.ref, _ptr(o), _stream(stream)), "gdn_replay_verify")


def gdn_replay_commit(prob: Problem, rb: Replay, accepted: torch.Tensor, stream=None) -> None:
    _check(accepted, "accepted", (torch.int32,), None)
    _raise(lib().gdn_replay_commit(prob.ref, rb.ref, _ptr(accepted), _stream(stream)),
           "gdn_replay_commit")


def gdn_read_device_error(prob: Problem, stream=None) -> int:
    """Synchronises the stream and returns the device error word (0 = none)."""
    code = ctypes.c_int32(0)
    st = lib().gdn_read_device_error(prob.ref, _stream(stream), ctypes.byref(code))
    if st not in (GDN_OK, GDN_ERR_DEVICE_ARG):
        _raise(st, "gdn_read_device_error")
    return int(code.value)


def gdn_select_algo(prob: Problem) -> int:
    return int(lib().gdn_select_algo(prob.ref))


def gdn_status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def gdn_last_error_string() -> str:
    return lib().gdn_last_error_string().decode()


def gdn_version() -> str:
    return lib().gdn_version().decode()


class PrevStep:
    """A gdn_prev_step plus references to the tensors it points into."""

    def __init__(self, c: gdn_prev_step, refs: tuple):
        self.c = c
        self.refs = refs

    @property
    def ref(self):
        return ctypes.byref(self.c)


def make_prev_step(*, k: torch.Tensor, alpha: torch.Tensor, w: torch.Tensor,
                   accepted: torch.Tensor, max_T: int,
                   cu_seqlens: Optional[torch.Tensor] = None) -> PrevStep:
    """The previous step of the same requests: its k [N_tok, H, dk], alpha [N_tok, H],
    the w its gdn_commit_verify wrote [N_tok, H, dv] fp32, its accepted [B] int32,
    and its row offsets [B+1] int32 or None (uniform length max_T)."""
    dev = k.device
    _check(k, "k", (torch.bfloat16, torch.float32), dev)
    _check(alpha, "alpha", (torch.float32,), dev)
    _check(w, "w", (torch.float32,), dev)
    _check(accepted, "accepted", (torch.int32,), dev)
    _check(cu_seqlens, "cu_seqlens", (torch.int32,), dev)
    c = gdn_prev_step()
    c.cu_seqlens = _ptr(cu_seqlens)
    c.max_T, c.reserved = int(max_T), 0
    c.n_tok = k.shape[0]
    c.k, c.alpha, c.w, c.accepted = _ptr(k), _ptr(alpha), _ptr(w), _ptr(accepted)
    return PrevStep(c, (k, alpha, w, accepted, cu_seqlens))


def gdn_commit_verify(prob: Problem, prev: Optional[PrevStep], o: torch.Tensor, w: torch.Tensor,
                      stream=None) -> None:
    """Commit `prev` (None: nothing), then verify `prob`; w: this step's W [N_tok, H, dv] fp32."""
    _check(o, "o", (_o_dtype(prob),), None)
    _check(w, "w", (torch.float32,), None)
    _raise(lib().gdn_commit_verify(prob.ref, None if prev is None else prev.ref, _ptr(o), _ptr(w),
                                   _stream(stream)), "gdn_commit_verify")
