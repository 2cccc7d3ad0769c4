"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/gdn.h declares, the Python struct matches the C layout, and host-side
validation rejects bad arguments before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

from speculative_decode_gated_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        import speculative_decode_gated_gb300 as pkg
        pkg.build()
    return binding.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", text)))


def test_header_declares_the_bound_symbols():
    assert declared_symbols() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (gdn_\w+)", out))
    for name in declared_symbols():
        assert name in exported, name
        assert hasattr(lib, name)


@pytest.mark.parametrize("cls,cname", [(binding.gdn_problem, "gdn_problem"),
                                       (binding.gdn_replay, "gdn_replay"),
                                       (binding.gdn_prev_step, "gdn_prev_step")])
def test_struct_layout_matches_c(tmp_path, cls, cname):
    fields = [f[0] for f in cls._fields_]
    prog = tmp_path / "layout.c"
    body = "\n".join(f'printf("%zu ", offsetof({cname}, {f}));' for f in fields)
    prog.write_text(f'#include <stdio.h>\n#include <stddef.h>\n#include "gdn.h"\n'
                    f'int main(void) {{ {body} printf("%zu\\n", sizeof({cname})); return 0; }}\n')
    exe = tmp_path / "layout"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(prog),
                    "-o", str(exe)], check=True)
    c_vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                             check=True).stdout.split()]
    py_vals = [getattr(cls, f).offset for f in fields]
    py_vals.append(ctypes.sizeof(cls))
    assert c_vals == py_vals


def fake_problem(**over):
    """A problem with plausible, aligned fake device addresses (never dereferenced)."""
    c = binding.gdn_problem()
    c.batch, c.heads, c.dk, c.dv, c.max_T = 2, 4, 128, 128, 8
    c.qkv_dtype, c.algo, c.flags = binding.GDN_BF16, 0, 0
    base = 1 << 40
    step = 1 << 32
    c.q, c.k, c.v = base, base + step, base + 2 * step
    c.alpha, c.beta = base + 3 * step, base + 4 * step
    c.pool, c.pool_slots = base + 5 * step, 8
    c.slot_ids = base + 6 * step
    c.cu_seqlens = None
    c.dev_err = base + 7 * step
    c.n_tok = 16
    for k, v in over.items():
        setattr(c, k, v)
    return c


O_PTR = (1 << 40) + 9 * (1 << 32)
ACC_PTR = (1 << 40) + 10 * (1 << 32)


def call(lib, fn, c, o=O_PTR, acc=ACC_PTR):
    if fn == "verify":
        return lib.gdn_verify(ctypes.byref(c), o, None)
    if fn == "commit":
        return lib.gdn_commit(ctypes.byref(c), acc, None)
    return lib.gdn_verify_commit_fused(ctypes.byref(c), acc, o, None)


@pytest.mark.parametrize("fn", ["verify", "commit", "fused"])
@pytest.mark.parametrize("over,status", [
    (dict(heads=0), 2), (dict(batch=-1), 2), (dict(max_T=-1), 2), (dict(max_T=1025), 2),
    (dict(flags=4), 2), (dict(flags=-1), 2), (dict(pool_slots=1), 2),
    (dict(cu_seqlens=(1 << 40) + 11 * (1 << 32), n_tok=-1), 2),
    (dict(qkv_dtype=5), 3),
    (dict(dk=48), 4), (dict(dk=512), 4), (dict(dv=48), 4), (dict(dv=160), 4), (dict(algo=9), 4),
    (dict(algo=2, qkv_dtype=0), 4), (dict(algo=2, dk=64, dv=64), 4),
    (dict(algo=3, qkv_dtype=0), 4), (dict(algo=3, dk=64, dv=64), 4), (dict(algo=4), 4),
    (dict(pool=None), 1), (dict(slot_ids=None), 1), (dict(k=None), 1), (dict(beta=None), 1),
    # token rows are 32-bit indices on the device
    (dict(batch=1 << 21, max_T=1024, pool_slots=1 << 22), 2),
    (dict(cu_seqlens=(1 << 40) + 11 * (1 << 32), n_tok=1 << 31), 2),
    (dict(q=(1 << 40) + 8), 7), (dict(pool=(1 << 40) + 5 * (1 << 32) + 4), 7),
    (dict(alpha=(1 << 40) + 3 * (1 << 32) + 2), 7),
    (dict(pool=1 << 40), 8),  # pool over q
])
def test_host_validation_rejects(lib, fn, over, status):
    assert call(lib, fn, fake_problem(**over)) == status


def test_q_is_required_only_with_outputs(lib):
    # verify and fused read q; a commit reads none.  The misaligned pool stops the
    # commit before any launch, after the pointer checks have passed.
    assert call(lib, "verify", fake_problem(q=None)) == 1
    assert call(lib, "fused", fake_problem(q=None)) == 1
    assert call(lib, "commit", fake_problem(q=None, pool=(1 << 40) + 5 * (1 << 32) + 4)) == 7


def test_output_checks(lib):
    c = fake_problem()
    assert lib.gdn_verify(ctypes.byref(c), None, None) == 1
    assert lib.gdn_commit(ctypes.byref(c), None, None) == 1
    assert lib.gdn_verify(ctypes.byref(c), O_PTR + 4, None) == 7
    assert lib.gdn_verify(ctypes.byref(c), c.v, None) == 8       # o over v
    assert lib.gdn_verify(ctypes.byref(c), c.pool, None) == 8    # o over the pool
    assert lib.gdn_verify(None, O_PTR, None) == 1


def test_empty_batch_is_a_no_op(lib):
    c = fake_problem(batch=0, q=None, k=None, v=None, pool=None)
    for fn in ("verify", "commit", "fused"):
        assert call(lib, fn, c) == 0


def test_select_algo(lib):
    assert lib.gdn_select_algo(ctypes.byref(fake_problem())) == binding.GDN_ALGO_CHUNK
    assert lib.gdn_select_algo(ctypes.byref(fake_problem(algo=1))) == 1
    assert lib.gdn_select_algo(ctypes.byref(fake_problem(qkv_dtype=0))) == 1
    assert lib.gdn_select_algo(ctypes.byref(fake_problem(dk=64))) == 1
    assert lib.gdn_select_algo(ctypes.byref(fake_problem(max_T=17))) == binding.GDN_ALGO_CHUNK
    assert lib.gdn_select_algo(ctypes.byref(fake_problem(max_T=1024))) == binding.GDN_ALGO_CHUNK
    assert lib.gdn_select_algo(ctypes.byref(fake_problem(dk=48))) == -1
    assert lib.gdn_select_algo(ctypes.byref(fake_problem(max_T=4096))) == -1


def test_status_strings(lib):
    for s in range(10):
        assert binding.gdn_status_string(s)
    assert binding.gdn_version().count(".") == 2
    assert binding.gdn_last_error_string() == ""


# ---------------------------------------------------------------- layer batches

def fake_layers(n, **over_last):
    """n problems that share the request-level fields and each own their arrays
    (disjoint fake addresses); overrides apply to the last one."""
    arr = (binding.gdn_problem * n)()
    for l in range(n):
        c = fake_problem()
        off = (l + 1) << 36
        c.q, c.k, c.v, c.alpha, c.beta, c.pool = (x + off for x in (c.q, c.k, c.v, c.alpha,
                                                                      c.beta, c.pool))
        arr[l] = c
    for k, v in over_last.items():
        setattr(arr[n - 1], k, v)
    return arr


def o_array(n, **set_at):
    arr = (ctypes.c_void_p * n)(*[O_PTR + ((l + 1) << 36) for l in range(n)])
    for i, v in set_at.items():
        arr[int(i[1:])] = v
    return arr


def call_layers(lib, fn, arr, n, o=None, acc=ACC_PTR):
    o = o_array(max(n, 1)) if o is None else o
    P = ctypes.cast(arr, ctypes.POINTER(binding.gdn_problem)) if arr is not None else None
    if fn == "verify":
        return lib.gdn_verify_layers(P, n, o, None)
    if fn == "commit":
        return lib.gdn_commit_layers(P, n, acc, None)
    return lib.gdn_verify_commit_fused_layers(P, n, acc, o, None)


@pytest.mark.parametrize("fn", ["verify", "commit", "fused"])
def test_layers_empty_and_null(lib, fn):
    assert call_layers(lib, fn, fake_layers(2), 0) == 0
    assert call_layers(lib, fn, fake_layers(2), -1) == 2
    assert call_layers(lib, fn, None, 2) == 1
    P = ctypes.cast(fake_layers(2), ctypes.POINTER(binding.gdn_problem))
    if fn == "verify":
        assert lib.gdn_verify_layers(P, 2, None, None) == 1           # no o array
    elif fn == "commit":
        assert lib.gdn_commit_layers(P, 2, None, None) == 1           # no accepted
    else:
        assert lib.gdn_verify_commit_fused_layers(P, 2, ACC_PTR, None, None) == 1


@pytest.mark.parametrize("fn", ["verify", "commit", "fused"])
@pytest.mark.parametrize("over,status", [
    (dict(heads=0), 2),                                  # a single-problem check on layer 2
    (dict(q=(1 << 40) + 8), 7),
    (dict(batch=1), 9), (dict(max_T=4), 9), (dict(pool_slots=16), 9),
    (dict(slot_ids=(1 << 40) + 6 * (1 << 32) + 64), 9), (dict(algo=1), 9),
    (dict(cu_seqlens=(1 << 40) + 11 * (1 << 32)), 9),
])
def test_layers_reject(lib, fn, over, status):
    assert call_layers(lib, fn, fake_layers(3, **over), 3) == status


def test_layers_cross_layer_aliasing(lib):
    # a layer's output over another layer's input or output
    arr = fake_layers(2)
    assert call_layers(lib, "verify", arr, 2, o=o_array(2, o1=arr[0].q)) == 8
    assert call_layers(lib, "fused", arr, 2, o=o_array(2, o1=arr[0].pool)) == 8
    assert call_layers(lib, "verify", arr, 2, o=o_array(2, o1=O_PTR + (1 << 36))) == 8
    # a committed pool over another layer's pool or tokens
    assert call_layers(lib, "commit", fake_layers(2, pool=fake_layers(1)[0].pool), 2) == 8
    assert call_layers(lib, "fused", fake_layers(2, pool=fake_layers(1)[0].k), 2) == 8


# ---------------------------------------------------------------- accept length

def call_accept(lib, batch=4, max_T=8, cu=None, n_tok=32, draft=(1 << 40), target=(1 << 40) + (1 << 32),
                acc=ACC_PTR, err=None):
    return lib.gdn_accept_prefix(batch, max_T, cu, n_tok, draft, target, acc, err, None)


def test_accept_prefix_validation(lib):
    assert call_accept(lib, batch=0, acc=None, draft=None, target=None) == 0  # nothing to do
    assert call_accept(lib, batch=-1) == 2
    assert call_accept(lib, max_T=1025) == 2
    assert call_accept(lib, max_T=-1) == 2
    assert call_accept(lib, cu=(1 << 40) + 11 * (1 << 32), n_tok=-1) == 2
    assert call_accept(lib, acc=None) == 1
    assert call_accept(lib, draft=None) == 1
    assert call_accept(lib, target=None) == 1
    assert call_accept(lib, acc=ACC_PTR + 2) == 7
    assert call_accept(lib, draft=(1 << 40) + 1) == 7
    assert call_accept(lib, acc=(1 << 40) + 16) == 8           # accepted over the draft ids
    assert call_accept(lib, err=ACC_PTR + 4) == 8              # accepted over the error word


def test_selftest_wait_timeout_validation(lib):
    # Both checks return before any CUDA call (no GPU here).
    assert lib.gdn_selftest_wait_timeout(None, None) == 1
    assert lib.gdn_selftest_wait_timeout((1 << 40) + 2, None) == 7



# ---------------------------------------------------------------- replay buffer

def fake_replay(**over):
    rb = binding.gdn_replay()
    base = (1 << 40) + 20 * (1 << 32)
    step = 1 << 32
    rb.capacity, rb.reserved = 32, 0
    rb.k, rb.v, rb.alpha, rb.beta = base, base + step, base + 2 * step, base + 3 * step
    rb.len_in, rb.len_out = base + 4 * step, base + 5 * step
    for k, v in over.items():
        setattr(rb, k, v)
    return rb


def call_replay(lib, fn, c=None, rb=None):
    c = fake_problem() if c is None else c
    rbp = None if rb is False else ctypes.byref(fake_replay() if rb is None else rb)
    if fn == "verify":
        return lib.gdn_replay_verify(ctypes.byref(c), rbp, O_PTR, None)
    return lib.gdn_replay_commit(ctypes.byref(c), rbp, ACC_PTR, None)


@pytest.mark.parametrize("fn", ["verify", "commit"])
def test_replay_validation(lib, fn):
    assert call_replay(lib, fn, rb=False) == 1
    assert call_replay(lib, fn, rb=fake_replay(reserved=1)) == 2
    assert call_replay(lib, fn, rb=fake_replay(capacity=0)) == 2
    assert call_replay(lib, fn, rb=fake_replay(capacity=7)) == 2       # below max_T = 8
    assert call_replay(lib, fn, rb=fake_replay(len_in=None)) == 1
    assert call_replay(lib, fn, rb=fake_replay(k=None)) == 1
    assert call_replay(lib, fn, rb=fake_replay(k=fake_replay().k + 8)) == 7
    assert call_replay(lib, fn, rb=fake_replay(len_in=fake_replay().len_in + 2)) == 7
    assert call_replay(lib, fn, c=fake_problem(dk=64, dv=64)) == 4      # chunked kernel only
    assert call_replay(lib, fn, c=fake_problem(algo=1)) == 4
    assert call_replay(lib, fn, c=fake_problem(qkv_dtype=0)) == 4
    assert call_replay(lib, fn, rb=fake_replay(k=fake_problem().pool)) == 8   # buffer over pool
    assert call_replay(lib, fn, c=fake_problem(batch=0, q=None, pool=None)) == 0


def test_replay_commit_output_checks(lib):
    assert call_replay(lib, "commit", rb=fake_replay(len_out=None)) == 1
    assert call_replay(lib, "commit", rb=fake_replay(len_out=fake_replay().len_in)) == 8
    assert call_replay(lib, "commit", rb=fake_replay(len_out=fake_problem().slot_ids)) == 8


# ---------------------------------------------------------------- commit then verify

W_PTR = (1 << 40) + 11 * (1 << 32)


def fake_prev(**over):
    pv = binding.gdn_prev_step()
    base = (1 << 40) + 30 * (1 << 32)
    step = 1 << 32
    pv.cu_seqlens, pv.max_T, pv.reserved, pv.n_tok = None, 8, 0, 16
    pv.k, pv.alpha, pv.w, pv.accepted = base, base + step, base + 2 * step, base + 3 * step
    for k, v in over.items():
        setattr(pv, k, v)
    return pv


def call_cv(lib, c=None, prev=None, o=O_PTR, w=W_PTR):
    c = fake_problem() if c is None else c
    pvp = None if prev is False else ctypes.byref(fake_prev() if prev is None else prev)
    return lib.gdn_commit_verify(ctypes.byref(c), pvp, o, w, None)


def test_commit_verify_validation(lib):
    assert call_cv(lib, w=None) == 1
    assert call_cv(lib, o=None) == 1
    assert call_cv(lib, w=W_PTR + 8) == 7
    assert call_cv(lib, c=fake_problem(max_T=17)) == 4          # single 16-token chunks
    assert call_cv(lib, prev=fake_prev(max_T=17)) == 4
    assert call_cv(lib, prev=fake_prev(reserved=1)) == 2
    assert call_cv(lib, prev=fake_prev(max_T=-1)) == 2
    assert call_cv(lib, c=fake_problem(dk=64, dv=64)) == 4      # chunked kernel only
    assert call_cv(lib, c=fake_problem(algo=1)) == 4
    assert call_cv(lib, c=fake_problem(algo=3)) == 4
    assert call_cv(lib, c=fake_problem(qkv_dtype=0)) == 4
    assert call_cv(lib, prev=fake_prev(w=None)) == 1
    assert call_cv(lib, prev=fake_prev(accepted=None)) == 1
    assert call_cv(lib, prev=fake_prev(k=fake_prev().k + 8)) == 7
    assert call_cv(lib, prev=fake_prev(w=fake_prev().w + 4)) == 7
    assert call_cv(lib, w=O_PTR) == 8                           # w over o
    assert call_cv(lib, w=fake_prev().w) == 8                   # w over the previous w
    assert call_cv(lib, w=fake_problem().q) == 8                # w over an input
    assert call_cv(lib, prev=fake_prev(w=fake_problem().pool)) == 8   # previous arrays over the pool
    assert call_cv(lib, prev=fake_prev(k=O_PTR)) == 8           # ... or over o
    assert call_cv(lib, c=fake_problem(batch=0, q=None, pool=None)) == 0
