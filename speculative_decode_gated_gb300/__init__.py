"""Gated DeltaNet speculative verify/commit on GB300 (sm_103a).

`binding` holds the Python side of the C ABI (include/gdn.h); `staging`
moves host problems (from `inputs`) into device tensors; `_build` compiles the
CUDA library in-tree.  Submodules load lazily so that `inputs` can be used on a
machine without a GPU or a built library.
"""
import importlib

__all__ = ["binding", "inputs", "staging", "build"]


def build(verbose: bool = False) -> str:
    from . import _build
    return _build.build(verbose=verbose)


def __getattr__(name):
    if name in ("binding", "inputs", "staging"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
