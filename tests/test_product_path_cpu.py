"""The product path stands on its own: it never loads the float64 oracle, no
product source refers to it, and without the CUDA library the binding raises
instead of falling back to anything else."""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "speculative_decode_gated_gb300")


def test_importing_the_package_does_not_load_the_oracle():
    code = ("import sys\n"
            "import speculative_decode_gated_gb300 as p\n"
            "from speculative_decode_gated_gb300 import binding, inputs, staging\n"
            "assert 'oracle' not in sys.modules, sorted(m for m in sys.modules if 'oracle' in m)\n"
            "print('ok')\n")
    res = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == "ok"


def _product_sources():
    for base in (PKG, os.path.join(ROOT, "include")):
        for dirpath, _, files in os.walk(base):
            if "__pycache__" in dirpath or os.sep + "_lib" in dirpath:
                continue
            for f in files:
                if f.endswith((".py", ".cu", ".cuh", ".h")):
                    yield os.path.join(dirpath, f)


def test_no_product_source_refers_to_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b|#\s*include\s+[<\"][^>\"]*oracle)"
                     r"|oracle/|gdn_oracle", re.M)
    offenders = []
    for path in _product_sources():
        with open(path, encoding="utf-8") as f:
            if pat.search(f.read()):
                offenders.append(os.path.relpath(path, ROOT))
    assert offenders == []


def test_missing_library_raises(monkeypatch, tmp_path):
    from speculative_decode_gated_gb300 import binding

    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "libgdn.so"))
    monkeypatch.setattr(binding, "_lib_handle", None)
    with pytest.raises(RuntimeError, match="no CPU or PyTorch fallback"):
        binding.lib()
