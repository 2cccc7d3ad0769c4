"""Planted mistakes in copies of the commit-then-verify oracle must each fail a pin.

Each mutant is a one-token edit of oracle/lagged.py, loaded as a module of the
oracle package from a temporary file; the real oracle is never modified.
"""
import importlib.util
import os
import sys

import pytest

import oracle
import test_lagged_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "lagged.py")

MUTANTS = {
    "verify_from_the_old_checkpoint": ("s0 = gather_s0(after, prob.slot_ids, prob.heads)",
                                       "s0 = gather_s0(pool, prob.slot_ids, prob.heads)"),
    "commit_the_new_step": ("after = commit(prev, pool, threads=threads)",
                            "after = commit(prob, pool, threads=threads)"),
    "first_step_commits": ("    else:\n        after = np.array(pool, dtype=np.float64, copy=True)",
                           "    else:\n        after = commit(prob, pool, threads=threads)"),
}


def run_pins():
    def chain_short():
        pins.test_chain_equals_one_run_over_the_accepted_rows(pins.SHORT)

    def chain_long():
        pins.test_chain_equals_one_run_over_the_accepted_rows(pins.LONG)

    checks = [chain_short, chain_long,
              pins.test_first_step_commits_nothing, pins.test_nothing_accepted_is_a_plain_verify]
    failed = []
    for check in checks:
        try:
            check()
        except (AssertionError, ValueError, IndexError):
            failed.append(check)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, monkeypatch, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, name
    path = tmp_path / "lagged_mutant.py"
    path.write_text(text.replace(old, new))
    spec = importlib.util.spec_from_file_location("oracle.lagged_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    monkeypatch.setitem(sys.modules, "oracle.lagged_mutant", mod)
    spec.loader.exec_module(mod)
    monkeypatch.setattr(oracle, "commit_verify", mod.commit_verify)
    assert run_pins(), f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_every_pin():
    assert not run_pins()
