"""Planted mistakes in copies of the accept-length oracle must each fail a pin.

Each mutant is a one-token edit of oracle/accept.py, loaded from a temporary
file; the real oracle is never modified.
"""
import importlib.util
import os

import pytest

import oracle
import test_accept_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "accept.py")

MUTANTS = {
    "count_every_match": ("                break\n", "                continue\n"),
    "start_at_one": ("        a = 0\n", "        a = 1\n"),
    "shifted_target": ("target[cu[r] + t]", "target[cu[r] + t - 1]"),
    "stop_on_match": ("!= target[cu[r] + t]", "== target[cu[r] + t]"),
}


def run_pins():
    failed = []
    checks = [pins.test_hand_fixture, pins.test_all_equal_and_all_different,
              pins.test_empty_batch] + [lambda s=s: pins.test_prefix_property_and_first_mismatch(s)
                                        for s in range(5)]
    for check in checks:
        try:
            check()
        except (AssertionError, IndexError, ValueError):
            failed.append(check)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, monkeypatch, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, name
    path = tmp_path / "accept_mutant.py"
    path.write_text(text.replace(old, new))
    spec = importlib.util.spec_from_file_location("accept_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    monkeypatch.setattr(oracle, "accept_prefix", mod.accept_prefix)
    assert run_pins(), f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_every_pin():
    assert not run_pins()
