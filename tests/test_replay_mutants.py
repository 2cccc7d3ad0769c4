"""Planted mistakes in copies of the ReplaySSM buffer oracle must each fail a pin.

Each mutant is a one-token edit of oracle/replay.py, loaded as a module of the
oracle package from a temporary file; the real oracle is never modified.
"""
import importlib.util
import os
import sys

import pytest

import oracle
import test_replay_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "replay.py")

MUTANTS = {
    "outputs_of_the_first_rows": ("o_seq[u, int(n[r]):int(n[r] + T[r])]", "o_seq[u, 0:int(T[r])]"),
    "flush_without_room_for_drafts": ("flushed = keep + int(prob.max_T) > C", "flushed = keep > C"),
    "commit_keeps_only_the_drafts": ("keep = n + prob.accepted.astype(np.int64)",
                                     "keep = prob.accepted.astype(np.int64)"),
    "rows_shifted": ("    lo = slot * C\n", "    lo = slot * C + 1\n"),
    "replay_skips_the_buffer": ("_slot_rows(buf, int(prob.slot_ids[r]), int(n[r] + T[r]))",
                                "_slot_rows(buf, int(prob.slot_ids[r]), int(T[r]))"),
}


def run_pins():
    checks = [pins.test_empty_buffers_are_the_plain_calls,
              pins.test_rows_past_the_drafts_never_matter_and_buffered_rows_do,
              pins.test_flush_bookkeeping, pins.test_rejects_overfull_buffers]
    checks += [lambda c=c: pins.test_steps_equal_committing_every_step(c) for c in (7, 12, 23)]
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
    path = tmp_path / "replay_mutant.py"
    path.write_text(text.replace(old, new))
    spec = importlib.util.spec_from_file_location("oracle.replay_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    monkeypatch.setitem(sys.modules, "oracle.replay_mutant", mod)
    spec.loader.exec_module(mod)
    monkeypatch.setattr(oracle, "replay_verify", mod.replay_verify)
    monkeypatch.setattr(oracle, "replay_commit", mod.replay_commit)
    assert run_pins(), f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_every_pin():
    assert not run_pins()
