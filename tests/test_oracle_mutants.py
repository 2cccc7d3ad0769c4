"""Planted mistakes in copies of the oracle must each fail at least one pin.

Every mutant is a one-token edit of the oracle's C source, compiled into a
temporary directory on the CPU; the real oracle is never modified.
"""
import os
import shutil

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTANTS = {
    "drop_write_term": ("+ b_t * v_t[j] * k_t[l]", "+ 0.0 * v_t[j] * k_t[l]"),
    "erase_sign": ("- b_t * k_t[i] * k_t[l]", "+ b_t * k_t[i] * k_t[l]"),
    "erase_without_beta": ("- b_t * k_t[i] * k_t[l]", "- k_t[i] * k_t[l]"),
    "gate_on_write_term": ("a_t * SE[j * dk + l] + b_t * v_t[j] * k_t[l]",
                           "a_t * (SE[j * dk + l] + b_t * v_t[j] * k_t[l])"),
    "no_gate": ("a_t * SE[j * dk + l]", "SE[j * dk + l]"),
    "wrong_index_in_product": ("S[j * dk + i] * E[i * dk + l]", "S[j * dk + l] * E[i * dk + l]"),
    "tile_not_transposed": ("S[j * dk + i] = tile[i * dv + j]", "S[j * dk + i] = tile[j * dk + i]"),
    "output_reads_key": ("S[j * dk + i] * q_t[i]", "S[j * dk + i] * k_t[i]"),
    "snapshot_off_by_one": ("t + 1 == a_r", "t == a_r"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, name
    src = tmp_path / "gdn_oracle.c"
    src.write_text(text.replace(old, new))
    shutil.copy(os.path.join(os.path.dirname(SRC), "gdn_oracle.h"), tmp_path / "gdn_oracle.h")
    lib = oracle.load(oracle.build(str(src), str(tmp_path / "libmutant.so")))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
