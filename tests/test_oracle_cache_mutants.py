"""Mutation check of the KV-cache step oracle's pins (CPU only).

Each case plants one plausible mistake in a private copy of
``oracle/gqa_cache.py`` (a wrong past or first-row formula, an off-by-one
bound, a wrong rotation sign or pair partner, query positions taken from the
append row, the attention seeing only the old rows, the latch ignored, ...),
loads the copy as a module and runs every pin of
``test_oracle_cache_pins.py`` against it.  Every mutant must fail at least
one pin; the unmodified copy must pass them all.
"""
import os
import types

import pytest

import oracle
import test_oracle_cache_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gqa_cache.py")

MUTANTS = [
    ("total_not_plus_one", "total = sk + 1", "total = sk"),
    ("past_from_q_seq", "        past = total - k_seq\n", "        past = total - q_seq\n"),
    ("first_from_k_seq", "first = total - q_seq", "first = total - k_seq"),
    ("capacity_bound_inclusive", "if total > capacity:", "if total >= capacity:"),
    ("past_bound_inclusive", "if past > capacity:", "if past >= capacity:"),
    ("position_bound_off_by_one", "if p < 0 or p >= cache_rows:", "if p < 0 or p > cache_rows:"),
    ("rotation_sign", "y[..., i0] = c * x0 - s * x1", "y[..., i0] = c * x0 + s * x1"),
    ("rotation_second_swapped", "y[..., i1] = s * x0 + c * x1", "y[..., i1] = c * x0 + s * x1"),
    ("half_split_partner", "(k, k + half, True)", "(k, k + half - 1, True)"),
    ("interleaved_pairs_swapped", "(2 * k, 2 * k + 1, True) if interleaved",
     "(2 * k + 1, 2 * k, True) if interleaved"),
    ("tail_pairs_shifted", "t = rot + 2 * (k - half)", "t = rot + 2 * (k - half) - 1"),
    ("query_positions_from_past", "P = positions([m[2] for m in meta], q_seq)",
     "P = positions([m[1] for m in meta], q_seq)"),
    ("append_at_first_row", "kc[b, :, past:past + k_seq]", "kc[b, :, first:first + k_seq]"),
    ("attend_old_rows_only", "totals = [m[0] for m in meta]", "totals = [m[1] for m in meta]"),
    ("position_ids_shifted", "return pos[:, :seq]", "return pos[:, :seq] + 1"),
    ("latch_ignored", "if poisoned:", "if False:"),
    ("queries_not_rotated", "    if rot:\n        P = positions([m[2]", "    if False:\n        P = positions([m[2]"),
]


def _load(src: str, name: str):
    mod = types.ModuleType(f"oracle._mutant_{name}")
    mod.__package__ = "oracle"
    exec(compile(src, f"gqa_cache_{name}.py", "exec"), mod.__dict__)
    return mod


def _failed_pins(mod):
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(mod)
        except Exception:  # an assertion, or a mutant that breaks outright
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_cache_pins_reject_mutant(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found once"
    assert _failed_pins(_load(src.replace(old, new), name)), f"mutant {name} passed every pin"


def test_unmutated_copy_passes_every_cache_pin():
    assert _failed_pins(_load(open(SRC).read(), "identity")) == []
