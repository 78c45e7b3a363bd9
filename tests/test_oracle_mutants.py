"""Mutation check of the oracle's pins (CPU only).

Each case below plants one plausible mistake in a private copy of
``oracle/pva_oracle.c`` (a dropped scale, a transposed head map, a wrong
causal offset, a softcap applied to the wrong quantity, a stale row offset,
masked rows not zeroed, ...), compiles the copy with gcc and runs the pin
checks against it.  Every mutant must be rejected by at least one pin; the
real oracle passes them all (``test_oracle_pins.py``).
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pva_oracle.c")

# (name, text in pva_oracle.c, replacement)
MUTANTS = [
    ("head_map_modulo", "const int g = h / group;", "const int g = h % Hkv;"),
    ("causal_offset_dropped", "i + (L_kv - L_q);", "i;"),
    ("causal_offset_sign", "i + (L_kv - L_q);", "i + (L_q - L_kv);"),
    ("causal_strict", "j > frontier", "j >= frontier"),
    ("scale_dropped", "double s = scale * dot;", "double s = dot;"),
    ("scale_squared", "double s = scale * dot;", "double s = scale * scale * dot;"),
    ("softcap_no_inner_divide", "softcap * tanh(s / softcap)", "softcap * tanh(s)"),
    ("softcap_dropped", "if (softcap != 0.0) s = softcap * tanh(s / softcap);", ""),
    ("no_max_subtract_zero_rows", "if (n_visible == 0) return;", ""),
    ("value_row_uses_key_stride", "((kv_start + j) * Hkv + g) * (int64_t)dv;",
     "((kv_start + j) * Hkv + g) * (int64_t)d;"),
    ("query_row_offset", "q + (tok * H + h) * (int64_t)d;", "q + (tok * H + h % 2) * (int64_t)d;"),
    ("kv_start_ignored", "const int64_t kv_start = cu_kv[b];", "const int64_t kv_start = cu_q[b];"),
    ("no_normalise", "const double p = scores[j] / l;", "const double p = scores[j];"),
    ("owner_off_by_one", "if ((int64_t)cu_q[mid] <= tok) lo = mid;", "if ((int64_t)cu_q[mid] < tok) lo = mid;"),
    ("window_off_by_one", "j < frontier + 1 - local_window", "j <= frontier + 1 - local_window"),
    ("window_from_row_not_limit", "j < frontier + 1 - local_window", "j < i + 1 - local_window"),
    ("window_ignored", "if (local_window > 0 && j < frontier + 1 - local_window)", "if (0)"),
    ("padded_frontier_dropped", "const int visible = j < limit &&", "const int visible ="),
    ("padded_offset_from_slot", "const int64_t offset = nonpad[b] - q_seq;",
     "const int64_t offset = kv_seq - q_seq;"),
    ("padded_frontier_inclusive", "const int visible = j < limit &&",
     "const int visible = j <= limit &&"),
    ("padded_head_map", "const int g = h / group;\n      const int64_t limit",
     "const int g = h % Hkv;\n      const int64_t limit"),
    ("padded_value_batch_stride", "v + (((int64_t)b * kv_seq + j)", "v + (((int64_t)b * q_seq + j)"),
    ("padded_no_normalise", "orow[c] += (w[j] / l) * vrow[c];", "orow[c] += w[j] * vrow[c];"),
]


def _compile(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(mutated)
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-std=c99", str(c),
                           "-o", str(so), "-lm"])
    return str(so)


def _pin_checks():
    """The pin tests, run as plain functions; returns the names that failed."""
    failed = []
    checks = [
        ("golden", lambda: [pins.test_worked_examples(c) for c in pins._golden_cases()]),
        ("sdpa_padded", lambda: [pins.test_padded_equal_lengths_match_sdpa(s, H, Hkv)
                                 for s in range(4) for H, Hkv in [(4, 2), (6, 1)]]),
        ("suffix", lambda: [pins.test_tail_aligned_is_suffix_of_self_attention(s) for s in range(4)]),
        ("nonpad", lambda: [pins.test_nonpad_kv_seqlen_prefix_sum_reproduces_padded_masking(s)
                            for s in range(4)]),
        ("bruteforce", lambda: [pins.test_bruteforce_tiny_random_against_sdpa(s) for s in range(6)]),
        ("window", lambda: ([pins.test_window_row_is_plain_attention_over_the_window_keys(s, c)
                             for s in range(2) for c in (False, True)],
                            pins.test_window_of_one_returns_the_value_row_at_the_causal_limit())),
        ("padded", lambda: ([pins.test_padded_form_matches_sdpa_with_both_frontiers(s)
                             for s in range(6)],
                            [pins.test_padded_form_equals_packed_form_on_the_prefix_sum(s)
                             for s in range(6)],
                            pins.test_padded_form_ignores_what_the_padding_holds())),
        ("closed_forms", lambda: (pins.test_constant_value_rows_return_that_row(),
                                  pins.test_zero_query_gives_mean_of_visible_values(),
                                  pins.test_empty_sequences_and_fully_masked_rows_are_zero())),
    ]
    for name, fn in checks:
        try:
            fn()
        except (AssertionError, ValueError):
            failed.append(name)
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, old, new):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    so = _compile(tmp_path, name, old, new)
    with oracle.use_library(so):
        failed = _pin_checks()
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_copy_passes_every_pin(tmp_path):
    so = _compile(tmp_path, "identity", "#include <math.h>", "#include <math.h>")
    with oracle.use_library(so):
        assert _pin_checks() == []
