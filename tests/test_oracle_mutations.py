"""Planted mistakes: each mutant copy of the oracle's C source must fail at
least one pin in test_oracle_pins.py, test_oracle_tails_pins.py or
test_oracle_prefill_pins.py.

This checks that the pins are sharp enough to catch the plausible slips a
hand-written attention oracle can make (wrong GQA head, swapped K/V, dropped
scale or max, wrong row order, off-by-one mask, broken merge weight, wrong
append slot; for per-decoder tails: another decoder's tail, the shared table
used for the tail, a dropped tail, an un-rebased tail position).  Mutants
are compiled on the CPU into a temporary directory; the real oracle is never
modified.  Partial prefill: attention that is not causal, that excludes the
token itself, or that writes rows head-major.
"""
import os
import subprocess

import pytest

import oracle
import tests.test_oracle_pins as pins
import tests.test_oracle_prefill_pins as prefill_pins
import tests.test_oracle_tails_pins as tail_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "shkv_oracle.c")

MUTANTS = {
    "gqa_head_modulo": ("return h / (Hq / Hkv);", "return h % Hkv;"),
    "keys_as_values": ("token_ptr(j, j->v_pages, b, g, t0 + i)", "token_ptr(j, j->k_pages, b, g, t0 + i)"),
    "no_scale": ("s[i] = scale * acc;", "s[i] = acc;"),
    "max_not_subtracted_in_numerator": ("double p = exp(s[i] - smax) / denom;", "double p = exp(s[i]) / denom;"),
    "head_major_rows": ("return (long)m * Hq + h;", "return (long)h * N + m;"),
    "mask_off_by_one": ("int t1 = j->t_end < L ? j->t_end : L;", "int t1 = j->t_end < L + 1 ? j->t_end : L + 1;"),
    "lse_without_log": ("*lse = smax + log(denom);", "*lse = smax + denom;"),
    "merge_weight_sign": ("double w = exp(l - M);", "double w = exp(M - l);"),
    "append_slot_shift": ("long dst = (((long)page * Hkv + g) * P + pos % P) * (long)D;",
                          "long dst = (((long)page * Hkv + g) * P + (pos + 1) % P) * (long)D;"),
    "token_slot_shift": ("return pool + (((long)page * Hkv + g) * P + t % P) * (long)D;",
                         "return pool + (((long)page * Hkv + g) * P + (t + 1) % P) * (long)D;"),
    # per-decoder unique tails
    "tail_of_first_decoder": ("page = j->tail_table[((long)b * j->N + m) * j->max_tail_pages + t / j->P];",
                              "page = j->tail_table[((long)b * j->N + 0) * j->max_tail_pages + t / j->P];"),
    "tail_through_shared_table": ("page = j->tail_table[((long)b * j->N + m) * j->max_tail_pages + t / j->P];",
                                  "page = j->block_table[(long)b * j->max_pages + t / j->P];"),
    "tail_dropped": ("const int n = j->seq_lens[b] + j->tail_lens[(long)b * j->N + m];",
                     "const int n = j->seq_lens[b];"),
    "tail_position_not_rebased": ("t = i - L;", "t = i;"),
    # partial-prefill attention
    "prefill_not_causal": ("const int n = L - j->n_new + i + 1;", "const int n = L;"),
    "prefill_excludes_itself": ("const int n = L - j->n_new + i + 1;", "const int n = L - j->n_new + i;"),
    "prefill_row_order": ("const long row = ((long)b * j->n_new + i) * j->Hq + h;",
                          "const long row = ((long)b * j->Hq + h) * j->n_new + i;"),
}

PIN_TESTS = ([getattr(pins, n) for n in dir(pins) if n.startswith("test_")] +
             [getattr(tail_pins, n) for n in dir(tail_pins) if n.startswith("test_")] +
             [getattr(prefill_pins, n) for n in dir(prefill_pins) if n.startswith("test_")])


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, mutant_dir, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in the oracle source"
    path_c = os.path.join(mutant_dir, f"{name}.c")
    path_so = os.path.join(mutant_dir, f"lib{name}.so")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", path_so, path_c, "-lm"])
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "build", lambda force=False: path_so)
    failed = []
    for t in PIN_TESTS:
        try:
            t()
        except (AssertionError, RuntimeError):
            failed.append(t.__name__)
    monkeypatch.setattr(oracle, "_lib", None)
    assert failed, f"no pin caught the planted mistake {name!r}"
