"""Plant plausible mistakes in a copy of the oracle and require a pin to catch each.

Each mutant is a textual edit of ``oracle/oracle.c`` compiled to a temporary
library (the committed oracle is untouched); every pin of ``oracle_pins`` is
run against it and at least one must fail.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "diagonal_excluded": ("if (causal && pk > pq)", "if (causal && pk >= pq)"),
    "window_off_by_one": ("pq - pk >= window", "pq - pk > window"),
    "gqa_modulo_map": ("const int g = h / G;", "const int g = h % Hkv;"),
    "subset_head_local_kv": ("const int g = h / G;", "const int g = (int)hr / G;"),
    "subset_rows_ignored": ("const int64_t i = rows ? rows[rr] : rr;", "const int64_t i = rr;"),
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "lse_log2": ("*ls = m + log(l);", "*ls = m + log2(l);"),
    "lse_unshifted": ("*ls = m + log(l);", "*ls = log(l);"),
    "no_normalisation": ("o[e] = acc[e] / l;", "o[e] = acc[e];"),
    "merge_weight_unnormalised": ("const double w = exp(x - L);", "const double w = exp(x - mx);"),
    "merge_lse_unshifted": ("const double L = mx + log(sum);", "const double L = log(sum);"),
    "merge_skips_first": ("for (int p = 0; p < n; ++p) {\n            const double x = lses[p][h * n_rows + r];\n            if (x == -INFINITY)",
                          "for (int p = 1; p < n; ++p) {\n            const double x = lses[p][h * n_rows + r];\n            if (x == -INFINITY)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "oracle_mut.c"
    so_path = tmp_path / "liboracle_mut.so"
    c_path.write_text(mutated)
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-shared", "-fPIC", str(c_path),
                           "-o", str(so_path), "-lm"])
    saved = oracle._lib
    oracle._lib = oracle._bind(ctypes.CDLL(str(so_path)))
    failures = []
    try:
        for check in pins.ALL_CHECKS:
            try:
                check()
            except AssertionError as e:
                failures.append(check.__name__)
    finally:
        oracle._lib = saved
    assert failures, f"mutant {name} passed every pin"
