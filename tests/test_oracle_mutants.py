"""Plant mistakes in copies of the oracle (on the CPU) and check that the pins
catch each one: a wrong nibble order, swapped scale/bias planes, a wrong group
size, a dropped bias, a sign error, weights rounded to bf16, a transposed
index, a dropped glue term and swapped gate and up halves must each fail at
least one pin."""
import os
import shutil
import tempfile

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "q4_oracle.c")

MUTANTS = {
    "nibble_order": ("return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 0x0F);",
                     "return (k & 1) ? (unsigned)(byte & 0x0F) : (unsigned)(byte >> 4);"),
    "planes_swapped": ("const uint8_t* plane = W + N * (K / 2);\n",
                       "const uint8_t* plane = W + N * (K / 2) + 2 * N * (K / Q4O_GROUP);\n"),
    "group_32": ("uint64_t g = k / Q4O_GROUP;", "uint64_t g = (k / 32) % (K / Q4O_GROUP);"),
    "bias_dropped": ("* (double)nib(W, K, n, k) + bias_at(W, N, K, n, g);",
                     "* (double)nib(W, K, n, k);"),
    "bias_sign": ("* (double)nib(W, K, n, k) + bias_at(W, N, K, n, g);",
                  "* (double)nib(W, K, n, k) - bias_at(W, N, K, n, g);"),
    "bf16_folded_w": ("for (uint64_t k = 0; k < K; ++k) j->wrow[k] = q4o_weight(j->W, j->N, K, n, k);",
                      "for (uint64_t k = 0; k < K; ++k) j->wrow[k] = bf16_to_f64(f64_to_bf16_rne("
                      "q4o_weight(j->W, j->N, K, n, k)));"),
    "row_index_transposed": ("uint8_t byte = W[n * (K / 2) + k / 2];",
                             "uint8_t byte = W[(k / 2) * 1 + n * 0 + (n * (K / 2)) * 0 + n];"),
    "glue_no_gate": ("if (kind == 2) a = a / (1.0 + exp(-a)) * (double)yr[K + k];",
                     "if (kind == 2) a = (double)yr[K + k];"),
    "tie_rounds_up": ("else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "else r = fl + 1.0;"),
    "gate_up_swapped": ("if (kind == 2) a = a / (1.0 + exp(-a)) * (double)yr[K + k];",
                        "if (kind == 2) { double u = (double)yr[K + k]; a = u / (1.0 + exp(-u)) * a; }"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    d = tempfile.mkdtemp(prefix="q4o_mut_")
    try:
        path = os.path.join(d, "m.c")
        open(path, "w").write(mutated)
        so = oracle.compile_oracle(src=path, out=os.path.join(d, "libm.so"))
        o = oracle.Oracle(oracle.load_library(so))
        failed = []
        for pin in P.ALL_PINS:
            try:
                pin(o)
            except AssertionError:
                failed.append(pin.__name__)
        assert failed, f"no pin caught mutant {name}"
    finally:
        shutil.rmtree(d, ignore_errors=True)
