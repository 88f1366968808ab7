"""Plants plausible mistakes in a copy of the C oracle (on the CPU) and checks
that the pins catch every one of them.  This is evidence that the pins in
test_oracle_pins.py constrain each part of the definition: the beta index, the
gate sign and base, the dot product, the sign of A, the orientation of the
result, the substitution's operand order, the diagonal and the chunk restart,
and in the unfused chain's halves the gate, the strictness of A and the
solve's operand order and sign."""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kkt_solve_oracle.c")

MUTANTS = {
    "beta_on_column": ("double bi = beta ? beta[i * ldb] : 1.0;",
                       "double bi = beta ? beta[j * ldb] : 1.0;"),
    "gate_sign": ("exp(g[i * ldg] - g[j * ldg])", "exp(g[j * ldg] - g[i * ldg])"),
    "gate_exp2": ("exp(g[i * ldg] - g[j * ldg])", "exp2(g[i * ldg] - g[j * ldg])"),
    "dot_drops_last_term": ("for (int64_t d = 0; d < K; ++d)", "for (int64_t d = 0; d < K - 1; ++d)"),
    "i_minus_a": ("v -= A[i * L + j] * X[j * L + c];", "v += A[i * L + j] * X[j * L + c];"),
    "transposed_operand": ("v -= A[i * L + j] * X[j * L + c];", "v -= A[j * L + i] * X[j * L + c];"),
    "transposed_result": ("out[i * ldo + c] = (c < L) ? X[i * L + c] : 0.0;",
                          "out[i * ldo + c] = (c < L) ? X[c * L + i] : 0.0;"),
    "no_unit_diagonal": ("double v = (i == c) ? 1.0 : 0.0;", "double v = 0.0;"),
    "global_chunk_grid": ("for (int64_t c0 = s; c0 < e; c0 += C) {",
                          "for (int64_t c0 = s - (s % C); c0 < e; c0 += C) {"),
    # the halves of the unfused chain
    "A_gate_divides": ("a = bi * dot * gate;", "a = bi * dot / gate;"),
    "A_keeps_diagonal": ("if (j < i) {", "if (j <= i) {"),
    "solve_reads_transposed_A": ("v -= Ain[i * lda + j] * X[j * L + c];",
                                 "v -= Ain[j * lda + i] * X[j * L + c];"),
    "solve_i_minus_a": ("v -= Ain[i * lda + j] * X[j * L + c];", "v += Ain[i * lda + j] * X[j * L + c];"),
}

# Pins to run against each mutant (function, kwargs).
PINS = [
    (pins.test_structure_and_residual, dict(L=17)),
    (pins.test_brute_force_gauss_jordan, dict(L=32)),
    (pins.test_single_coupled_pair_hand_value, {}),
    (pins.test_chain_L3_closed_form, {}),
    (pins.test_collinear_keys_delta_rule_product_form, {}),
    (pins.test_varlen_equals_separate_sequences, {}),
    (pins.test_golden_fixture_reproduces, {}),
    (pins.test_chunk_A_hand_values, {}),
    (pins.test_solve_tril_equals_library_inverse_and_reads_only_strict_lower, {}),
    (pins.test_solve_tril_L3_closed_form, {}),
    (pins.test_chain_of_halves_equals_fused_oracle, dict(name="B1_T256_H8_K128")),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, name
    mut = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mut)
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", str(so), str(c), "-lm"])
    lib = ctypes.CDLL(str(so))
    real = oracle._load()
    for fn in ("oracle_kkt_solve_chunk", "oracle_kkt_solve", "oracle_chunk_A_chunk",
               "oracle_solve_tril_chunk", "oracle_chunk_A", "oracle_solve_tril"):
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
        getattr(lib, fn).restype = getattr(real, fn).restype
    return lib


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_planted_mistake_is_caught(tmp_path, monkeypatch, name):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    oracle._load()
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for fn, kw in PINS:
        try:
            fn(**kw)
        except (AssertionError, RuntimeError):
            caught.append(fn.__name__)
    assert caught, f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_the_same_pins():
    for fn, kw in PINS:
        fn(**kw)
