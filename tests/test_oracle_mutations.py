"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake in a copy of the oracle's C source (on the
CPU, in a temporary directory), compiles it, and runs every pin of
test_oracle_pins.py, test_oracle_pins_bf16.py and test_oracle_pins_acc16.py
against the planted copy: at least one pin has to fail.  A mutation is one
(old, new) replacement or a list of them.
The committed oracle is never modified.
"""
import inspect
import os

import pytest

import oracle
import tests.test_oracle_pins as pins
import tests.test_oracle_pins_acc16 as pins_acc16
import tests.test_oracle_pins_bf16 as pins_bf16

_SRC = os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c")

MUTATIONS = {
    "fp32_accumulator": (
        "    double s = 0.0;\n    for (int64_t k = 0; k < K; ++k) s += g_f16_table[a[k]] * g_f16_table[b[k]];",
        "    float s = 0.0f;\n    for (int64_t k = 0; k < K; ++k) s += (float)(g_f16_table[a[k]] * g_f16_table[b[k]]);"),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k) s +=",
                          "for (int64_t k = 0; k + 1 < K; ++k) s +="),
    "reversed_k_index_of_B": ("g_f16_table[a[k]] * g_f16_table[b[k]]",
                              "g_f16_table[a[k]] * g_f16_table[b[K - 1 - k]]"),
    "sign_error": ("s += g_f16_table[a[k]] * g_f16_table[b[k]]",
                   "s -= g_f16_table[a[k]] * g_f16_table[b[k]]"),
    "truncating_round": ("if (rem > 0.5) {", "if (rem > 1.0) {"),
    "ties_away_from_zero": ("r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "r = fl + 1.0;"),
    "rounded_twice_via_fp32": ("j->C[m * j->ldc + n] = oracle_f64_to_f16(s);",
                               "j->C[m * j->ldc + n] = oracle_f64_to_f16((float)s);"),
    "subnormal_scale": ("v = ldexp((double)frac, -24);", "v = ldexp((double)frac, -25);"),
    "overflow_saturates": ("if (E > 15) return sign | 0x7c00;\n    if (E < -14)",
                           "if (E > 15) return sign | 0x7bff;\n    if (E < -14)"),
    "B_row_stride_ignored": ("j->B + n * j->ldb", "j->B + n * j->K"),
    "bf16_fp32_accumulator": (
        "    double s = 0.0;\n    for (int64_t k = 0; k < K; ++k) s += g_bf16_table[a[k]] * g_bf16_table[b[k]];",
        "    float s = 0.0f;\n    for (int64_t k = 0; k < K; ++k) s += (float)(g_bf16_table[a[k]] * g_bf16_table[b[k]]);"),
    "bf16_subnormal_scale": ("v = ldexp((double)frac, -133);", "v = ldexp((double)frac, -132);"),
    "bf16_exponent_bias": ("v = ldexp((double)(frac | 0x80), efield - 134);",
                           "v = ldexp((double)(frac | 0x80), efield - 133);"),
    "bf16_round_bias": ("double q = ldexp(a, 7 - E);", "double q = ldexp(a, 7 - E) + 0.25;"),
    "bf16_overflow_saturates": ("if (E > 127) return sign | 0x7f80;\n    if (E < -126)",
                                "if (E > 127) return sign | 0x7f7f;\n    if (E < -126)"),
    "bf16_reversed_k_index": ("g_bf16_table[a[k]] * g_bf16_table[b[k]]",
                              "g_bf16_table[a[k]] * g_bf16_table[b[K - 1 - k]]"),
    "acc16_step_32": ("#define ORACLE_ACC16_STEP 16", "#define ORACLE_ACC16_STEP 32"),
    "acc16_step_8": ("#define ORACLE_ACC16_STEP 16", "#define ORACLE_ACC16_STEP 8"),
    "acc16_accumulator_not_carried": ("double s = g_f16_table[acc];", "double s = 0.0;"),
    "acc16_rounded_only_at_end": [
        ("    uint16_t acc = 0;\n    for (int64_t k0 = 0;", "    uint16_t acc = 0;\n    double carry = 0.0;\n    for (int64_t k0 = 0;"),
        ("double s = g_f16_table[acc];", "double s = carry;"),
        ("        acc = oracle_f64_to_f16(s);\n", "        carry = s;\n        acc = oracle_f64_to_f16(s);\n")],
    "acc16_last_partial_step_dropped": ("int64_t k1 = k0 + ORACLE_ACC16_STEP < K ? k0 + ORACLE_ACC16_STEP : K;",
                                        "int64_t k1 = k0 + ORACLE_ACC16_STEP < K ? k0 + ORACLE_ACC16_STEP : k0;"),
}


def _pin_calls():
    """Every (name, function, kwargs) of the pin modules, parametrizations expanded."""
    calls = []
    for name, fn in (inspect.getmembers(pins, inspect.isfunction)
                     + inspect.getmembers(pins_bf16, inspect.isfunction)
                     + inspect.getmembers(pins_acc16, inspect.isfunction)):
        if not name.startswith("test_"):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((name, fn, {}))
            continue
        argnames, values = marks[0].args[0], marks[0].args[1]
        names = [a.strip() for a in argnames.split(",")]
        for v in values:
            v = v if isinstance(v, tuple) else (v,)
            calls.append((name, fn, dict(zip(names, v))))
    return calls


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation, tmp_path):
    edits = MUTATIONS[mutation]
    edits = edits if isinstance(edits, list) else [edits]
    src = open(_SRC).read()
    for old, new in edits:
        assert src.count(old) >= 1, f"mutation anchor for {mutation} not found: {old!r}"
        src = src.replace(old, new)
    mutated = tmp_path / "gemm_oracle_mutated.c"
    mutated.write_text(src)
    planted = oracle.Oracle(oracle.compile_source(str(mutated), str(tmp_path / "lib.so")))
    caught = []
    for name, fn, kw in _pin_calls():
        try:
            fn(planted, **kw)
        except AssertionError:
            caught.append(name)
    assert caught, f"no pin caught the planted mistake {mutation!r}"
