"""Plant plausible mistakes in copies of the oracle and check that the pins fail.

Each mutant is the oracle's C source with one textual edit, compiled into a
temporary directory and loaded next to the real oracle.  A mutant that passes
every fast pin would mean the pins cannot see that kind of mistake.
"""
import os

import pytest

import oracle as O
import oracle_pins as P

SRC = os.path.join(os.path.dirname(O.oracle.__file__), "w12_oracle.c")

# (name, text in the oracle, replacement)
MUTANTS = [
    ("window_one_binade_low", "return emax - 15;", "return emax - 16;"),
    ("window_one_binade_short", "e <= ebase + 15;", "e <= ebase + 14;"),
    ("floor_15_not_16", "if (emax < 16)\n        emax = 16;", "if (emax < 15)\n        emax = 15;"),
    ("inf_sets_window", "return e >= 1 && e <= 254;", "return e >= 1 && e <= 255;"),
    ("zero_in_window", "return is_finite_normal(b) && e >= ebase && e <= ebase + 15;",
     "return (is_finite_normal(b) && e >= ebase && e <= ebase + 15) || (b & 0x7FFF) == 0;"),
    ("decode_drops_B", "((A & 7) << 4) | B);", "((A & 7) << 4));"),
    ("decode_sign_shift", "(uint16_t)(((A >> 3) << 15) |", "(uint16_t)(((A >> 3) << 14) |"),
    ("decode_exponent_origin", "((ebase + E) << 7)", "((ebase + E - 1) << 7)"),
    ("A_low_bits_from_wrong_end", "return (bf16_sign(b) << 3) | (bf16_mant(b) >> 4);",
     "return (bf16_sign(b) << 3) | (bf16_mant(b) & 7);"),
    ("B_slots_odds_first", "return k8 / 2;         /* evens in slots 0..3 */",
     "return 4 + k8 / 2;"),
    ("AE_nibbles_swapped", "(uint8_t)((A << 4) | E);", "(uint8_t)((E << 4) | A);"),
    ("placeholder_without_sign", "return bf16_sign(b) << 3; /* R4 placeholder */", "return 0;"),
    ("escape_not_written_back", "out[(row - n0) * K + col] = (uint16_t)(entry & 0xFFFF);", ";"),
    ("escape_column_mod_128", "((uint32_t)(k - k0) << 16)", "((uint32_t)(k % 128) << 16)"),
    ("escape_row_field", "((uint32_t)(n - n0) << 24)", "((uint32_t)(n - n0) << 23)"),
    ("q8_keeps_B", "if (with_b) {\n                word", "if (1) {\n                word"),
    ("q8_patches_escapes", "if (!with_b)\n        return 0;", "if (0)\n        return 0;"),
    ("gemm_drops_first_term", "for (k = 0; k < K; k++)\n                acc += bf16_value",
     "for (k = 1; k < K; k++)\n                acc += bf16_value"),
    ("gemm_x_reversed", "acc += bf16_value(x[m * K + k]) * bf16_value(w[n * K + k]);",
     "acc += bf16_value(x[m * K + (K - 1 - k)]) * bf16_value(w[n * K + k]);"),
    ("gemm_float_accumulator", "            double acc = 0.0;\n            for (k = 0; k < K; k++)\n                acc +=",
     "            float acc = 0.0f;\n            for (k = 0; k < K; k++)\n                acc +="),
    ("abs_gemm_signed", "acc += p < 0 ? -p : p;", "acc += p;"),
    ("round_ties_away", "return (uint16_t)(((lo >> 16) & 1u) ? (hi >> 16) : (lo >> 16));",
     "return (uint16_t)(hi >> 16);"),
    ("round_truncates", "    if (dlo < dhi)\n        return (uint16_t)(lo >> 16);",
     "    if (1)\n        return (uint16_t)(lo >> 16);"),
    ("round_never_overflows", "ldexp(1.0, 128)", "HUGE_VAL"),
    ("silu_operands_swapped", "h[m * (N / 2) + i] = g / (1.0 + exp(-g)) * u;",
     "h[m * (N / 2) + i] = u / (1.0 + exp(-u)) * g;"),
    ("silu_sign", "g / (1.0 + exp(-g)) * u", "g / (1.0 + exp(g)) * u"),
    ("silu_pairs_shifted", "u = y[m * N + 2 * i + 1];", "u = y[m * N + (2 * i + 3) % N];"),
    ("count_max_ties_low", "if (c >= best) {", "if (c > best) {"),
    ("count_max_window_15_binades", "for (e = b; e <= b + 15; e++)\n            c += count[e];",
     "for (e = b; e <= b + 14; e++)\n            c += count[e];"),
    ("count_max_search_short", "for (b = 1; b <= b1; b++) {", "for (b = 1; b < b1; b++) {"),
    ("saturated_A_missing", "return (bf16_sign(b) << 3) | 7; /* R13 saturated placeholder */",
     "return bf16_sign(b) << 3;"),
    ("saturated_E_zero", "    if (above_window(b, ebase))\n        return 15;\n    return 0;\n}\n\nstatic int field_B",
     "    if (above_window(b, ebase))\n        return 0;\n    return 0;\n}\n\nstatic int field_B"),
    ("saturated_B_zero", "        return 15;\n    return 0;\n}\n\n/* R6", "        return 0;\n    return 0;\n}\n\n/* R6"),
    ("i8_round_half_away", "t = rintf(v / sc);", "t = roundf(v / sc);"),
    ("i8_scale_over_128", "sc = amax / 127.0f;", "sc = amax / 128.0f;"),
    ("i8_clamp_126", "if (t > 127.0f)\n                t = 127.0f;", "if (t > 126.0f)\n                t = 126.0f;"),
    ("i8_amax_counts_inf", "if (isfinite(v) && fabsf(v) > amax)", "if (!isnan(v) && fabsf(v) > amax)"),
    ("i8_gemm_drops_scale", "acc += bf16_value(x[m * K + k]) * ((double)q[n * K + k] * (double)scale[n]);",
     "acc += bf16_value(x[m * K + k]) * ((double)q[n * K + k]);"),
    ("above_one_binade_late", "return is_finite_normal(b) && bf16_exp(b) > ebase + 15;",
     "return is_finite_normal(b) && bf16_exp(b) > ebase + 16;"),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / "w12_oracle.c"
    src.write_text(source.replace(old, new, 1))
    path = O.oracle.build(src=str(src), build_dir=str(tmp_path), name=f"lib_{name}.so")
    lib = O.oracle.load(path)
    failures = []
    for pin in P.FAST_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, RuntimeError) as e:  # caught by a pin
            failures.append((pin.__name__, str(e)[:60]))
    assert failures, f"mutant {name} passed every pin"
