"""Mutation check of the oracle pins.

Each case below plants one plausible mistake in a copy of the oracle's source (a wrong
divisor, eps outside the square root, a dropped index, a flipped sign, swapped operands,
a wrong table row, ties rounded away from even, a second rounding, a wrong binary16
exponent bias, overflow or subnormal range), compiles the copy
with the host compiler into a temporary directory and runs the pin battery against it.
Every mutant must fail at least one pin. The real oracle is never modified.
"""

from __future__ import annotations

import os

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = {
    "mean divides by cols + 1":
        ("ss / static_cast<double>(cols)", "ss / static_cast<double>(cols + 1)"),
    "eps outside the square root":
        ("std::sqrt(mean_sq + eps)", "(std::sqrt(mean_sq) + eps)"),
    "weight index dropped":
        ("y[j] = x[j] / rms * w[j];", "y[j] = x[j] / rms * w[0];"),
    "absolute value instead of square":
        ("const double t = x[j] * x[j];", "const double t = std::fabs(x[j]);"),
    "sign of the first-half rotation":
        ("y[i] = x1 * c[i] - x2 * sn[i];", "y[i] = x1 * c[i] + x2 * sn[i];"),
    "halves transposed in the second output":
        ("y[i + half] = x2 * c[i] + x1 * sn[i];", "y[i + half] = x1 * c[i] + x2 * sn[i];"),
    "sin and cos swapped":
        ("rope_head(x + off, sin_t + s * half, cos_t + s * half, y + off, half);",
         "rope_head(x + off, cos_t + s * half, sin_t + s * half, y + off, half);"),
    "table row fixed at 0 in the storage path":
        ("const int64_t s = t - b * S;", "const int64_t s = 0 * (t - b * S);"),
    "ties rounded away from zero":
        ("if (frac > 0.5 || (frac == 0.5 && std::fmod(fl, 2.0) != 0.0)) m = fl + 1.0;\n"
         "    const double r = m * q;                    // exact: m <= 256",
         "if (frac >= 0.5) m = fl + 1.0;\n"
         "    const double r = m * q;                    // exact: m <= 256"),
    "binary16 ties rounded away from zero":
        ("if (frac > 0.5 || (frac == 0.5 && std::fmod(fl, 2.0) != 0.0)) m = fl + 1.0;\n"
         "    const double r = m * q;                     // exact: m <= 2048",
         "if (frac >= 0.5) m = fl + 1.0;\n"
         "    const double r = m * q;                     // exact: m <= 2048"),
    "rounded twice through fp32":
        ("static_cast<uint16_t*>(base)[i] = double_to_bf16(v);",
         "static_cast<uint16_t*>(base)[i] = double_to_bf16(static_cast<float>(v));"),
    "subnormal spacing wrong":
        ("if (E < -126) E = -126;", "if (E < -127) E = -127;"),
    "binary16 exponent bias 14":
        ("return static_cast<uint16_t>(sign | ((Er + 15) << 10) | mant);",
         "return static_cast<uint16_t>(sign | ((Er + 14) << 10) | mant);"),
    "binary16 overflow one binade late":
        ("if (r >= 65536.0) return static_cast<uint16_t>(sign | 0x7C00u);",
         "if (r >= 131072.0) return static_cast<uint16_t>(sign | 0x7C00u);"),
    "binary16 subnormals flushed to zero":
        ("        return static_cast<uint16_t>(sign | static_cast<uint16_t>(std::ldexp(r, 24)));",
         "        return sign;"),
    "add path normalizes x instead of h":
        ("hr[j] = load_elem(h, i, dtype);", "hr[j] = load_elem(x, i, dtype);"),
    "cache scatter uses the token index instead of its slot":
        ("store_elem(cache_n, slot * Dn + j, yn[j], dtype);",
         "store_elem(cache_n, (t % num_slots) * Dn + j, yn[j], dtype);"),
    "cache rope part uses the batch's first table row":
        ("sn[i] = static_cast<double>(sin_t[s * half + i]);\n                c[i] = static_cast<double>(cos_t[s * half + i]);\n            }\n            rmsnorm_row",
         "sn[i] = static_cast<double>(sin_t[0 * s * half + i]);\n                c[i] = static_cast<double>(cos_t[0 * s * half + i]);\n            }\n            rmsnorm_row"),
    "interleaved pair order swapped":
        ("store_elem(y, base + 2 * i, x0 * c - x1 * sn, dtype);",
         "store_elem(y, base + 2 * i, x1 * c - x0 * sn, dtype);"),
    "interleaved table row from the token, not its position":
        ("const double c = static_cast<double>(cos_t[p * half + i]);",
         "const double c = static_cast<double>(cos_t[(t % max_pos) * half + i]);"),
    "tables use theta^(-i/D)":
        ("const double freq = std::pow(theta, (-2.0 * static_cast<double>(i)) /",
         "const double freq = std::pow(theta, (-1.0 * static_cast<double>(i)) /"),
    "layernorm variance divides by n - 1":
        ("const double var = neumaier_sum(d2.data(), n) / static_cast<double>(n);",
         "const double var = neumaier_sum(d2.data(), n) / static_cast<double>(n - 1);"),
    "layernorm beta added before the weight":
        ("y[j] = xhat * g[j] + b[j];", "y[j] = (xhat + b[j]) * g[j];"),
    "kv repeat tiles the heads instead of interleaving them":
        ("const int64_t dst_row = (b * T + t) * Hout + h * n_rep + r;",
         "const int64_t dst_row = (b * T + t) * Hout + r * Hk + h;"),
    "kv new rows use the table row of their index among the new rows":
        ("sn[i] = static_cast<double>(sin_t[t * half + i]);\n                    c[i] = static_cast<double>(cos_t[t * half + i]);",
         "sn[i] = static_cast<double>(sin_t[(t - P) * half + i]);\n                    c[i] = static_cast<double>(cos_t[(t - P) * half + i]);"),
    "kv past rows rotated too":
        ("const bool rotate = !old_row && sin_t != nullptr;", "const bool rotate = sin_t != nullptr;"),
    "add path normalizes the unrounded sum":
        ("hr[j] = load_elem(h, i, dtype);",
         "hr[j] = load_elem(x, i, dtype) + load_elem(r, i, dtype);"),
}


def _battery(lib):
    """Run a fixed selection of pins; return the names of those that failed."""
    checks = [
        ("bf16 hand", lambda: [pins.test_bf16_round_hand(lib, v, b) for v, b in pins.BF16_HAND]),
        ("bf16 vs torch", lambda: pins.test_bf16_round_matches_torch_on_fp32_inputs(lib)),
        ("f16 hand", lambda: [pins.test_f16_round_hand(lib, v, b) for v, b in pins.F16_HAND]),
        ("f16 vs numpy", lambda: pins.test_f16_round_matches_numpy_on_fp64_inputs(lib)),
        ("f16 decode", lambda: pins.test_f16_value_matches_numpy_on_every_pattern(lib)),
        ("rms storage f16", lambda: pins.test_rmsnorm_storage_path_rounds_the_fp64_result_once(lib, "f16")),
        ("rms worked", lambda: [pins.test_rmsnorm_worked_cases(lib, [3.0, 4.0], [1.0, 1.0],
                                                                [3 / 12.5**0.5, 4 / 12.5**0.5]),
                                pins.test_rmsnorm_worked_cases(lib, [1.0, -1.0, 1.0, -1.0],
                                                                [0.5, 2.0, -3.0, 4.0],
                                                                [0.5, -2.0, -3.0, -4.0])]),
        ("rms constant row", lambda: pins.test_rmsnorm_constant_row_closed_form(lib, 0.01, 1e-5, 7)),
        ("rms eps in mean", lambda: pins.test_rmsnorm_eps_enters_the_mean_not_the_sum(lib)),
        ("rms numpy norm", lambda: pins.test_rmsnorm_matches_numpy_vector_norm(lib)),
        ("rms storage bf16", lambda: pins.test_rmsnorm_storage_path_rounds_the_fp64_result_once(lib, "bf16")),
        ("rope d2", lambda: pins.test_rope_worked_case_d2(lib)),
        ("rope complex", lambda: pins.test_rope_is_complex_multiplication(lib)),
        ("rope interleaved", lambda: pins.test_rope_rotate_half_equals_interleaved_on_deinterleaved_input(lib)),
        ("rope storage", lambda: pins.test_rope_storage_path_rounds_the_fp64_result_once(lib, "f32")),
        ("rope single rounding", lambda: pins.test_rope_single_rounding_crafted_case(lib)),
        ("kv cache", lambda: [pins.test_kv_cache_scatter_is_rmsnorm_and_rope_of_each_token(lib, d)
                              for d in ("bf16", "f32")]),
        ("rope interleaved", lambda: [pins.test_rope_interleaved_is_rotate_half_on_deinterleaved_input(lib, d)
                                      for d in ("bf16", "f32")]),
        ("rope tables", lambda: pins.test_rope_tables_match_numpy_and_closed_forms(lib)),
        ("layernorm worked", lambda: pins.test_layernorm_worked_case(lib)),
        ("layernorm numpy", lambda: pins.test_layernorm_matches_numpy_mean_and_std(lib)),
        ("kv cat repeat", lambda: [pins.test_kv_cat_repeat_without_tables_is_numpy_concatenate_and_repeat(
            lib, "bf16", 2, 5, 3, 3, 8, 4)]),
        ("kv cat repeat rope", lambda: pins.test_kv_cat_repeat_rotates_new_rows_at_their_absolute_positions(lib)),
        ("add rmsnorm", lambda: [pins.test_add_rmsnorm_h_is_the_library_sum_and_y_the_rmsnorm_of_h(lib, d)
                                 for d in ("bf16", "f32")]),
    ]
    failed = []
    for name, fn in checks:
        try:
            fn()
        except (AssertionError, ValueError):
            failed.append(name)
    return failed


def test_unmutated_oracle_passes_the_battery():
    assert _battery(oracle.load()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    pattern, replacement = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(pattern) == 1, f"mutation site not unique or missing: {pattern!r}"
    mutant_src = os.path.join(tmp_path, "mutant.cpp")
    with open(mutant_src, "w") as f:
        f.write(src.replace(pattern, replacement))
    lib_path = oracle.build(mutant_src, os.path.join(tmp_path, "libmutant.so"), force=True)
    failed = _battery(oracle.load(lib_path))
    assert failed, f"no pin caught the mutant '{name}'"
