"""The pins catch plausible mistakes: each test plants one mistake in a copy of
the oracle's C source, builds it on the CPU, and checks that at least one pin
fails against that broken build (and that the unbroken build passes them all).
No GPU is involved."""
import os
import subprocess
import types

import pytest

import oracle
import oracle_pins
from oracle import build as obuild

# (name, text in w4a16_oracle.c, replacement) -- one planted mistake each
MUTANTS = [
    ("twos_complement_off_by_one", "if (v >= 8) v -= 16;", "if (v > 8) v -= 16;"),
    ("nibble_order_reversed", "q[n * K + k] = (int8_t)nibble_value(word >> (4 * (k % 8)));",
     "q[n * K + k] = (int8_t)nibble_value(word >> (4 * (7 - k % 8)));"),
    ("gemv_nibble_order_reversed", "int q = nibble_value(word >> (4 * (k % 8)));",
     "int q = nibble_value(word >> (4 * (7 - k % 8)));"),
    ("group_index_wrong", "double s = orc_half_to_double(scales[n * (K / G) + k / G]);",
     "double s = orc_half_to_double(scales[n * (K / G) + (k / G) % 1]);"),
    ("unpack_transposed", "q[n * K + k] = (int8_t)", "q[k * N + n] = (int8_t)"),
    ("gemv_output_transposed", "y[m * N + n] = acc;", "y[n * M + m] = acc;"),
    ("dropped_last_term", "for (int64_t k = 0; k < K; ++k)\n        acc +=",
     "for (int64_t k = 0; k < K - 1; ++k)\n        acc +="),
    ("gemv_sign_flip", "acc += orc_half_to_double(x[m * K + k]) * w_hat(qweight, scales, K, G, n, k);\n      y[m * N + n]",
     "acc -= orc_half_to_double(x[m * K + k]) * w_hat(qweight, scales, K, G, n, k);\n      y[m * N + n]"),
    ("scale_divisor", "float d = amax / 7.0f;", "float d = amax / 8.0f;"),
    ("truncating_round", "double r = round((double)wg[k] / s);", "double r = trunc((double)wg[k] / s);"),
    ("ties_away_in_fp16", "return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;"),
    ("subnormal_scale", "double m = round_half_even(ldexp(a, 24));",
     "double m = round_half_even(ldexp(a, 23));"),
    ("exponent_bias", "v = ldexp((double)(1024 + f), e - 25);", "v = ldexp((double)(1024 + f), e - 24);"),
    ("x_index_transposed", "acc += orc_half_to_double(x[m * K + k]) * w_hat(qweight, scales, K, G, n, k);\n      y[m * N + n]",
     "acc += orc_half_to_double(x[k * M + m]) * w_hat(qweight, scales, K, G, n, k);\n      y[m * N + n]"),
    ("silu_exp_sign", "return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    ("silu_missing_one", "return v / (1.0 + exp(-v));", "return v / exp(-v);"),
    ("attn_missing_scale", "s[t] = dot * scale;", "s[t] = dot;"),
    ("attn_gqa_mapping_modulo", "const int64_t g = h / group;", "const int64_t g = h % n_kv_heads;"),
    ("attn_values_from_keys", "acc += s[t] * orc_half_to_double(v[(g * t_stride + t) * D + d]);",
     "acc += s[t] * orc_half_to_double(k[(g * t_stride + t) * D + d]);"),
    ("attn_dropped_last_key", "for (int64_t t = 0; t < T; ++t) {\n      s[t] = exp(s[t] - smax);",
     "for (int64_t t = 0; t < T - 1; ++t) {\n      s[t] = exp(s[t] - smax);"),
    ("attn_stride_ignored", "dot += orc_half_to_double(q[h * D + d]) * orc_half_to_double(k[(g * t_stride + t) * D + d]);",
     "dot += orc_half_to_double(q[h * D + d]) * orc_half_to_double(k[(g * T + t) * D + d]);"),
    ("a8_round_half_away", "const float r = nearbyintf(p);", "const float r = roundf(p);"),
    ("a8_scale_128", "const float sb = amax > 0.0f ? amax / 127.0f : 0.0f;",
     "const float sb = amax > 0.0f ? amax / 128.0f : 0.0f;"),
    ("a8_weight_scale_index", "scales[n * (K / G) + (b * ORC_A8_BLOCK) / G]", "scales[n * (K / G) + b / G]"),
    ("a8_activation_scale_dropped", "* (double)sx[b];", ";"),
    ("q4k_high_scale_bits_swapped", "*sc = (b[j + 4] & 15) | ((b[j - 4] >> 6) << 4);",
     "*sc = (b[j + 4] & 15) | ((b[j] >> 6) << 4);"),
    ("q4k_nibble_half_swapped", "return blk[16 + 32 * c + i] & 15;", "return blk[16 + 32 * c + i] >> 4;"),
    ("q4k_min_sign", "w[n * K + s * ORC_QK + e] = dq - m1;", "w[n * K + s * ORC_QK + e] = dq + m1;"),
    ("q4k_odd_subblock_index", "*j = 2 * c + 1;", "*j = 2 * c;"),
    ("swiglu_gate_up_swapped",
     "orc_silu(orc_half_to_double(g[i])) * orc_half_to_double(u[i])",
     "orc_silu(orc_half_to_double(u[i])) * orc_half_to_double(g[i])"),
    ("dequant_f64_transposed",
     "for (int64_t k = 0; k < K; ++k) w_out[n * K + k] = w_hat(qweight, scales, K, G, n, k);",
     "for (int64_t k = 0; k < K; ++k) w_out[k * N + n] = w_hat(qweight, scales, K, G, n, k);"),
]

# (name, text in oracle/__init__.py, replacement) -- planted mistakes in the
# Python-level tolerance machinery (row norms and the two checkers)
PY_MUTANTS = [
    ("row_norms_per_column", "return np.sqrt(np.sum(w * w, axis=1))", "return np.sqrt(np.sum(w * w, axis=0))"),
    ("row_norms_squared", "return np.sqrt(np.sum(w * w, axis=1))", "return np.sum(w * w, axis=1)"),
    ("check_gemv_strict_abs", "bool(np.all(max_err <= bound))", "bool(np.all(max_err < bound))"),
    ("check_gemv_strict_rel", "and rel <= rel_l2", "and rel < rel_l2"),
    ("check_gemv_x_norm_axis", "np.sqrt(np.sum(x_f64 * x_f64, axis=1))", "np.sqrt(np.sum(x_f64 * x_f64))"),
    ("check_gemv_max_per_column", "max_err = err.max(axis=1)", "max_err = err.max(axis=0).max() + 0 * err.max(axis=1)"),
    ("check_gemv_bound_one_row", "bound = abs_slope * np.sqrt(np.sum(x_f64 * x_f64, axis=1)) * max_row_norm + abs_floor",
     "bound = abs_slope * np.sqrt(np.sum(x_f64 * x_f64, axis=1)).max() * max_row_norm + abs_floor"),
    ("check_gemv_rel_per_row_max", "rel = float(np.sqrt(np.sum(err * err)) / denom)",
     "rel = float(np.sqrt(np.sum(err * err, axis=1)).max() / denom)"),
    ("check_attn_strict", "bool((err <= bound).all())", "bool((err < bound).all())"),
    ("check_attn_head_mapping_modulo", "vmax[np.arange(n_heads) // group]", "vmax[np.arange(n_heads) % Hkv]"),
    ("check_attn_whole_stride", "half_to_double(v[:, :T, :])", "half_to_double(v)"),
    ("check_attn_max_over_heads", "vmax = np.abs(half_to_double(v[:, :T, :])).reshape(Hkv, -1).max(axis=1)",
     "vmax = np.abs(half_to_double(v[:, :T, :])).reshape(Hkv, -1).max(axis=1).max() + 0 * np.arange(Hkv)"),
]


def _build_mutant(tmp_path, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = src.replace(old, new, 1)
    c = tmp_path / "mutant.c"
    c.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *obuild.CFLAGS, "-w", str(c), "-o", str(so), "-lm"], check=True)
    return oracle.lib(str(so))


def test_unbroken_oracle_passes_every_pin():
    assert oracle_pins.failing_pins(oracle.lib()) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    L = _build_mutant(tmp_path, old, new)
    failing = oracle_pins.failing_pins(L)
    assert failing, f"no pin caught the planted mistake {name}"


def _load_py_mutant(old, new):
    """A copy of the oracle's Python module with one planted mistake (it still
    loads the unbroken C library)."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "__init__.py")).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    mod.__package__ = "oracle"
    mod.__file__ = oracle.__file__
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_planted_checker_mistake_is_caught(name, old, new):
    O = _load_py_mutant(old, new)
    failing = oracle_pins.failing_pins(oracle.lib(), O)
    assert failing, f"no pin caught the planted mistake {name}"
