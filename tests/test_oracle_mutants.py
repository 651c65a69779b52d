"""The pins catch plausible mistakes: each test plants one mistake in a copy of
the oracle's C source, builds it on the CPU, and checks that at least one pin
fails against that broken build (and that the unbroken build passes them all).
No GPU is involved."""
import os
import subprocess

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
