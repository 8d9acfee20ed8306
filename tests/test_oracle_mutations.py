"""Planted mistakes in the oracle are caught by its pins (CPU only).

Each case copies ``oracle/oracle.c`` to a temporary directory, changes one
expression into a plausible mistake (a wrong comparison, a dropped term, a
wrong sign or index, a transposed operand, a different rounding), compiles
the copy and runs the pins on it: at least one pin must fail.  The real
oracle is never modified.
"""

import os
import shutil

import pytest

import oracle
import oracle_pins
from oracle import build_oracle

MUTATIONS = {
    "threshold_gt": ("if (x >= tau) hit = 1;", "if (x > tau) hit = 1;"),
    "absmax_includes_outliers": ("if (flag_buf[k]) continue;", "(void)0;"),
    "code_by_reciprocal": ("float q = rintf(num / a);", "float q = rintf(num * (1.0f / a));"),
    "code_truncates": ("float q = rintf(num / a);", "float q = truncf(num / a);"),
    "code_scale_128": ("float num = 127.0f * x;", "float num = 128.0f * x;"),
    "drop_outlier_term": ("double v = p / 16129.0 + out[r * N + n];", "double v = p / 16129.0;"),
    "outlier_term_sign": ("double v = p / 16129.0 + out[r * N + n];",
                          "double v = p / 16129.0 - out[r * N + n];"),
    "dequant_127": ("double v = p / 16129.0", "double v = p / 16384.0"),
    "weight_index_reversed": ("s += (int64_t)x[k] * (int64_t)w[k];",
                              "s += (int64_t)x[k] * (int64_t)w[K - 1 - k];"),
    "transposed_weight": ("const int8_t *w = Wq + n * K;", "const int8_t *w = Wq + n;"),
    "outlier_weight_from_row": ("elem_to_double(W16[n * K + O[j]], fmt);",
                                "elem_to_double(W16[O[j] * K + n % K], fmt);"),
    "half_round_floor": ("double n = rint(ldexp(a, 10 - E));", "double n = floor(ldexp(a, 10 - E));"),
    "weight_scale_first_col": ("if (x > a) a = x;\n    }\n    sw[n] = a;",
                               "if (k == 0) a = x;\n    }\n    sw[n] = a;"),
    "bias_dropped": ("if (bias) v += elem_to_double(bias[n], fmt);", "(void)bias;"),
    "bias_sign": ("if (bias) v += elem_to_double(bias[n], fmt);",
                  "if (bias) v -= elem_to_double(bias[n], fmt);"),
    "bias_of_next_channel": ("if (bias) v += elem_to_double(bias[n], fmt);",
                             "if (bias) v += elem_to_double(bias[(n + 1) % N], fmt);"),
    "bf16_round_floor": ("double n = rint(ldexp(a, 7 - E));", "double n = floor(ldexp(a, 7 - E));"),
    "bf16_exponent_bias": ("return sign | (uint16_t)(((E + 127) << 7) | ((int)n - 128));",
                           "return sign | (uint16_t)(((E + 126) << 7) | ((int)n - 128));"),
    "bf16_subnormal_quantum": ("double n = rint(ldexp(a, 133));", "double n = rint(ldexp(a, 132));"),
    "bf16_code_unscaled": ("return code_of(ldexpf(x, 1 - e), ldexpf(a, 1 - e));",
                           "return code_of(x, a);"),
    "bf16_read_as_fp16": ("return fmt ? orc_bf16_to_double(b) : orc_half_to_double(b);",
                          "return orc_half_to_double(b);"),
    "w16_free_scale_128": ("double w = (double)Wq[n * K + O[j]] * (double)sw[n] / 127.0;",
                           "double w = (double)Wq[n * K + O[j]] * (double)sw[n] / 128.0;"),
    "w16_free_column_by_position": ("double w = (double)Wq[n * K + O[j]] * (double)sw[n] / 127.0;",
                                    "double w = (double)Wq[n * K + j] * (double)sw[n] / 127.0;"),
    "w16_free_scale_of_row_0": ("double w = (double)Wq[n * K + O[j]] * (double)sw[n] / 127.0;",
                                "double w = (double)Wq[n * K + O[j]] * (double)sw[0] / 127.0;"),
    "blockwise_truncates": ("q[i] = (int8_t)rintf(num / as);", "q[i] = (int8_t)truncf(num / as);"),
    "blockwise_scale_of_whole_tensor": ("for (int64_t i = i0; i < i1; i++) {\n      const float v",
                                        "for (int64_t i = 0; i < n; i++) {\n      const float v"),
    "blockwise_block_shifted": ("const int64_t i0 = b * B, i1", "const int64_t i0 = b * B + 1, i1"),
    "blockwise_decode_128": ("y[i] = (prod / 127.0f) / s;", "y[i] = (prod / 128.0f) / s;"),
    "blockwise_unscaled": ("return a >= 0x1p120f ? 0x1p-8f : 1.0f;", "return (void)a, 1.0f;"),
    "blockwise_scale_threshold_late": ("return a >= 0x1p120f ? 0x1p-8f : 1.0f;",
                                       "return a >= 0x1p122f ? 0x1p-8f : 1.0f;"),
    "blockwise_scale_of_first": ("if (v > a) a = v;", "if (i == i0) a = v;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(build_oracle.SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    mut = tmp_path / "oracle_mut.c"
    mut.write_text(src.replace(old, new))
    lib = build_oracle.build(str(mut), str(tmp_path / "liboracle_mut.so"), extra=("-w",))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutation {name} survived every pin"
