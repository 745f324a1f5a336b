"""Plant plausible mistakes in copies of the oracle and check the pins catch them.

Each mutant is a textual edit of oracle/nvfp4_oracle.c compiled into a temporary
library on the CPU; the real oracle is never modified.  A mutant "survives" if
every pin in test_oracle_pins.py still passes against it -- that would mean the
pins cannot tell the mistake apart from the correct oracle.
"""
from __future__ import annotations

import os
import subprocess

import pytest

import oracle
from test_oracle_pins import ALL_CHECKS

SRC = os.path.join(os.path.dirname(oracle.__file__), "nvfp4_oracle.c")

MUTANTS = {
    "nibble_order_swapped": ("out[j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));",
                             "out[j] = (uint8_t)(c[2 * j + 1] | (c[2 * j] << 4));"),
    "e2m1_ties_away": ("double v = rint(a / quantum) * quantum;  /* ties to the even multiple */",
                       "double v = floor(a / quantum + 0.5) * quantum;"),
    "e4m3_ties_away": ("double v = rint(q / quantum) * quantum;",
                       "double v = floor(q / quantum + 0.5) * quantum;"),
    "e4m3_no_subnormal_binade": ("        e = -6;                /* subnormals",
                                 "        e = e;                 /* subnormals"),
    "e4m3_bias_8": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "e2m1_subnormal_wrong": ("double mag = (e == 0) ? 0.5 * m :", "double mag = (e == 0) ? 1.0 * m :"),
    "tensor_scale_without_6": ("float ts = amax / 2688.0f;", "float ts = amax / 448.0f;"),
    "scale_order_reassociated": ("float q = (bamax / 6.0f) / ts;", "float q = bamax / (6.0f * ts);"),
    "reciprocal_multiply": ("nvfp4_oracle_e2m1_encode(blk[j] / d);",
                            "nvfp4_oracle_e2m1_encode(blk[j] * (1.0f / d));"),
    "signed_zero_dropped": ("uint8_t sign = signbit(vf) ? 0x8 : 0x0;",
                            "uint8_t sign = (vf <= -0.25f) ? 0x8 : 0x0;"),
    "block_amax_first_only": ("                if (a > bamax)\n                    bamax = a;\n            }\n\n            /* Step 3b",
                              "                if (j == 0)\n                    bamax = a;\n            }\n\n            /* Step 3b"),
    "x_row_stride_wrong": ("const uint16_t *xn = x + n * K;", "const uint16_t *xn = x + n;"),
    "tensor_scale_dropped": ("y[i * n_rows + j] = (double)ts * sum;", "y[i * n_rows + j] = sum;"),
    "scale_block_off_by_one": ("nvfp4_oracle_e4m3_value(scales[m * (K / 16) + k / 16]);",
                               "nvfp4_oracle_e4m3_value(scales[m * (K / 16) + (k / 16 + 1) % (K / 16)]);"),
    "code_nibble_swapped_in_product": ("int code = (k & 1) ? (byte >> 4) : (byte & 0xF);",
                                       "int code = (k & 1) ? (byte & 0xF) : (byte >> 4);"),
    "silu_sign_flipped": ("h[o] = gv / (1.0 + exp(-gv)) * uv;", "h[o] = gv / (1.0 + exp(gv)) * uv;"),
    "clamp_at_4": ("if (a >= 6.0) {\n        code = 7;", "if (a >= 4.0) {\n        code = 6;"),
    "fp6_emax_3": ("shared = (e - 1) - 2;", "shared = (e - 1) - 3;"),
    "fp6_no_clamp": ("if (shared < -127)\n                    shared = -127;", ""),
    "fp6_subnormal_as_quarter": ("double mag = (e == 0) ? m / 8.0 :", "double mag = (e == 0) ? m / 4.0 :"),
    "fp6_ties_to_odd": ("if (d < best_d || (d == best_d && (c & 1) == 0)) {",
                        "if (d < best_d || (d == best_d && (c & 1) == 1)) {"),
    "fp6_sign_of_zero_dropped": ("(signbit(vf) ? 0x20 : 0)", "(vf < 0.0f ? 0x20 : 0)"),
    "fp6_multiply_by_scale": ("nvfp4_oracle_e2m3_encode(blk[i] / X)", "nvfp4_oracle_e2m3_encode(blk[i] * X)"),
    "fp6_unpack_misses_byte": ("if (bit % 8 > 2)", "if (bit % 8 > 4)"),
    "fp6_x_row_stride_wrong": ("const uint16_t *xrow = x + n * K;", "const uint16_t *xrow = x + n;"),
    "fp6_scale_bias_126": ("ldexp(1.0, (int)scales[m * (K / 128) + k / 128] - 127)",
                           "ldexp(1.0, (int)scales[m * (K / 128) + k / 128] - 126)"),
    "w4a4_activation_scale_dropped": ("const double scale = (double)x_ts * (double)ts;",
                                      "const double scale = (double)ts;"),
    "w4a4_token_index_is_position": ("weight_unscaled(x_codes, x_scales, K, n, k)",
                                     "weight_unscaled(x_codes, x_scales, K, i, k)"),
}


def _build_mutant(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path_c = tmp_path / f"{name}.c"
    path_c.write_text(src.replace(old, new))
    path_so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-w", "-shared", str(path_c), "-o", str(path_so), "-lm"],
                   check=True)
    return oracle.load_variant(str(path_so))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    lib = _build_mutant(name, old, new, tmp_path)
    caught = []
    for check in ALL_CHECKS:
        try:
            check(lib)
        except (AssertionError, ValueError, IndexError):
            caught.append(check.__name__)
    assert caught, f"mutant {name} passes every pin"
