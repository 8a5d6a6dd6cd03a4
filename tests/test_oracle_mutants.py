"""The oracle's pins must reject plausible mistakes.

Each case copies qk_oracle.c to a temporary directory, plants one mistake in
the copy (a dropped term, a flipped sign, a wrong index, a transposed
operand, a wrong rounding), compiles it and runs the pins of test_oracle.py
against it.  At least one pin has to fail for every planted mistake.  The
oracle source itself is never modified.
"""
import subprocess

import pytest

from oracle import oracle as orc
from tests import test_oracle as pins

MUTATIONS = {
    "drop_min_term": ("* (double)q - dmin * (double)m;", "* (double)q;"),
    "min_sign": ("* (double)q - dmin * (double)m;", "* (double)q + dmin * (double)m;"),
    "sc_high_bits_index": ("((scales[j - 4] >> 6) << 4);\n        *m", "((scales[j] >> 6) << 4);\n        *m"),
    "m_high_bits_index": ("((scales[j] >> 6) << 4);\n    }", "((scales[j - 4] >> 6) << 4);\n    }"),
    "m_low_index": ("*m = scales[j + 4] & 63;", "*m = scales[j] & 63;"),
    "nibble_swap": ("(byte & 15) : (byte >> 4)", "(byte >> 4) : (byte & 15)"),
    "qs_chunk_index": ("blk[16 + 32 * (j / 2) + i]", "blk[16 + 16 * j + i]"),
    "transposed_x": ("double p = w[c] * (double)x[b * K + c];", "double p = w[c] * (double)x[c * batch + b];"),
    "fp16_bias": ("e - 25);", "e - 24);"),
    "fp16_subnormal": ("ldexp((double)f, -24);", "ldexp((double)f, -25);"),
    "q8_block_stride": ("row + (c / 32) * 34;", "row + (c / 32) * 32;"),
    "q8_quant_offset": ("blk[2 + (c % 32)]", "blk[1 + (c % 32)]"),
    "abs_sum_drops_abs": ("acc += p;\n                mag += fabs(p);\n            }\n            y[b * n_rows + i] = acc;\n            if (s) s[b * n_rows + i] = mag;\n        }\n    }\n    free(w);\n    return 0;",
                          "acc += p;\n                mag += p;\n            }\n            y[b * n_rows + i] = acc;\n            if (s) s[b * n_rows + i] = mag;\n        }\n    }\n    free(w);\n    return 0;"),
    "bf16_ties_away": ("rest > 0x8000u ||", "rest >= 0x8000u ||"),
    "gemm_skips_x_rounding": ("xb[e] = qko_bf16_to_f64(qko_f32_to_bf16(x[e]));", "xb[e] = (double)x[e];"),
    "gemm_skips_w_rounding": ("w[c] = qko_bf16_to_f64(qko_f32_to_bf16((float)w[c]));", "w[c] = (double)(float)w[c];"),
    "q8_encode_no_clamp_sign": ("if (q < -127.0) q = -127.0;", "if (q < -127.0) q = 127.0;"),
    "q4_encode_high_nibble": ("(uint8_t)(best << 4);", "(uint8_t)(best << 3);"),
    "swiglu_gate_up_swapped": ("i < batch * n; ++i) h[i] = silu(g[i]) * u[i];", "i < batch * n; ++i) h[i] = silu(u[i]) * g[i];"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "q6_qh_shift": ("(blk[128 + 32 * n + l] >> (2 * t)) & 3;", "(blk[128 + 32 * n + l] >> t) & 3;"),
    "q6_ql_half": ("blk[64 * n + l + 32 * (t % 2)];", "blk[64 * n + l + 32 * (t / 2)];"),
    "q6_scale_index": ("blk[192 + i / 16];", "blk[192 + i / 32];"),
    "q6_offset": ("(double)(q - 32);", "(double)(q - 31);"),
    "q6_scale_unsigned": ("(int)(int8_t)blk[192 + i / 16];", "(int)blk[192 + i / 16];"),
    "experts_input_row_mod": ("x + (a / xk) * K, 1, y + a * rows", "x + (a % xk) * K, 1, y + a * rows"),
    "experts_ignores_id": ("idx[r] = e * rows + r;", "idx[r] = r;"),
    "swiglu_gemm_exact_gate": ("int rc = qko_gemm_bf16(fmt, wq, K, gate_rows, n, x, M, g, sg);",
                               "int rc = qko_gemv(fmt, wq, K, gate_rows, n, x, M, g, sg);"),
    "silu_missing_z": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    "swiglu_gemm_gate_up_swapped": ("i < M * n; ++i) h[i] = silu(g[i]) * u[i];", "i < M * n; ++i) h[i] = silu(u[i]) * g[i];"),
    "q4_row_stride": ("return ((K + 255) / 256) * 144;\n}", "return ((K + 255) / 256) * 128;\n}"),
    "q8_encode_divisor": ("qko_f64_to_fp16(amax / 127.0);", "qko_f64_to_fp16(amax / 128.0);"),
    "q4_sc_low_mask": ("*sc = scales[j] & 63;", "*sc = scales[j] & 31;"),
}

PINS = [
    (pins.test_fp16_decode_every_pattern, {}),
    (pins.test_fp16_encode_matches_numpy, {}),
    (pins.test_bf16_round_matches_torch, {}),
    (pins.test_layout_probes, {"fmt": "q8_0"}),
    (pins.test_layout_probes, {"fmt": "q4_k"}),
    (pins.test_layout_probes, {"fmt": "q6_k"}),
    (pins.test_unit_vectors_recover_matrix, {"fmt": "q4_k", "rows": 3, "K": 512}),
    (pins.test_unit_vectors_recover_matrix, {"fmt": "q8_0", "rows": 3, "K": 96}),
    (pins.test_all_zero_blocks, {"fmt": "q4_k"}),
    (pins.test_constant_block_closed_form, {"fmt": "q4_k", "w_const": 2.5, "n_blocks": 3}),
    (pins.test_constant_block_closed_form, {"fmt": "q8_0", "w_const": 3.0, "n_blocks": 7}),
    (pins.test_dot_matches_blas, {"fmt": "q8_0", "rows": 17, "K": 576, "B": 3}),
    (pins.test_q8_0_roundtrip_nearest, {}),
    (pins.test_q4_k_roundtrip_bound, {}),
    (pins.test_gemm_bf16_reference_matches_torch_rounding, {}),
    (pins.test_gemm_bf16_reference_exact_on_bf16_inputs, {}),
    (pins.test_swiglu_known_values, {}),
    (pins.test_swiglu_odd_part_identity, {"z": 1.75}),
    (pins.test_experts_select_expert_and_input_row, {"xk": 2}),
    (pins.test_swiglu_gemm_reference_rounds_to_bf16, {}),
    (pins.test_swiglu_gemm_reference_on_bf16_exact_inputs, {}),
    (pins.test_q4_k_unit_scales_reduce_to_plain_nibbles, {}),
    (pins.test_q8_0_requantise_reproduces_the_bytes, {}),
    (pins.test_q4_k_bytes_per_weight_give_the_page_intensity, {}),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(orc.SRC).read()
    assert src.count(old) == 1, f"mutation {name} does not match the oracle source exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = str(tmp_path / f"lib_{name}.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                           "-ffp-contract=off", str(path), "-o", lib, "-lm"])
    return lib


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(tmp_path, name):
    old, new = MUTATIONS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    caught = []
    with orc.using(lib):
        for fn, kw in PINS:
            try:
                fn(orc, **kw)
            except AssertionError:
                caught.append(fn.__name__)
    assert caught, f"no pin rejects the planted mistake {name}"


def test_unmutated_copy_passes_all_pins(tmp_path):
    lib = _build_mutant(tmp_path, "identity", "#include <math.h>", "#include <math.h>")
    with orc.using(lib):
        for fn, kw in PINS:
            fn(orc, **kw)
