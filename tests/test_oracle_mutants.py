"""Planted mistakes in copies of the oracle must turn its pins red (no GPU).

Each case copies ``oracle/qmm_oracle.c``, replaces one exact snippet (the
mistake: a dropped term, a wrong sign or index, a swapped order), compiles the
copy with gcc into a temporary directory and runs the named pins on it. The
test passes only when at least one of those pins fails on the mutant. The real
oracle source is never modified.
"""

import os

import pytest

import oracle
from tests import oracle_pins as P

MUTANTS = [
    ("fwht_sign", "v[i + h] = lo - hi;\n            }\n}\n\n/* The same transform in fp64",
     "v[i + h] = hi - lo;\n            }\n}\n\n/* The same transform in fp64", [P.pin_hadamard_matrix]),
    ("fwht_f64_dropped_stage", "for (int h = 1; h < n; h <<= 1)\n        for (int i = 0; i < n; i++)\n            if ((i & h) == 0) {\n                double",
     "for (int h = 2; h < n; h <<= 1)\n        for (int i = 0; i < n; i++)\n            if ((i & h) == 0) {\n                double",
     [P.pin_hadamard_matrix, P.pin_rotation_invariance]),
    ("nibble_high_first", "int u = (k & 1) ? (byte >> 4) : (byte & 0xf);",
     "int u = (k & 1) ? (byte & 0xf) : (byte >> 4);", [P.pin_nibble_order]),
    ("nibble_offset_binary", "q[(size_t)n * K + k] = (int8_t)(u >= 8 ? u - 16 : u);",
     "q[(size_t)n * K + k] = (int8_t)(u - 8);", [P.pin_nibble_order, P.pin_partials_brute_force]),
    ("round_ties_away", "float r = rintf(v[i] / s);", "float r = roundf(v[i] / s);", [P.pin_quant_fixture]),
    ("scale_128", "float s = amax / 127.0f;", "float s = amax / 128.0f;",
     [P.pin_quant_fixture, P.pin_quant_properties]),
    ("missing_rotation_factor", "sx[(size_t)m * G + g] = s * c;", "sx[(size_t)m * G + g] = s;",
     [P.pin_quant_fixture, P.pin_rotated_quant_exact, P.pin_quantized_rotation_end_to_end]),
    ("zero_group_scale", "sx[(size_t)m * G + g] = 0.0f;", "sx[(size_t)m * G + g] = 1.0f;",
     [P.pin_quant_fixture, P.pin_quant_properties]),
    ("partials_group_offset", "acc += (int64_t)q[(size_t)n * K + k] * a[(size_t)m * K + k];",
     "acc += (int64_t)q[(size_t)n * K + k] * a[(size_t)m * K + kl];", [P.pin_partials_brute_force]),
    ("gemm_scale_index", "double t = oracle_f16_to_f64(sw[(size_t)n * G + g]) * (double)sx[(size_t)m * G + g] * (double)p;",
     "double t = oracle_f16_to_f64(sw[(size_t)n * G + g]) * (double)sx[(size_t)m * G] * (double)p;",
     [P.pin_gemm_w4a8_dequant]),
    ("gemm_transposed_weight", "p += (int64_t)qrow[k] * a[(size_t)m * K + k];",
     "p += (int64_t)qrow[K - 1 - k] * a[(size_t)m * K + k];", [P.pin_gemm_w4a8_dequant]),
    ("tree_pairing", "S[(size_t)m * G + g] = ((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7]));",
     "S[(size_t)m * G + g] = ((c[0] + c[2]) + (c[1] + c[3])) + ((c[4] + c[6]) + (c[5] + c[7]));",
     [P.pin_group_sum_tree_fixture]),
    ("tree_flat", "S[(size_t)m * G + g] = ((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7]));",
     "S[(size_t)m * G + g] = (((((((c[0] + c[1]) + c[2]) + c[3]) + c[4]) + c[5]) + c[6]) + c[7]);",
     [P.pin_group_sum_tree_fixture]),
    ("chunk_right_to_left", "for (int i = 1; i < 8; i++) acc = acc + xg[8 * j + i];",
     "acc = xg[8 * j + 7]; for (int i = 6; i >= 0; i--) acc = acc + xg[8 * j + i];",
     [P.pin_group_sum_tree_fixture]),
    ("affine_bias_dropped", "y += sv * qx + bv * sumx;", "y += sv * qx;", [P.pin_affine_dequant_and_bias]),
    ("pack_natural_slots", "int s = (e % 2 == 0) ? e / 2 : 4 + e / 2;", "int s = e;", [P.pin_pack_positions]),
    ("pack_no_offset", "int u = variant == ORACLE_W4A8 ? q + 8 : q;", "int u = q;",
     [P.pin_pack_positions, P.pin_pack_roundtrip_and_invariance]),
    ("pack_piece_stride", "return (size_t)p * 2048 + (size_t)r * 16 + 4 * j + s / 2;",
     "return (size_t)p * 16 + (size_t)r * 32 + 4 * j + s / 2;", [P.pin_pack_positions]),
    ("f16_exponent", "v = ldexp((double)(1024 + f), e - 25);", "v = ldexp((double)(1024 + f), e - 24);",
     [P.pin_f16_to_f64]),
    ("cq4_cb_scale_dropped", "oracle_f16_to_f64(sw[(size_t)n * G + g]) * (double)cb_scale * (double)sx",
     "oracle_f16_to_f64(sw[(size_t)n * G + g]) * (double)sx", [P.pin_cq4_dequant_and_invariances]),
    ("cq4_gemm_no_lookup", "p += (int64_t)codebook[idx[k]] * a[(size_t)m * K + k];",
     "p += (int64_t)(idx[k] - 8) * a[(size_t)m * K + k];", [P.pin_cq4_dequant_and_invariances]),
    ("cq4_partials_signed_index", "acc += (int64_t)codebook[idx[(size_t)n * K + k]] * a[(size_t)m * K + k];",
     "acc += (int64_t)codebook[idx[(size_t)n * K + k] ^ 8] * a[(size_t)m * K + k];",
     [P.pin_cq4_identity_codebook_equals_w4a8, P.pin_cq4_partials_brute_force]),
    ("cq4_trailer_scale_offset", "memcpy(tr + 16, &cb_scale, 4);", "memcpy(tr + 20, &cb_scale, 4);",
     [P.pin_cq4_blob_trailer_and_roundtrip]),
    ("il4_rows_not_interleaved", "const uint8_t* piece = block + (size_t)c * 4 * cb + (size_t)ni * cb;",
     "const uint8_t* piece = block + (size_t)ni * (K / 2) + (size_t)c * cb;",
     [P.pin_interleaved4_fixture, P.pin_interleaved4_layout]),
    ("il4_block_stride", "const uint8_t* block = panels + (size_t)nb * 2 * K;",
     "const uint8_t* block = panels + (size_t)nb * K;", [P.pin_interleaved4_fixture, P.pin_interleaved4_layout]),
    ("il4_norms_row_major", "size_t at = ((size_t)nb * G + g) * 4 + ni;", "size_t at = (size_t)n * G + g;",
     [P.pin_interleaved4_fixture, P.pin_interleaved4_layout]),
    ("rot_transposed", "for (int k = 0; k < K; k++) acc = fmaf(Ri[k], xm[k], acc);",
     "for (int k = 0; k < K; k++) acc = fmaf(R[(size_t)k * K + i], xm[k], acc);",
     [P.pin_rotation_fixture, P.pin_rotation_properties]),
    ("rot_mul_then_add", "for (int k = 0; k < K; k++) acc = fmaf(Ri[k], xm[k], acc);",
     "for (int k = 0; k < K; k++) acc = acc + Ri[k] * xm[k];", [P.pin_rotation_fixture]),
    ("rot_reverse_order", "for (int k = 0; k < K; k++) acc = fmaf(Ri[k], xm[k], acc);",
     "for (int k = K - 1; k >= 0; k--) acc = fmaf(Ri[k], xm[k], acc);", [P.pin_rotation_fixture]),
    ("rot_skipped", "for (int k = 0; k < K; k++) acc = fmaf(Ri[k], xm[k], acc);",
     "acc = xm[i] + 0.0f * Ri[0];", [P.pin_rotation_fixture, P.pin_rotation_properties]),
    ("f16_round_truncate", "double q = rint(ldexp(a, 10 - E));", "double q = floor(ldexp(a, 10 - E));",
     [P.pin_f64_to_f16]),
]


@pytest.mark.parametrize("name,old,new,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, pins, tmp_path):
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"snippet for {name} not found exactly once"
    mutant_c = tmp_path / "qmm_oracle.c"
    mutant_c.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutant_c), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failures = 0
    for pin in pins:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            failures += 1
    assert failures > 0, f"planted mistake {name} passed every pin"
    assert os.path.getsize(oracle.SRC) == len(src.encode())
