"""Plant plausible mistakes in copies of the oracle and check that the pins catch
each one (no GPU).  A mistake is a textual edit of ``oracle/oracle.c``; the
edited copy is compiled into a temporary library and run against every pin.
"""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, replacement).  Each original must occur exactly once.
MUTATIONS = [
    # routed experts
    ("moe_first_expert_only", "const uint8_t *we = (id >= 0 && id < n_experts) ? (const uint8_t *)w[id] : NULL;",
     "const uint8_t *we = (id >= 0 && id < n_experts) ? (const uint8_t *)w[0] : NULL;"),
    ("moe_shared_x_always", "const size_t xo = (size_t)r * x_slot_stride;", "const size_t xo = 0 * x_slot_stride;"),
    ("moe_bad_id_zero", "if (we == NULL) {\n            for (size_t k = 0; k < out_n; ++k)\n                yr[k] = mr[k] = NAN;",
     "if (we == NULL) {\n            for (size_t k = 0; k < out_n; ++k)\n                yr[k] = mr[k] = 0.0;"),
    # fmt=4
    ("i4g_swapped_nibbles", "(i % 2 == 0) ? (byte & 0xF) : (byte >> 4);\n    return nib - 8;",
     "(i % 2 == 0) ? (byte >> 4) : (byte & 0xF);\n    return nib - 8;"),
    ("i4g_no_offset", "return nib - 8;", "return nib;"),
    ("i4g_group_off_by_one",
     "double sc = (double)scales[(size_t)o * ng + (size_t)(i / gs)];\n                double t = q * sc * (double)x",
     "double sc = (double)scales[(size_t)o * ng + (size_t)(i / gs > 0 ? i / gs - 1 : 0)];\n"
     "                double t = q * sc * (double)x"),
    ("i4g_scale_1pct", "double t = q * sc * (double)x", "double t = q * (sc * 1.01) * (double)x"),
    ("i4g_row_bytes_I_over_2", "size_t rb = ((size_t)I + 1) / 2;\n    size_t ng = ((size_t)I + (size_t)gs - 1) / (size_t)gs;\n    for (int s = 0; s < S; ++s) {\n        for (int o = 0; o < O; ++o) {\n            double acc = 0.0, m = 0.0;\n            for (int i = 0; i < I; ++i) {\n                double q = (double)i4g_value(w, rb, o, i);\n                double sc = (double)scales[(size_t)o * ng + (size_t)(i / gs)];\n                double t = q * sc * (double)x",
     "size_t rb = ((size_t)I) / 2;\n    size_t ng = ((size_t)I + (size_t)gs - 1) / (size_t)gs;\n    for (int s = 0; s < S; ++s) {\n        for (int o = 0; o < O; ++o) {\n            double acc = 0.0, m = 0.0;\n            for (int i = 0; i < I; ++i) {\n                double q = (double)i4g_value(w, rb, o, i);\n                double sc = (double)scales[(size_t)o * ng + (size_t)(i / gs)];\n                double t = q * sc * (double)x"),
    ("i4g_mag_signed", "acc += t;\n                m += fabs(t);\n            }\n            y[(size_t)s * O + o] = acc;\n            mag[(size_t)s * O + o] = m;\n        }\n    }\n}\n\n/* Batched",
     "acc += t;\n                m += t;\n            }\n            y[(size_t)s * O + o] = acc;\n            mag[(size_t)s * O + o] = m;\n        }\n    }\n}\n\n/* Batched"),
    ("i4g_gemm_mag_signed",
     "double t = q * sc * oracle_bf16_value(X[(size_t)s * I + i]);\n                acc += t;\n                m += fabs(t);",
     "double t = q * sc * oracle_bf16_value(X[(size_t)s * I + i]);\n                acc += t;\n                m += t;"),
    ("i4g_gemm_mag_x1000",
     "double t = q * sc * oracle_bf16_value(X[(size_t)s * I + i]);\n                acc += t;\n                m += fabs(t);",
     "double t = q * sc * oracle_bf16_value(X[(size_t)s * I + i]);\n                acc += t;\n                m += 1000.0 * fabs(t);"),
    ("i4g_gemm_group_off_by_one",
     "double sc = (double)scales[(size_t)o * ng + (size_t)(i / gs)];\n                double t = q * sc * oracle_bf16_value",
     "double sc = (double)scales[(size_t)o * ng + (size_t)(i / gs > 0 ? i / gs - 1 : 0)];\n"
     "                double t = q * sc * oracle_bf16_value"),
    ("moe_gemm_mag_rows_from_zero", "double *mg = mag + (size_t)off[g] * O;", "double *mg = mag;"),
    ("fp8_mag_signed",
     "double sc = (double)scale_inv[(size_t)(o / 128) * nbi + (size_t)(i / 128)];\n                double t = wv * sc * oracle_bf16_value(x[(size_t)s * I + i]);\n                acc += t;\n                m += fabs(t);",
     "double sc = (double)scale_inv[(size_t)(o / 128) * nbi + (size_t)(i / 128)];\n                double t = wv * sc * oracle_bf16_value(x[(size_t)s * I + i]);\n                acc += t;\n                m += t;"),
    ("fp8ue8m0_mag_x2",
     "double sc = oracle_e8m0_value(scale_e8m0[(size_t)(o / 128) * nbi + (size_t)(i / 128)]);\n                double t = wv * sc * oracle_bf16_value(x[(size_t)s * I + i]);\n                acc += t;\n                m += fabs(t);",
     "double sc = oracle_e8m0_value(scale_e8m0[(size_t)(o / 128) * nbi + (size_t)(i / 128)]);\n                double t = wv * sc * oracle_bf16_value(x[(size_t)s * I + i]);\n                acc += t;\n                m += 2.0 * fabs(t);"),
    ("q2_0_mag_signed", "i % 64) *\n                           oracle_bf16_value(x[(size_t)s * I + i]);\n                acc += t;\n                m += fabs(t);",
     "i % 64) *\n                           oracle_bf16_value(x[(size_t)s * I + i]);\n                acc += t;\n                m += t;"),
    ("mq4v2_mag_signed", "                    acc += t;\n                    m += fabs(t);", "                    acc += t;\n                    m += t;"),
    ("mq4_one_header_mag_signed", "sum_abs += fabs(t);", "sum_abs += t;"),
    ("quant_divisor_8", "volatile float sc = amax / 7.0f;", "volatile float sc = amax / 8.0f;"),
    ("quant_truncate", "float qr = rintf(r);\n                    if (qr < -8.0f)", "float qr = truncf(r);\n                    if (qr < -8.0f)"),
    # E4M3
    ("e4m3_bias_8", "v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3_all_e15_nan", "if (e == 15 && m == 7)\n        return NAN;", "if (e == 15)\n        return NAN;"),
    ("e4m3_no_nan", "if (e == 15 && m == 7)\n        return NAN;", "if (e == 16)\n        return NAN;"),
    ("e4m3_subnormal_exp", "v = ldexp((double)m / 8.0, 1 - 7);", "v = ldexp((double)m / 8.0, -7);"),
    ("e4m3_sign_dropped", "    return s ? -v : v;\n}\n\n/* IEEE 754 binary16", "    (void)s; return v;\n}\n\n/* IEEE 754 binary16"),
    # fmt=7
    ("fp8_block_transposed",
     "double sc = (double)scale_inv[(size_t)(o / 128) * nbi + (size_t)(i / 128)];",
     "double sc = (double)scale_inv[((size_t)(i / 128) * nbi + (size_t)(o / 128)) % (nbi * (((size_t)O + 127) / 128))];"),
    ("fp8_divide_scale",
     "double sc = (double)scale_inv[(size_t)(o / 128) * nbi + (size_t)(i / 128)];\n                double t = wv * sc",
     "double sc = (double)scale_inv[(size_t)(o / 128) * nbi + (size_t)(i / 128)];\n                double t = wv / sc"),
    ("fp8_block_64", "double sc = (double)scale_inv[(size_t)(o / 128) * nbi + (size_t)(i / 128)];",
     "double sc = (double)scale_inv[((size_t)(o / 128) * nbi + (size_t)(i / 64)) % (nbi * (((size_t)O + 127) / 128))];"),
    ("moe_gemm_rows_from_zero", "const uint16_t *xg = X + (size_t)off[g] * I;", "const uint16_t *xg = X;"),
    ("moe_gemm_expert_of_slot", "const int e = group_expert[g];", "const int e = group_expert[0];"),
    # Q2_0
    ("q2_0_no_offset", "    return (double)(code - 1) * d;\n}", "    return (double)code * d;\n}"),
    ("q2_0_shift_k", "int code = (block[2 + e / 4] >> (2 * (e % 4))) & 3;", "int code = (block[2 + e / 4] >> (e % 4)) & 3;"),
    ("q2_0_byte_transposed", "int code = (block[2 + e / 4] >> (2 * (e % 4))) & 3;",
     "int code = (block[2 + (e % 16)] >> (2 * (e / 16))) & 3;"),
    ("q2_0_stride_16", "double t = oracle_q2_0_weight(blocks + ((size_t)o * nb + (size_t)(i / 64)) * 18, i % 64) *",
     "double t = oracle_q2_0_weight(blocks + ((size_t)o * nb + (size_t)(i / 64)) * 16, i % 64) *"),
    ("q2_0_encoder_steps_8", "volatile float frac = 0.5f + (float)k / 16.0f;", "volatile float frac = 0.5f + (float)k / 8.0f;"),
    # UE8M0 scales
    ("e8m0_bias_126", "return ldexp(1.0, (int)e - 127);", "return ldexp(1.0, (int)e - 126);"),
    ("e8m0_no_nan", "    if (e == 255)\n        return NAN;\n    return ldexp", "    if (e == 256)\n        return NAN;\n    return ldexp"),
    ("fp8ue8m0_block_transposed",
     "double sc = oracle_e8m0_value(scale_e8m0[(size_t)(o / 128) * nbi + (size_t)(i / 128)]);",
     "double sc = oracle_e8m0_value(scale_e8m0[((size_t)(i / 128) * nbi + (size_t)(o / 128)) % (nbi * (((size_t)O + 127) / 128))]);"),
    # f16 / bf16
    ("f16_truncate", "double frac = rint((a / ldexp(1.0, e) - 1.0) * 1024.0);",
     "double frac = floor((a / ldexp(1.0, e) - 1.0) * 1024.0);"),
    ("f16_bias_14", "v = ldexp(1.0 + (double)f / 1024.0, e - 15);", "v = ldexp(1.0 + (double)f / 1024.0, e - 14);"),
    ("f16_subnormal_scale", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("bf16_shift", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    # MQ4-V2
    ("mq4_half_from_lane", "int h = byte_off >= 64 ? 1 : 0;", "int h = byte_off >= 32 ? 1 : 0;"),
    ("mq4_header_fields_swapped",
     "double sc = oracle_f16_value((uint16_t)(hd & 0xFFFFu));\n    double z = oracle_f16_value((uint16_t)(hd >> 16));",
     "double sc = oracle_f16_value((uint16_t)(hd >> 16));\n    double z = oracle_f16_value((uint16_t)(hd & 0xFFFFu));"),
    ("mq4_payload_plus4", "uint8_t byte = block[8 + byte_off];", "uint8_t byte = block[4 + byte_off];"),
    ("mq4_stride_132", "const uint8_t *blk = blocks + ((size_t)o * nb + b) * 136;",
     "const uint8_t *blk = blocks + ((size_t)o * nb + b) * 132;"),
    ("mq4_nibble_order", "int q = (j % 2 == 0) ? (byte & 0xF) : (byte >> 4);\n    return (double)q * sc + z;",
     "int q = (j % 2 == 0) ? (byte >> 4) : (byte & 0xF);\n    return (double)q * sc + z;"),
    ("mq4_enc_no_roundtrip", "float st = (float)oracle_f16_value(sc16);", "float st = step;"),
    ("mq4_enc_step_16", "volatile float step = diff / 15.0f;", "volatile float step = diff / 16.0f;"),
    ("mq4_enc_truncate", "float qr = rintf(r);\n                        if (qr < 0.0f)",
     "float qr = truncf(r);\n                        if (qr < 0.0f)"),
    # MQ4 v1 / MQ4C pad
    ("mq4v1_fields_swapped", "double scale = f32_at(block);\n    double zero = f32_at(block + 4);",
     "double scale = f32_at(block + 4);\n    double zero = f32_at(block);"),
    ("mq4c_reads_pad_as_zero", "double zero = oracle_f16_value((uint16_t)(pair >> 16));",
     "double zero = oracle_f16_value((uint16_t)(le32(block + 4) & 0xFFFFu));"),
    ("mq4_one_header_payload_plus4", "const uint8_t *payload = block + 8;", "const uint8_t *payload = block + 4;"),
    ("mq4_one_header_stride_132", "double t = weight(row + (size_t)(i / 256) * 136, i % 256) *",
     "double t = weight(row + (size_t)(i / 256) * 132, i % 256) *"),
    ("mq4_one_header_nibble_order", "return (j & 1) ? (b >> 4) : (b & 0xF);", "return (j & 1) ? (b & 0xF) : (b >> 4);"),
    ("mq4v1_enc_fp16_roundtrip", "scale = (hi == lo) ? 0.0f : step;\n                zero = lo;",
     "scale = (hi == lo) ? 0.0f : (float)oracle_f16_value(oracle_f16_from_f32(step));\n                zero = lo;"),
    ("mq4c_enc_no_pad_zero", "word1 = 0u;", "word1 = word0;"),
    ("mq4_one_header_enc_step_16", "volatile float step = span / 15.0f;", "volatile float step = span / 16.0f;"),
    # FWHT
    ("fwht_norm_8", "out[b * 256 + (size_t)j] = (float)(v[j] / 16.0);",
     "out[b * 256 + (size_t)j] = (float)(v[j] / 8.0);"),
    ("fwht_no_signs", "v[j] = (double)signs[j] * (double)in[b * 256 + (size_t)j];",
     "v[j] = (double)in[b * 256 + (size_t)j];"),
    ("fwht_butterfly_sign", "                    v[j] = a + c;\n                    v[j + len] = a - c;\n                }\n            }\n        }\n        for (int j = 0; j < 256; ++j)\n            out[b * 256 + (size_t)j] = (float)(v[j] / 16.0);",
     "                    v[j] = a + c;\n                    v[j + len] = c - a;\n                }\n            }\n        }\n        for (int j = 0; j < 256; ++j)\n            out[b * 256 + (size_t)j] = (float)(v[j] / 16.0);"),
]


def _run_pins(lib):
    orc = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            failed.append((pin.__name__, type(e).__name__))
    return failed


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation {name}: anchor occurs {src.count(old)} times"
    mutant = tmp_path / f"{name}.c"
    mutant.write_text(src.replace(old, new))
    lib_path = str(tmp_path / f"lib{name}.so")
    subprocess.run(["gcc", *[f for f in oracle.CFLAGS if f != "-Werror"], "-o", lib_path,
                    str(mutant), "-lm"], check=True)
    failed = _run_pins(oracle.load(lib_path))
    assert failed, f"mutation {name} passed every pin"
