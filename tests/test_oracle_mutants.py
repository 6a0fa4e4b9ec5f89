"""Planted mistakes: each variant of oracle.c below carries one plausible
error (a wrong constant, sign, index, rounding mode or dropped term).  Every
variant is compiled on the side and must fail the oracle's pin tests; a
variant that passes would show a blind spot in the pins.

The mistakes are planted in a copy of the oracle on the CPU only."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

import pytest

import oracle

ROOT = Path(__file__).resolve().parent.parent
PIN_FILES = ["tests/test_oracle_qgz.py", "tests/test_oracle_next.py", "tests/test_oracle_sr.py",
             "tests/test_oracle_qwz.py", "tests/test_oracle_bf16.py",
             "tests/test_oracle_quant.py"]

MUTANTS = {
    "scale_wrong_divisor": ("float scale = m / fq;", "float scale = m / (fq + 1.0f);"),
    "inverse_wrong_numerator": ("float inv = fq / m;", "float inv = (fq + 1.0f) / m;"),
    "round_half_away": ("float r = rintf(t);", "float r = roundf(t);"),
    "absmax_without_abs": ("float a = fabsf(x[i]);", "float a = x[i];"),
    "zero_block_bound_at_flt_min": ("if (m < fq * FLT_MIN) {", "if (m < FLT_MIN) {"),
    "compensation_sign": ("c[i] = gi + se;", "c[i] = gi - se;"),
    "error_scale_dropped": ("float se = s * e[in0 + i];", "float se = e[in0 + i];"),
    "residual_sign": ("float resid = c[i] - d;", "float resid = d - c[i];"),
    "beta_on_new_error": ("float kept = beta * e[in0 + i];",
                          "float kept = one_minus_beta * e[in0 + i];"),
    "one_minus_beta_on_old_error": ("float added = one_minus_beta * resid;",
                                    "float added = beta * resid;"),
    "send_order_identity": ("return l * G + gq;", "return gq * L + l;"),
    "nibble_order_swapped": ("if ((pos & 1) == 0) *byte", "if ((pos & 1) == 1) *byte"),
    "reader_nibble_order": ("int v = (pos & 1) ? (codes[pos >> 1] >> 4) : (codes[pos >> 1] & 0xF);",
                            "int v = (pos & 1) ? (codes[pos >> 1] & 0xF) : (codes[pos >> 1] >> 4);"),
    "flat_reduce_transposed": ("int64_t pos = (int64_t)r * N + (int64_t)k * S + i;",
                               "int64_t pos = (int64_t)k * N + (int64_t)r * S + i;"),
    "out_scale_dropped": ("float v = acc * out_scale;", "float v = acc;"),
    "hop2_wrong_subslice": ("int64_t pos = unit * G * S + (int64_t)g * S + i;",
                            "int64_t pos = unit * G * S + (int64_t)gq * S + i;"),
    "hop2_wrong_unit": ("int64_t unit = (int64_t)gq * L + l;",
                        "int64_t unit = (int64_t)l * G + gq;"),
    "hop1_wrong_chunk": ("int64_t pos = r * N + ((int64_t)l * G + gq) * S + b0 + i;",
                         "int64_t pos = r * N + ((int64_t)gq * L + l) * S + b0 + i;"),
    "hop1_wrong_rank": ("int64_t r = (int64_t)g * L + lq;", "int64_t r = (int64_t)lq * G + g;"),
    "bf16_ties_away": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))",
                       "if (lower >= 0x8000u)"),
    "bf16_truncate_in_dequant": ("w_out[i] = orc_f32_to_bf16_rne(orc_dequant(codes[i], scales[i / B]));",
                                 "w_out[i] = (uint16_t)(f32_bits(orc_dequant(codes[i], scales[i / B])) >> 16);"),
    "int8_wrong_qmax": ("orc_quant_block(x, B, 127, codes + b0, &scales[b0 / B]);",
                        "orc_quant_block(x, B, 128, codes + b0, &scales[b0 / B]);"),
    "sr_biased_half_bits": ("return (uint16_t)((u + r) >> 16);", "return (uint16_t)((u + (r >> 1)) >> 16);"),
    "sr_src_not_zeroed": ("        src[i] = 0;\n", "\n"),
    "sr_sum_dropped_src": ("float sum = orc_bf16_to_f32(dst[i]) + orc_bf16_to_f32(src[i]);",
                           "float sum = orc_bf16_to_f32(dst[i]);"),
    "hop1_ef_residual_sign": ("float resid1 = part[i] - d1;", "float resid1 = d1 - part[i];"),
    "hop1_ef_scale_dropped": ("float se1 = s * e1[out0 + i];", "float se1 = e1[out0 + i];"),
    "hop1_ef_beta_swapped": ("float kept1 = beta * e1[out0 + i];",
                             "float kept1 = one_minus_beta * e1[out0 + i];"),
    "bf16ef_truncates": ("e16[in0 + i] = orc_f32_to_bf16_rne(kh + ah);",
                         "e16[in0 + i] = (uint16_t)(f32_bits(kh + ah) >> 16);"),
    "bf16ef_beta_swapped": ("float kh = beta * eh;", "float kh = omb * eh;"),
    "bf16ef_compensation_sign": ("c[i] = gh + seh;", "c[i] = gh - seh;"),
    "replica_skips_dequant": ("    orc_qwz_dequant_int8(codes, scales, replica, n, B);\n", "\n"),
    "fmix_constant": ("h *= 0x85EBCA6Bu;", "h *= 0x85EBCA6Cu;"),
    "fmix_shift": ("h ^= h >> 13;", "h ^= h >> 12;"),
    "flat_reduce_reversed": ("for (int r = 0; r < R; ++r) {\n                int64_t pos = (int64_t)r * N",
                             "for (int r = R - 1; r >= 0; --r) {\n                int64_t pos = (int64_t)r * N"),
    "hop2_reversed": ("for (int gq = 0; gq < G; ++gq) {\n                int64_t unit",
                      "for (int gq = G - 1; gq >= 0; --gq) {\n                int64_t unit"),
    "hop1_reversed": ("for (int lq = 0; lq < L; ++lq) {", "for (int lq = L - 1; lq >= 0; --lq) {"),
    "hop1_ef_compensation_sign": ("acc = acc + se1;", "acc = acc - se1;"),
    "bf16ef_scale_dropped": ("float seh = s * eh;", "float seh = eh;"),
    "bf16ef_residual_sign": ("float rh = c[i] - dh;", "float rh = dh - c[i];"),
    "nibble_read_unsigned": ("return v >= 8 ? v - 16 : v;", "return v;"),
    "nibble_sign_off_by_one": ("return v >= 8 ? v - 16 : v;", "return v >= 8 ? v - 15 : v;"),
    "int8ef_stored_with_qmax_7": ("orc_quant_block(en8, B, 127, e8 + in0, &e8s[in0 / B]);",
                                  "orc_quant_block(en8, B, 7, e8 + in0, &e8s[in0 / B]);"),
    "int8ef_scale_in_send_order": ("float es8 = e8s[in0 / B];", "float es8 = e8s[out0 / B];"),
    "int8ef_beta_swapped": ("float k8 = beta * ev8[i];", "float k8 = one_mb * ev8[i];"),
    "int8ef_compensation_sign": ("c8[i] = g8 + se8;", "c8[i] = g8 - se8;"),
    "ef_update_as_difference": ("float added = one_minus_beta * resid;",
                                "float added = resid - beta * resid;"),
    "compensation_fused": ("c[i] = gi + se;", "c[i] = fmaf(s, e[in0 + i], gi);"),
    "scale_by_reciprocal": ("float scale = m / fq;", "float scale = m * (1.0f / fq);"),
    "bf16ef_update_as_difference": ("float ah = omb * rh;", "float ah = rh - beta * rh;"),
    "bf16ef_compensation_fused": ("c[i] = gh + seh;", "c[i] = fmaf(s, eh, gh);"),
    "int8ef_update_as_difference": ("float a8 = one_mb * r8;", "float a8 = r8 - beta * r8;"),
    "int8ef_compensation_fused": ("c8[i] = g8 + se8;", "c8[i] = fmaf(s, ev8[i], g8);"),
    "hop1_ef_update_as_difference": ("float added1 = one_minus_beta * resid1;",
                                     "float added1 = resid1 - beta * resid1;"),
    "hop1_ef_compensation_fused": ("acc = acc + se1;", "acc = fmaf(s, e1[out0 + i], acc);"),
    "code_from_exact_product": ("float r = rintf(t);", "float r = (float)rint((double)x[i] * inv);"),
    "bf16_output_unscaled": ("float v = acc * out_scale;",
                             "float v = out_bf16 ? acc : acc * out_scale;"),
    "reduce_starts_at_negative_zero": ("float acc = 0.0f;\n        if (G == 1) {",
                                       "float acc = -0.0f;\n        if (G == 1) {"),
    "sr_compare_form": ("return (uint16_t)((u + r) >> 16);",
                        "return (uint16_t)((u >> 16) + ((u & 0xFFFFu) > r ? 1u : 0u));"),
    "sr_step_ignored": ("uint32_t key = orc_mix32(orc_mix32(seed) ^ step);",
                        "uint32_t key = orc_mix32(orc_mix32(seed));"),
}


def _run_mutant(name, tmp: Path):
    old, new = MUTANTS[name]
    src = oracle.SOURCE.read_text()
    assert src.count(old) == 1, f"{name}: anchor not found exactly once"
    mpath = tmp / f"{name}.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.build(mpath, tmp / f"lib{name}.so", extra=["-w"])
    # one thread per child: the children already run one per core
    env = dict(os.environ, ORACLE_LIB=str(lib), OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               OPENBLAS_NUM_THREADS="1")
    proc = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           *PIN_FILES], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=900)
    return name, proc.returncode, proc.stdout[-2000:]


def test_every_planted_mistake_is_caught(tmp_path):
    workers = max(1, min(len(MUTANTS), os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda n: _run_mutant(n, tmp_path), sorted(MUTANTS)))
    survived = [(n, out) for n, rc, out in results if rc == 0]
    broken = [(n, rc, out) for n, rc, out in results if rc in (2, 3, 4, 5)]
    assert not broken, broken
    assert not survived, "mutants passing every pin: " + ", ".join(n for n, _ in survived)
