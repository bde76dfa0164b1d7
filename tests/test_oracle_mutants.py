"""The oracle's pins have teeth: plant one plausible mistake at a time in a copy
of the oracle's C source, build it, run the pin suite against that copy and
require it to fail.  Everything here runs on the CPU; the shipped oracle
source is never modified.
"""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "chord_oracle.c")

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("offset_7", "float d = (float)((int)q - 8);", "float d = (float)((int)q - 7);"),
    ("scale_then_subtract", "float p = d * f32_from_bf16(s);",
     "float p = (float)q * f32_from_bf16(s) - 8.0f * f32_from_bf16(s);"),
    ("ties_away", "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))", "if (rest >= 0x8000u)"),
    ("nibble_order", "int i = kpart * 2 + lower + 4 * odd;", "int i = kpart + 2 * lower + 4 * odd;"),
    ("nibble_order_layout2", "int i = (m % 2) * 4 + m / 2;", "int i = m;"),
    ("scale_half_layout2", "+ 4096u + (size_t)r * 4u\n               + (size_t)h * 2u;",
     "+ 4096u + (size_t)r * 4u\n               + (size_t)(1 - h) * 2u;"),
    ("scale_slot", "+ (size_t)(h * 8 + g) * 4u + (size_t)lower * 2u;", "+ (size_t)(g * 2 + h) * 4u + (size_t)lower * 2u;"),
    ("align_descending", "for (int64_t p = 0; p < P; ++p)\n            if (topk_ids[p] == e)",
     "for (int64_t p = P - 1; p >= 0; --p)\n            if (topk_ids[p] == e)"),
    ("gemm_k_shift", "                    acc += f32_from_bf16(a[k]) * w[k];",
     "                    acc += f32_from_bf16(a[k]) * w[(k + 1) % K];"),
    ("grouped_k_shift", "\n                acc += f32_from_bf16(a[k]) * w[k];",
     "\n                acc += f32_from_bf16(a[k]) * w[(k + 1) % K];"),
    ("gemm_row_mod", "const uint16_t *a = A + (size_t)(p / a_row_divisor) * (size_t)K;",
     "const uint16_t *a = A + (size_t)(p % a_row_divisor) * (size_t)K;"),
    ("gemm_group_64", "uint16_t s = scales[((size_t)e * N + n) * G + k / ORC_GROUP];",
     "uint16_t s = scales[((size_t)e * N + n) * G + k / 64];"),
    ("f32_output_rounded", "Cf[(size_t)p * N + n] = acc;",
     "Cf[(size_t)p * N + n] = f32_from_bf16(bf16_from_f32(acc));"),
    ("layer_rounds_down", "rc = orc_combine_f32(C2, topk_ids, topk_w, T, topk, E, H, out, nthreads);",
     "for (int64_t i = 0; i < P * H; ++i) C2[i] = f32_from_bf16(bf16_from_f32(C2[i]));\n"
     "    rc = orc_combine_f32(C2, topk_ids, topk_w, T, topk, E, H, out, nthreads);"),
    ("silu_sign", "float s = g / (1.0f + expf(-g));", "float s = g / (1.0f + expf(g));"),
    ("gate_up_swap", "float g = f32_from_bf16(C1[(size_t)p * 2 * I + j]);",
     "float g = f32_from_bf16(C1[(size_t)p * 2 * I + I + j]);"),
    ("interleave_up_first", "return 16 * (m / 8) + 8 + m % 8;", "return 16 * (m / 8) + m % 8 - 8 * (m % 8 > 7);"),
    ("interleave_by_16", "return 16 * (n / 8) + n % 8;", "return 16 * (n / 16) + n % 16;"),
    ("contiguous_takes_padding", "if (m_indices[m] == e)\n                rows[nr++] = m;",
     "if (m_indices[m] == e || m_indices[m] == -1)\n                rows[nr++] = m;"),
    ("masked_row_stride", "rows[r] = (int64_t)g * max_m + r;", "rows[r] = (int64_t)g * masked_m[g] + r;"),
    ("scale_range_half_included", "if (sign != 0 || expo < 1 || expo > 125)", "if (sign != 0 || expo < 1 || expo > 126)"),
    ("scale_range_subnormal_included", "if (sign != 0 || expo < 1 || expo > 125)", "if (sign != 0 || expo > 125)"),
    ("scale_range_sign_ignored", "if (sign != 0 || expo < 1 || expo > 125)", "if (expo < 1 || expo > 125)"),
    ("f64sum_binary32_accumulator", "double dacc = 0.0;", "float dacc = 0.0f;"),
    ("f64_rounds_through_binary32", "        if (r != 0.0) {\n            uint32_t keep", "        if (0) {\n            uint32_t keep"),
    ("f64_layer_rounds_down_sums", "rc = orc_combine_f64(C2, topk_ids, topk_w, T, topk, E, H, out, nthreads);",
     "for (int64_t i = 0; i < P * H; ++i) C2[i] = (double)(float)C2[i];\n"
     "    rc = orc_combine_f64(C2, topk_ids, topk_w, T, topk, E, H, out, nthreads);"),
    ("combine_nonlocal", "if (topk_ids[p] < 0 || topk_ids[p] >= E)\n                    continue;\n                float v",
     "if (topk_ids[p] >= E)\n                    continue;\n                float v"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    sys.path.insert(0, ROOT)
    import oracle
    subprocess.check_call(["gcc", *oracle.CFLAGS, str(msrc), "-o", str(so), "-lm"])
    env = dict(os.environ, CHORD_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
