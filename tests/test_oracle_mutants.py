"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Every mutant below is a plausible slip in the oracle (a swapped nibble, a
wrong index, a dropped term, a transposed operand, a sign, a rounding rule).
The test compiles an altered copy of the oracle source into a temporary
directory, runs the pin suite against it in a child process and expects the
suite to fail.  The committed oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = {
    "code_nibble_order": ("return (k % 2 == 0) ? (byte & 0x0f) : (byte >> 4);\n}\n\n/* Zero point",
                          "return (k % 2 == 1) ? (byte & 0x0f) : (byte >> 4);\n}\n\n/* Zero point"),
    "zero_nibble_order": ("return (b % 2 == 0) ? (byte & 0x0f) : (byte >> 4);",
                          "return (b % 2 == 1) ? (byte & 0x0f) : (byte >> 4);"),
    "zero_row_pitch": ("int64_t row_bytes = (nb + 1) / 2;", "int64_t row_bytes = nb / 2 + 1;"),
    "group_index": ("int64_t b = k / g;", "int64_t b = (k / g) % 2;"),
    "scale_row": ("return orc_f16_to_f32(scales[n * nb + b]);", "return orc_f16_to_f32(scales[b]);"),
    "sign": ("return (float)(q - z) * s;", "return (float)(z - q) * s;"),
    "symmetric_zero": ("        return 8;", "        return 7;"),
    "dropped_last_term": ("double p = w * (double)x[m * K + k];",
                          "double p = (k == K - 1) ? 0.0 : w * (double)x[m * K + k];"),
    "x_transposed": ("double p = w * (double)x[m * K + k];", "double p = w * (double)x[k * M + m];"),
    "f16_bias": ("v = ldexp((double)(1024 + frac), expo - 25);",
                 "v = ldexp((double)(1024 + frac), expo - 24);"),
    "f16_subnormal": ("v = ldexp((double)frac, -24);", "v = ldexp((double)frac, -25);"),
    "bf16_ties_away": ("(dropped == 0x8000u && (kept & 1u))", "(dropped == 0x8000u)"),
    "gemm_widen": ("double p = w * (double)orc_bf16_to_f32(a_bf16[m * K + k]);",
                   "double p = w * (double)orc_bf16_to_f32(a_bf16[m * K + k] & 0xfffe);"),
    "bound_signed": ("                mag += fabs(p);\n            }\n            y[m * N + n] = (float)acc;",
                     "                mag += p;\n            }\n            y[m * N + n] = (float)acc;"),
    "f32_control_index": ("double p = (double)W[n * K + k] * (double)x[m * K + k];",
                          "double p = (double)W[k * N + n] * (double)x[m * K + k];"),
    "rmsnorm_no_eps": ("double rms = sqrt(ss / (double)K + eps);", "double rms = sqrt(ss / (double)K);"),
    "rmsnorm_mean_over_k_minus_1": ("double rms = sqrt(ss / (double)K + eps);",
                                    "double rms = sqrt(ss / (double)(K - 1) + eps);"),
    "rmsnorm_gamma_index": ("/ rms * (double)gamma[k];", "/ rms * (double)gamma[K - 1 - k];"),
    "silu_sign": ("return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    "swiglu_swapped": ("out[i] = orc_silu(gate[i]) * up[i];", "out[i] = orc_silu(up[i]) * gate[i];"),
    "gemv_f64_dropped_first_term": ("double p = w * x[m * K + k];",
                                    "double p = (k == 0) ? 0.0 : w * x[m * K + k];"),
    "q40_scale_byte_order": ("uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));",
                             "uint16_t dbits = (uint16_t)(blk[1] | (blk[0] << 8));"),
    "q40_nibble_order": ("int q = (e % 2 == 0) ? (byte & 0x0f) : (byte >> 4);",
                         "int q = (e % 2 == 1) ? (byte & 0x0f) : (byte >> 4);"),
    "q40_block_pitch": ("const uint8_t *blk = blocks + (n * (K / 32) + k / 32) * 18;",
                        "const uint8_t *blk = blocks + (n * (K / 32) + k / 32) * 16;"),
    "gemm_a_transposed": ("double p = w * (double)orc_bf16_to_f32(a_bf16[m * K + k]);",
                          "double p = w * (double)orc_bf16_to_f32(a_bf16[k * M + m]);"),
    "gemm_dropped_last_term": ("                double p = w * (double)orc_bf16_to_f32(a_bf16[m * K + k]);",
                               "                double p = (k == K - 1) ? 0.0 : w * (double)orc_bf16_to_f32(a_bf16[m * K + k]);"),
    "gemm_output_transposed": ("            c[m * N + n] = (float)acc;", "            c[n * M + m] = (float)acc;"),
    "dequant_bf16_transposed": ("            wb[n * K + k] = orc_f32_to_bf16(", "            wb[k * N + n] = orc_f32_to_bf16("),
    "f32_control_bound_of_w": ("                double p = (double)W[n * K + k] * (double)x[m * K + k];\n                acc += p;\n                mag += fabs(p);",
                               "                double p = (double)W[n * K + k] * (double)x[m * K + k];\n                acc += p;\n                mag += fabs((double)W[n * K + k]);"),
    "probe_sum_skips_last": ("    for (int64_t i = 0; i < n; ++i)\n        acc += (double)buf[i];",
                             "    for (int64_t i = 0; i + 1 < n; ++i)\n        acc += (double)buf[i];"),
    "f16_inf_as_nan": ("        v = frac ? NAN : INFINITY;", "        v = NAN;"),
    "f16_sign_dropped": ("    return (float)(sign ? -v : v);", "    return (float)v;"),
    "bf16_widen_shift": ("    uint32_t u = (uint32_t)b << 16;", "    uint32_t u = (uint32_t)b << 15;"),
    "bf16_round_down_always": ("    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))",
                               "    if (0)"),
    "bf16_nan_not_quiet": ("        return (uint16_t)((u >> 16) | 0x0040u);", "        return (uint16_t)(u >> 16);"),
    "rmsnorm_sum_of_abs": ("            ss += v * v;", "            ss += fabs(v);"),
    "rmsnorm_no_sqrt": ("double rms = sqrt(ss / (double)K + eps);", "double rms = ss / (double)K + eps;"),
    "gemv_f64_bound_signed": ("                double p = w * x[m * K + k];\n                acc += p;\n                mag += fabs(p);",
                              "                double p = w * x[m * K + k];\n                acc += p;\n                mag += p;"),
    "q40_zero_point": ("    return (float)(q - 8) * orc_f16_to_f32(dbits);", "    return (float)(q - 7) * orc_f16_to_f32(dbits);"),
    "q80_unsigned_codes": ("    if (q >= 128)\n        q -= 256;\n", "\n"),
    "q80_block_pitch": ("const uint8_t *blk = blocks + (n * (K / 32) + k / 32) * 34;",
                        "const uint8_t *blk = blocks + (n * (K / 32) + k / 32) * 32;"),
    "q80_code_offset": ("int q = blk[2 + k % 32];", "int q = blk[1 + k % 32];"),
    "q80_scale_byte_order": ("uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));\n    int q = blk",
                             "uint16_t dbits = (uint16_t)(blk[1] | (blk[0] << 8));\n    int q = blk"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "q4_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mutant.c"
    c_path.write_text(mutated)
    so_path = str(tmp_path / "libmutant.so")
    oracle.build(force=True, src=str(c_path), out=so_path)
    env = dict(os.environ, Q4_ORACLE_LIB=so_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


# Plausible slips in the Python layer of the oracle (row-subset offsets, the SwiGLU
# pairing and tolerance).  The mutated source is executed over the real module's
# namespace by a plugin loaded before the pin suite is collected.
PY_MUTANTS = {
    "rows_zero_pitch": ("                          None if zeros is None else _ptr(zeros, _u8p, n * zrow),\n"
                        "                          _ptr(x, _f32p), M, 1, K, g, _ptr(yr, _f32p), _ptr(br, _f64p))",
                        "                          None if zeros is None else _ptr(zeros, _u8p, n * (nb // 2)),\n"
                        "                          _ptr(x, _f32p), M, 1, K, g, _ptr(yr, _f32p), _ptr(br, _f64p))"),
    "gemm_rows_a_offset": ("_ptr(a_bf16, _u16p, int(m) * K), 1, 1, K, g,", "_ptr(a_bf16, _u16p, int(m) * (K // 2)), 1, 1, K, g,"),
    "f32_rows_offset": ("lib().orc_f32_gemv(_ptr(W, _f32p, int(n) * K), _ptr(x, _f32p), M, 1, K,",
                        "lib().orc_f32_gemv(_ptr(W, _f32p, int(n) * (K - 1)), _ptr(x, _f32p), M, 1, K,"),
    "fused_pairs_swapped": ("        rows += [2 * i, 2 * i + 1]", "        rows += [2 * i + 1, 2 * i]"),
    "fused_bound_drops_up_error": ("    bound = (SILU_SLOPE_MAX * bg * (np.abs(up) + bu) + (sg + SILU_SLOPE_MAX * bg) * bu",
                                   "    bound = (SILU_SLOPE_MAX * bg * (np.abs(up) + bu) + 0 * bu"),
    "fused_bound_drops_gate_error": ("    bound = (SILU_SLOPE_MAX * bg * (np.abs(up) + bu) + (sg + SILU_SLOPE_MAX * bg) * bu",
                                     "    bound = ((sg + SILU_SLOPE_MAX * bg) * bu"),
    "silu_slope_too_small": ("SILU_SLOPE_MAX = 1.1 ", "SILU_SLOPE_MAX = 1.0 "),
    "q40_rows_pitch": ("    row_bytes = (K // 32) * 18", "    row_bytes = (K // 32) * 16"),
    "q80_rows_pitch": ("    row_bytes = (K // 32) * 34", "    row_bytes = (K // 32) * 32"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_planted_mistake_in_the_python_layer_is_caught(name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    old, new = PY_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found"
    mutated = tmp_path / "mutated_oracle_source.py"
    mutated.write_text(src.replace(old, new))
    (tmp_path / "oracle_mutation_plugin.py").write_text(
        "import sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import oracle\n"
        f"exec(compile(open({str(mutated)!r}).read(), oracle.__file__, 'exec'), oracle.__dict__)\n")
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([str(tmp_path), os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-p", "oracle_mutation_plugin", os.path.join(HERE, "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert "passed" in r.stdout or "failed" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
