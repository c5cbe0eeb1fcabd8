"""The oracle pins must catch plausible mistakes.

Each case plants one mistake in a private copy of oracle/oracle.c (a dropped
term, a wrong sign or index, a transposed operand, the wrong rounding),
builds it on the CPU, and runs the pin suite against that build in a child
process: at least one pin must fail.  The real oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

ORACLE_SRC = os.path.join(ROOT, "oracle", "oracle.c")
sys.path.insert(0, ROOT)
from oracle import build as oracle_build  # noqa: E402

MUTATIONS = {
    "gemm_zero_point_sign": ("((int64_t)uA[i * K + k] - (int64_t)zeroA[i])",
                             "((int64_t)uA[i * K + k] + (int64_t)zeroA[i])"),
    "gemm_scaleA_by_column": ("val = val * scaleA[i];", "val = val * scaleA[j % M];"),
    "gemm_bias_dropped": ("if (bias) val = val + bias[j];", "(void)bias;"),
    "gemm_B_transposed": ("* (int64_t)iB[k * N + j];", "* (int64_t)iB[(j * K + k) % (K * N)];"),
    "gemm_scales_not_applied_in_order": ("val = val * scaleB[j];", "val = val / scaleB[j];"),
    "round_half_away": ("double r = (double)rintf(v) + (double)zp;", "double r = (double)roundf(v) + (double)zp;"),
    "quantize_zero_point_dropped": ("store_q(y, ytype, i, sat_rint_plus(q, zp, lo, hi));",
                                    "store_q(y, ytype, i, sat_rint_plus(q, 0, lo, hi));"),
    "quantize_axis_index_shifted": ("      int64_t c = per_axis ? a : 0;\n      float s = y_scale[c];",
                                    "      int64_t c = per_axis ? (a + 1) % axis_len : 0;\n      float s = y_scale[c];"),
    "dequantize_zero_point_sign": ("float d = (float)(load_q(x, xtype, i) - zp);",
                                   "float d = (float)(load_q(x, xtype, i) + zp);"),
    "row_zero_from_max": ("z = sat_rint_plus(-mn / s, 0, 0, 255);", "z = sat_rint_plus(mx / s, 0, 0, 255);"),
    "narrow_range_64": ("const int64_t qmax = avoid_overflow ? 63 : 127;",
                        "const int64_t qmax = avoid_overflow ? 64 : 127;"),
    "conv_pad_reads_code_zero": ("if (iw < 0 || iw >= W) continue;",
                                 "if (iw < 0 || iw >= W) { acc += (0 - (int64_t)x_zero_point) * "
                                 "(load_q(w, wtype, ((m * Cg + cc) * kH + kh) * kW + kw) - wz); continue; }"),
    "conv_requant_multiplies_y_scale": ("v = v / y_scale;", "v = v * y_scale;"),
    "conv_bias_dropped": ("if (B) acc += B[m];", "(void)B;"),
    "conv_weight_zero_point_per_tensor": ("const int64_t wz = w_zero_point[per_channel ? m : 0];",
                                          "const int64_t wz = w_zero_point[0];"),
    "lstm_gates_o_f_swapped": ("float fg = input_forget ? 1.0f - ig : sigmoid_f32(g[2]);",
                               "float fg = input_forget ? 1.0f - ig : sigmoid_f32(g[1]);"),
    "lstm_peephole_o_uses_old_cell": ("if (P) vo = vo + P[H + u] * c;", "if (P) vo = vo + P[H + u] * cp;"),
    "lstm_coupled_gate_is_i": ("float fg = input_forget ? 1.0f - ig : sigmoid_f32(g[2]);",
                               "float fg = input_forget ? ig : sigmoid_f32(g[2]);"),
    "lstm_clip_skips_candidate": ("        if (q != 1) {\n          if (Wb) v = v + Wb[n];\n          if (Rb) v = v + Rb[n];\n          if (clip > 0.0f)",
                                  "        if (q != 1) {\n          if (Wb) v = v + Wb[n];\n          if (Rb) v = v + Rb[n];\n          if (clip > 0.0f && q != 3)"),
    "zp_product_zero_point_per_tensor": ("const int64_t zb = zeroB ? zeroB[n_zb == N ? j : 0] : 0;",
                                         "const int64_t zb = zeroB ? zeroB[0] : 0;"),
    "lstm_recurrent_bias_dropped": ("if (Rb) v = v + Rb[n];", "(void)Rb;"),
    "bf16_truncates": ("u += 0x7fffu + lsb;", "(void)lsb;"),
    "qgemm_b_zero_point_per_tensor": ("const int64_t bz = b_zero_point ? b_zero_point[n_b == N ? j : 0] : 0;",
                                      "const int64_t bz = b_zero_point ? b_zero_point[0] : 0;"),
    "qgemm_transB_ignored": ("const int64_t bv = load_q(B, btype, transB ? j * K + k : k * N + j);",
                             "const int64_t bv = load_q(B, btype, k * N + j);"),
    "qgemm_C_broadcast_rows": ("if (C) acc += C[(c_rows == 1 ? 0 : i) * c_cols + (c_cols == 1 ? 0 : j)];",
                               "if (C) acc += C[(c_cols == 1 ? 0 : j)];"),
    "qgemm_alpha_dropped": ("float mul = alpha * a_scale;", "float mul = a_scale;"),
    "mitf_a_zero_point_per_tensor": ("const int64_t az = a_zero_point ? a_zero_point[pa] : 0;",
                                     "const int64_t az = a_zero_point ? a_zero_point[0] : 0;"),
    "mitf_bias_dropped": ("if (bias) v = v + bias[j];", "(void)bias;"),
    "mitf_scale_by_row_of_b": ("float mul = a_scale[pa] * b_scale[pb];", "float mul = a_scale[pa] * b_scale[0];"),
    "bcast_index_reversed": ("    if (sh[d] != 1) off += idx * stride;", "    if (sh[d] != 1) off += (sh[d] - 1 - idx) * stride;"),
    "qadd_b_scale_on_a": ("float fb = b_scale * (float)b;", "float fb = a_scale * (float)b;"),
    "qmul_divides_by_scale_product": ("v = (float)(a * b) * m;", "v = (float)(a * b) / m;"),
    "leaky_alpha_on_positive": ("f = d < 0.0f ? alpha * d : d;", "f = d > 0.0f ? alpha * d : d;"),
    "mul_integer_zero_point_b_dropped": ("const int64_t b = load_q(B, btype, bcast_offset(i, out_shape, b_shape, rank)) - b_zp;",
                                         "const int64_t b = load_q(B, btype, bcast_offset(i, out_shape, b_shape, rank));"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(ORACLE_SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", *oracle_build.CFLAGS, str(mutant), "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB_UNDER_TEST=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin failed for planted mistake {name}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
