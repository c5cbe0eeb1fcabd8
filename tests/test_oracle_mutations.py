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
    "lstm_gates_o_f_swapped": ("float fg = input_forget ? 1.0f - ig : F_(g[2]);",
                               "float fg = input_forget ? 1.0f - ig : F_(g[1]);"),
    "lstm_peephole_o_uses_old_cell": ("if (P) vo = vo + P[H + u] * c;", "if (P) vo = vo + P[H + u] * cp;"),
    "lstm_coupled_gate_is_i": ("float fg = input_forget ? 1.0f - ig : F_(g[2]);",
                               "float fg = input_forget ? ig : F_(g[2]);"),
    "exp_low_part_of_ln2_dropped": ("  r = fmaf(-nf, EF_LN2_LO, r);\n  float p", "  float p"),
    "exp_taylor_coefficient": ("p = fmaf(p, r, 0x1.111112p-7f);  /* 1/5! */", "p = fmaf(p, r, 0x1.555556p-5f);  /* 1/5! */"),
    "exp_scale_halves_wrong": ("const int n1 = n / 2, n2 = n - n1;\n  return", "const int n1 = n / 2, n2 = n1;\n  return"),
    "expm1_missing_2n_minus_1": ("return fmaf(t, q, t - 1.0f);", "return t * q;"),
    "log1p_range_step_dropped": ("return fmaf(k, EF_LN2_HI, l);", "return l;"),
    "tanh_large_argument_threshold": ("  if (a <= 9.5f) {", "  if (a <= 4.0f) {"),
    "tanh_quotient_denominator": ("? e : 2.0f) / (e + 2.0f);", "? e : 2.0f) / (e + 1.0f);"),
    "tanh_forms_swapped": ("t = a < 0.625f ? q : 1.0f - q;", "t = a < 0.625f ? 1.0f - q : q;"),
    "sigmoid_sign": ("static float ef_sigmoid(float x) { return 1.0f / (1.0f + ef_exp(-x)); }",
                     "static float ef_sigmoid(float x) { return 1.0f / (1.0f + ef_exp(x)); }"),
    "softplus_positive_branch": ("return x > 0.0f ? x + ef_log1p01(ef_exp(-x))", "return x > 0.0f ? ef_log1p01(ef_exp(-x))"),
    "lstm_candidate_uses_f": ("float ct = G_(g[3]);", "float ct = F_(g[3]);"),
    "lstm_output_uses_g": ("h_out[b * H + u] = og * H_(c);", "h_out[b * H + u] = og * G_(c);"),
    "activation_hard_sigmoid_unclamped": ("return v < 0.0f ? 0.0f : (v > 1.0f ? 1.0f : v);", "return v;"),
    "activation_thresholded_relu_at_zero": ("case OR_LA_THRESHOLDED_RELU: return x > alpha ? x : 0.0f;",
                                            "case OR_LA_THRESHOLDED_RELU: return x > 0.0f ? x : 0.0f;"),
    "activation_elu_without_alpha": ("case OR_LA_ELU: return x >= 0.0f ? x : alpha * ef_expm1(x);",
                                     "case OR_LA_ELU: return x >= 0.0f ? x : ef_expm1(x);"),
    "activation_scaled_tanh_beta_dropped": ("case OR_LA_SCALED_TANH: return alpha * ef_tanh(beta * x);",
                                            "case OR_LA_SCALED_TANH: return alpha * ef_tanh(x);"),
    "activation_affine_beta_dropped": ("case OR_LA_AFFINE: return alpha * x + beta;", "case OR_LA_AFFINE: return alpha * x;"),
    "activation_softsign_sign": ("case OR_LA_SOFTSIGN: return x / (1.0f + fabsf(x));",
                                 "case OR_LA_SOFTSIGN: return x / (1.0f + x);"),
    "activation_leaky_relu_on_positive": ("case OR_LA_LEAKY_RELU: return x >= 0.0f ? x : alpha * x;",
                                          "case OR_LA_LEAKY_RELU: return x >= 0.0f ? alpha * x : x;"),
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


def _run_mutant(name, workdir):
    """Build the oracle with mutation `name` planted and run the pin suite
    against it in a child process; returns (returncode, stdout)."""
    old, new = MUTATIONS[name]
    src = open(ORACLE_SRC).read()
    if src.count(old) < 1:
        return None, f"mutation anchor for {name} not found"
    mutant = os.path.join(workdir, f"oracle_{name}.c")
    with open(mutant, "w") as f:
        f.write(src.replace(old, new, 1))
    so = os.path.join(workdir, f"liboracle_{name}.so")
    subprocess.run(["gcc", *oracle_build.CFLAGS, mutant, "-o", so, "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB_UNDER_TEST=so, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    """Every planted mistake, built and run concurrently (one child process
    per mutation, as many at once as this host has cores)."""
    from concurrent.futures import ThreadPoolExecutor
    workdir = str(tmp_path_factory.mktemp("mutants"))
    with ThreadPoolExecutor(max_workers=max(1, len(os.sched_getaffinity(0)))) as ex:
        futs = {n: ex.submit(_run_mutant, n, workdir) for n in MUTATIONS}
        return {n: f.result() for n, f in futs.items()}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, mutant_results):
    rc, out = mutant_results[name]
    assert rc is not None, out
    assert rc != 0, f"no pin failed for planted mistake {name}:\n{out[-2000:]}"
    assert "failed" in out
