"""Mutation check of the oracle pins.

Each case plants one plausible mistake in a copy of the oracle's C source,
builds it on the CPU, and runs the pin suite against it; the suite must go
red. This shows the pins constrain every term of the definition rather than
re-deriving the oracle from itself.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "rmsnorm_oracle.c")

MUTATIONS = {
    "sum_instead_of_mean": ("const double ms = ss / (double)N;", "const double ms = ss;"),
    "eps_outside_root": ("1.0 / sqrt(ms + jb->eps)", "1.0 / (sqrt(ms) + jb->eps)"),
    "offset_dropped_fwd": ("const double factor = jb->w ? jb->offset + load_elem",
                           "const double factor = jb->w ? load_elem"),
    "w_index_reversed": ("load_elem(jb->wdtype, jb->w, j) : 1.0;\n            const double yj",
                         "load_elem(jb->wdtype, jb->w, N - 1 - j) : 1.0;\n            const double yj"),
    "bwd_sign_flip": ("rstd * (g - xhat * c)", "rstd * (g + xhat * c)"),
    "bwd_c_not_mean": ("c /= (double)N;\n        cabs /= (double)N;", "c /= 1.0;\n        cabs /= (double)N;"),
    "bwd_offset_dropped": ("wpo[j] = jb->w ? jb->offset + load_elem", "wpo[j] = jb->w ? 0.0 * jb->offset + load_elem"),
    "dw_uses_g": ("jb->dw[j] += dyj * xhat;", "jb->dw[j] += g * xhat;"),
    "dw_missing_rstd": ("jb->dw[j] += dyj * xhat;", "jb->dw[j] += dyj * hv[j];"),
    "dres_dropped": ("rstd * (fabs(g) + fabs(xhat * c));\n            if (jb->dres) {\n"
                     "                const double d = load_elem(jb->dtype, jb->dres, base + j);\n"
                     "                dxj += d;",
                     "rstd * (fabs(g) + fabs(xhat * c));\n            if (jb->dres) {\n"
                     "                const double d = load_elem(jb->dtype, jb->dres, base + j);\n"
                     "                dxj += 0.0 * d;"),
    "ln_fused_h_unrounded": ("h[j] = round_to(jb->dtype, xv + load_elem(jb->dtype, jb->residual, base + j));\n"
                             "            else\n                h[j] = xv;\n        }\n        double sum = 0.0;",
                             "h[j] = xv + load_elem(jb->dtype, jb->residual, base + j);\n"
                             "            else\n                h[j] = xv;\n        }\n        double sum = 0.0;"),
    "ln_dres_dropped": ("rstd * (fabs(g) + fabs(mg) + fabs(xhat * c));\n            if (jb->dres) {\n"
                        "                const double d = load_elem(jb->dtype, jb->dres, base + j);\n"
                        "                dxj += d;",
                        "rstd * (fabs(g) + fabs(mg) + fabs(xhat * c));\n            if (jb->dres) {\n"
                        "                const double d = load_elem(jb->dtype, jb->dres, base + j);\n"
                        "                dxj += 0.0 * d;"),
    "fused_h_unrounded": ("/* h: the row that is normalised */\n        for (int64_t j = 0; j < N; ++j) {\n"
                          "            double xv = load_elem(jb->dtype, jb->x, base + j);\n"
                          "            if (jb->residual)\n"
                          "                h[j] = round_to(jb->dtype, xv + load_elem(jb->dtype, jb->residual, base + j));",
                          "/* h: the row that is normalised */\n        for (int64_t j = 0; j < N; ++j) {\n"
                          "            double xv = load_elem(jb->dtype, jb->x, base + j);\n"
                          "            if (jb->residual)\n"
                          "                h[j] = xv + load_elem(jb->dtype, jb->residual, base + j);"),
    "bf16_via_binary32": ("int oracle_bf16_round(double v, uint16_t *out)\n{\n",
                          "int oracle_bf16_round(double v, uint16_t *out)\n{\n    v = (double)(float)v;\n"),
    "f16_via_binary32": ("int oracle_f16_round(double v, uint16_t *out)\n{\n",
                         "int oracle_f16_round(double v, uint16_t *out)\n{\n    v = (double)(float)v;\n"),
    "bf16_ties_away": ("double q = rint(ldexp(m, 8));", "double q = round(ldexp(m, 8));"),
    "f16_ties_away": ("double q = rint(ldexp(m, 11));", "double q = round(ldexp(m, 11));"),
    "f16_subnormal_quantum": ("double q = rint(ldexp(a, 24));", "double q = rint(ldexp(a, 23));"),
    "non_affine_keeps_offset": ("load_elem(jb->wdtype, jb->w, j) : 1.0;\n            const double yj",
                                "load_elem(jb->wdtype, jb->w, j) : jb->offset + 1.0;\n            const double yj"),
    "e4m3_ties_away": ("double q = rint(ldexp(m, 4));", "double q = round(ldexp(m, 4));"),
    "e4m3_exponent_bias": ("const int be = e - 1 + 7;", "const int be = e - 1 + 8;"),
    "e4m3_subnormal_quantum": ("double q = rint(ldexp(a, 9));", "double q = rint(ldexp(a, 8));"),
    "e4m3_decode_bias": ("ldexp((double)(f + 8), e - 10)", "ldexp((double)(f + 8), e - 11)"),
    "e4m3_overflow_to_nan": ("if (a >= 448.0) { *out = (uint8_t)(sign | 0x7eu); return 0; }",
                             "if (a >= 448.0) { *out = (uint8_t)(sign | 0x7fu); return 0; }"),
    "fp8_row_scale_not_to_448": ("sc = amax > 0.0 ? 448.0 / amax : 1.0;", "sc = amax > 0.0 ? 256.0 / amax : 1.0;"),
    "fp8_scale_divides": ("const double v = yrow[j] * sc;", "const double v = yrow[j] / sc;"),
    "fp8_amax_of_h": ("if (fabs(yj) > amax) amax = fabs(yj);", "if (fabs(h[j]) > amax) amax = fabs(h[j]);"),
    "ln_unbiased_variance": ("const double var = sq / (double)N;", "const double var = sq / (double)(N > 1 ? N - 1 : 1);"),
    "ln_variance_not_centred": ("for (int64_t j = 0; j < N; ++j) sq += (h[j] - mu) * (h[j] - mu);",
                                "for (int64_t j = 0; j < N; ++j) sq += h[j] * h[j];"),
    "ln_beta_dropped": ("const double yj = (h[j] - mu) * rstd * factor + bias;",
                        "const double yj = (h[j] - mu) * rstd * factor + 0.0 * bias;"),
    "ln_mean_not_subtracted_in_y": ("const double yj = (h[j] - mu) * rstd * factor + bias;",
                                    "const double yj = h[j] * rstd * factor + bias;"),
    "ln_offset_dropped": ("gpo[j] = jb->gamma ? jb->offset + load_elem", "gpo[j] = jb->gamma ? 0.0 * jb->offset + load_elem"),
    "ln_dx_missing_mean_g": ("double dxj = rstd * (g - mg - xhat * c);", "double dxj = rstd * (g - xhat * c);"),
    "ln_dx_missing_xhat_term": ("double dxj = rstd * (g - mg - xhat * c);", "double dxj = rstd * (g - mg);"),
    "ln_dbeta_uses_g": ("jb->db[j] += dyj;", "jb->db[j] += g;"),
    "ln_dgamma_uses_h": ("jb->dg[j] += dyj * xhat;", "jb->dg[j] += dyj * hv[j];"),
    "ln_bwd_ignores_given_mean": ("mu = (double)jb->mean_in[i];", "mu = 0.0 * (double)jb->mean_in[i];"),
    "weight_read_as_activation_type": ("wpo[j] = jb->w ? jb->offset + load_elem(jb->wdtype",
                                       "wpo[j] = jb->w ? jb->offset + load_elem(jb->dtype"),
    "fp8_scale_inv_not_reciprocal": ("if (jb->scale_inv) jb->scale_inv[i] = 1.0 / sc;",
                                     "if (jb->scale_inv) jb->scale_inv[i] = sc;"),
    "ln_mean_over_n_plus_1": ("const double mu = sum / (double)N;", "const double mu = sum / (double)(N + 1);"),
    "bwd_ignores_given_rstd": ("double rstd;\n        if (jb->rstd_in) {\n            rstd = (double)jb->rstd_in[i];\n",
                               "double rstd;\n        if (jb->rstd_in) {\n            rstd = 1.0 + 0.0 * (double)jb->rstd_in[i];\n"),
    "e4m3_saturates_late": ("if (a >= 448.0) { *out = (uint8_t)(sign | 0x7eu); return 0; }",
                            "if (a >= 480.0) { *out = (uint8_t)(sign | 0x7eu); return 0; }"),
    "ln_dgamma_uncentred": ("jb->dg[j] += dyj * xhat;", "jb->dg[j] += dyj * (hv[j] * rstd);"),
    "fp8_tensor_scale_ignored": ("double sc = jb->fp8_scale;", "double sc = 1.0;"),
    "dres_subtracted": ("rstd * (fabs(g) + fabs(xhat * c));\n            if (jb->dres) {\n"
                        "                const double d = load_elem(jb->dtype, jb->dres, base + j);\n"
                        "                dxj += d;",
                        "rstd * (fabs(g) + fabs(xhat * c));\n            if (jb->dres) {\n"
                        "                const double d = load_elem(jb->dtype, jb->dres, base + j);\n"
                        "                dxj -= d;"),
    "bwd_recomputed_rstd_without_eps": ("rstd = 1.0 / sqrt(ss / (double)N + jb->eps);",
                                        "rstd = 1.0 / sqrt(ss / (double)N);"),
    "ln_mean_g_over_n_minus_1": ("mg /= (double)N;", "mg /= (double)(N > 1 ? N - 1 : 1);"),
    "rstd_saved_as_std": ("if (jb->rstd32) jb->rstd32[i] = (float)rstd;\n        if (jb->fp8_mode",
                          "if (jb->rstd32) jb->rstd32[i] = (float)(1.0 / rstd);\n        if (jb->fp8_mode"),
    "ln_mean32_not_saved": ("if (jb->mean32) jb->mean32[i] = (float)mu;", "if (jb->mean32) jb->mean32[i] = 0.0f;"),
    "fp8_amax_after_scaling": ("if (jb->amax_row) jb->amax_row[i] = amax;",
                               "if (jb->amax_row) jb->amax_row[i] = amax * sc;"),
    "ln_bwd_recomputed_var_uncentred": ("for (int64_t j = 0; j < N; ++j) sq += (hv[j] - mu) * (hv[j] - mu);",
                                        "for (int64_t j = 0; j < N; ++j) sq += hv[j] * hv[j];"),
    "ln_beta_takes_offset": ("const double bias = jb->beta ? load_elem(jb->wdtype, jb->beta, j) : 0.0;",
                             "const double bias = jb->beta ? jb->offset + load_elem(jb->wdtype, jb->beta, j) : 0.0;"),
    "fp8_zero_row_scale_zero": ("sc = amax > 0.0 ? 448.0 / amax : 1.0;", "sc = amax > 0.0 ? 448.0 / amax : 0.0;"),
    # the tolerance scales the GPU checks are widened by
    "cabs_not_mean": ("c /= (double)N;\n        cabs /= (double)N;",
        "c /= (double)N;\n        cabs /= 1.0;"),
    "dw_abs_signed": ("jb->dw_abs[j] += fabs(dyj * xhat);",
        "jb->dw_abs[j] += dyj * xhat;"),
    "dw_abs_double_counted": ("sa += jobs[t].dw_abs[j];",
        "sa += 2.0 * jobs[t].dw_abs[j];"),
    "dx_scale_drops_dres": ("rstd * (fabs(g) + fabs(xhat * c));\n            if (jb->dres) {\n                const double d = load_elem(jb->dtype, jb->dres, base + j);\n                dxj += d;\n                scale += fabs(d);",
        "rstd * (fabs(g) + fabs(xhat * c));\n            if (jb->dres) {\n                const double d = load_elem(jb->dtype, jb->dres, base + j);\n                dxj += d;\n                scale += 0.0 * fabs(d);"),
    "dx_scale_missing_xhat_c": ("double scale = rstd * (fabs(g) + fabs(xhat * c));",
        "double scale = rstd * fabs(g);"),
    "dx_scale_missing_rstd": ("double scale = rstd * (fabs(g) + fabs(xhat * c));",
        "double scale = (fabs(g) + fabs(xhat * c));"),
    "dx_cscale_missing_xhat": ("jb->dx_cscale[base + j] = rstd * fabs(xhat) * cabs;",
        "jb->dx_cscale[base + j] = rstd * cabs;"),
    "dx_cscale_signed_sum": ("cabs += fabs(g * (hv[j] * rstd));",
        "cabs += g * (hv[j] * rstd);"),
    "ln_dx_scale_missing_mean_g": ("double scale = rstd * (fabs(g) + fabs(mg) + fabs(xhat * c));",
        "double scale = rstd * (fabs(g) + fabs(xhat * c));"),
    "ln_dx_scale_drops_dres": ("rstd * (fabs(g) + fabs(mg) + fabs(xhat * c));\n            if (jb->dres) {\n                const double d = load_elem(jb->dtype, jb->dres, base + j);\n                dxj += d;\n                scale += fabs(d);",
        "rstd * (fabs(g) + fabs(mg) + fabs(xhat * c));\n            if (jb->dres) {\n                const double d = load_elem(jb->dtype, jb->dres, base + j);\n                dxj += d;\n                scale += 0.0 * fabs(d);"),
    "ln_cscale_missing_mean_abs_g": ("jb->dx_cscale[base + j] = rstd * (mgabs + fabs(xhat) * cabs);",
        "jb->dx_cscale[base + j] = rstd * fabs(xhat) * cabs;"),
    "ln_cscale_missing_xhat": ("jb->dx_cscale[base + j] = rstd * (mgabs + fabs(xhat) * cabs);",
        "jb->dx_cscale[base + j] = rstd * (mgabs + cabs);"),
    "ln_mean_abs_g_not_mean": ("mgabs /= (double)N;",
        "mgabs /= 1.0;"),
    "ln_dg_abs_signed": ("jb->dg_abs[j] += fabs(dyj * xhat);",
        "jb->dg_abs[j] += dyj * xhat;"),
    "ln_db_abs_signed": ("jb->db_abs[j] += fabs(dyj);",
        "jb->db_abs[j] += dyj;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=gnu99", "-fPIC", "-shared", "-ffp-contract=off",
                           "-o", str(lib), str(mutated), "-lm", "-lpthread"])
    env = dict(os.environ, RMSNORM_ORACLE_LIB_OVERRIDE=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"
