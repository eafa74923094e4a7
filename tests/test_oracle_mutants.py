"""Planted mistakes: each broken copy of the oracle must fail the pins.

Every mutant is a one-line edit of ``oracle/ce_oracle.c`` compiled into a
temporary library; the pin suite then runs against it in a subprocess and
must fail.  This checks that the pins constrain every term of the oracle,
not that the oracle is right (the pins themselves do that).
"""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ce_oracle.c")

MUTANTS = {
    "target_not_divided_by_T": ("- x[t] / T);", "- x[t]);"),
    "softplus_sign": ("fmax(a, 0.0) + log1p(", "fmax(a, 0.0) - log1p("),
    "target_left_in_others": ("        if (j == skip)\n            continue;\n        sum_add",
                              "        sum_add"),
    "target_grad_exp_minus_one": ("scale * (expm1(lp)", "scale * ((exp(lp) - 1.0)"),
    "grad_missing_inverse_T": ("double scale = (dft ? exp(lp) * g : g) / T;",
                               "double scale = (dft ? exp(lp) * g : g);"),
    "mean_grad_not_divided": ("g = count > 0 ? grad_out[0] / (double)count : 0.0;",
                              "g = grad_out[0];"),
    "mean_loss_not_divided": ("*loss = count > 0 ? sum_value(&total) / (double)count : 0.0;",
                              "*loss = sum_value(&total);"),
    "ignored_rows_counted": ("if (labels[r] != ignore_index)\n            ++count;",
                             "++count;"),
    "grad_sign_flipped": ("dr[j] = scale * (exp(xr[j] / T - zy + lp) - u);",
                          "dr[j] = -scale * (exp(xr[j] / T - zy + lp) - u);"),
    "other_logit_target_swap": ("scale * (exp(xr[j] / T - zy + lp)",
                                "scale * (exp(zy - xr[j] / T + lp)"),
    "masked_rows_computed": ("if (row_mask && row_mask[r] == 0) {\n                *o = 0.0;",
                             "if (0) {\n                *o = 0.0;"),
    "sel_bwd_target_term_sign": ("dr[t] = (-g_t * expm1(lp) - (Gv - g_t) * exp(lp)) / T;",
                                 "dr[t] = (g_t * expm1(lp) - (Gv - g_t) * exp(lp)) / T;"),
    "sel_bwd_others_use_all_of_G": ("- (Gv - g_t) * exp(lp)) / T;", "- Gv * exp(lp)) / T;"),
    "sel_bwd_duplicates_not_summed": ("                if (idx[r * K + i] == t)\n                    sum_add(&gt",
                                      "                if (i == k)\n                    sum_add(&gt"),
    "entropy_target_term_dropped": ("    sum_add(&h, neg_plogp(lp_d));\n", ""),
    "entropy_lse_sign": (": x[d] / T - lp_d;", ": x[d] / T + lp_d;"),
    "entropy_reference_not_dominant": ("    const int64_t d = row_argmax(x, V);\n    const double lp_d",
                                       "    const int64_t d = 0;\n    const double lp_d"),
    "ent_bwd_sign": ("dr[j] -= (gH / T) * pj * (j == d ? Hd : lpj + H);",
                     "dr[j] += (gH / T) * pj * (j == d ? Hd : lpj + H);"),
    "ent_bwd_dominant_by_difference": ("dr[j] -= (gH / T) * pj * (j == d ? Hd : lpj + H);",
                                       "dr[j] -= (gH / T) * pj * (lpj + H);"),
    "ent_bwd_gap_sign": ("sum_add(&q, pj * ((xr[d] - xr[j]) / T));",
                         "sum_add(&q, pj * ((xr[j] - xr[d]) / T));"),
    "ent_bwd_target_drops_H": ("* exp(lp) * (t == d ? Hd : lp + H);", "* exp(lp) * (t == d ? Hd : lp);"),
    "smoothing_off_by_one_class": ("const double u = eps / (double)V;",
                                   "const double u = eps / (double)(V - 1);"),
    "smoothing_mean_not_over_V": ("eps * (sum_value(&nl) / (double)V)", "eps * sum_value(&nl)"),
    "dft_weight_missing_in_gradient": ("double scale = (dft ? exp(lp) * g : g) / T;",
                                       "double scale = g / T;"),
    "softcap_chain_factor_dropped": ("dx[r * ldx + j] *= sech * sech;", "dx[r * ldx + j] *= 1.0;"),
    "softcap_chain_factor_cancels": ("dx[r * ldx + j] *= sech * sech;",
                                     "dx[r * ldx + j] *= 1.0 - tanh(x[r * ld + j] / softcap)"
                                     " * tanh(x[r * ld + j] / softcap);"),
    "softcap_not_rescaled": ("z[r * V + j] = softcap * tanh(x[r * ld + j] / softcap);",
                             "z[r * V + j] = tanh(x[r * ld + j] / softcap);"),
    "sel_bwd_missing_inverse_T": ("dr[j] = -(Gv / T) * pj;",
                                  "dr[j] = -Gv * pj;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
                    "-shared", "-fPIC", str(mutated), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, GBCE_ORACLE_LIB=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"pins passed with mutant {name}:\n{res.stdout[-2000:]}"
