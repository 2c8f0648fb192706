"""The oracle's pins catch plausible mistakes: each case plants one mistake
(a flipped sign, a dropped factor, a swapped operand or population, a
non-strict comparison, an off-by-one) in a copy of oracle.c in a temporary
directory and requires tests/test_oracle_pins.py to fail on that copy.  The
oracle under test is never modified."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "k3_sign": ("q.k3 = r_minus_1 - log_r;", "q.k3 = r_minus_1 + log_r;"),
    "delta_sign": ("double d = (double)l_tr - (double)l_ro;", "double d = (double)l_ro - (double)l_tr;"),
    "weight_max_for_min": ("q.w = r < C ? r : C;", "q.w = r > C ? r : C;"),
    "rel_over_rollout": ("q.rel = fabs(d) / (fabs((double)l_tr) + 1e-8);",
                         "q.rel = fabs(d) / (fabs((double)l_ro) + 1e-8);"),
    "k2_without_half": ("q.k2 = 0.5 * log_r * log_r;", "q.k2 = log_r * log_r;"),
    "clip_not_strict": ("q.clip = (double)d32 > logC;", "q.clip = (double)d32 >= logC;"),
    "lse_without_max": ("double lse = m + log(S);", "double lse = log(S);"),
    "temperature_multiplies": ("z[v] = acc / temperature;", "z[v] = acc * temperature;"),
    "quantile_position_nq": ("const double h = (double)(n - 1) * q;", "const double h = (double)n * q;"),
    "ppo_clip_eps_swapped": ("const double rclip = A > 0.0 ? 1.0 + eps_high : 1.0 - eps_low;",
                             "const double rclip = A > 0.0 ? 1.0 + eps_low : 1.0 - eps_high;"),
    "ppo_grad_through_clip": ("grad = ppo_clipped ? 0.0 : -w * r * A;", "grad = -w * r * A;"),
    "seqmean_k1_wrong_field": ("b_mk1 += o[SQ_MEAN_K1];", "b_mk1 += o[SQ_MEAN_K2];"),
    "clip_ratio_over_used": ("batch[BT_CLIP_RATIO] = mean_or_zero(b_clip, b_mask);",
                             "batch[BT_CLIP_RATIO] = mean_or_zero(b_clip, b_used);"),
    "default_tau_sign": ("const double tau = isnan(tau_seq) ? (C - 1.0) - logC : tau_seq;",
                         "const double tau = isnan(tau_seq) ? (C - 1.0) + logC : tau_seq;"),
    "ppo_thresholds_eps_swapped": ("const double log_hi = log1p(eps_high), log_lo = log1p(-eps_low)",
                                   "const double log_hi = log1p(eps_low), log_lo = log1p(-eps_high)"),
    "ppo_weight_not_truncated": ("const double w = rc < C ? rc : C;", "const double w = rc;"),
    "k1_sign": ("q.k1 = -log_r;", "q.k1 = log_r;"),
    "logp_plus_lse": ("*out_logp = (a >= 0 && (int64_t)a < V) ? z[a] - lse : NAN;",
                      "*out_logp = (a >= 0 && (int64_t)a < V) ? z[a] + lse : NAN;"),
    "ratio_quantile_without_exp": ("out[MO_RATIO_Q01] = quantile_sorted(d, n, 0.01, 1);",
                                   "out[MO_RATIO_Q01] = quantile_sorted(d, n, 0.01, 0);"),
    "extreme_not_strict": ("const int ext = used && fabs((double)d32) > tau_tok;",
                           "const int ext = used && fabs((double)d32) >= tau_tok;"),
    "n_mask_counts_used": ("n_mask += mask[t] != 0;", "n_mask += q.used;"),
    "mean_abs_delta_signed": ("sad += fabs(q.delta);", "sad += q.delta;"),
    "nan_ratio_over_used": ("batch[BT_NAN_RATIO] = mean_or_zero(b_nan, b_mask);",
                            "batch[BT_NAN_RATIO] = mean_or_zero(b_nan, b_used);"),
    "p95_on_signed_delta": ("out[MO_P95_ABS_DELTA] = quantile_sorted(ad, n, 0.95, 0);",
                            "out[MO_P95_ABS_DELTA] = quantile_sorted(d, n, 0.95, 0);"),
    "backward_softmax_sign": ("((v == targets[t] ? 1.0 : 0.0) - p) / temperature;",
                              "(p - (v == targets[t] ? 1.0 : 0.0)) / temperature;"),
    "backward_without_temperature": ("((v == targets[t] ? 1.0 : 0.0) - p) / temperature;",
                                     "((v == targets[t] ? 1.0 : 0.0) - p);"),
    "backward_dh_times_h": ("dht[d] += dzv * bf16_value(w[d]);", "dht[d] += dzv * hd[d];"),
    "backward_dw_times_w": ("dwv[d] += dzv * hd[d];", "dwv[d] += dzv * bf16_value(w[d]);"),
    "target_off_by_one": ("*out_logp = (a >= 0 && (int64_t)a < V) ? z[a] - lse : NAN;",
                          "*out_logp = (a >= 0 && (int64_t)a < V) ? z[a > 0 ? a - 1 : a] - lse : NAN;"),
    "seqmean_over_all_sequences": ("batch[BT_SEQMEAN_K3] = mean_or_zero(b_mk3, b_nonempty);",
                                   "batch[BT_SEQMEAN_K3] = mean_or_zero(b_mk3, (double)S);"),
    "rejection_on_k2": ("double stat = seq_estimator == 3 ? o[SQ_MEAN_K3] : fabs(o[SQ_MEAN_K1]);",
                        "double stat = seq_estimator == 3 ? o[SQ_MEAN_K2] : fabs(o[SQ_MEAN_K1]);"),
    "token_rejection_ignores_mask": ("const int ext = used && fabs((double)d32) > tau_tok;",
                                     "const int ext = isfinite(d32) && fabs((double)d32) > tau_tok;"),
    "ppo_loss_sign": ("loss = ppo_clipped ? -w * rclip * A : -w * r * A;",
                      "loss = ppo_clipped ? w * rclip * A : w * r * A;"),
    "ppo_clip_on_ties": ("(A > 0.0 && (double)dt32 > log_hi) || (A < 0.0 && (double)dt32 < log_lo)",
                         "(A > 0.0 && (double)dt32 >= log_hi) || (A < 0.0 && (double)dt32 <= log_lo)"),
    "max_of_signed_delta": ("        if (fabs(q.delta) > z.mx)\n            z.mx = fabs(q.delta);",
                            "        if (q.delta > z.mx)\n            z.mx = q.delta;"),
    "nan_counted_when_masked_out": ("q.nan = in && !fin;", "q.nan = !fin;"),
    "quantile_interpolation_sign": ("return lo + (h - fl) * (hi - lo);", "return lo + (h - fl) * (hi + lo);"),
    "extreme_on_signed_delta": ("const int ext = used && fabs((double)d32) > tau_tok;",
                                "const int ext = used && (double)d32 > tau_tok;"),
    "extreme_fraction_over_all_tokens": ("out[MO_FRAC_EXTREME] = mean_or_zero((double)n_ext, (double)n);",
                                         "out[MO_FRAC_EXTREME] = mean_or_zero((double)n_ext, (double)N);"),
    "median_ratio_of_abs_delta": ("out[MO_RATIO_Q50] = quantile_sorted(d, n, 0.5, 1);",
                                  "out[MO_RATIO_Q50] = quantile_sorted(ad, n, 0.5, 1);"),
}


def _copy_tree(dst):
    ignore = shutil.ignore_patterns("*.so", "__pycache__")
    for d in ("oracle", "workloads"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(dst, d), ignore=ignore)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    for f in ("tests/conftest.py", "tests/test_oracle_pins.py", "pytest.ini"):
        shutil.copy(os.path.join(ROOT, f), os.path.join(dst, f))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_a_planted_oracle_mistake_fails_the_pins(name, tmp_path):
    old, new = MUTATIONS[name]
    _copy_tree(str(tmp_path))
    path = tmp_path / "oracle" / "oracle.c"
    src = path.read_text()
    assert src.count(old) == 1, "the mutation no longer matches oracle.c: " + name
    path.write_text(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-q", "-x",
                        "-p", "no:cacheprovider"], cwd=str(tmp_path), capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 1, (name, r.stdout[-400:], r.stderr[-400:])
