"""The pins catch plausible mistakes in the oracle.

Each case below copies the oracle's source, plants one mistake (a transposed index, a dropped term,
a wrong order of normalisations, a wrong mean, a misplaced eps, a wrong rounding rule ...),
compiles the copy on the CPU and runs the whole pin battery against it: at least one pin must
fail. The real oracle passes every pin (``test_oracle_pins.py``).
"""

import os
import subprocess

import pytest

import oracle
import pins

MUTANTS = {
    "hc_post_comb_transposed": ("comb[j * hc + k]) * bf16_to_double(X[j * d + i]);",
                                "comb[k * hc + j]) * bf16_to_double(X[j * d + i]);"),
    "hc_post_drops_delta": ("double acc = static_cast<double>(post[k]) * bf16_to_double(delta[i]);",
                            "double acc = 0.0;"),
    "hc_post_wrong_post_index": ("static_cast<double>(post[k]) * bf16_to_double(delta[i])",
                                 "static_cast<double>(post[0]) * bf16_to_double(delta[i])"),
    "mixes_mean_over_d": ("double r = 1.0 / std::sqrt(ss / D + norm_eps);",
                          "double r = 1.0 / std::sqrt(ss / d + norm_eps);"),
    "mixes_no_rsqrt": ("mixes[m] = dot * r;", "mixes[m] = dot;"),
    "mixes_eps_outside_sqrt": ("double r = 1.0 / std::sqrt(ss / D + norm_eps);",
                               "double r = 1.0 / (std::sqrt(ss / D) + norm_eps);"),
    "pre_wrong_scale": ("pre[j] = sigmoid(m[j] * s0 + hc_base[j]) + eps;",
                        "pre[j] = sigmoid(m[j] * s1 + hc_base[j]) + eps;"),
    "pre_no_eps": ("pre[j] = sigmoid(m[j] * s0 + hc_base[j]) + eps;",
                   "pre[j] = sigmoid(m[j] * s0 + hc_base[j]);"),
    "post_no_factor_two": ("post[j] = 2.0 * sigmoid(", "post[j] = 1.0 * sigmoid("),
    "post_wrong_offset": ("sigmoid(m[hc + j] * s1 + hc_base[hc + j])", "sigmoid(m[hc + j] * s1 + hc_base[j])"),
    "comb_logits_transposed": ("C[j * hc + k] = m[2 * hc + j * hc + k] * s2 + hc_base[2 * hc + j * hc + k];",
                               "C[j * hc + k] = m[2 * hc + k * hc + j] * s2 + hc_base[2 * hc + k * hc + j];"),
    "softmax_eps_inside": ("C[j * hc + k] = C[j * hc + k] / sum + eps;",
                           "C[j * hc + k] = C[j * hc + k] / (sum + eps);"),
    "softmax_over_columns": ("for (int k = 0; k < hc; ++k) C[j * hc + k] = C[j * hc + k] / sum + eps;",
                             "for (int k = 0; k < hc; ++k) C[j * hc + k] = C[j * hc + k] / sum + eps;\n"
                             "    }\n    for (int j = 0; j < hc; ++j) { for (int k = 0; k < j; ++k) "
                             "std::swap(C[j * hc + k], C[k * hc + j]);"),
    "sinkhorn_row_first": ("    col_normalise();\n    for (int it = 0; it < iters - 1; ++it) {\n"
                           "        row_normalise();\n        col_normalise();",
                           "    row_normalise();\n    for (int it = 0; it < iters - 1; ++it) {\n"
                           "        col_normalise();\n        row_normalise();"),
    "sinkhorn_one_iteration_short": ("for (int it = 0; it < iters - 1; ++it)", "for (int it = 0; it < iters - 2; ++it)"),
    "sinkhorn_colsum_eps_dropped": ("C[j * hc + k] = C[j * hc + k] / (cs[k] + eps);",
                                    "C[j * hc + k] = C[j * hc + k] / cs[k];"),
    "hc_pre_wrong_weight": ("double term = static_cast<double>(pre_mix[j]) * bf16_to_double(X[j * d + i]);",
                            "double term = static_cast<double>(pre_mix[0]) * bf16_to_double(X[j * d + i]);"),
    "rmsnorm_no_eps": ("double r = 1.0 / std::sqrt(ss / d + eps);", "double r = 1.0 / std::sqrt(ss / d);"),
    "rmsnorm_no_weight": ("double v = static_cast<double>(w[i]) * (bf16_to_double(x[i]) * r);",
                          "double v = bf16_to_double(x[i]) * r;"),
    "round_ties_away": ("(frac == 0.5 && std::fmod(r, 2.0) != 0.0)", "(frac == 0.5)"),
    "round_truncates": ("if (frac > 0.5 || (frac == 0.5 && std::fmod(r, 2.0) != 0.0)) r += 1.0;", ""),
    "pre_step_norms_unrounded_y": ("rmsnorm_token(d, y.data(), norm_w, norm_eps, y_normed + t * d, nullptr);",
                                   "{ std::vector<double> ye(d); pre_token(hc, d, Xt, pre_mix + t * hc, y.data(), ye.data(), nullptr);"
                                   " double ss = 0; for (int i = 0; i < d; ++i) ss += ye[i] * ye[i];"
                                   " double rr = 1.0 / std::sqrt(ss / d + norm_eps);"
                                   " for (int i = 0; i < d; ++i) y_normed[t * d + i] = double_to_bf16(norm_w[i] * (ye[i] * rr)); }"),
    "expand_interleaved": ("for (int j = 0; j < hc; ++j) std::copy(h, h + d, X + static_cast<int64_t>(j) * d);",
                           "for (int i = 0; i < d; ++i) for (int j = 0; j < hc; ++j) X[i * hc + j] = h[i];"),
    "expand_identity_not_normalised": ("pm[j] = 1.0f / static_cast<float>(hc);", "pm[j] = 1.0f;"),
    "expand_identity_one_hot_wrong_scale": ("pm[j] = 1.0f / static_cast<float>(hc);",
                                            "pm[j] = (j == 0) ? 0.5f : 0.0f;"),
    "final_uses_fixed_eps": ("rmsnorm_token(d, y.data(), norm_w, norm_eps, z + t * d, z_exact ? z_exact + t * d : nullptr);",
                             "rmsnorm_token(d, y.data(), norm_w, 1e-6, z + t * d, z_exact ? z_exact + t * d : nullptr);"),
    "final_skips_collapse_rounding": ("pre_token(hc, d, X + t * hc * d, pre_mix + t * hc, y.data(), nullptr, nullptr);\n"
                                      "        rmsnorm_token(d, y.data(), norm_w, norm_eps, z + t * d",
                                      "pre_token(hc, d, X + t * hc * d, pre_mix + t * hc, y.data(), nullptr, nullptr);\n"
                                      "        for (int i = 0; i < d; ++i) y[i] = X[t * hc * d + i];\n"
                                      "        rmsnorm_token(d, y.data(), norm_w, norm_eps, z + t * d"),
    "post_then_final_skips_post": ("oracle_hc_post(n, hc, d, X, delta, post, comb, X_out, threads);\n"
                                   "    oracle_hc_final(",
                                   "std::copy(X, X + n * hc * d, X_out);\n    oracle_hc_final("),
    "stream_mean_over_columns": ("for (int j = 0; j < hc; ++j) acc += bf16_to_double(X[(t * hc + j) * d + i]);",
                                 "for (int j = 0; j < hc; ++j) acc += bf16_to_double(X[t * hc * d + i * hc + j]);"),
    "stream_mean_sum_not_mean": ("const double m = acc / hc;", "const double m = acc;"),
}


def _build_mutant(name, tmp_path):
    with open(oracle._SRC) as f:
        src = f.read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, "mutation site not found: %s" % name
    src = src.replace(old, new, 1)
    path = tmp_path / ("mut_%s.cpp" % name)
    path.write_text(src)
    out = str(tmp_path / ("libmut_%s.so" % name))
    oracle.build(force=True, src=str(path), out=out)
    return oracle.load(out)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    lib = _build_mutant(name, tmp_path)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "no pin caught the planted mistake %r" % name
