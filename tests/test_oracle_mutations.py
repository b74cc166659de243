"""Mutation check of the oracle's pins: plant plausible mistakes in a copy of the
oracle's C source (on the CPU, in a temporary directory), rebuild it there, and
require the pin suite to fail for every one of them."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "anvil_oracle.c")

MUTATIONS = {
    "dropped_b_term": ("Bf[e] = b * Af[e] + c * P[e];", "Bf[e] = c * P[e];"),
    "sign_of_c": ("Bf[e] = b * Af[e] + c * P[e];", "Bf[e] = b * Af[e] - c * P[e];"),
    "a_times_C": ("X[e] = f32_to_bf16(a * Xf[e] + Cf[e]);", "X[e] = f32_to_bf16(Xf[e] + a * Cf[e]);"),
    "A_over_d": ("const float d2 = d * d;", "const float d2 = d;"),
    "no_margin": ("const float d = sqrtf(tr) * margin + eps;", "const float d = sqrtf(tr) + eps;"),
    "trace_wrong_index": ("tr += bf16_to_f32(A[(size_t)i * s + i]);", "tr += bf16_to_f32(A[(size_t)i * s]);"),
    "slow_rail_fast_beta": ("float v1 = lerp32(v_slow[e], g, w_slow);", "float v1 = lerp32(v_slow[e], g, w_fast);"),
    "blend_weights_swapped": ("float blend = w * v0 + one_minus_w * v1;", "float blend = one_minus_w * v0 + w * v1;"),
    "lerp_reversed": ("g = lerp32(g, blend, momentum);", "g = lerp32(blend, g, momentum);"),
    "tall_transposed_update": ("if (is_tall) matmul_f32(Xf, Bf, Cf, rows, cols, cols);",
                               "if (is_tall) { transpose_f32(Xf, T, rows, cols); matmul_f32(Bf, T, P, cols, cols, rows); transpose_f32(P, Cf, cols, rows); }"),
    "first_gram_recomputed": ("if (k > 0) gram_bf16(Xf, rows, cols, is_tall, T, Af, A);",
                              "gram_bf16(Xf, rows, cols, is_tall, T, Af, A);"),
    "no_bf16_round_of_B": ("to_bf16(Bf, B, nA);\n        to_f32(B, Bf, nA);", "to_bf16(Bf, B, nA);"),
    "ema_weight_beta2": ("const float w = 1.0f - beta2;", "const float w = beta2;"),
    "lanes_wrong_dim": ("const int lanes_are_rows = rows >= cols;", "const int lanes_are_rows = rows < cols;"),
    "gate_sign_reversed": ("const float aligned = (gate[e] * w >= 0.0f) ? 1.0f : 0.0f;",
                           "const float aligned = (gate[e] * w <= 0.0f) ? 1.0f : 0.0f;"),
    "decay_without_lr": ("w = (w - ((w * aligned) * wd) * lrm) - u * lrm;", "w = (w - (w * aligned) * wd) - u * lrm;"),
    "no_norm_restore": ("const float ratio = pre_norm / post_norm;", "const float ratio = 1.0f;"),
    "adam_mask_reversed": ("const float mask = (u * p[e] > 0.0f) ? 1.0f : 0.0f;",
                           "const float mask = (u * p[e] < 0.0f) ? 1.0f : 0.0f;"),
    "adam_second_moment_unsquared": ("(c2 * g[e]) * g[e]", "(c2 * g[e])"),
    "scale_not_rounded_to_bf16": ("for (int l = 0; l < nl; ++l) scale[l] = round_bf16(scale[l] * ratio);",
                                  "for (int l = 0; l < nl; ++l) scale[l] = scale[l] * ratio;"),
    "power_mean_over_lane_count": ("power[l] = s / (float)lane_len;", "power[l] = s / (float)nl;"),
    "gain_from_old_energy": ("            le[l] = lerp32(le[l], power[l], w);\n"
                             "            const float gain = rsqrt_rn(le[l] > 1e-10f ? le[l] : 1e-10f);",
                             "            const float gain = rsqrt_rn(le[l] > 1e-10f ? le[l] : 1e-10f);\n"
                             "            le[l] = lerp32(le[l], power[l], w);"),
    "adam_eps_inside_sqrt": ("float u = (m / (sqrtf(v) + eps)) * step_size;", "float u = (m / sqrtf(v + eps)) * step_size;"),
    "no_nesterov_lookahead": ("g = lerp32(g, blend, momentum);", "g = blend;"),
    "X_over_d_squared": ("X[e] = f32_to_bf16(bf16_to_f32(X[e]) / d);", "X[e] = f32_to_bf16(bf16_to_f32(X[e]) / d2);"),
    "maps_reversed": ("const float a = maps[3 * k], b = maps[3 * k + 1], c = maps[3 * k + 2];",
                      "const int kr = nmaps - 1 - k;\n        const float a = maps[3 * kr], b = maps[3 * kr + 1], c = maps[3 * kr + 2];"),
    "trace_from_unrounded_gram": ("tr += bf16_to_f32(A[(size_t)i * s + i]);", "tr += Af[(size_t)i * s + i];"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, name
    src = tmp_path / "anvil_oracle.c"
    src.write_text(text.replace(old, new))
    env = dict(os.environ, ANVIL_ORACLE_SRC=str(src), ANVIL_ORACLE_BUILD=str(tmp_path / "b"))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_tail.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutation {name} survived:\n{r.stdout[-2000:]}"
