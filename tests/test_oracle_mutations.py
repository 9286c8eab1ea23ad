"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle source (never
in the committed oracle, and never on a GPU), builds it, and runs the pin
suite against that copy, which must then fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.cpp")

MUTATIONS = {
    "gate_up_interleave_swapped": ("glu(gu[2 * j], gu[2 * j + 1])",
                                   "glu(gu[2 * j + 1], gu[2 * j])"),
    "gate_up_bias_dropped": ("gu[n] = acc + bf16_value(L->b_gu[gu_row0 + n]);",
                             "gu[n] = acc;"),
    "down_bias_dropped": ("y_out[n] = acc + bf16_value(L->b_d[d_row0 + n]);",
                          "y_out[n] = acc;"),
    "ties_to_higher_index": ("logit[e] > logit[best]", "logit[e] >= logit[best]"),
    "glu_constant_wrong": ("sigmoid(1.702f * gate)", "sigmoid(1.0f * gate)"),
    "up_lower_clamp_missing": ("if (up < -7.0f) up = -7.0f;", ""),
    "gate_lower_clamp_added": ("if (gate > 7.0f) gate = 7.0f;",
                               "if (gate > 7.0f) gate = 7.0f; if (gate < -7.0f) gate = -7.0f;"),
    "up_plus_one_dropped": ("return (up + 1.0f) * g;", "return up * g;"),
    "down_transposed": ("weight_at(L->wfmt, L->w_d, s_d, d_row0 + n, j, I)",
                        "weight_at(L->wfmt, L->w_d, s_d, d_row0 + j, n, I)"),
    "combine_weight_dropped": ("acc += w[static_cast<size_t>(p) * k + j] *\n                       y[",
                               "acc += 1.0f *\n                       y["),
    "router_bias_dropped": ("return acc + bf16_value(L->br[e]);", "return acc;"),
    "nibble_order_swapped": ("(col & 1) ? (byte >> 4) : (byte & 0xFu)",
                             "(col & 1) ? (byte & 0xFu) : (byte >> 4)"),
    "fp8_act_scale_wrong": ("const float inv = amax > 0.0f ? 448.0f / amax : 1.0f;",
                            "const float inv = amax > 0.0f ? 240.0f / amax : 1.0f;"),
    "fp8_h_scale_wrong": ("hv[j] = e4m3_value(e4m3_round(h[j] * 8.0f));",
                          "hv[j] = e4m3_value(e4m3_round(h[j] * 4.0f));"),
    "fp8_ties_to_odd": ("(d == best_d && (c & 1) == 0)", "(d == best_d && (c & 1) == 1)"),
    "fp8_no_saturation": ("for (int c = 0; c <= 0x7E; ++c) {", "for (int c = 0; c <= 0x7D; ++c) {"),
    "fp8_weight_scale_twice": ("const float gu_scale = sw_gu[e] * xs;",
                               "const float gu_scale = sw_gu[e] * sw_gu[e] * xs;"),
    "mx_shared_exponent_off_by_one": ("shared = (ex - 1) - 8;", "shared = ex - 8;"),
    "mx_low_clamp_missing": ("if (shared < -127) shared = -127;", ""),
    "mx_block_scale_dropped": ("xv[32 * b + i] = e4m3_value(xq[32 * b + i]) * e8m0_value(sx);",
                               "xv[32 * b + i] = e4m3_value(xq[32 * b + i]);"),
    "mx_h_scale_wrong": ("hv[j] = e4m3_value(e4m3_round(h[j] * 8.0f)) * 0.125f;",
                         "hv[j] = e4m3_value(e4m3_round(h[j] * 8.0f)) * 0.25f;"),
    "ep_range_off_by_one": ("if (e < ex_lo || e >= ex_lo + ex_n) continue;",
                            "if (e < ex_lo || e > ex_lo + ex_n) continue;"),
    "att_sink_not_in_denominator": (
        "double denom = std::isinf(sinks[h]) && sinks[h] < 0 ? 0.0 : std::exp(sinks[h] - m);",
        "double denom = 0.0;"),
    "att_window_off_by_one": ("std::max(0, pos - window + 1)", "std::max(0, pos - window)"),
    "att_gqa_mapping_wrong": ("const int hk = h / rep;", "const int hk = h % Hkv;"),
    "scale_bias_off_by_one": ("static_cast<int>(s) - 127", "static_cast<int>(s) - 128"),
    "softmax_over_all_experts": ("    for (int j = 0; j < k; ++j) w[j] = ex[j] / denom;",
                                 "    for (int e = 0; e < E; ++e) if (!taken[e]) denom += std::exp(logit[e] - m);\n"
                                 "    for (int j = 0; j < k; ++j) w[j] = ex[j] / denom;"),
    "permutation_unstable": ("const int r = next[ids[a]]++;",
                             "const int r = offsets[ids[a] + 1] - 1 - (next[ids[a]]++ - offsets[ids[a]]);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found once"
    mutated = tmp_path / "moe_oracle.cpp"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC",
                           "-shared", "-ffp-contract=off",
                           "-I", os.path.join(ROOT, "oracle"), str(mutated),
                           "-o", str(so)])
    env = dict(os.environ, GPT_OSS_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p",
                        "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"pins did not catch {name}:\n{r.stdout[-2000:]}"
