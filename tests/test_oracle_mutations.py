"""The pins must reject plausible mistakes in the oracle.

Each case copies the oracle's C source, plants one mistake by a textual
substitution (a wrong table entry, swapped nibble order, wrong block size, a
sign error, a dropped term, a transposed operand, a slot mix-up, ...),
compiles the broken copy on the CPU and runs the pin checks against it
through ``oracle.using_library``.  At least one pin has to fail for every
mutation; the unmodified source has to pass them all.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTATIONS = {
    "e2m1_table_entry": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 4.0, 6.0}"),
    "e2m1_sign_bit": ("return (code & 8u) ? -v : v;", "return (code & 4u) ? -v : v;"),
    "nibble_order": ("unsigned code = (k & 1) ? (byte >> 4) : (byte & 0xF);\n    double s = moe_oracle_scale",
                     "unsigned code = (k & 1) ? (byte & 0xF) : (byte >> 4);\n    double s = moe_oracle_scale"),
    "nv_block_size": ("return fmt == ORACLE_MXFP4 ? 32 : 16;", "return fmt == ORACLE_MXFP4 ? 32 : 32;"),
    "ue8m0_bias": ("return ldexp(1.0, (int)b - 127);", "return ldexp(1.0, (int)b - 128);"),
    "e4m3_bias": ("else v = ldexp(1.0 + (double)m / 8.0, e - 7);", "else v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_subnormal": ("if (e == 0) v = ldexp((double)m / 8.0, -6);", "if (e == 0) v = ldexp((double)m / 8.0, -7);"),
    "silu_sign": ("return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    "dropped_up": ("return silu(gate) * up;", "return silu(gate);"),
    "gate_up_swapped": ("return silu(gate) * up;", "return silu(up) * gate;"),
    "up_rows_offset": ("up += x[k] * weight_at(nib, sc, H, fmt, gu, I + n, k);",
                       "up += x[k] * weight_at(nib, sc, H, fmt, gu, n, k);"),
    "nv_global_swapped": ("double gg = fmt == ORACLE_NVFP4 ? (double)g13[2 * e + 0] : 1.0;\n    double gu = fmt == ORACLE_NVFP4 ? (double)g13[2 * e + 1] : 1.0;\n    double gate = 0.0",
                          "double gg = fmt == ORACLE_NVFP4 ? (double)g13[2 * e + 1] : 1.0;\n    double gu = fmt == ORACLE_NVFP4 ? (double)g13[2 * e + 0] : 1.0;\n    double gate = 0.0"),
    "down_global_dropped": ("double gd = fmt == ORACLE_NVFP4 ? (double)g2[e] : 1.0;\n    double acc = 0.0;",
                            "double gd = 1.0;\n    double acc = 0.0;"),
    "router_weight_ignored": ("double w = (double)tw[j];", "double w = 1.0;"),
    "router_weight_wrong_slot": ("double w = (double)tw[j];", "double w = (double)tw[0];"),
    "invalid_upper_bound": ("return e >= 0 && e < E;", "return e >= 0 && e <= E;"),
    "accumulate_instead_of_overwrite": ("double o = 0.0; /* overwrite", "double o = out[v]; /* overwrite"),
    "fc2_index_transposed": ("for (int n = 0; n < I; ++n) acc += weight_at(nib, sc, I, fmt, gd, m, n) * h[n];",
                             "for (int n = 0; n < I; ++n) acc += weight_at(nib, sc, I, fmt, gd, m, (n + 1) % I) * h[n];"),
    "quant_global_rule": ("volatile float six448 = 6.0f * 448.0f;", "volatile float six448 = 6.0f * 256.0f;"),
    "quant_tie_rule": ("if (d < bestd || (d == bestd && (c & 1) == 0)) {\n            bestd = d;\n            best = c;\n        }\n    }\n    if (signbit(v))",
                       "if (d <= bestd) {\n            bestd = d;\n            best = c;\n        }\n    }\n    if (signbit(v))"),
    "quant_negative_zero": ("if (signbit(v)) best |= 8;", "if (best != 0 && v < 0.0f) best |= 8;"),
    "gelu_cubic_coefficient": ("(gate + 0.044715 * gate * gate * gate)", "(gate + 0.0447 * gate * gate * gate)"),
    "gelu_half_dropped": ("return 0.5 * gate * (1.0 + tanh(", "return gate * (1.0 + tanh("),
    "swiglu_beta_multiplied": ("return (u + a->beta) * g / (1.0 + exp(-a->alpha * g));",
                               "return (u * a->beta) * g / (1.0 + exp(-a->alpha * g));"),
    "swiglu_gate_unclamped": ("double g = gate < a->limit ? gate : a->limit;", "double g = gate;"),
    "swiglu_up_clamp_dropped": ("double u = up < -a->limit ? -a->limit : (up > a->limit ? a->limit : up);",
                                "double u = up;"),
    "swiglu_alpha_outside": ("return (u + a->beta) * g / (1.0 + exp(-a->alpha * g));",
                             "return a->alpha * (u + a->beta) * g / (1.0 + exp(-g));"),
    "mxfp8_scale_floor": ("e = (m == 0.5) ? ex - 1 : ex;         /* ceil(log2(amax/448)) */",
                          "e = ex - 1;"),
    "mxfp8_scale_bias": ("s[b] = (uint8_t)(e + 127);\n        double scale = ldexp(1.0, e);",
                         "s[b] = (uint8_t)(e + 128);\n        double scale = ldexp(1.0, e);"),
    "mxfp8_sign_dropped": ("if (signbit(v)) c |= 0x80;", "if (v < 0.0f && c != 0) c |= 0x80;"),
    "mxfp8_h_unquantised": ("moe_oracle_quant_mxfp8_row(hf, I, hq, hs);\n                dequant_mxfp8_row(hq, hs, I, hd);",
                            "moe_oracle_quant_mxfp8_row(hf, I, hq, hs);\n                for (int n = 0; n < I; ++n) hd[n] = h[n];"),
    "relu2_square_dropped": ("h[n] = r * r;", "h[n] = r;"),
    "relu2_relu_dropped": ("double r = u > 0.0 ? u : 0.0;\n                    h[n] = r * r;", "double r = u;\n                    h[n] = r * r;"),
    "prefill_relu2_relu_dropped": ("double r = u > 0.0 ? u : 0.0;\n                    hf[n]", "double r = u;\n                    hf[n]"),
    "relu2_rows_shifted": ("for (int k = 0; k < H; ++k) u += x[k] * weight_at(nib, sc, H, fmt, g, n, k);",
                           "for (int k = 0; k < H; ++k) u += x[k] * weight_at(nib, sc, H, fmt, g, (n + 1) % I, k);"),
    "prefill_bf16_staging_dropped": ("hf[n] = bf16_round((float)h[n]);\n                float hG;",
                                     "hf[n] = (float)h[n];\n                float hG;"),
    "prefill_h_takes_x_multiplier": ("hf[n] = bf16_round((float)h[n]);\n                float hG;\n                moe_oracle_quant_nvfp4_row(hf, I, hq, hs, &hG);\n                dequant_nvfp4_row(hq, hs, hG, I, hd);",
                                     "hf[n] = bf16_round((float)h[n]);\n                float hG;\n                moe_oracle_quant_nvfp4_row(hf, I, hq, hs, &hG);\n                dequant_nvfp4_row(hq, hs, xG, I, hd);"),
    "prefill_h_dequant_skipped": ("hf[n] = bf16_round((float)h[n]);\n                float hG;\n                moe_oracle_quant_nvfp4_row(hf, I, hq, hs, &hG);\n                dequant_nvfp4_row(hq, hs, hG, I, hd);\n                expert_fc2(hd,",
                                  "hf[n] = bf16_round((float)h[n]);\n                float hG;\n                moe_oracle_quant_nvfp4_row(hf, I, hq, hs, &hG);\n                dequant_nvfp4_row(hq, hs, hG, I, hd);\n                expert_fc2(h,"),
    "prefill_x_multiplier_dropped": ("if (xg_out) xg_out[i] = xG;\n            dequant_nvfp4_row(xq, xs, xG, H, xd);",
                                     "if (xg_out) xg_out[i] = xG;\n            dequant_nvfp4_row(xq, xs, 1.0f, H, xd);"),
    "prefill_h_multiplier_per_token": ("hf[n] = bf16_round((float)h[n]);\n                float hG;\n                moe_oracle_quant_nvfp4_row(hf, I, hq, hs, &hG);",
                                       "hf[n] = bf16_round((float)h[n]);\n                float hG;\n                static float shared_hG;\n                moe_oracle_quant_nvfp4_row(hf, I, hq, hs, &hG);\n                if (j > 0) hG = shared_hG; else shared_hG = hG;"),
    "prefill_relu2_square_dropped": ("hf[n] = bf16_round((float)(r * r));", "hf[n] = bf16_round((float)r);"),
    "prefill_relu2_h_unquantised": ("dequant_nvfp4_row(hq, hs, hG, I, hd);\n                expert_fc2(hd, w2, s2, g2, e, H, I, fmt, y);\n                double w = (double)topk_w[(size_t)t * top_k + j];\n                for (int m = 0; m < H; ++m) o[m] += w * y[m];\n            }\n        }\n        free(xf); free(xq); free(xs); free(xd); free(hf);",
                                    "dequant_nvfp4_row(hq, hs, hG, I, hd);\n                for (int n = 0; n < I; ++n) hd[n] = hf[n];\n                expert_fc2(hd, w2, s2, g2, e, H, I, fmt, y);\n                double w = (double)topk_w[(size_t)t * top_k + j];\n                for (int m = 0; m < H; ++m) o[m] += w * y[m];\n            }\n        }\n        free(xf); free(xq); free(xs); free(xd); free(hf);"),
    "route_order": ("for (int t = 0; t < M; ++t)\n            for (int j = 0; j < top_k; ++j)\n                if (topk_ids[(size_t)t * top_k + j] == e) perm[r++] = t * top_k + j;",
                    "for (int j = 0; j < top_k; ++j)\n            for (int t = 0; t < M; ++t)\n                if (topk_ids[(size_t)t * top_k + j] == e) perm[r++] = t * top_k + j;"),
}


def _run_pins():
    """Run the pin checks; return the names of those that fail."""
    failures = []
    checks = [
        ("e2m1", pins.test_e2m1_all_codes_closed_form),
        ("ue8m0", pins.test_ue8m0_all_codes),
        ("e4m3", pins.test_e4m3_all_codes_match_library),
        ("e4m3_round", pins.test_e4m3_rounding_matches_library),
        ("e2m1_round", pins.test_e2m1_rounding_golden),
        ("dequant_mx", lambda: pins.test_dequant_structure(0)),
        ("dequant_nv", lambda: pins.test_dequant_structure(1)),
        ("quant_rules", pins.test_quant_row_global_and_scale_rules),
        ("quant_nearest", pins.test_quant_row_codes_are_nearest),
        ("route", pins.test_route_is_stable_counting_sort),
        ("top1_mx", lambda: pins.test_top1_is_gated_mlp(0)),
        ("top1_nv", lambda: pins.test_top1_is_gated_mlp(1)),
        ("gelu_mx", lambda: pins.test_top1_gelu_tanh_is_gated_mlp(0)),
        ("gelu_nv", lambda: pins.test_top1_gelu_tanh_is_gated_mlp(1)),
        ("swiglu_reductions", lambda: pins.test_swigluoai_reductions(_small_case())),
        ("swiglu_relu", lambda: pins.test_swigluoai_large_alpha_is_relu_gated(0)),
        ("swiglu_clamps", pins.test_swigluoai_hand_worked_clamps),
        ("mxfp8_library", pins.test_mxfp8_quantiser_matches_library),
        ("mxfp8_grid", pins.test_mxfp8_exact_on_grid),
        ("w4a8_golden", pins.test_w4a8_hand_worked_layer),
        ("w4a8_invariants", pins.test_w4a8_invariants_and_accuracy),
        ("w4a8_brute", pins.test_w4a8_layer_brute_force),
        ("relu2_golden", pins.test_relu2_hand_worked_layer),
        ("relu2_mlp_mx", lambda: pins.test_relu2_is_a_plain_mlp_mixture(0)),
        ("relu2_mlp_nv", lambda: pins.test_relu2_is_a_plain_mlp_mixture(1)),
        ("prefill_brute_nv", lambda: pins.test_prefill_mirror_brute_force(1)),
        ("prefill_brute_mx", lambda: pins.test_prefill_mirror_brute_force(0)),
        ("prefill_per_row_h", pins.test_prefill_mirror_quantises_h_per_routed_row),
        ("prefill_relu2_nv", lambda: pins.test_prefill_relu2_mirror_brute_force(1)),
        ("prefill_relu2_mx", lambda: pins.test_prefill_relu2_mirror_brute_force(0)),
    ]
    for case in pins._golden_cases():
        checks.append(("golden_" + case["name"], lambda c=case: pins.test_hand_worked_layers(c)))
    checks.append(("brute_mx", lambda: _brute_once(0)))
    checks.append(("brute_nv", lambda: _brute_once(1)))
    for name, fn in checks:
        try:
            fn()
        except (AssertionError, ValueError):
            failures.append(name)
    return failures


def _small_case():
    E, H, I, M, k = 6, 64, 32, 3, 4
    w = pins._tiny_weights(E, H, I, pins.gen.MXFP4, seed=21)
    x = pins.gen.draw_activations(M, H, seed=22)
    ids = np.array([[0, 3, 5, 1], [2, 2, 4, 0], [5, 1, 3, 2]], np.int32)
    tw = np.random.default_rng(23).uniform(0.05, 1.0, (M, k)).astype(np.float32)
    return E, H, I, M, k, w, x, ids, tw


def _brute_once(fmt):
    E, H, I, M, k = 3, 32, 32, 2, 3
    w = pins._tiny_weights(E, H, I, fmt, seed=99)
    x = pins.gen.draw_activations(M, H, seed=98)
    ids = np.array([[0, 2, -1], [1, 1, 3]], np.int32)
    tw = np.array([[0.3, 0.6, 0.1], [0.2, 0.5, 0.3]], np.float32)
    got = oracle.forward(x, w, ids, tw, E, H, I, k, fmt)
    want = pins._np_layer(x.to(torch.float64).numpy(), w, ids, tw, E, H, I, fmt)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12 * np.abs(want).max())


def _build_variant(tmp_path, name, src_text):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(src_text)
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
                    "-o", str(so), str(c), "-lm"], check=True)
    return str(so)


def test_unmodified_oracle_passes_all_pins():
    assert _run_pins() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutation(tmp_path, name):
    src = open(SRC).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/present"
    so = _build_variant(tmp_path, name, src.replace(old, new))
    with oracle.using_library(so):
        failed = _run_pins()
    assert failed, f"no pin caught mutation {name}"
