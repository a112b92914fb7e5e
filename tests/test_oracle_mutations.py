"""The oracle's pins are strong enough: plant plausible mistakes in copies of the
oracle (on the CPU only) and check that at least one pin fails for each.

Each mutant is compiled from a string-edited copy of ``oracle/oracle.c`` into a
temporary library; the pin functions of ``test_oracle_pins`` run against it.
"""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_backward_pins as bwd
import test_oracle_fp8_pins as fp8
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "silu_on_up_projection": ("silu(gate) * up", "silu(up) * gate"),
    "w3_transposed": ("elem(w3, base3 + (size_t)i * c + j, wdt)", "elem(w3, base3 + (size_t)j * d + i, wdt)"),
    "ties_to_higher_index": ("if (best < 0 || z[j] > z[best]) best = j;", "if (best < 0 || z[j] >= z[best]) best = j;"),
    "renorm_over_all_experts": ("for (int s = 0; s < k; ++s) den += exp(z[e[s]] - zmax);",
                                "for (int j = 0; j < E; ++j) den += exp(z[j] - zmax);"),
    "sigmoid_norm_unnormalised": ("w[s] = sigmoid(z[e[s]]) / den;", "w[s] = sigmoid(z[e[s]]);"),
    "bias_dropped": ("if (bias) acc += (double)bias[j];", ""),
    "partial_wiring_uses_o_k": ("if (wiring == ORACLE_WIRE_PARTIAL) nxt = os_k;", "if (wiring == ORACLE_WIRE_PARTIAL) nxt = o_k;"),
    "outdated_wiring_uses_o_star": ("else if (wiring == ORACLE_WIRE_OUTDATED) nxt = o_km1;",
                                    "else if (wiring == ORACLE_WIRE_OUTDATED) nxt = os_k;"),
    "o_star_without_shared": ("o_star[(size_t)t * d + i] = oracle_round(op + sv, out_storage);",
                              "o_star[(size_t)t * d + i] = oracle_round(op, out_storage);"),
    "gate_weight_dropped": ("for (int i = 0; i < d; ++i) R[i] += w * oracle_round(y[i], cfg->storage);",
                            "for (int i = 0; i < d; ++i) R[i] += oracle_round(y[i], cfg->storage);"),
    "dispatch_unstable": ("for (int t = 0; t < T; ++t) {\n        for (int s = 0; s < k; ++s) {\n            int e = topk_idx[(size_t)t * k + s];\n            int p = cursor[e]++;",
                          "for (int t = T - 1; t >= 0; --t) {\n        for (int s = 0; s < k; ++s) {\n            int e = topk_idx[(size_t)t * k + s];\n            int p = cursor[e]++;"),
    "combine_weight_dropped": ("r += (double)topk_w[(size_t)t * k + s] * elem(y_perm, p * d + i, in_dtype);",
                               "r += elem(y_perm, p * d + i, in_dtype);"),
    "rounding_ties_away": ("double r = nearbyint(x / q) * q;", "double r = round(x / q) * q;"),
    "attn_mlp_input_misses_routed": ("for (size_t i = 0; i < n; ++i) ubuf[i] = oracle_round(o_k[i], cfg->storage);\n                a_in = abuf;",
                                     "for (size_t i = 0; i < n; ++i) ubuf[i] = oracle_round(os_k[i], cfg->storage);\n                a_in = abuf;"),
    "attn_output_dropped": ("double op = o_prev[(size_t)t * d + i] + (extra ? extra[(size_t)t * d + i] : 0.0);",
                            "double op = o_prev[(size_t)t * d + i];"),
    "hidden_storage_rounding_dropped": (
        "h[j] = oracle_round(silu(gate) * up, storage);\n    }\n    for (int i = 0; i < d; ++i) {\n        double acc = 0.0;\n        for (int j = 0; j < c; ++j) acc += h[j]",
        "h[j] = silu(gate) * up;\n    }\n    for (int i = 0; i < d; ++i) {\n        double acc = 0.0;\n        for (int j = 0; j < c; ++j) acc += h[j]"),
    "routed_output_storage_rounding_dropped": (
        "for (int i = 0; i < d; ++i) R[i] += w * oracle_round(y[i], cfg->storage);",
        "for (int i = 0; i < d; ++i) R[i] += w * y[i];"),
    "shared_sum_rounded_per_expert": ("for (int i = 0; i < d; ++i) S[i] += y[i];",
                                      "for (int i = 0; i < d; ++i) S[i] += (sh == 0 ? y[i] : 0.0);"),
    # FP8 expert path
    "e4m3_without_subnormal_floor": ("    if (lead < -6) lead = -6;       /* below the smallest normal 2^-6 the quantum stays 2^-9 */\n", ""),
    "e4m3_ties_away": ("double r = nearbyint(a / q) * q; /* ties to even */", "double r = round(a / q) * q;"),
    "fp8_scale_search_starts_high": ("int s = e - 10;", "int s = e - 8;"),
    "fp8_scale_boundary_exclusive": ("while (amax > ldexp(448.0, s)) ++s;", "while (amax >= ldexp(448.0, s)) ++s;"),
    "fp8_hidden_not_quantised": ("    quant_blocks(hq, c, bc, NULL, NULL);\n", ""),
    "fp8_gate_uses_up_row_exponent": ("const int eg = e2[(size_t)j * nbd + b], eu = e1[(size_t)j * nbd + b];",
                                      "const int eg = e1[(size_t)j * nbd + b], eu = e1[(size_t)j * nbd + b];"),
    "fp8_down_exponent_by_column": ("const int ed = e3[(size_t)i * nbc + b];",
                                    "const int ed = e3[(size_t)((int)b * bc % d) * nbc + b];"),
    "fp8_token_row_not_quantised_in_block": ("            quant_blocks(aq, d, fp8_blk(cfg, d), NULL, NULL);\n", ""),
    "fp8_shared_down_read_as_one_matrix": ("size_t off = base3 + (size_t)(jj / cw) * d * cw + (size_t)i * cw + (size_t)(jj % cw);",
                                           "size_t off = base3 + (size_t)i * c + (size_t)jj;"),
    "fp8_shared_down_exponent_first_expert": ("                    const int sh = jj / cs, j = jj % cs;",
                                              "                    const int sh = 0, j = jj % cs;"),
    # block-scaled (MX) FP8
    "mx_blocks_of_16": ("#define ORACLE_MX_BLOCK 32", "#define ORACLE_MX_BLOCK 16"),
    "mx_weight_row_uses_first_block_exponent": ("const int eg = e2[(size_t)j * nbd + b], eu = e1[(size_t)j * nbd + b];",
                                                "const int eg = e2[(size_t)j * nbd + b], eu = e1[(size_t)j * nbd];"),
    "mx_hidden_row_scaled": ("    quant_blocks(hq, c, bc, NULL, NULL);\n", "    quant_blocks(hq, c, c, NULL, NULL);\n"),
    "mx_token_row_scaled_in_block": ("            quant_blocks(aq, d, fp8_blk(cfg, d), NULL, NULL);\n",
                                     "            quant_blocks(aq, d, d, NULL, NULL);\n"),
    # backward
    "bwd_silu_grad_sign": ("return sg * (1.0 + g * (1.0 - sg));", "return sg * (1.0 - g * (1.0 - sg));"),
    "bwd_dg_without_up": ("dg[jj] = oracle_round(dh * a[jj] * silu_grad(g[jj]), storage);",
                          "dg[jj] = oracle_round(dh * silu_grad(g[jj]), storage);"),
    "bwd_dy_without_gate_weight": ("for (int i = 0; i < d; ++i) dy[i] = oracle_round(w[ts] * dR[i], st);",
                                   "for (int i = 0; i < d; ++i) dy[i] = oracle_round(dR[i], st);"),
    "bwd_renorm_without_normaliser_term": ("for (int r = 0; r < k; ++r) dz[e[r]] = w[r] * (dw[r] - c);",
                                           "for (int r = 0; r < k; ++r) dz[e[r]] = w[r] * dw[r];"),
    "bwd_softmax_without_other_experts": ("for (int j = 0; j < E; ++j) dz[j] = -c * exp(z[j] - zmax) / den;",
                                          "for (int j = 0; j < E; ++j) dz[j] = 0.0;"),
    "bwd_sigmoid_norm_without_den": ("dz[e[r]] = (dw[r] - c) / den * sg * (1.0 - sg);",
                                     "dz[e[r]] = (dw[r] - c) * sg * (1.0 - sg);"),
    "bwd_gate_up_swapped_in_dx": (
        "acc += dg[j] * elem(w2, base12 + (size_t)j * d + i, wdt) + da[j] * elem(w1, base12 + (size_t)j * d + i, wdt);",
        "acc += dg[j] * elem(w1, base12 + (size_t)j * d + i, wdt) + da[j] * elem(w2, base12 + (size_t)j * d + i, wdt);"),
    "bwd_partial_grad_to_o": ("else if (wiring == ORACLE_WIRE_PARTIAL) target = gos + n * (b - 1);",
                              "else if (wiring == ORACLE_WIRE_PARTIAL) target = go + n * (b - 1);"),
    "bwd_outdated_grad_one_block_late": ("else if (wiring == ORACLE_WIRE_OUTDATED) target = go + n * (b - 2);",
                                         "else if (wiring == ORACLE_WIRE_OUTDATED) target = go + n * (b - 1);"),
    "bwd_shared_without_dOs": ("double dsv = dO[(size_t)t * d + i] + (dOs ? dOs[(size_t)t * d + i] : 0.0);",
                               "double dsv = dO[(size_t)t * d + i];"),
    "bwd_router_input_grad_dropped": ("                dut[i] += acc;\n", ""),
    "bwd_wgrad_wrong_token": ("const double* x = u + (ts / k) * d;", "const double* x = u + (ts % n_tok) * d;"),
    "bwd_slots_not_summed": ("for (int i = 0; i < d; ++i) dut[i] += oracle_round(dx[i], st);",
                             "for (int i = 0; i < d; ++i) dut[i] = oracle_round(dx[i], st);"),
}

PIN_TESTS = [
    lambda: [pins.test_golden_gates(g) for g in ("softmax", "softmax_renorm", "sigmoid", "sigmoid_norm")],
    pins.test_golden_tie_and_bias,
    pins.test_golden_mlp,
    pins.test_golden_dispatch,
    pins.test_golden_rounding,
    pins.test_golden_storage_roundings,
    lambda: [pins.test_router_vs_library(g) for g in ("softmax", "softmax_renorm", "sigmoid", "sigmoid_norm")],
    pins.test_dispatch_vs_library,
    lambda: [pins.test_brute_force_dense_moe(g) for g in ("softmax", "softmax_renorm", "sigmoid", "sigmoid_norm")],
    pins.test_tp_slice_identity,
    lambda: [pins.test_telescoping_and_wiring(w) for w in ("partial", "outdated", "disabled")],
    pins.test_disabled_is_plain_recurrence_and_L1_agrees,
    lambda: [pins.test_dispatch_combine_round_trip(k, w) for k, w in ((1, 1.0), (2, 0.5), (4, 0.25))],
    pins.test_attn_farskip_wiring_identities,
    pins.test_attn_plain_is_the_ordinary_layer,
    fp8.test_every_e4m3_code_is_a_fixed_point,
    fp8.test_e4m3_rounding_matches_the_library,
    fp8.test_row_scales_brute_force,
    fp8.test_gate_up_reduces_to_exact_on_representable_operands,
    fp8.test_down_projection_reduces_to_the_quantised_hidden,
    fp8.test_down_projection_with_representable_weights_is_a_matmul_of_the_quantised_hidden,
    fp8.test_block_sums_are_the_per_row_fp8_experts,
    fp8.test_mx_block_scales_brute_force,
    fp8.test_mx_gate_up_reduces_to_exact_on_representable_operands,
    fp8.test_mx_down_projection_is_a_matmul_of_the_block_quantised_hidden,
    lambda: [fp8.test_mx_block_sums_are_the_per_row_mx_experts(w) for w in (False, True)],
    lambda: [fp8.test_mx_expert_matches_a_library_form_on_a_wide_dynamic_range(l)
             for l in ("across_blocks", "within_blocks")],
    lambda: [bwd.test_stack_backward_finite_differences_wirings(w) for w in ("partial", "outdated", "disabled")],
    lambda: [bwd.test_stack_backward_finite_differences_gates(g) for g in ("softmax", "softmax_renorm", "sigmoid",
                                                                          "sigmoid_norm")],
    bwd.test_stack_backward_finite_differences_no_shared_top1,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: %s" % name
    mut = src.replace(old, new)
    cpath = tmp_path / "oracle_mut.c"
    cpath.write_text(mut)
    so = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-std=c11", "-shared", "-fPIC",
                           "-I", os.path.dirname(SRC), "-o", str(so), str(cpath), "-lm"])
    mutant = ctypes.CDLL(str(so))
    mutant.oracle_round.restype = ctypes.c_double
    mutant.oracle_round.argtypes = [ctypes.c_double, ctypes.c_int]
    saved = oracle.lib()
    oracle._lib = mutant
    caught = []
    try:
        for t in PIN_TESTS:
            try:
                t()
            except (AssertionError, RuntimeError):
                caught.append(t)
    finally:
        oracle._lib = saved
    assert caught, "no pin catches the mutant %s" % name
