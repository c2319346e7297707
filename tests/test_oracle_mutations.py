"""Planted mistakes: each case copies the oracle's C source, changes one
expression into a plausible mistake (a dropped term, a wrong sign, index or
operand order), builds it on the CPU and checks that at least one pin in
``oracle_pins.py`` rejects that build. This shows the pins constrain every
part of the oracle rather than restating it."""
import os
import tempfile

import pytest

import oracle as oracle_pkg
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "moe_oracle.c")

# (name, exact text in the source, replacement). Each original must occur
# exactly once.
MUTATIONS = [
    ("silu_on_up_branch", "h[j] = silu(a) * b;", "h[j] = a * silu(b);"),
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("down_weight_transposed", "widen(wdtype, wd, (size_t)c * d_ff + j)", "widen(wdtype, wd, (size_t)j * d + c)"),
    ("gate_weight_transposed", "a += widen(wdtype, wg, (size_t)j * d + i) * x[i];", "a += widen(wdtype, wg, (size_t)i * d_ff + j) * x[i];"),
    ("router_weight_transposed", "widen(wdtype, w_router, (size_t)e * d + j)", "widen(wdtype, w_router, (size_t)j * N + e)"),
    ("tie_to_higher_index", "if (best < 0 || key[i] > key[best]) best = i;", "if (best < 0 || key[i] >= key[best]) best = i;"),
    ("softmax_sign", "p[i] = exp(r[i] - m);", "p[i] = exp(m - r[i]);"),
    ("selection_bias_in_gates", "r[e] = (double)rt[e];", "r[e] = (double)rt[e] + (sel_bias ? (double)sel_bias[e] : 0.0);"),
    ("logit_bias_dropped", "if (logit_bias) acc += logit_bias[e];", ""),
    ("no_renormalisation", "g[s] = p[idx[s]] / z;", "g[s] = p[idx[s]];"),
    ("shared_expert_dropped", "G[q] = 1.0;", "G[q] = 0.0;"),
    ("permute_descending_tokens", "for (int t = 0; t < T; ++t)\n      for (int s = 0; s < k; ++s)\n        if (topk_idx[(size_t)t * k + s] == e) {\n          int32_t pair", "for (int t = T - 1; t >= 0; --t)\n      for (int s = 0; s < k; ++s)\n        if (topk_idx[(size_t)t * k + s] == e) {\n          int32_t pair"),
    ("capacity_keeps_the_last_pairs", "for (int t = 0; t < T; ++t)\n      for (int s = 0; s < k; ++s)\n        if (topk_idx[(size_t)t * k + s] == e) {\n          keep", "for (int t = T - 1; t >= 0; --t)\n      for (int s = 0; s < k; ++s)\n        if (topk_idx[(size_t)t * k + s] == e) {\n          keep"),
    ("capacity_off_by_one", "(capacity == 0 || taken < capacity)", "(capacity == 0 || taken <= capacity)"),
    ("dropped_pair_still_runs", "if (s < k && keep && !keep[(size_t)t * k + s]) {", "if (0) {"),
    ("balance_loss_without_N", "return alpha * (double)N * s;", "return alpha * s;"),
    ("f_over_tokens_not_assignments", "f[i] = (double)counts[i] / ((double)T * (double)k);", "f[i] = (double)counts[i] / (double)T;"),
    ("gated_sum_transposed", "acc += G[i] * E[(size_t)i * dim + c];", "acc += G[i] * E[(size_t)c * n_terms + i];"),
    ("prob_sum_from_gates", "for (int e = 0; e < N; ++e) prob_sum[e] += p[e];", "for (int s = 0; s < k; ++s) prob_sum[it[s]] += topk_w[(size_t)t * k + s];"),
    ("bf16_widen_wrong_half", "uint32_t u = (uint32_t)((const uint16_t*)base)[i] << 16;", "uint32_t u = (uint32_t)((const uint16_t*)base)[i];"),
    ("order_margin_skips_last_gap", "for (int s = 0; s + 1 < m; ++s)", "for (int s = 0; s + 2 < m; ++s)"),
    ("e4m3_exponent_bias", "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    ("e4m3_ties_away_from_even", "if (d < bd || (d == bd && (c & 1) == 0)) {", "if (d <= bd) {"),
    ("e4m3_direct_no_carry", "  if (m == 8) {\n    m = 0;\n    ++E;\n  }", ""),
    ("fp8_scale_over_240", "const float s = amax / 448.0f;", "const float s = amax / 240.0f;"),
    ("fp8_codes_over_240", "const float inv = amax > 0.0f ? 448.0f / amax : 0.0f;", "const float inv = amax > 0.0f ? 240.0f / amax : 0.0f;"),
    ("fp8_h_not_quantized", "(oracle_e4m3_decode(hq[j]) * (double)hs);", "(double)h[j];"),
    ("e2m1_exponent_bias", "ldexp(1.0 + 0.5 * m, e - 1);", "ldexp(1.0 + 0.5 * m, e - 2);"),
    ("e2m1_ties_away_from_even", "if (d < bd || (d == bd && !(c & 1))) {", "if (d <= bd) {"),
    ("e2m1_direct_no_saturation", "c = a >= 6.0 ? 7 : 6 + (int)rint(0.5 * (a - 4.0));", "c = 6 + (int)rint(0.5 * (a - 4.0));"),
    ("e2m1_direct_truncates", "c = 4 + (int)rint(a - 2.0);", "c = 4 + (int)floor(a - 2.0);"),
    ("nvfp4_block_scale_from_row_amax", "oracle_e4m3_encode(bmax * to_block) : 0;", "oracle_e4m3_encode(amax * to_block) : 0;"),
    ("nvfp4_row_scale_over_448", "scale[r] = amax / 2688.0f;", "scale[r] = amax / 448.0f;"),
    ("nvfp4_codes_over_448", "const float to_code = amax > 0.0f ? 2688.0f / amax : 0.0f;", "const float to_code = amax > 0.0f ? 448.0f / amax : 0.0f;"),
    ("nvfp4_value_without_block_scale", "return oracle_e2m1_decode(q[r * cols + c]) * oracle_e4m3_decode(bs[r * (cols / 16) + c / 16]) *", "return oracle_e2m1_decode(q[r * cols + c]) *"),
    ("nvfp4_h_not_quantized", "             nvfp4_value(hq, hb, &hs, d_ff, 0, j);", "             (double)h[j];"),
    ("nvfp4_token_not_quantized", "for (int i = 0; i < d; ++i) xt[i] = nvfp4_value(xq, xb, &xs, d, 0, i);", "for (int i = 0; i < d; ++i) xt[i] = widen(xdtype, x, (size_t)t * d + i);"),
    ("nvfp4_sign_dropped", "const uint8_t sign = signbit(v) ? 8 : 0;\n  const double a = fabs((double)v);\n  int c;", "const uint8_t sign = 0;\n  const double a = fabs((double)v);\n  int c;"),
    ("fp8_wrong_weight_row_scale", "out[c] = acc * (double)q->ds[c];", "out[c] = acc * (double)q->ds[d - 1 - c];"),
    ("reroute_tie_to_higher_index", "if (best < 0 || key > best_key) {", "if (best < 0 || key >= best_key) {"),
    ("reroute_accepts_descending_pairs", "for (size_t p = 0; p < P; ++p) {\n      const int e = prop[p];", "for (size_t p = P; p-- > 0;) {\n      const int e = prop[p];"),
    ("reroute_ignores_held_experts", "if (held[(size_t)t * N + e] || room[e] <= 0 || tried[e]) continue;", "if (room[e] <= 0 || tried[e]) continue;"),
    ("reroute_slots_propose_the_same_expert", "if (held[(size_t)t * N + e] || room[e] <= 0 || tried[e]) continue;", "if (held[(size_t)t * N + e] || room[e] <= 0) continue;"),
    ("reroute_ignores_selection_bias", "float key = sel_bias ? (float)((double)r + (double)sel_bias[e]) : r;", "float key = r;"),
    ("reroute_nan_not_lowest", "if (isnan(key)) key = -INFINITY;", ""),
    ("reroute_accepts_up_to_capacity", "if (taken[e] < room[e]) {", "if (taken[e] < capacity) {"),
    ("reroute_room_not_spent", "for (int e = 0; e < N; ++e) room[e] -= taken[e];", ""),
    ("reroute_without_cut", "  /* round 0: the capacity cut */\n  oracle_capacity_keep(T, k, N, topk_idx, capacity, keep);", "  /* round 0: the capacity cut */\n  oracle_capacity_keep(T, k, N, topk_idx, 0, keep);"),
    ("reroute_accepted_expert_not_held", "        held[(p / k) * N + e] = 1;\n        taken[e] += 1;", "        taken[e] += 1;"),
    ("bwd_reroute_ignored", "    return R->run[q];", "    return R->idx[q];"),
    ("selection_ignores_bias", "key[e] = sel_bias ? (float)((double)rt[e] + (double)sel_bias[e]) : rt[e];", "key[e] = rt[e];"),
    ("bwd_silu_grad_missing_term", "return s * (1.0 + z * (1.0 - s));", "return s;"),
    ("bwd_db_uses_silu_grad", "db[j] = dh * silu(a[j]);", "db[j] = dh * silu_grad(a[j]);"),
    ("bwd_gate_grad_from_weighted_output", "dG += dyt[c] * o;", "dG += dyt[c] * o * G;"),
    ("bwd_balance_sign", "for (int i = 0; i < N; ++i) dr[i] += scale * p[i] * (f[i] - pf);", "for (int i = 0; i < N; ++i) dr[i] -= scale * p[i] * (f[i] - pf);"),
    ("bwd_balance_not_centred", "dr[i] += scale * p[i] * (f[i] - pf);", "dr[i] += scale * p[i] * f[i];"),
    ("bwd_renorm_not_centred", "dp[idx[s]] = (dG[s] - gdG) / Z;", "dp[idx[s]] = dG[s] / Z;"),
    ("bwd_dx_without_router_term", "        acc += DR[(size_t)t * N + e] * widen(wdtype, w_router, (size_t)e * d + i);\n      dx[(size_t)t * d + i] = acc;", "      dx[(size_t)t * d + i] = acc;"),
    ("bwd_down_grad_from_da", "rd[j] += DO[q * d + c] * H[q * d_ff + j];", "rd[j] += DO[q * d + c] * DA[q * d_ff + j];"),
    ("bwd_gate_grad_transposed", "acc += widen(wdtype, wg, (size_t)j * d + i) * da[j] +", "acc += widen(wdtype, wu, (size_t)j * d + i) * da[j] +"),
]


def _all_pins_pass(o):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except Exception as e:  # a crash in a mutant counts as a failed pin
            failed.append((pin.__name__, type(e).__name__))
    return failed


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} must occur exactly once"
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "mutant.c")
        so = os.path.join(tmp, "libmutant.so")
        with open(c, "w") as f:
            f.write(src.replace(old, new))
        oracle_pkg.compile_oracle(c, so)
        o = oracle_pkg.Oracle(oracle_pkg.load(so))
        failed = _all_pins_pass(o)
    assert failed, f"no pin caught the planted mistake {name}"
