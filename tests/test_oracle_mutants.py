"""Plant plausible mistakes in copies of the oracle's C source (on the CPU, in a temp directory) and
check that at least one pin catches each: a dropped term, a wrong sign, a wrong index, a transposed
operand, a flipped tie rule, an off-by-one.  The real oracle is untouched."""
import os

import pytest

import oracle
from tests.oracle_pins import ALL_PINS

# (name, text in moe_oracle.c, replacement)
MUTANTS = [
    ("noisy_sign", "s += (double)eps[(size_t)t * E + e] * softplus(noise);",
     "s -= (double)eps[(size_t)t * E + e] * softplus(noise);"),
    ("softplus_drops_log1p", "return log1p(exp(z));", "return exp(z);"),
    ("gelu_missing_sqrt2", "erf(z / sqrt(2.0))", "erf(z)"),
    ("tie_to_higher_id", "if (best < 0 || s[e] > s[best]) best = e;", "if (best < 0 || s[e] >= s[best]) best = e;"),
    ("topk_norm_over_all", "if (norm == NORM_ALL) {", "if (1) {"),
    ("all_norm_over_topk", "for (int e = 0; e < E; ++e) den += exp(s[e] - m);",
     "for (int e = 0; e < k; ++e) den += exp(s[idx[(size_t)t * k + e]] - m);"),
    ("capacity_floor", "return (int)ceil(", "return (int)floor("),
    ("keep_one_too_many", "slot[(size_t)t * k + j] = pos < C ? pos : -1;", "slot[(size_t)t * k + j] = pos <= C ? pos : -1;"),
    ("rank_major_slots", "    for (int t = 0; t < T; ++t) {\n        for (int j = 0; j < k; ++j) {\n            int e = idx",
     "    for (int j = 0; j < k; ++j) {\n        for (int t = 0; t < T; ++t) {\n            int e = idx"),
    ("count_only_kept", "int pos = count[e]++;", "int pos = count[e]; if (pos < C) count[e]++;"),
    ("rank_priority_in_token_order", "        for (int r = 0; r < k; ++r)\n            for (int tok = 0; tok < T; ++tok) {",
     "        for (int tok = 0; tok < T; ++tok)\n            for (int r = 0; r < k; ++r) {"),
    ("rank_priority_keeps_one_too_many", "slot[i] = q < C ? q : -1;", "slot[i] = q <= C ? q : -1;"),
    ("rank_priority_ignored", "if (priority == PRIORITY_RANK) {", "if (0) {"),
    ("cosine_no_emb_norm", "if (ne < 1e-12) ne = 1e-12;", "ne = 1.0;"),
    ("cosine_times_temperature", "num / (nu * ne) / temperature", "num / (nu * ne) * temperature"),
    ("cosine_emb_transposed", "elem(emb, (size_t)e * (size_t)p + (size_t)j, dtype)",
     "elem(emb, (size_t)j * (size_t)E + (size_t)e, dtype)"),
    ("dot_off_by_one", "for (int i = 0; i < n; ++i)\n        s += elem(a", "for (int i = 0; i < n - 1; ++i)\n        s += elem(a"),
    ("gate_reads_token0", "double s = dot_rows(x, xo, dtype, w_gate", "double s = dot_rows(x, 0, dtype, w_gate"),
    ("b1_dropped", "if (b1) z += elem(b1,", "if (0) z += elem(b1,"),
    ("b2_dropped", "if (b2) z += elem(b2,", "if (0) z += elem(b2,"),
    ("w2_transposed", "elem(w2, w2_off + (size_t)n * (size_t)h + (size_t)i, wdtype)",
     "elem(w2, w2_off + (size_t)i * (size_t)d + (size_t)n, wdtype)"),
    ("w1_reads_x_dtype", "w1_off + (size_t)n * (size_t)d, wdtype, d);", "w1_off + (size_t)n * (size_t)d, dtype, d);"),
    ("gelu_grad_drops_density", " + z * exp(-0.5 * z * z) / sqrt(2.0 * pi);", ";"),
    ("topk_gate_grad_sign", "gate[(size_t)t * k + j] * (dg[j] - sum);", "gate[(size_t)t * k + j] * (sum - dg[j]);"),
    ("dropped_pair_gets_gradient", "            dg[j] = 0.0;\n            if (slot[i] < 0) continue;",
     "            dg[j] = 0.0;"),
    ("noisy_grad_without_eps", "ds[e] * (double)eps[(size_t)t * E + e] * sigmoid(nl)", "ds[e] * sigmoid(nl)"),
    ("dw2_from_preactivation", "dw2[(e * d + m) * (size_t)h + n] += dy * a[n];", "dw2[(e * d + m) * (size_t)h + n] += dy * z[n];"),
    ("all_norm_grad_drops_softmax", "((e == idx[(size_t)t * k + j] ? 1.0 : 0.0) - p[e])",
     "(e == idx[(size_t)t * k + j] ? 1.0 : 0.0)"),
    ("dx_misses_gate_path", "gx[m] += ds[e] * elem(w_gate,", "gx[m] += 0.0 * elem(w_gate,"),
    ("fp8_exponent_bias_8", "mag = ldexp(1.0 + (double)man / 8.0, ex - 7);", "mag = ldexp(1.0 + (double)man / 8.0, ex - 8);"),
    ("fp8_subnormal_as_normal", "mag = ldexp((double)man / 8.0, -6);", "mag = ldexp(1.0 + (double)man / 8.0, -7);"),
    ("fp8_sign_dropped", "return sign ? -mag : mag;", "return mag;"),
    ("fp8_scale_block_transposed", "scale[(size_t)(r / block) * sc + (c / block)]",
     "scale[(size_t)(c / block) * sc + (r / block)]"),
    ("combine_drops_gate", "o[n] += g * y[n];", "o[n] += y[n];"),
    ("combine_keeps_dropped", "if (slot[(size_t)t * k + j] < 0) continue;", ""),
    ("std_over_n", "0.1 * sqrt(ss / (double)(E - 1))", "0.1 * sqrt(ss / (double)E)"),
    ("importance_counts_pairs", "importance[idx[i]] += gate[i];", "importance[idx[i]] += 1.0;"),
    ("drops_counts_kept", "if (slot && slot[i] < 0) ++drops;", "if (slot && slot[i] >= 0) ++drops;"),
    ("bf16_widening_wrong_half", "uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;",
     "uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 15;"),
    ("sampled_dw1_drops_gelu_grad", "const double dzn = dan * gelu_grad(zn);", "const double dzn = dan;"),
    ("sampled_dw2_drops_gate", "const double dy = gate[q] * dout[xo + m];", "const double dy = dout[xo + m];"),
    ("sampled_dx_noise_sign", "for (int m = 0; m < d; ++m) gx[m] += dn * elem(w_noise, (size_t)e * d + m, dtype);",
     "for (int m = 0; m < d; ++m) gx[m] -= dn * elem(w_noise, (size_t)e * d + m, dtype);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, "mutation site of %s not found exactly once" % name
    path = os.path.join(tmp_path, "mutant.c")
    open(path, "w").write(src.replace(old, new))
    o = oracle.Oracle(oracle.compile_source(path, os.path.join(tmp_path, "mutant.so")))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "no pin catches the planted mistake %s" % name
