"""The oracle's pins catch plausible mistakes: each case plants one error in a copy
of oracle.c (on the CPU), builds it, and runs the oracle pin tests against it; at
least one pin must fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = ["test_oracle_conversions.py", "test_oracle_router.py", "test_oracle_sigmoid.py",
        "test_oracle_topk.py", "test_oracle_lists.py", "test_oracle_mxfp8.py", "test_oracle_finalize.py",
        "test_oracle_front.py", "test_oracle_units.py", "test_oracle_norm.py"]

MUTATIONS = {
    "router_wrong_row": ("const uint16_t* wr = w + (size_t)e * H;\n      for", "const uint16_t* wr = w + (size_t)(e ? e - 1 : 0) * H;\n      for"),
    "exp_degree6": ("float p = INV_FACT[7];\n  for (int i = 6;", "float p = INV_FACT[6];\n  for (int i = 5;"),
    "exp_no_lo_part": ("r = fmaf(-n, LN2_LO, r);", "r = r;"),
    "sigmoid_sign": ("float e = oracle_exp_spec(-x);", "float e = oracle_exp_spec(x);"),
    "topk_tie_high_index": ("  return ia < ib;\n}", "  return ia > ib;\n}"),
    "topk_weights_biased": ("for (int k = 0; k < K; ++k) S = S + s[id[k]];", "for (int k = 0; k < K; ++k) S = S + c[id[k]];"),
    "topk_no_bias": ("c[e] = bias ? s[e] + bias[e] : s[e];", "c[e] = s[e];"),
    "topk_scale_before": ("wk = (S == 0.0f) ? 0.0f : s[id[k]] / S;", "wk = (S == 0.0f) ? 0.0f : (s[id[k]] * scale) / S;"),
    "lists_slot_major": ("for (int t = 0; t < T; ++t)\n    for (int k = 0; k < K; ++k) {\n      int e = ids[(size_t)t * K + k];",
                         "for (int k = 0; k < K; ++k)\n    for (int t = 0; t < T; ++t) {\n      int e = ids[(size_t)t * K + k];"),
    "lists_inclusive_scan": ("offsets[e + 1] = offsets[e] + fill[e];", "offsets[e + 1] = offsets[e] + fill[e] + (e == 0);"),
    "mx_scale_off_by_one": ("int se = bf16_floor_log2(amax_bits) - 8;", "int se = bf16_floor_log2(amax_bits) - 7;"),
    "mx_round_half_up": ("  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;", "  return f + 1.0;"),
    "mx_saturate_to_nan": ("if (a > 448.0) return sign | 0x7E;", "if (a > 448.0) return sign | 0x7F;"),
    "mx_subnormal_step": ("double m = rne_nonneg(a * 512.0);", "double m = rne_nonneg(a * 256.0);"),
    "fin_reverse_k": ("for (int k = 0; k < K; ++k) {\n        if (idx[k] == -1) continue;\n        acc = fmaf(w[k],",
                      "for (int k = K - 1; k >= 0; --k) {\n        if (idx[k] == -1) continue;\n        acc = fmaf(w[k],"),
    "fin_mul_add": ("acc = fmaf(w[k], bf16_to_f32(rows[(size_t)idx[k] * H + c]), acc);",
                    "acc = acc + w[k] * bf16_to_f32(rows[(size_t)idx[k] * H + c]);"),
    "fin_no_scale": ("if (scale != 1.0f) wk = wk * scale;\n      if (r == -1)", "if (r == -1)"),
    "fin_shared_twice": ("if (shared) acc = acc + bf16_to_f32(shared[(size_t)t * H + c]);",
                         "if (shared) acc = acc + 2.0f * bf16_to_f32(shared[(size_t)t * H + c]);"),
    "bf16_truncate": ("  u += 0x7FFFu + lsb;", "  u += 0u * lsb;"),
    "f64_bf16_via_f32": ("const double r = nearbyint(a / step) * step;", "const double r = (double)(float)a;"),
    "f64_bf16_nine_bits": ("const double step = ldexp(1.0, lead - 7);", "const double step = ldexp(1.0, lead - 8);"),
    "units_len_full": ("if (len > window) len = window;", "len = window;"),
    "units_one_per_expert": ("pos += window) {", "pos += window + offsets[e + 1]) {"),
    "norm_sum_not_mean": ("const double inv = 1.0 / sqrt(ss / (double)H + eps);", "const double inv = 1.0 / sqrt(ss + eps);"),
    "norm_eps_outside": ("const double inv = 1.0 / sqrt(ss / (double)H + eps);", "const double inv = 1.0 / (sqrt(ss / (double)H) + eps);"),
    "norm_no_gamma": ("* inv * (double)bf16_to_f32(g[c]);", "* inv;"),
    "mx_ceil_always_up": ("if (rule == 1 && (double)amax > ldexp(448.0, se)) se += 1;", "if (rule == 1) se += 1;"),
    "mx_tiles_line_swap": ("out[tile * 512 + 16 * (rr % 32) + 4 * (rr / 32) + cc]", "out[tile * 512 + 4 * (rr % 32) + 16 * (rr / 32) + cc]"),
    "mx_tiles_column_major": ("const size_t tile = (size_t)(r / 128) * ct + (size_t)(c / 4);",
                              "const size_t tile = (size_t)(c / 4) * ((size_t)(rows + 127) / 128) + (size_t)(r / 128);"),
    "mx_ceil_at_448": ("if (rule == 1 && (double)amax > ldexp(448.0, se)) se += 1;",
                       "if (rule == 1 && (double)amax >= ldexp(448.0, se)) se += 1;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/absent: {name}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", str(mutated), "-o", str(lib), "-lm"])
    env = dict(os.environ, MOE_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       cwd=os.path.join(ROOT, "tests"), env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"no pin caught mutation {name}:\n{r.stdout[-2000:]}"
