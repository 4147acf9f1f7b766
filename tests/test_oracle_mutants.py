"""Planted mistakes in the oracle must each fail at least one pin (CPU only).

Every mutant is a copy of ``oracle/gq_oracle.c`` with one plausible mistake --
a dropped term, a wrong sign, index or rounding rule -- compiled to a temporary
library.  The pins of ``oracle_pins.py`` run against it, and at least one must
fail.  The real oracle is never modified.
"""
import functools

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "tie_to_odd": ("c = (lo % 2 == 0) ? lo : hi;", "c = (lo % 2 == 0) ? hi : lo;"),
    "ties_away": ("c = (lo % 2 == 0) ? lo : hi;", "c = hi;"),
    "no_saturation": ("return (uint8_t)(sign | 0x7E);\n  /* invariant",
                      "return (uint8_t)(sign | 0x7F);\n  /* invariant"),
    "eps_dropped": ("float d = amax > GQO_EPS ? amax : GQO_EPS;",
                    "float d = amax > 0.0f ? amax : 1.0f;"),
    "eps_wrong": ("#define GQO_EPS 1e-12f", "#define GQO_EPS 1e-6f"),
    "reciprocal_scale": ("return GQO_FP8_MAX / d;", "return d / GQO_FP8_MAX;"),
    "zero_sign_dropped": ("return (uint8_t)(sign | c);",
                          "return (uint8_t)(c == 0 ? 0 : (sign | c));"),
    "subnormal_exponent": ("mag = ldexp((double)m, -9);",
                           "mag = ldexp((double)m, -10);"),
    "exponent_bias": ("mag = ldexp(1.0 + m / 8.0, e - 7);",
                      "mag = ldexp(1.0 + m / 8.0, e - 8);"),
    "product_via_reciprocal": (
        "float v = gqo_bf16_to_float(x_bf16) * scale;",
        "float v = gqo_bf16_to_float(x_bf16) / (1.0f / scale);"),
    "group_start_off_by_one": ("start[g] = prev;",
                               "start[g] = prev + (g > 0 ? 1 : 0);"),
    "no_running_max": ("if (e < prev) e = prev;", ""),
    "amax_without_abs": (
        "float a = fabsf(gqo_bf16_to_float(x[r * K + k]));",
        "float a = gqo_bf16_to_float(x[r * K + k]);"),
    "amax_whole_column": ("for (r = start[g]; r < end[g]; ++r)\n      for (k = 0; k < K; ++k) {\n        float a",
                          "for (r = 0; r < M; ++r)\n      for (k = 0; k < K; ++k) {\n        float a"),
    "colwise_scale_of_group0": (
        "q[r * K + k] = gqo_quant(x[r * K + k], scales[(int64_t)g * K + k]);",
        "q[r * K + k] = gqo_quant(x[r * K + k], scales[k]);"),
    "rowwise_not_transposed": ("qt[m * N + n] = gqo_quant(a[n * Mg + m], s);",
                               "qt[n * Mg + m] = gqo_quant(a[n * Mg + m], s);"),
    "rowwise_scale_layout": ("scales[n * n_groups + g] = s;",
                             "scales[g * N + n] = s;"),
    "pow2_rounds_up": ("return ldexpf(1.0f, e - 1);", "return ldexpf(1.0f, e);"),
    "mx_floor_off_by_one": ("E = (e - 1) - 8;", "E = e - 8;"),
    "mx_rceil_as_floor": ("E = (frexpf(v, &e) == 0.5f) ? e - 1 : e;",
                          "frexpf(v, &e); E = e - 1;"),
    "mx_zero_block": ("if (amax == 0.0f) return -127;", "if (amax == 0.0f) return 0;"),
    "expert_amax_ignores_expert": ("float a = fabsf(gqo_bf16_to_float(w[(e * K + k) * N + n]));",
                                   "float a = fabsf(gqo_bf16_to_float(w[k * N + n]));"),
    "expert_rowwise_amax_of_first_row": ("float a = fabsf(gqo_bf16_to_float(w[row + k]));",
                                         "float a = fabsf(gqo_bf16_to_float(w[e * N * K + k]));"),
    "expert_rowwise_scale_of_previous_row": ("for (k = 0; k < K; ++k) q[row + k] = gqo_quant(w[row + k], s);",
                                             "for (k = 0; k < K; ++k) q[row + k] = gqo_quant(w[row + k], n ? scales[e * N + n - 1] : s);"),
    "wgrad_drops_last_token": ("for (t = start[g]; t < end[g]; ++t)\n      for (n = 0; n < N; ++n) {",
                               "for (t = start[g]; t + 1 < end[g]; ++t)\n      for (n = 0; n < N; ++n) {"),
    "wgrad_operand_transposed": ("const double a = dec[qa_t[t * N + n]];",
                                 "const double a = dec[qa_t[n * T + t]];"),
    "wgrad_scale_of_wrong_group": ("(double)sa[n * n_groups + g]",
                                   "(double)sa[n * n_groups + (g > 0 ? g - 1 : 0)]"),
    "wgrad_sx_ignored": (" * (double)sx[(int64_t)g * K + k];", ";"),
    "wgrad_abs_dropped": ("mag[n * K + k] += fabs(p);", "mag[n * K + k] += p;"),
    "pow2_ignored": ("return pow2 ? gqo_scale_pow2(amax) : gqo_scale(amax);",
                     "return gqo_scale(amax);"),
}


def _fast_pins():
    pins = []
    for p in oracle_pins.ALL_PINS:
        if p is oracle_pins.pin_encode_vs_torch:
            p = functools.partial(p, stride=13, neg_stride=7)
        pins.append(p)
    return pins


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found once"
    mpath = tmp_path / "gq_oracle_mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mpath), str(tmp_path / "libmutant.so"))
    o = oracle.Oracle(lib)
    failed = []
    for pin in _fast_pins():
        try:
            pin(o)
        except AssertionError:
            failed.append(getattr(pin, "__name__", getattr(pin, "func", pin).__name__))
            break
    assert failed, f"mutant {name} passed every pin"
