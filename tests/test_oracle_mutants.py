"""The oracle's pins must reject a plausibly broken oracle.

Each case plants one mistake in a copy of oracle.c (on the CPU, in a temporary
directory), builds it, and runs every pin of the oracle suites against that
copy: at least one pin has to fail. The shipped oracle.c is never modified."""
import inspect
import os

import pytest

pytestmark = pytest.mark.filterwarnings("ignore:overflow encountered in cast")

import oracle
from tests import test_oracle_attention, test_oracle_codec, test_oracle_gemm, test_oracle_softmax, test_oracle_w4

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement) -- one planted mistake each
MUTANTS = [
    ("transposed_B", "a * lut[brow[j]]", "a * lut[B[j * K + k]]"),
    ("dropped_last_k", "for (int64_t k = 0; k < K; ++k) {\n                double a",
     "for (int64_t k = 0; k + 1 < K; ++k) {\n                double a"),
    ("bias_per_row", "(bias ? oracle_half_to_double(bias[j]) : 0.0)",
     "(bias ? oracle_half_to_double(bias[j % 2]) : 0.0)"),
    ("gelu_wrong_scale", "erf(x / sqrt(2.0))", "erf(x / 2.0)"),
    ("gelu_tanh_form", "0.5 * x * (1.0 + erf(x / sqrt(2.0)))",
     "0.5 * x * (1.0 + tanh(0.7978845608028654 * (x + 0.044715 * x * x * x)))"),
    ("gelu_before_bias", "double x = s + (bias ? oracle_half_to_double(bias[j]) : 0.0);\n    return gelu ? oracle_gelu(x) : x;",
     "double x = (gelu ? oracle_gelu(s) : s);\n    return x + (bias ? oracle_half_to_double(bias[j]) : 0.0);"),
    ("rounding_through_fp32", "if (C) C[r * N + j] = oracle_double_to_half(y);",
     "if (C) C[r * N + j] = oracle_double_to_half((double)(float)y);"),
    ("round_ties_away", "double q = nearbyint(ldexp(a, 10 - e));", "double q = round(ldexp(a, 10 - e));"),
    ("subnormal_exponent", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("normal_exponent_bias", "v = ldexp((double)(1024 + f), e - 25);", "v = ldexp((double)(1024 + f), e - 24);"),
    ("overflow_threshold", "if (a >= 65520.0)", "if (a >= 65504.0)"),
    ("fp32_accumulation", "double* acc = (double*)malloc((size_t)N * sizeof(double));",
     "float* acc = (float*)malloc((size_t)N * sizeof(float));"),
    ("sampled_wrong_index", "oracle_half_to_double(B[k * N + j])", "oracle_half_to_double(B[j * K + k])"),
    ("int4_nibble_order", "row[k / 2], (k % 2) ? 4 : 0", "row[k / 2], (k % 2) ? 0 : 4"),
    ("int4_rows_along_k", "const uint8_t* row = Bq + n * (K / 2);", "const uint8_t* row = Bq + (n ^ 1) * (K / 2);"),
    ("int4_unsigned", "return v >= 8 ? v - 16 : v;", "return v;"),
    ("int4_group_index", "scales + (k / group) * N;", "scales + (k % group) * N;"),
    ("int4_no_rounding_of_weights", "W[k * N + n] = oracle_double_to_half(q * oracle_half_to_double(srow[n]));",
     "W[k * N + n] = oracle_double_to_half(q) ; (void)srow;"),
    ("e2m1_exponent_bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e)"),
    ("e2m1_subnormal_as_normal", "(e == 0) ? 0.5 * m :", "(e == 0) ? ldexp(1.0 + 0.5 * m, -1) :"),
    ("e2m1_mantissa_weight", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.25 * m, e - 1)"),
    ("e2m1_sign_bit", "const int s = (v >> 3) & 1, e", "const int s = v & 1, e"),
    ("fp4_format_ignored", "return format == 1 ? oracle_e2m1_value", "return format == 2 ? oracle_e2m1_value"),
    ("attn_no_max_shift", "const double pj = exp(sc[j] - m);", "const double pj = exp(sc[j]);"),
    ("attn_causal_drops_diagonal", "const int64_t visible = causal ? si + 1 : S;",
     "const int64_t visible = causal ? (si > 0 ? si : 1) : S;"),
    ("attn_causal_sees_next", "const int64_t visible = causal ? si + 1 : S;",
     "const int64_t visible = causal ? (si + 2 < S ? si + 2 : S) : S;"),
    ("attn_wrong_scale", "sc[j] = dot * scale;", "sc[j] = dot * scale * scale;"),
    ("attn_no_normalisation", "const double y = acc[d] / l;", "const double y = acc[d];"),
    ("attn_value_of_query_row", "const uint16_t* vr = V + ((b * S + j) * H + h) * D;",
     "const uint16_t* vr = V + ((b * S + si) * H + h) * D;"),
    ("softmax_no_max_shift", "for (int64_t j = 0; j < N; ++j) l += exp(lut[x[j]] - m);",
     "m = 0.0; for (int64_t j = 0; j < N; ++j) l += exp(lut[x[j]] - m);"),
    ("softmax_max_skips_last", "for (int64_t j = 0; j < N; ++j)\n            if (lut[x[j]] > m) m = lut[x[j]];",
     "for (int64_t j = 0; j + 1 < N; ++j)\n            if (lut[x[j]] > m) m = lut[x[j]];"),
    ("softmax_sum_skips_first", "for (int64_t j = 0; j < N; ++j) l += exp(lut[x[j]] - m);",
     "for (int64_t j = 1; j < N; ++j) l += exp(lut[x[j]] - m);"),
    ("softmax_wrong_row", "const uint16_t* x = X + (row0 + r) * N;", "const uint16_t* x = X + r * N;"),
    ("attn_key_of_head_zero", "const uint16_t* kr = K + ((b * S + j) * H + h) * D;",
     "const uint16_t* kr = K + ((b * S + j) * H + 0) * D;"),
]


def _pins():
    fns = []
    for mod in (test_oracle_codec, test_oracle_gemm, test_oracle_w4, test_oracle_attention, test_oracle_softmax):
        for name, fn in inspect.getmembers(mod, inspect.isfunction):
            if name.startswith("test_") and "oracle_lib" in inspect.signature(fn).parameters:
                fns.append(fn)
    return fns


def test_every_pin_passes_on_the_shipped_oracle(oracle_lib):
    for fn in _pins():
        fn(oracle_lib)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(text.replace(old, new))
    lib = oracle.load_library(oracle.compile_source(str(src), str(tmp_path / f"lib_{name}.so")))
    failures = []
    for fn in _pins():
        try:
            fn(lib)
        except (AssertionError, RuntimeError, ValueError) as e:
            failures.append(fn.__name__)
    assert failures, f"no pin caught the planted mistake {name}"
