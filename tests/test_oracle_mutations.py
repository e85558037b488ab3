"""Planted mistakes: each edit below is a plausible bug in the oracle (a wrong
sign or bound, a dropped term, a wrong index, a transposed operand).  The edit
is made to a temporary copy of the oracle source on the CPU, compiled, and the
pin suite must reject it: at least one pin has to fail for every mistake."""
import pytest

import oracle
from test_oracle_pins import PINS

MUTATIONS = {
    "causal_off_by_one": ("if (j > pos) return 0;", "if (j >= pos) return 0;"),
    "window_off_by_one": ("j < pos - window + 1) return 0;",
                          "j < pos - window) return 0;"),
    "sink_dropped": ("if (has_x) z += exp(x - m);", ""),
    "sink_scaled": ("(sinks != NULL) ? sinks[h] : 0.0",
                    "(sinks != NULL) ? scale * sinks[h] : 0.0"),
    "smooth_dropped": ("const int has_x = (sinks != NULL) || smooth;",
                       "const int has_x = (sinks != NULL);"),
    "kv_head_interleaved": ("const int g = h / G;", "const int g = h % Hkv;"),
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "prefix_ignored": ("const long pos = P + i;", "const long pos = i;"),
    "k_and_v_swapped": ("const double* kr = k + ((size_t)(base + j) * Hkv + g) * d;",
                        "const double* kr = v + ((size_t)(base + j) * Hkv + g) * d;"),
    "lse_without_log": ("m + log(z);", "m + z;"),
    "max_not_subtracted_from_sink": ("if (has_x) z += exp(x - m);",
                                     "if (has_x) z += exp(x);"),
    "census_live_off_by_one": ("if (n0 <= pos && n1 >= lo) {",
                               "if (n0 <= pos && n1 > lo) {"),
    "census_masked_off_by_one": ("if (n0 < lo || n1 > pos) { ++masked; break; }",
                                 "if (n0 < lo || n1 >= pos) { ++masked; break; }"),
    "custom_mask_ignored": ("if (mask == NULL || j < P) return 1;", "return 1;"),
    "custom_mask_transposed": (
        "const uint32_t word = mask[(long)mask_indptr[b] + i * W + jp / 32];\n"
        "    return (int)((word >> (jp % 32)) & 1u);",
        "const uint32_t word = mask[(long)mask_indptr[b] + jp * W + i / 32];\n"
        "    return (int)((word >> (i % 32)) & 1u);"),
    "custom_mask_bit_off_by_one": ("return (int)((word >> (jp % 32)) & 1u);",
                                   "return (int)((word >> ((jp + 1) % 32)) & 1u);"),
    "custom_mask_row_stride": ("const long W = (E + 31) / 32;", "const long W = E / 32;"),
    "census_window_ignored": ("long lo = (window > 0) ? pos - window + 1 : 0;",
                              "long lo = 0;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert old in src, f"mutation anchor for {name} not found"
    path = oracle.compile_variant(src.replace(old, new))
    try:
        lib = oracle.load(path)
        failures = []
        for pin in PINS:
            try:
                pin(lib)
            except AssertionError:
                failures.append(pin.__name__)
        assert failures, f"no pin caught the planted mistake {name}"
    finally:
        oracle.remove_variant(path)
