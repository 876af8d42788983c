"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each mutation is a textual edit of a temporary copy of ``oracle/pagedkv_oracle.c``
(the committed oracle is never touched): a wrong head-to-group index, a dropped
scale, an off-by-one causal window, a wrong block offset, a dropped softmax
normalisation, a transposed V operand, a wrong cache-write offset, a dropped
merge denominator, a wrong size rule, an off-by-one sliding window, E4M3
rounding ties away from zero, a wrong E4M3 exponent bias, a dropped FP8 scale,
a signed instead of absolute row maximum, and a block copy from the wrong
source.  The copy is compiled with gcc and the
whole pin suite is run against it; at least one pin must fail.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pagedkv_oracle.c")

MUTATIONS = {
    "group_index_mod": [("return h / G;", "return h % n_kv;"),
                        ("const int32_t g = h / G;", "const int32_t g = h % n_kv;")],
    "scale_dropped": [("s[j] = scale * key_dot(", "s[j] = key_dot(")],
    "causal_off_by_one": [("const int32_t nvis = pos + 1;", "const int32_t nvis = pos + (pos > 0 ? 0 : 1);")],
    "block_offset": [("s[j] = scale * key_dot(qrow, kc, trow[j / block_size], j % block_size, g,",
                      "s[j] = scale * key_dot(qrow, kc, trow[j / block_size], (j + 1) % block_size, g,")],
    "softmax_not_normalised": [("const double w = s[j] / l;", "const double w = s[j];")],
    "v_transposed": [("head_dim, k);\n            }\n            if (lse)",
                      "head_dim, (k % 2) ? k - 1 : k + 1);\n            }\n            if (lse)")],
    "cache_write_offset": [("int64_t off = slot % block_size;", "int64_t off = (slot + 1) % block_size;")],
    "merge_no_denominator": [("o[k] /= den;", "o[k] /= 1.0;")],
    "size_rule_half": [("return 2 * layers * n_kv * head_dim * dtype_size;",
                        "return layers * n_kv * head_dim * dtype_size;")],
    "window_off_by_one": [("pos + 1 - window : 0;", "pos + 2 - window : 0;")],
    "e4m3_ties_away": [("if (rem > 0.5 || (rem == 0.5 && fmod(n, 2.0) == 1.0))", "if (rem >= 0.5)")],
    "e4m3_bias_8": [("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)")],
    "fp8_scale_dropped": [("* (double)c.scale[row];", "* 1.0;")],
    "fp8_signed_amax": [("const float v = (float)fabs(bf16_to_double(src[k]));",
                         "const float v = (float)bf16_to_double(src[k]);")],
    "copy_blocks_source": [("cache[dst * block_bytes + b] = cache[src * block_bytes + b];",
                            "cache[dst * block_bytes + b] = cache[(src + 1) * block_bytes + b];")],
    "table_row_stride": [("const int32_t *trow = block_tables + (int64_t)b * max_blocks;\n            const uint16_t *qrow = q + ((int64_t)row",
                          "const int32_t *trow = block_tables + (int64_t)b * (max_blocks - (max_blocks > 1));\n            const uint16_t *qrow = q + ((int64_t)row")],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    text = open(SRC).read()
    for old, new in MUTATIONS[name]:
        assert old in text, f"mutation {name}: pattern not found in the oracle source"
        text = text.replace(old, new)
    src = tmp_path / "mutant.c"
    src.write_text(text)
    so = oracle.build(force=True, src=str(src), out=str(tmp_path / "libmutant.so"))
    lib = oracle.load_library(so)
    failures = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(lib)
        except (AssertionError, ValueError, IndexError) as exc:
            failures.append((check.__name__, str(exc)[:80]))
            break
    assert failures, f"no pin caught the planted mistake {name!r}"
