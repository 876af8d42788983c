"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each mutation is a textual edit of a temporary copy of ``oracle/pagedkv_oracle.c``
(the committed oracle is never touched): a wrong head-to-group index, a dropped
scale, an off-by-one causal window, a wrong block offset, a dropped softmax
normalisation, a transposed V operand, a wrong cache-write offset, a dropped
merge denominator and a wrong size rule.  The copy is compiled with gcc and the
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
    "block_offset": [("key_dot(qrow, k_cache, trow[j / block_size], j % block_size, g, n_kv,\n                                       block_size",
                      "key_dot(qrow, k_cache, trow[j / block_size], (j + 1) % block_size, g, n_kv,\n                                       block_size")],
    "softmax_not_normalised": [("const double w = s[j] / l;", "const double w = s[j];")],
    "v_transposed": [("orow[k] += w * bf16_to_double(vrow[k]);",
                      "orow[k] += w * bf16_to_double(vrow[(k % 2) ? k - 1 : k + 1]);")],
    "cache_write_offset": [("int64_t off = slot % block_size;", "int64_t off = (slot + 1) % block_size;")],
    "merge_no_denominator": [("o[k] /= den;", "o[k] /= 1.0;")],
    "size_rule_half": [("return 2 * layers * n_kv * head_dim * dtype_size;",
                        "return layers * n_kv * head_dim * dtype_size;")],
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
