"""Plants plausible mistakes in copies of the oracle source and checks that the
pins catch every one of them (no GPU needed).

Each mutant is a textual edit of ``oracle/topk_oracle.cpp`` compiled into a
temporary library; the committed oracle itself is never modified.
"""

import os

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    # ranking reversed: worst scores selected
    "ascending_order": ("if (a > b) return true;", "if (a < b) return true;"),
    # signed zero ignored: -0 and +0 treated as equal
    "no_signed_zero_rule": ("return !std::signbit(a) && std::signbit(b);", "return false;"),
    # ties resolved by the highest index
    "highest_index_ties": ("return i < j;", "return i > j;"),
    # one selected slot too few
    "m_off_by_one": ("const int64_t m = std::min<int64_t>(k, n);",
                     "const int64_t m = std::min<int64_t>(k, n) - (n > 0 ? 1 : 0);"),
    # padding written as 0 instead of -1
    "padding_zero": ("for (int64_t j = m; j < k; ++j) out_row[j] = -1;",
                     "for (int64_t j = m; j < k; ++j) out_row[j] = 0;"),
    # page offset taken from the wrong operand
    "page_offset_swapped": ("* page_size + idx % page_size;", "* page_size + idx / page_size;"),
    # page number computed with the wrong operator
    "page_number_modulo": ("const int64_t page = idx / page_size;",
                           "const int64_t page = idx % page_size;"),
    # negative lengths read as their magnitude
    "negative_length_abs": ("if (len < 0) return 0;", "if (len < 0) return std::min<int64_t>(-static_cast<int64_t>(len), stride);"),
    # length not clamped to the width: reads one row into the next
    "length_clamp_off_by_one": ("return std::min<int64_t>(len, stride);",
                                "return std::min<int64_t>(len, stride - 1);"),
    # NaN inside the valid prefix accepted silently
    "nan_accepted": ("if (std::isnan(row[i])) return ORACLE_ENAN;", "(void)row;"),
    # block key misses the last score of each block
    "amax_block_short": ("for (int64_t j = 8 * i; j < 8 * i + 8; ++j) {",
                         "for (int64_t j = 8 * i; j < 8 * i + 7; ++j) {"),
    # block key keeps the first of two equal-comparing scores (-0 / +0 order-dependent)
    "amax_first_of_equals": ("if (ranks_above(row[j], m)) m = row[j];", "if (row[j] > m) m = row[j];"),
    # newest block not forced to +inf
    "amax_no_inf": ("out_row[nb - 1] = INFINITY;", "out_row[nb - 1] = row[8 * (nb - 1)];"),
    # rows with exactly topk blocks not skipped
    "amax_skip_strict": ("if (nb == 0 || (topk > 0 && nb <= topk)) continue;",
                         "if (nb == 0 || (topk > 0 && nb < topk)) continue;"),
    # block table sorted descending
    "blocks_descending": ("std::sort(ids.begin(), ids.end());",
                          "std::sort(ids.begin(), ids.end(), [](int32_t a, int32_t b) { return a > b; });"),
    # a row with exactly k blocks not treated as the identity
    "blocks_identity_strict": ("    if (nb <= k) {\n      for (int64_t j = 0; j < nb; ++j)",
                               "    if (nb < k) {\n      for (int64_t j = 0; j < nb; ++j)"),
    # blocks per page taken as the page size itself
    "blocks_bpp_page_size": ("const int64_t bpp = page_size / 8;", "const int64_t bpp = page_size;"),
    # padding written as -1 instead of INT32_MAX
    "blocks_pad_minus_one": ("        row[j] = INT32_MAX;\n        pages[j] = INT32_MAX;",
                             "        row[j] = -1;\n        pages[j] = -1;"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.source_path()) as f:
        return f.read()


def _build_variant(tmp_path, src_text, name):
    src = tmp_path / f"{name}.cpp"
    src.write_text(src_text)
    lib = tmp_path / f"lib{name}.so"
    oracle.build(str(src), str(lib))
    return oracle.Oracle(str(lib))


def test_unmutated_copy_passes(tmp_path, source):
    P.run_all_pins(_build_variant(tmp_path, source, "clean"), quick=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, source, name):
    before, after = MUTANTS[name]
    assert source.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    orc = _build_variant(tmp_path, source.replace(before, after), name)
    with pytest.raises((AssertionError, RuntimeError)):
        P.run_all_pins(orc, quick=True)
