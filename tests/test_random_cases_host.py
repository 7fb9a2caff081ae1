"""The seeded random-case generator of the parity tests, on CPU: it is
deterministic, keeps every case within its size bound, never puts a NaN where
a call may read, draws well-formed page tables, and covers the regimes the GPU
tests are meant to reach (short and long rows, rows at or under k, paging,
every row offset). The oracle runs on a few small cases."""

import numpy as np

import oracle
import oracle_pins as P
from random_cases import MAX_ELEMENTS, N_CASES, draw_case


def _valid(lengths, width):
    return np.clip(lengths.astype(np.int64), 0, width)


def test_cases_are_deterministic():
    for i in (0, 7, 41):
        a, b = draw_case(i), draw_case(i)
        assert np.array_equal(a[0], b[0], equal_nan=True)
        assert np.array_equal(a[1], b[1]) and a[2:4] == b[2:4]
        assert (a[4] is None) == (b[4] is None) and (a[4] is None or np.array_equal(a[4], b[4]))


def test_cases_are_well_formed_and_cover_the_regimes():
    seen = {"short": 0, "long": 0, "at_or_under_k": 0, "over_k": 0, "paged": 0, "ragged": 0}
    offsets = set()
    for i in range(0, N_CASES, 4):
        scores, lengths, k, offset, pt, page_size = draw_case(i)
        B, width = scores.shape
        assert 1 <= width <= 300000 and 1 <= k <= 2048 and 0 <= offset <= 3
        assert B == 1 or B * width <= MAX_ELEMENTS
        assert lengths.dtype == np.int32 and lengths.shape == (B,)
        n = _valid(lengths, width)
        inside = np.arange(width)[None, :] < n[:, None]
        assert not np.isnan(scores[inside]).any(), "a NaN where a call reads"
        assert np.isnan(scores[~inside]).all(), "the padding is NaN"
        if pt is not None:
            assert pt.shape == (B, -(-width // page_size)) and page_size in (1, 7, 16, 64)
            assert np.array_equal(np.sort(pt.ravel()), np.arange(pt.size))
            seen["paged"] += 1
        else:
            seen["ragged"] += 1
        seen["short" if width <= 16384 else "long"] += 1
        seen["at_or_under_k"] += int((n <= k).sum())
        seen["over_k"] += int((n > k).sum())
        offsets.add(offset)
    assert all(v > 0 for v in seen.values()), seen
    assert offsets == {0, 1, 2, 3}


def test_the_oracle_runs_on_small_cases():
    """The oracle's output on the small random cases meets the invariants of
    an exact top-k (the checks of the oracle pins)."""
    done = 0
    for i in range(N_CASES):
        scores, lengths, k, offset, pt, page_size = draw_case(i)
        if scores.size > 200_000:
            continue
        P.check_selection(scores, lengths, k, oracle.topk_ragged(scores, lengths, k))
        done += 1
        if done == 12:
            break
    assert done == 12
