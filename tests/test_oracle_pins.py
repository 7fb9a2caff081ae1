"""The CPU oracle against facts outside itself (no GPU needed)."""

import numpy as np
import pytest

import oracle
import oracle_pins as P
from synth import make_rows, make_workload


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def test_golden_fixtures(orc):
    P.pin_golden(orc)


def test_closed_forms(orc):
    P.pin_closed_forms(orc)


def test_nan_inside_length_is_refused(orc):
    P.pin_nan_rejected(orc)


def test_bruteforce_tiny_rows(orc):
    P.pin_bruteforce(orc, cases=1500)


@pytest.mark.parametrize("k", [1, 7, 64, 512, 2048])
def test_invariants_and_lexsort(orc, k):
    scores, lengths = P.small_inputs()
    out = orc.topk_ragged(scores, lengths, k)
    P.check_selection(scores, lengths, k, out)
    P.pin_lexsort(orc, scores, lengths, k)


@pytest.mark.parametrize("config", [1, 2, 3, 4, 5])
def test_invariants_on_workload_rows(orc, config):
    # a few rows of every workload, full width, with the workload's own k
    rows = {1: range(4), 2: [0, 1, 40, 63], 3: [0, 511, 1023], 4: [0, 777], 5: range(0, 128, 7)}
    w = make_rows(config, rows[config])
    out = orc.topk_ragged(w.scores, w.lengths, w.k)
    P.check_selection(w.scores, w.lengths, w.k, out)
    P.pin_lexsort(orc, w.scores, w.lengths, w.k)


def test_torch_topk_values(orc):
    w = make_workload(1)
    P.pin_torch_topk(orc, w.scores, w.lengths, w.k)
    w = make_rows(3, [3, 9])
    P.pin_torch_topk(orc, w.scores, w.lengths, w.k)


def test_paged_formula(orc):
    w = make_rows(4, [0, 5, 1000])
    P.pin_paged_formula(orc, w.scores, w.lengths, w.k, w.page_table, w.page_size)


def test_capacity_boundaries(orc):
    # Rows whose best scores share one narrow band, with the band's population
    # at the capacities the pages report failures at (4096, 16384/16385) and
    # around them; the oracle must still return the exact selection.
    rng = np.random.default_rng(3)
    k = 2048
    for pop in (4095, 4096, 4097, 16384, 16385):
        n = pop + 5000
        x = rng.standard_normal(n).astype(np.float32) - 10.0
        band = (np.uint32(0x3F800000) + rng.integers(0, 8193, pop).astype(np.uint32)).view(np.float32)
        pos = rng.permutation(n)[:pop]
        x[pos] = band
        out = orc.topk_ragged(x[None], np.array([n], np.int32), k)
        P.check_selection(x[None], np.array([n]), k, out)
        P.pin_lexsort(orc, x[None], np.array([n]), k)


def test_check_selection_catches_a_swap(orc):
    # the invariant checker itself fails on a corrupted answer
    scores, lengths = P.small_inputs()
    out = orc.topk_ragged(scores, lengths, 64)
    bad = out.copy()
    b = 0
    n = P.valid_len(lengths[b], scores.shape[1])
    unselected = np.setdiff1d(np.arange(n), out[b])
    worst = unselected[np.argmin(P.total_order(scores[b, unselected]))]
    bad[b, 10] = worst
    with pytest.raises(AssertionError):
        P.check_selection(scores, lengths, 64, bad)
