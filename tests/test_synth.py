"""The seeded generators: determinism, row-subset consistency, workload shapes."""

import numpy as np

from synth import CONFIGS, make_rows, make_workload
from synth.workloads import CFG5_LENGTHS


def test_rows_regenerate_bit_identically():
    full = make_workload(2, B=8)
    sub = make_rows(2, [6, 1])
    assert np.array_equal(sub.scores.view(np.uint32), full.scores[[6, 1]].view(np.uint32))
    assert np.array_equal(sub.lengths, full.lengths[[6, 1]])
    again = make_rows(2, [6, 1])
    assert np.array_equal(again.scores.view(np.uint32), sub.scores.view(np.uint32))


def test_ragged_lengths_and_padding():
    for cfg in (2, 3, 4):
        spec = CONFIGS[cfg]
        w = make_rows(cfg, range(0, spec.B, max(1, spec.B // 16)))
        assert w.lengths.min() >= int(np.ceil(0.8 * spec.stride)) and w.lengths.max() <= spec.stride
        for b, n in enumerate(w.lengths):
            assert not np.isnan(w.scores[b, :n]).any()
            assert np.isnan(w.scores[b, n:]).all()


def test_config1_and_config5_lengths():
    assert make_workload(1).lengths.tolist() == [0, 300, 512, 8192]
    w = make_rows(5, range(0, 128, 6))
    assert w.lengths.tolist() == [CFG5_LENGTHS[(r // 6) % 9] for r in range(0, 128, 6)]


def test_config2_narrow_band_and_config5_kinds():
    w = make_rows(2, [40])
    x = w.scores[0, : w.lengths[0]]
    assert x.min() >= 1.0 and x.max() <= 1.0 + 2.0 ** -10
    assert np.unique(x).size > 8000
    w = make_rows(5, [6 * 8 + k for k in range(6)])  # length 98307 for all six kinds
    const, asc, low, huge, special, peaks = w.scores
    assert np.unique(const).size == 1
    assert np.array_equal(asc, np.arange(asc.size, dtype=np.float32))
    assert np.unique(low).size <= 1024 and low.min() >= 1.0 and low.max() < 1.0 + 2 ** -13
    assert huge.min() >= 65504.0
    assert np.isneginf(special).any() and np.isposinf(special).any()
    assert (np.signbit(special) & (special == 0)).any()
    assert (peaks > 50).sum() == 1024 // 4


def test_config4_page_table_is_a_permutation():
    w = make_rows(4, [0, 1023])
    assert w.page_table.shape == (2, 4096)
    full_pt = make_rows(4, [0]).page_table
    assert np.array_equal(full_pt[0], w.page_table[0])
    assert np.unique(w.page_table).size == 2 * 4096
    assert w.page_table.min() >= 0 and w.page_table.max() < 1024 * 4096
