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


def test_bf16_rounding_is_nearest_even():
    """The BF16 inputs are the float32 scores rounded to the nearest bfloat16
    (ties to even), checked against the two neighbouring bfloat16 values."""
    from synth import bf16_bits_to_float, to_bf16_bits

    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(5000).astype(np.float32),
                        np.array([1.00390625, 1.01171875, -2.0078125, 0.0, -0.0, 1e-40],
                                 dtype=np.float32)])
    b = to_bf16_bits(x)
    got = bf16_bits_to_float(b).astype(np.float64)
    lo = bf16_bits_to_float((x.view(np.uint32) >> 16).astype(np.uint16)).astype(np.float64)
    hi = bf16_bits_to_float(((x.view(np.uint32) >> 16) + 1).astype(np.uint16)).astype(np.float64)
    xv = x.astype(np.float64)
    # the result is one of the two neighbours (truncation and one ulp further out) ...
    assert np.all((got == lo) | (got == hi))
    # ... the nearer one, and on an exact tie the one with an even last bit
    d_lo, d_hi = np.abs(xv - lo), np.abs(xv - hi)
    nearer = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.nan))
    tie = np.isnan(nearer)
    assert np.all(got[~tie] == nearer[~tie])
    assert np.all((b[tie] & 1) == 0)
    assert np.array_equal(bf16_bits_to_float(b[-6:-1]),
                          np.array([1.0, 1.015625, -2.0, 0.0, -0.0], dtype=np.float32))


def test_config3_offsets_config4_spikes_and_prefill_rows():
    """The value recipes: N(0,1) plus one offset per row in [-4, 4] (workload
    3); N(0,1) with about 1 % of positions raised by U(3, 6) (workload 4);
    N(0,1) rows of 80-100 % length for the prefill shapes (workloads 6, 7)."""
    w = make_rows(3, range(16))
    means = np.array([w.scores[b, : w.lengths[b]].mean() for b in range(16)])
    stds = np.array([w.scores[b, : w.lengths[b]].std() for b in range(16)])
    assert np.all(np.abs(means) < 4.02) and np.ptp(means) > 1.0  # offsets differ per row
    assert np.all(np.abs(stds - 1.0) < 0.02)
    w = make_rows(4, [0, 1])
    for b in range(2):
        x = w.scores[b, : w.lengths[b]].astype(np.float64)
        # spikes: x > 2.5 is N(0,1)'s 0.6 % tail plus ~1 % raised by at least 3
        frac = float(np.mean(x > 2.5))
        assert 0.013 < frac < 0.019, frac
        assert x.max() < 6.0 + 6.0  # U(3, 6) over N(0,1)
    for cfg in (6, 7):
        spec = CONFIGS[cfg]
        w = make_rows(cfg, [0, spec.B // 2, spec.B - 1])
        assert w.scores.shape == (3, spec.stride)
        assert w.lengths.min() >= int(np.ceil(0.8 * spec.stride)) and w.lengths.max() <= spec.stride
        x = w.scores[0, : w.lengths[0]]
        assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1.0) < 0.05
