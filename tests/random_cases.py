"""Seeded random cases of the parity tests (host-side generator, numpy only).

Each case draws a batch size, a row width (1 to 300000), k, a length mode
(full, 80-100 %, anything from -2 to past the width, around k, up to 2k, up
to k + 16384), per-row value kinds (N(0,1), offsets, few distinct values,
infinities and signed zeros, ascending, descending, constant, sparse peaks),
a row start offset of 0 to 3 floats, and paging. Scores past a row's length
are NaN: no call may read them. The GPU tests in test_gpu_random.py and
test_zz_no_alloc.py run these cases; test_random_cases_host.py checks the
generator itself on CPU.
"""

import numpy as np

N_CASES = 96
MAX_ELEMENTS = 12_000_000  # per case, so that the oracle's full sorts stay quick


def row_values(rng, kind, width):
    if kind == 0:
        return rng.standard_normal(width)
    if kind == 1:  # an offset, as in the decode workload
        return rng.standard_normal(width) + rng.uniform(-4, 4)
    if kind == 2:  # few distinct values: ties at every cutoff
        return rng.integers(-3, 4, width).astype(np.float64) * 0.25
    if kind == 3:  # infinities and signed zeros over N(0,1)
        x = rng.standard_normal(width)
        pick = rng.integers(0, 8, width)
        x[pick == 0] = np.inf
        x[pick == 1] = -np.inf
        x[pick == 2] = -0.0
        x[pick == 3] = 0.0
        return x
    if kind == 4:
        return np.arange(width, dtype=np.float64)
    if kind == 5:
        return -np.arange(width, dtype=np.float64)
    if kind == 6:
        return np.full(width, rng.standard_normal())
    return np.where(rng.random(width) < 0.01, rng.uniform(3, 6, width), 0.0) + rng.standard_normal(width)


def draw_lengths(rng, mode, B, width, k):
    if mode == 0:
        return np.full(B, width, dtype=np.int64)
    if mode == 1:
        lo = (8 * width + 9) // 10
        return rng.integers(lo, width + 1, B)
    if mode == 2:
        return rng.integers(-2, width + 21, B)
    if mode == 3:
        return k + rng.integers(-1, 2, B)
    if mode == 4:  # a little over k: split halves and cluster slices with few scores
        return rng.integers(k + 1, 2 * k + 2, B)
    return rng.integers(k + 1, k + 16385, B)  # around the sampled cutoff's gate


def draw_case(i):
    rng = np.random.default_rng([0x5EED, 0xF022, i])
    if rng.random() < 0.3:  # long rows: the sampled cutoff, clusters and split rows
        width = int(rng.integers(65536, 300001))
    else:
        width = int(np.exp(rng.uniform(0.0, np.log(300000.0))))
    B = int(np.exp(rng.uniform(0.0, np.log(1200.0))))
    while B > 1 and B * width > MAX_ELEMENTS:
        B //= 2
    k = int(rng.choice([1, 2, 17, 100, 511, 512, 513, 1000, 1024, 2047, 2048, int(rng.integers(1, 2049))]))
    lengths = draw_lengths(rng, int(rng.integers(0, 6)), B, width, k)
    scores = np.full((B, width), np.nan, dtype=np.float32)
    for b in range(B):
        n = int(min(max(lengths[b], 0), width))
        scores[b, :n] = row_values(rng, int(rng.integers(0, 8)), n).astype(np.float32)
    offset = int(rng.integers(0, 4))  # floats before row 0 in the device buffer
    paged = bool(rng.integers(0, 2))
    page_size = int(rng.choice([1, 7, 16, 64]))
    pages = -(-width // page_size)
    pt = rng.permutation(B * pages).astype(np.int32).reshape(B, pages) if paged else None
    return scores, np.clip(lengths, -2**31, 2**31 - 1).astype(np.int32), k, offset, pt, page_size
