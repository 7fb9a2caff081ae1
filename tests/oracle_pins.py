"""Checks that pin the CPU oracle to facts outside itself.

Each ``pin_*`` takes an oracle object (``topk_ragged`` / ``topk_paged`` on
numpy arrays) and raises ``AssertionError`` when the oracle disagrees with

* brute force over every index subset of tiny rows,
* the invariants that define a top-k selection,
* closed forms (constant, ascending, descending, short, empty, all -inf rows),
* an independent library ordering (numpy's stable ``lexsort``) and
  ``torch.topk`` values,
* the hand-derived fixtures under ``tests/golden/``.

The same functions run against the real oracle and against deliberately
broken builds of it (the mutation test), so every plausible slip in the
oracle trips at least one of them.
"""

from __future__ import annotations

import glob
import itertools
import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
NEG_ZERO_STANDIN = -1e-320  # a float64 between every negative float32 and +0


def total_order(x) -> np.ndarray:
    """float64 values ordered like the scores' total order (-0 just below +0)."""
    v = np.asarray(x, dtype=np.float32).astype(np.float64)
    v[(v == 0) & np.signbit(v)] = NEG_ZERO_STANDIN
    return v


def valid_len(length: int, stride: int) -> int:
    return min(max(int(length), 0), stride)


def check_selection(scores: np.ndarray, lengths: np.ndarray, k: int, out: np.ndarray,
                    lowest_index_ties: bool = True, ordered: bool = True) -> None:
    """Invariants of an exact top-k output, row by row.

    * exactly m = min(k, n) valid indices, unique, inside [0, n); -1 after them
    * every selected score ranks at or above every unselected one
    * count(score > cut) < m <= count(score >= cut) for the m-th best score cut
    * (ordered) best first, equal scores by ascending index
    * (lowest_index_ties) the tied scores at the cut that are taken are the
      lowest indices among them
    """
    B, stride = scores.shape
    assert out.shape == (B, k), (out.shape, (B, k))
    for b in range(B):
        n = valid_len(lengths[b], stride)
        m = min(k, n)
        row = out[b]
        assert np.all(row[m:] == -1), f"row {b}: slots past m={m} must be -1"
        sel = row[:m]
        assert np.all((sel >= 0) & (sel < n)), f"row {b}: index outside [0, {n})"
        assert np.unique(sel).size == m, f"row {b}: duplicate indices"
        if m == 0:
            continue
        tov = total_order(scores[b, :n])
        chosen = np.zeros(n, dtype=bool)
        chosen[sel] = True
        if m < n:
            assert tov[chosen].min() >= tov[~chosen].max(), f"row {b}: unselected outranks selected"
        cut = tov[chosen].min()
        assert np.count_nonzero(tov > cut) < m <= np.count_nonzero(tov >= cut), f"row {b}: cut count"
        if ordered:
            t = tov[sel]
            assert np.all(t[:-1] >= t[1:]), f"row {b}: not best first"
            same = t[:-1] == t[1:]
            assert np.all(sel[:-1][same] < sel[1:][same]), f"row {b}: ties not by index"
        if lowest_index_ties:
            tied = np.flatnonzero(tov == cut)
            need = m - np.count_nonzero(tov > cut)
            assert np.array_equal(np.sort(sel[tov[sel] == cut]), tied[:need]), \
                f"row {b}: ties at the cut are not the lowest indices"


def _run(orc, scores, lengths, k, page_table=None, page_size=0):
    scores = np.asarray(scores, dtype=np.float32)
    if scores.ndim == 1:
        scores = scores[None, :]
    lengths = np.asarray(lengths, dtype=np.int32)
    if page_table is None:
        return orc.topk_ragged(scores, lengths, k)
    return orc.topk_paged(scores, lengths, k, np.asarray(page_table, dtype=np.int32), page_size)


# --------------------------------------------------------------------------
# brute force

POOL = (-math.inf, -2.5, -1.0, -0.0, 0.0, 0.5, 1.0, 3.0, math.inf)


def _order_key(v: float):
    return (v, 0 if (v == 0 and math.copysign(1.0, v) < 0) else 1)


def brute_force_row(vals, k):
    """Best-first index list by enumerating every subset of size min(k, n).

    The winning subset maximises its sorted score vector; among the winners
    the lexicographically smallest index tuple (= lowest indices at ties)."""
    n = len(vals)
    m = min(k, n)
    best_vec, best_set = None, ()
    for subset in itertools.combinations(range(n), m):
        vec = sorted((_order_key(vals[i]) for i in subset), reverse=True)
        if best_vec is None or vec > best_vec:
            best_vec, best_set = vec, subset
    return sorted(best_set, key=lambda i: (tuple(-c for c in _order_key(vals[i])), i))


def pin_bruteforce(orc, cases: int = 400, seed: int = 1234) -> None:
    rng = np.random.default_rng(seed)
    stride = 8
    for _ in range(cases):
        n = int(rng.integers(0, stride + 1))
        vals = [POOL[i] for i in rng.integers(0, len(POOL), size=n)]
        k = int(rng.choice([1, 2, 3, 5, 8]))
        row = np.full(stride, np.nan, dtype=np.float32)
        row[:n] = vals
        got = _run(orc, row, [n], k)[0]
        want = brute_force_row(vals, k)
        m = len(want)
        assert list(got[:m]) == want, (vals, k, got, want)
        assert np.all(got[m:] == -1)
        # the value multiset, bit for bit
        gb = np.sort(row[got[:m]].view(np.uint32))
        wb = np.sort(row[np.array(want, dtype=np.int64)].view(np.uint32)) if m else gb
        assert np.array_equal(gb, wb)


# --------------------------------------------------------------------------
# library cross-checks


def lexsort_reference(scores: np.ndarray, lengths: np.ndarray, k: int) -> np.ndarray:
    """numpy's stable lexsort: score descending, +0 before -0, index ascending."""
    B, stride = scores.shape
    out = np.full((B, k), -1, dtype=np.int32)
    for b in range(B):
        n = valid_len(lengths[b], stride)
        x = scores[b, :n].astype(np.float64)
        pos_zero = ((x == 0) & ~np.signbit(x)).astype(np.int8)
        idx = np.arange(n)
        order = np.lexsort((idx, -pos_zero, -x))
        m = min(k, n)
        out[b, :m] = order[:m]
    return out


def pin_lexsort(orc, scores, lengths, k) -> None:
    got = _run(orc, scores, lengths, k)
    want = lexsort_reference(np.asarray(scores, np.float32), np.asarray(lengths), k)
    assert np.array_equal(got, want), "oracle differs from numpy lexsort ordering"


def pin_torch_topk(orc, scores, lengths, k) -> None:
    """torch.topk values (float compare; no signed zeros in these rows)."""
    import torch

    got = _run(orc, scores, lengths, k)
    B, stride = scores.shape
    for b in range(B):
        n = valid_len(lengths[b], stride)
        m = min(k, n)
        if m == 0:
            continue
        row = torch.from_numpy(np.ascontiguousarray(scores[b, :n]))
        tv = torch.topk(row, m, largest=True, sorted=True).values.numpy()
        gv = np.sort(scores[b, got[b, :m]])[::-1]
        assert np.array_equal(gv.view(np.uint32), tv.view(np.uint32)), f"row {b}: torch.topk values"


# --------------------------------------------------------------------------
# closed forms


def pin_closed_forms(orc) -> None:
    stride, k = 64, 8
    # constant row: the m lowest indices
    out = _run(orc, np.full(stride, 2.5), [40], k)[0]
    assert list(out) == list(range(k))
    # ascending x[i] = i: the last m indices, best first
    out = _run(orc, np.arange(stride), [50], k)[0]
    assert list(out) == list(range(49, 49 - k, -1))
    # descending: the first m
    out = _run(orc, -np.arange(stride), [50], k)[0]
    assert list(out) == list(range(k))
    # n <= k: every valid index, then -1
    x = np.linspace(-1, 1, stride)
    out = _run(orc, x, [5], k)[0]
    assert sorted(out[:5]) == [0, 1, 2, 3, 4] and list(out[5:]) == [-1] * (k - 5)
    # n = 0 and negative lengths: all -1
    for n in (0, -1, -1000):
        assert list(_run(orc, x, [n], k)[0]) == [-1] * k
    # all -inf: -inf is a legal score, never replaced by padding
    out = _run(orc, np.full(stride, -np.inf), [6], k)[0]
    assert list(out) == [0, 1, 2, 3, 4, 5, -1, -1]
    # one +inf among ordinary scores comes first
    rng = np.random.default_rng(7)
    x = rng.standard_normal(stride).astype(np.float32)
    x[37] = np.inf
    out = _run(orc, x, [stride], k)[0]
    assert out[0] == 37
    # length past the stride is clamped to the stride
    out = _run(orc, np.arange(stride), [stride + 17], k)[0]
    assert list(out) == list(range(stride - 1, stride - 1 - k, -1))


def pin_nan_rejected(orc) -> None:
    """A NaN inside the valid prefix is outside the contract and is refused;
    NaN past the length is never looked at."""
    x = np.arange(16, dtype=np.float32)
    x[10:] = np.nan
    out = _run(orc, x, [10], 4)[0]
    assert list(out) == [9, 8, 7, 6]
    try:
        _run(orc, x, [12], 4)
    except RuntimeError:
        return
    raise AssertionError("NaN inside the valid prefix was not refused")


# --------------------------------------------------------------------------
# golden fixtures


def golden_cases():
    for path in sorted(glob.glob(os.path.join(GOLDEN, "*.json"))):
        with open(path) as f:
            yield os.path.basename(path), json.load(f)


def pin_golden(orc) -> None:
    for name, doc in golden_cases():
        if "amax8_cases" in doc:
            pin_golden_amax8(orc, name, doc["amax8_cases"])
        elif "cases" in doc:
            for case in doc["cases"]:
                got = _run(orc, case["scores"], case["lengths"], case["k"])
                assert got.tolist() == case["expected"], (name, case, got.tolist())
        else:  # paged fixture
            scores = np.array(doc["scores"], dtype=np.float32)
            got = _run(orc, scores, doc["lengths"], doc["k"])
            assert got.tolist() == doc["expected_ragged"], (name, got.tolist())
            got = _run(orc, scores, doc["lengths"], doc["k"], doc["page_table"], doc["page_size"])
            assert got.tolist() == doc["expected_paged"], (name, got.tolist())


def _golden_floats(rows, fill):
    """JSON rows of numbers and the strings "inf", "-inf", "sentinel" as float32."""
    conv = {"inf": np.inf, "-inf": -np.inf, "sentinel": fill}
    return np.array([[conv.get(v, v) if isinstance(v, str) else v for v in r] for r in rows],
                    dtype=np.float32)


def pin_golden_amax8(orc, name, cases) -> None:
    """Block keys compared bit for bit (a float compare would take -0 for +0)."""
    for case in cases:
        scores = _golden_floats(case["scores"], np.nan)
        want = _golden_floats(case["expected"], SENTINEL)
        init = np.full(want.shape, SENTINEL, dtype=np.float32)
        got = orc.amax8_varlen(scores, np.array(case["lengths"], np.int32), case["topk"], init)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (name, got.tolist())


def page_map_reference(ragged_out, page_table, page_size):
    """The docstring's formula, written out in numpy on the ragged output."""
    out = ragged_out.astype(np.int64)
    valid = out >= 0
    rows = np.broadcast_to(np.arange(out.shape[0])[:, None], out.shape)
    mapped = page_table[rows[valid], out[valid] // page_size].astype(np.int64) * page_size \
        + out[valid] % page_size
    res = np.full(out.shape, -1, dtype=np.int64)
    res[valid] = mapped
    return res.astype(np.int32)


def pin_paged_formula(orc, scores, lengths, k, page_table, page_size) -> None:
    ragged = _run(orc, scores, lengths, k)
    paged = _run(orc, scores, lengths, k, page_table, page_size)
    assert np.array_equal(paged, page_map_reference(ragged, np.asarray(page_table), page_size))


# --------------------------------------------------------------------------
# inputs for the randomized pins


def small_inputs(seed: int = 99):
    """A few small rows with the value mixes of the five workloads: normal,
    narrow range, offsets, spikes, constants, ramps, low-bit ties, huge values,
    +-inf and signed zeros, sparse peaks; ragged lengths including -1 and
    past-the-width."""
    rng = np.random.default_rng(seed)
    stride = 3000
    rows, lens = [], []
    kinds = ["normal", "narrow", "offset", "spike", "const", "asc", "lowbits", "huge",
             "special", "peaks"]
    for i, kind in enumerate(kinds * 2):
        if kind == "normal":
            x = rng.standard_normal(stride)
        elif kind == "narrow":
            x = (np.uint32(0x3F800000) + rng.integers(0, 8193, stride).astype(np.uint32)).view(np.float32)
        elif kind == "offset":
            x = rng.standard_normal(stride) + rng.uniform(-4, 4)
        elif kind == "spike":
            x = rng.standard_normal(stride)
            s = rng.random(stride) < 0.01
            x[s] += rng.uniform(3, 6, s.sum())
        elif kind == "const":
            x = np.full(stride, rng.standard_normal())
        elif kind == "asc":
            x = np.arange(stride, dtype=np.float64)
        elif kind == "lowbits":
            x = (np.uint32(0x3F800000) | rng.integers(0, 1024, stride).astype(np.uint32)).view(np.float32)
        elif kind == "huge":
            x = rng.uniform(65504, 1e6, stride)
        elif kind == "special":
            x = rng.standard_normal(stride)
            p = rng.integers(0, 8, stride)
            x[p == 0], x[p == 1], x[p == 2], x[p == 3] = -np.inf, np.inf, -0.0, 0.0
        else:
            x = rng.random(stride)
            x[np.arange(0, stride, 64)[:16]] += 150
        rows.append(np.asarray(x, dtype=np.float32))
        lens.append([stride, 2500, 1, 0, -1, stride + 17, 700, 64, 65, 1999][i % 10])
    scores = np.stack(rows)
    lengths = np.array(lens, dtype=np.int32)
    for b, n in enumerate(lengths):
        scores[b, valid_len(n, stride):] = np.nan
    return scores, lengths


# ------------------------------------------------ two-level indexer helpers

INT32_MAX = np.iinfo(np.int32).max
SENTINEL = np.float32(-12345.5)


def amax8_reference(scores, lengths, topk, width):
    """Block keys by numpy: pad each row to whole blocks of 8 with -inf and
    take the maximum over axis 1 of the [blocks, 8] view."""
    B, stride = scores.shape
    out = np.full((B, width), SENTINEL, dtype=np.float32)
    for b in range(B):
        n = valid_len(lengths[b], stride)
        nb = -(-n // 8)
        if nb == 0 or (topk > 0 and nb <= topk):
            continue
        padded = np.full(nb * 8, -np.inf, dtype=np.float32)
        padded[:n] = scores[b, :n]
        out[b, :nb] = padded.reshape(nb, 8).max(axis=1)
        out[b, nb - 1] = np.inf
    return out


def pin_amax8(orc) -> None:
    rng = np.random.default_rng(81)
    stride = 203
    scores = rng.standard_normal((40, stride)).astype(np.float32)
    scores[3] = np.arange(stride, dtype=np.float32)  # ascending: block i's max is 8i + 7
    scores[4] = -np.inf
    lengths = np.array([0, 1, 7, 8, 9, 16, 17, 203, 204, -5] + list(rng.integers(0, 260, 30)),
                       dtype=np.int32)
    lengths[3] = 203
    width = -(-stride // 8)
    for topk in (0, 1, 2, 3, 25, 26):
        init = np.full((40, width), SENTINEL, dtype=np.float32)
        got = orc.amax8_varlen(scores, lengths, topk, init)
        want = amax8_reference(scores, lengths, topk, width)
        assert np.array_equal(got, want), f"block keys differ (topk={topk})"
    got = orc.amax8_varlen(scores[3:4], lengths[3:4], 0, np.full((1, width), SENTINEL, np.float32))
    nb = -(-203 // 8)
    assert np.array_equal(got[0, : nb - 1], np.arange(nb - 1, dtype=np.float32) * 8 + 7)
    assert got[0, nb - 1] == np.inf


def blocks_reference(blocks, lengths, stride, page_table, page_size):
    """Block table by numpy: np.sort of the valid ids (identity when a row has
    at most k blocks), INT32_MAX padding, slots by the pool formula."""
    B, k = blocks.shape
    bpp = page_size // 8
    ids_out = np.full((B, k), INT32_MAX, dtype=np.int64)
    pages = np.full((B, k), INT32_MAX, dtype=np.int64)
    for b in range(B):
        nb = -(-valid_len(lengths[b], stride) // 8)
        ids = np.arange(nb) if nb <= k else np.sort(blocks[b][blocks[b] >= 0])
        ids_out[b, : len(ids)] = ids
        pages[b, : len(ids)] = page_table[b, ids // bpp].astype(np.int64) * bpp + ids % bpp
    return ids_out.astype(np.int32), pages.astype(np.int32)


def pin_sort_candidate_blocks(orc) -> None:
    rng = np.random.default_rng(82)
    B, k, stride = 24, 16, 800  # up to 100 blocks per row
    lengths = np.array([0, 1, 8, 128, 129, 136, 800, 900, -3] + list(rng.integers(0, 800, 15)),
                       dtype=np.int32)
    blocks = np.full((B, k), -7, dtype=np.int32)  # rows with <= k blocks: input ignored
    for b in range(B):
        nb = -(-valid_len(lengths[b], stride) // 8)
        if nb > k:
            sel = rng.choice(nb, k, replace=False).astype(np.int32)
            blocks[b] = sel  # any order
    for page_size in (8, 16, 64):
        bpp = page_size // 8
        pt = rng.permutation(B * (100 // bpp + 1)).astype(np.int32).reshape(B, -1)
        got_ids, got_pages = orc.sort_candidate_blocks(blocks, lengths, stride, pt, page_size)
        want_ids, want_pages = blocks_reference(blocks, lengths, stride, pt, page_size)
        assert np.array_equal(got_ids, want_ids), f"block ids differ (page {page_size})"
        assert np.array_equal(got_pages, want_pages), f"pool slots differ (page {page_size})"
    # a row with exactly k blocks is the identity; a padded (-1) entry in a row
    # that needs k ids, or a duplicate, is refused
    one = np.full((1, k), -1, dtype=np.int32)
    ids, _ = orc.sort_candidate_blocks(one, np.array([8 * k], np.int32), stride,
                                       np.zeros((1, 100), np.int32), 8)
    assert np.array_equal(ids[0], np.arange(k))
    bad = np.arange(k, dtype=np.int32)[None, :].copy()
    bad[0, 3] = -1
    for b_ in (bad, np.where(np.arange(k) == 5, 4, np.arange(k)).astype(np.int32)[None, :]):
        try:
            orc.sort_candidate_blocks(b_, np.array([8 * k + 8], np.int32), stride,
                                      np.zeros((1, 100), np.int32), 8)
        except RuntimeError:
            continue
        raise AssertionError("a malformed block row was accepted")


def run_all_pins(orc, quick: bool = False) -> None:
    pin_golden(orc)
    pin_closed_forms(orc)
    pin_nan_rejected(orc)
    pin_bruteforce(orc, cases=150 if quick else 600)
    scores, lengths = small_inputs()
    for k in (64, 512):
        out = _run(orc, scores, lengths, k)
        check_selection(scores, lengths, k, out)
        pin_lexsort(orc, scores, lengths, k)
    rng = np.random.default_rng(5)
    pt = rng.permutation(scores.shape[0] * 48).astype(np.int32).reshape(scores.shape[0], 48)
    pin_paged_formula(orc, scores, lengths, 64, pt, 64)
    pin_amax8(orc)
    pin_sort_candidate_blocks(orc)
