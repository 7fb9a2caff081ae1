"""Full-size workloads (B=1024 x 131072 / 262144), in the launch configuration
the benchmark times: every row is checked by properties that hold at any size,
and a sample of rows is compared element by element with the CPU oracle."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle_pins as P  # noqa: E402
from gpu_helpers import assert_parity, run_oracle, to_dev  # noqa: E402
from synth import make_workload  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_indexer_fp32_gb300 as tk  # noqa: E402

SAMPLED_ROWS = 24


def _properties_all_rows(scores, lengths, k, out):
    """Exactly min(k, n) unique indices in [0, n), -1 after them, and no
    unselected score outranking a selected one - for every row."""
    B, stride = scores.shape
    for b in range(B):
        n = P.valid_len(lengths[b], stride)
        m = min(k, n)
        sel = out[b, :m]
        assert np.all(out[b, m:] == -1), b
        assert np.all((sel >= 0) & (sel < n)), b
        assert np.unique(sel).size == m, b
        if m < n:
            tov = P.total_order(scores[b, :n])
            chosen = np.zeros(n, dtype=bool)
            chosen[sel] = True
            assert tov[chosen].min() >= tov[~chosen].max(), b


@pytest.mark.parametrize("config", [3, 4])
def test_full_size_workload(config):
    w = make_workload(config)
    s, l = to_dev(w.scores), to_dev(w.lengths)
    ragged = tk.topk_ragged(s, l, w.k).cpu().numpy()
    _properties_all_rows(w.scores, w.lengths, w.k, ragged)

    # the last rows of the batch are the ones split over two CTAs
    rows = np.concatenate([np.random.default_rng(config).choice(w.B - 8, SAMPLED_ROWS, replace=False),
                           np.arange(w.B - 8, w.B)])
    want = run_oracle(w.scores[rows], w.lengths[rows], w.k)
    assert_parity(w.scores[rows], w.lengths[rows], w.k, ragged[rows], want, rows=rows)

    if w.paged:
        pt = to_dev(w.page_table)
        paged = tk.topk_paged(s, l, w.k, pt, w.page_size).cpu().numpy()
        assert np.array_equal(paged, P.page_map_reference(ragged, w.page_table, w.page_size))
        want_p = run_oracle(w.scores[rows], w.lengths[rows], w.k, w.page_table[rows], w.page_size)
        assert_parity(w.scores[rows], w.lengths[rows], w.k, paged[rows], want_p, rows=rows,
                      page_table=w.page_table)
    # the same answer on a second call, and without splitting any row
    again = tk.topk_ragged(s, l, w.k).cpu().numpy()
    assert np.array_equal(again, ragged)
    unsplit = tk.topk_ragged(s, l, w.k, split=False).cpu().numpy()
    assert np.array_equal(unsplit, ragged)


@pytest.mark.parametrize("config", [3, 4])
def test_full_size_deterministic_over_100_calls(config):
    """The benchmarked launch (one CTA per row, the last rows split over two
    CTAs and merged by whichever half finishes second) gives byte-identical
    output on 100 calls with the same input, and that output is the oracle's
    on sampled rows, the split ones included."""
    w = make_workload(config)
    s, l = to_dev(w.scores), to_dev(w.lengths)
    out = torch.empty((w.B, w.k), dtype=torch.int32, device="cuda:0")
    if w.paged:
        pt = to_dev(w.page_table)
        call = lambda: tk.topk_paged(s, l, w.k, pt, w.page_size, out=out)  # noqa: E731
    else:
        call = lambda: tk.topk_ragged(s, l, w.k, out=out)  # noqa: E731
    first = call().clone()
    differing = 0
    for _ in range(99):
        call()
        differing += int(not torch.equal(out, first))
    assert differing == 0, f"{differing} of 99 repeated calls differ from the first"
    rows = np.array([0, 1, w.B // 2, w.B - 120, w.B - 3, w.B - 2, w.B - 1])
    got = first.cpu().numpy()[rows]
    pt_rows = w.page_table[rows] if w.paged else None
    want = run_oracle(w.scores[rows], w.lengths[rows], w.k, pt_rows, w.page_size)
    assert_parity(w.scores[rows], w.lengths[rows], w.k, got, want, rows=rows, page_table=pt_rows)
