"""Parity of the two-level indexer's helpers (block-max keys and the
candidate block table) with the CPU oracle, alone and chained around the
top-k (needs an sm_103 GPU)."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpu_helpers import to_dev  # noqa: E402
from synth import make_workload  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_indexer_fp32_gb300 as tk  # noqa: E402

SENTINEL = np.float32(-12345.5)
INT32_MAX = np.iinfo(np.int32).max


@pytest.mark.parametrize("stride", [4096, 4093, 65536])
@pytest.mark.parametrize("topk", [0, 3, 64])
def test_amax8_matches_the_oracle(stride, topk):
    """Aligned rows (vector loads) and an odd stride (scalar loads); lengths
    around block boundaries; rows skipped by topk keep the sentinel."""
    rng = np.random.default_rng(stride + topk)
    B = 24
    scores = rng.standard_normal((B, stride)).astype(np.float32)
    scores[2] = -np.inf
    # blocks whose maximum is a zero of either sign, in either order
    zeros = rng.choice([-0.0, 0.0, -1.0, -np.inf], size=(4, stride), p=[0.4, 0.1, 0.4, 0.1])
    scores[10:14] = zeros.astype(np.float32)
    scores[10, :16] = [-0.0, 0.0, -1, -1, -1, -1, -1, -1, 0.0, -0.0, -1, -1, -1, -1, -1, -1]
    lengths = np.array([0, 1, 7, 8, 9, 24, 25, stride, stride + 3, -1]
                       + list(rng.integers(0, stride, B - 10)), dtype=np.int32)
    width = -(-stride // 8)
    init = np.full((B, width), SENTINEL, dtype=np.float32)
    out = to_dev(init)
    tk.amax8_varlen(to_dev(scores), to_dev(lengths), topk, out=out)
    torch.cuda.synchronize()
    want = oracle.amax8_varlen(scores, lengths, topk, init)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), "keys differ (bit for bit)"
    if topk == 0:  # the case does hold zero maxima of both signs
        z = want[10:14].view(np.uint32)
        assert (z == 0).any() and (z == 0x80000000).any()


@pytest.mark.parametrize("page_size", [8, 64])
@pytest.mark.parametrize("k", [1, 100, 2048])
def test_sort_candidate_blocks_matches_the_oracle(page_size, k):
    rng = np.random.default_rng(k + page_size)
    B, stride = 16, 131072
    lengths = np.array([0, 5, 8 * k, 8 * k + 1, stride, 8 * k - 8] + list(rng.integers(0, stride, B - 6)),
                       dtype=np.int32)
    blocks = np.full((B, k), -1, dtype=np.int32)
    for b in range(B):
        nb = -(-min(max(int(lengths[b]), 0), stride) // 8)
        if nb > k:
            blocks[b] = rng.choice(nb, k, replace=False)
        else:
            blocks[b] = rng.integers(-1, 5, k)  # ignored: the identity table
    bpp = page_size // 8
    pt = rng.permutation(B * (stride // 8 // bpp)).astype(np.int32).reshape(B, -1)
    d_blocks = to_dev(blocks)
    pages = tk.sort_candidate_blocks(d_blocks, to_dev(lengths), stride, to_dev(pt), page_size)
    torch.cuda.synchronize()
    want_ids, want_pages = oracle.sort_candidate_blocks(blocks, lengths, stride, pt, page_size)
    assert np.array_equal(d_blocks.cpu().numpy(), want_ids)
    assert np.array_equal(pages.cpu().numpy(), want_pages)


def test_two_level_pipeline_matches_the_oracle_pipeline():
    """Block keys -> top-k over the keys (lengths ceil(n / 8)) -> block table,
    on rows of the 262144-wide paged workload, against the oracle's chain."""
    w = make_workload(4, B=32)
    k_blocks, page_size = 512, 64
    nb = -(-np.clip(w.lengths.astype(np.int64), 0, w.stride) // 8)
    blen = nb.astype(np.int32)
    width = -(-w.stride // 8)
    s, l = to_dev(w.scores), to_dev(w.lengths)
    init = np.full((w.B, width), SENTINEL, dtype=np.float32)
    keys = tk.amax8_varlen(s, l, k_blocks, out=to_dev(init))
    sel = tk.topk_ragged(keys, to_dev(blen), k_blocks)
    pt = w.page_table[:, : width * 8 // page_size]  # 64-token pages of blocks
    pages = tk.sort_candidate_blocks(sel, l, w.stride, to_dev(pt), page_size)
    torch.cuda.synchronize()

    want_keys = oracle.amax8_varlen(w.scores, w.lengths, k_blocks, init)
    assert np.array_equal(keys.cpu().numpy(), want_keys)
    want_sel = oracle.topk_ragged(want_keys, blen, k_blocks)
    want_ids, want_pages = oracle.sort_candidate_blocks(want_sel, w.lengths, w.stride, pt, page_size)
    assert np.array_equal(sel.cpu().numpy(), want_ids)
    assert np.array_equal(pages.cpu().numpy(), want_pages)
