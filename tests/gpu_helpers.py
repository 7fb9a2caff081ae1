"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
binding and compare with the CPU oracle on the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import oracle_pins as P
import sparse_attention_indexer_fp32_gb300 as tk


def to_dev(a: np.ndarray, device="cuda:0") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def run_gpu(scores: np.ndarray, lengths: np.ndarray, k: int, page_table=None, page_size=0,
            **opts) -> np.ndarray:
    s = to_dev(scores)
    l = to_dev(lengths.astype(np.int32))
    pt = None if page_table is None else to_dev(page_table.astype(np.int32))
    if opts:
        out = tk.topk_select_ex(s, l, k, pt, page_size, **opts)
    elif pt is None:
        out = tk.topk_ragged(s, l, k)
    else:
        out = tk.topk_paged(s, l, k, pt, page_size)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def run_oracle(scores, lengths, k, page_table=None, page_size=0) -> np.ndarray:
    if page_table is None:
        return oracle.topk_ragged(scores, lengths, k)
    return oracle.topk_paged(scores, lengths, k, page_table, page_size)


def assert_parity(scores, lengths, k, got, want, rows=None, page_table=None) -> None:
    """Row by row: identical -1 pattern, identical index sets (both sides take
    the lowest indices among ties at the cutoff), and - for ragged output -
    bit-identical selected value multisets."""
    B = got.shape[0]
    assert got.shape == want.shape, (got.shape, want.shape)
    stride = scores.shape[1]
    bad = []
    for b in range(B):
        n = P.valid_len(lengths[b], stride)
        m = min(k, n)
        g, w_ = got[b], want[b]
        if not np.all(g[m:] == -1):
            bad.append((b, "padding"))
            continue
        gs, ws = np.sort(g[:m]), np.sort(w_[:m])
        if not np.array_equal(gs, ws):
            if page_table is None and m and np.all((g[:m] >= 0) & (g[:m] < n)):
                gv = np.sort(scores[b, g[:m]].view(np.uint32))
                wv = np.sort(scores[b, w_[:m]].view(np.uint32))
                bad.append((b, "index set differs; values " +
                            ("equal" if np.array_equal(gv, wv) else "DIFFER")))
            else:
                bad.append((b, "index set differs"))
    label = "" if rows is None else f" (rows {list(rows)[:8]}...)"
    assert not bad, f"{len(bad)} rows differ{label}: {bad[:10]}"


def check_against_oracle(scores, lengths, k, page_table=None, page_size=0, **opts):
    got = run_gpu(scores, lengths, k, page_table, page_size, **opts)
    want = run_oracle(scores, lengths, k, page_table, page_size)
    assert_parity(scores, lengths, k, got, want, page_table=page_table)
    return got


def counters_tensor():
    return torch.zeros(tk.NUM_COUNTERS, dtype=torch.int32, device="cuda:0")
