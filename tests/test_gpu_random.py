"""Seeded random cases through the automatic dispatch (needs an sm_103 GPU).

The other GPU tests force each path or run the fixed workloads; here every
case draws a batch size, a row width (1 to 300000), k, a length mode (full,
80-100 %, anything, around k, up to 2k, up to k + 16384), value
kinds with ties, infinities and signed zeros, a row start that may not sit on
16 bytes, and paging, and lets the library choose its path (short-row kernel,
sampled cutoff, clusters, split rows). Each result must equal the oracle's
(identical -1 pattern, index set and value multiset), the split and unsplit
calls must agree slot for slot, and a second call must repeat the first.
Each case also runs once on a randomly forced path (clusters of 1 to 16,
split rows, the short-row kernel, sampling on or off, the smallest candidate
buffer). Rows of at most 16384 scores also go through the BF16 entry point,
compared with the oracle on the BF16-rounded values.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gpu_helpers import assert_parity, run_oracle, to_dev  # noqa: E402
from synth import bf16_bits_to_float, to_bf16_bits  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_indexer_fp32_gb300 as tk  # noqa: E402

N_CASES = 96
MAX_ELEMENTS = 12_000_000  # per case, so that the oracle's full sorts stay quick


def _row_values(rng, kind, width):
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


def _lengths(rng, mode, B, width, k):
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


def _case(i):
    rng = np.random.default_rng([0x5EED, 0xF022, i])
    if rng.random() < 0.3:  # long rows: the sampled cutoff, clusters and split rows
        width = int(rng.integers(65536, 300001))
    else:
        width = int(np.exp(rng.uniform(0.0, np.log(300000.0))))
    B = int(np.exp(rng.uniform(0.0, np.log(1200.0))))
    while B > 1 and B * width > MAX_ELEMENTS:
        B //= 2
    k = int(rng.choice([1, 2, 17, 100, 511, 512, 513, 1000, 1024, 2047, 2048, int(rng.integers(1, 2049))]))
    lengths = _lengths(rng, int(rng.integers(0, 6)), B, width, k)
    scores = np.full((B, width), np.nan, dtype=np.float32)
    for b in range(B):
        n = int(min(max(lengths[b], 0), width))
        scores[b, :n] = _row_values(rng, int(rng.integers(0, 8)), n).astype(np.float32)
    offset = int(rng.integers(0, 4))  # floats before row 0 in the device buffer
    paged = bool(rng.integers(0, 2))
    page_size = int(rng.choice([1, 7, 16, 64]))
    pages = -(-width // page_size)
    pt = rng.permutation(B * pages).astype(np.int32).reshape(B, pages) if paged else None
    return scores, np.clip(lengths, -2**31, 2**31 - 1).astype(np.int32), k, offset, pt, page_size


def _device_rows(scores, offset):
    B, width = scores.shape
    flat = np.full(B * width + 4, np.nan, dtype=np.float32)
    flat[offset: offset + B * width] = scores.ravel()
    return to_dev(flat)[offset: offset + B * width].view(B, width)


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_case_through_the_automatic_path(case):
    scores, lengths, k, offset, pt, page_size = _case(case)
    s, l = _device_rows(scores, offset), to_dev(lengths)
    if pt is None:
        got = tk.topk_ragged(s, l, k)
        again = tk.topk_ragged(s, l, k)
        unsplit = tk.topk_ragged(s, l, k, split=False)
        want = run_oracle(scores, lengths, k)
    else:
        dpt = to_dev(pt)
        got = tk.topk_paged(s, l, k, dpt, page_size)
        again = tk.topk_paged(s, l, k, dpt, page_size)
        unsplit = tk.topk_paged(s, l, k, dpt, page_size, split=False)
        want = run_oracle(scores, lengths, k, pt, page_size)
    torch.cuda.synchronize()
    assert torch.equal(got, again)
    assert torch.equal(got, unsplit)
    assert_parity(scores, lengths, k, got.cpu().numpy(), want, page_table=pt)


def _forced_options(case, B, stride, k):
    """A random forced path for the case: the streaming kernel on clusters of
    1 to 16, split rows, or the short-row kernel, with random sampling and
    candidate-buffer capacity."""
    rng = np.random.default_rng([0x5EED, 0xF023, case])
    cap_max = 2560 if k <= 512 else 5120
    caps = [c for c in (0, k + 2048, cap_max) if c == 0 or k + 2048 <= c <= cap_max]
    opts = {"sample_mode": int(rng.integers(0, 3)), "stash_capacity": int(rng.choice(caps))}
    kind = int(rng.integers(0, 3))
    if kind == 2 and stride <= 16384:
        return {"short_rows": 1, "sample_mode": opts["sample_mode"]}
    opts["short_rows"] = -1
    if kind == 1:
        m = int(rng.integers(1, min(B, 1024) + 1))
        opts["split_rows"] = m
        opts["workspace"] = torch.zeros(tk.workspace_bytes(k, m), dtype=torch.uint8, device="cuda:0")
    else:
        opts["cluster_size"] = int(rng.choice([1, 2, 4, 8, 16]))
    return opts


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_case_on_a_forced_path(case):
    scores, lengths, k, offset, pt, page_size = _case(case)
    B, stride = scores.shape
    opts = _forced_options(case, B, stride, k)
    s, l = _device_rows(scores, offset), to_dev(lengths)
    dpt = None if pt is None else to_dev(pt)
    got = tk.topk_select_ex(s, l, k, dpt, page_size if pt is not None else 0, **opts)
    torch.cuda.synchronize()
    if "workspace" in opts:
        assert not torch.any(opts["workspace"][:4096]), "arrival counters must be left at zero"
    want = run_oracle(scores, lengths, k) if pt is None else run_oracle(scores, lengths, k, pt, page_size)
    assert_parity(scores, lengths, k, got.cpu().numpy(), want, page_table=pt)


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_case_in_bf16(case):
    scores, lengths, k, offset, pt, page_size = _case(case)
    if scores.shape[1] > 16384:
        pytest.skip("BF16 rows hold at most 16384 scores")
    bits = to_bf16_bits(scores)
    vals = bf16_bits_to_float(bits)
    B, width = bits.shape
    flat = np.zeros(B * width + 8, dtype=np.uint16)
    flat[offset: offset + B * width] = bits.ravel()
    s = torch.from_numpy(flat.view(np.int16)).to("cuda:0")[offset: offset + B * width].view(B, width)
    s = s.view(torch.bfloat16)
    l = to_dev(lengths)
    if pt is None:
        got = tk.topk_select_bf16(s, l, k)
        want = run_oracle(vals, lengths, k)
    else:
        got = tk.topk_select_bf16(s, l, k, to_dev(pt), page_size)
        want = run_oracle(vals, lengths, k, pt, page_size)
    torch.cuda.synchronize()
    assert_parity(vals, lengths, k, got.cpu().numpy(), want, page_table=pt)


N_CHAIN_CASES = 24


@pytest.mark.parametrize("case", range(N_CHAIN_CASES))
def test_random_two_level_chain(case):
    """Block keys (padded output rows), top-k over the keys, block table:
    each step against the oracle's, bit for bit, on seeded random shapes."""
    import oracle

    rng = np.random.default_rng([0x5EED, 0xF024, case])
    stride = int(np.exp(rng.uniform(np.log(8.0), np.log(70000.0))))
    B = int(rng.integers(1, 201))
    while B > 1 and B * stride > MAX_ELEMENTS // 2:
        B //= 2
    k_blocks = int(rng.choice([1, 17, 100, 512, 1000, 2048]))
    lengths = _lengths(rng, int(rng.integers(0, 3)), B, stride, 8 * k_blocks)
    lengths = np.clip(lengths, -2, stride + 20).astype(np.int32)
    scores = np.full((B, stride), np.nan, dtype=np.float32)
    for b in range(B):
        n = int(min(max(lengths[b], 0), stride))
        scores[b, :n] = _row_values(rng, int(rng.integers(0, 8)), n).astype(np.float32)
    width = -(-stride // 8)
    out_stride = width + int(rng.integers(0, 10))
    init = np.full((B, out_stride), np.float32(-12345.5), dtype=np.float32)
    page_size = int(rng.choice([8, 16, 64]))
    bpp = page_size // 8
    pt = rng.permutation(B * -(-width // bpp)).astype(np.int32).reshape(B, -1)
    nb = -(-np.clip(lengths.astype(np.int64), 0, stride) // 8)
    blen = nb.astype(np.int32)

    keys = tk.amax8_varlen(to_dev(scores), to_dev(lengths), k_blocks, out=to_dev(init))
    sel = tk.topk_ragged(keys, to_dev(blen), k_blocks)
    pages = tk.sort_candidate_blocks(sel, to_dev(lengths), stride, to_dev(pt), page_size)
    torch.cuda.synchronize()

    want_keys = oracle.amax8_varlen(scores, lengths, k_blocks, init)
    assert np.array_equal(keys.cpu().numpy().view(np.uint32), want_keys.view(np.uint32))
    want_sel = oracle.topk_ragged(want_keys, blen, k_blocks)
    want_ids, want_pages = oracle.sort_candidate_blocks(want_sel, lengths, stride, pt, page_size)
    assert np.array_equal(sel.cpu().numpy(), want_ids)
    assert np.array_equal(pages.cpu().numpy(), want_pages)


@pytest.mark.parametrize("case", range(0, N_CASES, 6))
def test_random_case_replayed_from_a_graph_with_new_lengths(case):
    """The automatic call captured in a CUDA graph (its path fixed at capture
    from B, the width and k), replayed after the lengths were rewritten in
    place with another draw: the oracle's result for the new lengths."""
    scores, lengths, k, offset, pt, page_size = _case(case)
    B, width = scores.shape
    rng = np.random.default_rng([0x5EED, 0xF025, case])
    new_lengths = _lengths(rng, int(rng.integers(0, 6)), B, width, k)
    new_lengths = np.clip(new_lengths, -2, width + 20).astype(np.int32)
    full = np.asarray(scores, dtype=np.float32).copy()
    for b in range(B):  # valid scores wherever either draw reads
        n = int(min(max(max(lengths[b], new_lengths[b]), 0), width))
        holes = np.isnan(full[b, :n])
        full[b, :n][holes] = rng.standard_normal(int(holes.sum())).astype(np.float32)
    s, l = _device_rows(full, offset), to_dev(lengths)
    dpt = None if pt is None else to_dev(pt)
    out = torch.empty((B, k), dtype=torch.int32, device="cuda:0")
    stream = torch.cuda.Stream()

    def call():
        if dpt is None:
            tk.topk_ragged(s, l, k, out=out)
        else:
            tk.topk_paged(s, l, k, dpt, page_size, out=out)

    with torch.cuda.stream(stream):
        call()  # creates the stream's workspace outside the capture
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            call()
        l.copy_(torch.from_numpy(new_lengths))
        graph.replay()
        stream.synchronize()
    want = run_oracle(full, new_lengths, k) if pt is None else run_oracle(full, new_lengths, k, pt, page_size)
    assert_parity(full, new_lengths, k, out.cpu().numpy(), want, page_table=pt)
