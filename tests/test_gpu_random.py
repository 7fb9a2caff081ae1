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

from random_cases import MAX_ELEMENTS, N_CASES, draw_case, draw_lengths, row_values  # noqa: E402


def _device_rows(scores, offset):
    B, width = scores.shape
    flat = np.full(B * width + 4, np.nan, dtype=np.float32)
    flat[offset: offset + B * width] = scores.ravel()
    return to_dev(flat)[offset: offset + B * width].view(B, width)


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_case_through_the_automatic_path(case):
    scores, lengths, k, offset, pt, page_size = draw_case(case)
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
    scores, lengths, k, offset, pt, page_size = draw_case(case)
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
    scores, lengths, k, offset, pt, page_size = draw_case(case)
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
    lengths = draw_lengths(rng, int(rng.integers(0, 3)), B, stride, 8 * k_blocks)
    lengths = np.clip(lengths, -2, stride + 20).astype(np.int32)
    scores = np.full((B, stride), np.nan, dtype=np.float32)
    for b in range(B):
        n = int(min(max(lengths[b], 0), stride))
        scores[b, :n] = row_values(rng, int(rng.integers(0, 8)), n).astype(np.float32)
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
    scores, lengths, k, offset, pt, page_size = draw_case(case)
    B, width = scores.shape
    rng = np.random.default_rng([0x5EED, 0xF025, case])
    new_lengths = draw_lengths(rng, int(rng.integers(0, 6)), B, width, k)
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
