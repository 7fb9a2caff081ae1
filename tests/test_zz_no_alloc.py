"""The allocation-free entry point, topk_select_noalloc (needs an sm_103 GPU).

Some callers cannot allocate device memory at the moment they select: a
serving engine that reserves nearly all of HBM for its KV cache and forbids
allocation on the decode path, or a plugin with no access to its host
framework's allocator. For them the library keeps the scratch of split rows
in a fixed array of its own. These tests call that entry point through the C
ABI and require exactly the output of the regular entry point, on two calls in
a row (the second one finds the array as the first left it), and the CPU
oracle's selection on a sample of rows that includes the split ones.

The file is named to be collected last, so that a run stopping at the first
failure has run every other test before it.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gpu_helpers import assert_parity, counters_tensor, run_oracle, to_dev  # noqa: E402
from synth import make_workload  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_indexer_fp32_gb300 as tk  # noqa: E402


def _noalloc(lib, s, l, k, out, pt=None, page_size=0):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.topk_select_noalloc(s.data_ptr(), s.shape[1], l.data_ptr(), s.shape[0], k,
                                   None if pt is None else pt.data_ptr(),
                                   0 if pt is None else pt.shape[1], page_size, out.data_ptr(),
                                   stream)


def _sm_count() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def _split_rows_expected(B: int, stride: int, sms: int) -> int:
    """Rows the library splits in a batch of one-CTA rows: the ones that fill
    the slots (two CTAs per SM) that the last partial wave leaves idle, rows
    of width 196608 and more only."""
    slots = 2 * sms
    if stride < 196608:
        return 0
    r = B % slots if B >= slots else B
    return min(r, slots - r)


@pytest.mark.parametrize("paged", [False, True])
def test_noalloc_matches_the_regular_entry_point_on_two_calls(paged):
    lib = tk.load_library()
    sms = _sm_count()
    # A few more rows of width 262144 than the GPU has SMs: too many for a
    # cluster per row, and all but 8 of them are split over two CTAs (they fill
    # the two slots per SM that one-CTA rows leave idle), so the call goes
    # through the static scratch.
    B = sms + 8
    w = make_workload(4, B=B)
    s, l = to_dev(w.scores), to_dev(w.lengths)
    pt = to_dev(w.page_table) if paged else None
    ps = w.page_size if paged else 0
    if paged:
        want = tk.topk_paged(s, l, w.k, pt, w.page_size, split=False)
    else:
        want = tk.topk_ragged(s, l, w.k, split=False)

    # The automatic policy does split these rows (seen through the regular
    # workspace call with counters).
    cnt = counters_tensor()
    ws = torch.zeros(tk.workspace_bytes(w.k), dtype=torch.uint8, device="cuda:0")
    tk.topk_select_ex(s, l, w.k, pt, ps, workspace=ws, counters=cnt)
    torch.cuda.synchronize()
    split = _split_rows_expected(B, w.stride, sms)
    assert split == sms - 8
    assert int(cnt[tk.Counter.SPLIT_ROWS]) == split

    for call in range(2):
        got = torch.full_like(want, -7)
        status = _noalloc(lib, s, l, w.k, got, pt, ps)
        assert status == tk.Status.OK, lib.topk_status_string(status)
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"call {call}: output differs from the regular entry point"

    # and the oracle's selection, on rows before and inside the split range
    rows = np.array([0, 3, B - split - 1, B - split, B - split + 1, B - 2, B - 1])
    pt_rows = w.page_table[rows] if paged else None
    assert_parity(w.scores[rows], w.lengths[rows], w.k, got.cpu().numpy()[rows],
                  run_oracle(w.scores[rows], w.lengths[rows], w.k, pt_rows, ps), rows=rows,
                  page_table=pt_rows)


def test_noalloc_refuses_calls_beyond_its_scratch():
    """One row more than the GPU has SMs, of width 196608 at k = 2048: all but
    one row would be split (32 KiB of scratch each), more than the 4 MiB array
    holds, so the call is refused before anything runs and the output is
    untouched. A smaller k fits."""
    lib = tk.load_library()
    sms = _sm_count()
    B, stride, k = sms + 1, 196608, 2048
    split = _split_rows_expected(B, stride, sms)
    if split * 2 * k * 8 <= 4 * 1024 * 1024:
        pytest.skip(f"{sms} SMs: every split of this shape fits the array")
    s = torch.zeros((B, stride), dtype=torch.float32, device="cuda:0")
    l = torch.full((B,), stride, dtype=torch.int32, device="cuda:0")
    out = torch.full((B, k), -7, dtype=torch.int32, device="cuda:0")
    status = _noalloc(lib, s, l, k, out)
    assert status == tk.Status.ESCRATCH
    assert b"static workspace" in lib.topk_status_string(status)
    torch.cuda.synchronize()
    assert torch.all(out == -7)
    # a smaller k fits (512: 8 KiB per split row)
    out512 = torch.empty((B, 512), dtype=torch.int32, device="cuda:0")
    assert _noalloc(lib, s, l, 512, out512) == tk.Status.OK
    torch.cuda.synchronize()
    assert np.array_equal(np.sort(out512.cpu().numpy(), axis=1),
                          np.broadcast_to(np.arange(512, dtype=np.int32), (B, 512)))


def test_noalloc_deterministic_over_100_calls():
    """The allocation-free call on the paged full-size batch (its last rows
    split through the static scratch), 100 times: byte-identical output."""
    lib = tk.load_library()
    w = make_workload(4)
    s, l, pt = to_dev(w.scores), to_dev(w.lengths), to_dev(w.page_table)
    first = torch.empty((w.B, w.k), dtype=torch.int32, device="cuda:0")
    assert _noalloc(lib, s, l, w.k, first, pt, w.page_size) == tk.Status.OK
    out = torch.empty_like(first)
    differing = 0
    for _ in range(99):
        assert _noalloc(lib, s, l, w.k, out, pt, w.page_size) == tk.Status.OK
        differing += int(not torch.equal(out, first))
    assert differing == 0
    assert torch.equal(first, tk.topk_paged(s, l, w.k, pt, w.page_size, split=False))


@pytest.mark.parametrize("B,stride,k", [(300, 8192, 512), (200, 16384, 2048), (4, 262144, 512),
                                        (40, 98307, 1024)])
def test_noalloc_without_scratch_paths(B, stride, k):
    """Calls that split no row (short rows, a small batch on clusters, rows
    narrower than the split gate) go through the same entry point and match
    the regular call and the oracle."""
    lib = tk.load_library()
    rng = np.random.default_rng(B + stride)
    scores = rng.standard_normal((B, stride)).astype(np.float32)
    lengths = rng.integers(stride * 4 // 5, stride + 1, B).astype(np.int32)
    s, l = to_dev(scores), to_dev(lengths)
    want = tk.topk_ragged(s, l, k)
    got = torch.full_like(want, -7)
    assert _noalloc(lib, s, l, k, got) == tk.Status.OK
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    rows = np.arange(0, B, max(1, B // 6))
    assert_parity(scores[rows], lengths[rows], k, got.cpu().numpy()[rows],
                  run_oracle(scores[rows], lengths[rows], k), rows=rows)


@pytest.mark.parametrize("case", range(24))
def test_noalloc_on_random_cases(case):
    """The seeded random cases of the automatic-path tests (any batch, width,
    k, length mode, row offset and paging) through the allocation-free entry
    point: the regular call's output and the oracle's selection, or a refusal
    that leaves the output untouched when the split rows need more scratch
    than the array holds."""
    import test_gpu_random as R
    from random_cases import draw_case

    lib = tk.load_library()
    scores, lengths, k, offset, pt, page_size = draw_case(case)
    s, l = R._device_rows(scores, offset), to_dev(lengths)
    dpt = None if pt is None else to_dev(pt)
    want = tk.topk_ragged(s, l, k) if pt is None else tk.topk_paged(s, l, k, dpt, page_size)
    got = torch.full_like(want, -7)
    status = _noalloc(lib, s, l, k, got, dpt, page_size if pt is not None else 0)
    torch.cuda.synchronize()
    if status == tk.Status.ESCRATCH:
        assert torch.all(got == -7)
        return
    assert status == tk.Status.OK, lib.topk_status_string(status)
    assert torch.equal(got, want)
    assert_parity(scores, lengths, k, got.cpu().numpy(),
                  run_oracle(scores, lengths, k) if pt is None else run_oracle(scores, lengths, k, pt, page_size),
                  page_table=pt)
