"""The allocation-free entry point, topk_select_noalloc (needs an sm_103 GPU).

Some callers cannot allocate device memory at the moment they select: a
serving engine that reserves nearly all of HBM for its KV cache and forbids
allocation on the decode path, or a plugin with no access to its host
framework's allocator. For them the library keeps the scratch of split rows
in a fixed array of its own. These tests call that entry point through the C
ABI and require exactly the output of the regular entry point, on two calls in
a row (the second one finds the array as the first left it).

The file is named to be collected last, so that a run stopping at the first
failure has run every other test before it.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gpu_helpers import counters_tensor, to_dev  # noqa: E402
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


@pytest.mark.parametrize("paged", [False, True])
def test_noalloc_matches_the_regular_entry_point_on_two_calls(paged):
    lib = tk.load_library()
    # 160 rows of width 262144: too many rows for a cluster per row, and the
    # last 144 are split over two CTAs (they fill the 2 x 152 slots that 160
    # one-CTA rows leave idle), so the call goes through the static scratch.
    w = make_workload(4, B=160)
    s, l = to_dev(w.scores), to_dev(w.lengths)
    pt = to_dev(w.page_table) if paged else None
    if paged:
        want = tk.topk_paged(s, l, w.k, pt, w.page_size, split=False)
    else:
        want = tk.topk_ragged(s, l, w.k, split=False)

    # The automatic policy does split these rows (seen through the regular
    # workspace call with counters).
    cnt = counters_tensor()
    ws = torch.zeros(tk.workspace_bytes(w.k), dtype=torch.uint8, device="cuda:0")
    tk.topk_select_ex(s, l, w.k, pt, w.page_size if paged else 0, workspace=ws, counters=cnt)
    torch.cuda.synchronize()
    assert int(cnt[tk.Counter.SPLIT_ROWS]) == 144

    for call in range(2):
        got = torch.full_like(want, -7)
        status = _noalloc(lib, s, l, w.k, got, pt, w.page_size if paged else 0)
        assert status == tk.Status.OK, lib.topk_status_string(status)
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"call {call}: output differs from the regular entry point"


def test_noalloc_refuses_calls_beyond_its_scratch():
    """153 rows of width 196608 at k = 2048 would split 151 rows (32 KiB of
    scratch each, 4.7 MiB in all): more than the 4 MiB array holds, so the
    call is refused before anything runs and the output is untouched."""
    lib = tk.load_library()
    B, stride, k = 153, 196608, 2048
    s = torch.zeros((B, stride), dtype=torch.float32, device="cuda:0")
    l = torch.full((B,), stride, dtype=torch.int32, device="cuda:0")
    out = torch.full((B, k), -7, dtype=torch.int32, device="cuda:0")
    status = _noalloc(lib, s, l, k, out)
    assert status == tk.Status.ESCRATCH
    assert b"static workspace" in lib.topk_status_string(status)
    torch.cuda.synchronize()
    assert torch.all(out == -7)
    # a smaller k fits
    out512 = torch.empty((B, 512), dtype=torch.int32, device="cuda:0")
    assert _noalloc(lib, s, l, 512, out512) == tk.Status.OK
    torch.cuda.synchronize()
    assert np.array_equal(np.sort(out512.cpu().numpy(), axis=1),
                          np.broadcast_to(np.arange(512, dtype=np.int32), (B, 512)))
