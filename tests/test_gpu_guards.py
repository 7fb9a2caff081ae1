"""Guard zones around every output and workspace (needs an sm_103 GPU).

compute-sanitizer is not available on the GPUs these tests run on, so writes
outside the buffers a call owns are caught the plain way: each output is the
inner view of a larger buffer whose guard rows (before row 0 and after row
B - 1) hold a sentinel, and a workspace is followed by a guard tail. After
calls on every path the library has - sampled and unsampled streaming,
in-buffer compaction, clusters of 8, split rows, paged output, the short-row
kernel, BF16 scores, the allocation-free entry point, the block keys (with
padding columns past each row's width) and the block table - every guard
must still hold its sentinel, and the results must still match the CPU
oracle.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpu_helpers import assert_parity, counters_tensor, run_oracle, to_dev  # noqa: E402
from synth import make_rows, make_workload, to_bf16_bits  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_indexer_fp32_gb300 as tk  # noqa: E402

GUARD_ROWS = 3
SENT = 0x5A5A5A5A  # as int32: neither an index, -1, nor the device-error mark
SENT_F = np.float32(-12345.5)


def guarded(B, k, dtype=torch.int32, fill=SENT):
    """A [B + 2 * GUARD_ROWS, k] buffer of sentinels and its inner [B, k] view."""
    buf = torch.full((B + 2 * GUARD_ROWS, k), fill, dtype=dtype, device="cuda:0")
    return buf, buf[GUARD_ROWS: GUARD_ROWS + B]


def assert_guards(buf, B, fill=SENT, what="out"):
    torch.cuda.synchronize()
    head, tail = buf[:GUARD_ROWS], buf[GUARD_ROWS + B:]
    assert torch.all(head == fill), f"{what}: a write before row 0"
    assert torch.all(tail == fill), f"{what}: a write after row B - 1"


def guarded_workspace(k, m):
    """Workspace of exactly topk_workspace_bytes(k, m) bytes (counters zero)
    followed by a 4 KiB sentinel tail; returns (buffer, inner view)."""
    nbytes = tk.workspace_bytes(k, m)
    buf = torch.full((nbytes + 4096,), 0xA5, dtype=torch.uint8, device="cuda:0")
    buf[:4096].zero_()
    return buf, buf[:nbytes]


def assert_ws_tail(buf, nbytes):
    torch.cuda.synchronize()
    assert torch.all(buf[nbytes:] == 0xA5), "workspace: a write past its end"
    assert not torch.any(buf[:4096]), "workspace: arrival counters not left at zero"


def _check(w, got_view, page_table=None, page_size=0):
    got = got_view.cpu().numpy()
    want = run_oracle(w.scores, w.lengths, w.k, page_table, page_size)
    assert_parity(w.scores, w.lengths, w.k, got, want, page_table=page_table)


# ------------------------------------------------------- streaming kernel

@pytest.mark.parametrize("opts", [
    dict(sample_mode=1, cluster_size=1),                          # unsampled
    dict(sample_mode=2, cluster_size=1),                          # sampled cutoff
    dict(sample_mode=1, cluster_size=1, stash_capacity=2048 + 2048),  # many compactions
    dict(sample_mode=2, cluster_size=8),                          # cluster of 8, DSMEM merge
    dict(sample_mode=1, cluster_size=2, stash_capacity=2048 + 2048),
], ids=["unsampled", "sampled", "compaction", "cluster8", "cluster2_compaction"])
def test_streaming_paths_write_only_their_rows(opts):
    # narrow-range rows (compaction and ties) and normal rows, ragged lengths
    w = make_rows(2, [0, 1, 2, 32, 33, 34, 62, 63])
    s, l = to_dev(w.scores), to_dev(w.lengths)
    buf, out = guarded(w.B, w.k)
    tk.topk_select_ex(s, l, w.k, out=out, **opts)
    assert_guards(buf, w.B)
    _check(w, out)


@pytest.mark.parametrize("k", [512, 2048])
def test_split_rows_write_only_their_rows_and_workspace(k):
    w = make_workload(3, B=6)
    s, l = to_dev(w.scores), to_dev(w.lengths)
    for m, sample_mode in ((6, 1), (6, 2), (3, 0)):
        wbuf, ws = guarded_workspace(k, m)
        buf, out = guarded(w.B, k)
        cnt = counters_tensor()
        tk.topk_select_ex(s, l, k, out=out, split_rows=m, workspace=ws, sample_mode=sample_mode,
                          counters=cnt)
        assert_guards(buf, w.B)
        assert_ws_tail(wbuf, ws.numel())
        assert int(cnt[tk.Counter.SPLIT_ROWS]) == m
        got = out.cpu().numpy()
        assert_parity(w.scores, w.lengths, k, got, run_oracle(w.scores, w.lengths, k))


def test_paged_split_rows_write_only_their_rows():
    w = make_workload(4, B=4)
    s, l, pt = to_dev(w.scores), to_dev(w.lengths), to_dev(w.page_table)
    wbuf, ws = guarded_workspace(w.k, 4)
    buf, out = guarded(w.B, w.k)
    tk.topk_select_ex(s, l, w.k, pt, w.page_size, out=out, split_rows=4, workspace=ws)
    assert_guards(buf, w.B)
    assert_ws_tail(wbuf, ws.numel())
    _check(w, out, w.page_table, w.page_size)


def test_default_calls_write_only_their_rows():
    """The binding's default calls (cached workspace, automatic policy) on
    the adversarial workload: rows at every 4-byte offset, lengths -1 ..
    width, the short and streaming paths both taken across the batch."""
    w = make_workload(5)
    s, l = to_dev(w.scores), to_dev(w.lengths)
    buf, out = guarded(w.B, w.k)
    tk.topk_ragged(s, l, w.k, out=out)
    assert_guards(buf, w.B)
    _check(w, out)


# ------------------------------------------------------- short-row kernel

@pytest.mark.parametrize("sample_mode", [0, 1])
@pytest.mark.parametrize("paged", [False, True])
def test_short_rows_write_only_their_rows(sample_mode, paged):
    rng = np.random.default_rng(7)
    B, stride, k, ps = 40, 16384 - 3, 1024, 64
    scores = rng.standard_normal((B, stride)).astype(np.float32)
    scores[5:10] = 1.0  # ties: the register path
    lengths = np.array([-1, 0, 1, k - 1, k, k + 1, stride, stride + 17] * 5, np.int32)
    pt = rng.permutation(B * 256).astype(np.int32).reshape(B, 256) if paged else None
    buf, out = guarded(B, k)
    tk.topk_select_ex(to_dev(scores), to_dev(lengths), k, None if pt is None else to_dev(pt),
                      ps if paged else 0, out=out, sample_mode=sample_mode, short_rows=1)
    assert_guards(buf, B)
    got = out.cpu().numpy()
    assert_parity(scores, lengths, k, got, run_oracle(scores, lengths, k, pt, ps if paged else 0),
                  page_table=pt)


def test_bf16_rows_write_only_their_rows():
    rng = np.random.default_rng(8)
    B, stride, k = 33, 8192, 512
    f = rng.standard_normal((B, stride)).astype(np.float32)
    bits = to_bf16_bits(f)
    lengths = np.array([0, 1, k, k + 1, stride, stride + 5, 3000] * 5, np.int32)[:B]
    s = torch.from_numpy(bits.view(np.int16)).to("cuda:0").view(torch.bfloat16)
    buf, out = guarded(B, k)
    tk.topk_select_bf16(s, to_dev(lengths), k, out=out)
    assert_guards(buf, B)
    conv = (bits.astype(np.uint32) << 16).view(np.float32)
    assert_parity(conv, lengths, k, out.cpu().numpy(), run_oracle(conv, lengths, k))


# ------------------------------------------------------- allocation-free call

def test_noalloc_writes_only_its_rows():
    lib = tk.load_library()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    w = make_workload(4, B=sms + 8)  # the last sms - 8 rows are split
    s, l = to_dev(w.scores), to_dev(w.lengths)
    buf, out = guarded(w.B, w.k)
    st = lib.topk_select_noalloc(s.data_ptr(), w.stride, l.data_ptr(), w.B, w.k, None, 0, 0,
                                 out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == tk.Status.OK
    assert_guards(buf, w.B)
    rows = np.array([0, w.B - 9, w.B - 8, w.B - 1])
    got = out.cpu().numpy()[rows]
    assert_parity(w.scores[rows], w.lengths[rows], w.k, got,
                  run_oracle(w.scores[rows], w.lengths[rows], w.k), rows=rows)


# ------------------------------------------------------- two-level helpers

@pytest.mark.parametrize("stride", [4096, 4093])
def test_amax8_writes_only_its_blocks(stride):
    """Keys go to slots [0, nb_b) of each row only: not to the padding columns
    past the row's width, not to slots at or past nb_b, not to skipped rows,
    not outside the rows."""
    rng = np.random.default_rng(stride)
    B, topk, pad = 20, 3, 5
    scores = rng.standard_normal((B, stride)).astype(np.float32)
    lengths = np.array([0, 1, 7, 8, 9, 24, 25, stride, stride + 3, -1]
                       + list(rng.integers(0, stride, B - 10)), dtype=np.int32)
    width = -(-stride // 8)
    buf = torch.full((B + 2 * GUARD_ROWS, width + pad), float(SENT_F), dtype=torch.float32,
                     device="cuda:0")
    out = buf[GUARD_ROWS: GUARD_ROWS + B, :width]
    tk.amax8_varlen(to_dev(scores), to_dev(lengths), topk, out=out)
    assert_guards(buf, B, fill=float(SENT_F), what="block keys")
    assert torch.all(buf[:, width:] == float(SENT_F)), "block keys: a write into the padding"
    want = oracle.amax8_varlen(scores, lengths, topk, np.full((B, width), SENT_F, np.float32))
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_block_table_writes_only_its_rows():
    rng = np.random.default_rng(3)
    B, stride, k, ps = 12, 65536, 100, 64
    lengths = np.array([0, 5, 8 * k, 8 * k + 1, stride, -1] + list(rng.integers(0, stride, B - 6)),
                       np.int32)
    blocks = np.full((B, k), -1, np.int32)
    for b in range(B):
        nb = -(-min(max(int(lengths[b]), 0), stride) // 8)
        if nb > k:
            blocks[b] = rng.choice(nb, k, replace=False)
    pt = rng.permutation(B * (stride // ps)).astype(np.int32).reshape(B, -1)
    bbuf, d_blocks = guarded(B, k)
    d_blocks.copy_(to_dev(blocks))
    pbuf, pages = guarded(B, k)
    tk.sort_candidate_blocks(d_blocks, to_dev(lengths), stride, to_dev(pt), ps, out_pages=pages)
    assert_guards(bbuf, B, what="block ids")
    assert_guards(pbuf, B, what="pool slots")
    want_ids, want_pages = oracle.sort_candidate_blocks(blocks, lengths, stride, pt, ps)
    assert np.array_equal(d_blocks.cpu().numpy(), want_ids)
    assert np.array_equal(pages.cpu().numpy(), want_pages)
