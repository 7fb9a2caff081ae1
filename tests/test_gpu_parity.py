"""Parity of the CUDA path with the CPU oracle (needs an sm_103 GPU).

Every case runs the C ABI through the Python binding and compares with the
oracle on the same seeded inputs: identical -1 pattern, identical index set
(both take the lowest indices among ties at the cutoff, so the sets match even
with ties), identical selected value multiset.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gpu_helpers import (assert_parity, check_against_oracle, counters_tensor, run_gpu,  # noqa: E402
                         run_oracle, to_dev)
from synth import make_rows, make_workload  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_indexer_fp32_gb300 as tk  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    tk.load_library()


# ---------------------------------------------------------------- workloads


@pytest.mark.parametrize("config", [1, 2, 5])
def test_workload_full(config):
    w = make_workload(config)
    check_against_oracle(w.scores, w.lengths, w.k)


@pytest.mark.parametrize("config", [3, 4])
def test_workload_leading_rows(config):
    w = make_workload(config, B=48)
    if w.paged:
        check_against_oracle(w.scores, w.lengths, w.k, w.page_table, w.page_size)
    check_against_oracle(w.scores, w.lengths, w.k)


# ------------------------------------------------------------ forced paths


def _mixed_rows():
    """Rows of every workload kind at moderate width, with lengths that hit
    the head/tail and stage boundaries."""
    w2 = make_rows(2, [0, 1, 33, 40, 63])
    w5 = make_rows(5, list(range(90, 108)))
    stride = 70001
    scores = np.full((w2.B + w5.B, stride), np.nan, dtype=np.float32)
    lengths = np.zeros(w2.B + w5.B, dtype=np.int32)
    for i in range(w2.B):
        n = min(int(w2.lengths[i]), stride)
        scores[i, :n] = w2.scores[i, :n]
        lengths[i] = n
    for i in range(w5.B):
        n = min(max(int(w5.lengths[i]), 0), stride)
        scores[w2.B + i, :n] = w5.scores[i, :n]
        lengths[w2.B + i] = w5.lengths[i] if w5.lengths[i] < stride else stride + 17
    return scores, lengths


@pytest.mark.parametrize("k", [512, 1024, 2048])
@pytest.mark.parametrize("sample_mode", [1, 2])
@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
def test_forced_paths(k, sample_mode, cluster):
    scores, lengths = _mixed_rows()
    check_against_oracle(scores, lengths, k, sample_mode=sample_mode, cluster_size=cluster)


@pytest.mark.parametrize("k", [512, 1024, 2048])
@pytest.mark.parametrize("cluster", [1, 4, 16])
def test_compaction_path(k, cluster):
    """Smallest candidate buffer (k + 2048 entries): the in-buffer compaction
    runs many times, and on the ascending rows the hits of one group exceed
    the room left even after compaction, so quarters of the group append in
    turn."""
    scores, lengths = _mixed_rows()
    cnt = counters_tensor()
    check_against_oracle(scores, lengths, k, sample_mode=1, cluster_size=cluster,
                         stash_capacity=k + 2048, counters=cnt)
    assert int(cnt[tk.Counter.COMPACTIONS]) > 0


@pytest.mark.parametrize("cluster", [1, 2, 8, 16])
def test_underflow_rescan_path(cluster):
    """A sampled cutoff set far too high keeps fewer than k candidates: every
    sampled row must be rescanned and still come out exact."""
    w = make_workload(3, B=8)
    cnt = counters_tensor()
    check_against_oracle(w.scores, w.lengths, w.k, sample_mode=2, sample_z=-1e4,
                         cluster_size=cluster, counters=cnt)
    assert int(cnt[tk.Counter.SAMPLED]) == 8
    assert int(cnt[tk.Counter.RESCAN]) == 8


def test_sampled_rows_are_counted():
    w = make_workload(4, B=16)
    cnt = counters_tensor()
    check_against_oracle(w.scores, w.lengths, w.k, w.page_table, w.page_size, counters=cnt)
    assert int(cnt[tk.Counter.ROWS]) == 16
    assert int(cnt[tk.Counter.SAMPLED]) == 16
    assert int(cnt[tk.Counter.DEVICE_ERRORS]) == 0


# ------------------------------------------------------------ split rows


def _workspace(k, rows):
    return torch.zeros(tk.workspace_bytes(k, rows), dtype=torch.uint8, device="cuda:0")


def _nontrivial(lengths, stride, k):
    n = np.clip(lengths.astype(np.int64), 0, stride)
    return int(np.sum(n > k))


@pytest.mark.parametrize("k", [512, 1024, 2048])
@pytest.mark.parametrize("sample_mode", [0, 1, 2])
def test_split_rows_forced(k, sample_mode):
    """Every row streamed by two independent CTAs that meet in the workspace:
    rows of every kind, lengths at the head/tail and stage boundaries, halves
    with no stage at all."""
    scores, lengths = _mixed_rows()
    B = scores.shape[0]
    ws = _workspace(k, B)
    cnt = counters_tensor()
    check_against_oracle(scores, lengths, k, sample_mode=sample_mode, split_rows=B,
                         workspace=ws, counters=cnt)
    assert int(cnt[tk.Counter.SPLIT_ROWS]) == _nontrivial(lengths, scores.shape[1], k)
    assert not torch.any(ws[:4096]), "arrival counters must be left at zero"


@pytest.mark.parametrize("k", [512, 1024, 2048])
@pytest.mark.parametrize("paged", [False, True])
def test_split_halves_that_hand_over_their_whole_stash(k, paged):
    """Rows just longer than k, split: a half that holds no more than k
    scores hands its whole stash over, right after its last stream group
    (with no scalar tail after it when the row's start and length line up),
    and the merge must see every entry of it. Rows at all four 4-byte
    offsets, repeated calls, each against the oracle."""
    rng = np.random.default_rng(k + paged)
    B, stride = 64, 140003  # odd: the rows start at every 4-byte offset
    lengths = (k + 1 + np.arange(B) % 4).astype(np.int32)
    scores = np.full((B, stride), np.nan, dtype=np.float32)
    for b in range(B):
        x = rng.standard_normal(lengths[b]).astype(np.float32)
        if b % 8 == 7:
            x = np.round(x * 2) / 2  # ties at the cut
        scores[b, :lengths[b]] = x
    pt, ps = None, 0
    if paged:
        ps = 64
        pages = -(-stride // ps)
        pt = rng.permutation(B * pages).astype(np.int32).reshape(B, pages)
    want = run_oracle(scores, lengths, k, pt, ps)
    ws = _workspace(k, B)
    for _ in range(10):
        got = run_gpu(scores, lengths, k, pt, ps, split_rows=B, workspace=ws)
        assert_parity(scores, lengths, k, got, want, page_table=pt)
    assert not torch.any(ws[:4096])


@pytest.mark.parametrize("k", [512, 2048])
def test_split_rows_compaction_and_rescan(k):
    """Halves that compact their own candidate buffer (smallest capacity), and
    halves whose sampled cutoff keeps too few (forced rescan)."""
    scores, lengths = _mixed_rows()
    B = scores.shape[0]
    ws = _workspace(k, B)
    cnt = counters_tensor()
    check_against_oracle(scores, lengths, k, sample_mode=1, stash_capacity=k + 2048,
                         split_rows=B, workspace=ws, counters=cnt)
    assert int(cnt[tk.Counter.COMPACTIONS]) > 0
    w = make_workload(3, B=6)
    cnt = counters_tensor()
    check_against_oracle(w.scores, w.lengths, w.k, sample_mode=2, sample_z=-1e4, split_rows=6,
                         workspace=_workspace(w.k, 6), counters=cnt)
    assert int(cnt[tk.Counter.RESCAN]) == 12  # both halves of every row


def test_split_rows_partial_and_paged():
    """Only the last m rows split (m < B); paged output through the merge."""
    w = make_workload(4, B=20)
    ws = _workspace(w.k, 20)
    for m in (1, 7, 20):
        cnt = counters_tensor()
        check_against_oracle(w.scores, w.lengths, w.k, w.page_table, w.page_size, split_rows=m,
                             workspace=ws, counters=cnt)
        assert int(cnt[tk.Counter.SPLIT_ROWS]) == m
    assert not torch.any(ws[:4096])


def test_split_rows_workspace_reused_and_too_small():
    """Calls in a row on one workspace (the counters return to zero after
    each); a workspace that holds fewer rows than forced is refused, and
    automatic splitting splits only what fits."""
    w = make_workload(5, B=30)
    ws = _workspace(w.k, 30)
    first = run_gpu(w.scores, w.lengths, w.k, split_rows=30, workspace=ws)
    for _ in range(3):
        assert np.array_equal(run_gpu(w.scores, w.lengths, w.k, split_rows=30, workspace=ws), first)
    assert_parity(w.scores, w.lengths, w.k, first, run_oracle(w.scores, w.lengths, w.k))
    small = _workspace(w.k, 4)
    with pytest.raises(tk.TopkError) as e:
        run_gpu(w.scores, w.lengths, w.k, split_rows=5, workspace=small)
    assert e.value.status == tk.Status.EINVAL
    # rows wide enough to be split automatically: only as many as the workspace holds
    w4 = make_workload(4, B=30)
    cnt = counters_tensor()
    got = run_gpu(w4.scores, w4.lengths, w4.k, cluster_size=1, workspace=_workspace(w4.k, 4),
                  counters=cnt)
    assert int(cnt[tk.Counter.SPLIT_ROWS]) == 4
    assert_parity(w4.scores, w4.lengths, w4.k, got, run_oracle(w4.scores, w4.lengths, w4.k))


def test_split_rows_wait_limit():
    """A half whose wait runs out hands over a failure; the merging half marks
    the row failed, and the workspace is left ready for the next call."""
    w = make_workload(3, B=4)
    ws = _workspace(w.k, 4)
    cnt = counters_tensor()
    out = run_gpu(w.scores, w.lengths, w.k, split_rows=4, workspace=ws, counters=cnt,
                  probe_stage=2, probe_wait_us=2000)
    assert np.all(out == tk.DEVICE_ERROR_INDEX)
    assert int(cnt[tk.Counter.DEVICE_ERRORS]) == 8
    assert not torch.any(ws[:4096])
    check_against_oracle(w.scores, w.lengths, w.k, split_rows=4, workspace=ws)


# ------------------------------------------------------------ edge cases


def test_capacity_boundaries_without_sampling():
    """Row lengths around the candidate-buffer capacity: the buffer fills
    exactly, one short of, and one past its end."""
    rng = np.random.default_rng(11)
    for k, cap in ((512, 2560), (1024, 5120), (2048, 5120)):
        ns = [cap - 1, cap, cap + 1, cap + 2047, cap + 2048, cap + 2049, 2 * cap + 5]
        stride = max(ns) + 3
        scores = rng.standard_normal((len(ns), stride)).astype(np.float32)
        lengths = np.array(ns, dtype=np.int32)
        check_against_oracle(scores, lengths, k, sample_mode=1, cluster_size=1)


def test_pages_capacity_boundaries():
    """One narrow band holding the top scores with the populations the pages
    report failures at (4096, 16384, 16385) and around them."""
    rng = np.random.default_rng(3)
    pops = [4095, 4096, 4097, 16384, 16385]
    stride = 16385 + 7000
    scores = np.full((len(pops), stride), np.nan, dtype=np.float32)
    lengths = np.zeros(len(pops), dtype=np.int32)
    for i, pop in enumerate(pops):
        n = pop + 5000
        x = rng.standard_normal(n).astype(np.float32) - 10.0
        band = (np.uint32(0x3F800000) + rng.integers(0, 8193, pop).astype(np.uint32)).view(np.float32)
        x[rng.permutation(n)[:pop]] = band
        scores[i, :n] = x
        lengths[i] = n
    for k in (512, 2048):
        check_against_oracle(scores, lengths, k)
        check_against_oracle(scores, lengths, k, sample_mode=1)


@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_unaligned_rows(offset):
    """Row starts at every 4-byte offset from a 16-byte boundary; odd stride."""
    rng = np.random.default_rng(offset)
    B, stride = 6, 20011
    flat = rng.standard_normal(B * stride + 4).astype(np.float32)
    lengths = np.array([stride, 20000, 9999, 2049, 2050, 3], dtype=np.int32)
    buf = to_dev(flat)
    s = buf[offset: offset + B * stride].view(B, stride)
    l = to_dev(lengths)
    host = flat[offset: offset + B * stride].reshape(B, stride)
    for k in (1, 17, 512, 2048):
        out = tk.topk_ragged(s, l, k)
        torch.cuda.synchronize()
        assert_parity(host, lengths, k, out.cpu().numpy(), run_oracle(host, lengths, k))


@pytest.mark.parametrize("width,B", [(2000003, 3), (1 << 24, 1)])
@pytest.mark.parametrize("k", [512, 2048])
def test_very_wide_rows(width, B, k):
    """Rows far wider than the workloads' (2,000,003 scores, odd; 2^24
    scores): the index arithmetic of every stage, sample and page-table
    lookup, on the automatic path (clusters of 16 for so few rows), ragged
    and paged."""
    rng = np.random.default_rng(width + k)
    scores = rng.standard_normal((B, width)).astype(np.float32)
    scores[:, width // 3] = np.inf  # one clear maximum far into the row
    lengths = np.array([width, width - 5, width // 2][:B], dtype=np.int32)
    check_against_oracle(scores, lengths, k)
    ps = 64
    pages = -(-width // ps)
    pt = rng.permutation(B * pages).astype(np.int32).reshape(B, pages)
    check_against_oracle(scores, lengths, k, pt, ps)


@pytest.mark.parametrize("B,width,k", [(300000, 5, 3), (70000, 40, 17), (5000, 20000, 512)])
def test_large_batches(B, width, k):
    """Many rows: a grid of hundreds of thousands of CTAs on the short-row
    kernel, and thousands of rows just past its width on the streaming
    kernel (several waves, the split tail), ragged."""
    rng = np.random.default_rng(B + width)
    scores = rng.standard_normal((B, width)).astype(np.float32)
    lengths = rng.integers(-1, width + 2, B).astype(np.int32)
    check_against_oracle(scores, lengths, k)


@pytest.mark.parametrize("k", [1, 2, 3, 100, 511, 513, 2047])
def test_other_k_values(k):
    w = make_rows(5, list(range(0, 128, 5)))
    check_against_oracle(w.scores, w.lengths, k)


def test_special_values():
    rng = np.random.default_rng(8)
    stride = 40000
    rows = []
    rows.append(np.full(stride, -np.inf))                      # all -inf
    rows.append(np.full(stride, np.inf))                       # all +inf
    x = np.zeros(stride); x[::2] = -0.0; rows.append(x)        # signed zeros
    x = np.where(rng.random(stride) < 0.5, -0.0, 0.0); rows.append(x)
    rows.append(np.full(stride, 7.25))                         # constant
    x = np.arange(stride, dtype=np.float64)[::-1].copy(); rows.append(x)  # descending
    x = rng.standard_normal(stride); x[12345] = np.inf; rows.append(x)
    x = rng.uniform(65504, 1e6, stride); rows.append(x)        # above the fp16 range
    x = np.full(stride, np.float32(3.4028235e38)); x[::3] = -np.float32(3.4028235e38); rows.append(x)
    x = (np.float32(1.4e-45) * rng.integers(-3, 4, stride)); rows.append(x)  # subnormals
    scores = np.stack([np.asarray(r, dtype=np.float32) for r in rows])
    lengths = np.array([stride, 300, stride, 30000, stride, stride, stride, 31111, stride, stride],
                       dtype=np.int32)
    for k in (512, 1024, 2048):
        for mode in (0, 1, 2):
            check_against_oracle(scores, lengths, k, sample_mode=mode)


def test_lengths_convention():
    rng = np.random.default_rng(1)
    stride = 5000
    scores = rng.standard_normal((8, stride)).astype(np.float32)
    lengths = np.array([-5, -1, 0, 1, 511, 512, 513, stride + 17], dtype=np.int32)
    check_against_oracle(scores, lengths, 512)


def test_empty_batch_is_a_noop():
    s = torch.zeros((0, 128), dtype=torch.float32, device="cuda:0")
    l = torch.zeros((0,), dtype=torch.int32, device="cuda:0")
    out = tk.topk_ragged(s, l, 512)
    assert out.shape == (0, 512)


def test_paged_full_mapping():
    w = make_workload(4, B=24)
    got = run_gpu(w.scores, w.lengths, w.k, w.page_table, w.page_size)
    want = run_oracle(w.scores, w.lengths, w.k, w.page_table, w.page_size)
    assert_parity(w.scores, w.lengths, w.k, got, want, page_table=w.page_table)
    # odd page size and short rows
    rng = np.random.default_rng(2)
    B, stride, ps = 5, 9000, 7
    scores = rng.standard_normal((B, stride)).astype(np.float32)
    lengths = np.array([9000, 700, 513, 512, 0], dtype=np.int32)
    pt = rng.permutation(B * 1300).astype(np.int32).reshape(B, 1300)
    check_against_oracle(scores, lengths, 512, pt, ps)


@pytest.mark.parametrize("cluster", [2, 4, 8, 16])
def test_paged_output_from_clusters(cluster):
    """Paged output written by every CTA of a cluster (each maps its own
    share of the selection through the table), with an odd page size too."""
    w = make_workload(4, B=6)
    check_against_oracle(w.scores, w.lengths, w.k, w.page_table, w.page_size, cluster_size=cluster)
    rng = np.random.default_rng(cluster)
    pt = rng.permutation(6 * 40000).astype(np.int32).reshape(6, 40000)
    check_against_oracle(w.scores, w.lengths, 1024, pt, 7, cluster_size=cluster, sample_mode=2)


def test_status_codes():
    s = torch.zeros((2, 64), dtype=torch.float32, device="cuda:0")
    l = torch.full((2,), 64, dtype=torch.int32, device="cuda:0")
    for bad_k in (0, -1, 2049):
        with pytest.raises(tk.TopkError) as e:
            tk.topk_ragged(s, l, bad_k)
        assert e.value.status == tk.Status.EUNSUPPORTED_K
    pt = torch.zeros((2, 1), dtype=torch.int32, device="cuda:0")
    with pytest.raises(tk.TopkError) as e:  # page table too narrow for the width
        tk.topk_paged(s, l, 8, pt, 16)
    assert e.value.status == tk.Status.EINVAL
    with pytest.raises(tk.TopkError) as e:
        tk.topk_select_ex(s, l, 8, stash_capacity=100)
    assert e.value.status == tk.Status.EINVAL


# ------------------------------------------------------------ determinism


@pytest.mark.parametrize("config", [2, 5])
def test_deterministic_over_100_calls(config):
    w = make_workload(config)
    s, l = to_dev(w.scores), to_dev(w.lengths)
    first = tk.topk_ragged(s, l, w.k).clone()
    for _ in range(99):
        again = tk.topk_ragged(s, l, w.k)
        assert torch.equal(first, again)
    torch.cuda.synchronize()


@pytest.mark.parametrize("k", [512, 1024, 2048])
@pytest.mark.parametrize("cluster", [1, 2])
def test_wait_limit_reports_device_error(cluster, k):
    """A wait that runs out (on a barrier nothing completes) is reported: the
    rows carry TOPK_DEVICE_ERROR_INDEX in every slot, the error is counted,
    the call returns, and the context keeps working. The output starts out
    holding a third value, so a slot written by a selection after (or
    instead of) the failure mark would show."""
    w = make_workload(3, B=4)
    s, l = to_dev(w.scores), to_dev(w.lengths)
    cnt = counters_tensor()
    out = torch.full((w.B, k), 0x1234567, dtype=torch.int32, device="cuda:0")
    tk.topk_select_ex(s, l, k, out=out, cluster_size=cluster, counters=cnt,
                      probe_stage=2, probe_wait_us=2000)
    torch.cuda.synchronize()
    assert torch.all(out == tk.DEVICE_ERROR_INDEX), "a slot of a failed row holds something else"
    assert int(cnt[tk.Counter.DEVICE_ERRORS]) == 4 * cluster
    assert int(cnt[tk.Counter.SPLIT_ROWS]) == 0
    check_against_oracle(w.scores, w.lengths, k, cluster_size=cluster)


def test_capture_before_the_streams_first_call_runs_unsplit():
    """A stream that captures a graph before any call on it has no workspace
    yet; zeroing one inside the capture would happen only at replay, so the
    binding's default call runs unsplit there. The replays match the oracle,
    and a later eager call on the same stream creates the workspace, splits
    the last rows, and gives the same indices."""
    from sparse_attention_indexer_fp32_gb300 import _binding

    w = make_workload(4, B=160)  # 262144-wide rows: the last 144 are split when a workspace is given
    s, l = to_dev(w.scores), to_dev(w.lengths)
    tk.topk_ragged(s, l, w.k)  # the library's one-time set-up, on the current stream
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    key = (0, int(stream.cuda_stream))
    _binding._workspaces.pop(key, None)  # streams come from a pool: forget an earlier test's
    out = torch.empty((w.B, w.k), dtype=torch.int32, device="cuda:0")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        tk.topk_ragged(s, l, w.k, out=out)
    assert key not in _binding._workspaces
    graph.replay()
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    rows = np.arange(w.B - 24, w.B)
    assert_parity(w.scores[rows], w.lengths[rows], w.k, got[rows],
                  run_oracle(w.scores[rows], w.lengths[rows], w.k), rows=rows)
    with torch.cuda.stream(stream):
        eager = tk.topk_ragged(s, l, w.k)
    stream.synchronize()
    assert key in _binding._workspaces
    assert np.array_equal(eager.cpu().numpy(), got)


@pytest.mark.parametrize("paged,split", [(False, False), (True, False), (False, True)])
def test_cuda_graph_replay_with_mutated_lengths(paged, split):
    """One captured call replayed with the row lengths (and once the scores)
    rewritten in place between replays, as a decode step would: every replay
    matches the oracle on the inputs current at that replay. The split case
    streams every row with two CTAs that meet in a workspace."""
    rng = np.random.default_rng(21)
    B, stride, k, ps = 6, 98307 + 3, 1024, 64
    scores = rng.standard_normal((B, stride)).astype(np.float32)
    pt = rng.permutation(B * 1600).astype(np.int32).reshape(B, 1600) if paged else None
    s, l = to_dev(scores), to_dev(np.full(B, stride, np.int32))
    dpt = to_dev(pt) if paged else None
    out = torch.empty((B, k), dtype=torch.int32, device="cuda:0")
    ws = _workspace(k, B) if split else None
    torch.cuda.synchronize()  # the workspace is zeroed on another stream

    def call():
        if split:
            tk.topk_select_ex(s, l, k, out=out, split_rows=B, workspace=ws)
        elif paged:
            tk.topk_paged(s, l, k, dpt, ps, out=out)
        else:
            tk.topk_ragged(s, l, k, out=out)

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):  # warm the library (attributes, device query) first
        call()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    boundary = [-1, 0, 1, k - 1, k, 32769, 65535, 98307, stride, stride + 17]
    for rep in range(4):
        lengths = np.array([boundary[(rep * B + i) % len(boundary)] for i in range(B)], np.int32)
        if rep == 2:
            scores = -scores  # flip the scores once
            s.copy_(to_dev(scores))
        l.copy_(to_dev(lengths))
        graph.replay()
        torch.cuda.synchronize()
        want = run_oracle(scores, lengths, k, pt, ps if paged else 0)
        assert_parity(scores, lengths, k, out.cpu().numpy(), want, page_table=pt)



def test_cluster_residency_answers():
    """The CUDA driver's cluster residency answers that the automatic policy uses:
    clusters of 2, 4 and 8 fit; larger clusters never fit more at once."""
    for k in (512, 2048):
        for paged in (False, True):
            n = [tk.max_active_clusters(k, paged, g) for g in (2, 4, 8, 16)]
            assert n[0] > 0 and n[1] > 0 and n[2] > 0, n
            assert n[0] >= n[1] >= n[2] >= n[3] >= 0, n


@pytest.mark.parametrize("B,stride,clustered", [(1, 262144, True), (4, 131072, True),
                                                (2, 65536, True), (8, 262144, True),
                                                (5, 131072, True), (9, 196608, True),
                                                (16, 131072, True), (17, 131072, True),
                                                (32, 131072, True), (33, 131072, True),
                                                (64, 131072, True), (4, 32768, False),
                                                (32, 65536, False), (64, 65536, False),
                                                (200, 262144, False)])
def test_automatic_cluster_policy(B, stride, clustered):
    """Small batches of long rows run on clusters, short rows and larger
    batches on one CTA per row (the gates the dispatch sweep measured); the
    result is the oracle's either way."""
    rng = np.random.default_rng(B + stride)
    scores = rng.standard_normal((B, stride)).astype(np.float32)
    lengths = rng.integers(stride * 4 // 5, stride + 1, B).astype(np.int32)
    cnt = counters_tensor()
    check_against_oracle(scores, lengths, 512, counters=cnt)
    assert int(cnt[tk.Counter.CLUSTER_ROWS]) == (B if clustered else 0)


def _sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("B,stride,k,expect", [
    (64, 131072, 1024, "all"),       # a few dozen rows: every row split, not clustered
    (33, 131072, 1024, "clusters"),  # up to 40 rows: clusters of 4
    (128, 131072, 512, "all"),       # up to half the slots: every row
    (128, 131072, 2048, "none"),     # 131072 scores, k = 2048, beyond 74 rows: none
    (192, 262144, 512, "fill"),      # beyond half the slots: the rows that fill the idle ones
    (256, 262144, 512, "none"),      # beyond 200 rows one CTA per row keeps HBM busy
])
def test_automatic_split_policy(B, stride, k, expect):
    """With a workspace the automatic policy splits the rows the dispatch
    sweep found faster split, gives small batches clusters instead, and
    matches the unsplit call and the oracle either way."""
    slots = 2 * _sm_count()
    want_split = {"all": B, "fill": slots - B, "none": 0, "clusters": 0}[expect]
    rng = np.random.default_rng(B * 7 + k)
    scores = rng.standard_normal((B, stride)).astype(np.float32)
    lengths = rng.integers(stride * 4 // 5, stride + 1, B).astype(np.int32)
    s, l = to_dev(scores), to_dev(lengths)
    ws = torch.zeros(tk.workspace_bytes(k, B), dtype=torch.uint8, device="cuda:0")
    cnt = counters_tensor()
    got = tk.topk_select_ex(s, l, k, workspace=ws, counters=cnt)
    want = tk.topk_select_ex(s, l, k, split_rows=-1)
    torch.cuda.synchronize()
    assert int(cnt[tk.Counter.SPLIT_ROWS]) == want_split
    assert int(cnt[tk.Counter.CLUSTER_ROWS]) == (B if expect == "clusters" else 0)
    assert torch.equal(got, want)
    rows = np.array([0, B // 2, B - 1])
    assert_parity(scores[rows], lengths[rows], k, got.cpu().numpy()[rows],
                  run_oracle(scores[rows], lengths[rows], k), rows=rows)
