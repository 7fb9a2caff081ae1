"""Parity of the short-row kernel (rows of at most 16384 scores, FP32 and
BF16) with the CPU oracle (needs an sm_103 GPU).

The short-row kernel serves the prefill-shaped batches (many rows of a few
thousand scores) and every BF16 call. Its fast path filters against a
sampled cutoff into a shared-memory stash; its exact path runs the radix
passes over the registers (underflow, overflow, or sampling off). Every case
compares with the oracle element by element: identical -1 pattern, identical
index set (both take the lowest indices among ties), identical value
multiset.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gpu_helpers import assert_parity, check_against_oracle, counters_tensor, run_oracle, to_dev  # noqa: E402
from synth import bf16_bits_to_float, make_rows, make_workload, to_bf16_bits  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_indexer_fp32_gb300 as tk  # noqa: E402


def _short_rows(width):
    """Rows of every adversarial kind of the 98307-wide workload, cut to
    `width`, with lengths around k and the width."""
    w5 = make_rows(5, list(range(0, 36)))
    rng = np.random.default_rng(width)
    B = w5.B + 6
    scores = np.full((B, width), np.nan, dtype=np.float32)
    lengths = np.zeros(B, dtype=np.int32)
    for i in range(w5.B):
        n = min(max(int(w5.lengths[i]), 0), width)
        scores[i, :n] = w5.scores[i, :n]
        lengths[i] = w5.lengths[i] if w5.lengths[i] < width else width + 5
    extra = [width, width - 1, 2049, 2048, 1025, 513]
    for j, n in enumerate(extra):
        scores[w5.B + j, :n] = rng.standard_normal(n).astype(np.float32)
        lengths[w5.B + j] = n
    return scores, lengths


@pytest.mark.parametrize("width", [8192, 16384, 9001, 4000])
@pytest.mark.parametrize("k", [1, 17, 512, 1024, 2048])
@pytest.mark.parametrize("sample_mode", [0, 1])
def test_short_rows_forced(width, k, sample_mode):
    """Widths for 32 and 64 scores per thread, an odd width (rows at every
    4-byte offset: scalar loads), and a width below the thread count x 32."""
    scores, lengths = _short_rows(width)
    cnt = counters_tensor()
    check_against_oracle(scores, lengths, k, short_rows=1, sample_mode=sample_mode, counters=cnt)
    assert int(cnt[tk.Counter.SHORT_ROWS]) == scores.shape[0]
    if sample_mode == 1:  # the stash path off: every row with n > k takes the register census
        n = np.clip(lengths.astype(np.int64), 0, width)
        assert int(cnt[tk.Counter.SHORT_EXACT]) == int(np.sum(n > k))


def test_short_rows_fall_back_to_the_exact_path():
    """The exact register path, forced (sample_mode 1) and taken by itself on
    constant rows (all scores tie: more candidates than the stash holds),
    comes out exact."""
    rng = np.random.default_rng(5)
    width = 16384
    scores = rng.standard_normal((6, width)).astype(np.float32)
    scores[3:] = np.float32(0.75)
    lengths = np.array([width, 12000, 9000, width, 10000, 4097], dtype=np.int32)
    for k in (512, 2048):
        cnt = counters_tensor()
        check_against_oracle(scores[:3], lengths[:3], k, short_rows=1, sample_mode=1, counters=cnt)
        assert int(cnt[tk.Counter.SHORT_EXACT]) == 3
        cnt = counters_tensor()
        check_against_oracle(scores[3:], lengths[3:], k, short_rows=1, counters=cnt)
        assert int(cnt[tk.Counter.SHORT_EXACT]) == 3


@pytest.mark.parametrize("config", [6, 7])
def test_prefill_workload_rows(config):
    """The first rows of the prefill-shaped workloads take the short-row
    kernel automatically; ragged and paged; and the streaming kernel forced."""
    w = make_workload(config, B=96)
    cnt = counters_tensor()
    check_against_oracle(w.scores, w.lengths, w.k, counters=cnt)
    assert int(cnt[tk.Counter.SHORT_ROWS]) == w.B
    cnt = counters_tensor()
    check_against_oracle(w.scores, w.lengths, w.k, short_rows=-1, counters=cnt)
    assert int(cnt[tk.Counter.SHORT_ROWS]) == 0
    cnt = counters_tensor()
    check_against_oracle(w.scores, w.lengths, w.k, counters=cnt)
    # nearly every row through the stash (a row whose k-th largest score's
    # coarse bin is selected whole, or holds too many scores, is served from
    # registers instead)
    assert int(cnt[tk.Counter.SHORT_EXACT]) <= w.B // 16
    rng = np.random.default_rng(config)
    pt = rng.permutation(w.B * 300).astype(np.int32).reshape(w.B, 300)
    check_against_oracle(w.scores, w.lengths, w.k, pt, 64)


def test_short_rows_special_values():
    rng = np.random.default_rng(9)
    width = 12000
    rows = [np.full(width, -np.inf), np.full(width, np.inf),
            np.where(rng.random(width) < 0.5, -0.0, 0.0),
            np.float32(1.4e-45) * rng.integers(-3, 4, width),
            rng.uniform(65504, 1e6, width),
            np.arange(width, dtype=np.float64)[::-1].copy()]
    x = rng.standard_normal(width)
    x[rng.integers(0, width, 50)] = np.inf
    x[rng.integers(0, width, 50)] = -np.inf
    rows.append(x)
    scores = np.stack([np.asarray(r, dtype=np.float32) for r in rows])
    lengths = np.array([width, 700, width, width, 11000, width, width], dtype=np.int32)
    for k in (512, 1024, 2048):
        for mode in (0, 1):
            check_against_oracle(scores, lengths, k, short_rows=1, sample_mode=mode)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_short_rows_unaligned(offset):
    rng = np.random.default_rng(offset)
    B, stride = 5, 8192
    flat = rng.standard_normal(B * stride + 4).astype(np.float32)
    host = flat[offset: offset + B * stride].reshape(B, stride)
    lengths = np.array([8192, 8000, 3000, 2049, 100], dtype=np.int32)
    s = to_dev(flat)[offset: offset + B * stride].view(B, stride)
    l = to_dev(lengths)
    for k in (512, 2048):
        out = tk.topk_ragged(s, l, k)
        torch.cuda.synchronize()
        assert_parity(host, lengths, k, out.cpu().numpy(), run_oracle(host, lengths, k))


# ------------------------------------------------------------------- BF16


def _bf16_case(width, B, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, width)).astype(np.float32)
    x[1] = rng.uniform(-3, 3, width).astype(np.float32) * 1e-3  # dense ties after rounding
    x[2, ::3] = np.inf
    x[3] = np.where(rng.random(width) < 0.5, -0.0, 0.0)
    bits = to_bf16_bits(x)
    return bits, bf16_bits_to_float(bits)


@pytest.mark.parametrize("width", [8192, 16384, 5001])
@pytest.mark.parametrize("k", [512, 1024, 2048])
def test_bf16_matches_the_oracle_on_the_converted_scores(width, k):
    B = 8
    bits, vals = _bf16_case(width, B, width + k)
    lengths = np.array([width, width - 3, width, 4000, 2048, 2049, 0, -1], dtype=np.int32)
    s = torch.from_numpy(bits.view(np.int16)).to("cuda:0").view(torch.bfloat16)
    l = to_dev(lengths)
    out = tk.topk_select_bf16(s, l, k)
    torch.cuda.synchronize()
    assert_parity(vals, lengths, k, out.cpu().numpy(), run_oracle(vals, lengths, k))
    rng = np.random.default_rng(k)
    pages = -(-width // 64)
    pt = rng.permutation(B * pages).astype(np.int32).reshape(B, pages)
    out = tk.topk_select_bf16(s, l, k, to_dev(pt), 64)
    torch.cuda.synchronize()
    assert_parity(vals, lengths, k, out.cpu().numpy(), run_oracle(vals, lengths, k, pt, 64),
                  page_table=pt)


def test_bf16_refuses_wide_rows():
    s = torch.zeros((2, 16385), dtype=torch.bfloat16, device="cuda:0")
    l = torch.full((2,), 100, dtype=torch.int32, device="cuda:0")
    with pytest.raises(tk.TopkError) as e:
        tk.topk_select_bf16(s, l, 8)
    assert e.value.status == tk.Status.EINVAL


def test_short_rows_deterministic_over_100_calls():
    w = make_workload(6, B=300)
    s, l = to_dev(w.scores), to_dev(w.lengths)
    first = tk.topk_ragged(s, l, w.k).clone()
    for _ in range(99):
        assert torch.equal(tk.topk_ragged(s, l, w.k), first)
    torch.cuda.synchronize()


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda:0").view(torch.bfloat16)


@pytest.mark.parametrize("width", [8192, 16384, 9001, 4000])
@pytest.mark.parametrize("k", [1, 17, 700, 2048])
def test_bf16_adversarial_rows(width, k):
    """The adversarial rows (constant rows, dense ties, +-inf, +-0, lengths
    around k and the width) rounded to BF16: both register layouts (32 and 64
    keys per thread), an odd width (rows that do not start on 16 bytes: scalar
    loads), the stash path and the register census, ragged and paged with an
    odd page size."""
    scores, lengths = _short_rows(width)
    bits = to_bf16_bits(scores)
    vals = bf16_bits_to_float(bits)
    s, l = _bf16_dev(bits), to_dev(lengths)
    out = tk.topk_select_bf16(s, l, k)
    torch.cuda.synchronize()
    assert_parity(vals, lengths, k, out.cpu().numpy(), run_oracle(vals, lengths, k))
    rng = np.random.default_rng(width * 7 + k)
    pages = -(-width // 7)
    pt = rng.permutation(scores.shape[0] * pages).astype(np.int32).reshape(scores.shape[0], pages)
    out = tk.topk_select_bf16(s, l, k, to_dev(pt), 7)
    torch.cuda.synchronize()
    assert_parity(vals, lengths, k, out.cpu().numpy(), run_oracle(vals, lengths, k, pt, 7), page_table=pt)


@pytest.mark.parametrize("width", [8192, 16384, 9001])
@pytest.mark.parametrize("k", [1, 512, 2048])
def test_bf16_rows_of_negative_infinity(width, k):
    """Rows whose k-th largest score is -inf, the lowest key any score has
    (slots past a row's end sit below it): ragged lengths that end inside a
    warp's range, mixed with a few finite scores and with -max, the lowest
    finite BF16 value."""
    rng = np.random.default_rng(width + k)
    lengths = np.array([width, width - 1, width - 77, 5000, 4097, 2049, k + 1, 3000], dtype=np.int32)
    scores = np.full((lengths.size, width), np.nan, dtype=np.float32)
    for i, n in enumerate(lengths):
        scores[i, :n] = -np.inf
    scores[1, rng.integers(0, lengths[1], 100)] = rng.standard_normal(100).astype(np.float32)
    scores[2, :lengths[2]:5] = np.float32(-3.3895314e38)  # -max in BF16
    scores[4, lengths[4] - 1] = 0.0
    scores[5, 0] = -np.inf
    scores[6, lengths[6] - 1] = np.float32(-3.3895314e38)
    bits = to_bf16_bits(scores)
    vals = bf16_bits_to_float(bits)
    s, l = _bf16_dev(bits), to_dev(lengths)
    out = tk.topk_select_bf16(s, l, k)
    torch.cuda.synchronize()
    assert_parity(vals, lengths, k, out.cpu().numpy(), run_oracle(vals, lengths, k))


@pytest.mark.parametrize("width,k", [(8192, 512), (16384, 2048)])
def test_bf16_and_fp32_kernels_agree(width, k):
    """The BF16 kernel's 16-bit keys are the high halves of the FP32 keys of
    the same values, with the same tie rule: on BF16-representable scores it
    returns exactly what the FP32 short-row kernel returns, slot by slot."""
    scores, lengths = _short_rows(width)
    bits = to_bf16_bits(scores)
    vals = np.ascontiguousarray(bf16_bits_to_float(bits))
    got16 = tk.topk_select_bf16(_bf16_dev(bits), to_dev(lengths), k)
    got32 = tk.topk_select_ex(to_dev(vals), to_dev(lengths), k, short_rows=1)
    torch.cuda.synchronize()
    assert torch.equal(got16, got32)


def test_bf16_deterministic_over_100_calls():
    w = make_workload(6, B=300)
    bits = to_bf16_bits(w.scores)
    s, l = _bf16_dev(bits), to_dev(w.lengths)
    first = tk.topk_select_bf16(s, l, w.k).clone()
    for _ in range(99):
        assert torch.equal(tk.topk_select_bf16(s, l, w.k), first)
    torch.cuda.synchronize()


def _group_rows(width, rng):
    """Rows whose cutoff falls inside the coarse bin of [1, 1.25) (or of
    (-1.25, -1]) with that bin's entries in group 0, in group 63, across all
    64 groups of 32 second-pass bins, or sharing their top 22 key bits (a
    third pass); the rest of each row far below."""
    def fill(m_lo, m_hi, count, sign=1.0):
        m = rng.integers(m_lo, m_hi, size=count, dtype=np.int64)
        x = (1.0 + m.astype(np.float64) * 2.0 ** -23).astype(np.float32)
        return sign * x
    rows = []
    for sign in (1.0, -1.0):
        for lo, hi in ((0, 1 << 15), (63 << 15, 64 << 15), (0, 1 << 21), (0, 1 << 10)):
            r = np.full(width, -8.0 if sign > 0 else -64.0, dtype=np.float32)
            pos = rng.choice(width, size=900, replace=False)
            r[pos] = fill(lo, hi, 900, sign)
            rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("width", [8192, 16384])
@pytest.mark.parametrize("k", [512, 700, 2048])
def test_short_rows_grouped_second_pass_extremes(width, k):
    """The second pass's group sums at their extremes (every entry of the
    cutoff bin in the first or the last group of 32 bins, or spread over all
    64) and a third pass over a shared 22-bit prefix, for positive and
    negative cutoffs, on the short-row kernel and through the default call."""
    rng = np.random.default_rng(width + k)
    scores = _group_rows(width, rng)
    lengths = np.full(scores.shape[0], width, dtype=np.int32)
    lengths[1::3] = width - 7
    cnt = counters_tensor()
    check_against_oracle(scores, lengths, k, short_rows=1, counters=cnt)
    assert int(cnt[tk.Counter.SHORT_ROWS]) == scores.shape[0]
    out = tk.topk_ragged(to_dev(scores), to_dev(lengths), k)
    torch.cuda.synchronize()
    assert_parity(scores, lengths, k, out.cpu().numpy(), run_oracle(scores, lengths, k))
