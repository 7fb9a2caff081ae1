"""Seeded synthetic workloads for batched ragged FP32 top-k.

Every workload is drawn on the host with numpy's Philox counter-based bit
generator. Each row has its own stream, keyed by ``SeedSequence([seed, row])``,
so any subset of rows can be regenerated bit-identically without drawing the
others (the full-size parity tests use this to check sampled rows).

The first five shapes follow the decode-step workloads named for this path: the
sampled-filter PR of vLLM (PR 56346, "执行摘要": B=1024, 80-100 % ragged,
128K/k=2048 and 256K/k=512), the narrow-range and >65504 failure triggers of
the vLLM issue "persistent_topk silently drops top-k candidates ..." (原因分析),
and the boundary lengths and distributions of the same PR's graph test
(实现拆解 4). Shapes 6 and 7 are the prefill side of the same operation (many
rows of at most 8192 / 16384 scores, the short-row regime the sampled-filter
PR's dispatch sends to a separate path, 实现拆解 3), N(0,1) with lengths
uniform in [0.8 w, w].

Positions at and beyond a row's length are filled with ``PAD_VALUE`` (a quiet
NaN). The selection contract never looks there, so any read past a row's
length shows up as a wrong answer instead of passing silently.
"""

from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

PAD_VALUE = np.float32(np.nan)

#: Base of the per-config seeds: config ``c`` (1-based) uses ``0x5EED0000 + c``.
SEED_BASE = 0x5EED0000

#: Lengths used by config 5, cycled every 6 rows (``-1`` means "no token").
CFG5_LENGTHS = (-1, 0, 1, 1023, 1024, 32769, 65535, 65536, 98307)


@dataclasses.dataclass
class Workload:
    """One batch of synthetic input.

    ``scores`` is float32 ``[B, stride]`` row-major, ``lengths`` int32 ``[B]``,
    ``page_table`` int32 ``[B, pt_stride]`` or ``None`` for ragged output.
    ``rows`` lists which global row ids were drawn (all of them unless a subset
    was requested).
    """

    name: str
    config: int
    B: int
    stride: int
    k: int
    scores: np.ndarray
    lengths: np.ndarray
    page_table: Optional[np.ndarray] = None
    page_size: int = 0
    rows: Optional[np.ndarray] = None

    @property
    def paged(self) -> bool:
        return self.page_table is not None

    @property
    def pt_stride(self) -> int:
        return 0 if self.page_table is None else int(self.page_table.shape[1])


@dataclasses.dataclass(frozen=True)
class ConfigSpec:
    index: int
    name: str
    B: int
    stride: int
    k: int
    page_size: int = 0


CONFIGS = {
    1: ConfigSpec(1, "B4_w8192_k512_latency", 4, 8192, 512),
    2: ConfigSpec(2, "B64_w65536_k2048_samebin", 64, 65536, 2048),
    3: ConfigSpec(3, "B1024_w131072_k2048_ragged", 1024, 131072, 2048),
    4: ConfigSpec(4, "B1024_w262144_k512_paged64", 1024, 262144, 512, page_size=64),
    5: ConfigSpec(5, "B128_w98307_k1024_adversarial", 128, 98307, 1024),
    # Prefill-shaped batches: many short rows (one per query token of a chunk).
    6: ConfigSpec(6, "B16384_w8192_k512_prefill", 16384, 8192, 512),
    7: ConfigSpec(7, "B8192_w16384_k2048_prefill", 8192, 16384, 2048),
}


def config_seed(config: int) -> int:
    return SEED_BASE + int(config)


def _row_rng(seed: int, row: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, row])))


def _ragged_len(rng: np.random.Generator, width: int) -> int:
    """Integer length uniform in [ceil(0.8 * width), width], inclusive."""
    lo = -((-8 * width) // 10)
    return int(rng.integers(lo, width, endpoint=True))


def _normal(rng, n):
    return rng.standard_normal(n, dtype=np.float32)


def _row_cfg1(rng, row, stride):
    lengths = (0, 300, 512, 8192)
    return _normal(rng, stride), lengths[row % 4]


def _row_cfg2(rng, row, stride):
    n = _ragged_len(rng, stride)
    if row < 32:
        x = _normal(rng, stride)
    else:
        # Uniform over the float32 values in [1.0, 1.0 + 2^-10]: the mantissa
        # offsets 0..8192 above 1.0 are exactly those values, equally spaced.
        bits = np.uint32(0x3F800000) + rng.integers(0, 8192, size=stride, endpoint=True,
                                                    dtype=np.uint32)
        x = bits.view(np.float32)
    return x, n


def _row_cfg3(rng, row, stride):
    n = _ragged_len(rng, stride)
    offset = np.float32(rng.uniform(-4.0, 4.0))
    x = _normal(rng, stride) + offset
    return x, n


def _row_cfg4(rng, row, stride):
    n = _ragged_len(rng, stride)
    x = _normal(rng, stride)
    spike = rng.random(stride, dtype=np.float32) < np.float32(0.01)
    x[spike] += rng.uniform(3.0, 6.0, size=int(spike.sum())).astype(np.float32)
    return x, n


def _row_cfg5(rng, row, stride, k=1024):
    n = CFG5_LENGTHS[(row // 6) % len(CFG5_LENGTHS)]
    kind = row % 6
    if kind == 0:  # constant row, value drawn per row
        x = np.full(stride, _normal(rng, 1)[0], dtype=np.float32)
    elif kind == 1:  # ascending x[i] = i (exact: every i < 2^24)
        x = np.arange(stride, dtype=np.float32)
    elif kind == 2:  # exponent of 2^0, random low 10 mantissa bits: 1024 distinct values
        bits = np.uint32(0x3F800000) | rng.integers(0, 1024, size=stride, dtype=np.uint32)
        x = bits.view(np.float32)
    elif kind == 3:  # above the fp16 maximum
        x = rng.uniform(65504.0, 1.0e6, size=stride).astype(np.float32)
    elif kind == 4:  # -inf / +inf / -0 / +0, each with probability 1/8, over N(0,1)
        x = _normal(rng, stride)
        pick = rng.integers(0, 8, size=stride)
        x[pick == 0] = -np.inf
        x[pick == 1] = np.inf
        x[pick == 2] = np.float32(-0.0)
        x[pick == 3] = np.float32(0.0)
    else:  # k/4 peaks of +U(100,200) over U(0,1), on a 64-element grid
        x = rng.random(stride, dtype=np.float32)
        pos = np.arange(k // 4, dtype=np.int64) * 64
        pos = pos[pos < max(n, 0)]
        x[pos] += rng.uniform(100.0, 200.0, size=pos.size).astype(np.float32)
    return x, n


def _row_prefill(rng, row, stride):
    n = _ragged_len(rng, stride)
    return _normal(rng, stride), n


_ROW_FNS = {1: _row_cfg1, 2: _row_cfg2, 3: _row_cfg3, 4: _row_cfg4, 5: _row_cfg5,
            6: _row_prefill, 7: _row_prefill}


def _page_table_cfg4(seed: int, B: int, pt_stride: int) -> np.ndarray:
    """One global random permutation of [0, B*pt_stride) reshaped to [B, pt_stride]."""
    rng = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 0xFA6E])))
    return rng.permutation(B * pt_stride).astype(np.int32).reshape(B, pt_stride)


def make_rows(config: int, rows: Sequence[int], seed: Optional[int] = None) -> Workload:
    """Draw only the listed rows of a config (same bits as in the full batch)."""
    spec = CONFIGS[config]
    seed = config_seed(config) if seed is None else seed
    rows = np.asarray(list(rows), dtype=np.int64)
    scores = np.empty((rows.size, spec.stride), dtype=np.float32)
    lengths = np.empty(rows.size, dtype=np.int32)
    fn = _ROW_FNS[config]
    for j, r in enumerate(rows):
        x, n = fn(_row_rng(seed, int(r)), int(r), spec.stride)
        n_valid = min(max(int(n), 0), spec.stride)
        x = np.asarray(x, dtype=np.float32)
        x[n_valid:] = PAD_VALUE
        scores[j] = x
        lengths[j] = n
    page_table = None
    if spec.page_size:
        pt_stride = -(-spec.stride // spec.page_size)
        page_table = _page_table_cfg4(seed, spec.B, pt_stride)[rows]
    return Workload(spec.name, config, rows.size, spec.stride, spec.k, scores, lengths,
                    page_table, spec.page_size, rows)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), rounding to nearest even;
    inputs for the BF16 call (NaN is never produced by the generators)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_float(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> the float32 values they denote (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def make_workload(config: int, seed: Optional[int] = None, B: Optional[int] = None) -> Workload:
    """Draw a whole config (or its first ``B`` rows)."""
    spec = CONFIGS[config]
    n = spec.B if B is None else int(B)
    return make_rows(config, range(n), seed)
