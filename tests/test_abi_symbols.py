"""The C-ABI library builds, loads and exports every function the header
declares; host-side argument checks return their codes without a GPU."""

import ctypes
import os
import re

import pytest

import sparse_attention_indexer_fp32_gb300 as tk
from sparse_attention_indexer_fp32_gb300 import build as cuda_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "topk_indexer.h")


@pytest.fixture(scope="module")
def lib():
    if cuda_build.is_stale():
        cuda_build.build()
    return tk.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(topk_[a-z_]+)\s*\(", text)))


def test_header_declares_the_two_calls():
    names = declared_functions()
    assert "topk_ragged" in names and "topk_paged" in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} missing from {cuda_build.LIB}"


def test_abi_version_and_status_strings(lib):
    assert lib.topk_abi_version() == 3
    for code in range(5):
        assert lib.topk_status_string(code)
    assert b"unknown" in lib.topk_status_string(99)


def test_argument_checks_need_no_gpu(lib):
    # All of these fail (or succeed, for B = 0) before any CUDA call.
    P = ctypes.c_void_p
    some = ctypes.c_void_p(0x1000)
    assert lib.topk_ragged(some, 64, some, 0, 512, some, None) == tk.Status.OK
    assert lib.topk_ragged(some, 64, some, 2, 0, some, None) == tk.Status.EUNSUPPORTED_K
    assert lib.topk_ragged(some, 64, some, 2, 2049, some, None) == tk.Status.EUNSUPPORTED_K
    assert lib.topk_ragged(some, 64, some, -1, 512, some, None) == tk.Status.EINVAL
    assert lib.topk_ragged(some, 0, some, 2, 512, some, None) == tk.Status.EINVAL
    assert lib.topk_ragged(P(None), 64, some, 2, 512, some, None) == tk.Status.EINVAL
    assert lib.topk_ragged(ctypes.c_void_p(0x1002), 64, some, 2, 512, some, None) == tk.Status.EINVAL
    assert lib.topk_paged(some, 64, some, 2, 512, P(None), 4, 16, some, None) == tk.Status.EINVAL
    assert lib.topk_paged(some, 64, some, 2, 512, some, 4, 0, some, None) == tk.Status.EINVAL
    assert lib.topk_paged(some, 64, some, 2, 512, some, 3, 16, some, None) == tk.Status.EINVAL


def test_workspace_checks_need_no_gpu(lib):
    some = ctypes.c_void_p(0x1000)
    ws, big = ctypes.c_void_p(0x100000), 1 << 24
    # misaligned or too small to hold the counters
    assert lib.topk_ragged_ws(some, 64, some, 2, 512, some, ctypes.c_void_p(0x100008), big,
                              None) == tk.Status.EINVAL
    assert lib.topk_ragged_ws(some, 64, some, 2, 512, some, ws, 12287, None) == tk.Status.EINVAL
    assert lib.topk_paged_ws(some, 64, some, 2, 512, some, 3, 16, some, ws, big,
                             None) == tk.Status.EINVAL
    assert lib.topk_ragged_ws(some, 64, some, 0, 512, some, ws, big, None) == tk.Status.OK
    assert lib.topk_ragged_ws(some, 64, some, 2, 4096, some, ws, big, None) == \
        tk.Status.EUNSUPPORTED_K


def test_bf16_checks_need_no_gpu(lib):
    some = ctypes.c_void_p(0x1000)
    # rows wider than 16384 scores, an odd (misaligned) score pointer, k out of range
    assert lib.topk_select_bf16(some, 16385, some, 2, 512, None, 0, 0, some, None) == tk.Status.EINVAL
    assert lib.topk_select_bf16(ctypes.c_void_p(0x1001), 64, some, 2, 8, None, 0, 0, some,
                                None) == tk.Status.EINVAL
    assert lib.topk_select_bf16(some, 64, some, 2, 2049, None, 0, 0, some, None) == \
        tk.Status.EUNSUPPORTED_K
    assert lib.topk_select_bf16(some, 64, some, 0, 8, None, 0, 0, some, None) == tk.Status.OK


def test_block_helper_checks_need_no_gpu(lib):
    some = ctypes.c_void_p(0x1000)
    # out rows narrower than ceil(stride / 8), negative topk, B = 0
    assert lib.topk_amax8_varlen(some, 64, some, 2, 0, some, 7, None) == tk.Status.EINVAL
    assert lib.topk_amax8_varlen(some, 64, some, 2, -1, some, 8, None) == tk.Status.EINVAL
    assert lib.topk_amax8_varlen(some, 64, some, 0, 0, some, 8, None) == tk.Status.OK
    # page size not a power of two >= 8, page table too narrow, rows too wide
    assert lib.topk_sort_candidate_blocks(some, 2, 8, some, 64, some, 8, 12, some, None) == tk.Status.EINVAL
    assert lib.topk_sort_candidate_blocks(some, 2, 8, some, 64, some, 8, 4, some, None) == tk.Status.EINVAL
    assert lib.topk_sort_candidate_blocks(some, 2, 8, some, 640, some, 9, 64, some, None) == tk.Status.EINVAL
    assert lib.topk_sort_candidate_blocks(some, 2, 8, some, (1 << 20) + 8, some, 1 << 17, 8, some,
                                          None) == tk.Status.EINVAL
    assert lib.topk_sort_candidate_blocks(some, 0, 8, some, 64, some, 8, 8, some, None) == tk.Status.OK


def test_workspace_bytes(lib):
    out = ctypes.c_size_t(0)
    # 12 KiB of counters, then per split row and half k keys and k indices
    assert lib.topk_workspace_bytes(512, 10, ctypes.byref(out)) == tk.Status.OK
    assert out.value == 12288 + 10 * 2 * 512 * 8
    assert lib.topk_workspace_bytes(2048, 1024, ctypes.byref(out)) == tk.Status.OK
    assert out.value == 12288 + 1024 * 2 * 2048 * 8
    assert lib.topk_workspace_bytes(0, 10, ctypes.byref(out)) == tk.Status.EUNSUPPORTED_K
    assert lib.topk_workspace_bytes(512, -1, ctypes.byref(out)) == tk.Status.EINVAL
    assert lib.topk_workspace_bytes(512, 1025, ctypes.byref(out)) == tk.Status.EINVAL
    assert lib.topk_workspace_bytes(512, 10, None) == tk.Status.EINVAL


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from sparse_attention_indexer_fp32_gb300 import _binding

    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _binding.load_library(str(tmp_path / "missing.so"))


def _opts(**kw):
    from sparse_attention_indexer_fp32_gb300._binding import _DebugOpts

    o = _DebugOpts()
    for name, value in kw.items():
        setattr(o, name, value)
    return o


def test_debug_option_checks_need_no_gpu(lib):
    """Every option outside its documented range is refused before anything
    is enqueued (rows of 65536 scores at k = 512: the streaming kernel's
    options apply)."""
    some = ctypes.c_void_p(0x1000)

    def call(B=2, stride=65536, k=512, **kw):
        return lib.topk_select_ex(some, stride, some, B, k, None, 0, 0, some,
                                  ctypes.byref(_opts(**kw)), None)

    bad = [
        dict(sample_mode=-1), dict(sample_mode=3),
        dict(stash_capacity=512 + 2047), dict(stash_capacity=512 + 2048 + 1),  # [k + 2048, default]
        dict(stash_capacity=512 + 4096 + 1),
        dict(cluster_size=3), dict(cluster_size=32), dict(cluster_size=-1),
        dict(counters=0x1002),  # misaligned
        dict(probe_stage=-1), dict(probe_stage=1, probe_wait_us=0),
        dict(probe_stage=1, probe_wait_us=5000001),
        dict(split_rows=-2), dict(split_rows=3),  # more than B
        dict(split_rows=1),  # no workspace
        dict(split_rows=1, workspace=0x100000, workspace_bytes=1 << 20, cluster_size=2),
        dict(split_rows=1, workspace=0x100008, workspace_bytes=1 << 20),  # misaligned
        dict(split_rows=1, workspace=0x100000, workspace_bytes=12287),  # below the counters
        dict(short_rows=2), dict(short_rows=-2),
    ]
    for kw in bad:
        assert call(**kw) == tk.Status.EINVAL, kw
    # the short-row kernel: rows of at most 16384 scores, no streaming-kernel option
    assert call(stride=16385, short_rows=1) == tk.Status.EINVAL
    assert call(stride=8192, short_rows=1, cluster_size=2) == tk.Status.EINVAL
    assert call(stride=8192, short_rows=1, stash_capacity=4000) == tk.Status.EINVAL
    # k is checked first; B = 0 is a no-op whatever the options
    assert call(k=2049, sample_mode=3) == tk.Status.EUNSUPPORTED_K
    assert call(B=0, cluster_size=3) == tk.Status.OK


def test_noalloc_checks_need_no_gpu(lib):
    """Every argument check of the allocation-free call runs before it looks
    at the device or sizes its scratch: an invalid call gets the same code as
    from topk_ragged / topk_paged, never TOPK_ESCRATCH."""
    some = ctypes.c_void_p(0x1000)
    assert lib.topk_select_noalloc(some, 64, some, 0, 512, None, 0, 0, some, None) == tk.Status.OK
    assert lib.topk_select_noalloc(some, 64, some, 2, 0, None, 0, 0, some, None) == \
        tk.Status.EUNSUPPORTED_K
    assert lib.topk_select_noalloc(some, 64, some, 2, 2049, None, 0, 0, some, None) == \
        tk.Status.EUNSUPPORTED_K
    assert lib.topk_select_noalloc(some, 64, some, -1, 512, None, 0, 0, some, None) == \
        tk.Status.EINVAL
    assert lib.topk_select_noalloc(some, 0, some, 2, 512, None, 0, 0, some, None) == \
        tk.Status.EINVAL
    # a call big enough to need more scratch than the array holds (153 rows
    # of 196608 at k = 2048), with one argument broken at a time
    big = dict(scores=some, stride=196608, lengths=some, B=153, k=2048, pt=None, pt_stride=0,
               page_size=0, out=some)

    def noalloc(**kw):
        a = dict(big, **kw)
        return lib.topk_select_noalloc(a["scores"], a["stride"], a["lengths"], a["B"], a["k"],
                                       a["pt"], a["pt_stride"], a["page_size"], a["out"], None)

    assert noalloc(scores=None) == tk.Status.EINVAL
    assert noalloc(lengths=None) == tk.Status.EINVAL
    assert noalloc(out=None) == tk.Status.EINVAL
    assert noalloc(scores=ctypes.c_void_p(0x1002)) == tk.Status.EINVAL  # misaligned
    assert noalloc(stride=2 ** 31) == tk.Status.EINVAL
    assert noalloc(pt=some, pt_stride=3071, page_size=64) == tk.Status.EINVAL  # table too narrow
    assert noalloc(pt=some, pt_stride=3072, page_size=0) == tk.Status.EINVAL
    assert noalloc(pt=ctypes.c_void_p(0x1001), pt_stride=3072, page_size=64) == tk.Status.EINVAL
    assert b"scratch" in lib.topk_status_string(tk.Status.ESCRATCH)


def test_cluster_residency_query_checks_need_no_gpu(lib):
    out = ctypes.c_int32(0)
    assert lib.topk_max_active_clusters(0, 0, 2, ctypes.byref(out)) == tk.Status.EUNSUPPORTED_K
    assert lib.topk_max_active_clusters(512, 0, 2, None) == tk.Status.EINVAL
    for g in (0, 1, 3, 32):
        assert lib.topk_max_active_clusters(512, 0, g, ctypes.byref(out)) == tk.Status.EINVAL
