"""ctypes binding of ``libtopk_indexer.so`` (argument marshalling only).

Every step of the selection runs in the library's CUDA kernels; this module
only checks tensor dtypes/devices/shapes, takes their device pointers and the
current CUDA stream, and turns status codes into exceptions. There is no CPU
fallback: without the built library every call raises.
"""

from __future__ import annotations

import ctypes
import enum
import os
import threading
from typing import Optional

import torch

from . import build as _build

LIB_PATH = _build.LIB

TOPK_MAX_K = 2048
DEVICE_ERROR_INDEX = -(2 ** 31)


class Status(enum.IntEnum):
    OK = 0
    EINVAL = 1
    EUNSUPPORTED_K = 2
    ECUDA = 3
    EDEVICE = 4
    ESCRATCH = 5


class Counter(enum.IntEnum):
    ROWS = 0
    TRIVIAL = 1
    SAMPLED = 2
    RESCAN = 3
    COMPACTIONS = 4
    DEVICE_ERRORS = 5
    CLUSTER_ROWS = 6
    SPLIT_ROWS = 7
    SHORT_ROWS = 8
    SHORT_EXACT = 9


NUM_COUNTERS = 16


class TopkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class _DebugOpts(ctypes.Structure):
    _fields_ = [("sample_mode", ctypes.c_int32), ("cluster_size", ctypes.c_int32),
                ("stash_capacity", ctypes.c_int32), ("sample_z", ctypes.c_float),
                ("counters", ctypes.c_void_p), ("probe_stage", ctypes.c_int32),
                ("probe_wait_us", ctypes.c_uint32), ("split_rows", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("short_rows", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads the CUDA library (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library not built: {path} is missing. Build it with "
                "`python -m sparse_attention_indexer_fp32_gb300.build` "
                "(nvcc, sm_103a).")
        lib = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        lib.topk_ragged.argtypes = [vp, i64, vp, i32, i32, vp, vp]
        lib.topk_ragged.restype = ctypes.c_int
        lib.topk_paged.argtypes = [vp, i64, vp, i32, i32, vp, i64, i32, vp, vp]
        lib.topk_paged.restype = ctypes.c_int
        lib.topk_select_ex.argtypes = [vp, i64, vp, i32, i32, vp, i64, i32, vp,
                                       ctypes.POINTER(_DebugOpts), vp]
        lib.topk_select_ex.restype = ctypes.c_int
        sz = ctypes.c_size_t
        lib.topk_ragged_ws.argtypes = [vp, i64, vp, i32, i32, vp, vp, sz, vp]
        lib.topk_ragged_ws.restype = ctypes.c_int
        lib.topk_paged_ws.argtypes = [vp, i64, vp, i32, i32, vp, i64, i32, vp, vp, sz, vp]
        lib.topk_paged_ws.restype = ctypes.c_int
        lib.topk_workspace_bytes.argtypes = [i32, i32, ctypes.POINTER(sz)]
        lib.topk_workspace_bytes.restype = ctypes.c_int
        lib.topk_select_noalloc.argtypes = [vp, i64, vp, i32, i32, vp, i64, i32, vp, vp]
        lib.topk_select_noalloc.restype = ctypes.c_int
        lib.topk_select_bf16.argtypes = [vp, i64, vp, i32, i32, vp, i64, i32, vp, vp]
        lib.topk_select_bf16.restype = ctypes.c_int
        lib.topk_amax8_varlen.argtypes = [vp, i64, vp, i32, i32, vp, i64, vp]
        lib.topk_amax8_varlen.restype = ctypes.c_int
        lib.topk_sort_candidate_blocks.argtypes = [vp, i32, i32, vp, i64, vp, i64, i32, vp, vp]
        lib.topk_sort_candidate_blocks.restype = ctypes.c_int
        lib.topk_max_active_clusters.argtypes = [i32, i32, i32, ctypes.POINTER(i32)]
        lib.topk_max_active_clusters.restype = ctypes.c_int
        lib.topk_status_string.argtypes = [ctypes.c_int]
        lib.topk_status_string.restype = ctypes.c_char_p
        lib.topk_abi_version.restype = ctypes.c_int32
        _lib = lib
        return lib


def _check(status: int) -> None:
    if status != Status.OK:
        msg = load_library().topk_status_string(status).decode()
        raise TopkError(status, f"top-k call failed: {msg}")


def _stream(device, stream):
    """The torch stream a call is enqueued on (default: the current one);
    ``device`` a torch.device or a device index."""
    return torch.cuda.current_stream(device) if stream is None else stream


def _stream_handle(device, stream) -> int:
    return int(_stream(device, stream).cuda_stream)


def _on_device(index: int, fn):
    """Runs ``fn`` with CUDA device ``index`` current (the library launches
    on the current device), switching only when another one is current."""
    if torch.cuda.current_device() == index:
        return fn()
    with torch.cuda.device(index):
        return fn()


def workspace_bytes(k: int = TOPK_MAX_K, max_split_rows: int = 0) -> int:
    """Workspace size for calls with this k that split up to
    ``max_split_rows`` rows (0: the most the library splits on the current
    device)."""
    out = ctypes.c_size_t(0)
    _check(load_library().topk_workspace_bytes(int(k), int(max_split_rows), ctypes.byref(out)))
    return int(out.value)


# One zero-initialised workspace per (device, stream): calls on one stream run
# one after another, so they can share it; the library leaves its counters
# zero after every call.
_workspaces = {}
_ws_lock = threading.Lock()


def _workspace(device, stream) -> Optional[torch.Tensor]:
    """The cached workspace of this device and stream, created (and zeroed on
    that stream, so that the first call is ordered after the zeroing) on first
    use. None while the stream captures a CUDA graph and has no workspace yet:
    zeroing it inside the capture would run only at replay, so the call takes
    the unsplit path instead (same results). ``device`` a torch.device or a
    device index; ``stream`` a torch stream or None (the current one)."""
    index = device if isinstance(device, int) else device.index
    stream = _stream(index, stream)
    key = (index, int(stream.cuda_stream))
    ws = _workspaces.get(key)  # entries are only ever added
    if ws is not None:
        return ws
    with _ws_lock:
        ws = _workspaces.get(key)
        if ws is None:
            with torch.cuda.stream(stream):
                if torch.cuda.is_current_stream_capturing():
                    return None
                ws = torch.zeros(workspace_bytes(TOPK_MAX_K), dtype=torch.uint8, device=index)
            _workspaces[key] = ws
    return ws


def _prepare(scores: torch.Tensor, lengths: torch.Tensor, k: int, out: Optional[torch.Tensor]):
    if not isinstance(scores, torch.Tensor) or scores.dim() != 2:
        raise ValueError("scores must be a 2-D tensor [B, stride]")
    if not scores.is_cuda or scores.dtype != torch.float32 or not scores.is_contiguous():
        raise ValueError("scores must be a contiguous float32 CUDA tensor")
    B, stride = scores.shape
    if lengths.dtype != torch.int32 or lengths.device != scores.device or lengths.numel() != B \
            or not lengths.is_contiguous():
        raise ValueError("lengths must be a contiguous int32 tensor [B] on the scores' device")
    if out is None:
        # an unsupported k is reported by the library itself (TOPK_EUNSUPPORTED_K)
        out = torch.empty((B, max(int(k), 1)), dtype=torch.int32, device=scores.device)
    elif (out.dtype != torch.int32 or out.device != scores.device
          or tuple(out.shape) != (B, max(int(k), 1)) or not out.is_contiguous()):
        raise ValueError("out must be a contiguous int32 tensor [B, k] on the scores' device")
    return B, stride, out


def topk_ragged(scores: torch.Tensor, lengths: torch.Tensor, k: int,
                out: Optional[torch.Tensor] = None, stream=None,
                split: bool = True) -> torch.Tensor:
    """Indices of the ``min(k, lengths[b])`` largest scores of every row, ``-1`` after them.

    ``scores`` float32 ``[B, stride]`` (CUDA, contiguous), ``lengths`` int32
    ``[B]``. Returns ``out`` (int32 ``[B, k]``), enqueued on ``stream`` (default:
    the current stream). With ``split`` (the default) the call goes through
    ``topk_ragged_ws`` with a workspace cached per device and stream, so that
    the last rows of a large batch may be split over two CTAs; the result is
    the same either way. A stream's workspace is created by its first call
    outside a CUDA graph capture: a call captured before that runs unsplit."""
    lib = load_library()
    B, stride, out = _prepare(scores, lengths, k, out)
    index = scores.get_device()
    st = _stream(index, stream)
    sh = int(st.cuda_stream)

    def call():
        ws = _workspace(index, st) if split else None
        if ws is not None:
            return lib.topk_ragged_ws(scores.data_ptr(), stride, lengths.data_ptr(), B, k,
                                      out.data_ptr(), ws.data_ptr(), ws.numel(), sh)
        return lib.topk_ragged(scores.data_ptr(), stride, lengths.data_ptr(), B, k, out.data_ptr(), sh)

    _check(_on_device(index, call))
    return out


def topk_paged(scores: torch.Tensor, lengths: torch.Tensor, k: int, page_table: torch.Tensor,
               page_size: int, out: Optional[torch.Tensor] = None, stream=None,
               split: bool = True) -> torch.Tensor:
    """As :func:`topk_ragged`, each selected index ``i`` of row ``b`` written as
    ``page_table[b, i // page_size] * page_size + i % page_size``."""
    lib = load_library()
    B, stride, out = _prepare(scores, lengths, k, out)
    if (page_table.dtype != torch.int32 or page_table.device != scores.device
            or page_table.dim() != 2 or page_table.shape[0] != B or not page_table.is_contiguous()):
        raise ValueError("page_table must be a contiguous int32 tensor [B, pages] on the scores' device")
    index = scores.get_device()
    st = _stream(index, stream)
    sh = int(st.cuda_stream)

    def call():
        ws = _workspace(index, st) if split else None
        if ws is not None:
            return lib.topk_paged_ws(scores.data_ptr(), stride, lengths.data_ptr(), B, k,
                                     page_table.data_ptr(), page_table.shape[1], page_size,
                                     out.data_ptr(), ws.data_ptr(), ws.numel(), sh)
        return lib.topk_paged(scores.data_ptr(), stride, lengths.data_ptr(), B, k,
                              page_table.data_ptr(), page_table.shape[1], page_size, out.data_ptr(), sh)

    _check(_on_device(index, call))
    return out


def topk_select_ex(scores: torch.Tensor, lengths: torch.Tensor, k: int,
                   page_table: Optional[torch.Tensor] = None, page_size: int = 0,
                   out: Optional[torch.Tensor] = None, *, sample_mode: int = 0,
                   cluster_size: int = 0, stash_capacity: int = 0, sample_z: float = 0.0,
                   counters: Optional[torch.Tensor] = None, probe_stage: int = 0,
                   probe_wait_us: int = 0, split_rows: int = 0,
                   workspace: Optional[torch.Tensor] = None, short_rows: int = 0,
                   stream=None) -> torch.Tensor:
    """Diagnostic variant: same result, with the internal path forced (see the
    header's ``topk_debug_opts``). ``counters`` is an optional int32/uint32
    CUDA tensor of ``NUM_COUNTERS`` entries that the kernel increments;
    ``workspace`` an optional uint8 CUDA tensor (first 4 KiB zero) that lets
    rows be split (``split_rows``)."""
    lib = load_library()
    B, stride, out = _prepare(scores, lengths, k, out)
    pt_ptr, pt_stride = None, 0
    if page_table is not None:
        if page_table.dtype != torch.int32 or not page_table.is_contiguous():
            raise ValueError("page_table must be contiguous int32")
        pt_ptr, pt_stride = page_table.data_ptr(), page_table.shape[1]
    if workspace is not None and (not workspace.is_cuda or workspace.dtype != torch.uint8
                                  or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous uint8 CUDA tensor")
    opts = _DebugOpts(sample_mode, cluster_size, stash_capacity, sample_z,
                      None if counters is None else counters.data_ptr(), probe_stage, probe_wait_us,
                      split_rows, None if workspace is None else workspace.data_ptr(),
                      0 if workspace is None else workspace.numel(), short_rows)
    if counters is not None and (counters.numel() < NUM_COUNTERS or not counters.is_cuda
                                 or counters.element_size() != 4):
        raise ValueError("counters must be a 4-byte CUDA tensor of NUM_COUNTERS entries")
    index = scores.get_device()
    sh = _stream_handle(index, stream)
    _check(_on_device(index, lambda: lib.topk_select_ex(scores.data_ptr(), stride, lengths.data_ptr(), B, k,
                                                        pt_ptr, pt_stride, page_size, out.data_ptr(),
                                                        ctypes.byref(opts), sh)))
    return out


def topk_select_bf16(scores: torch.Tensor, lengths: torch.Tensor, k: int,
                     page_table: Optional[torch.Tensor] = None, page_size: int = 0,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Top-k over bfloat16 scores ``[B, stride]`` (``stride <= 16384``): the
    indices, ``-1`` padded, or with ``page_table`` the mapped slots, as
    :func:`topk_ragged` / :func:`topk_paged` on the scores converted to
    float32."""
    lib = load_library()
    if not isinstance(scores, torch.Tensor) or scores.dim() != 2 or scores.dtype != torch.bfloat16 \
            or not scores.is_cuda or not scores.is_contiguous():
        raise ValueError("scores must be a contiguous bfloat16 CUDA tensor [B, stride]")
    B, stride = scores.shape
    if lengths.dtype != torch.int32 or lengths.device != scores.device or lengths.numel() != B \
            or not lengths.is_contiguous():
        raise ValueError("lengths must be a contiguous int32 tensor [B] on the scores' device")
    if out is None:
        out = torch.empty((B, max(int(k), 1)), dtype=torch.int32, device=scores.device)
    pt_ptr, pt_stride = None, 0
    if page_table is not None:
        if (page_table.dtype != torch.int32 or page_table.device != scores.device
                or page_table.dim() != 2 or page_table.shape[0] != B
                or not page_table.is_contiguous()):
            raise ValueError("page_table must be a contiguous int32 tensor [B, pages]")
        pt_ptr, pt_stride = page_table.data_ptr(), page_table.shape[1]
    index = scores.get_device()
    sh = _stream_handle(index, stream)
    _check(_on_device(index, lambda: lib.topk_select_bf16(scores.data_ptr(), stride, lengths.data_ptr(), B, k,
                                                          pt_ptr, pt_stride, page_size, out.data_ptr(), sh)))
    return out


def amax8_varlen(scores: torch.Tensor, lengths: torch.Tensor, topk: int = 0,
                 out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Level-one block keys of the two-level indexer (max of every 8 scores,
    the newest block +inf, rows with at most ``topk`` blocks skipped). ``out``
    float32 ``[B, >= ceil(stride / 8)]``; allocated (uninitialised) when not
    given."""
    lib = load_library()
    if not isinstance(scores, torch.Tensor) or scores.dim() != 2 or scores.dtype != torch.float32 \
            or not scores.is_cuda or not scores.is_contiguous():
        raise ValueError("scores must be a contiguous float32 CUDA tensor [B, stride]")
    B, stride = scores.shape
    if lengths.dtype != torch.int32 or lengths.device != scores.device or lengths.numel() != B:
        raise ValueError("lengths must be an int32 tensor [B] on the scores' device")
    if out is None:
        out = torch.empty((B, (stride + 7) // 8), dtype=torch.float32, device=scores.device)
    elif out.dtype != torch.float32 or out.device != scores.device or out.dim() != 2 \
            or out.shape[0] != B or out.stride(1) != 1:
        raise ValueError("out must be a float32 tensor [B, width] with unit inner stride")
    index = scores.get_device()
    sh = _stream_handle(index, stream)
    _check(_on_device(index, lambda: lib.topk_amax8_varlen(scores.data_ptr(), stride, lengths.data_ptr(), B,
                                                           int(topk), out.data_ptr(), out.stride(0), sh)))
    return out


def sort_candidate_blocks(blocks: torch.Tensor, lengths: torch.Tensor, stride: int,
                          page_table: torch.Tensor, page_size: int,
                          out_pages: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Rewrites ``blocks`` (int32 ``[B, k]``, selected block ids in any order,
    -1 padded) in ascending order with ``INT32_MAX`` padding, and returns the
    ids' pool slots ``page_table[b, id // bpp] * bpp + id % bpp`` (``bpp =
    page_size // 8``) in ``out_pages``."""
    lib = load_library()
    if blocks.dtype != torch.int32 or not blocks.is_cuda or blocks.dim() != 2 \
            or not blocks.is_contiguous():
        raise ValueError("blocks must be a contiguous int32 CUDA tensor [B, k]")
    B, k = blocks.shape
    if out_pages is None:
        out_pages = torch.empty_like(blocks)
    if page_table.dtype != torch.int32 or not page_table.is_contiguous() or page_table.dim() != 2:
        raise ValueError("page_table must be a contiguous int32 tensor [B, pages]")
    index = blocks.get_device()
    sh = _stream_handle(index, stream)
    _check(_on_device(index, lambda: lib.topk_sort_candidate_blocks(
        blocks.data_ptr(), B, k, lengths.data_ptr(), int(stride), page_table.data_ptr(),
        page_table.shape[1], int(page_size), out_pages.data_ptr(), sh)))
    return out_pages


def max_active_clusters(k: int, paged: bool, cluster_size: int) -> int:
    """Clusters of ``cluster_size`` CTAs of the streaming kernel (this k
    bucket and output kind) resident at once on the current device, as the
    driver answers it."""
    out = ctypes.c_int32(0)
    _check(load_library().topk_max_active_clusters(int(k), int(bool(paged)), int(cluster_size),
                                                   ctypes.byref(out)))
    return int(out.value)


def raw_library() -> ctypes.CDLL:
    """The loaded ctypes library, for callers that pass raw pointers."""
    return load_library()
