"""ctypes front end of the CPU oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. It compiles ``topk_oracle.cpp`` with the host C++
compiler on first use (or via :func:`build`) and exposes the two selections
and the two-level indexer's block helpers on numpy arrays. The library it loads is unrelated to the CUDA library of the
product package; they share no source.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "topk_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

ORACLE_OK, ORACLE_EARG, ORACLE_ENAN, ORACLE_EPAGE = 0, 1, 2, 3
_ERRORS = {ORACLE_EARG: "bad arguments", ORACLE_ENAN: "NaN inside a row's valid prefix",
           ORACLE_EPAGE: "page index or mapped slot out of range"}

_lib = None


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle error {code}: {_ERRORS.get(code, 'unknown')}")
        self.code = code


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", *extra_flags, src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _stale() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))


class Oracle:
    """Bound oracle library. ``Oracle(path)`` loads another build of the same
    source (the mutation tests use this)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_topk_ragged.argtypes = [f32p, ctypes.c_int64, i32p, ctypes.c_int32,
                                           ctypes.c_int32, i32p]
        lib.oracle_topk_ragged.restype = ctypes.c_int
        lib.oracle_topk_paged.argtypes = [f32p, ctypes.c_int64, i32p, ctypes.c_int32,
                                          ctypes.c_int32, i32p, ctypes.c_int64, ctypes.c_int32,
                                          i32p]
        lib.oracle_topk_paged.restype = ctypes.c_int
        lib.oracle_amax8_varlen.argtypes = [f32p, ctypes.c_int64, i32p, ctypes.c_int32,
                                            ctypes.c_int32, f32p, ctypes.c_int64]
        lib.oracle_amax8_varlen.restype = ctypes.c_int
        lib.oracle_sort_candidate_blocks.argtypes = [i32p, ctypes.c_int32, ctypes.c_int32, i32p,
                                                     ctypes.c_int64, i32p, ctypes.c_int64,
                                                     ctypes.c_int32, i32p]
        lib.oracle_sort_candidate_blocks.restype = ctypes.c_int
        lib.oracle_abi_version.restype = ctypes.c_int
        self._lib = lib
        self.path = path

    @staticmethod
    def _f32(a):
        return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))

    @staticmethod
    def _i32(a):
        return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def topk_ragged(self, scores: np.ndarray, lengths: np.ndarray, k: int) -> np.ndarray:
        """Indices ``[B, k]`` of each row's ``min(k, len)`` best scores, best
        first (ties by ascending index), ``-1`` after them."""
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        lengths = np.ascontiguousarray(lengths, dtype=np.int32)
        B, stride = scores.shape
        out = np.empty((B, k), dtype=np.int32)
        rc = self._lib.oracle_topk_ragged(self._f32(scores), stride, self._i32(lengths), B, k,
                                          self._i32(out))
        if rc != ORACLE_OK:
            raise OracleError(rc)
        return out

    def topk_paged(self, scores: np.ndarray, lengths: np.ndarray, k: int,
                   page_table: np.ndarray, page_size: int) -> np.ndarray:
        """As :meth:`topk_ragged`, each valid index mapped through the page table."""
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        lengths = np.ascontiguousarray(lengths, dtype=np.int32)
        page_table = np.ascontiguousarray(page_table, dtype=np.int32)
        B, stride = scores.shape
        out = np.empty((B, k), dtype=np.int32)
        rc = self._lib.oracle_topk_paged(self._f32(scores), stride, self._i32(lengths), B, k,
                                         self._i32(page_table), page_table.shape[1], page_size,
                                         self._i32(out))
        if rc != ORACLE_OK:
            raise OracleError(rc)
        return out


    def amax8_varlen(self, scores: np.ndarray, lengths: np.ndarray, topk: int,
                     out: np.ndarray) -> np.ndarray:
        """Level-one block keys written into ``out`` (float32 ``[B, >= ceil(stride/8)]``,
        pre-filled by the caller: slots the definition does not write keep
        their value)."""
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        lengths = np.ascontiguousarray(lengths, dtype=np.int32)
        out = np.ascontiguousarray(out, dtype=np.float32).copy()
        B, stride = scores.shape
        rc = self._lib.oracle_amax8_varlen(self._f32(scores), stride, self._i32(lengths), B, topk,
                                           self._f32(out), out.shape[1])
        if rc != ORACLE_OK:
            raise OracleError(rc)
        return out

    def sort_candidate_blocks(self, blocks: np.ndarray, lengths: np.ndarray, stride: int,
                              page_table: np.ndarray, page_size: int):
        """(ascending block table, pool slots), both int32 ``[B, k]``."""
        blocks = np.ascontiguousarray(blocks, dtype=np.int32).copy()
        lengths = np.ascontiguousarray(lengths, dtype=np.int32)
        page_table = np.ascontiguousarray(page_table, dtype=np.int32)
        B, k = blocks.shape
        pages = np.empty_like(blocks)
        rc = self._lib.oracle_sort_candidate_blocks(self._i32(blocks), B, k, self._i32(lengths),
                                                    stride, self._i32(page_table),
                                                    page_table.shape[1], page_size,
                                                    self._i32(pages))
        if rc != ORACLE_OK:
            raise OracleError(rc)
        return blocks, pages


def load(rebuild_if_stale: bool = True) -> Oracle:
    """The oracle built from this directory's source (compiled if missing)."""
    global _lib
    if _lib is None:
        if rebuild_if_stale and _stale():
            build()
        _lib = Oracle(_LIB_PATH)
    return _lib


def topk_ragged(scores, lengths, k):
    return load().topk_ragged(scores, lengths, k)


def topk_paged(scores, lengths, k, page_table, page_size):
    return load().topk_paged(scores, lengths, k, page_table, page_size)


def amax8_varlen(scores, lengths, topk, out):
    return load().amax8_varlen(scores, lengths, topk, out)


def sort_candidate_blocks(blocks, lengths, stride, page_table, page_size):
    return load().sort_candidate_blocks(blocks, lengths, stride, page_table, page_size)


def source_path() -> str:
    return _SRC


def library_path() -> Optional[str]:
    return _LIB_PATH if os.path.exists(_LIB_PATH) else None
