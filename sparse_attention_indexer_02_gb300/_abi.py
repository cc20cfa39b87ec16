"""ctypes binding of libqsa.so (include/qsa.h): argument marshalling only.

Every step of scoring and selection runs in the library's CUDA kernels; this
module converts torch tensors (or raw integer addresses) to pointers, fills
the descriptor struct and raises on a non-OK status.  If the library is not
built the import of a call fails loudly - there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqsa.so")

QSA_OK, QSA_ERR_INVALID_ARG, QSA_ERR_UNSUPPORTED, QSA_ERR_CUDA = 0, 1, 2, 3
KV_BF16, KV_FP8_E4M3 = 0, 1
Q_BF16, Q_FP8_E4M3 = 0, 1
VARIANT_AUTO, VARIANT_ROWCORE, VARIANT_UMMA, VARIANT_UMMA_TOPK, VARIANT_UMMA_LEAN = -1, 0, 1, 2, 3
VARIANT_NAMES = {VARIANT_ROWCORE: "rowcore", VARIANT_UMMA: "umma", VARIANT_UMMA_TOPK: "umma+topk",
                 VARIANT_UMMA_LEAN: "umma_lean"}

# Every symbol include/qsa.h declares.
EXPORTED = ("qsa_paged_mqa_logits", "qsa_paged_mqa_logits_ragged", "qsa_paged_mqa_logits_ex", "qsa_paged_mqa_topk",
            "qsa_paged_mqa_topk_workspace", "qsa_paged_mqa_topk_noalloc",
            "qsa_paged_mqa_topk_noalloc_counters", "qsa_select_topk", "qsa_select_topk_bounded", "qsa_plan_variant",
            "qsa_plan_variant_ex", "qsa_force_variant",
            "qsa_last_variant", "qsa_status_string", "qsa_last_error", "qsa_abi_version", "qsa_device_status",
            "qsa_page_stream")


class QSAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


class PagedDesc(ctypes.Structure):
    _fields_ = [
        ("num_requests", ctypes.c_int32),
        ("rows_per_req", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_cols", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("out_cols", ctypes.c_int64),
        ("key_page_stride", ctypes.c_int64),
        ("scale_page_stride", ctypes.c_int64),
    ]


_lib = None


def load_library():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.qsa_paged_mqa_logits.restype = ctypes.c_int
        lib.qsa_paged_mqa_logits.argtypes = [ctypes.POINTER(PagedDesc), vp, vp, vp, vp, vp, vp, vp, vp]
        lib.qsa_paged_mqa_logits_ragged.restype = ctypes.c_int
        lib.qsa_paged_mqa_logits_ragged.argtypes = [ctypes.POINTER(PagedDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.qsa_paged_mqa_logits_ex.restype = ctypes.c_int
        lib.qsa_paged_mqa_logits_ex.argtypes = [ctypes.POINTER(PagedDesc), i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.qsa_paged_mqa_topk.restype = ctypes.c_int
        lib.qsa_paged_mqa_topk.argtypes = [ctypes.POINTER(PagedDesc), i32, vp, vp, vp, vp, vp, vp, vp, i32, i64, vp,
                                           vp, vp, ctypes.c_size_t, vp]
        lib.qsa_paged_mqa_topk_noalloc.restype = ctypes.c_int
        lib.qsa_paged_mqa_topk_noalloc.argtypes = [ctypes.POINTER(PagedDesc), i32, vp, vp, vp, vp, vp, vp, vp, i32,
                                                   i64, vp, vp, vp]
        lib.qsa_paged_mqa_topk_workspace.restype = ctypes.c_int
        lib.qsa_paged_mqa_topk_workspace.argtypes = [ctypes.POINTER(PagedDesc), ctypes.POINTER(ctypes.c_size_t)]
        lib.qsa_select_topk.restype = ctypes.c_int
        lib.qsa_select_topk.argtypes = [vp, i64, i64, vp, i32, vp, vp]
        lib.qsa_select_topk_bounded.restype = ctypes.c_int
        lib.qsa_select_topk_bounded.argtypes = [vp, i64, i64, vp, i64, i32, vp, vp]
        lib.qsa_plan_variant.restype = ctypes.c_int
        lib.qsa_plan_variant.argtypes = [ctypes.POINTER(PagedDesc), ctypes.POINTER(i32)]
        lib.qsa_plan_variant_ex.restype = ctypes.c_int
        lib.qsa_plan_variant_ex.argtypes = [ctypes.POINTER(PagedDesc), i32, ctypes.POINTER(i32)]
        lib.qsa_force_variant.restype = None
        lib.qsa_force_variant.argtypes = [i32]
        lib.qsa_last_variant.restype = i32
        lib.qsa_last_variant.argtypes = []
        lib.qsa_status_string.restype = ctypes.c_char_p
        lib.qsa_status_string.argtypes = [i32]
        lib.qsa_last_error.restype = ctypes.c_char_p
        lib.qsa_last_error.argtypes = []
        lib.qsa_abi_version.restype = i32
        lib.qsa_abi_version.argtypes = []
        lib.qsa_paged_mqa_topk_noalloc_counters.restype = ctypes.c_int
        lib.qsa_paged_mqa_topk_noalloc_counters.argtypes = [ctypes.POINTER(ctypes.c_void_p),
                                                            ctypes.POINTER(ctypes.c_size_t)]
        lib.qsa_device_status.restype = ctypes.c_int
        lib.qsa_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        lib.qsa_page_stream.restype = ctypes.c_int
        lib.qsa_page_stream.argtypes = [ctypes.c_void_p, ctypes.c_int64, i32, ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        _lib = lib
    return _lib


def status_string(st: int) -> str:
    return load_library().qsa_status_string(int(st)).decode()


def last_error() -> str:
    return load_library().qsa_last_error().decode()


def _addr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int):
    if st != QSA_OK:
        raise QSAError(st, last_error())


def make_desc(num_requests, rows_per_req, num_heads, page_cols, max_pages, num_pages, out_cols,
              key_page_stride, kv_dtype=KV_BF16, scale_page_stride=0, head_dim=128) -> PagedDesc:
    return PagedDesc(int(num_requests), int(rows_per_req), int(num_heads), int(head_dim), int(page_cols),
                     int(max_pages), int(num_pages), int(kv_dtype), int(out_cols), int(key_page_stride),
                     int(scale_page_stride))


def paged_mqa_logits(desc: PagedDesc, q, weights, kv_cache, scales, block_table, visible_cols,
                     out_logits, stream=None, next_n_lens=None, q_dtype: int = Q_BF16) -> None:
    lib = load_library()
    if q_dtype != Q_BF16:
        st = lib.qsa_paged_mqa_logits_ex(ctypes.byref(desc), int(q_dtype), _addr(q), _addr(weights),
                                         _addr(kv_cache), _addr(scales), _addr(block_table),
                                         _addr(visible_cols), _addr(next_n_lens), _addr(out_logits),
                                         _stream(stream))
    elif next_n_lens is None:
        st = lib.qsa_paged_mqa_logits(ctypes.byref(desc), _addr(q), _addr(weights), _addr(kv_cache),
                                      _addr(scales), _addr(block_table), _addr(visible_cols),
                                      _addr(out_logits), _stream(stream))
    else:
        st = lib.qsa_paged_mqa_logits_ragged(ctypes.byref(desc), _addr(q), _addr(weights), _addr(kv_cache),
                                             _addr(scales), _addr(block_table), _addr(visible_cols),
                                             _addr(next_n_lens), _addr(out_logits), _stream(stream))
    _check(st)


def paged_mqa_topk(desc: PagedDesc, q, weights, kv_cache, scales, block_table, visible_cols, k: int,
                   out_logits, out_idx, workspace, workspace_bytes: int, stream=None, next_n_lens=None,
                   q_dtype: int = Q_BF16, max_visible: int = 0) -> None:
    """qsa_paged_mqa_topk: scoring and the per-row top-k in one call."""
    st = load_library().qsa_paged_mqa_topk(ctypes.byref(desc), int(q_dtype), _addr(q), _addr(weights),
                                           _addr(kv_cache), _addr(scales), _addr(block_table),
                                           _addr(visible_cols), _addr(next_n_lens), int(k), int(max_visible),
                                           _addr(out_logits), _addr(out_idx), _addr(workspace),
                                           int(workspace_bytes), _stream(stream))
    _check(st)


def paged_mqa_topk_noalloc(desc: PagedDesc, q, weights, kv_cache, scales, block_table, visible_cols, k: int,
                           out_logits, out_idx, stream=None, next_n_lens=None, q_dtype: int = Q_BF16,
                           max_visible: int = 0) -> None:
    """qsa_paged_mqa_topk_noalloc: the one-call form with the library's fixed counters."""
    st = load_library().qsa_paged_mqa_topk_noalloc(ctypes.byref(desc), int(q_dtype), _addr(q), _addr(weights),
                                                   _addr(kv_cache), _addr(scales), _addr(block_table),
                                                   _addr(visible_cols), _addr(next_n_lens), int(k),
                                                   int(max_visible), _addr(out_logits), _addr(out_idx),
                                                   _stream(stream))
    _check(st)


def topk_workspace_bytes(desc: PagedDesc) -> int:
    """Workspace bytes paged_mqa_topk needs for this shape (zeroed before first use)."""
    n = ctypes.c_size_t(0)
    _check(load_library().qsa_paged_mqa_topk_workspace(ctypes.byref(desc), ctypes.byref(n)))
    return n.value


def select_topk(logits, num_rows: int, row_stride: int, visible_cols, k: int, out_idx, stream=None) -> None:
    st = load_library().qsa_select_topk(_addr(logits), int(num_rows), int(row_stride), _addr(visible_cols),
                                        int(k), _addr(out_idx), _stream(stream))
    _check(st)


def select_topk_bounded(logits, num_rows: int, row_stride: int, visible_cols, max_visible: int, k: int, out_idx,
                        stream=None) -> None:
    st = load_library().qsa_select_topk_bounded(_addr(logits), int(num_rows), int(row_stride), _addr(visible_cols),
                                                int(max_visible), int(k), _addr(out_idx), _stream(stream))
    _check(st)


def page_stream(base, page_stride: int, page_bytes: int, pages, num_listed: int, pool_pages: int, checksum,
                stream=None) -> None:
    """qsa_page_stream (include/qsa.h): the measurement stream of listed pages."""
    _check(load_library().qsa_page_stream(_addr(base), int(page_stride), int(page_bytes), _addr(pages),
                                          int(num_listed), int(pool_pages), _addr(checksum), _stream(stream)))


def plan_variant(desc: PagedDesc, q_dtype: int | None = None) -> int:
    v = ctypes.c_int32(-1)
    if q_dtype is None:
        _check(load_library().qsa_plan_variant(ctypes.byref(desc), ctypes.byref(v)))
    else:
        _check(load_library().qsa_plan_variant_ex(ctypes.byref(desc), int(q_dtype), ctypes.byref(v)))
    return v.value


def force_variant(v: int) -> None:
    load_library().qsa_force_variant(int(v))


def last_variant() -> int:
    return load_library().qsa_last_variant()


def noalloc_counters() -> tuple[int, int]:
    """(device address, bytes) of qsa_paged_mqa_topk_noalloc's counter array on
    the current device."""
    ptr, n = ctypes.c_void_p(0), ctypes.c_size_t(0)
    _check(load_library().qsa_paged_mqa_topk_noalloc_counters(ctypes.byref(ptr), ctypes.byref(n)))
    return int(ptr.value or 0), int(n.value)


def device_status(clear: bool = True) -> int:
    """Device fault word (non-zero: a kernel gave up on a barrier wait); synchronises."""
    v = ctypes.c_uint32(0)
    _check(load_library().qsa_device_status(ctypes.byref(v), 1 if clear else 0))
    return v.value


def abi_version() -> int:
    return load_library().qsa_abi_version()
