"""torch-tensor form of the C-ABI calls (argument marshalling only).

The descriptor is read off the tensors' shapes and strides; every byte of the
result is computed by libqsa.so.  All tensors must be on the current CUDA
device; work is enqueued on the current torch stream unless one is given.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _abi


def _desc_from(q, kv_cache, block_table, page_cols, out_cols, kv_dtype, scale_offset):
    R, H, D = q.shape
    B, max_pages = block_table.shape
    if B == 0 or R % B:
        raise ValueError("rows must be a whole number of rows per request")
    page_stride = kv_cache.stride(0) * kv_cache.element_size()
    scales = None
    scale_stride = 0
    if kv_dtype == _abi.KV_FP8_E4M3:
        if scale_offset < 0:
            raise ValueError("fp8 keys need the scale offset inside a block")
        scales = kv_cache.data_ptr() + scale_offset
        scale_stride = page_stride
    desc = _abi.make_desc(B, R // B, H, page_cols, max_pages, kv_cache.shape[0], out_cols, page_stride,
                          kv_dtype=kv_dtype, scale_page_stride=scale_stride, head_dim=D)
    q_dtype = _abi.Q_FP8_E4M3 if q.dtype in (torch.float8_e4m3fn, torch.uint8) else _abi.Q_BF16
    return desc, scales, q_dtype


def paged_mqa_logits(q: torch.Tensor, weights: torch.Tensor, kv_cache: torch.Tensor,
                     block_table: torch.Tensor, visible_cols: torch.Tensor, *, page_cols: int,
                     out_cols: int, kv_dtype: int = _abi.KV_BF16, scale_offset: int = -1,
                     out: Optional[torch.Tensor] = None, stream=None,
                     next_n_lens: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Index logits fp32 [R, out_cols] (include/qsa.h, qsa_paged_mqa_logits).

    q: bf16 [R, H, 128], or float8_e4m3fn (fp8 keys only: qsa_paged_mqa_logits_ex
    with fp8 q); weights: fp32 [R, H]; kv_cache: [num_pages, ...] paged
    keys whose dim-0 stride is the page stride; block_table: int32
    [num_requests, max_pages]; visible_cols: int32 [R].  For fp8 keys in the
    block-flat layout pass kv_dtype=KV_FP8_E4M3 and the byte offset of the
    scales inside a block (page_cols * 128).  next_n_lens (int32
    [num_requests]) selects qsa_paged_mqa_logits_ragged: a request's rows past
    its count are -inf."""
    desc, scales, q_dtype = _desc_from(q, kv_cache, block_table, page_cols, out_cols, kv_dtype, scale_offset)
    if out is None:
        out = torch.empty((q.shape[0], out_cols), dtype=torch.float32, device=q.device)
    _abi.paged_mqa_logits(desc, q, weights, kv_cache, scales, block_table, visible_cols, out, stream,
                          next_n_lens=next_n_lens, q_dtype=q_dtype)
    return out


def select_topk(logits: torch.Tensor, visible_cols: torch.Tensor, k: int,
                out: Optional[torch.Tensor] = None, stream=None, max_visible: int = 0) -> torch.Tensor:
    """Top-k column indices int32 [rows, k] (include/qsa.h, qsa_select_topk;
    with max_visible > 0, qsa_select_topk_bounded: the visible counts are
    clamped to that host bound)."""
    rows = logits.shape[0]
    if out is None:
        out = torch.empty((rows, k), dtype=torch.int32, device=logits.device)
    if max_visible > 0:
        _abi.select_topk_bounded(logits, rows, logits.stride(0), visible_cols, max_visible, k, out, stream)
    else:
        _abi.select_topk(logits, rows, logits.stride(0), visible_cols, k, out, stream)
    return out


def page_stream(pool: torch.Tensor, page_stride: int, page_bytes: int, pages: torch.Tensor,
                checksum: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Stream the listed pages of `pool` (a device buffer of whole pages) and
    XOR their 32-bit words into `checksum` (include/qsa.h, qsa_page_stream)."""
    if checksum is None:
        checksum = torch.zeros(1, dtype=torch.int32, device=pool.device)
    pool_pages = pool.numel() * pool.element_size() // page_stride
    _abi.page_stream(pool, page_stride, page_bytes, pages, pages.numel(), pool_pages, checksum, stream)
    return checksum


_workspaces: dict = {}


def topk_workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    """A zeroed workspace of at least nbytes on `device`, kept for later calls
    (every completed qsa_paged_mqa_topk call leaves it zero again).  One per
    device: calls that may overlap on other streams need their own."""
    key = torch.device(device).index if torch.device(device).index is not None else torch.cuda.current_device()
    ws = _workspaces.get(key)
    if ws is None or ws.numel() * 4 < nbytes:
        ws = torch.zeros(max(64, (nbytes + 3) // 4), dtype=torch.int32, device=device)
        _workspaces[key] = ws
    return ws


def paged_mqa_topk(q: torch.Tensor, weights: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                   visible_cols: torch.Tensor, k: int, *, page_cols: int, out_cols: int,
                   kv_dtype: int = _abi.KV_BF16, scale_offset: int = -1, max_visible: int = 0,
                   out_logits: Optional[torch.Tensor] = None, out_idx: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None,
                   next_n_lens: Optional[torch.Tensor] = None):
    """(logits fp32 [R, out_cols], top-k int32 [R, k]) in one call
    (include/qsa.h, qsa_paged_mqa_topk); arguments as paged_mqa_logits, plus k
    and the host bound max_visible of the visible counts (0: unknown)."""
    desc, scales, q_dtype = _desc_from(q, kv_cache, block_table, page_cols, out_cols, kv_dtype, scale_offset)
    R = q.shape[0]
    if out_logits is None:
        out_logits = torch.empty((R, out_cols), dtype=torch.float32, device=q.device)
    if out_idx is None:
        out_idx = torch.empty((R, k), dtype=torch.int32, device=q.device)
    nbytes = _abi.topk_workspace_bytes(desc)
    if workspace is None and nbytes:
        workspace = topk_workspace(nbytes, q.device)
    _abi.paged_mqa_topk(desc, q, weights, kv_cache, scales, block_table, visible_cols, k, out_logits, out_idx,
                        workspace, 0 if workspace is None else workspace.numel() * workspace.element_size(),
                        stream, next_n_lens=next_n_lens, q_dtype=q_dtype, max_visible=max_visible)
    return out_logits, out_idx
