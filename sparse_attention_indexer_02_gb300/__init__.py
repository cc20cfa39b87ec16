"""GB300 (sm_103a) QSA-indexer hot path: paged MQA-logits scoring and per-row top-k.

The compute lives in libqsa.so (CUDA kernels behind the C ABI in include/qsa.h).
This package is its thin binding: :mod:`._abi` marshals pointers and sizes
through ctypes, :mod:`.torch_api` takes torch tensors and passes their device
pointers and the current stream, and :mod:`.build` compiles the library.
"""
from ._abi import (EXPORTED, KV_BF16, KV_FP8_E4M3, LIB_PATH, Q_BF16, Q_FP8_E4M3, QSA_ERR_CUDA, QSA_ERR_INVALID_ARG,
                   QSA_ERR_UNSUPPORTED, QSA_OK, VARIANT_AUTO, VARIANT_NAMES, VARIANT_ROWCORE,
                   VARIANT_UMMA, VARIANT_UMMA_LEAN, VARIANT_UMMA_TOPK, PagedDesc, QSAError, abi_version, device_status,
                   force_variant, last_error, last_variant, load_library, make_desc, page_stream, paged_mqa_logits,
                   paged_mqa_topk, plan_variant, select_topk, select_topk_bounded, status_string,
                   topk_workspace_bytes)

__all__ = [
    "EXPORTED", "KV_BF16", "KV_FP8_E4M3", "LIB_PATH", "Q_BF16", "Q_FP8_E4M3", "QSA_OK", "QSA_ERR_INVALID_ARG", "QSA_ERR_UNSUPPORTED",
    "QSA_ERR_CUDA", "VARIANT_AUTO", "VARIANT_ROWCORE", "VARIANT_UMMA", "VARIANT_UMMA_LEAN", "VARIANT_UMMA_TOPK", "VARIANT_NAMES",
    "PagedDesc", "QSAError", "abi_version", "device_status", "force_variant", "last_error", "last_variant",
    "load_library", "make_desc", "page_stream", "paged_mqa_logits", "paged_mqa_topk", "plan_variant", "select_topk",
    "select_topk_bounded", "status_string", "topk_workspace_bytes",
]
