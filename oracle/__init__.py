"""CPU oracle for paged MQA-logits scoring and per-row top-k.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU baseline / ``--impl reference`` arm import this package.
The product library never loads it, and it shares no code with the CUDA path.

Two independent CPU implementations live here:

* ``qsa_oracle.c`` (built by :func:`build`): the definition written out element
  by element in double precision, with pthreads over rows.  This is the oracle
  the GPU parity tests compare against.
* ``brute.py``: a numpy restatement for tiny inputs (dense de-paged keys,
  ``einsum`` in float64), used only to cross-check the C oracle.

Each function cites the page and section it follows in ``qsa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_qsa.so")
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc a C oracle source into a shared library (IEEE double, no FMA contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile qsa_oracle.c into liboracle_qsa.so next to it (skipped when up to date)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _load():
    global _lib
    if _lib is None:
        # QSA_ORACLE_LIB points the pins at a deliberately broken build (mutation test).
        path = os.environ.get("QSA_ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        lib.qsa_oracle_bf16_value.restype = ctypes.c_double
        lib.qsa_oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.qsa_oracle_e4m3_value.restype = ctypes.c_double
        lib.qsa_oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        lib.qsa_oracle_paged_mqa_logits.restype = ctypes.c_int
        lib.qsa_oracle_paged_mqa_logits.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i64, i64,
                                                    i64, vp, vp, vp, vp, vp, vp, vp, i64, vp, i32]
        lib.qsa_oracle_paged_mqa_logits_ex.restype = ctypes.c_int
        lib.qsa_oracle_paged_mqa_logits_ex.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i64, i64,
                                                       i64, i32, vp, vp, vp, vp, vp, vp, vp, i64, vp, i32]
        lib.qsa_oracle_select_topk.restype = ctypes.c_int
        lib.qsa_oracle_select_topk.argtypes = [vp, i64, i64, vp, i32, vp, i32]
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def bf16_value(bits: int) -> float:
    return _load().qsa_oracle_bf16_value(int(bits))


def e4m3_value(code: int) -> float:
    return _load().qsa_oracle_e4m3_value(int(code))


def paged_mqa_logits(inp, rows: Optional[Sequence[int]] = None, threads: Optional[int] = None,
                     *, q=None, weights=None, kv=None, block_table=None, visible=None,
                     next_n_lens="spec") -> np.ndarray:
    """Oracle logits for ``inp`` (a ``qsa_inputs.Inputs``) as float32 [len(rows) or R, out_cols].

    Keyword overrides replace single tensors (for invariance tests).  With live-row
    counts (``next_n_lens``, default: the spec's), aiter #4221 "Ragged next_n":
    request b's leading min(next_n_lens[b], rows_per_req) rows are scored and every
    column of its other rows is -inf, i.e. those rows see no column."""
    lib = _load()
    s = inp.spec
    q_dtype = getattr(s, "q_dtype", 0)
    q = np.ascontiguousarray(inp.q if q is None else q, dtype=np.uint16 if q_dtype == 0 else np.uint8)
    w = np.ascontiguousarray(inp.weights if weights is None else weights, dtype=np.float32)
    kvb = np.ascontiguousarray(inp.kv if kv is None else kv, dtype=np.uint8)
    bt = np.ascontiguousarray(inp.block_table if block_table is None else block_table, dtype=np.int32)
    vis = np.ascontiguousarray(s.visible if visible is None else visible, dtype=np.int32)
    nn = s.next_n_lens if isinstance(next_n_lens, str) else next_n_lens
    if nn is not None:
        live_n = np.clip(np.asarray(nn, dtype=np.int64), 0, s.rows_per_req)
        live = (np.arange(s.rows_per_req)[None, :] < live_n[:, None]).reshape(-1)
        vis = np.ascontiguousarray(np.where(live, vis, 0), dtype=np.int32)
    sel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = s.num_rows if sel is None else len(sel)
    out = np.empty((n, s.out_cols), dtype=np.float32)
    if n == 0:
        return out
    scales = None
    if s.kv_dtype == 1:
        scales = ctypes.c_void_p(kvb.ctypes.data + inp.scale_offset)
    st = lib.qsa_oracle_paged_mqa_logits_ex(
        s.num_requests, s.rows_per_req, s.num_heads, s.head_dim, s.page_cols, s.max_pages,
        kvb.shape[0], s.kv_dtype, s.out_cols, inp.key_page_stride, inp.key_page_stride, q_dtype,
        _ptr(q), _ptr(w), _ptr(kvb), scales, _ptr(bt), _ptr(vis), _ptr(sel),
        n, _ptr(out), threads or default_threads())
    if st != 0:
        raise ValueError(f"oracle rejected the inputs (status {st})")
    return out


def select_topk(logits: np.ndarray, visible: np.ndarray, k: int, threads: Optional[int] = None) -> np.ndarray:
    """Oracle top-k: int32 [rows, k], each row's set in ascending column order, -1 padded."""
    lib = _load()
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    vis = np.ascontiguousarray(visible, dtype=np.int32)
    rows, stride = lg.shape
    out = np.empty((rows, k), dtype=np.int32)
    if rows == 0:
        return out
    st = lib.qsa_oracle_select_topk(_ptr(lg), rows, stride, _ptr(vis), int(k), _ptr(out),
                                    threads or default_threads())
    if st != 0:
        raise ValueError(f"oracle top-k rejected the inputs (status {st})")
    return out


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(force="--force" in sys.argv))
