"""Numpy brute force for tiny inputs (test infrastructure only).

An independent restatement used to cross-check the C oracle: it de-pages each
request's visible keys into a dense matrix with numpy fancy indexing, decodes
bf16 by placing the 16 bits in the top half of a float32, decodes e4m3 (fp8
keys, and fp8 q) with torch's float8_e4m3fn cast, and contracts with
``einsum`` in float64:

    S[r, h, c] = sum_d q[r, h, d] * key[c, d]
    logit[r, c] = sum_h w[r, h] * max(S[r, h, c], 0)      for c < visible[r]
                = -inf                                     otherwise

(ReLU per head before the weighted head sum: ROCm/ATOM #2651 "Changes";
aiter #4221 "Technical details".)  The top-k brute force is Python's
``sorted`` on (-value, column).
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def dense_keys(inp, b: int, ncols: int) -> np.ndarray:
    """float64 [ncols, D]: request b's first ncols keys, dequantised."""
    s = inp.spec
    D, pc = s.head_dim, s.page_cols
    cols = np.arange(ncols)
    pages = inp.block_table[b, cols // pc].astype(np.int64)
    slots = cols % pc
    if s.kv_dtype == 0:
        words = inp.kv.view(np.uint16).reshape(inp.kv.shape[0], -1)
        idx = slots[:, None] * D + np.arange(D)[None, :]
        return bf16_to_f64(words[pages[:, None], idx])
    idx = slots[:, None] * D + np.arange(D)[None, :]
    codes = inp.kv[pages[:, None], idx]
    sc_bytes = inp.kv[pages[:, None], inp.scale_offset + slots[:, None] * 4 + np.arange(4)[None, :]]
    scales = np.ascontiguousarray(sc_bytes).view(np.float32).reshape(-1).astype(np.float64)
    return e4m3_to_f64(codes) * scales[:, None]


def logits(inp) -> np.ndarray:
    s = inp.spec
    R, out_cols = s.num_rows, s.out_cols
    out = np.full((R, out_cols), -np.inf, dtype=np.float32)
    q = bf16_to_f64(inp.q) if getattr(s, "q_dtype", 0) == 0 else e4m3_to_f64(inp.q)  # [R, H, D]
    w = inp.weights.astype(np.float64)
    for b in range(s.num_requests):
        rows = range(b * s.rows_per_req, (b + 1) * s.rows_per_req)
        vmax = int(max(s.visible[r] for r in rows))
        if vmax == 0:
            continue
        K = dense_keys(inp, b, vmax)  # [vmax, D]
        for r in rows:
            v = int(s.visible[r])
            S = np.einsum("hd,cd->hc", q[r], K[:v])
            lg = (w[r][:, None] * np.maximum(S, 0.0)).sum(axis=0).astype(np.float32)
            out[r, :v] = lg + np.float32(0.0)
    return out


def topk(logits_rows: np.ndarray, visible, k: int) -> np.ndarray:
    rows = logits_rows.shape[0]
    out = np.full((rows, k), -1, dtype=np.int32)
    for r in range(rows):
        n = int(visible[r])
        if n <= k:
            out[r, :n] = np.arange(n)
            continue
        order = sorted(range(n), key=lambda c: (-float(logits_rows[r, c]), c))
        out[r] = np.sort(np.asarray(order[:k], dtype=np.int32))
    return out
