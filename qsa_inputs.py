"""Seeded synthetic inputs for paged MQA-logits scoring and per-row top-k.

This module is shared by the CPU oracle tests, the GPU parity tests, ``smoke()``
and ``bench.py``.  It only draws random numbers and lays them out in the paged
formats the scorer reads; it computes none of the method's arithmetic (no dot
products, no ReLU, no head sum, no selection).  Both the oracle and the CUDA
path consume exactly the bytes produced here.

Workload shapes follow the workloads the QSA-indexer pages measure:

* "[ROCm/ATOM #2651] Performance": MTP-3 verify decode, 9 requests x 4 rows on
  64K-128K prompts, index block 16 or 64.
* "[vllm #62589] Performance": logits width 65,600 (max_model_len / 4), top-k
  2048, 4 heads, head_dim 128, 32K-262K contexts, one or four rows a request.
* "[aiter #4221] honest pool sizing commit": fp8 block-flat cache, B=16,
  kv_len 32768, KV block 64, pool sized from the blocks the batch needs.
* "[ATOM #2651] Performance" prefill profile: a 16,384-row chunk at ~96K.

Recipe (identical on every machine): numpy PCG64 seeded per workload; q and
keys ~ N(0,1) rounded to bf16 (round-to-nearest-even, by torch's CPU cast);
weights ~ U(0,1) fp32; fp8 keys are N(0,1) quantised per key with
scale = amax/448 (fp32) and torch's saturating-free e4m3fn cast after a clamp
to +-448.  The page pool holds exactly the pages the batch needs plus one
"poison" page filled with NaN; physical page ids are a random permutation and
every block-table entry past a request's needed pages points at the poison
page, so an over-read shows up as NaN instead of passing silently.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

HEAD_DIM = 128
KV_BF16 = 0
KV_FP8 = 1
Q_BF16 = 0
Q_FP8 = 1
BF16_NAN_BITS = 0x7FC0
FP8_NAN_CODE = 0x7F
# Rows of a given config are drawn from seed BASE_SEED + config index.
BASE_SEED = 1000


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even via torch."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 (already within +-448) -> OCP e4m3fn codes (uint8) via torch."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = torch.clamp(t, -448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@dataclasses.dataclass
class Spec:
    """Shape of one scoring + top-k call."""

    name: str
    num_requests: int
    rows_per_req: int
    num_heads: int
    page_cols: int
    out_cols: int
    k: int
    kv_dtype: int
    visible: np.ndarray  # int32 [R]
    seed: int
    head_dim: int = HEAD_DIM
    max_pages: Optional[int] = None  # block-table row width; default covers out_cols
    next_n_lens: Optional[np.ndarray] = None  # int32 [B] live rows per request (ragged call), or None
    q_dtype: int = Q_BF16  # Q_FP8: q as e4m3 codes (fp8 keys only)

    def __post_init__(self):
        self.visible = np.ascontiguousarray(self.visible, dtype=np.int32)
        assert self.visible.shape == (self.num_rows,)
        if self.next_n_lens is not None:
            self.next_n_lens = np.ascontiguousarray(self.next_n_lens, dtype=np.int32)
            assert self.next_n_lens.shape == (self.num_requests,)
        if self.max_pages is None:
            self.max_pages = max(1, -(-self.out_cols // self.page_cols))

    def live_rows(self) -> np.ndarray:
        """bool [R]: row i of request b is live when i < next_n_lens[b] (all rows without it)."""
        if self.next_n_lens is None:
            return np.ones(self.num_rows, dtype=bool)
        nn = np.clip(self.next_n_lens.astype(np.int64), 0, self.rows_per_req)
        return (np.arange(self.rows_per_req)[None, :] < nn[:, None]).reshape(-1)

    def live_visible(self) -> np.ndarray:
        """Visible counts with dead rows at 0 (the columns whose keys are read)."""
        return np.where(self.live_rows(), self.visible, 0).astype(np.int32)

    @property
    def num_rows(self) -> int:
        return self.num_requests * self.rows_per_req

    @property
    def key_bytes_per_col(self) -> int:
        return self.head_dim * 2 if self.kv_dtype == KV_BF16 else self.head_dim + 4

    def pages_needed(self) -> np.ndarray:
        """Per request: pages that hold at least one visible column of a live row."""
        vis = self.live_visible().reshape(self.num_requests, self.rows_per_req).max(axis=1)
        return -(-vis.astype(np.int64) // self.page_cols)

    def key_bytes_touched(self) -> int:
        """Algorithmic key-cache bytes: each request's visible columns (live rows), once."""
        vis = self.live_visible().reshape(self.num_requests, self.rows_per_req).max(axis=1)
        return int(vis.astype(np.int64).sum()) * self.key_bytes_per_col


@dataclasses.dataclass
class Inputs:
    spec: Spec
    q: np.ndarray  # uint16 bf16 bits, or uint8 e4m3 codes (fp8 q), [R, H, D]
    weights: np.ndarray  # float32 [R, H]
    kv: np.ndarray  # uint8 [num_pages, key_page_stride] raw paged cache
    key_page_stride: int  # bytes between pages (blocks)
    scale_offset: int  # fp8 block-flat: byte offset of the scales inside a block; -1 for bf16
    block_table: np.ndarray  # int32 [B, max_pages]
    poison_page: int

    @property
    def num_pages(self) -> int:
        return self.kv.shape[0]

    @property
    def visible(self) -> np.ndarray:
        return self.spec.visible


def build_inputs(spec: Spec, rng: Optional[np.random.Generator] = None) -> Inputs:
    """Draw q, weights and a permuted paged cache for ``spec``."""
    rng = rng if rng is not None else np.random.default_rng(spec.seed)
    R, H, D, pc = spec.num_rows, spec.num_heads, spec.head_dim, spec.page_cols
    B = spec.num_requests
    needed = spec.pages_needed()
    assert (needed <= spec.max_pages).all(), "visible count beyond the block table"
    total_needed = int(needed.sum())
    num_pages = total_needed + 1  # + one poison page

    if spec.q_dtype == Q_BF16:
        q = _bf16_bits(rng.standard_normal((R, H, D), dtype=np.float32))
    else:  # e4m3 codes of N(0,1) draws (no q scale: the weights carry it)
        q = _e4m3_codes(rng.standard_normal((R, H, D), dtype=np.float32))
    weights = rng.random((R, H), dtype=np.float32)

    perm = rng.permutation(num_pages).astype(np.int32)
    poison = int(perm[total_needed])
    block_table = np.full((B, spec.max_pages), poison, dtype=np.int32)
    pos = 0
    for b in range(B):
        n = int(needed[b])
        block_table[b, :n] = perm[pos : pos + n]
        pos += n

    if spec.kv_dtype == KV_BF16:
        stride = pc * D * 2
        kv = np.empty((num_pages, stride), dtype=np.uint8)
        # Draw page by page in chunks to bound peak host memory on large pools.
        chunk = max(1, (64 << 20) // stride)
        for p0 in range(0, num_pages, chunk):
            p1 = min(num_pages, p0 + chunk)
            vals = rng.standard_normal((p1 - p0, pc * D), dtype=np.float32)
            kv[p0:p1] = _bf16_bits(vals).view(np.uint8).reshape(p1 - p0, stride)
        kv[poison] = np.frombuffer(
            np.full(pc * D, BF16_NAN_BITS, dtype=np.uint16).tobytes(), dtype=np.uint8
        )
        scale_offset = -1
    else:
        stride = pc * (D + 4)
        kv = np.empty((num_pages, stride), dtype=np.uint8)
        chunk = max(1, (64 << 20) // stride)
        for p0 in range(0, num_pages, chunk):
            p1 = min(num_pages, p0 + chunk)
            vals = rng.standard_normal((p1 - p0, pc, D), dtype=np.float32)
            amax = np.abs(vals).max(axis=2).astype(np.float32)
            scale = (amax / np.float32(448.0)).astype(np.float32)
            safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
            codes = _e4m3_codes(vals / safe[:, :, None])
            codes[scale == 0] = 0
            kv[p0:p1, : pc * D] = codes.reshape(p1 - p0, pc * D)
            kv[p0:p1, pc * D :] = scale.view(np.uint8).reshape(p1 - p0, pc * 4)
        kv[poison, : pc * D] = FP8_NAN_CODE
        kv[poison, pc * D :] = np.full(pc, np.nan, dtype=np.float32).view(np.uint8)
        scale_offset = pc * D
    return Inputs(spec, q, weights, kv, stride, scale_offset, block_table, poison)


# ---------------------------------------------------------------------------
# Visible-column rules of the workloads (row -> number of compressed columns).
# ---------------------------------------------------------------------------


def decode_visible(context_tokens: Sequence[int], rows_per_req: int, ratio: int = 4) -> np.ndarray:
    """Verify row i of a request with L prompt tokens sees ceil((L + i) / ratio) columns."""
    out = []
    for L in context_tokens:
        for i in range(rows_per_req):
            out.append(-(-(int(L) + i) // ratio))
    return np.asarray(out, dtype=np.int32)


def prefill_visible(first_pos: int, num_rows: int, ratio: int = 4) -> np.ndarray:
    """Causal prefill: the row at position p sees floor((p + 1) / ratio) columns."""
    p = np.arange(first_pos, first_pos + num_rows, dtype=np.int64)
    return ((p + 1) // ratio).astype(np.int32)


# ---------------------------------------------------------------------------
# The five workloads (index = seed offset).
# ---------------------------------------------------------------------------


def tiny_mtp() -> Spec:
    """2 requests x 4 MTP rows, L = 4000 / 10000 tokens, page 64 columns, k 256."""
    vis = decode_visible([4000, 10000], 4)
    return Spec("tiny_mtp_2x4_p64", 2, 4, 4, 64, 2560, 256, KV_BF16, vis, BASE_SEED + 0)


def single_row_decode() -> Spec:
    """16 requests x 1 row at 32K tokens (8192 columns), page 16, width 65,600, k 2048."""
    vis = np.full(16, 8192, dtype=np.int32)
    return Spec("single_row_16x1_32k_p16", 16, 1, 4, 16, 65600, 2048, KV_BF16, vis, BASE_SEED + 1)


def mtp3_verify(page_cols: int = 16) -> Spec:
    """9 requests x 4 rows, prompts ~ U[64K, 128K] tokens, width 65,600, k 2048."""
    rng = np.random.default_rng(BASE_SEED + 2)
    L = rng.integers(65536, 131072 + 1, size=9)
    vis = decode_visible(L.tolist(), 4)
    return Spec(f"mtp3_9x4_64k-128k_p{page_cols}", 9, 4, 4, page_cols, 65600, 2048, KV_BF16, vis,
                BASE_SEED + 2)


def mtp3_large(page_cols: int = 16) -> Spec:
    """64 requests x 4 rows at 262,144 tokens, width 65,600, k 2048."""
    vis = decode_visible([262144] * 64, 4)
    return Spec(f"mtp3_64x4_262k_p{page_cols}", 64, 4, 4, page_cols, 65600, 2048, KV_BF16, vis,
                BASE_SEED + 2)


def fp8_h64() -> Spec:
    """16 requests x 1 row, 32,768 columns, 64 heads, fp8 block-flat KV block 64, k 2048."""
    vis = np.full(16, 32768, dtype=np.int32)
    return Spec("fp8_h64_16x1_kv32k_kvb64", 16, 1, 64, 64, 32768, 2048, KV_FP8, vis, BASE_SEED + 3)


def prefill_chunk() -> Spec:
    """1 request, 16,384 rows at positions 81,920..98,303, page 64, width 24,576, k 2048."""
    vis = prefill_visible(81920, 16384)
    return Spec("prefill_16384rows_at_81920_p64", 1, 16384, 4, 64, 24576, 2048, KV_BF16, vis,
                BASE_SEED + 4)


def prefill_chunk_4k() -> Spec:
    """The last 4,096 rows of prefill_chunk (positions 94,208..98,303): the same tile shape
    (64 rows x 4 heads = N 256) on a quarter of the logits, small enough for a full
    profiler capture."""
    vis = prefill_visible(94208, 4096)
    return Spec("prefill_4096rows_at_94208_p64", 1, 4096, 4, 64, 24576, 2048, KV_BF16, vis, BASE_SEED + 6)


def ragged_nn8() -> Spec:
    """aiter #4221 ragged mix: 116 requests x next_n 8, next_n_lens ~ U{1..8}, fp8 q and
    fp8 block-flat keys (KV block 64), 32 heads, prompts ~ U[32K, 128K] tokens, k 2048."""
    rng = np.random.default_rng(BASE_SEED + 5)
    L = rng.integers(32768, 131072 + 1, size=116)
    nn = rng.integers(1, 8 + 1, size=116).astype(np.int32)
    vis = decode_visible(L.tolist(), 8)
    return Spec("ragged_116x8_nn1-8_fp8q_h32", 116, 8, 32, 64, 32832, 2048, KV_FP8, vis, BASE_SEED + 5,
                next_n_lens=nn, q_dtype=Q_FP8)


def fp8q_h64() -> Spec:
    """fp8_h64 with fp8 q: 16 requests x 1 row, 32,768 columns, 64 heads, q and keys e4m3."""
    vis = np.full(16, 32768, dtype=np.int32)
    return Spec("fp8q_h64_16x1_kv32k_kvb64", 16, 1, 64, 64, 32768, 2048, KV_FP8, vis, BASE_SEED + 3,
                q_dtype=Q_FP8)


WORKLOADS = {
    "tiny_mtp": tiny_mtp,
    "single_row_decode": single_row_decode,
    "mtp3_verify_p16": lambda: mtp3_verify(16),
    "mtp3_verify_p64": lambda: mtp3_verify(64),
    "mtp3_large_p16": lambda: mtp3_large(16),
    "mtp3_large_p64": lambda: mtp3_large(64),
    "fp8_h64": fp8_h64,
    "prefill_chunk": prefill_chunk,
    "prefill_chunk_4k": prefill_chunk_4k,
    "ragged_nn8": ragged_nn8,
    "fp8q_h64": fp8q_h64,
}


def custom(name: str, num_requests: int, rows_per_req: int, num_heads: int, page_cols: int,
           visible: Sequence[int], out_cols: int, k: int = 64, kv_dtype: int = KV_BF16,
           seed: int = 7, max_pages: Optional[int] = None,
           next_n_lens: Optional[Sequence[int]] = None, q_dtype: int = Q_BF16) -> Spec:
    """Small ad-hoc shapes for tests."""
    nn = None if next_n_lens is None else np.asarray(next_n_lens, dtype=np.int32)
    return Spec(name, num_requests, rows_per_req, num_heads, page_cols, out_cols, k, kv_dtype,
                np.asarray(visible, dtype=np.int32), seed, max_pages=max_pages, next_n_lens=nn,
                q_dtype=q_dtype)


def random_logit_rows(rng: np.random.Generator, num_rows: int, width: int,
                      visible: Sequence[int], zero_frac: float = 0.06) -> np.ndarray:
    """Logit-like rows for top-k tests: mostly positive floats with exact +0.0
    entries (all-negative head dots give exactly 0 after the ReLU) and -inf past
    the visible count."""
    x = np.abs(rng.standard_normal((num_rows, width))).astype(np.float32) * np.float32(3.0)
    z = rng.random((num_rows, width)) < zero_frac
    x[z] = 0.0
    for r, v in enumerate(visible):
        x[r, int(v):] = -np.inf
    return x


def gather_rows_for(spec: Spec, max_rows: int, rng: np.random.Generator, group_rows: int = 0,
                    edge_groups: int = 0) -> List[int]:
    """A stratified sample of row indices: the first and last rows; with
    group_rows, the edge rows (first and last, and the row before) of the first
    three and of `edge_groups` more groups of `group_rows` consecutive rows
    spread over the batch, the last group among them; then random rows, up to
    max_rows or at least four of them past the edge rows."""
    R = spec.num_rows
    if R <= max_rows:
        return list(range(R))
    picks = {0, R - 1}
    if group_rows > 0 and edge_groups > 0:
        n_groups = -(-R // group_rows)
        spread = np.linspace(0, n_groups - 1, edge_groups).round().astype(int).tolist()
        for g in sorted(set([0, 1, 2] + spread) & set(range(n_groups))):
            first = int(g) * group_rows
            picks.update({first, min(R, first + group_rows) - 1})
            if first > 0:
                picks.add(first - 1)
    target = min(R, max(max_rows, len(picks) + 4))
    while len(picks) < target:
        picks.add(int(rng.integers(0, R)))
    return sorted(picks)


# ---------------------------------------------------------------------------
# Host -> device copies (plumbing only).
# ---------------------------------------------------------------------------


def device_tensors(inp: Inputs, device="cuda", pin: bool = False) -> dict:
    """torch tensors of ``inp`` on ``device`` (or pinned host memory with pin=True).

    q is bf16 [R, H, D]; kv is the raw paged cache as uint8 [num_pages, stride];
    scales (fp8 only) is a view at the block-flat scale offset."""
    import torch

    def t(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        return x.pin_memory() if pin else x.to(device)

    d = {
        "q": (t(inp.q.view(np.int16)).view(torch.bfloat16) if inp.spec.q_dtype == Q_BF16
              else t(inp.q).view(torch.float8_e4m3fn)),
        "weights": t(inp.weights),
        "kv": t(inp.kv),
        "block_table": t(inp.block_table),
        "visible": t(inp.spec.visible),
    }
    if inp.spec.next_n_lens is not None:  # ragged call: live rows per request, and the
        d["next_n_lens"] = t(inp.spec.next_n_lens)  # visible counts a top-k of it reads
        d["visible_live"] = t(inp.spec.live_visible())
    return d
