"""Shared helpers for the parity tests: tolerances, comparisons, GPU runners.

Tolerances (written here, used by every parity test):
* bf16 keys: |gpu - oracle| <= 5e-5 + 5e-5 * |oracle| elementwise (the fp32
  summation-order bound ROCm/ATOM #2651 "Accuracy" holds its kernels to).
* fp8 keys: |gpu - oracle| <= 1e-3 * |oracle| + 1e-5 elementwise, and the
  global similarity 1 - 2*sum(g*o) / sum(g^2 + o^2) <= 1e-3 (this library's
  reading of the aiter #4221 gate "calc_diff < 1e-3", which the page does not
  define).
* the -inf mask is bit-exact (0xFF800000) and zero logits are +0.0.
"""
from __future__ import annotations

import numpy as np

import qsa_inputs as qi

NEG_INF_BITS = 0xFF800000
BF16_TOL = (5e-5, 5e-5)  # (atol, rtol)
FP8_TOL = (1e-5, 1e-3)


def tol_for(kv_dtype: int):
    return BF16_TOL if kv_dtype == 0 else FP8_TOL


def assert_logits_match(gpu: np.ndarray, ref: np.ndarray, kv_dtype: int, where: str = ""):
    gpu = np.asarray(gpu, np.float32)
    ref = np.asarray(ref, np.float32)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    gb = gpu.view(np.uint32)
    masked = np.isneginf(ref)
    bad_mask = masked & (gb != NEG_INF_BITS)
    assert not bad_mask.any(), f"{where}: {int(bad_mask.sum())} masked entries are not exactly -inf " \
                               f"(first at {np.argwhere(bad_mask)[0].tolist()})"
    fin = ~masked
    assert np.isfinite(ref[fin]).all(), f"{where}: oracle produced non-finite visible logits"
    g, o = gpu[fin].astype(np.float64), ref[fin].astype(np.float64)
    assert np.isfinite(g).all(), f"{where}: GPU produced non-finite visible logits " \
                                 f"({int((~np.isfinite(g)).sum())} entries)"
    atol, rtol = tol_for(kv_dtype)
    err = np.abs(g - o)
    lim = atol + rtol * np.abs(o)
    bad = err > lim
    if bad.any():
        i = int(np.argmax(err / lim))
        raise AssertionError(f"{where}: {int(bad.sum())} of {g.size} logits out of tolerance; "
                             f"worst gpu={g[i]!r} oracle={o[i]!r} err={err[i]:.3g} lim={lim[i]:.3g}")
    if kv_dtype != 0 and g.size:
        denom = float((g * g + o * o).sum())
        if denom > 0:
            diff = 1.0 - 2.0 * float((g * o).sum()) / denom
            assert diff <= 1e-3, f"{where}: global similarity diff {diff}"
    zeros = gpu[fin] == 0
    assert (gpu[fin][zeros].view(np.uint32) == 0).all(), f"{where}: a zero logit is -0.0"


def assert_topk_strict(gpu_idx: np.ndarray, oracle_idx: np.ndarray, where: str = ""):
    """Same logits in, same index set out, bit for bit (both sides ascending)."""
    # both sides list the set in ascending column order with -1 padding last;
    # sort anyway (unused slots last) so only the set is compared
    big = np.iinfo(np.int32).max
    g = np.asarray(gpu_idx).astype(np.int64)
    g = np.sort(np.where(g < 0, big, g), axis=1)
    g = np.where(g == big, -1, g)
    o = np.asarray(oracle_idx)
    bad = (g != o).any(axis=1)
    assert not bad.any(), f"{where}: top-k differs in rows {np.flatnonzero(bad)[:8].tolist()}"


def assert_topk_within_tie_tolerance(gpu_idx: np.ndarray, oracle_logits: np.ndarray, visible, k: int,
                                     kv_dtype: int, where: str = ""):
    """GPU set (from GPU logits) vs oracle set (from oracle logits): they may differ
    only in columns whose oracle logit is within the logits tolerance of the
    oracle's k-th value."""
    atol, rtol = tol_for(kv_dtype)
    for r in range(gpu_idx.shape[0]):
        n = int(visible[r])
        row = oracle_logits[r, :n].astype(np.float64)
        g = set(int(c) for c in gpu_idx[r] if c >= 0)
        if n <= k:
            assert g == set(range(n)), f"{where}: row {r} should select all {n} columns"
            assert (np.asarray(gpu_idx[r]) == -1).sum() == k - n
            continue
        order = sorted(range(n), key=lambda c: (-row[c], c))
        o = set(order[:k])
        kth = row[order[k - 1]]
        for c in g ^ o:
            assert abs(row[c] - kth) <= 2 * (atol + rtol * abs(kth)), \
                f"{where}: row {r} column {c} differs (logit {row[c]}, k-th {kth})"
        assert len(g) == k


def nan_filled(shape, dtype, device):
    import torch

    t = torch.empty(shape, dtype=dtype, device=device)
    if dtype == torch.float32:
        t.fill_(float("nan"))
    else:
        t.fill_(-7)
    return t


def int_bf16(vals):
    return qi._bf16_bits(np.asarray(vals, dtype=np.float32))


def exact_case(kv_dtype, spec=None):
    """q, keys in {-3..3}; weights and scales powers of two: every partial sum is an
    integer multiple of a power of two below 2^24, so the result is exact."""
    rng = np.random.default_rng(5)
    if spec is None:
        spec = qi.custom("exact", 2, 2, 3, 8, [19, 20, 5, 24], 24, kv_dtype=kv_dtype, seed=3)
    inp = qi.build_inputs(spec)
    qv = rng.integers(-3, 4, size=inp.q.shape)
    inp.q = int_bf16(qv)
    inp.weights = rng.choice(np.array([0.25, 0.5, 1.0, 2.0], dtype=np.float32), size=inp.weights.shape)
    D, pc = spec.head_dim, spec.page_cols
    kvals = rng.integers(-3, 4, size=(inp.num_pages, pc, D))
    if kv_dtype == qi.KV_BF16:
        inp.kv = int_bf16(kvals.reshape(inp.num_pages, -1)).view(np.uint8).reshape(inp.num_pages, -1).copy()
        scales = np.ones((inp.num_pages, pc))
    else:
        codes = qi._e4m3_codes(kvals.astype(np.float32)).reshape(inp.num_pages, pc * D)
        scales = rng.choice(np.array([0.5, 1.0, 2.0], dtype=np.float32), size=(inp.num_pages, pc))
        kv = np.empty((inp.num_pages, pc * (D + 4)), dtype=np.uint8)
        kv[:, : pc * D] = codes
        kv[:, pc * D:] = scales.astype(np.float32).view(np.uint8).reshape(inp.num_pages, pc * 4)
        inp.kv = kv
    return inp, qv, kvals, scales
