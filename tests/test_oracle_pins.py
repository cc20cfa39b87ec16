"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test fixes the oracle to something it cannot agree with by construction:
a format definition or an independent library cast, an exact closed form,
brute force by a second implementation, an invariant the pages state, or a
value the pages print (fixtures under tests/golden/, each with its source).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import qsa_inputs as qi
from oracle import brute
from qsa_testlib import exact_case as _exact_case, int_bf16 as _int_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------


def test_bf16_decode_matches_library_cast_on_all_codes(oracle_mod):
    codes = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_mod.bf16_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    assert (np.signbit(got[~nan]) == np.signbit(ref[~nan])).all()


def test_bf16_decode_definition_points(oracle_mod):
    v = oracle_mod.bf16_value
    assert v(0x3F80) == 1.0 and v(0xC000) == -2.0 and v(0x3FC0) == 1.5
    assert v(0x0001) == 2.0 ** -133  # smallest subnormal
    assert v(0x0080) == 2.0 ** -126  # smallest normal
    assert v(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127
    assert math.isinf(v(0x7F80)) and math.isnan(v(0x7FC0))
    assert math.copysign(1.0, v(0x8000)) == -1.0


def test_e4m3_decode_matches_library_cast_on_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_mod.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_e4m3_decode_definition_points(oracle_mod):
    v = oracle_mod.e4m3_value
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0  # largest finite
    assert v(0x01) == 2.0 ** -9  # smallest subnormal
    assert v(0x07) == 7 * 2.0 ** -9
    assert v(0x08) == 2.0 ** -6  # smallest normal
    assert v(0x38) == 1.0 and v(0x40) == 2.0 and v(0x3C) == 1.5
    assert math.isnan(v(0x7F)) and math.isnan(v(0xFF))
    assert math.copysign(1.0, v(0x80)) == -1.0
    finite = [v(c) for c in range(256) if c not in (0x7F, 0xFF)]
    assert max(finite) == 448.0 and len(set(finite)) == 253  # +0 and -0 compare equal


def test_every_finite_e4m3_value_is_exact_in_bf16(oracle_mod):
    """The GPU path widens fp8 keys to bf16; that step must lose nothing."""
    vals = np.array([oracle_mod.e4m3_value(c) for c in range(256) if c not in (0x7F, 0xFF)])
    rt = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    assert (rt == vals).all()


# --------------------------------------------------------------------------
# Logits: brute force, exact cases, closed forms, invariants
# --------------------------------------------------------------------------

SMALL_SPECS = [
    dict(name="b2x4_p16", num_requests=2, rows_per_req=4, num_heads=4, page_cols=16,
         visible=[0, 33, 57, 64], out_cols=80),
    dict(name="b3x1_p64_h8", num_requests=3, rows_per_req=1, num_heads=8, page_cols=64,
         visible=[130, 1, 64], out_cols=192),
    dict(name="b1x3_p5_h1", num_requests=1, rows_per_req=3, num_heads=1, page_cols=5,
         visible=[11, 12, 13], out_cols=20),
    dict(name="b2x2_p16_h3", num_requests=2, rows_per_req=2, num_heads=3, page_cols=16,
         visible=[40, 40, 17, 0], out_cols=48),
]


def _spec(d, kv_dtype=qi.KV_BF16, seed=11):
    vis = d["visible"]
    if len(vis) != d["num_requests"] * d["rows_per_req"]:
        vis = (vis * d["num_requests"] * d["rows_per_req"])[: d["num_requests"] * d["rows_per_req"]]
    return qi.custom(d["name"], d["num_requests"], d["rows_per_req"], d["num_heads"],
                     d["page_cols"], vis, d["out_cols"], kv_dtype=kv_dtype, seed=seed)


def _close_1ulp(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    fin = np.isfinite(b)
    if not (np.isfinite(a) == fin).all():
        return False
    if not (a[~fin].view(np.uint32) == b[~fin].view(np.uint32)).all():
        return False
    ia = a[fin].view(np.int32).astype(np.int64)
    ib = b[fin].view(np.int32).astype(np.int64)
    return bool((np.abs(ia - ib) <= 1).all())


@pytest.mark.parametrize("d", SMALL_SPECS, ids=lambda d: d["name"])
@pytest.mark.parametrize("kv_dtype", [qi.KV_BF16, qi.KV_FP8], ids=["bf16", "fp8"])
def test_logits_match_numpy_bruteforce(oracle_mod, d, kv_dtype):
    inp = qi.build_inputs(_spec(d, kv_dtype))
    got = oracle_mod.paged_mqa_logits(inp)
    ref = brute.logits(inp)
    assert _close_1ulp(got, ref)


@pytest.mark.parametrize("kv_dtype", [qi.KV_BF16, qi.KV_FP8], ids=["bf16", "fp8"])
def test_exact_integer_case_is_bit_exact(oracle_mod, kv_dtype):
    inp, qv, kvals, scales = _exact_case(kv_dtype)
    s = inp.spec
    got = oracle_mod.paged_mqa_logits(inp)
    for r in range(s.num_rows):
        b = r // s.rows_per_req
        for c in range(s.out_cols):
            if c >= s.visible[r]:
                assert got[r, c] == -np.inf
                continue
            p = int(inp.block_table[b, c // s.page_cols])
            j = c % s.page_cols
            acc = Fraction(0)
            for h in range(s.num_heads):
                dot = Fraction(0)
                for d in range(s.head_dim):
                    dot += Fraction(int(qv[r, h, d])) * Fraction(int(kvals[p, j, d])) * Fraction(float(scales[p, j]))
                acc += Fraction(float(inp.weights[r, h])) * max(dot, Fraction(0))
            want = np.float32(float(acc))
            assert got[r, c].view(np.uint32) == (want + np.float32(0)).view(np.uint32), (r, c)


def _one_col_inputs(qrows, key, weights, kv_dtype=qi.KV_BF16, scale=1.0):
    H = len(qrows)
    spec = qi.custom("onecol", 1, 1, H, 1, [1], 1, kv_dtype=kv_dtype, seed=1)
    inp = qi.build_inputs(spec)
    D = spec.head_dim
    q = np.zeros((1, H, D), np.float32)
    for h, qr in enumerate(qrows):
        q[0, h, : len(qr)] = qr
    inp.q = _int_bf16(q)
    inp.weights = np.asarray([weights], dtype=np.float32)
    k = np.zeros(D, np.float32)
    k[: len(key)] = key
    page = int(inp.block_table[0, 0])
    if kv_dtype == qi.KV_BF16:
        inp.kv[page] = _int_bf16(k).view(np.uint8)
    else:
        inp.kv[page, :D] = qi._e4m3_codes(k)
        inp.kv[page, D:] = np.asarray([scale], np.float32).view(np.uint8)
    return inp


def test_relu_applies_per_head_before_the_weighted_sum(oracle_mod):
    # head dots: +3 and -6; weights (2, -1).  Per-head ReLU then weight: 2*3 + (-1)*0 = 6.
    # ReLU after the head sum would give max(0, 6 + 6) = 12; weight before ReLU gives 6 + 6 = 12;
    # no ReLU gives 12; dropping the weight gives 3.
    inp = _one_col_inputs([[1.0, 1.0], [-2.0, -2.0]], [1.5, 1.5], [2.0, -1.0])
    assert oracle_mod.paged_mqa_logits(inp)[0, 0] == 6.0


def test_zero_logit_is_positive_zero(oracle_mod):
    # every head dot negative -> exactly 0; with a negative weight w*0 would be -0.0
    inp = _one_col_inputs([[1.0], [2.0]], [-1.0], [-1.0, 3.0])
    v = oracle_mod.paged_mqa_logits(inp)[0, 0]
    assert v.view(np.uint32) == 0


def test_fp8_scale_dequantises_the_key_before_relu(oracle_mod):
    # key codes +2, scale -0.5: dequantised key is -1, dot -1 -> ReLU -> 0.
    # Applying the scale after the ReLU would give -0.5 * 2 = -1.
    inp = _one_col_inputs([[1.0]], [2.0], [1.0], kv_dtype=qi.KV_FP8, scale=-0.5)
    assert oracle_mod.paged_mqa_logits(inp)[0, 0] == 0.0
    inp = _one_col_inputs([[1.0]], [2.0], [1.0], kv_dtype=qi.KV_FP8, scale=0.25)
    assert oracle_mod.paged_mqa_logits(inp)[0, 0] == 0.5


def test_fp8_nonnegative_scale_hoists_out_of_the_relu(oracle_mod):
    """aiter #4221 (comment-trim commit): ReLU(s*x) = s*ReLU(x) for s >= 0, so a
    power-of-two per-key scale multiplies each logit exactly."""
    spec = qi.custom("hoist", 2, 1, 4, 16, [40, 29], 48, kv_dtype=qi.KV_FP8, seed=9)
    inp = qi.build_inputs(spec)
    pc, D = spec.page_cols, spec.head_dim
    ones = np.ones((inp.num_pages, pc), np.float32)
    inp1 = qi.build_inputs(spec)
    inp1.kv[:, pc * D:] = ones.view(np.uint8).reshape(inp.num_pages, -1)
    inp4 = qi.build_inputs(spec)
    inp4.kv[:, pc * D:] = (4 * ones).view(np.uint8).reshape(inp.num_pages, -1)
    l1 = oracle_mod.paged_mqa_logits(inp1)
    l4 = oracle_mod.paged_mqa_logits(inp4)
    fin = np.isfinite(l1)
    assert (l4[fin] == 4 * l1[fin]).all()
    assert (l4[~fin] == -np.inf).all()


def test_single_head_unit_weight_nonnegative_is_a_plain_matmul(oracle_mod):
    spec = qi.custom("mm", 2, 3, 1, 16, [50, 50, 50, 31, 47, 0], 64, seed=21)
    inp = qi.build_inputs(spec)
    rng = np.random.default_rng(4)
    inp.q = _int_bf16(np.abs(rng.standard_normal(inp.q.shape)).astype(np.float32))
    D = spec.head_dim
    kvals = np.abs(rng.standard_normal((inp.num_pages, spec.page_cols * D))).astype(np.float32)
    inp.kv = _int_bf16(kvals).view(np.uint8).reshape(inp.num_pages, -1).copy()
    inp.weights = np.ones_like(inp.weights)
    got = oracle_mod.paged_mqa_logits(inp)
    qf = brute.bf16_to_f64(inp.q)[:, 0, :]
    for r in range(spec.num_rows):
        b = r // spec.rows_per_req
        v = int(spec.visible[r])
        K = brute.dense_keys(inp, b, v)
        want = np.matmul(K, qf[r]).astype(np.float32)
        assert _close_1ulp(got[r, :v], want)
        assert (got[r, v:] == -np.inf).all()


def test_page_permutation_leaves_logits_bit_identical(oracle_mod):
    spec = qi.custom("perm", 3, 2, 4, 16, [70, 71, 5, 6, 40, 33], 96, seed=31)
    inp = qi.build_inputs(spec)
    base = oracle_mod.paged_mqa_logits(inp)
    perm = np.random.default_rng(8).permutation(inp.num_pages)
    new_kv = np.empty_like(inp.kv)
    new_kv[perm] = inp.kv  # page p moves to slot perm[p]
    new_bt = perm[inp.block_table].astype(np.int32)
    moved = oracle_mod.paged_mqa_logits(inp, kv=new_kv, block_table=new_bt)
    assert (moved.view(np.uint32) == base.view(np.uint32)).all()


def test_zero_padded_heads_add_exactly_nothing(oracle_mod):
    """SGLang #48649 Accuracy Tests: heads padded with zero queries add 0 after the ReLU."""
    spec = qi.custom("pad4", 2, 2, 4, 16, [37, 38, 20, 21], 48, seed=41)
    inp = qi.build_inputs(spec)
    base = oracle_mod.paged_mqa_logits(inp)
    spec16 = qi.custom("pad16", 2, 2, 16, 16, [37, 38, 20, 21], 48, seed=41)
    inp16 = qi.build_inputs(spec16)
    inp16.kv, inp16.block_table = inp.kv, inp.block_table
    q16 = np.zeros((4, 16, 128), np.uint16)
    q16[:, :4] = inp.q
    w16 = np.random.default_rng(2).random((4, 16)).astype(np.float32) * 100
    w16[:, :4] = inp.weights
    padded = oracle_mod.paged_mqa_logits(inp16, q=q16, weights=w16)
    assert (padded.view(np.uint32) == base.view(np.uint32)).all()


def test_mask_is_exact_negative_infinity_past_visible(oracle_mod):
    spec = qi.custom("mask", 2, 3, 4, 16, [0, 1, 16, 17, 63, 64], 64, seed=51)
    inp = qi.build_inputs(spec)
    got = oracle_mod.paged_mqa_logits(inp)
    for r, v in enumerate(spec.visible):
        assert np.isfinite(got[r, :v]).all()
        assert (got[r, v:].view(np.uint32) == 0xFF800000).all()


def test_poison_page_is_never_read_for_visible_columns(oracle_mod):
    spec = qi.custom("poison", 2, 1, 4, 16, [20, 3], 64, seed=61)
    inp = qi.build_inputs(spec)
    assert (inp.block_table[:, 2:] == inp.poison_page).all()
    got = oracle_mod.paged_mqa_logits(inp)
    assert not np.isnan(got).any()
    # a block table that points a visible column at the poison page shows NaN
    bt = inp.block_table.copy()
    bt[0, 0] = inp.poison_page
    bad = oracle_mod.paged_mqa_logits(inp, block_table=bt)
    assert np.isnan(bad[0, :16]).all()


def test_oracle_rejects_visible_beyond_block_table(oracle_mod):
    spec = qi.custom("cap", 1, 1, 4, 16, [16], 64, seed=71, max_pages=1)
    inp = qi.build_inputs(spec)
    with pytest.raises(ValueError):
        oracle_mod.paged_mqa_logits(inp, visible=np.array([17], np.int32))


def test_row_subset_matches_full_run(oracle_mod):
    spec = qi.custom("subset", 3, 2, 4, 16, [70, 71, 5, 6, 40, 33], 96, seed=31)
    inp = qi.build_inputs(spec)
    full = oracle_mod.paged_mqa_logits(inp, threads=1)
    sub = oracle_mod.paged_mqa_logits(inp, rows=[5, 0, 3], threads=3)
    assert (sub.view(np.uint32) == full[[5, 0, 3]].view(np.uint32)).all()


# --------------------------------------------------------------------------
# fp8 q (aiter #4221 "Motivation": q and keys as e4m3 codes, weights and key scales fp32)
# --------------------------------------------------------------------------


def _q8_spec(seed=3):
    return qi.custom("q8", 3, 2, 8, 64, [130, 131, 64, 65, 1, 0], 192, kv_dtype=qi.KV_FP8, seed=seed,
                     q_dtype=qi.Q_FP8)


def test_fp8_q_equals_bf16_q_of_the_same_values(oracle_mod):
    """Every finite e4m3 value is exact in bf16, so the fp8-q oracle must equal
    the (separately pinned) bf16-q oracle on the decoded values, bit for bit."""
    inp = qi.build_inputs(_q8_spec())
    got = oracle_mod.paged_mqa_logits(inp)
    as_bf16 = torch.from_numpy(inp.q).view(torch.float8_e4m3fn).to(torch.bfloat16)
    inp16 = qi.build_inputs(_q8_spec())
    inp16.spec.q_dtype = qi.Q_BF16
    inp16.q = as_bf16.view(torch.int16).numpy().view(np.uint16)
    ref = oracle_mod.paged_mqa_logits(inp16)
    assert (got.view(np.uint32) == ref.view(np.uint32)).all()


def test_fp8_q_matches_numpy_bruteforce(oracle_mod):
    inp = qi.build_inputs(_q8_spec(seed=4))
    assert _close_1ulp(oracle_mod.paged_mqa_logits(inp), brute.logits(inp))


# --------------------------------------------------------------------------
# Ragged live rows (aiter #4221 "Ragged next_n for confidence-scheduled
# verification": the leading next_n_lens[b] rows of a request are live, the
# rest stay -inf; the page's test plan edits the q of dead rows and expects
# no live logit to change)
# --------------------------------------------------------------------------


def _ragged_spec(kv_dtype, nn):
    vis = [90, 91, 92, 93, 17, 18, 19, 20, 60, 61, 62, 63, 33, 34, 35, 36]
    return qi.custom("ragged", 4, 4, 4, 16, vis, 96, kv_dtype=kv_dtype, seed=41, next_n_lens=nn)


@pytest.mark.parametrize("kv_dtype", [qi.KV_BF16, qi.KV_FP8], ids=["bf16", "fp8"])
def test_ragged_rows_match_bruteforce_with_dead_rows_neg_inf(oracle_mod, kv_dtype):
    nn = [0, 2, 4, 7]  # none live, two, all, more than the rows (all)
    inp = qi.build_inputs(_ragged_spec(kv_dtype, nn))
    got = oracle_mod.paged_mqa_logits(inp)
    # brute force over every row (dense, no live-row rule), then the rule by hand
    ref = brute.logits(inp)
    for b, n in enumerate(nn):
        for i in range(4):
            if i >= min(n, 4):
                ref[b * 4 + i, :] = -np.inf
    assert _close_1ulp(got, ref)
    assert np.isneginf(got[0:4]).all() and np.isneginf(got[6:8]).all()


def test_ragged_dead_row_inputs_change_nothing(oracle_mod):
    nn = [1, 3, 0, 2]
    inp = qi.build_inputs(_ragged_spec(qi.KV_BF16, nn))
    base = oracle_mod.paged_mqa_logits(inp)
    live = inp.spec.live_rows()
    q = inp.q.copy()
    w = inp.weights.copy()
    q[~live] = _int_bf16(np.full((int((~live).sum()), 4, 128), 3.0))
    w[~live] = np.nan
    vis = inp.spec.visible.copy()
    vis[~live] = 96
    got = oracle_mod.paged_mqa_logits(inp, q=q, weights=w, visible=vis)
    assert (got.view(np.uint32) == base.view(np.uint32)).all()


def test_ragged_full_counts_equal_the_uniform_call(oracle_mod):
    inp = qi.build_inputs(_ragged_spec(qi.KV_BF16, [4, 4, 9, 4]))
    got = oracle_mod.paged_mqa_logits(inp)
    plain = oracle_mod.paged_mqa_logits(inp, next_n_lens=None)
    assert (got.view(np.uint32) == plain.view(np.uint32)).all()


# --------------------------------------------------------------------------
# Top-k
# --------------------------------------------------------------------------


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_topk_matches_bruteforce_sort(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    vis = [0, 1, 7, 8, 9, 50, 200, 300]
    x = qi.random_logit_rows(rng, len(vis), 300, vis, zero_frac=0.3)
    got = oracle_mod.select_topk(x, np.array(vis, np.int32), 8)
    assert (got == brute.topk(x, vis, 8)).all()


def test_topk_rows_with_at_most_k_visible_select_everything(oracle_mod):
    x = np.zeros((3, 10), np.float32)
    got = oracle_mod.select_topk(x, np.array([0, 3, 5], np.int32), 5)
    assert got.tolist() == [[-1] * 5, [0, 1, 2, -1, -1], [0, 1, 2, 3, 4]]


def test_topk_zero_ties_keep_the_lowest_columns(oracle_mod):
    x = np.zeros((1, 12), np.float32)
    x[0, [3, 9]] = 1.0
    got = oracle_mod.select_topk(x, np.array([12], np.int32), 5)
    assert got.tolist() == [[0, 1, 2, 3, 9]]


def test_topk_one_ulp_boundary_from_the_pages(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "topk_tie_1ulp.json")))
    hi = np.array([int(g["higher_bits"], 16)], np.uint32).view(np.float32)[0]
    lo = np.array([int(g["lower_bits"], 16)], np.uint32).view(np.float32)[0]
    assert np.nextafter(lo, np.float32(np.inf)) == hi  # the page's pair is 1 ulp apart
    rank = g["boundary_rank"]
    rng = np.random.default_rng(3)
    n = 2000
    row = (rng.random(n).astype(np.float32) * 0.5)  # all below both candidates
    above = rng.choice(n, rank - 2, replace=False)
    row[above] = 2.0 + rng.random(rank - 2).astype(np.float32)
    free = np.setdiff1d(np.arange(n), above)
    c_lo, c_hi = int(free[10]), int(free[-10])  # the larger value sits at the higher column
    row[c_lo], row[c_hi] = lo, hi
    k = rank - 1  # exactly one of the two fits
    sel = set(oracle_mod.select_topk(row[None], np.array([n], np.int32), k)[0].tolist())
    assert c_hi in sel and c_lo not in sel
    row[c_hi] = lo  # made exactly equal: the lower column wins the tie
    sel = set(oracle_mod.select_topk(row[None], np.array([n], np.int32), k)[0].tolist())
    assert c_lo in sel and c_hi not in sel


def test_topk_changes_under_last_ulp_flips_only_at_near_ties(oracle_mod):
    """SGLang #48649 test_decode_selection_equivalent: a 1-ulp change matters only at ties."""
    rng = np.random.default_rng(12)
    vis = [900] * 16
    x = qi.random_logit_rows(rng, 16, 900, vis, zero_frac=0.0)
    k = 100
    base = oracle_mod.select_topk(x, np.array(vis, np.int32), k)
    flip = rng.choice([-1, 1], size=x.shape).astype(np.float32)
    y = np.where(flip > 0, np.nextafter(x, np.float32(np.inf)), np.nextafter(x, np.float32(-np.inf)))
    y = y.astype(np.float32)
    pert = oracle_mod.select_topk(y, np.array(vis, np.int32), k)
    for r in range(16):
        srt = np.sort(x[r])[::-1]
        gap_ulps = abs(int(srt[k - 1].view(np.int32)) - int(srt[k].view(np.int32)))
        if gap_ulps > 2:
            assert set(base[r]) == set(pert[r])


# --------------------------------------------------------------------------
# Golden facts printed on the pages
# --------------------------------------------------------------------------


def test_fp8_block_flat_pool_sizes_from_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "fp8_block_flat_pool.json")))
    spec = qi.fp8_h64()
    assert spec.num_requests == g["batch"] and spec.visible.max() == g["kv_len"]
    assert spec.page_cols == g["kv_block"] and spec.head_dim == g["head_dim"]
    assert int(spec.pages_needed().sum()) == g["block_references"]
    block_bytes = spec.page_cols * (spec.head_dim + 4)
    assert round(g["block_references"] * block_bytes / 1e6) == g["needed_working_set_mb"]
    assert round(g["wrapped_pool_blocks"] * block_bytes / 1e6, 2) == g["wrapped_pool_mb"]
    assert spec.key_bytes_touched() == g["block_references"] * block_bytes


def test_workload_recipe_constants_from_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "workload_recipe.json")))
    assert g["max_model_len_tokens"] // g["compress_ratio"] == g["logits_width"]
    for name in ("single_row_decode", "mtp3_verify_p16", "mtp3_large_p64"):
        s = qi.WORKLOADS[name]()
        assert s.out_cols == g["logits_width"] and s.k == g["topk"]
        assert s.num_heads == g["num_heads"] and s.head_dim == g["head_dim"]
    m = qi.mtp3_verify(16)
    assert m.num_requests == g["decode_requests"] and m.num_rows == g["decode_rows"]
    assert m.rows_per_req * m.num_heads == g["rows_times_heads"]
    p = qi.prefill_chunk()
    assert p.num_rows == g["prefill_rows"]
    assert p.visible.max() == g["prefill_context"] // g["compress_ratio"]


def test_block_flat_layout_is_keys_then_scales():
    """aiter #4221, KVBlockSize>=1 commit: KVB fp8 key rows first, then KVB fp32 scales."""
    spec = qi.custom("layout", 1, 1, 4, 16, [16], 16, kv_dtype=qi.KV_FP8, seed=2)
    inp = qi.build_inputs(spec)
    assert inp.key_page_stride == 16 * (128 + 4) and inp.scale_offset == 16 * 128
    p = int(inp.block_table[0, 0])
    scales = inp.kv[p, 16 * 128:].view(np.float32)
    keys = brute.e4m3_to_f64(inp.kv[p, : 16 * 128].reshape(16, 128))
    amax = np.abs(keys).max(axis=1)
    # quantised with scale = amax/448: the largest code of each key is +-448
    assert (amax == 448.0).all() and (scales > 0).all()
