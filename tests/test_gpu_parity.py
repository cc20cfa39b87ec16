"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every case uses the seeded generator, a NaN-prefilled output buffer and a
NaN poison page behind every unused block-table entry.  Logits are compared
element by element (tolerances in qsa_testlib); the -inf mask is bit-exact;
top-k is bit-exact against the oracle's top-k of the same GPU logits, and
within tie tolerance against the oracle's own logits.
"""
import numpy as np
import pytest

import qsa_inputs as qi
from qsa_testlib import (assert_logits_match, assert_topk_strict, assert_topk_within_tie_tolerance,
                         exact_case, nan_filled)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_indexer_02_gb300 as qsa  # noqa: E402
from sparse_attention_indexer_02_gb300 import torch_api  # noqa: E402

VARIANTS = {"auto": qsa.VARIANT_AUTO, "rowcore": qsa.VARIANT_ROWCORE, "umma": qsa.VARIANT_UMMA,
            "lean": qsa.VARIANT_UMMA_LEAN}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qsa.load_library()
    yield
    qsa.force_variant(qsa.VARIANT_AUTO)


def desc_of(inp):
    s = inp.spec
    stride = inp.key_page_stride
    return qsa.make_desc(s.num_requests, s.rows_per_req, s.num_heads, s.page_cols, s.max_pages,
                         inp.num_pages, s.out_cols, stride, kv_dtype=s.kv_dtype,
                         scale_page_stride=stride if s.kv_dtype == qi.KV_FP8 else 0)


def supported(inp, variant):
    qsa.force_variant(variant)
    try:
        qsa.plan_variant(desc_of(inp), inp.spec.q_dtype)
        return True
    except qsa.QSAError as e:
        if e.status == qsa.QSA_ERR_UNSUPPORTED:
            return False
        raise
    finally:
        qsa.force_variant(qsa.VARIANT_AUTO)


def gpu_logits(inp, variant=qsa.VARIANT_AUTO, dev=None, stream=None):
    s = inp.spec
    d = dev if dev is not None else qi.device_tensors(inp)
    out = nan_filled((s.num_rows, s.out_cols), torch.float32, "cuda")
    qsa.force_variant(variant)
    try:
        torch_api.paged_mqa_logits(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"],
                                   page_cols=s.page_cols, out_cols=s.out_cols, kv_dtype=s.kv_dtype,
                                   scale_offset=inp.scale_offset, out=out, stream=stream,
                                   next_n_lens=d.get("next_n_lens"))
        ran = qsa.last_variant()
    finally:
        qsa.force_variant(qsa.VARIANT_AUTO)
    torch.cuda.synchronize()
    return out, ran, d


def gpu_topk(logits_t, visible_t, k, max_visible=0):
    idx = nan_filled((logits_t.shape[0], k), torch.int32, "cuda")
    torch_api.select_topk(logits_t, visible_t, k, out=idx, max_visible=max_visible)
    torch.cuda.synchronize()
    return idx.cpu().numpy()


# (name, B, rows/req, H, page_cols, visible list (cycled), out_cols, k)
SMALL = [
    ("grid_6_100_700_p64", 3, 1, 4, 64, [6, 100, 700], 704, 64),  # SGLang decode_grid_covers_every_group
    ("mtp4_multi_tile_ragged", 2, 4, 4, 16, [1000, 1001, 1002, 1003, 300, 301, 302, 303], 1100, 256),
    ("mtp4_p64", 3, 4, 4, 64, [517, 518, 518, 519, 64, 65, 65, 66, 129, 130, 130, 131], 576, 100),
    ("single_row_h4_p16", 5, 1, 4, 16, [33, 129, 0, 640, 257], 640, 32),
    ("single_row_h1", 2, 1, 1, 16, [200, 77], 256, 16),
    ("h2_rows3", 2, 3, 2, 16, [150, 151, 152, 40, 41, 42], 160, 20),
    ("h3_odd_page5", 2, 2, 3, 5, [61, 62, 13, 14], 70, 10),
    ("h8_rows2_p32", 2, 2, 8, 32, [300, 301, 129, 130], 320, 50),
    ("h16_rows4", 2, 4, 16, 16, [270, 271, 272, 273, 5, 6, 7, 8], 288, 64),
    ("h64_single_row", 2, 1, 64, 64, [400, 257], 448, 64),
    ("rows16_p64", 1, 16, 4, 64, list(range(300, 316)), 320, 128),
    ("rows64_prefill_like", 1, 80, 4, 64, [200 + i // 4 for i in range(80)], 256, 64),
    ("visible_full_and_empty", 3, 2, 4, 16, [96, 96, 0, 0, 95, 1], 96, 8),
    ("page128_single", 2, 2, 4, 128, [700, 701, 129, 128], 768, 100),
    # more than 256 rows: the schedule is built by the whole CTA
    ("rows300_one_request", 1, 300, 4, 64, [100 + i // 3 for i in range(300)], 256, 32),
    ("rows260_single_row_requests", 260, 1, 4, 16, [0, 17, 130, 255, 256], 288, 16),
]


def small_spec(case, kv_dtype, seed=123):
    name, B, rpr, H, pc, vis, oc, k = case
    R = B * rpr
    v = (vis * R)[:R]
    return qi.custom(name, B, rpr, H, pc, v, oc, k=k, kv_dtype=kv_dtype, seed=seed)


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("kv_dtype", [qi.KV_BF16, qi.KV_FP8], ids=["bf16", "fp8"])
@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes_match_oracle(oracle_mod, case, kv_dtype, variant):
    if kv_dtype == qi.KV_FP8 and (case[4] * 132) % 16:
        pytest.skip("a block-flat fp8 page of this size is not 16-byte aligned")
    inp = qi.build_inputs(small_spec(case, kv_dtype))
    if not supported(inp, VARIANTS[variant]):
        pytest.skip(f"{variant} does not serve this shape")
    out, ran, d = gpu_logits(inp, VARIANTS[variant])
    if variant != "auto":
        assert ran == VARIANTS[variant]
    g = out.cpu().numpy()
    ref = oracle_mod.paged_mqa_logits(inp)
    assert_logits_match(g, ref, kv_dtype, where=f"{case[0]}/{variant}")
    k = inp.spec.k
    idx = gpu_topk(out, d["visible"], k)
    assert_topk_strict(idx, oracle_mod.select_topk(g, inp.spec.visible, k), where=case[0])
    assert_topk_within_tie_tolerance(idx, ref, inp.spec.visible, k, kv_dtype, where=case[0])


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("kv_dtype", [qi.KV_BF16, qi.KV_FP8], ids=["bf16", "fp8"])
def test_exact_integer_inputs_are_bit_exact(oracle_mod, kv_dtype, variant):
    """Integer q/keys and power-of-two weights/scales: fp32 is exact in any order."""
    spec = qi.custom("exact_gpu", 2, 4, 4, 16, [300, 301, 302, 303, 17, 18, 19, 0], 320, kv_dtype=kv_dtype,
                     seed=4)
    inp, _, _, _ = exact_case(kv_dtype, spec)
    if not supported(inp, VARIANTS[variant]):
        pytest.skip(f"{variant} does not serve this shape")
    out, _, _ = gpu_logits(inp, VARIANTS[variant])
    ref = oracle_mod.paged_mqa_logits(inp)
    assert (out.cpu().numpy().view(np.uint32) == ref.view(np.uint32)).all()


def test_variants_agree_with_each_other(oracle_mod):
    inp = qi.build_inputs(small_spec(SMALL[1], qi.KV_BF16))
    a, _, d = gpu_logits(inp, qsa.VARIANT_ROWCORE)
    if not supported(inp, qsa.VARIANT_UMMA):
        pytest.skip("tcgen05 scorer does not serve this shape")
    b, _, _ = gpu_logits(inp, qsa.VARIANT_UMMA, dev=d)
    assert_logits_match(b.cpu().numpy(), a.cpu().numpy(), qi.KV_BF16, where="umma vs rowcore")


def test_repeat_calls_are_bit_identical():
    inp = qi.build_inputs(small_spec(SMALL[2], qi.KV_BF16))
    a, _, d = gpu_logits(inp)
    b, _, _ = gpu_logits(inp, dev=d)
    assert (a.cpu().numpy().view(np.uint32) == b.cpu().numpy().view(np.uint32)).all()
    ia = gpu_topk(a, d["visible"], 100)
    ib = gpu_topk(b, d["visible"], 100)
    assert (ia == ib).all()


def test_side_stream(oracle_mod):
    inp = qi.build_inputs(small_spec(SMALL[3], qi.KV_BF16))
    s = torch.cuda.Stream()
    d = qi.device_tensors(inp)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out, _, _ = gpu_logits(inp, dev=d, stream=s)
    assert_logits_match(out.cpu().numpy(), oracle_mod.paged_mqa_logits(inp), qi.KV_BF16)


def test_cuda_graph_capture_and_replay(oracle_mod):
    """vLLM #62589 Validation: capture, then replay with new queries and lengths written in place."""
    spec = small_spec(SMALL[1], qi.KV_BF16)
    inp = qi.build_inputs(spec)
    d = qi.device_tensors(inp)
    s = inp.spec
    out = torch.empty((s.num_rows, s.out_cols), dtype=torch.float32, device="cuda")
    idx = torch.empty((s.num_rows, s.k), dtype=torch.int32, device="cuda")

    def step():
        torch_api.paged_mqa_logits(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"],
                                   page_cols=s.page_cols, out_cols=s.out_cols, out=out)
        torch_api.select_topk(out, d["visible"], s.k, out=idx)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside capture (first-call setup)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    # new queries and shorter lengths, written in place
    rng = np.random.default_rng(99)
    new_q = qi._bf16_bits(rng.standard_normal(inp.q.shape, dtype=np.float32))
    new_vis = np.maximum(spec.visible - rng.integers(0, 200, size=spec.visible.shape), 0).astype(np.int32)
    d["q"].copy_(torch.from_numpy(new_q.view(np.int16)).view(torch.bfloat16))
    d["visible"].copy_(torch.from_numpy(new_vis))
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    inp.q = new_q
    ref = oracle_mod.paged_mqa_logits(inp, visible=new_vis)
    got = out.cpu().numpy()
    assert_logits_match(got, ref, qi.KV_BF16, where="graph replay")
    assert_topk_strict(idx.cpu().numpy(), oracle_mod.select_topk(got, new_vis, s.k))


PRECEDED = [SMALL[1], SMALL[3], SMALL[14]]


@pytest.mark.parametrize("form", ["two-call", "one-call"])
@pytest.mark.parametrize("case", PRECEDED + [None], ids=[c[0] for c in PRECEDED] + ["single_row_decode_full"])
def test_inputs_written_by_the_kernel_just_before(oracle_mod, case, form):
    """The scoring kernel may start while the kernel before it in the stream is
    still running and loads q, weights and keys only after that kernel has
    completed: values written by the kernels just before the call (here q * -2,
    weights * 0.5, then every key negated, the largest write last) are the ones
    scored, and the selection right after reads the logits just written.  The
    row metadata (visible counts, block table) is not written there, as the
    header's contract asks."""
    spec = qi.single_row_decode() if case is None else small_spec(case, qi.KV_BF16)
    inp = qi.build_inputs(spec)
    d = qi.device_tensors(inp)
    s = inp.spec
    stride = d["kv"].shape[1]
    sign = torch.zeros(stride, dtype=torch.uint8, device="cuda")
    sign[1::2] = 0x80  # high byte of every little-endian bf16 key element

    def one_call():
        return torch_api.paged_mqa_topk(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"], s.k,
                                        page_cols=s.page_cols, out_cols=s.out_cols,
                                        max_visible=int(s.visible.max()))

    if form == "one-call":
        one_call()  # its workspace is allocated (and zero-filled) here, not just before the call
    torch.cuda.synchronize()
    torch.mul(d["q"], -2.0, out=d["q"])
    torch.mul(d["weights"], 0.5, out=d["weights"])
    torch.bitwise_xor(d["kv"], sign, out=d["kv"])
    if form == "two-call":
        out = torch.empty((s.num_rows, s.out_cols), dtype=torch.float32, device="cuda")
        torch_api.paged_mqa_logits(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"],
                                   page_cols=s.page_cols, out_cols=s.out_cols, out=out)
        idx = torch_api.select_topk(out, d["visible"], s.k)
    else:
        out, idx = one_call()
    torch.cuda.synchronize()
    q_new = qi._bf16_bits((inp.q.astype(np.uint32) << 16).view(np.float32) * np.float32(-2.0))
    kv_new = inp.kv.copy()
    kv_new[:, 1::2] ^= np.uint8(0x80)
    ref = oracle_mod.paged_mqa_logits(inp, q=q_new, weights=inp.weights * np.float32(0.5), kv=kv_new)
    got = out.cpu().numpy()
    assert_logits_match(got, ref, qi.KV_BF16, where=f"{s.name} {form}")
    assert_topk_strict(idx.cpu().numpy(), oracle_mod.select_topk(got, s.visible, s.k), where=f"{s.name} {form}")


# --------------------------------------------------------------------------
# fp8 q x fp8 keys (qsa_paged_mqa_logits_ex)
# --------------------------------------------------------------------------

Q8_CASES = [c for c in SMALL if (c[4] * 132) % 16 == 0]


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("case", Q8_CASES, ids=[c[0] for c in Q8_CASES])
def test_fp8_q_small_shapes_match_oracle(oracle_mod, case, variant):
    name, B, rpr, H, pc, vis, oc, k = case
    R = B * rpr
    spec = qi.custom(name, B, rpr, H, pc, (vis * R)[:R], oc, k=k, kv_dtype=qi.KV_FP8, seed=321,
                     q_dtype=qi.Q_FP8)
    inp = qi.build_inputs(spec)
    if not supported(inp, VARIANTS[variant]):
        pytest.skip(f"{variant} does not serve this shape")
    out, ran, d = gpu_logits(inp, VARIANTS[variant])
    if variant != "auto":
        assert ran == VARIANTS[variant]
    g = out.cpu().numpy()
    ref = oracle_mod.paged_mqa_logits(inp)
    assert_logits_match(g, ref, qi.KV_FP8, where=f"q8 {name}/{variant}")
    idx = gpu_topk(out, d["visible"], k)
    assert_topk_strict(idx, oracle_mod.select_topk(g, spec.visible, k), where=name)


@pytest.mark.parametrize("variant", ["rowcore", "umma", "lean"])
def test_fp8_q_exact_integer_case_is_bit_exact(oracle_mod, variant):
    """q and keys in {-3..3}, power-of-two scales and weights: exact in fp32."""
    spec = qi.custom("exact_q8", 2, 4, 4, 16, [300, 301, 302, 303, 17, 18, 19, 0], 320,
                     kv_dtype=qi.KV_FP8, seed=3, q_dtype=qi.Q_FP8)
    inp, qv, _, _ = exact_case(qi.KV_FP8, spec)
    inp.q = qi._e4m3_codes(qv.astype(np.float32))
    out, ran, _ = gpu_logits(inp, VARIANTS[variant])
    assert ran == VARIANTS[variant]
    ref = oracle_mod.paged_mqa_logits(inp)
    assert (out.cpu().numpy().view(np.uint32) == ref.view(np.uint32)).all()


# --------------------------------------------------------------------------
# Ragged live rows (qsa_paged_mqa_logits_ragged)
# --------------------------------------------------------------------------

RAGGED = [
    # (name, B, rows/req, H, page_cols, visible (cycled), out_cols, next_n_lens)
    ("nn8_h4_p16", 5, 8, 4, 16, [700 + i for i in range(8)], 768, [1, 8, 0, 3, 11]),
    ("nn4_h32_p64", 3, 4, 32, 64, [300, 301, 302, 303, 129, 130, 131, 132], 320, [2, 4, 1]),
    ("nn2_h64_p64", 4, 2, 64, 64, [200, 201], 256, [1, 2, 0, 1]),
    ("nn3_h3_page5", 2, 3, 3, 5, [41, 42, 43], 48, [2, 1]),  # CUDA-core scorer only
]


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("kv_dtype,q_dtype", [(qi.KV_BF16, qi.Q_BF16), (qi.KV_FP8, qi.Q_BF16),
                                             (qi.KV_FP8, qi.Q_FP8)], ids=["bf16", "fp8", "fp8q"])
@pytest.mark.parametrize("case", RAGGED, ids=[c[0] for c in RAGGED])
def test_ragged_rows_match_oracle(oracle_mod, case, kv_dtype, q_dtype, variant):
    name, B, rpr, H, pc, vis, oc, nn = case
    if kv_dtype == qi.KV_FP8 and (pc * 132) % 16:
        pytest.skip("a block-flat fp8 page of this size is not 16-byte aligned")
    R = B * rpr
    spec = qi.custom(name, B, rpr, H, pc, (vis * R)[:R], oc, k=32, kv_dtype=kv_dtype, seed=77,
                     next_n_lens=nn, q_dtype=q_dtype)
    inp = qi.build_inputs(spec)
    if not supported(inp, VARIANTS[variant]):
        pytest.skip(f"{variant} does not serve this shape")
    out, ran, d = gpu_logits(inp, VARIANTS[variant])
    g = out.cpu().numpy()
    assert_logits_match(g, oracle_mod.paged_mqa_logits(inp), kv_dtype, where=f"{name}/{variant}")
    dead = ~spec.live_rows()
    assert (g[dead].view(np.uint32) == 0xFF800000).all()
    # the top-k of the live visible counts: dead rows select nothing
    idx = gpu_topk(out, d["visible_live"], 32)
    assert_topk_strict(idx, oracle_mod.select_topk(g, spec.live_visible(), 32), where=name)


def test_ragged_dead_row_inputs_change_nothing():
    """aiter #4221 "Test plan": editing the q of a request's rows past its live count
    leaves every live logit as it was."""
    spec = qi.custom("dead", 4, 8, 4, 16, [500 + i for i in range(8)] * 4, 512, kv_dtype=qi.KV_BF16,
                     seed=5, next_n_lens=[3, 8, 1, 5])
    inp = qi.build_inputs(spec)
    base, _, d = gpu_logits(inp)
    dead = torch.from_numpy(~spec.live_rows()).cuda()
    d["q"][dead] = 7.0
    d["weights"][dead] = float("nan")
    got, _, _ = gpu_logits(inp, dev=d)
    assert torch.equal(got.view(torch.int32), base.view(torch.int32))


def test_fp8_q_graph_replay_with_new_q(oracle_mod):
    spec = qi.custom("q8_graph", 2, 4, 32, 64, [300, 301, 302, 303] * 2, 320, kv_dtype=qi.KV_FP8, seed=19,
                     q_dtype=qi.Q_FP8)
    inp = qi.build_inputs(spec)
    d = qi.device_tensors(inp)
    out = torch.empty((spec.num_rows, spec.out_cols), dtype=torch.float32, device="cuda")

    def call():
        torch_api.paged_mqa_logits(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"],
                                   page_cols=spec.page_cols, out_cols=spec.out_cols, kv_dtype=spec.kv_dtype,
                                   scale_offset=inp.scale_offset, out=out)

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    rng = np.random.default_rng(4)
    for _ in range(2):
        inp.q = qi._e4m3_codes(rng.standard_normal(inp.q.shape, dtype=np.float32))
        d["q"].copy_(torch.from_numpy(inp.q).view(torch.float8_e4m3fn))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_logits_match(out.cpu().numpy(), oracle_mod.paged_mqa_logits(inp), qi.KV_FP8, where="q8 graph")


def test_ragged_counts_rewritten_between_graph_replays(oracle_mod):
    spec = qi.custom("ragged_graph", 3, 4, 4, 16, [300, 301, 302, 303] * 3, 320, seed=9,
                     next_n_lens=[4, 4, 4])
    inp = qi.build_inputs(spec)
    d = qi.device_tensors(inp)
    out = torch.empty((spec.num_rows, spec.out_cols), dtype=torch.float32, device="cuda")

    def call():
        torch_api.paged_mqa_logits(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"],
                                   page_cols=spec.page_cols, out_cols=spec.out_cols, out=out,
                                   next_n_lens=d["next_n_lens"])

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for nn in ([1, 2, 3], [0, 4, 2]):
        d["next_n_lens"].copy_(torch.tensor(nn, dtype=torch.int32))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_mod.paged_mqa_logits(inp, next_n_lens=np.array(nn, np.int32))
        assert_logits_match(out.cpu().numpy(), ref, qi.KV_BF16, where=f"graph {nn}")


# --------------------------------------------------------------------------
# Top-k kernel on its own
# --------------------------------------------------------------------------


def _topk_case(rows, width, vis, k, zero_frac=0.06, seed=0):
    rng = np.random.default_rng(seed)
    x = qi.random_logit_rows(rng, rows, width, vis, zero_frac)
    return x


@pytest.mark.parametrize("k", [1, 7, 256, 2048])
def test_topk_edge_rows(oracle_mod, k):
    vis = [0, 1, k - 1 if k > 1 else 0, k, k + 1, 3 * k + 5, 4000, 9000]
    width = max(vis) + 3
    x = _topk_case(len(vis), width, vis, k, zero_frac=0.2, seed=k)
    # a row of all-equal values and a row mixing -0.0 and +0.0
    x[6, :4000] = 1.25
    x[7, :9000:2] = -0.0
    x[7, 1:9000:2] = 0.0
    xt = torch.from_numpy(x).cuda()
    vt = torch.tensor(vis, dtype=torch.int32, device="cuda")
    idx = gpu_topk(xt, vt, k)
    assert_topk_strict(idx, oracle_mod.select_topk(x, np.array(vis, np.int32), k))
    for r, n in enumerate(vis):
        if n <= k:
            assert idx[r].tolist() == list(range(n)) + [-1] * (k - n)


def test_topk_rows_longer_than_the_shared_memory_cache(oracle_mod):
    vis = [65537, 60000, 49153, 49152]
    x = _topk_case(4, 65600, vis, 2048, seed=5)
    xt = torch.from_numpy(x).cuda()
    vt = torch.tensor(vis, dtype=torch.int32, device="cuda")
    idx = gpu_topk(xt, vt, 2048)
    assert_topk_strict(idx, oracle_mod.select_topk(x, np.array(vis, np.int32), 2048))


@pytest.mark.parametrize("rows", [3, 40, 100, 200])
def test_topk_cluster_sizes_and_single_cta_path(oracle_mod, rows):
    """Few rows are split over clusters of 8 or 2 CTAs (3 and 40 rows), many
    rows use one CTA a row (100 and 200); rows of 4003..40000 columns, the
    stride not a multiple of 4 (plain loads fill the cache)."""
    rng = np.random.default_rng(rows)
    vis = rng.integers(2000, 40000, size=rows).astype(np.int32)
    vis[:3] = [40000, 12288, 12289]
    x = qi.random_logit_rows(rng, rows, 40003, vis, zero_frac=0.1)
    xt = torch.from_numpy(x).cuda()
    for k in (1000, 2048):
        idx = gpu_topk(xt, torch.from_numpy(vis).cuda(), k)
        assert_topk_strict(idx, oracle_mod.select_topk(x, vis, k))


@pytest.mark.parametrize("rows", [1, 3, 40])
def test_topk_short_rows(oracle_mod, rows):
    """Rows of at most 12288 columns with a 16-byte aligned stride (bulk copies
    fill the cache), over clusters of 8 (1 and 3 rows) and 2 CTAs (40 rows)."""
    rng = np.random.default_rng(rows + 11)
    vis = rng.integers(2049, 12288, size=rows).astype(np.int32)
    vis[0] = 12288
    x = qi.random_logit_rows(rng, rows, 12288, vis, zero_frac=0.1)
    xt = torch.from_numpy(x).cuda()
    idx = gpu_topk(xt, torch.from_numpy(vis).cuda(), 2048)
    assert_topk_strict(idx, oracle_mod.select_topk(x, vis, 2048))


def test_topk_many_long_rows_read_from_global_memory(oracle_mod):
    """More rows than the cluster path takes, each longer than the shared-memory cache."""
    rows = 160
    rng = np.random.default_rng(77)
    vis = np.full(rows, 50000, np.int32)
    vis[::7] = 49153
    x = qi.random_logit_rows(rng, rows, 50004, vis, zero_frac=0.05)
    xt = torch.from_numpy(x).cuda()
    idx = gpu_topk(xt, torch.from_numpy(vis).cuda(), 2048)
    assert_topk_strict(idx, oracle_mod.select_topk(x, vis, 2048))


@pytest.mark.parametrize("rows,n", [(200, 30000), (2, 65536)])
def test_topk_candidate_list_overflow(oracle_mod, rows, n):
    """Rows whose first-digit bin holds more keys than a CTA's candidate list
    (all values equal): the CTAs fall back to scanning their whole segment; the
    lowest columns win the tie (one CTA a row for 200 rows, clusters of 8 for 2)."""
    x = np.full((rows, n + 4), 1.5, np.float32)
    x[:, n:] = 9.0  # past the visible count: never selected
    x[1, 100] = 2.0  # one larger value in row 1
    vis = np.full(rows, n, np.int32)
    xt = torch.from_numpy(x).cuda()
    idx = gpu_topk(xt, torch.from_numpy(vis).cuda(), 2048)
    assert_topk_strict(idx, oracle_mod.select_topk(x, vis, 2048))
    assert idx[0].tolist() == list(range(2048))


def test_topk_threshold_ties_take_the_lowest_columns(oracle_mod):
    # 3000 exact zeros around the k-th place: the lowest-column zeros must win
    x = np.zeros((2, 5000), np.float32)
    x[:, 4000:] = 2.0
    x[1, ::7] = 0.5
    vis = np.array([5000, 4999], np.int32)
    xt = torch.from_numpy(x).cuda()
    idx = gpu_topk(xt, torch.from_numpy(vis).cuda(), 1500)
    assert_topk_strict(idx, oracle_mod.select_topk(x, vis, 1500))


@pytest.mark.parametrize("n", [4096, 8192, 32768])
def test_topk_threshold_bin_taken_whole(oracle_mod, n):
    """Row 0: exactly k keys fall in one first-digit bin ([1, 1.25): sign, exponent
    and two mantissa bits), every other key is lower, and one of them is the float
    just below 1.0 (the bin's lowest key minus one): the selection may stop after
    the first digit and must take exactly the bin.  Row 1: the bin holds one key
    more than wanted, so the later digits decide."""
    k = 2048
    rng = np.random.default_rng(n)
    x = np.empty((2, n), np.float32)
    below = np.nextafter(np.float32(1.0), np.float32(0.0))
    top = np.nextafter(np.float32(1.25), np.float32(0.0))
    for r in range(2):
        hi = k + r
        vals = np.concatenate([np.minimum(rng.uniform(1.0, 1.25, hi).astype(np.float32), top),
                               rng.uniform(0.25, 0.3, n - hi).astype(np.float32)])
        vals[hi] = below
        x[r] = vals[rng.permutation(n)]
    vis = np.array([n, n], np.int32)
    idx = gpu_topk(torch.from_numpy(x).cuda(), torch.from_numpy(vis).cuda(), k)
    assert_topk_strict(idx, oracle_mod.select_topk(x, vis, k))
    assert sorted(idx[0].tolist()) == np.flatnonzero(x[0] >= 1.0).tolist()


KEY_SPANS = [1, 2, 2047, 2048, 2049, 4095, (1 << 22) - 1, 1 << 22, (1 << 22) + 1, (1 << 24) + 3, None]


def key_span_rows(rng, rows, n):
    """Rows of n columns whose order-preserving keys cover exactly KEY_SPANS[r]
    (row r cycles through them): float32 bit patterns 1.0 + offsets in
    [0, span] with both ends present, so small spans hold many equal values;
    None is a row of both signs from -1e30 to 1e30 (a span near 2^32)."""
    x = np.empty((rows, n), np.float32)
    for r in range(rows):
        span = KEY_SPANS[r % len(KEY_SPANS)]
        if span is None:
            v = rng.uniform(-1e30, 1e30, n).astype(np.float32)
            v[rng.integers(n)], v[rng.integers(n)] = np.float32(-1e30), np.float32(1e30)
        else:
            off = rng.integers(0, span + 1, n, dtype=np.int64)
            off[rng.integers(n)], off[rng.integers(n)] = 0, span
            v = (np.uint32(0x3F800000) + off.astype(np.uint32)).view(np.float32)
        x[r] = v
    return x


@pytest.mark.parametrize("rows,n", [(11, 8192), (11, 5001), (200, 22528)])
def test_topk_key_spans_at_the_digit_boundaries(oracle_mod, rows, n):
    """One CTA a row takes its digits from the keys' offsets above the smallest
    one, as many bits as the span needs: spans below 2048 end after one digit,
    below 2^22 after two, the rest take three; the rows put the span on each
    side of those boundaries (the register path for 8192 and 5001 columns, the
    sampled pivot's candidate select for 22528)."""
    rng = np.random.default_rng(n)
    x = key_span_rows(rng, rows, n)
    vis = np.full(rows, n, np.int32)
    for k in (2048, 1):
        idx = gpu_topk(torch.from_numpy(x).cuda(), torch.from_numpy(vis).cuda(), k)
        assert_topk_strict(idx, oracle_mod.select_topk(x, vis, k))


# --------------------------------------------------------------------------
# qsa_select_topk_bounded: the caller's bound clamps the visible counts; a
# bound of at most 8192 columns takes the register form (1024 threads)
# --------------------------------------------------------------------------


@pytest.mark.parametrize("k", [1, 7, 256, 2048])
def test_bounded_topk_register_form_edge_rows(oracle_mod, k):
    """Rows of 0, 1, k - 1, k, k + 1, 3k + 5 and 8192 visible columns, an
    all-equal row and a row of -0.0 / +0.0, in a 65,603-column stride (as the
    decode logits, far wider than the bound) under the bound 8192."""
    vis = [0, 1, max(k - 1, 0), k, k + 1, 3 * k + 5, 8192, 8192, 8192]
    width = 65603
    x = _topk_case(len(vis), width, vis, k, zero_frac=0.2, seed=k + 1)
    x[7, :8192] = 1.25
    x[8, :8192:2] = -0.0
    x[8, 1:8192:2] = 0.0
    vis_np = np.array(vis, np.int32)
    idx = gpu_topk(torch.from_numpy(x).cuda(), torch.from_numpy(vis_np).cuda(), k, max_visible=8192)
    assert_topk_strict(idx, oracle_mod.select_topk(x, vis_np, k))


@pytest.mark.parametrize("rows,width,bound", [(16, 65600, 8192), (40, 8192, 8192), (320, 4099, 5000),
                                              (3, 8191, 8191), (5, 1000, 700)])
def test_bounded_topk_rows_within_the_bound(oracle_mod, rows, width, bound):
    """Random rows no longer than the bound (counts past the stride are
    clamped to it): the widths are not multiples of 4 except two (plain and
    vector loads); 320 rows is more than two an SM (152 SMs), which takes the
    general form."""
    rng = np.random.default_rng(rows * 7 + width)
    vis = rng.integers(0, min(bound, width) + 1, size=rows).astype(np.int32)
    vis[0] = min(bound, width)
    if width < bound:
        vis[-1] = bound  # past the stride
    x = qi.random_logit_rows(rng, rows, width, np.minimum(vis, width), zero_frac=0.1)
    k = 2048 if bound > 2048 else 256
    idx = gpu_topk(torch.from_numpy(x).cuda(), torch.from_numpy(vis).cuda(), k, max_visible=bound)
    assert_topk_strict(idx, oracle_mod.select_topk(x, np.minimum(vis, width).astype(np.int32), k))


@pytest.mark.parametrize("rows,width", [(16, 40003), (40, 12288)])
def test_bounded_topk_rows_past_a_wrong_bound(oracle_mod, rows, width):
    """A bound of 8192 columns that some rows exceed (up to 40,000 columns):
    the register form's launch still selects them exactly (candidate
    compaction from global memory).  Continuous values, then every row's
    first-digit bin crowded (all values equal but a few)."""
    rng = np.random.default_rng(rows + width)
    vis = rng.integers(2000, width + 1, size=rows).astype(np.int32)
    vis[0], vis[1], vis[2] = width, 8192, 8193
    base = qi.random_logit_rows(rng, rows, width, vis, zero_frac=0.05)
    flat = np.where(np.isfinite(base), np.float32(1.5), base)
    flat[:, 5::997] = np.where(np.isfinite(flat[:, 5::997]), np.float32(2.0), flat[:, 5::997])
    for x in (base, flat):
        for k in (2048, 100):
            idx = gpu_topk(torch.from_numpy(x).cuda(), torch.from_numpy(vis).cuda(), k, max_visible=8192)
            assert_topk_strict(idx, oracle_mod.select_topk(x, vis, k))
    assert qsa.device_status() == 0


def test_bounded_topk_cluster_launch_with_a_wrong_bound(oracle_mod):
    """Three rows of a 70,003-column stride under a bound of 16,000: a cluster
    launch of 8 CTAs whose plan, going by the bound, has no segment cache.
    Row 0 (70,003 columns, past the bound) takes candidate compaction from
    global memory, row 1 (12,000) is selected by the first CTA alone (the
    sampled pivot), row 2 (30,000) by the register path in every CTA.
    Continuous values, then every row's first-digit bin crowded."""
    rng = np.random.default_rng(70003)
    width = 70003
    vis = np.array([70003, 12000, 30000], np.int32)
    base = qi.random_logit_rows(rng, 3, width, vis, zero_frac=0.05)
    flat = np.where(np.isfinite(base), np.float32(1.5), base)
    flat[:, 3::1001] = np.where(np.isfinite(flat[:, 3::1001]), np.float32(2.0), flat[:, 3::1001])
    for x in (base, flat):
        for k in (2048, 300):
            idx = gpu_topk(torch.from_numpy(x).cuda(), torch.from_numpy(vis).cuda(), k, max_visible=16000)
            assert_topk_strict(idx, oracle_mod.select_topk(x, vis, k))
    assert qsa.device_status() == 0


def test_bounded_topk_key_spans_and_unaligned_rows(oracle_mod):
    """The key-span rows under a bound of 8192 columns, with the logits
    starting one float past a 16-byte boundary and a stride of 8195 floats
    (every row misaligned: plain loads)."""
    rng = np.random.default_rng(44)
    rows, n = 11, 8192
    x = key_span_rows(rng, rows, n)
    buf = np.zeros((rows, 8195), np.float32)
    buf[:, :n] = x
    flat = torch.from_numpy(np.concatenate([np.zeros(1, np.float32), buf.ravel()])).cuda()
    xt = flat[1:].view(rows, 8195)
    vis = np.full(rows, n, np.int32)
    for k in (2048, 1):
        idx = gpu_topk(xt, torch.from_numpy(vis).cuda(), k, max_visible=n)
        assert_topk_strict(idx, oracle_mod.select_topk(buf, vis, k))


def test_bounded_topk_gives_the_plain_calls_indices_for_any_bound():
    """The bound only chooses the launch: none (0, negative), at or above the
    stride, above 8192 (the general form) or below the rows (the register
    form) all give exactly the plain call's indices."""
    rng = np.random.default_rng(9)
    rows, width = 16, 20000
    vis = rng.integers(1000, width, size=rows).astype(np.int32)
    x = qi.random_logit_rows(rng, rows, width, vis, zero_frac=0.05)
    xt, vt = torch.from_numpy(x).cuda(), torch.from_numpy(vis).cuda()
    ref = gpu_topk(xt, vt, 2048)
    for bound in (0, -3, width, width + 100, 12000, 8192, 3000):
        assert (gpu_topk(xt, vt, 2048, max_visible=bound) == ref).all(), bound
    assert qsa.device_status() == 0


@pytest.mark.parametrize("rows,n", [(4, 16000), (200, 22528), (160, 65537), (400, 22528)])
def test_topk_long_rows_sampled_pivot(oracle_mod, rows, n):
    """Rows one CTA selects alone and longer than its keys-in-registers limit
    (4 rows of 16000 columns, 200 of 22528, 160 of 65537 - sampled more
    sparsely - and 400 of 22528, more rows than twice the SMs: the narrow
    256-thread form): a sample of every 8th block of 128 columns sets a threshold, the
    exact selection runs on the candidates above it.  Continuous values, then every sampled block raised far above
    the rest (the sample's threshold lets fewer than k columns through, so the
    full path must take over), then exact zeros spanning the k-th place (the
    lowest zero columns win)."""
    k = 2048
    rng = np.random.default_rng(rows)
    vis = np.full(rows, n, np.int32)
    vis[1] = n - 123
    base = qi.random_logit_rows(rng, rows, n, vis, zero_frac=0.0)
    high = base.copy()
    blk = np.arange(n) // 128
    high[:, blk % 8 == 0] += np.float32(10.0)
    ties = np.where(np.isfinite(base), np.float32(-1.0), base)
    for r in range(rows):
        cols = rng.permutation(int(vis[r]))
        ties[r, cols[:1500]] = 2.0
        ties[r, cols[1500:4500]] = 0.0
    for x in (base, high, ties):
        idx = gpu_topk(torch.from_numpy(x).cuda(), torch.from_numpy(vis).cuda(), k)
        assert_topk_strict(idx, oracle_mod.select_topk(x, vis, k))


def test_topk_more_rows_than_resident_ctas(oracle_mod):
    """More rows than the device holds CTAs at once (the narrow 256-thread form,
    whose register path ends at 4096 columns), mixing every path a row can
    take: at most k columns, keys in registers, the sampled pivot, and its
    fallback (all values equal)."""
    rows, width, k = 700, 12000, 1024
    rng = np.random.default_rng(700)
    vis = rng.integers(9000, width + 1, size=rows).astype(np.int32)
    vis[::7] = rng.integers(0, k + 1, size=vis[::7].shape)      # fit in k
    vis[3::7] = rng.integers(k + 1, 8192, size=vis[3::7].shape)  # registers
    x = qi.random_logit_rows(rng, rows, width, vis, zero_frac=0.05)
    x[5::50, :] = np.where(np.isfinite(x[5::50, :]), np.float32(0.75), x[5::50, :])  # all equal
    idx = gpu_topk(torch.from_numpy(x).cuda(), torch.from_numpy(vis).cuda(), k)
    assert_topk_strict(idx, oracle_mod.select_topk(x, vis, k))


def test_topk_visible_beyond_stride_is_clamped():
    x = np.arange(40, dtype=np.float32).reshape(2, 20)
    xt = torch.from_numpy(x).cuda()
    vt = torch.tensor([1000, -5], dtype=torch.int32, device="cuda")
    idx = gpu_topk(xt, vt, 4)
    assert sorted(idx[0].tolist()) == [16, 17, 18, 19]
    assert idx[1].tolist() == [-1, -1, -1, -1]


# --------------------------------------------------------------------------
# Full-size workloads in the bench launch configuration (auto dispatch),
# checked on sampled rows (logits) and on every row (top-k vs oracle top-k
# of the same logits).
# --------------------------------------------------------------------------

FULL = ["tiny_mtp", "single_row_decode", "mtp3_verify_p16", "mtp3_verify_p64", "fp8_h64", "prefill_chunk",
        "mtp3_large_p16", "mtp3_large_p64", "ragged_nn8", "fp8q_h64"]


def scorer_group_rows(spec):
    """Rows the tcgen05 scorer stacks into one MMA (rows x heads <= 256, within
    a request): the sample takes both edge rows of several such groups."""
    return min(max(1, 256 // spec.num_heads), spec.rows_per_req)


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled(oracle_mod, name):
    spec = qi.WORKLOADS[name]()
    inp = qi.build_inputs(spec)
    out, ran, d = gpu_logits(inp)
    # first, last and random rows, and the edge rows of 8 row groups spread
    # over the batch (the last group included): 63/64, 127/128, ... for the
    # prefill chunk's 64-row groups, a request's first and last rows for MTP
    rows = qi.gather_rows_for(spec, 6 if spec.num_heads > 4 else 12, np.random.default_rng(1),
                              group_rows=scorer_group_rows(spec), edge_groups=8)
    ref = oracle_mod.paged_mqa_logits(inp, rows=rows)
    sub = out[torch.tensor(rows, device="cuda")].cpu().numpy()
    assert_logits_match(sub, ref, spec.kv_dtype, where=f"{name} rows {rows}")
    idx_t = nan_filled((spec.num_rows, spec.k), torch.int32, "cuda")
    vis_live = d.get("visible_live", d["visible"])  # ragged: dead rows select nothing
    # the bench's call: the batch's longest visible count as the host bound
    torch_api.select_topk(out, vis_live, spec.k, out=idx_t, max_visible=int(spec.live_visible().max()))
    torch.cuda.synchronize()
    idx = idx_t.cpu().numpy()
    # strict top-k on a bounded set of rows (the oracle sorts each row)
    trows = rows if spec.num_rows > 512 else list(range(spec.num_rows))
    g_rows = out[torch.tensor(trows, device="cuda")].cpu().numpy()
    assert_topk_strict(idx[trows], oracle_mod.select_topk(g_rows, spec.live_visible()[trows], spec.k), where=name)
    assert_topk_within_tie_tolerance(idx[rows], ref, spec.live_visible()[rows], spec.k, spec.kv_dtype, where=name)
    # every masked entry of every row, bit-exact
    vis_t = vis_live.long()
    cols = torch.arange(spec.out_cols, device="cuda")
    masked = cols[None, :] >= vis_t[:, None]
    bits = out.view(torch.int32)
    assert bool((bits[masked] == np.int32(np.uint32(0xFF800000).view(np.int32))).all())
    assert not bool(torch.isnan(out[~masked]).any())


def test_no_kernel_gave_up_on_a_barrier():
    """Every bounded wait above completed: the device fault word is still clear."""
    assert qsa.device_status(clear=True) == 0


@pytest.mark.parametrize("variant", ["rowcore", "umma"])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_fp8_every_finite_code_including_subnormals(oracle_mod, variant, sign):
    """Column c holds code c in element 0 (all other elements zero); q = +-e0, w = 1,
    scale = 2: the logit is relu(+-2 * e4m3(c)), exact in fp32 - so every code,
    subnormals included, must decode exactly (no flush to zero)."""
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
    n = len(codes)
    spec = qi.custom("fp8_codes", 1, 1, 1, 16, [n], 256, k=8, kv_dtype=qi.KV_FP8, seed=3)
    inp = qi.build_inputs(spec)
    D, pc = 128, 16
    inp.kv[:, : pc * D] = 0
    inp.kv[:, pc * D:] = np.full((inp.num_pages, pc), 2.0, np.float32).view(np.uint8).reshape(inp.num_pages, -1)
    for ci, code in enumerate(codes):
        page = int(inp.block_table[0, ci // pc])
        inp.kv[page, (ci % pc) * D] = code
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = sign
    inp.q = qi._bf16_bits(q)
    inp.weights = np.ones((1, 1), np.float32)
    if not supported(inp, VARIANTS[variant]):
        pytest.skip(f"{variant} does not serve this shape")
    out, _, _ = gpu_logits(inp, VARIANTS[variant])
    ref = oracle_mod.paged_mqa_logits(inp)
    assert (out.cpu().numpy().view(np.uint32) == ref.view(np.uint32)).all()
