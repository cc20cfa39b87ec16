"""GPU parity of qsa_paged_mqa_topk, scoring with the per-row selection in the
same call, against the CPU oracle.

The call is defined as the scoring call followed by the top-k of every row
over its scored visible count (live rows; dead rows select nothing).  Logits
are compared with the scoring tolerances, selections bit-exactly against the
oracle's top-k of the same GPU logits, and within tie tolerance against the
oracle's own logits.  The fused kernel (decode-sized calls) and the two-launch
form (long rows by the caller's bound, more than 256 rows) are both covered,
and the workspace must read zero after every call.
"""
import numpy as np
import pytest

import qsa_inputs as qi
from qsa_testlib import assert_logits_match, assert_topk_strict, assert_topk_within_tie_tolerance, nan_filled

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_indexer_02_gb300 as qsa  # noqa: E402
from sparse_attention_indexer_02_gb300 import torch_api  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qsa.load_library()
    yield
    qsa.force_variant(qsa.VARIANT_AUTO)


@pytest.fixture(autouse=True)
def _fuse_every_shape():
    """The dispatch fuses single-row requests only; these tests cover the fused
    kernel on every shape it serves, so they force it (tests of the dispatch
    itself set AUTO)."""
    qsa.force_variant(qsa.VARIANT_UMMA_TOPK)
    yield
    qsa.force_variant(qsa.VARIANT_AUTO)


def scored_visible(spec):
    """n[r]: the row's visible count as scored (live rows, clamped to the row)."""
    cap = min(spec.out_cols, spec.max_pages * spec.page_cols)
    return np.clip(spec.live_visible(), 0, cap).astype(np.int32)


def run_fused(inp, k, max_visible=0, dev=None, workspace=None, stream=None):
    s = inp.spec
    d = dev if dev is not None else qi.device_tensors(inp)
    logits = nan_filled((s.num_rows, s.out_cols), torch.float32, "cuda")
    idx = nan_filled((s.num_rows, k), torch.int32, "cuda")
    torch_api.paged_mqa_topk(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"], k,
                             page_cols=s.page_cols, out_cols=s.out_cols, kv_dtype=s.kv_dtype,
                             scale_offset=inp.scale_offset, max_visible=max_visible, out_logits=logits,
                             out_idx=idx, workspace=workspace, stream=stream, next_n_lens=d.get("next_n_lens"))
    ran = qsa.last_variant()
    torch.cuda.synchronize()
    return logits, idx, ran, d


def check(oracle_mod, inp, logits, idx, k, where):
    s = inp.spec
    g = logits.cpu().numpy()
    ref = oracle_mod.paged_mqa_logits(inp)
    assert_logits_match(g, ref, s.kv_dtype, where=where)
    n = scored_visible(s)
    got = idx.cpu().numpy()
    assert_topk_strict(got, oracle_mod.select_topk(g, n, k), where=where)
    assert_topk_within_tie_tolerance(got, ref, n, k, s.kv_dtype, where=where)


def workspace_is_zero():
    torch.cuda.synchronize()
    return all(int(ws.abs().sum()) == 0 for ws in torch_api._workspaces.values())


# (name, B, rows/req, H, page_cols, visible list (cycled), out_cols, k)
CASES = [
    ("decode_h4_p16", 6, 1, 4, 16, [300, 1000, 2049, 5, 4096, 777], 4160, 256),
    ("decode_k2048_p64", 4, 1, 4, 64, [8192, 6000, 2048, 9000], 9024, 2048),
    ("mtp4_groups_helpers", 3, 4, 4, 64, [1500, 1501, 1502, 1503, 700, 701, 702, 703, 90, 91, 92, 93], 1536, 100),
    ("rows16_one_group", 1, 16, 4, 64, list(range(3000, 3016)), 3072, 512),
    ("h1_many_rows_per_group", 2, 40, 1, 16, [200 + i for i in range(40)], 256, 16),
    ("h16_rows4", 2, 4, 16, 16, [2700, 2701, 2702, 2703, 50, 51, 52, 53], 2720, 64),
    ("h64_single_row", 3, 1, 64, 64, [4000, 2570, 1], 4032, 1024),
    ("empty_groups", 3, 2, 4, 16, [960, 960, 0, 0, 950, 1], 960, 8),
    ("all_rows_fit_k", 2, 2, 4, 16, [30, 31, 32, 0], 64, 32),
    ("page128", 2, 2, 4, 128, [7000, 7001, 1290, 128], 7040, 1000),
    # more than 256 rows: the scoring call and the top-k launch
    ("rows260_two_launches", 260, 1, 4, 16, [0, 17, 130, 255, 256], 288, 16),
]


def case_spec(case, kv_dtype, q_dtype=qi.Q_BF16, seed=2024):
    name, B, rpr, H, pc, vis, oc, k = case
    R = B * rpr
    return qi.custom(name, B, rpr, H, pc, (vis * R)[:R], oc, k=k, kv_dtype=kv_dtype, seed=seed, q_dtype=q_dtype)


KINDS = [(qi.KV_BF16, qi.Q_BF16), (qi.KV_FP8, qi.Q_BF16), (qi.KV_FP8, qi.Q_FP8)]


@pytest.mark.parametrize("kv_dtype,q_dtype", KINDS, ids=["bf16", "fp8", "fp8q"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_matches_oracle(oracle_mod, case, kv_dtype, q_dtype):
    if kv_dtype == qi.KV_FP8 and (case[4] * 132) % 16:
        pytest.skip("a block-flat fp8 page of this size is not 16-byte aligned")
    inp = qi.build_inputs(case_spec(case, kv_dtype, q_dtype))
    k = case[7]
    logits, idx, ran, _ = run_fused(inp, k)
    expect = qsa.VARIANT_UMMA if inp.spec.num_rows > 256 else qsa.VARIANT_UMMA_TOPK
    assert ran == expect, (ran, expect)
    check(oracle_mod, inp, logits, idx, k, where=case[0])
    assert workspace_is_zero()


@pytest.mark.parametrize("max_visible", [1, 0, 20000])
def test_caller_bound_steers_dispatch_only(oracle_mod, max_visible):
    """A bound below the real counts still gives the defined result (the pages'
    single_row_decode flag: a wrong flag costs speed only)."""
    case = ("bound", 4, 1, 4, 64, [9000, 16000, 30000, 100], 30016, 2048)
    inp = qi.build_inputs(case_spec(case, qi.KV_BF16))
    logits, idx, ran, _ = run_fused(inp, 2048, max_visible=max_visible)
    # unknown (0) and large bounds leave these 30016-column rows to the top-k launch
    assert ran == (qsa.VARIANT_UMMA_TOPK if max_visible == 1 else qsa.VARIANT_UMMA_LEAN)
    check(oracle_mod, inp, logits, idx, 2048, where=f"bound {max_visible}")
    assert workspace_is_zero()


@pytest.mark.parametrize("vis,max_visible", [([9000, 16000, 30000, 100], 5000), ([8000, 100, 8192, 5000], 8192),
                                              ([9000, 16000, 30000, 100], 30016)])
def test_one_call_bound_chooses_the_topk_form_only(oracle_mod, vis, max_visible):
    """With the automatic dispatch the one call runs the scoring and top-k
    launches, and its bound picks the top-k form: the register form for a
    bound of at most 8192 columns, whether right or wrong (rows of up to 30,000
    columns under a bound of 5,000 are still selected exactly), the default
    form above it."""
    qsa.force_variant(qsa.VARIANT_AUTO)
    case = ("bound_form", 4, 1, 4, 64, vis, 30016, 2048)
    inp = qi.build_inputs(case_spec(case, qi.KV_BF16))
    logits, idx, ran, _ = run_fused(inp, 2048, max_visible=max_visible)
    assert ran == qsa.VARIANT_UMMA_LEAN
    check(oracle_mod, inp, logits, idx, 2048, where=f"bound {max_visible}")
    assert qsa.device_status() == 0


def test_fused_rows_longer_than_the_shared_memory_cache(oracle_mod):
    """Columns past the selection's cache are read back from L2 by the fused kernel."""
    for kv_dtype, q_dtype in KINDS:
        case = ("long", 2, 1, 4, 64, [60000, 45000], 60032, 2048)
        inp = qi.build_inputs(case_spec(case, kv_dtype, q_dtype, seed=5))
        logits, idx, ran, _ = run_fused(inp, 2048, max_visible=1)
        assert ran == qsa.VARIANT_UMMA_TOPK
        check(oracle_mod, inp, logits, idx, 2048, where=f"long kv{kv_dtype} q{q_dtype}")
    assert workspace_is_zero()


RAGGED = [
    ("nn8_h4_p16", 5, 8, 4, 16, [1700 + i for i in range(8)], 1728, [1, 8, 0, 3, 11]),
    ("nn4_h32_p64", 3, 4, 32, 64, [3000, 3001, 3002, 3003, 129, 130, 131, 132], 3008, [2, 4, 1]),
    ("nn2_h64_p64", 4, 2, 64, 64, [200, 201], 256, [1, 2, 0, 1]),
]


@pytest.mark.parametrize("kv_dtype,q_dtype", KINDS, ids=["bf16", "fp8", "fp8q"])
@pytest.mark.parametrize("case", RAGGED, ids=[c[0] for c in RAGGED])
def test_fused_ragged_rows(oracle_mod, case, kv_dtype, q_dtype):
    name, B, rpr, H, pc, vis, oc, nn = case
    R = B * rpr
    spec = qi.custom(name, B, rpr, H, pc, (vis * R)[:R], oc, k=64, kv_dtype=kv_dtype, seed=78,
                     next_n_lens=nn, q_dtype=q_dtype)
    inp = qi.build_inputs(spec)
    logits, idx, ran, _ = run_fused(inp, 64)
    assert ran == qsa.VARIANT_UMMA_TOPK
    check(oracle_mod, inp, logits, idx, 64, where=name)
    dead = ~spec.live_rows()
    assert (idx.cpu().numpy()[dead] == -1).all()
    assert workspace_is_zero()


def test_fused_matches_the_two_calls_bit_for_bit():
    inp = qi.build_inputs(case_spec(CASES[2], qi.KV_BF16))
    s = inp.spec
    logits, idx, ran, d = run_fused(inp, s.k)
    assert ran == qsa.VARIANT_UMMA_TOPK
    ref = torch_api.paged_mqa_logits(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"],
                                     page_cols=s.page_cols, out_cols=s.out_cols)
    ridx = torch_api.select_topk(ref, d["visible"], s.k)
    torch.cuda.synchronize()
    assert torch.equal(logits.view(torch.int32), ref.view(torch.int32))
    assert torch.equal(idx, ridx)


def test_repeat_calls_and_side_stream(oracle_mod):
    inp = qi.build_inputs(case_spec(CASES[0], qi.KV_BF16))
    a_l, a_i, _, d = run_fused(inp, 256)
    s = torch.cuda.Stream()
    ws = torch.zeros(1024, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        b_l, b_i, ran, _ = run_fused(inp, 256, dev=d, workspace=ws, stream=s)
    assert ran == qsa.VARIANT_UMMA_TOPK
    assert torch.equal(a_l.view(torch.int32), b_l.view(torch.int32)) and torch.equal(a_i, b_i)
    assert int(ws.abs().sum()) == 0


def test_fused_graph_replay_with_new_inputs(oracle_mod):
    """vLLM #62589 Validation: capture once, replay with new q and lengths written in place."""
    spec = case_spec(CASES[2], qi.KV_BF16)
    inp = qi.build_inputs(spec)
    d = qi.device_tensors(inp)
    s = inp.spec
    logits = torch.empty((s.num_rows, s.out_cols), dtype=torch.float32, device="cuda")
    idx = torch.empty((s.num_rows, s.k), dtype=torch.int32, device="cuda")

    def call():
        torch_api.paged_mqa_topk(d["q"], d["weights"], d["kv"], d["block_table"], d["visible"], s.k,
                                 page_cols=s.page_cols, out_cols=s.out_cols, out_logits=logits, out_idx=idx)

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    rng = np.random.default_rng(11)
    for _ in range(3):
        inp.q = qi._bf16_bits(rng.standard_normal(inp.q.shape, dtype=np.float32))
        new_vis = np.maximum(spec.visible - rng.integers(0, 600, size=spec.visible.shape), 0).astype(np.int32)
        d["q"].copy_(torch.from_numpy(inp.q.view(np.int16)).view(torch.bfloat16))
        d["visible"].copy_(torch.from_numpy(new_vis))
        logits.fill_(float("nan"))
        idx.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_mod.paged_mqa_logits(inp, visible=new_vis)
        got = logits.cpu().numpy()
        assert_logits_match(got, ref, qi.KV_BF16, where="fused graph replay")
        assert_topk_strict(idx.cpu().numpy(), oracle_mod.select_topk(got, new_vis, s.k))
        assert workspace_is_zero()


def test_fused_call_with_the_cuda_core_scorer(oracle_mod):
    """A forced CUDA-core scorer makes the call the scoring launch + the top-k
    launch (the fused selection lives in the tcgen05 kernel only)."""
    inp = qi.build_inputs(case_spec(CASES[2], qi.KV_BF16))
    qsa.force_variant(qsa.VARIANT_ROWCORE)
    try:
        logits, idx, ran, _ = run_fused(inp, inp.spec.k, max_visible=int(inp.spec.visible.max()))
    finally:
        qsa.force_variant(qsa.VARIANT_UMMA_TOPK)
    assert ran == qsa.VARIANT_ROWCORE
    check(oracle_mod, inp, logits, idx, inp.spec.k, where="rowcore composition")
    assert workspace_is_zero()


@pytest.mark.parametrize("name", ["single_row_decode", "tiny_mtp"])
def test_fused_full_size_decode_workloads(oracle_mod, name):
    """The one-call form at the full size the bench times it (its host bound of
    the visible counts, so the selection runs in the scoring kernel): every
    row's logits and selection against the oracle."""
    spec = qi.WORKLOADS[name]()
    inp = qi.build_inputs(spec)
    logits, idx, ran, _ = run_fused(inp, spec.k, max_visible=int(spec.live_visible().max()))
    assert ran == qsa.VARIANT_UMMA_TOPK
    check(oracle_mod, inp, logits, idx, spec.k, where=f"{name} full size")
    assert workspace_is_zero()


@pytest.mark.parametrize("case,fused", [(CASES[0], False), (CASES[2], False), (CASES[3], False)],
                         ids=["single_row", "mtp4", "rows16"])
def test_auto_dispatch_takes_the_two_launches(oracle_mod, case, fused):
    """AUTO: the scorer the dispatch picks and the top-k launch (measured
    faster than the fused kernel at every decode shape)."""
    qsa.force_variant(qsa.VARIANT_AUTO)
    inp = qi.build_inputs(case_spec(case, qi.KV_BF16))
    k = case[7]
    logits, idx, ran, _ = run_fused(inp, k, max_visible=int(inp.spec.visible.max()))
    s = inp.spec
    scorer = qsa.plan_variant(qsa.make_desc(s.num_requests, s.rows_per_req, s.num_heads, s.page_cols, s.max_pages,
                                            inp.num_pages, s.out_cols, inp.key_page_stride))
    assert ran == (qsa.VARIANT_UMMA_TOPK if fused else scorer)
    check(oracle_mod, inp, logits, idx, k, where=f"auto {case[0]}")


def test_no_fused_kernel_gave_up_on_a_barrier():
    assert qsa.device_status(clear=True) == 0
