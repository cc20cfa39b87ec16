"""qsa_paged_mqa_topk_noalloc (the fused call on the library's fixed counter
array) against qsa_paged_mqa_topk with a caller workspace: two calls in a row
each, identical logits and selections.  Kept in its own file, collected last,
and independent of every other test's state."""
import numpy as np
import pytest

import qsa_inputs as qi
from qsa_testlib import nan_filled

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import sparse_attention_indexer_02_gb300 as qsa  # noqa: E402
from sparse_attention_indexer_02_gb300 import _abi, torch_api  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qsa.load_library()
    # the counters serve the selection inside the scoring kernel, which the
    # dispatch runs for single-row requests only: force it for every case
    qsa.force_variant(qsa.VARIANT_UMMA_TOPK)
    yield
    qsa.force_variant(qsa.VARIANT_AUTO)


def _desc(inp):
    s = inp.spec
    stride = inp.key_page_stride
    return qsa.make_desc(s.num_requests, s.rows_per_req, s.num_heads, s.page_cols, s.max_pages, inp.num_pages,
                         s.out_cols, stride, kv_dtype=s.kv_dtype,
                         scale_page_stride=stride if s.kv_dtype == qi.KV_FP8 else 0)


def _call(inp, d, k, noalloc, ws=None):
    s = inp.spec
    logits = nan_filled((s.num_rows, s.out_cols), torch.float32, "cuda")
    idx = nan_filled((s.num_rows, k), torch.int32, "cuda")
    scales = d["kv"].data_ptr() + inp.scale_offset if s.kv_dtype == qi.KV_FP8 else None
    q_dtype = qsa.Q_FP8_E4M3 if s.q_dtype == qi.Q_FP8 else qsa.Q_BF16
    mv = int(s.live_visible().max())
    if noalloc:
        _abi.paged_mqa_topk_noalloc(_desc(inp), d["q"], d["weights"], d["kv"], scales, d["block_table"],
                                    d["visible"], k, logits, idx, next_n_lens=d.get("next_n_lens"),
                                    q_dtype=q_dtype, max_visible=mv)
    else:
        _abi.paged_mqa_topk(_desc(inp), d["q"], d["weights"], d["kv"], scales, d["block_table"], d["visible"], k,
                            logits, idx, ws, ws.numel() * 4, next_n_lens=d.get("next_n_lens"), q_dtype=q_dtype,
                            max_visible=mv)
    ran = qsa.last_variant()
    torch.cuda.synchronize()
    return logits, idx, ran


CASES = [
    # (name, B, rows/req, H, page_cols, visible (cycled), out_cols, k, kv, q, next_n_lens)
    ("decode_16x1", 16, 1, 4, 16, [8192, 3000, 2049, 7777], 8192, 2048, qi.KV_BF16, qi.Q_BF16, None),
    ("mtp_4x4_fp8", 4, 4, 4, 64, [2500, 2501, 2502, 2503, 900, 901, 902, 903], 2560, 256, qi.KV_FP8, qi.Q_BF16,
     None),
    ("ragged_fp8q", 5, 4, 32, 64, [3000, 3001, 3002, 3003], 3008, 512, qi.KV_FP8, qi.Q_FP8, [4, 1, 0, 3, 2]),
    # 300 rows: scoring + top-k launches (no counters used), within the array's 128 groups
    ("rows300_two_launches", 1, 300, 4, 64, [1000 + i for i in range(300)], 1344, 64, qi.KV_BF16, qi.Q_BF16,
     None),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_the_workspace_call_on_two_calls_in_a_row(case):
    name, B, rpr, H, pc, vis, oc, k, kv, qd, nn = case
    R = B * rpr
    spec = qi.custom(name, B, rpr, H, pc, (vis * R)[:R], oc, k=k, kv_dtype=kv, seed=31, q_dtype=qd,
                     next_n_lens=nn)
    inp = qi.build_inputs(spec)
    d = qi.device_tensors(inp)
    ws = torch.zeros(max(64, _abi.topk_workspace_bytes(_desc(inp)) // 4 + 1), dtype=torch.int32, device="cuda")
    for _ in range(2):
        ref_l, ref_i, ran_ref = _call(inp, d, k, noalloc=False, ws=ws)
        got_l, got_i, ran = _call(inp, d, k, noalloc=True)
        assert ran == ran_ref == (qsa.VARIANT_UMMA if spec.num_rows > 256 else qsa.VARIANT_UMMA_TOPK)
        assert torch.equal(got_l.view(torch.int32), ref_l.view(torch.int32))
        assert torch.equal(got_i, ref_i)
        assert int(ws.abs().sum()) == 0
    assert qsa.device_status(clear=True) == 0


class _DeviceWords:
    """int32 view of device memory the library owns (zero-copy, through the
    CUDA array interface), so the test can write the counter array directly."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (ptr, False), "version": 2,
                                         "strides": None}


def test_device_status_clear_zeroes_counters_a_failed_call_left():
    """A no-alloc call that gave up on a barrier (qsa_device_status bit 0) may
    leave counts in the array; here they are planted from the host instead.
    qsa_device_status(clear) zeroes the array, and the next calls match the
    workspace call again."""
    addr, nbytes = _abi.noalloc_counters()
    assert addr != 0 and nbytes == 4 * 257
    words = torch.as_tensor(_DeviceWords(addr, nbytes // 4), device="cuda")
    words.copy_(torch.arange(1, nbytes // 4 + 1, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(words.abs().sum()) > 0
    assert qsa.device_status(clear=True) == 0
    assert int(words.abs().sum()) == 0
    test_noalloc_matches_the_workspace_call_on_two_calls_in_a_row(CASES[0])
    assert int(words.abs().sum()) == 0
