"""C-ABI library checks that need no GPU: it builds, loads, exports every
symbol include/qsa.h declares, and its host-side validation and dispatch
behave.  No call here reaches a kernel launch: every compute call below is
rejected by host validation before anything is enqueued."""
import ctypes
import os
import re

import pytest

import sparse_attention_indexer_02_gb300 as qsa
from sparse_attention_indexer_02_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qsa.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"{n} declared in qsa.h but not exported"
    assert set(names) == set(qsa.EXPORTED)


def test_abi_version_and_status_strings(lib):
    assert qsa.abi_version() == 1
    assert qsa.status_string(qsa.QSA_OK) == "QSA_OK"
    assert qsa.status_string(qsa.QSA_ERR_UNSUPPORTED) == "QSA_ERR_UNSUPPORTED"
    assert "unknown" in qsa.status_string(99)


def _desc(**kw):
    base = dict(num_requests=2, rows_per_req=4, num_heads=4, page_cols=16, max_pages=8, num_pages=16,
                out_cols=128, key_page_stride=16 * 128 * 2)
    base.update(kw)
    return qsa.make_desc(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), qsa.QSA_ERR_UNSUPPORTED),
    (dict(num_heads=65), qsa.QSA_ERR_UNSUPPORTED),
    (dict(num_heads=0), qsa.QSA_ERR_INVALID_ARG),
    (dict(rows_per_req=0), qsa.QSA_ERR_INVALID_ARG),
    (dict(num_requests=-1), qsa.QSA_ERR_INVALID_ARG),
    (dict(page_cols=0), qsa.QSA_ERR_INVALID_ARG),
    (dict(out_cols=-5), qsa.QSA_ERR_INVALID_ARG),
    (dict(key_page_stride=16 * 128 * 2 - 16), qsa.QSA_ERR_INVALID_ARG),
    (dict(key_page_stride=16 * 128 * 2 + 8), qsa.QSA_ERR_INVALID_ARG),
    (dict(kv_dtype=7), qsa.QSA_ERR_INVALID_ARG),
    (dict(kv_dtype=qsa.KV_FP8_E4M3, key_page_stride=16 * 132, scale_page_stride=2), qsa.QSA_ERR_INVALID_ARG),
])
def test_descriptor_validation(lib, kw, status):
    d = _desc(**kw)
    with pytest.raises(qsa.QSAError) as e:
        qsa.plan_variant(d)
    assert e.value.status == status
    with pytest.raises(qsa.QSAError) as e:
        qsa.paged_mqa_logits(d, None, None, None, None, None, None, None, stream=0)
    assert e.value.status == status


def test_mixed_operand_types_rejected(lib):
    """SGLang #48649 test list: rejects_mixed_operand_dtypes."""
    with pytest.raises(qsa.QSAError) as e:  # bf16 keys with a scales pointer
        qsa.paged_mqa_logits(_desc(), 16, 16, 16, 16, 16, 16, 16, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG and "mixed" in str(e.value)
    d8 = _desc(kv_dtype=qsa.KV_FP8_E4M3, key_page_stride=16 * 132, scale_page_stride=16 * 132)
    with pytest.raises(qsa.QSAError) as e:  # fp8 keys without scales
        qsa.paged_mqa_logits(d8, 16, 16, 16, None, 16, 16, 16, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG


def test_fp8_q_needs_fp8_keys_and_a_known_q_dtype(lib):
    """fp8 q with bf16 keys is a mixed-operand call (SGLang #48649 rejects_mixed_operand_dtypes)."""
    with pytest.raises(qsa.QSAError) as e:
        qsa.paged_mqa_logits(_desc(), 16, 16, 16, None, 16, 16, 16, stream=0, q_dtype=qsa.Q_FP8_E4M3)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG and "mixed" in str(e.value)
    d8 = _desc(kv_dtype=qsa.KV_FP8_E4M3, key_page_stride=16 * 132, scale_page_stride=16 * 132)
    with pytest.raises(qsa.QSAError) as e:
        qsa.paged_mqa_logits(d8, 16, 16, 16, 16, 16, 16, 16, stream=0, q_dtype=7)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG and "q_dtype" in str(e.value)


def test_null_and_misaligned_pointers_rejected(lib):
    with pytest.raises(qsa.QSAError) as e:
        qsa.paged_mqa_logits(_desc(), None, 16, 16, None, 16, 16, 16, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG
    with pytest.raises(qsa.QSAError) as e:  # q not 16-byte aligned
        qsa.paged_mqa_logits(_desc(), 24, 16, 16, None, 16, 16, 16, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG
    with pytest.raises(qsa.QSAError) as e:  # out not 4-byte aligned
        qsa.paged_mqa_logits(_desc(), 16, 16, 16, None, 16, 16, 18, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG


def test_empty_calls_are_no_ops(lib):
    qsa.paged_mqa_logits(_desc(num_requests=0), None, None, None, None, None, None, None, stream=0)
    qsa.paged_mqa_logits(_desc(out_cols=0), None, None, None, None, None, None, None, stream=0)
    qsa.select_topk(None, 0, 10, None, 8, None, stream=0)
    for bound in (0, -5, 1, 8192, 1 << 40):
        qsa.select_topk_bounded(None, 0, 10, None, bound, 8, None, stream=0)


@pytest.mark.parametrize("k", [0, -1, 2049])
def test_topk_k_range(lib, k):
    with pytest.raises(qsa.QSAError) as e:
        qsa.select_topk(16, 4, 100, 16, k, 16, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG
    with pytest.raises(qsa.QSAError) as e:
        qsa.select_topk_bounded(16, 4, 100, 16, 64, k, 16, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG


TOPK_BAD_ARGS = [(16, -1, 100, 16, 8, 16), (16, 4, 0, 16, 8, 16), (None, 4, 100, 16, 8, 16),
                 (18, 4, 100, 16, 8, 16), (16, 4, 100, None, 8, 16), (16, 4, 100, 16, 8, None),
                 (16, 4, 100, 18, 8, 16), (16, 4, 100, 16, 8, 18)]


@pytest.mark.parametrize("args", TOPK_BAD_ARGS)
def test_topk_argument_checks(lib, args):
    with pytest.raises(qsa.QSAError) as e:
        qsa.select_topk(*args, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG


@pytest.mark.parametrize("bound", [0, 100, 8192, 1 << 40])
@pytest.mark.parametrize("args", TOPK_BAD_ARGS)
def test_bounded_topk_argument_checks(lib, args, bound):
    """qsa_select_topk_bounded rejects what qsa_select_topk rejects, whatever
    the bound (which is never itself an error)."""
    logits, rows, stride, vis, k, out = args
    with pytest.raises(qsa.QSAError) as e:
        qsa.select_topk_bounded(logits, rows, stride, vis, bound, k, out, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG


def test_last_error_names_the_problem(lib):
    with pytest.raises(qsa.QSAError):
        qsa.plan_variant(_desc(head_dim=96))
    assert "head_dim" in qsa.last_error()


def test_dispatch_decisions(lib):
    """Host dispatch on host metadata only (vLLM #62589 'Dispatch')."""
    qsa.force_variant(qsa.VARIANT_AUTO)
    # single-row bf16 decode: the lean tcgen05 form
    assert qsa.plan_variant(_desc(rows_per_req=1)) == qsa.VARIANT_UMMA_LEAN
    # odd page size: only the CUDA-core scorer serves it
    assert qsa.plan_variant(_desc(page_cols=5, key_page_stride=5 * 256)) == qsa.VARIANT_ROWCORE
    # MTP verify rows (4 rows x 4 heads = N 16): lean; 256 rows still lean, 260 not
    assert qsa.plan_variant(_desc()) == qsa.VARIANT_UMMA_LEAN
    assert qsa.plan_variant(_desc(num_requests=64)) == qsa.VARIANT_UMMA_LEAN
    assert qsa.plan_variant(_desc(num_requests=65)) == qsa.VARIANT_UMMA
    # groups wider than 64 rows x heads (32 rows x 4 heads = N 128), or whose q
    # leaves the lean form's shared memory fewer than three 32 KB key stages
    # (bf16 at N 64): the full form
    assert qsa.plan_variant(_desc(rows_per_req=32)) == qsa.VARIANT_UMMA
    assert qsa.plan_variant(_desc(rows_per_req=16)) == qsa.VARIANT_UMMA
    assert qsa.plan_variant(_desc(rows_per_req=8)) == qsa.VARIANT_UMMA_LEAN
    # fp8 keys (with bf16 q, which qsa_plan_variant assumes): the converter of the full form
    d8 = _desc(rows_per_req=1, num_heads=64, page_cols=64, key_page_stride=64 * 132,
               kv_dtype=qsa.KV_FP8_E4M3, scale_page_stride=64 * 132)
    assert qsa.plan_variant(d8) == qsa.VARIANT_UMMA
    # head counts the tcgen05 epilogue is not built for -> CUDA-core scorer
    assert qsa.plan_variant(_desc(num_heads=3)) == qsa.VARIANT_ROWCORE
    qsa.force_variant(qsa.VARIANT_ROWCORE)
    assert qsa.plan_variant(_desc()) == qsa.VARIANT_ROWCORE
    qsa.force_variant(qsa.VARIANT_UMMA)
    assert qsa.plan_variant(_desc()) == qsa.VARIANT_UMMA
    with pytest.raises(qsa.QSAError) as e:
        qsa.plan_variant(_desc(page_cols=5, key_page_stride=5 * 256))
    assert e.value.status == qsa.QSA_ERR_UNSUPPORTED
    qsa.force_variant(qsa.VARIANT_UMMA_LEAN)
    assert qsa.plan_variant(_desc()) == qsa.VARIANT_UMMA_LEAN
    for bad in (d8, _desc(num_requests=65), _desc(rows_per_req=32)):
        with pytest.raises(qsa.QSAError) as e:
            qsa.plan_variant(bad)
        assert e.value.status == qsa.QSA_ERR_UNSUPPORTED and "lean" in str(e.value)
    qsa.force_variant(qsa.VARIANT_AUTO)


def test_fused_call_workspace_size_and_argument_checks(lib):
    """qsa_paged_mqa_topk: host checks before anything is enqueued (the fused
    kernel forced, so the call needs a workspace)."""
    qsa.force_variant(qsa.VARIANT_UMMA_TOPK)
    d = _desc(rows_per_req=1)  # 2 single-row requests: two row groups
    assert qsa.topk_workspace_bytes(d) == 4 * (2 * 2 + 1)
    # the CUDA-core scorer's shapes never run the fused selection
    assert qsa.topk_workspace_bytes(_desc(page_cols=5, key_page_stride=5 * 256)) == 0
    args = (d, 16, 16, 16, None, 16, 16)
    for k in (0, 2049):
        with pytest.raises(qsa.QSAError) as e:
            qsa.paged_mqa_topk(*args, k, 16, 16, 16, 64, stream=0)
        assert e.value.status == qsa.QSA_ERR_INVALID_ARG and "k must" in str(e.value)
    with pytest.raises(qsa.QSAError) as e:  # no workspace
        qsa.paged_mqa_topk(*args, 8, 16, 16, None, 0, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG and "workspace" in str(e.value)
    with pytest.raises(qsa.QSAError) as e:  # workspace too small
        qsa.paged_mqa_topk(*args, 8, 16, 16, 16, 16, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG and "20 bytes" in str(e.value)
    with pytest.raises(qsa.QSAError) as e:  # misaligned out_idx
        qsa.paged_mqa_topk(*args, 8, 16, 18, 16, 64, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG
    with pytest.raises(qsa.QSAError) as e:  # the scoring checks come first
        qsa.paged_mqa_topk(_desc(head_dim=64), 16, 16, 16, None, 16, 16, 8, 16, 16, 16, 64, stream=0)
    assert e.value.status == qsa.QSA_ERR_UNSUPPORTED
    qsa.paged_mqa_topk(_desc(num_requests=0), None, None, None, None, None, None, 8, None, None, None, 0,
                       stream=0)  # no rows: nothing to do
    qsa.force_variant(qsa.VARIANT_AUTO)


def test_one_call_fuses_only_when_forced(lib):
    """The dispatch of qsa_paged_mqa_topk: the scoring and top-k launches
    (measured faster than the fused kernel at every decode shape; no
    workspace), the selection inside the scoring kernel only with
    QSA_VARIANT_UMMA_TOPK forced (a workspace), never for a forced scorer."""
    qsa.force_variant(qsa.VARIANT_AUTO)
    try:
        assert qsa.topk_workspace_bytes(_desc(rows_per_req=1)) == 0
        assert qsa.topk_workspace_bytes(_desc()) == 0
        assert qsa.topk_workspace_bytes(_desc(rows_per_req=1, page_cols=5, key_page_stride=5 * 256)) == 0
        qsa.force_variant(qsa.VARIANT_UMMA_TOPK)
        assert qsa.topk_workspace_bytes(_desc()) == 4 * (2 * 2 + 1)
        assert qsa.topk_workspace_bytes(_desc(rows_per_req=1)) == 4 * (2 * 2 + 1)
        assert qsa.plan_variant(_desc()) == qsa.VARIANT_UMMA_LEAN  # scoring dispatch unchanged
        for forced in (qsa.VARIANT_UMMA, qsa.VARIANT_UMMA_LEAN, qsa.VARIANT_ROWCORE):
            qsa.force_variant(forced)
            assert qsa.topk_workspace_bytes(_desc(rows_per_req=1)) == 0
    finally:
        qsa.force_variant(qsa.VARIANT_AUTO)


def test_noalloc_call_rejects_shapes_past_its_counters(lib):
    """qsa_paged_mqa_topk_noalloc holds counters for 128 row groups: a call
    that would select inside the scoring kernel (forced) over more is refused
    before anything is enqueued."""
    d = _desc(num_requests=200, rows_per_req=1)  # 200 groups of one row
    qsa.force_variant(qsa.VARIANT_UMMA_TOPK)
    try:
        with pytest.raises(qsa.QSAError) as e:
            qsa._abi.paged_mqa_topk_noalloc(d, 16, 16, 16, None, 16, 16, 8, 16, 16, stream=0)
        assert e.value.status == qsa.QSA_ERR_UNSUPPORTED and "128 row groups" in str(e.value)
        with pytest.raises(qsa.QSAError) as e:  # the scoring checks come first
            qsa._abi.paged_mqa_topk_noalloc(_desc(head_dim=64), 16, 16, 16, None, 16, 16, 8, 16, 16, stream=0)
        assert e.value.status == qsa.QSA_ERR_UNSUPPORTED and "head_dim" in str(e.value)
    finally:
        qsa.force_variant(qsa.VARIANT_AUTO)
