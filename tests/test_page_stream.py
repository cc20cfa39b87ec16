"""qsa_page_stream, the measurement stream of listed pages: argument checks (no
GPU needed: they fail before any CUDA call) and, on the GPU, its checksum -
the XOR of every 32-bit word of every listed page copy - against numpy's, bit
for bit, over lists with repeats, out-of-range indices (clamped) and more
pages than the CTAs' rings hold."""
import numpy as np
import pytest

import sparse_attention_indexer_02_gb300 as qsa


@pytest.fixture(scope="module")
def lib():
    return qsa.load_library()


@pytest.mark.parametrize("args", [
    (None, 256, 128, 16, 4, 8, 16),        # null base
    (16, 256, 128, None, 4, 8, 16),        # null page list
    (16, 256, 128, 16, 4, 8, None),        # null checksum
    (24, 256, 128, 16, 4, 8, 16),          # base not 16-byte aligned
    (16, 264, 128, 16, 4, 8, 16),          # stride not a multiple of 16
    (16, 256, 8, 16, 4, 8, 16),            # page_bytes below 16
    (16, 256, 136, 16, 4, 8, 16),          # page_bytes not a multiple of 16
    (16, 256, 272, 16, 4, 8, 16),          # page_bytes above the stride
    (16, 1 << 20, 65552, 16, 4, 8, 16),    # page_bytes above 65536
    (16, 256, 128, 16, 4, 0, 16),          # empty pool
    (16, 256, 128, 18, 4, 8, 16),          # page list not 4-byte aligned
    (16, 256, 128, 16, -1, 8, 16),         # negative count
])
def test_argument_checks(lib, args):
    base, stride, nbytes, pages, n, pool, checksum = args
    with pytest.raises(qsa.QSAError) as e:
        qsa.page_stream(base, stride, nbytes, pages, n, pool, checksum, stream=0)
    assert e.value.status == qsa.QSA_ERR_INVALID_ARG


def test_empty_list_is_a_no_op(lib):
    qsa.page_stream(None, 256, 128, None, 0, 0, None, stream=0)


def xor_words(pool_u32, stride_words, nwords, pages, pool_pages):
    pg = np.clip(np.asarray(pages, np.int64), 0, pool_pages - 1)
    x = np.uint32(0)
    for p in pg:
        x ^= np.bitwise_xor.reduce(pool_u32[p * stride_words:p * stride_words + nwords])
    return int(x)


@pytest.mark.gpu
@pytest.mark.parametrize("stride,nbytes,pool_pages,listed", [
    (8448, 8448, 300, 2000),    # fp8 block-flat page (64 keys + their scales), more pages than rings hold
    (4096, 4096, 97, 1),        # one bf16 page of 16 keys
    (16384, 8192, 50, 777),     # half of each page
    (65536, 65536, 9, 40),      # the largest copy (one stage a CTA)
])
def test_checksum_matches_numpy(lib, stride, nbytes, pool_pages, listed):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_attention_indexer_02_gb300 import torch_api
    rng = np.random.default_rng(stride + listed)
    pool = rng.integers(0, 2**32, size=pool_pages * stride // 4, dtype=np.uint32)
    pages = rng.integers(-3, pool_pages + 3, size=listed).astype(np.int32)   # repeats and clamped indices
    d_pool = torch.from_numpy(pool.view(np.int32)).cuda()
    d_pages = torch.from_numpy(pages).cuda()
    got = torch_api.page_stream(d_pool, stride, nbytes, d_pages)
    torch.cuda.synchronize()
    assert qsa.device_status() == 0
    want = xor_words(pool, stride // 4, nbytes // 4, pages, pool_pages)
    assert int(got.cpu().numpy().view(np.uint32)[0]) == want
