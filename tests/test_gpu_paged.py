"""GPU: paged KV input and output.  Encoding pages gathered from a pool must
give the oracle's container of the gathered tensor, byte for byte; decoding
into a pool must fill exactly the listed pages (bit-exact) and leave every
other byte of the pool as it was; bad page indices are reported."""
import numpy as np
import pytest
import torch

import oracle
import lossless_kv_cache_gb300 as sz
from lossless_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(splitzip_lib):
    assert torch.cuda.is_available()
    return splitzip_lib


def pool_of(dtype, pages, page_elems, seed):
    n = pages * page_elems
    if dtype == sz.BF16:
        x = W.escape_stress(seed, chunks=-(-n // 65536), chunk_elems=65536)[:n]
    else:
        x = W.kv_cache_layer_e5m2(seed, 5, tokens=-(-n // 2048))[:n]
    return x.cuda()


def host(t, dtype):
    a = t.cpu().numpy()
    return a.view(np.uint16) if dtype == sz.BF16 else a


@pytest.mark.parametrize("dtype", [sz.BF16, sz.FP8_E5M2])
@pytest.mark.parametrize("chunk,page_elems", [(65536, 16384), (4096, 16384), (65536, 65536), (1024, 4096)])
def test_paged_roundtrip_matches_oracle(dtype, chunk, page_elems):
    if page_elems % min(chunk, 8192 if dtype == sz.BF16 else 16384):
        pytest.skip("pages must hold whole encoder tiles")
    pool_pages = 11
    pool = pool_of(dtype, pool_pages, page_elems, 5)
    order = [7, 2, 9, 0, 10, 3, 2]  # a page may be listed twice
    pages = torch.tensor(order, dtype=torch.int32, device="cuda")
    gathered = torch.cat([pool[p * page_elems:(p + 1) * page_elems] for p in order])
    g_host = host(gathered, dtype)
    exps = oracle.calibrate(oracle.histogram(g_host, dtype), dtype)
    cb = sz.Codebook.make(dtype, [int(e) for e in exps])
    n = len(order) * page_elems
    bufs = sz.EncodeBuffers(n, dtype, chunk)
    sz.encode_paged_into(pool, pages, page_elems, cb, bufs)
    torch.cuda.synchronize()
    assert int(bufs.status[0]) == sz.OK
    blob = bufs.out[: int(bufs.size[0])]
    assert np.array_equal(blob.cpu().numpy(), oracle.encode(g_host, dtype, exps, chunk))
    # scatter into other pages of another pool
    fill = 0x5A5A if dtype == sz.BF16 else 0x5A
    dst = torch.full((13 * page_elems,), fill, dtype=pool.dtype, device="cuda")
    dst_order = [12, 1, 5, 4, 8, 0, 6]
    dpages = torch.tensor(dst_order, dtype=torch.int32, device="cuda")
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    sz.decode_paged_into(blob, blob.numel(), dst, dpages, page_elems, dtype, status)
    torch.cuda.synchronize()
    assert int(status[0]) == sz.OK
    for i, p in enumerate(dst_order):
        assert torch.equal(dst[p * page_elems:(p + 1) * page_elems], gathered[i * page_elems:(i + 1) * page_elems])
    untouched = [p for p in range(13) if p not in dst_order]
    for p in untouched:
        assert bool((dst[p * page_elems:(p + 1) * page_elems] == fill).all())


@pytest.mark.parametrize("dtype", [sz.BF16, sz.FP8_E5M2])
def test_paged_bad_page_index_is_reported(dtype):
    page_elems, pool_pages = 16384, 4
    pool = pool_of(dtype, pool_pages, page_elems, 6)
    cb = sz.Codebook.make(dtype, range(16) if dtype == sz.FP8_E5M2 else range(118, 134))
    for bad in ([0, 4, 1], [2, -1]):
        pages = torch.tensor(bad, dtype=torch.int32, device="cuda")
        bufs = sz.EncodeBuffers(len(bad) * page_elems, dtype)
        sz.encode_paged_into(pool, pages, page_elems, cb, bufs)
        torch.cuda.synchronize()
        assert int(bufs.status[0]) == sz.ERR_INVALID_ARG
    # a good container decoded through a bad page list: reported, the pool's
    # other pages untouched
    good = torch.tensor([1, 3], dtype=torch.int32, device="cuda")
    bufs = sz.EncodeBuffers(2 * page_elems, dtype)
    sz.encode_paged_into(pool, good, page_elems, cb, bufs)
    torch.cuda.synchronize()
    assert int(bufs.status[0]) == sz.OK
    fill = 0x1234 if dtype == sz.BF16 else 0x12
    dst = torch.full((pool_pages * page_elems,), fill, dtype=pool.dtype, device="cuda")
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    sz.decode_paged_into(bufs.out, bufs.capacity, dst, torch.tensor([2, 9], dtype=torch.int32, device="cuda"),
                         page_elems, dtype, status)
    torch.cuda.synchronize()
    assert int(status[0]) == sz.ERR_INVALID_ARG
    assert torch.equal(dst[2 * page_elems:3 * page_elems], pool[page_elems:2 * page_elems])
    for p in (0, 1, 3):
        assert bool((dst[p * page_elems:(p + 1) * page_elems] == fill).all())
