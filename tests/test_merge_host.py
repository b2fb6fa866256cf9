"""CPU: splitzip_merge joins the containers of consecutive whole-chunk pieces
into the container of the whole tensor.

The pieces and the expected whole container come from the oracle; the merge is
the library's (host code, no GPU needed).  Byte equality is required, for both
dtypes, several chunk sizes, empty pieces and a ragged last piece; pieces that
cannot be joined are refused.
"""
import ctypes

import numpy as np
import pytest

import oracle
import lossless_kv_cache_gb300 as sz
from lossless_kv_cache_gb300 import workloads as W


def _tensor(dtype, n):
    if dtype == 0:
        return W.escape_stress(3, chunks=5, chunk_elems=65536).numpy().view(np.uint16)[:n]
    if dtype == 2:
        return W.kv_cache_layer_fp16(1, 2, tokens=160).numpy().view(np.uint16)[:n]
    return W.kv_cache_layer_e5m2(1, 2, tokens=300).numpy()[:n]


@pytest.mark.parametrize("dtype", [0, 1, 2])
@pytest.mark.parametrize("chunk", [64, 4096, 65536])
def test_merge_of_oracle_pieces_is_the_whole_container(dtype, chunk):
    n = 5 * 65536 - 333
    x = _tensor(dtype, n)
    cb = oracle.calibrate(oracle.histogram(x, dtype), dtype)
    whole = oracle.encode(x, dtype, cb, chunk)
    C = -(-n // chunk)
    rng = np.random.default_rng(chunk + dtype)
    for pieces in (1, 2, 3, 7):
        inner = sorted(rng.choice(np.arange(0, C), size=pieces - 1, replace=True)) if pieces > 1 else []
        cuts = [0] + [int(c) * chunk for c in inner] + [n]  # repeated cuts give empty pieces
        parts = [oracle.encode(x[a:b], dtype, cb, chunk) for a, b in zip(cuts, cuts[1:])]
        np.testing.assert_array_equal(sz.merge(parts), whole)


def test_merge_size_query_and_capacity():
    x = _tensor(0, 3 * 4096 + 5)
    cb = oracle.calibrate(oracle.histogram(x, 0), 0)
    whole = oracle.encode(x, 0, cb, 4096)
    parts = [oracle.encode(x[:8192], 0, cb, 4096), oracle.encode(x[8192:], 0, cb, 4096)]
    ptrs = (ctypes.c_void_p * 2)(*[p.ctypes.data for p in parts])
    sizes = (ctypes.c_uint64 * 2)(*[p.size for p in parts])
    got = ctypes.c_uint64(0)
    assert sz.splitzip_merge(ptrs, sizes, 2, None, 0, got) == sz.OK and got.value == whole.size
    out = np.zeros(whole.size, np.uint8)
    assert sz.splitzip_merge(ptrs, sizes, 2, out.ctypes.data, whole.size - 1, got) == sz.ERR_CAPACITY
    assert sz.splitzip_merge(ptrs, sizes, 2, out.ctypes.data, whole.size, got) == sz.OK
    np.testing.assert_array_equal(out, whole)


def test_merge_refuses_pieces_that_do_not_join():
    x = _tensor(0, 4 * 4096)
    cb = oracle.calibrate(oracle.histogram(x, 0), 0)
    a, b = oracle.encode(x[:8192], 0, cb, 4096), oracle.encode(x[8192:], 0, cb, 4096)

    def merge_status(parts):
        arrs = [np.ascontiguousarray(p) for p in parts]
        ptrs = (ctypes.c_void_p * len(arrs))(*[p.ctypes.data for p in arrs])
        sizes = (ctypes.c_uint64 * len(arrs))(*[p.size for p in arrs])
        return sz.splitzip_merge(ptrs, sizes, len(arrs), None, 0, ctypes.c_uint64(0))

    assert merge_status([a, b]) == sz.OK
    # a first piece that ends in a partial chunk
    assert merge_status([oracle.encode(x[:8000], 0, cb, 4096), b]) == sz.ERR_INVALID_ARG
    # another codebook, another chunk size, another dtype
    cb2 = cb.copy()
    cb2[[0, 1]] = cb2[[1, 0]]
    assert merge_status([a, oracle.encode(x[8192:], 0, cb2, 4096)]) == sz.ERR_INVALID_ARG
    assert merge_status([a, oracle.encode(x[8192:], 0, cb, 2048)]) == sz.ERR_INVALID_ARG
    e = W.kv_cache_layer_e5m2(0, 0, tokens=8)
    ecb = oracle.calibrate(oracle.histogram(e.numpy(), 1), 1)
    assert merge_status([a, oracle.encode(e.numpy(), 1, ecb, 4096)]) == sz.ERR_INVALID_ARG
    # an index whose offsets are not the prefix of its counts, a truncated piece
    bad = b.copy()
    bad[64 + 8] ^= 1
    assert merge_status([a, bad]) == sz.ERR_CORRUPT
    assert merge_status([a, b[:-1]]) == sz.ERR_CORRUPT
    assert sz.splitzip_merge(None, None, 0, None, 0, ctypes.c_uint64(0)) == sz.ERR_INVALID_ARG
