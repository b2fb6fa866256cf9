"""The allocation-free encode entry point, splitzip_encode_noalloc.

It serves callers that cannot allocate device memory when they encode (an
engine whose KV pool already owns nearly all GPU memory, or a path that must
not call cudaMalloc/cudaFree because they can synchronise the device).  Its
scratch is a fixed 32 MiB device array inside the library.  These tests call
it through the C ABI and require byte-identical output to splitzip_encode on
two calls in a row (the second call finds the first call's scratch contents),
and a clean error for sizes beyond the array.  This file is collected last so
a failure here cannot hide the result of any other test.
"""
import numpy as np
import pytest
import torch

import lossless_kv_cache_gb300 as sz
from lossless_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _regular(x, cb, dtype, chunk):
    bufs = sz.EncodeBuffers(x.numel(), dtype, chunk)
    sz.encode_into(x, cb, bufs)
    torch.cuda.synchronize()
    assert int(bufs.status[0]) == sz.OK
    return bufs.out[: int(bufs.size[0])].cpu()


def _noalloc(x, cb, dtype, chunk):
    cap = sz.max_compressed_size(x.numel(), dtype, chunk)
    out = torch.full((cap,), 0xA5, dtype=torch.uint8, device="cuda")
    size = torch.zeros(2, dtype=torch.int64, device="cuda")
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    st = sz.splitzip_encode_noalloc(x.data_ptr(), x.numel(), dtype, cb, chunk, out.data_ptr(), cap,
                                    size.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == sz.OK, sz.splitzip_status_string(st)
    torch.cuda.synchronize()
    assert int(status[0]) == sz.OK
    return out[: int(size[0])].cpu()


def test_noalloc_matches_encode_on_two_calls_in_a_row(splitzip_lib):
    assert torch.cuda.is_available()
    # call 1: a BF16 layer slice with ordinary escape rates, default chunk
    x1 = W.llama_layer_kv(0, tokens=2048).to("cuda")  # 4,194,304 elements
    cb1, _ = sz.calibrate(x1, sz.BF16)
    got1 = _noalloc(x1, cb1, sz.BF16, 65536)
    assert torch.equal(got1, _regular(x1, cb1, sz.BF16, 65536))
    # call 2: heavier escapes, a ragged size and a smaller chunk, so the
    # scratch still holds call 1's staged records at other offsets
    x2 = W.escape_stress(1, chunks=96, chunk_elems=65536)[: 6_000_001].to("cuda")
    cb2 = sz.Codebook.make(sz.BF16, range(118, 134))
    got2 = _noalloc(x2, cb2, sz.BF16, 4096)
    assert torch.equal(got2, _regular(x2, cb2, sz.BF16, 4096))
    # the containers decode back to the inputs
    for x, blob in ((x1, got1), (x2, got2)):
        y = sz.decode(blob.to("cuda"), x.numel(), sz.BF16)
        assert torch.equal(y, x)


def test_noalloc_fp8_e5m2(splitzip_lib):
    x = W.kv_cache_layer_e5m2(2, 1, tokens=4000).to("cuda")  # 8,192,000 elements
    cb, _ = sz.calibrate(x, sz.FP8_E5M2)
    for _ in range(2):
        assert torch.equal(_noalloc(x, cb, sz.FP8_E5M2, 65536), _regular(x, cb, sz.FP8_E5M2, 65536))


def test_noalloc_rejects_sizes_beyond_its_scratch(splitzip_lib):
    # largest n whose workspace fits 32 MiB at the default chunk size
    for dtype, n_max in ((sz.BF16, 8_372_224), (sz.FP8_E5M2, 8_372_224)):
        assert sz.workspace_size(n_max, dtype, 65536) <= sz.NOALLOC_SCRATCH_BYTES
        assert sz.workspace_size(n_max + 1, dtype, 65536) > sz.NOALLOC_SCRATCH_BYTES
    limit = 8_372_224
    cb = sz.Codebook.make(sz.BF16, range(16))
    A = 1 << 20  # never dereferenced: the size check comes first
    st = sz.splitzip_encode_noalloc(A, limit + 1, sz.BF16, cb, 65536, A, 1 << 40, A, A, 0)
    assert st == sz.ERR_CAPACITY
