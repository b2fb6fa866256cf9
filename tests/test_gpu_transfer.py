"""GPU: the transfer path (encode -> D2H -> H2D -> decode per piece, four
streams) against the oracle.  The destination must equal the source bit for
bit, the bytes that crossed the link must be the oracle's container sizes of
the pieces, and the last container left in the host staging area must be the
oracle's container of the last piece, byte for byte."""
import ctypes

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


def slot_layout(x):
    """(slot stride, alignment) of the transfer's staging ring: slots and the
    area's base on 2 MiB boundaries, 64 KiB ones for slots under 2 MiB."""
    a = 2 << 20 if x >= 2 << 20 else 64 << 10
    return -(-x // a) * a, a


def bits(dtype, n, seed):
    if dtype == sz.BF16:
        x = W.escape_stress(seed, chunks=-(-n // 65536), chunk_elems=65536)[:n]
        return x.numpy().view(np.uint16), x.cuda()
    if dtype == sz.FP16:
        x = W.kv_cache_layer_fp16(seed, 3, tokens=-(-n // 2048))[:n]
        return x.numpy().view(np.uint16), x.cuda()
    x = W.kv_cache_layer_e5m2(seed, 3, tokens=-(-n // 1024))[:n]
    return x.numpy(), x.cuda()


@pytest.mark.parametrize("dtype", [sz.BF16, sz.FP8_E5M2, sz.FP16])
@pytest.mark.parametrize("chunk,piece", [(65536, 65536), (4096, 3 * 4096)])
def test_transfer_matches_oracle(dtype, chunk, piece):
    n = 9 * 65536 + 12345  # ten or more pieces: the ring of four slots is reused; a ragged last piece
    host, x = bits(dtype, n, 7)
    exps = oracle.calibrate(oracle.histogram(host, dtype), dtype)
    cb = sz.Codebook.make(dtype, [int(e) for e in exps])
    for compress in (True, False):
        y = torch.full_like(x, 0x55 if dtype == sz.FP8_E5M2 else 0x5555)
        bufs = sz.TransferBuffers(n, dtype, piece, compress, chunk)
        ms, link = sz.transfer(x, y, cb, bufs)
        torch.cuda.synchronize()
        assert torch.equal(y, x)
        assert ms > 0
        eb = 1 if dtype == sz.FP8_E5M2 else 2
        pieces = [(i, min(piece, n - i)) for i in range(0, n, piece)]
        if not compress:
            assert link == n * eb
            continue
        sizes = []
        for lo, m in pieces:
            E = int(oracle.chunk_escape_counts(host[lo:lo + m], dtype, exps, chunk).sum())
            sizes.append(oracle.container_size(m, dtype, chunk, E))
        assert link == sum(sizes)
        # the last piece's container is still in its staging slot
        lo, m = pieces[-1]
        ref = oracle.encode(host[lo:lo + m], dtype, exps, chunk)
        k = (len(pieces) - 1) % 4
        cap, a = slot_layout(sz.max_compressed_size(piece, dtype, chunk))
        base = -bufs.host.data_ptr() % a  # the ring starts at the next multiple of a
        got = bufs.host[base + k * cap: base + k * cap + ref.size].numpy()
        assert np.array_equal(got, ref)


def test_transfer_rejects_pageable_host_memory():
    n, piece = 65536, 65536
    x = torch.zeros(n, dtype=torch.int16, device="cuda")
    d, h = sz.transfer_scratch_size(n, sz.BF16, piece, True)
    dev = torch.empty(d, dtype=torch.uint8, device="cuda")
    pageable = torch.empty(h + 16, dtype=torch.uint8)  # not page-locked
    cb = sz.Codebook.make(sz.BF16, range(16))
    st = sz.splitzip_transfer(x.data_ptr(), x.data_ptr(), n, sz.BF16, cb, 65536, piece, 1, dev.data_ptr(), d,
                              pageable.data_ptr() + (-pageable.data_ptr()) % 16, h, None, None, 0)
    assert st == sz.ERR_INVALID_ARG


@pytest.mark.parametrize("compress", [True, False])
def test_transfer_with_bases_off_the_slot_alignment(compress):
    # 16-byte-aligned bases 16 bytes past an allocation (so off the slot
    # alignment, the worst case for the call's rounding up) and exactly the
    # scratch sizes reported: the output is exact and not a byte outside the
    # areas passed in is written
    n, piece = 5 * 65536 + 7, 65536
    host, x = bits(sz.BF16, n, 11)
    exps = oracle.calibrate(oracle.histogram(host, sz.BF16), sz.BF16)
    cb = sz.Codebook.make(sz.BF16, [int(e) for e in exps])
    d, h = sz.transfer_scratch_size(n, sz.BF16, piece, compress)
    pad = 16
    dev = torch.full((d + 2 * pad + 16,), 0xA7, dtype=torch.uint8, device="cuda")
    hst = torch.full((h + 2 * pad + 16,), 0x5C, dtype=torch.uint8).pin_memory()
    assert dev.data_ptr() % 16 == 0 and hst.data_ptr() % 16 == 0
    y = torch.zeros_like(x)
    link, ms = ctypes.c_uint64(0), ctypes.c_float(0.0)
    st = sz.splitzip_transfer(x.data_ptr(), y.data_ptr(), n, sz.BF16, cb if compress else None, 65536, piece,
                              int(compress), dev.data_ptr() + pad if compress else 0, d if compress else 0,
                              hst.data_ptr() + pad, h, link, ms, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == sz.OK
    assert torch.equal(y, x)
    dv, hv = dev.cpu(), hst
    assert bool((dv[:pad] == 0xA7).all()) and bool((dv[pad + d:] == 0xA7).all())
    assert bool((hv[:pad] == 0x5C).all()) and bool((hv[pad + h:] == 0x5C).all())
