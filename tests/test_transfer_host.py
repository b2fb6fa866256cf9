"""The transfer path's host side (no GPU): scratch sizes and the argument
checks that splitzip_transfer makes before any GPU work."""
import ctypes

import numpy as np

import lossless_kv_cache_gb300 as sz


def a16(x):
    return (x + 15) // 16 * 16


def slot(x):
    """(slot stride, alignment): 2 MiB slots from 2 MiB on, 64 KiB below."""
    a = 2 << 20 if x >= 2 << 20 else 64 << 10
    return -(-x // a) * a, a


def test_transfer_scratch_sizes(splitzip_lib):
    for dtype, eb in ((sz.BF16, 2), (sz.FP8_E5M2, 1)):
        for n, piece in ((10 * 65536 + 5, 65536), (3 * 65536, 2 * 65536), (65536, 65536), (1, 4096),
                         (3 << 20, 1 << 20), (5 << 21, 1 << 21)):
            chunk = 65536 if piece % 65536 == 0 else 4096
            pieces = -(-n // piece)
            ring = min(4, pieces)
            cap, a = slot(sz.max_compressed_size(piece, dtype, chunk))
            ws = a16(sz.workspace_size(piece, dtype, chunk))
            d, h = sz.transfer_scratch_size(n, dtype, piece, True, chunk)
            assert d == (a - 16) + 2 * ring * cap + ws + 16 * pieces
            assert h == (a - 16) + ring * cap + 16 * pieces
            d, h = sz.transfer_scratch_size(n, dtype, piece, False, chunk)
            raw, a = slot(piece * eb)
            assert d == 0
            assert h == (a - 16) + ring * raw
    # both alignments occur above
    assert slot(sz.max_compressed_size(1 << 20, sz.FP8_E5M2, 65536))[1] == 2 << 20
    assert slot(sz.max_compressed_size(65536, sz.BF16, 65536))[1] == 64 << 10


def test_transfer_argument_errors(splitzip_lib):
    out_d, out_h = ctypes.c_uint64(0), ctypes.c_uint64(0)
    f = sz.splitzip_transfer_scratch_size
    assert f(1000, sz.BF16, 65536, 65536 + 64, 1, out_d, out_h) == sz.ERR_INVALID_ARG  # not whole chunks
    assert f(0, sz.BF16, 65536, 65536, 1, out_d, out_h) == sz.ERR_INVALID_ARG          # n = 0
    assert f(1000, sz.BF16, 65536, 0, 1, out_d, out_h) == sz.ERR_INVALID_ARG           # no piece
    assert f(1000, sz.BF16, 100, 200, 1, out_d, out_h) == sz.ERR_INVALID_ARG           # chunk not a power of 2
    cb = sz.Codebook.make(sz.BF16, range(16))
    A = 1 << 20  # a 16-aligned fake device address: no call below reaches the GPU
    n, piece = 3 * 65536, 65536
    d, h = sz.transfer_scratch_size(n, sz.BF16, piece, True)
    good = dict(d_src=A, d_dst=A, n=n, dtype=sz.BF16, cb=cb, chunk_elems=65536, piece_elems=piece, compress=1,
                d_scratch=A, d_scratch_bytes=d, h_stage=A, h_stage_bytes=h, out_link_bytes=None, out_ms=None,
                stream=0)

    def call(**kw):
        return sz.splitzip_transfer(**dict(good, **kw))

    assert call(dtype=3) == sz.ERR_INVALID_ARG
    assert call(compress=2) == sz.ERR_INVALID_ARG
    assert call(piece_elems=65536 + 16) == sz.ERR_INVALID_ARG
    assert call(d_src=None) == sz.ERR_INVALID_ARG
    assert call(d_dst=A + 8) == sz.ERR_INVALID_ARG
    assert call(h_stage=None) == sz.ERR_INVALID_ARG
    assert call(cb=None) == sz.ERR_INVALID_ARG
    assert call(d_scratch=None) == sz.ERR_INVALID_ARG
    assert call(d_scratch_bytes=d - 1) == sz.ERR_CAPACITY
    assert call(h_stage_bytes=h - 1) == sz.ERR_CAPACITY
    # host memory that is not page-locked cannot be the link's staging area
    pageable = np.zeros(h + 64, dtype=np.uint8)
    addr = pageable.ctypes.data
    addr += (-addr) % 16
    assert call(h_stage=addr) == sz.ERR_INVALID_ARG
