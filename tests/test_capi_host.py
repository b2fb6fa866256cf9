"""C ABI checks that need no GPU: the library loads and exports every entry
point include/splitzip.h declares, and the host-side logic (sizes, argument
checks, codebook calibration, header parsing) agrees with the CPU oracle."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import lossless_kv_cache_gb300 as sz
from lossless_kv_cache_gb300 import workloads as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "splitzip.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(splitzip_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("splitzip_calibrate", "splitzip_max_compressed_size", "splitzip_encode", "splitzip_decode",
                     "splitzip_exponent_histogram", "splitzip_parse_header"):
        assert required in names


def test_library_exports_every_declared_symbol(splitzip_lib):
    for name in declared_functions():
        assert hasattr(splitzip_lib, name), name
    # the binding mirrors the C names
    assert set(sz.SIGNATURES) == set(declared_functions())
    for name in declared_functions():
        assert callable(getattr(sz, name))


def test_status_strings(splitzip_lib):
    assert sz.splitzip_status_string(sz.OK) == "ok"
    assert "corrupt" in sz.splitzip_status_string(sz.ERR_CORRUPT)
    assert sz.splitzip_status_string(99) == "unknown status"


@pytest.mark.parametrize("dtype", [sz.BF16, sz.FP8_E5M2, sz.FP16])
@pytest.mark.parametrize("chunk", [64, 256, 8192, 65536])
def test_sizes_match_oracle(splitzip_lib, dtype, chunk):
    for n in (0, 1, 2, 7, 31, 64, 65, 1000, 65537, 2**31 + 3, 2**32):
        for E in {0, 1, n // 3, n}:
            if E > n:
                continue
            assert sz.compressed_size(n, dtype, chunk, E) == oracle.container_size(n, dtype, chunk, E)
        assert sz.max_compressed_size(n, dtype, chunk) == oracle.max_container_size(n, dtype, chunk)


def test_workspace_size(splitzip_lib):
    # per-group totals, per-(tile, consumer warp) counts, per-tile first
    # record indices, then a staging slot of tile_elems 4-byte records per
    # tile; a tile is 16 KB of input (8,192 BF16 or 16,384 E5M2 elements) or
    # the chunk when chunks are smaller
    a16 = lambda x: -(-x // 16) * 16
    head = lambda tiles: a16(a16(a16(4 * -(-tiles // 256)) + 32 * tiles) + 8 * tiles)
    n = 5 * 8192 + 3
    assert sz.workspace_size(n, sz.BF16, 65536) == head(6) + 4 * 6 * 8192
    assert sz.workspace_size(n, sz.FP8_E5M2, 65536) == head(3) + 4 * 3 * 16384
    tiles = -(-n // 1024)  # tiles = chunks when chunks are smaller than a tile
    assert sz.workspace_size(n, sz.BF16, 1024) == head(tiles) + 4 * tiles * 1024
    assert sz.workspace_size(n, sz.FP8_E5M2, 1024) == head(tiles) + 4 * tiles * 1024
    n = 300 * 8192 * 2
    assert sz.workspace_size(n, sz.BF16, 65536) == head(600) + 4 * 600 * 8192
    assert sz.workspace_size(0, sz.BF16, 65536) == 0


def test_size_argument_errors(splitzip_lib):
    out = ctypes.c_uint64(0)
    assert sz.splitzip_max_compressed_size(10, 3, 65536, out) == sz.ERR_INVALID_ARG      # dtype
    assert sz.splitzip_max_compressed_size(10, 0, 100, out) == sz.ERR_INVALID_ARG        # not pow2
    assert sz.splitzip_max_compressed_size(10, 0, 32, out) == sz.ERR_INVALID_ARG         # < 64
    assert sz.splitzip_max_compressed_size(10, 0, 131072, out) == sz.ERR_INVALID_ARG     # > 65536
    assert sz.splitzip_compressed_size(10, 0, 64, 11, out) == sz.ERR_INVALID_ARG         # E > n
    assert sz.splitzip_max_compressed_size(2**49, 0, 65536, out) == sz.ERR_UNSUPPORTED


def _cb(dtype, exps=None):
    return sz.Codebook.make(dtype, exps if exps is not None else range(16))


def test_encode_argument_errors_are_host_side(splitzip_lib):
    n, chunk = 1000, 64
    cap = sz.max_compressed_size(n, 0, chunk)
    ws = sz.workspace_size(n, 0, chunk)
    A = 1 << 20  # a 16-aligned fake device address: no call below reaches the GPU
    good = dict(d_in=A, n=n, dtype=0, cb=_cb(0), chunk_elems=chunk, d_out=A, out_capacity=cap, d_ws=A,
                ws_bytes=ws, d_out_size=A, d_status=A, stream=0)

    def call(**kw):
        args = dict(good, **kw)
        return sz.splitzip_encode(**args)

    assert call(dtype=5) == sz.ERR_INVALID_ARG
    assert call(chunk_elems=96) == sz.ERR_INVALID_ARG
    assert call(d_in=None) == sz.ERR_INVALID_ARG
    assert call(d_in=A + 8) == sz.ERR_INVALID_ARG          # misaligned
    assert call(d_out=None) == sz.ERR_INVALID_ARG
    assert call(d_out_size=None) == sz.ERR_INVALID_ARG
    assert call(d_status=None) == sz.ERR_INVALID_ARG
    assert call(out_capacity=cap - 1) == sz.ERR_CAPACITY
    assert call(ws_bytes=ws - 1) == sz.ERR_CAPACITY
    assert call(d_ws=None) == sz.ERR_INVALID_ARG
    assert call(cb=_cb(1)) == sz.ERR_INVALID_ARG            # codebook of another dtype
    assert call(cb=_cb(0, [1] * 16)) == sz.ERR_INVALID_ARG  # duplicate exponents
    assert call(dtype=1, cb=_cb(1, range(20, 36))) == sz.ERR_INVALID_ARG  # E5M2 exponent >= 32


def test_decode_argument_errors_are_host_side(splitzip_lib):
    A = 1 << 20
    assert sz.splitzip_decode(None, 64, A, 10, 0, A, 0) == sz.ERR_INVALID_ARG
    assert sz.splitzip_decode(A + 4, 64, A, 10, 0, A, 0) == sz.ERR_INVALID_ARG
    assert sz.splitzip_decode(A, 64, A, 10, 3, A, 0) == sz.ERR_INVALID_ARG
    assert sz.splitzip_decode(A, 64, A, 10, 0, None, 0) == sz.ERR_INVALID_ARG
    assert sz.splitzip_decode(A, 63, A, 10, 0, A, 0) == sz.ERR_CORRUPT


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_call_without_gpu_reports_cuda_error(splitzip_lib):
    A = 1 << 20
    st = sz.splitzip_decode(A, 1 << 20, A, 10, 0, A, 0)
    assert st in (sz.ERR_CUDA, sz.ERR_UNSUPPORTED)


@pytest.mark.parametrize("seed", range(8))
def test_calibrate_host_histogram_matches_oracle(splitzip_lib, seed):
    rng = np.random.default_rng(seed)
    for dtype, bins in ((sz.BF16, 256), (sz.FP8_E5M2, 32)):
        h = np.zeros(256, dtype=np.uint64)
        support = rng.choice(bins, size=rng.integers(1, bins + 1), replace=False)
        h[support] = rng.integers(0, 4, size=support.size) * rng.integers(1, 1 << 40)
        cb = sz.Codebook()
        assert sz.splitzip_calibrate(h.ctypes.data, 0, dtype, cb) == sz.OK
        assert cb.dtype == dtype
        np.testing.assert_array_equal(np.array(cb.values(), np.uint8), oracle.calibrate(h, dtype))


def test_calibrate_rejects_bad_e5m2_histogram(splitzip_lib):
    h = np.zeros(256, dtype=np.uint64)
    h[33] = 1
    assert sz.splitzip_calibrate(h.ctypes.data, 0, sz.FP8_E5M2, sz.Codebook()) == sz.ERR_INVALID_ARG


def test_parse_header_matches_oracle(splitzip_lib):
    x = W.escape_stress(2, chunks=3, chunk_elems=4096).numpy().view(np.uint16)[:10001]
    cb = oracle.calibrate(oracle.histogram(x, 0), 0)
    blob = oracle.encode(x, 0, cb, 2048)
    h = sz.parse_header(blob)
    st, ref = oracle.parse_header(blob)
    assert st == oracle.OK
    assert (h.n_elems, h.total_escapes, h.size, h.chunk_elems, h.n_chunks, h.dtype) == (
        ref.n, ref.total_escapes, ref.size, ref.chunk_elems, ref.n_chunks, ref.dtype)
    assert list(h.codebook) == list(ref.codebook)
    assert h.size == blob.size
    # header-level corruptions are rejected like the oracle rejects them
    from tests.test_oracle_pins import corruptions
    for name, bad in corruptions(blob):
        o_st, _ = oracle.parse_header(bad)
        buf = np.ascontiguousarray(bad)
        st = sz.splitzip_parse_header(buf.ctypes.data, buf.size, sz.Header())
        assert (st == sz.OK) == (o_st == oracle.OK), name


def test_pointer_arguments_reject_non_addresses(splitzip_lib):
    # a str or bytes must never reach the library as an address (plain
    # c_void_p would pass the address of the object's host buffer)
    cb = sz.Codebook.make(sz.BF16, range(16))
    for bad in ("encode", b"\x00" * 16, 1.5, True):
        with pytest.raises(ctypes.ArgumentError):
            sz.splitzip_encode(1 << 20, 8, sz.BF16, cb, 65536, bad, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 0)
        with pytest.raises(ctypes.ArgumentError):
            sz.splitzip_decode(bad, 1 << 20, 1 << 20, 8, sz.BF16, 1 << 20, 0)
    # integers, None and objects with data_ptr() are addresses
    class T:
        def data_ptr(self):
            return 1 << 20
    assert sz._Address.from_param(None) is None
    assert sz._Address.from_param(T()).value == 1 << 20
    assert sz._Address.from_param(1 << 40).value == 1 << 40


def test_online_calibration_argument_errors(splitzip_lib):
    A = 1 << 20  # fake device addresses: every call below fails before the GPU
    assert sz.splitzip_calibrate_device(A, 100, sz.BF16, A, None, 0) == sz.ERR_INVALID_ARG      # no codebook
    assert sz.splitzip_calibrate_device(A, 100, 7, A, A, 0) == sz.ERR_INVALID_ARG               # dtype
    assert sz.splitzip_calibrate_device(A, 100, sz.BF16, A + 8, A, 0) == sz.ERR_INVALID_ARG     # misaligned
    ws = sz.workspace_size(1000, sz.BF16, 64)
    cap = sz.max_compressed_size(1000, sz.BF16, 64)
    f = sz.splitzip_encode_device_codebook
    assert f(A, 1000, sz.BF16, None, 64, A, cap, A, ws, A, A, 0) == sz.ERR_INVALID_ARG          # no codebook
    assert f(A, 1000, sz.BF16, A, 96, A, cap, A, ws, A, A, 0) == sz.ERR_INVALID_ARG             # chunk
    assert f(A, 1000, sz.BF16, A, 64, A, cap - 1, A, ws, A, A, 0) == sz.ERR_CAPACITY            # output


def test_paged_argument_errors(splitzip_lib):
    A = 1 << 20  # fake device addresses: every call below fails before the GPU
    cb = sz.Codebook.make(sz.BF16, range(16))
    n_pages, page = 4, 16384
    cap = sz.max_compressed_size(n_pages * page, sz.BF16, 65536)
    ws = sz.workspace_size(n_pages * page, sz.BF16, 65536)
    f = sz.splitzip_encode_paged
    ok = (A, 8, A, n_pages, page, sz.BF16, cb, 65536, A, cap, A, ws, A, A, 0)

    def call(**kw):
        args = list(ok)
        names = ["pool", "pool_pages", "pages", "n_pages", "page_elems", "dtype", "cb", "chunk", "out", "cap", "ws",
                 "ws_bytes", "size", "status", "stream"]
        for k, v in kw.items():
            args[names.index(k)] = v
        return f(*args)

    assert call(page_elems=3 * 8192) == sz.ERR_INVALID_ARG      # not a power of two
    assert call(page_elems=4096) == sz.ERR_INVALID_ARG          # smaller than a BF16 tile at chunk 65,536
    assert call(pages=None) == sz.ERR_INVALID_ARG
    assert call(pages=A + 2) == sz.ERR_INVALID_ARG              # misaligned page table
    assert call(n_pages=0) == sz.ERR_INVALID_ARG
    assert call(pool_pages=0) == sz.ERR_INVALID_ARG
    assert call(cap=cap - 1) == sz.ERR_CAPACITY
    d = sz.splitzip_decode_paged
    assert d(A, 1 << 20, A, 8, A, 4, 24, sz.BF16, A, 0) == sz.ERR_INVALID_ARG   # not a power of two
    assert d(A, 1 << 20, A, 8, A, 4, 8, sz.BF16, A, 0) == sz.ERR_INVALID_ARG    # fewer than 16 elements
    assert d(A, 1 << 20, A, 8, None, 4, 4096, sz.BF16, A, 0) == sz.ERR_INVALID_ARG
    assert d(A, 1 << 20, A, 0, A, 4, 4096, sz.BF16, A, 0) == sz.ERR_INVALID_ARG


def test_ablation_argument_errors(splitzip_lib):
    A = 1 << 20  # fake device addresses: every call below fails before the GPU
    out = ctypes.c_uint64(0)
    assert sz.splitzip_ablation_max_size(100, sz.BF16, 64, 3, out) == sz.ERR_INVALID_ARG
    assert sz.splitzip_ablation_max_size(100, sz.BF16, 96, 1, out) == sz.ERR_INVALID_ARG
    assert sz.splitzip_ablation_max_size(100, sz.BF16, 64, 1, out) == sz.OK
    # two chunks: 64 + 2 * 12 -> 96; 3 * 13 code bytes -> 48; 100 sign|mantissa bytes -> 112; 300 escape bytes
    assert out.value == 96 + 48 + 112 + 300
    cap = sz.ablation_max_size(1000, sz.BF16, 1, 64)
    f = sz.splitzip_ablation_encode
    good = sz.Codebook.make(sz.BF16, list(range(8)) + [0] * 8)
    assert f(A, 1000, sz.BF16, good, 64, 1, A, cap - 1, A, A, 0) == sz.ERR_CAPACITY
    tail = sz.Codebook.make(sz.BF16, list(range(8)) + [0] * 7 + [9])           # byte 15 must be zero
    assert f(A, 1000, sz.BF16, tail, 64, 1, A, cap, A, A, 0) == sz.ERR_INVALID_ARG
    dup = sz.Codebook.make(sz.BF16, [3, 3] + list(range(4, 10)) + [0] * 8)       # duplicate exponent
    assert f(A, 1000, sz.BF16, dup, 64, 1, A, cap, A, A, 0) == sz.ERR_INVALID_ARG
    assert f(A, 1000, sz.FP8_E5M2, good, 64, 1, A, cap, A, A, 0) == sz.ERR_INVALID_ARG  # other dtype
    assert sz.splitzip_ablation_decode(A, 1 << 20, A, 10, sz.BF16, 5, A, 0) == sz.ERR_INVALID_ARG
    assert sz.splitzip_ablation_decode(A, 63, A, 10, sz.BF16, 1, A, 0) == sz.ERR_CORRUPT


def test_selftest_argument_errors(splitzip_lib):
    # the bounded-wait self-test checks its arguments before any CUDA call
    A = 1 << 20  # never dereferenced: the checks come first
    assert sz.splitzip_selftest_bounded_wait(0, A, None, 0) == sz.ERR_INVALID_ARG
    assert sz.splitzip_selftest_bounded_wait(3_000_000_000, A, None, 0) == sz.ERR_INVALID_ARG
    assert sz.splitzip_selftest_bounded_wait(100, None, None, 0) == sz.ERR_INVALID_ARG
    assert sz.splitzip_selftest_bounded_wait(100, A + 2, None, 0) == sz.ERR_INVALID_ARG
    assert sz.splitzip_selftest_bounded_wait(100, A, A + 4, 0) == sz.ERR_INVALID_ARG


def test_fp16_calibrate_and_ablation_refusal(splitzip_lib):
    # FP16 histograms have 32 bins; the ablation formats are defined for BF16 and E5M2 only
    h = np.zeros(256, dtype=np.uint64)
    h[[3, 15, 16, 14]] = [5, 900, 400, 400]
    cb = sz.Codebook()
    assert sz.splitzip_calibrate(h.ctypes.data, 0, sz.FP16, cb) == sz.OK
    np.testing.assert_array_equal(np.array(cb.values(), np.uint8), oracle.calibrate(h, sz.FP16))
    h[40] = 1
    assert sz.splitzip_calibrate(h.ctypes.data, 0, sz.FP16, cb) == sz.ERR_INVALID_ARG
    out = ctypes.c_uint64(0)
    assert sz.splitzip_ablation_max_size(100, sz.FP16, 65536, 1, out) == sz.ERR_INVALID_ARG


def test_batch_workspace_and_argument_errors(splitzip_lib):
    ns = [0, 1, 70000, 1 << 20]
    arr = (ctypes.c_uint64 * 4)(*ns)
    out = ctypes.c_uint64(0)
    assert sz.splitzip_encode_batch_workspace_size(arr, 4, sz.BF16, 65536, out) == sz.OK
    assert out.value == sum(-(-sz.workspace_size(n, sz.BF16) // 256) * 256 for n in ns)
    assert sz.splitzip_encode_batch_workspace_size(arr, 0, sz.BF16, 65536, out) == sz.ERR_INVALID_ARG
    assert sz.splitzip_encode_batch_workspace_size(arr, 257, sz.BF16, 65536, out) == sz.ERR_INVALID_ARG
    big = (ctypes.c_uint64 * 1)(sz.MAX_BATCH_ITEM_ELEMS + 1)
    assert sz.splitzip_encode_batch_workspace_size(big, 1, sz.BF16, 65536, out) == sz.ERR_UNSUPPORTED

    A = 1 << 20  # never dereferenced: the checks come first
    cb = sz.Codebook.make(sz.BF16, range(16))
    cap = sz.max_compressed_size(1000, sz.BF16)
    ws = sz.batch_workspace_size([1000], sz.BF16)

    def enc(**kw):
        it = dict(d_in=A, n=1000, d_out=A, out_capacity=cap, d_out_size=A)
        it.update({k: v for k, v in kw.items() if k in it})
        items = (sz.EncodeItem * 1)(sz.EncodeItem(it["d_in"], it["n"], it["d_out"], it["out_capacity"], it["d_out_size"]))
        return sz.splitzip_encode_batch(items, kw.get("count", 1), kw.get("dtype", sz.BF16), kw.get("cb", cb), 65536,
                                        A, kw.get("ws", ws), kw.get("status", A), 0)

    assert enc(count=0) == sz.ERR_INVALID_ARG
    assert enc(dtype=3) == sz.ERR_INVALID_ARG
    assert enc(cb=sz.Codebook.make(sz.FP8_E5M2, range(16))) == sz.ERR_INVALID_ARG
    assert enc(d_in=A + 8) == sz.ERR_INVALID_ARG
    assert enc(d_out=None) == sz.ERR_INVALID_ARG
    assert enc(d_out_size=A + 4) == sz.ERR_INVALID_ARG
    assert enc(out_capacity=cap - 1) == sz.ERR_CAPACITY
    assert enc(ws=ws - 1) == sz.ERR_CAPACITY
    assert enc(status=None) == sz.ERR_INVALID_ARG
    assert enc(n=sz.MAX_BATCH_ITEM_ELEMS + 1, out_capacity=1 << 40) == sz.ERR_UNSUPPORTED

    def dec(**kw):
        it = dict(d_in=A, in_bytes=1 << 20, d_out=A, n=1000)
        it.update({k: v for k, v in kw.items() if k in it})
        items = (sz.DecodeItem * 1)(sz.DecodeItem(it["d_in"], it["in_bytes"], it["d_out"], it["n"]))
        return sz.splitzip_decode_batch(items, kw.get("count", 1), kw.get("dtype", sz.BF16), kw.get("status", A), 0)

    assert dec(count=257) == sz.ERR_INVALID_ARG
    assert dec(dtype=7) == sz.ERR_INVALID_ARG
    assert dec(d_in=A + 2) == sz.ERR_INVALID_ARG
    assert dec(d_out=A + 2) == sz.ERR_INVALID_ARG
    assert dec(in_bytes=63) == sz.ERR_CORRUPT
    assert dec(n=sz.MAX_BATCH_ITEM_ELEMS + 1) == sz.ERR_UNSUPPORTED
    assert dec(status=A + 1) == sz.ERR_INVALID_ARG
