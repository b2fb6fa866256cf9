"""GPU: batched encode and decode (one launch sequence for a list of
tensors), and the small-tensor path that single calls take, against the CPU
oracle.

Each item of a batch must get exactly the oracle's container of that item
(byte equality), and batched decoding must give back every item bit for bit
(tolerance 0: integer work).  Sizes straddle the thresholds where single
calls switch between the small-tensor kernels and the persistent ones, so
both paths are compared with the oracle at neighbouring sizes.
"""
import numpy as np
import pytest
import torch

import oracle
import lossless_kv_cache_gb300 as sz
from lossless_kv_cache_gb300 import workloads as W
from tests.test_gpu_parity import gpu_decode, gpu_encode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(splitzip_lib):
    assert torch.cuda.is_available()
    return splitzip_lib


def host(x, dtype):
    a = x.cpu().numpy()
    return a if dtype == sz.FP8_E5M2 else a.view(np.uint16)


def tensor(dtype, n, seed):
    if dtype == sz.BF16:
        return W.escape_stress(seed, chunks=-(-n // 65536) or 1, chunk_elems=65536, sigma=2.0)[:n]
    if dtype == sz.FP16:
        return W.kv_cache_layer_fp16(seed, 1, tokens=-(-n // 2048) or 1)[:n]
    return W.kv_cache_layer_e5m2(seed, 2, tokens=-(-n // 2048) or 1)[:n]


SIZES = [0, 1, 63, 4096, 8193, 65536, 65537, 200001, 1 << 20]


@pytest.mark.parametrize("dtype", [sz.BF16, sz.FP8_E5M2, sz.FP16])
@pytest.mark.parametrize("chunk", [65536, 4096])
def test_batch_encode_and_decode_match_oracle(dtype, chunk):
    rng = np.random.default_rng(dtype * 7 + chunk)
    sizes = [int(v) for v in rng.permutation(SIZES)]
    xs = [tensor(dtype, n, 20 + i) for i, n in enumerate(sizes)]
    allh = np.concatenate([host(x, dtype) for x in xs if x.numel()])
    exps = oracle.calibrate(oracle.histogram(allh, dtype), dtype)
    cb = sz.Codebook.make(dtype, [int(e) for e in exps])
    dev = [x.cuda() for x in xs]
    blobs = sz.encode_batch(dev, cb, dtype, chunk)
    refs = [oracle.encode(host(x, dtype), dtype, exps, chunk) for x in xs]
    for n, b, r in zip(sizes, blobs, refs):
        np.testing.assert_array_equal(b.cpu().numpy(), r, err_msg="item of %d elements" % n)
    st, ys = sz.decode_batch_status(blobs, sizes, dtype)
    assert st == sz.OK
    for x, y in zip(dev, ys):
        assert torch.equal(y, x)
    # the oracle's containers decode the same way
    st, ys = sz.decode_batch_status([torch.from_numpy(r).cuda() for r in refs], sizes, dtype)
    assert st == sz.OK and all(torch.equal(y, x) for x, y in zip(dev, ys))


def test_batch_of_256_items():
    dtype, chunk = sz.BF16, 65536
    sizes = [(i * 7919) % 30000 for i in range(256)]  # includes 0
    x = tensor(dtype, sum(sizes), 3).cuda()
    xs, lo = [], 0
    for n in sizes:  # each item its own allocation: item pointers must be 16-byte aligned
        xs.append(x[lo: lo + n].clone())
        lo += n
    cb = sz.Codebook.make(dtype, range(118, 134))
    blobs = sz.encode_batch(xs, cb, dtype, chunk)
    for i in range(0, 256, 17):
        np.testing.assert_array_equal(blobs[i].cpu().numpy(),
                                      oracle.encode(host(xs[i], dtype), dtype, np.arange(118, 134, dtype=np.uint8), chunk))
    st, ys = sz.decode_batch_status(blobs, sizes, dtype)
    assert st == sz.OK and all(torch.equal(a, b) for a, b in zip(xs, ys))


def test_batch_decode_reports_a_corrupt_item():
    dtype = sz.BF16
    xs = [tensor(dtype, n, 40 + n % 7) for n in (70000, 5000, 130000)]
    exps = oracle.calibrate(oracle.histogram(host(xs[0], dtype), dtype), dtype)
    refs = [oracle.encode(host(x, dtype), dtype, exps, 65536) for x in xs]
    bad = refs[1].copy()
    a16 = lambda v: (v + 15) // 16 * 16
    rec = a16(64 + 12) + a16((5000 + 1) // 2) + a16(5000)  # one chunk: header + index, nibbles, sign|mantissa
    assert oracle.parse_header(bad)[1].total_escapes >= 2
    bad[rec + 3: rec + 5] = bad[rec: rec + 2]  # positions not ascending
    assert oracle.decode_status(bad, 5000, dtype)[0] == oracle.CORRUPT
    blobs = [torch.from_numpy(b).cuda() for b in (refs[0], bad, refs[2])]
    st, ys = sz.decode_batch_status(blobs, [x.numel() for x in xs], dtype)
    assert st == sz.ERR_CORRUPT
    assert torch.equal(ys[0].cpu(), xs[0]) and torch.equal(ys[2].cpu(), xs[2])


@pytest.mark.parametrize("dtype", [sz.BF16, sz.FP8_E5M2])
def test_single_calls_on_both_sides_of_the_small_encode_limit(dtype):
    # 8,192 tiles: BF16 tiles are 8,192 elements, E5M2 tiles 16,384
    tile = 8192 if dtype == sz.BF16 else 16384
    limit = 8192 * tile
    big = tensor(dtype, limit + 4097, 5)
    exps = oracle.calibrate(oracle.histogram(host(big[:1 << 20], dtype), dtype), dtype)
    cb = sz.Codebook.make(dtype, [int(e) for e in exps])
    for n in (limit, limit + 4097):
        x = big[:n]
        blob = gpu_encode(x.cuda(), cb, dtype, 65536)
        np.testing.assert_array_equal(blob.cpu().numpy(), oracle.encode(host(x, dtype), dtype, exps, 65536))


@pytest.mark.parametrize("dtype", [sz.BF16, sz.FP16])
def test_single_calls_on_both_sides_of_the_small_decode_limit(dtype):
    limit = 1 << 21
    big = tensor(dtype, limit + 4097, 6)
    exps = oracle.calibrate(oracle.histogram(host(big[:1 << 20], dtype), dtype), dtype)
    for n in (limit, limit + 4097):
        x = big[:n]
        ref = oracle.encode(host(x, dtype), dtype, exps, 65536)
        st, y = gpu_decode(torch.from_numpy(ref).cuda(), n, dtype)
        assert st == sz.OK and torch.equal(y.cpu(), x)
