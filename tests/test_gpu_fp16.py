"""GPU parity for FP16 (the library's extension to the page's "other
formats", reading R16), through the C ABI, against the CPU oracle.

Byte equality of the container and bit equality of the decoded tensor
(tolerance 0: integer work) on every FP16 bit pattern at three chunk sizes,
ragged sizes, special values and an all-escape chunk, a cache workload with
the device histogram and codebook, corrupt containers, chunk shards joined by
splitzip_merge, and paged input and output (the transfer path's FP16 cases
are in test_gpu_transfer.py).
"""
import numpy as np
import pytest
import torch

import oracle
import lossless_kv_cache_gb300 as sz
from lossless_kv_cache_gb300 import workloads as W
from tests.test_gpu_parity import SIZES, gpu_decode, gpu_encode, roundtrip_vs_oracle
from tests.test_oracle_pins import corruptions

pytestmark = pytest.mark.gpu
FP16 = sz.FP16


@pytest.fixture(scope="module", autouse=True)
def _lib(splitzip_lib):
    assert torch.cuda.is_available()
    return splitzip_lib


def bits16(t):
    return t.numpy().view(np.uint16)


@pytest.mark.parametrize("chunk", [65536, 4096, 64])
def test_exhaustive_fp16(chunk):
    x = np.arange(65536, dtype=np.uint16)
    ref = roundtrip_vs_oracle(x, FP16, np.arange(16), chunk)
    assert oracle.parse_header(ref)[1].total_escapes == 32768
    roundtrip_vs_oracle(x[::-1].copy(), FP16, [15, 14, 16, 13, 17, 0, 31, 12, 18, 11, 19, 10, 20, 9, 21, 1], chunk)


@pytest.mark.parametrize("chunk", [64, 512, 4096, 65536])
def test_fp16_sizes_and_ragged_tails(chunk):
    rng = np.random.default_rng(chunk + 2)
    cb = [15, 14, 16, 13, 12, 17, 11, 18, 10, 9, 19, 8, 7, 20, 6, 5]
    for n in SIZES:
        x = bits16(W.kv_cache_layer_fp16(n, 0, tokens=-(-n // 2048) or 1))[:n].copy()
        k = rng.integers(0, max(n, 1), size=n // 20)
        x[k] = rng.integers(0, 65536, size=k.size).astype(np.uint16)
        roundtrip_vs_oracle(x, FP16, cb, chunk)


def test_fp16_special_values_and_all_escape_chunk():
    sp = bits16(W.special_fp16_patterns())
    x = np.concatenate([np.tile(sp, 4000), np.full(65536, 0x3C00, np.uint16), sp]).astype(np.uint16)
    # codebook 16..31 holds no exponent 15: the run of 1.0 is one all-escape chunk
    roundtrip_vs_oracle(x, FP16, np.arange(16, 32), 65536)
    roundtrip_vs_oracle(x, FP16, np.arange(16), 64)


def test_fp16_cache_workload_with_device_calibration():
    x = torch.cat([W.kv_cache_layer_fp16(0, l, tokens=1024) for l in (0, 5)])  # 4,194,304 elements
    cal = W.kv_cache_layer_fp16(1, 0, tokens=1024)
    cb, hist = sz.calibrate(cal.cuda(), FP16)
    ref_hist = oracle.histogram(bits16(cal), FP16)
    np.testing.assert_array_equal(hist.numpy().view(np.uint64), ref_hist)
    ref_cb = oracle.calibrate(ref_hist, FP16)
    np.testing.assert_array_equal(np.array(cb.values(), np.uint8), ref_cb)
    ref = roundtrip_vs_oracle(bits16(x), FP16, ref_cb, 65536)
    # online calibration: device histogram + Top-16, encode reading it from device memory
    xd = x.cuda()
    h, dcb = sz.calibrate_device(xd, FP16)
    own_cb = oracle.calibrate(oracle.histogram(bits16(x), FP16), FP16)
    np.testing.assert_array_equal(dcb[1:17].cpu().numpy(), own_cb)
    assert int(dcb[0]) == FP16
    bufs = sz.EncodeBuffers(x.numel(), FP16, 65536)
    sz.encode_into_device_codebook(xd, dcb, bufs)
    torch.cuda.synchronize()
    assert int(bufs.status[0]) == sz.OK
    np.testing.assert_array_equal(bufs.out[: int(bufs.size[0])].cpu().numpy(),
                                  oracle.encode(bits16(x), FP16, own_cb, 65536))
    assert ref.size > 0


def test_fp16_corrupt_containers_rejected_like_oracle():
    x = bits16(W.kv_cache_layer_fp16(11, 2, tokens=6))[:12000]
    cb = oracle.calibrate(oracle.histogram(x, FP16), FP16)
    blob = oracle.encode(x, FP16, cb, 4096)
    assert gpu_decode(torch.from_numpy(blob).cuda(), x.size, FP16)[0] == sz.OK
    cases = [c for c in corruptions_fp16(blob)]
    assert len(cases) >= 5
    for name, bad in cases:
        o_st, _ = oracle.decode_status(bad, x.size, FP16)
        st, _ = gpu_decode(torch.from_numpy(bad).cuda(), x.size, FP16)
        assert st == sz.ERR_CORRUPT and o_st == oracle.CORRUPT, name
    # read as BF16 or E5M2 the container is refused
    assert gpu_decode(torch.from_numpy(blob).cuda(), x.size, sz.BF16)[0] == sz.ERR_CORRUPT


def corruptions_fp16(blob):
    st, h = oracle.parse_header(blob)
    C, E, n = h.n_chunks, h.total_escapes, h.n
    a16 = lambda v: (v + 15) // 16 * 16
    rec = a16(64 + 12 * C) + a16((n + 1) // 2) + a16(11 * (-(-n // 8)))
    out = []
    for name, f in (("magic", lambda b: b.__setitem__(0, 0)),
                    ("codebook exponent >= 32", lambda b: b.__setitem__(32, 40)),
                    ("offset not a prefix", lambda b: b.__setitem__(64 + 8, b[64 + 8] ^ 1)),
                    ("escape exponent >= 32", lambda b: b.__setitem__(rec + 2, 0x20)),
                    ("position outside the chunk", lambda b: b[rec: rec + 2].__setitem__(slice(None), [0xFF, 0xFF])),
                    ("positions not ascending", lambda b: b[rec + 3: rec + 5].__setitem__(slice(None), b[rec: rec + 2]))):
        b = blob.copy()
        f(b)
        out.append((name, b))
    out.append(("truncated", blob[:-1].copy()))
    return out


def test_fp16_shards_merge_into_the_whole_container():
    chunk = 65536
    x = torch.cat([W.kv_cache_layer_fp16(3, l, tokens=1024) for l in (1, 2)])[: 5 * chunk + 999].cuda()
    cb = sz.Codebook.make(FP16, [int(e) for e in oracle.calibrate(oracle.histogram(bits16(x.cpu()), FP16), FP16)])
    whole = gpu_encode(x, cb, FP16, chunk).cpu().numpy()
    parts = [gpu_encode(x[a:b], cb, FP16, chunk).cpu().numpy() for a, b in ((0, 2 * chunk), (2 * chunk, 3 * chunk),
                                                                             (3 * chunk, x.numel()))]
    np.testing.assert_array_equal(sz.merge(parts), whole)
    np.testing.assert_array_equal(whole, oracle.encode(bits16(x.cpu()), FP16, np.array(cb.values(), np.uint8), chunk))


@pytest.mark.parametrize("page_elems,chunk", [(16384, 65536), (8192, 4096)])
def test_fp16_paged_encode_and_decode(page_elems, chunk):
    pool_pages = 40
    pool = W.kv_cache_layer_fp16(9, 3, tokens=pool_pages * page_elems // 2048).cuda()
    g = torch.Generator().manual_seed(page_elems)
    pages = torch.randperm(pool_pages, generator=g)[:29].to(torch.int32)
    gathered = pool.view(pool_pages, page_elems)[pages.long().cuda()].reshape(-1)
    cb_exps = oracle.calibrate(oracle.histogram(bits16(gathered.cpu()), FP16), FP16)
    cb = sz.Codebook.make(FP16, [int(e) for e in cb_exps])
    n = pages.numel() * page_elems
    bufs = sz.EncodeBuffers(n, FP16, chunk)
    sz.encode_paged_into(pool, pages.cuda(), page_elems, cb, bufs)
    torch.cuda.synchronize()
    assert int(bufs.status[0]) == sz.OK
    blob = bufs.out[: int(bufs.size[0])]
    np.testing.assert_array_equal(blob.cpu().numpy(), oracle.encode(bits16(gathered.cpu()), FP16, cb_exps, chunk))
    # decode into other pages of a fresh pool: exactly the listed pages change
    dst_pages = torch.randperm(pool_pages, generator=g)[:29].to(torch.int32).cuda()
    out_pool = torch.full((pool_pages * page_elems,), 0x1234, dtype=torch.int16, device="cuda")
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    sz.decode_paged_into(blob, blob.numel(), out_pool, dst_pages, page_elems, FP16, status)
    torch.cuda.synchronize()
    assert int(status[0]) == sz.OK
    view = out_pool.view(pool_pages, page_elems)
    assert torch.equal(view[dst_pages.long()].reshape(-1), gathered)
    untouched = torch.ones(pool_pages, dtype=torch.bool, device="cuda")
    untouched[dst_pages.long()] = False
    assert bool((view[untouched] == 0x1234).all())

