"""GPU: online calibration (histogram + Top-16 on the device) and the encode
that takes its codebook from device memory, against the oracle."""
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


def cases():
    few = torch.tensor([0x3F80, 0xBF80, 0x4000, 0x3F00] * 1000 + [0x4000] * 7, dtype=torch.int32).to(torch.int16)
    return [
        ("bf16 escape stress", sz.BF16, W.escape_stress(3, chunks=5, chunk_elems=65536)[:300001]),
        ("bf16 three exponents", sz.BF16, few),
        ("bf16 all patterns", sz.BF16, W.all_bf16_patterns()),
        ("bf16 llama layer", sz.BF16, W.llama_layer_kv(2, tokens=512)),
        ("e5m2 cache layer", sz.FP8_E5M2, W.kv_cache_layer_e5m2(4, 9, tokens=300)),
        ("e5m2 all patterns", sz.FP8_E5M2, W.all_e5m2_patterns()),
    ]


def host_bits(t, dtype):
    a = t.numpy()
    return a.view(np.uint16) if dtype == sz.BF16 else a


@pytest.mark.parametrize("case", range(6))
def test_device_codebook_matches_oracle(case):
    name, dtype, x = cases()[case]
    h = host_bits(x, dtype)
    ref_hist = oracle.histogram(h, dtype)
    ref_cb = oracle.calibrate(ref_hist, dtype)
    hist, dcb = sz.calibrate_device(x.cuda(), dtype)
    torch.cuda.synchronize()
    assert np.array_equal(hist.cpu().numpy().astype(np.uint64), ref_hist), name
    got = dcb.cpu().numpy()
    assert got[0] == dtype, name
    assert np.array_equal(got[1:17], ref_cb), name
    # the encode that reads it: byte-identical to the oracle's container
    bufs = sz.EncodeBuffers(x.numel(), dtype, 4096)
    sz.encode_into_device_codebook(x.cuda(), dcb, bufs)
    torch.cuda.synchronize()
    assert int(bufs.status[0]) == sz.OK, name
    blob = bufs.out[: int(bufs.size[0])].cpu().numpy()
    assert np.array_equal(blob, oracle.encode(h, dtype, ref_cb, 4096)), name


def test_uniform_histograms_give_the_first_sixteen_exponents():
    # every exponent equally frequent: ties go to the smaller exponent
    for dtype, x in ((sz.BF16, W.all_bf16_patterns()), (sz.FP8_E5M2, W.all_e5m2_patterns())):
        _, dcb = sz.calibrate_device(x.cuda(), dtype)
        assert list(dcb.cpu().numpy()[1:17]) == list(range(16))


@pytest.mark.parametrize("dtype,bad", [
    (sz.BF16, [sz.BF16] + [5] * 2 + list(range(14))),             # duplicate exponent
    (sz.BF16, [sz.FP8_E5M2] + list(range(16))),                   # codebook of the other dtype
    (sz.FP8_E5M2, [sz.FP8_E5M2] + list(range(15)) + [40]),        # E5M2 exponent >= 32
])
def test_bad_device_codebook_is_reported(dtype, bad):
    x = (W.escape_stress(1, chunks=1, chunk_elems=65536) if dtype == sz.BF16
         else W.kv_cache_layer_e5m2(1, 0, tokens=64)).cuda()
    dcb = torch.tensor(bad + [0] * (32 - len(bad)), dtype=torch.uint8, device="cuda")
    bufs = sz.EncodeBuffers(x.numel(), dtype)
    sz.encode_into_device_codebook(x, dcb, bufs)
    torch.cuda.synchronize()
    assert int(bufs.status[0]) == sz.ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", [sz.BF16, sz.FP8_E5M2])
def test_calibrate_reads_device_histogram_from_a_nonblocking_stream(dtype):
    """splitzip_exponent_histogram on a torch side stream (non-blocking), kept
    busy first so the histogram is still pending when the host returns, then
    splitzip_calibrate(d_hist, hist_is_device=1) straight away with no host
    synchronisation in between: the call must wait for the histogram."""
    x = W.escape_stress(7, chunks=16) if dtype == sz.BF16 else W.kv_cache_layer_e5m2(6, 2, tokens=2048)
    ref = oracle.calibrate(oracle.histogram(host_bits(x, dtype), dtype), dtype)
    xd = x.to("cuda")
    hist = torch.empty(256, dtype=torch.int64, device="cuda")
    # a stale histogram whose codebook differs from the true one
    stale = np.zeros(256, dtype=np.int64)
    stale[:32] = np.arange(32, 0, -1) * 1000
    hist.copy_(torch.from_numpy(stale))
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    busy = torch.empty(1 << 28, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(side):
        for i in range(40):  # ~10 GB of writes queued ahead of the histogram
            busy.fill_(i)
        assert sz.splitzip_exponent_histogram(xd.data_ptr(), xd.numel(), dtype, hist.data_ptr(),
                                              side.cuda_stream) == sz.OK
    cb = sz.Codebook()
    assert sz.splitzip_calibrate(hist.data_ptr(), 1, dtype, cb) == sz.OK
    np.testing.assert_array_equal(np.array(cb.values(), np.uint8), ref)
    assert cb.dtype == dtype
    side.synchronize()
