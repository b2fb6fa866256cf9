"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer/bit work, so the bar is byte equality of the container and bit
equality of the decoded tensor (tolerance 0).  Small and medium workloads are
compared whole; the two 4.3 GB workloads are compared chunk by chunk, every
chunk (the oracle encodes blocks of whole chunks on host threads; a chunk's
sections do not depend on other chunks), with the header and padding bytes
checked against the layout formula, plus properties that hold at any size:
the index is the prefix of the counts, E equals the exponent mass outside the
codebook (counted by torch.bincount, not by this library), the size formula,
and decode(encode(x)) == x; an oracle-built container of one whole layer is
decoded on the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
import lossless_kv_cache_gb300 as sz
from lossless_kv_cache_gb300 import workloads as W
from tests import goldens
from tests.test_oracle_pins import corruptions

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib(splitzip_lib):
    assert torch.cuda.is_available()
    return splitzip_lib


def a16(x):
    return (x + 15) // 16 * 16


def np_bits(t, dtype):
    a = t.cpu().numpy()
    return a if dtype == sz.FP8_E5M2 else a.view(np.uint16)


def sm_stream_bytes(n, dtype):
    return n if dtype == sz.BF16 else (11 if dtype == sz.FP16 else 3) * (-(-n // 8))


def gpu_encode(x_dev, cb, dtype, chunk, dirty=True):
    bufs = sz.EncodeBuffers(x_dev.numel(), dtype, chunk)
    if dirty:  # every byte of the container must be written by the encoder
        bufs.out.fill_(0xA5)
        bufs.ws.fill_(0x5A)
        bufs.status.fill_(-1)
    sz.encode_into(x_dev, cb, bufs)
    torch.cuda.synchronize()
    assert int(bufs.status[0]) == sz.OK
    return bufs.out[: int(bufs.size[0])]


def gpu_decode(blob_dev, n, dtype, in_bytes=None):
    out = torch.empty(max(n, 1), dtype=torch.uint8 if dtype == sz.FP8_E5M2 else torch.int16, device=DEV)
    status = torch.full((4,), -1, dtype=torch.int32, device=DEV)
    sz.decode_into(blob_dev, blob_dev.numel() if in_bytes is None else in_bytes, out, n, dtype, status)
    torch.cuda.synchronize()
    return int(status[0]), out[:n]


def codebook_of(exps, dtype):
    return sz.Codebook.make(dtype, [int(e) for e in exps])


def roundtrip_vs_oracle(bits, dtype, cb_exps, chunk):
    """Encode on the GPU and with the oracle; bytes must match; both
    containers decode on the GPU to the input."""
    x = torch.from_numpy(bits if dtype == sz.FP8_E5M2 else bits.view(np.int16)).to(DEV)
    blob = gpu_encode(x, codebook_of(cb_exps, dtype), dtype, chunk)
    ref = oracle.encode(bits, dtype, np.asarray(cb_exps, np.uint8), chunk)
    got = blob.cpu().numpy()
    assert got.size == ref.size
    if not np.array_equal(got, ref):
        bad = np.nonzero(got != ref)[0]
        raise AssertionError("container differs at %d bytes, first at %s" % (bad.size, bad[:8]))
    st, y = gpu_decode(blob, bits.size, dtype)
    assert st == sz.OK
    assert torch.equal(y, x)
    st, y2 = gpu_decode(torch.from_numpy(ref).to(DEV), bits.size, dtype)
    assert st == sz.OK and torch.equal(y2, x)
    return ref


# ------------------------------------------------------------------ goldens

@pytest.mark.parametrize("name", goldens.CONTAINER_FIXTURES)
def test_golden_containers(name):
    fx = goldens.load_container(name)
    ref = roundtrip_vs_oracle(fx["input"], fx["dtype"], fx["codebook"], fx["chunk_elems"])
    np.testing.assert_array_equal(ref, fx["expected"])


# ------------------------------------------------------------ exhaustive

@pytest.mark.parametrize("chunk", [65536, 4096, 64])
def test_exhaustive_bf16(chunk):
    roundtrip_vs_oracle(np.arange(65536, dtype=np.uint16), sz.BF16, np.arange(16), chunk)
    # and a codebook around the common exponents, in frequency order
    roundtrip_vs_oracle(np.arange(65536, dtype=np.uint16)[::-1].copy(), sz.BF16,
                        [127, 126, 128, 125, 129, 0, 255, 124, 130, 1, 254, 123, 131, 2, 122, 132], chunk)


@pytest.mark.parametrize("chunk", [64, 8192])
def test_exhaustive_e5m2(chunk):
    x = np.tile(np.arange(256, dtype=np.uint8), 300)
    roundtrip_vs_oracle(x, sz.FP8_E5M2, np.arange(16), chunk)
    roundtrip_vs_oracle(x, sz.FP8_E5M2, [15, 14, 16, 13, 17, 0, 31, 12, 18, 11, 19, 10, 20, 9, 21, 1], chunk)


# --------------------------------------------------------- sizes and tails

SIZES = [0, 1, 2, 7, 8, 9, 15, 16, 17, 31, 33, 63, 64, 65, 127, 511, 512, 513, 4095, 8191, 8192, 8193,
         16385, 65535, 65536, 65537, 131073, 270000]


@pytest.mark.parametrize("dtype", [sz.BF16, sz.FP8_E5M2])
@pytest.mark.parametrize("chunk", [64, 512, 4096, 65536])
def test_sizes_and_ragged_tails(dtype, chunk):
    rng = np.random.default_rng(chunk + dtype)
    for n in SIZES:
        if dtype == sz.BF16:
            # mostly common exponents plus a sprinkle of arbitrary patterns
            x = (W.kv_tile_k_only(n, tokens=-(-n // 1024) or 1).numpy().view(np.uint16)[:n]).copy()
            k = rng.integers(0, max(n, 1), size=n // 20)
            x[k] = rng.integers(0, 65536, size=k.size).astype(np.uint16)
            cb = [127, 126, 128, 125, 124, 129, 123, 130, 122, 131, 121, 132, 120, 119, 133, 118]
        else:
            x = rng.integers(0, 256, size=n).astype(np.uint8)
            cb = [15, 14, 16, 13, 17, 12, 18, 11, 19, 10, 20, 9, 21, 8, 22, 7]
        roundtrip_vs_oracle(x, dtype, cb, chunk)


def test_special_values_and_all_escape_chunk():
    sp = W.special_bf16_patterns().numpy().view(np.uint16)
    x = np.concatenate([np.tile(sp, 4000), np.full(65536, 0x3F80, np.uint16), sp]).astype(np.uint16)
    # codebook without 127: the 65,536-element run of 1.0 is one all-escape chunk
    roundtrip_vs_oracle(x, sz.BF16, np.arange(16), 65536)
    roundtrip_vs_oracle(x, sz.BF16, np.arange(16), 64)
    e = W.special_e5m2_patterns().numpy()
    roundtrip_vs_oracle(np.tile(e, 5000), sz.FP8_E5M2, np.arange(16, 32), 4096)


# ---------------------------------------------------- the workloads, whole

SMALL_WORKLOADS = ["kv_tile_1x1024x8x128_bf16", "llama_layer_2x8192x8x128_bf16", "escape_stress_64x65536_bf16"]


@pytest.mark.parametrize("name", SMALL_WORKLOADS)
def test_workload_whole(name):
    dtype = W.dtype_of(name)
    xc = W.make(name, 0)
    calc = W.calibration_tensor(name)
    # calibration: device histogram and codebook against the oracle's
    cb, hist = sz.calibrate(calc.to(DEV), dtype)
    ref_hist = oracle.histogram(np_bits(calc, dtype), dtype)
    np.testing.assert_array_equal(hist.numpy().view(np.uint64), ref_hist)
    ref_cb = oracle.calibrate(ref_hist, dtype)
    np.testing.assert_array_equal(np.array(cb.values(), np.uint8), ref_cb)
    roundtrip_vs_oracle(np_bits(xc, dtype), dtype, ref_cb, 65536)


def test_escape_stress_in_band_sigma():
    x = W.escape_stress(0, sigma=2.0)
    cal = W.escape_stress(1, sigma=2.0)
    ref_cb = oracle.calibrate(oracle.histogram(np_bits(cal, 0), 0), 0)
    ref = roundtrip_vs_oracle(np_bits(x, 0), 0, ref_cb, 65536)
    E = oracle.parse_header(ref)[1].total_escapes
    assert 0.01 < E / x.numel() < 0.05


def test_histogram_e5m2_and_tail():
    x = W.kv_cache_layer_e5m2(4, 3, tokens=33)[:-5]  # n not a multiple of 16
    cb, hist = sz.calibrate(x.to(DEV), sz.FP8_E5M2)
    np.testing.assert_array_equal(hist.numpy().view(np.uint64), oracle.histogram(x.numpy(), sz.FP8_E5M2))
    y = W.kv_tile_k_only(3, tokens=5)[:-3]
    _, h2 = sz.calibrate(y.to(DEV), sz.BF16)
    np.testing.assert_array_equal(h2.numpy().view(np.uint64), oracle.histogram(np_bits(y, 0), 0))


# ----------------------------------------------------- streams and reuse

def test_side_stream_and_reused_workspace():
    """Encode on a non-default stream twice into the same buffers (the
    workspace keeps the first call's look-back state); both match the oracle."""
    x = W.escape_stress(5, chunks=5, chunk_elems=65536)[:300001]
    bits = np_bits(x, 0)
    cb_exps = np.arange(120, 136)
    ref = oracle.encode(bits, 0, cb_exps.astype(np.uint8), 65536)
    xd = x.to(DEV)
    bufs = sz.EncodeBuffers(x.numel(), 0, 65536)
    s = torch.cuda.Stream()
    for fill in (0x11, 0xEE):
        bufs.out.fill_(fill)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            sz.encode_into(xd, codebook_of(cb_exps, 0), bufs, stream=s)
        s.synchronize()
        assert int(bufs.status[0]) == sz.OK
        got = bufs.out[: int(bufs.size[0])].cpu().numpy()
        np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------- corruption

def test_corrupt_containers_rejected_like_oracle():
    x = W.escape_stress(11, chunks=3, chunk_elems=4096).numpy().view(np.uint16)[:12000]
    cb = oracle.calibrate(oracle.histogram(x, 0), 0)
    blob = oracle.encode(x, 0, cb, 4096)
    st, _ = gpu_decode(torch.from_numpy(blob).to(DEV), x.size, 0)
    assert st == sz.OK
    for name, bad in corruptions(blob):
        o_st, _ = oracle.decode_status(bad, x.size, 0)
        st, _ = gpu_decode(torch.from_numpy(bad).to(DEV), x.size, 0)
        assert st == sz.ERR_CORRUPT and o_st == oracle.CORRUPT, name
    # caller's n or dtype disagreeing with the header
    d = torch.from_numpy(blob).to(DEV)
    assert gpu_decode(d, x.size - 1, 0)[0] == sz.ERR_CORRUPT
    assert gpu_decode(d, x.size, 1)[0] == sz.ERR_CORRUPT
    # a status word left at an error by an earlier call is reset
    assert gpu_decode(d, x.size, 0)[0] == sz.OK


# --------------------------------------------- sharding by whole chunks

def test_chunk_aligned_shards_match_single_container():
    """Chunks are independent: encoding two chunk-aligned halves separately
    gives containers whose dense sections and per-chunk escapes are the
    corresponding slices of the single-container encode."""
    chunk = 65536
    x = W.make("escape_stress_64x65536_bf16", 0)[: 10 * chunk + 777].to(DEV)
    cb = codebook_of(np.arange(118, 134), 0)
    whole = gpu_encode(x, cb, 0, chunk).cpu().numpy()
    parts = [gpu_encode(x[: 6 * chunk], cb, 0, chunk).cpu().numpy(), gpu_encode(x[6 * chunk:], cb, 0, chunk).cpu().numpy()]
    hw = sz.parse_header(whole)
    hp = [sz.parse_header(p) for p in parts]
    assert hw.total_escapes == sum(h.total_escapes for h in hp)
    nw = whole[hw.nibble_off: hw.nibble_off + (x.numel() + 1) // 2]
    np.testing.assert_array_equal(nw, np.concatenate([parts[0][hp[0].nibble_off: hp[0].nibble_off + 3 * chunk],
                                                      parts[1][hp[1].nibble_off: hp[1].nibble_off + (hp[1].n_elems + 1) // 2]]))
    cw = whole[hw.counts_off: hw.counts_off + 4 * hw.n_chunks].view(np.uint32)
    cp = np.concatenate([p[h.counts_off: h.counts_off + 4 * h.n_chunks].view(np.uint32) for p, h in zip(parts, hp)])
    np.testing.assert_array_equal(cw, cp)
    E0 = hp[0].total_escapes
    rw = whole[hw.escrec_off: hw.escrec_off + 3 * hw.total_escapes]
    np.testing.assert_array_equal(rw[: 3 * E0], parts[0][hp[0].escrec_off: hp[0].escrec_off + 3 * E0])
    np.testing.assert_array_equal(rw[3 * E0:], parts[1][hp[1].escrec_off: hp[1].size])
    # and the library's merge joins the two shard containers into the whole one
    np.testing.assert_array_equal(sz.merge(parts), whole)


# ------------------------------------------- the 4.3 GB workloads, whole

def _layout(n, dtype, chunk, E):
    C = -(-n // chunk)
    nib = a16(64 + 12 * C)
    sm = nib + a16((n + 1) // 2)
    sm_bytes = sm_stream_bytes(n, dtype)
    rec = sm + a16(sm_bytes)
    return dict(C=C, index=64, counts=64 + 8 * C, index_end=64 + 12 * C, nib=nib, sm=sm, sm_bytes=sm_bytes,
                rec=rec, size=rec + 3 * E)


def _expected_header(n, dtype, chunk, C, E, cb):
    h = np.zeros(64, np.uint8)
    h[0:4] = np.frombuffer(np.uint32(0x50495A53).tobytes(), np.uint8)
    h[4:6] = (1, 0)
    h[6] = dtype
    h[8:16] = np.frombuffer(np.uint64(n).tobytes(), np.uint8)
    h[16:20] = np.frombuffer(np.uint32(chunk).tobytes(), np.uint8)
    h[20:24] = np.frombuffer(np.uint32(C).tobytes(), np.uint8)
    h[24:32] = np.frombuffer(np.uint64(E).tobytes(), np.uint8)
    h[32:48] = cb
    return h


def _compare_all_chunks(hb, xh, dtype, cb, chunk, L, off, cnt, block_chunks=16):
    """Every chunk of the GPU container against the oracle: the tensor is cut
    into blocks of whole chunks, each block encoded by the oracle into its own
    container on a host thread (a chunk's sections do not depend on other
    chunks), and the block's nibble, sign|mantissa, count and record bytes
    compared with the matching slices of the GPU container."""
    from concurrent.futures import ThreadPoolExecutor
    n = xh.size
    C = L["C"]

    def one(c0):
        c1 = min(C, c0 + block_chunks)
        lo, hi = c0 * chunk, min(n, c1 * chunk)
        ref = oracle.encode(xh[lo:hi], dtype, cb, chunk)
        R = _layout(hi - lo, dtype, chunk, (ref.size - _layout(hi - lo, dtype, chunk, 0)["size"]) // 3)
        checks = [
            ("nibbles", hb[L["nib"] + lo // 2: L["nib"] + (hi + 1) // 2], ref[R["nib"]: R["nib"] + (hi - lo + 1) // 2]),
            ("sign|mantissa", hb[L["sm"] + sm_stream_bytes(lo, dtype): L["sm"] + sm_stream_bytes(hi, dtype)],
             ref[R["sm"]: R["sm"] + R["sm_bytes"]]),
            ("counts", hb[L["counts"] + 4 * c0: L["counts"] + 4 * c1], ref[R["counts"]: R["index_end"]]),
            ("records", hb[L["rec"] + 3 * int(off[c0]): L["rec"] + 3 * (int(off[c0]) + int(cnt[c0:c1].sum()))],
             ref[R["rec"]: R["size"]]),
        ]
        for what, got, want in checks:
            if got.size != want.size or not np.array_equal(got, want):
                return "chunks %d..%d: %s differ" % (c0, c1 - 1, what)
        return None

    import os
    with ThreadPoolExecutor(max(1, os.cpu_count() or 1)) as pool:
        bad = [r for r in pool.map(one, range(0, C, block_chunks)) if r]
    assert not bad, bad[:5]
    return C


def _full_size_check(name):
    dtype = W.dtype_of(name)
    n_layers, _ = W.layers_of(name)
    x = W.make_layers(name, 0, n_layers, DEV)
    n = x.numel()
    assert n == W.numel(name)
    cal = W.calibration_tensor(name, DEV)
    cb, hist = sz.calibrate(cal, dtype)
    # calibration on the calibration layer against the oracle
    ref_cb = oracle.calibrate(oracle.histogram(np_bits(cal, dtype), dtype), dtype)
    np.testing.assert_array_equal(np.array(cb.values(), np.uint8), ref_cb)
    del cal

    chunk = 65536
    blob = gpu_encode(x, cb, dtype, chunk, dirty=True)
    E = int(blob[24:32].cpu().numpy().view(np.uint64)[0])
    L = _layout(n, dtype, chunk, E)
    assert blob.numel() == L["size"]
    hb = blob.cpu().numpy()

    # header and inter-section padding, from the layout formula
    np.testing.assert_array_equal(hb[:64], _expected_header(n, dtype, chunk, L["C"], E, ref_cb))
    for lo, hi in ((L["index_end"], L["nib"]), (L["nib"] + (n + 1) // 2, L["sm"]), (L["sm"] + L["sm_bytes"], L["rec"])):
        assert not hb[lo:hi].any(), "padding [%d, %d) not zero" % (lo, hi)

    # E = exponent mass outside the codebook, counted by torch on the device
    if dtype == sz.BF16:
        e = (x.view(torch.int16).to(torch.int32) >> 7) & 0xFF
    elif dtype == sz.FP16:
        e = (x.view(torch.int16).to(torch.int32) >> 10) & 0x1F
    else:
        e = (x.to(torch.int32) >> 2) & 0x1F
    counts = torch.bincount(e.flatten(), minlength=256).cpu().numpy()
    del e
    in_cb = np.zeros(256, bool)
    in_cb[ref_cb] = True
    assert E == int(counts[~in_cb].sum())

    # index = exclusive prefix of the counts
    cnt = hb[L["counts"]: L["counts"] + 4 * L["C"]].view(np.uint32).astype(np.uint64)
    off = hb[L["index"]: L["index"] + 8 * L["C"]].view(np.uint64)
    np.testing.assert_array_equal(off, np.concatenate([[0], np.cumsum(cnt)[:-1]]))
    assert int(cnt.sum()) == E

    # every chunk against the oracle
    xh = np_bits(x, dtype)
    assert _compare_all_chunks(hb, xh, dtype, ref_cb, chunk, L, off, cnt) == L["C"]
    del hb

    st, y = gpu_decode(blob, n, dtype)
    assert st == sz.OK
    assert torch.equal(y, x)
    del y, blob

    # an oracle-built container of a whole layer, decoded on the GPU
    per = n // n_layers
    ref = oracle.encode(xh[:per], dtype, ref_cb, chunk)
    st, y = gpu_decode(torch.from_numpy(ref).to(DEV), per, dtype)
    assert st == sz.OK
    assert torch.equal(y, x[:per])
    return E / n


@pytest.mark.slow
def test_kv_cache_32_layer_bf16_full_size():
    rate = _full_size_check("kv_cache_32x2x32768x8x128_bf16")
    assert 0.0 < rate < 0.5


@pytest.mark.slow
def test_kv_cache_32_layer_e5m2_full_size():
    rate = _full_size_check("kv_cache_32x2x65536x8x128_e5m2")
    assert 0.0 < rate < 0.5


@pytest.mark.slow
def test_kv_cache_32_layer_fp16_full_size():
    rate = _full_size_check("kv_cache_32x2x32768x8x128_fp16")
    assert 0.0 < rate < 0.5
