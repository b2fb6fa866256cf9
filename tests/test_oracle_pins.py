"""Pins of the CPU oracle to facts fixed outside it.

The pins come from the SplitZip page ("SplitZip: Ultra Fast Lossless KV
Compression for Disaggregated LLM Serving", section "Method: SplitZip"):
bit-exact reconstruction ("Decoding strategy: Correction"), 4-bit codes two per
byte ("Fixed-length coding"), 16 + 8 bits per escape ("Escape stream"), raw
sign|mantissa ("Sign/mantissa preservation"), and from arithmetic: closed-form
escape counts and sizes for exhaustive inputs, float semantics of the exponent
field (numpy frexp), library sorts for the Top-16 selection, and hand-worked
containers under tests/golden/.
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_kv_cache_gb300 import workloads as W
from tests import goldens

BF16, E5M2, FP16 = oracle.BF16, oracle.E5M2, oracle.FP16


def a16(x):
    return (x + 15) // 16 * 16


# ---------------------------------------------------------------- hand-worked

@pytest.mark.parametrize("name", goldens.CONTAINER_FIXTURES)
def test_golden_container_bytes(name):
    fx = goldens.load_container(name)
    blob = oracle.encode(fx["input"], fx["dtype"], fx["codebook"], fx["chunk_elems"])
    assert blob.size == fx["size"]
    np.testing.assert_array_equal(blob, fx["expected"])


@pytest.mark.parametrize("name", goldens.CONTAINER_FIXTURES)
def test_golden_container_decodes(name):
    fx = goldens.load_container(name)
    y = oracle.decode(fx["expected"], fx["n"], fx["dtype"])
    np.testing.assert_array_equal(y, fx["input"])


def test_golden_calibration():
    for case in goldens.load_calibration_cases():
        np.testing.assert_array_equal(oracle.calibrate(case["hist"], case["dtype"]), case["expect"])


# (bits, exponent field, sign|mantissa) worked by hand from the bit layouts:
# BF16 = 1 sign, 8 exponent, 7 mantissa bits; E5M2 = 1, 5, 2.
HAND_BF16 = [(0x3F80, 127, 0x00), (0xC000, 128, 0x80), (0x7FC1, 255, 0x41),
             (0x0001, 0, 0x01), (0x8000, 0, 0x80), (0xFF80, 255, 0x80), (0x4049, 128, 0x49)]
HAND_E5M2 = [(0x3C, 15, 0), (0xFF, 31, 7), (0x80, 0, 4), (0x01, 0, 1), (0x7C, 31, 0), (0xBE, 15, 6)]
# FP16 = 1 sign, 5 exponent, 10 mantissa bits; s11 = sign << 10 | mantissa
HAND_FP16 = [(0x3C00, 15, 0x000), (0xFFFF, 31, 0x7FF), (0x8000, 0, 0x400), (0x0001, 0, 0x001),
             (0x7C00, 31, 0x000), (0xBE00, 15, 0x600), (0x4555, 17, 0x155), (0xC248, 16, 0x648)]


@pytest.mark.parametrize("bits,exp,sm", HAND_BF16)
def test_hand_split_bf16(bits, exp, sm):
    x = np.array([bits], dtype=np.uint16)
    # codebook without `exp`: the element escapes with its exponent and position 0
    cb = np.array([v for v in range(256) if v != exp][:16], dtype=np.uint8)
    blob = oracle.encode(x, BF16, cb, 64)
    # C=1: nibbles at 80, sign|mantissa at 96, the escape record at 112
    assert blob[96] == sm
    assert blob.size == 115
    assert blob[80] == 0 and blob[112] == 0 and blob[113] == 0 and blob[114] == exp
    # codebook with `exp` as code 5: the nibble holds 5, no escape
    cb2 = cb.copy()
    cb2[5] = exp
    blob2 = oracle.encode(x, BF16, cb2, 64)
    assert blob2.size == 112 and blob2[80] == 5 and blob2[96] == sm


@pytest.mark.parametrize("bits,exp,s3", HAND_E5M2)
def test_hand_split_e5m2(bits, exp, s3):
    x = np.array([bits], dtype=np.uint8)
    cb = np.array([v for v in range(32) if v != exp][:16], dtype=np.uint8)
    blob = oracle.encode(x, E5M2, cb, 64)
    assert blob[96] == s3 and blob[114] == exp


@pytest.mark.parametrize("bits,exp,s11", HAND_FP16)
def test_hand_split_fp16(bits, exp, s11):
    x = np.array([bits], dtype=np.uint16)
    cb = np.array([v for v in range(32) if v != exp][:16], dtype=np.uint8)
    blob = oracle.encode(x, FP16, cb, 64)
    # one element: s11 in the low 11 bits of the 2-byte stream (11 * 1 bytes padded)
    assert blob[96] == s11 & 0xFF and blob[97] == s11 >> 8
    assert blob.size == 96 + 16 + 3 and blob[114] == exp and blob[80] == 0
    cb2 = cb.copy()
    cb2[9] = exp
    blob2 = oracle.encode(x, FP16, cb2, 64)
    assert blob2.size == 112 and blob2[80] == 9


# ------------------------------------------------------------- exhaustive sets

@pytest.mark.parametrize("chunk", [65536, 64, 4096])
def test_exhaustive_bf16(chunk):
    """All 65,536 BF16 patterns: every exponent value appears 2*128 = 256
    times, so the tie rule gives codebook 0..15 and E = 65536 - 16*256."""
    x = np.arange(65536, dtype=np.uint16)
    h = oracle.histogram(x, BF16)
    assert (h == 256).all()
    cb = oracle.calibrate(h, BF16)
    np.testing.assert_array_equal(cb, np.arange(16))
    blob = oracle.encode(x, BF16, cb, chunk)
    st, hdr = oracle.parse_header(blob)
    assert st == oracle.OK and hdr.total_escapes == 61440
    C = 65536 // chunk
    assert blob.size == a16(64 + 12 * C) + 32768 + 65536 + 2 * 61440 + 61440
    np.testing.assert_array_equal(oracle.decode(blob, 65536, BF16), x)


def test_exhaustive_e5m2():
    """All 256 E5M2 patterns: each of the 32 exponents appears 8 times, the
    codebook is 0..15 and the 16 exponents 16..31 escape: E = 128."""
    x = np.arange(256, dtype=np.uint8)
    h = oracle.histogram(x, E5M2)
    assert (h[:32] == 8).all() and (h[32:] == 0).all()
    cb = oracle.calibrate(h, E5M2)
    np.testing.assert_array_equal(cb, np.arange(16))
    blob = oracle.encode(x, E5M2, cb, 64)
    st, hdr = oracle.parse_header(blob)
    assert hdr.total_escapes == 128
    assert blob.size == a16(64 + 12 * 4) + 128 + 96 + 256 + 128
    np.testing.assert_array_equal(oracle.decode(blob, 256, E5M2), x)


@pytest.mark.parametrize("chunk", [65536, 64])
def test_exhaustive_fp16(chunk):
    """All 65,536 FP16 patterns: each of the 32 exponents appears 2 * 1024 =
    2,048 times, the codebook is 0..15 and E = 65536 - 16 * 2048 = 32768;
    the sign|mantissa stream holds 11 bits per element (90,112 bytes)."""
    x = np.arange(65536, dtype=np.uint16)
    h = oracle.histogram(x, FP16)
    assert (h[:32] == 2048).all() and (h[32:] == 0).all()
    cb = oracle.calibrate(h, FP16)
    np.testing.assert_array_equal(cb, np.arange(16))
    blob = oracle.encode(x, FP16, cb, chunk)
    st, hdr = oracle.parse_header(blob)
    assert st == oracle.OK and hdr.total_escapes == 32768
    C = 65536 // chunk
    assert blob.size == a16(64 + 12 * C) + 32768 + 90112 + 3 * 32768
    np.testing.assert_array_equal(oracle.decode(blob, 65536, FP16), x)


# ----------------------------------------------- float semantics cross-checks

def exponent_field_from_floats_bf16(bits):
    """Biased exponent field of BF16 values derived through float semantics
    (numpy frexp), not through bit shifts."""
    with np.errstate(invalid="ignore"):
        f = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    e = np.zeros(bits.size, dtype=np.int64)
    special = ~np.isfinite(f)
    tiny = np.isfinite(f) & (np.abs(f) < 2.0 ** -126)
    normal = ~special & ~tiny
    e[special] = 255
    e[normal] = np.frexp(f[normal])[1] + 126
    return e


def exponent_field_from_floats_e5m2(bits):
    f = torch.from_numpy(bits).view(torch.float8_e5m2).float().numpy().astype(np.float64)
    e = np.zeros(bits.size, dtype=np.int64)
    special = ~np.isfinite(f)
    tiny = np.isfinite(f) & (np.abs(f) < 2.0 ** -14)
    normal = ~special & ~tiny
    e[special] = 31
    e[normal] = np.frexp(f[normal])[1] + 14
    return e


def exponent_field_from_floats_fp16(bits):
    with np.errstate(invalid="ignore"):
        f = bits.view(np.float16).astype(np.float64)
    e = np.zeros(bits.size, dtype=np.int64)
    special = ~np.isfinite(f)
    tiny = np.isfinite(f) & (np.abs(f) < 2.0 ** -14)
    normal = ~special & ~tiny
    e[special] = 31
    e[normal] = np.frexp(f[normal])[1] + 14
    return e


def test_histogram_matches_float_semantics_fp16():
    x = W.kv_cache_layer_fp16(3, 2, tokens=64).numpy().view(np.uint16)
    x = np.concatenate([x, W.special_fp16_patterns().numpy().view(np.uint16), np.arange(65536, dtype=np.uint16)])
    expect = np.bincount(exponent_field_from_floats_fp16(x), minlength=256)
    np.testing.assert_array_equal(oracle.histogram(x, FP16), expect)


def test_sign_mantissa_bits_match_float_semantics_fp16():
    """The 11-bit sign|mantissa field (reading R16) of normal FP16 values is
    (signbit << 10) | round(1024 * (2|m| - 1)), m the frexp mantissa; read back
    from the packed stream bit by bit."""
    x = W.kv_cache_layer_fp16(5, 1, tokens=8).numpy().view(np.uint16)
    f = x.view(np.float16).astype(np.float64)
    keep = np.isfinite(f) & (np.abs(f) >= 2.0 ** -14)
    x, f = x[keep][:3000].copy(), f[keep][:3000]
    m = np.frexp(np.abs(f))[0]
    expect = (np.signbit(f).astype(np.int64) << 10) | np.rint(1024 * (2 * m - 1)).astype(np.int64)
    cb = oracle.calibrate(oracle.histogram(x, FP16), FP16)
    blob = oracle.encode(x, FP16, cb, 65536)
    sm_off = a16(64 + 12) + a16((x.size + 1) // 2)
    bits = np.unpackbits(blob[sm_off: sm_off + 11 * (-(-x.size // 8))], bitorder="little")
    got = (bits[: 11 * x.size].reshape(-1, 11).astype(np.int64) << np.arange(11)).sum(axis=1)
    np.testing.assert_array_equal(got, expect)


def test_histogram_matches_float_semantics_bf16():
    x = W.llama_layer_kv(3, tokens=256).numpy().view(np.uint16)
    x = np.concatenate([x, W.special_bf16_patterns().numpy().view(np.uint16)])
    expect = np.bincount(exponent_field_from_floats_bf16(x), minlength=256)
    np.testing.assert_array_equal(oracle.histogram(x, BF16), expect)


def test_histogram_matches_float_semantics_e5m2():
    x = W.kv_cache_layer_e5m2(3, 0, tokens=64).numpy()
    x = np.concatenate([x, W.special_e5m2_patterns().numpy()])
    expect = np.bincount(exponent_field_from_floats_e5m2(x), minlength=256)
    np.testing.assert_array_equal(oracle.histogram(x, E5M2), expect)


def test_sign_mantissa_byte_matches_float_semantics_bf16():
    """The raw sign|mantissa byte (reading R3) of normal BF16 values equals
    (signbit << 7) | round(128 * (2|m| - 1)) with m the frexp mantissa."""
    x = W.kv_tile_k_only(5, tokens=64).numpy().view(np.uint16)
    f = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    keep = np.isfinite(f) & (np.abs(f) >= 2.0 ** -126)
    x, f = x[keep][:4000], f[keep][:4000]
    m = np.frexp(np.abs(f))[0]
    expect = (np.signbit(f).astype(np.int64) << 7) | np.rint(128 * (2 * m - 1)).astype(np.int64)
    cb = oracle.calibrate(oracle.histogram(x, BF16), BF16)
    blob = oracle.encode(x, BF16, cb, 65536)
    _, hdr = oracle.parse_header(blob)
    sm_off = a16(64 + 12) + a16((x.size + 1) // 2)
    np.testing.assert_array_equal(blob[sm_off : sm_off + x.size], expect)


# -------------------------------------------------- codebook vs library sort

@pytest.mark.parametrize("seed", range(6))
def test_calibrate_matches_lexsort(seed):
    """Top-16 = first 16 of a stable sort by (count desc, value asc)."""
    rng = np.random.default_rng(seed)
    for dtype, bins in ((BF16, 256), (E5M2, 32), (FP16, 32)):
        h = np.zeros(256, dtype=np.uint64)
        support = rng.choice(bins, size=rng.integers(1, bins), replace=False)
        h[support] = rng.integers(0, 6, size=support.size)  # many ties
        values = np.arange(bins)
        order = np.lexsort((values, -h[:bins].astype(np.int64)))
        np.testing.assert_array_equal(oracle.calibrate(h, dtype), order[:16])


def test_calibrate_rejects_e5m2_mass_above_31():
    h = np.zeros(256, dtype=np.uint64)
    h[40] = 1
    for dtype in (E5M2, FP16):
        with pytest.raises(ValueError):
            oracle.calibrate(h, dtype)


def test_fp16_and_bf16_containers_differ_only_where_the_formats_do():
    """The same 16-bit words encoded as FP16 and as BF16 give different
    dtype bytes and exponents, and neither decodes as the other."""
    x = W.kv_cache_layer_fp16(2, 0, tokens=4).numpy().view(np.uint16)
    b = oracle.encode(x, BF16, oracle.calibrate(oracle.histogram(x, BF16), BF16), 4096)
    f = oracle.encode(x, FP16, oracle.calibrate(oracle.histogram(x, FP16), FP16), 4096)
    assert b[6] == BF16 and f[6] == FP16
    assert oracle.decode_status(f, x.size, BF16)[0] == oracle.CORRUPT
    assert oracle.decode_status(b, x.size, FP16)[0] == oracle.CORRUPT
    np.testing.assert_array_equal(oracle.decode(f, x.size, FP16), x)


# ---------------------------------------- escape count, size and ratio laws

def _random_cases():
    yield "kv_tile", BF16, W.kv_tile_k_only(7, tokens=200).numpy().view(np.uint16), 65536
    yield "llama", BF16, W.llama_layer_kv(7, tokens=64).numpy().view(np.uint16), 4096
    yield "stress", BF16, W.escape_stress(7, chunks=2, chunk_elems=8192).numpy().view(np.uint16), 8192
    yield "e5m2", E5M2, W.kv_cache_layer_e5m2(7, 1, tokens=40).numpy(), 1024
    rng = np.random.default_rng(0)
    yield "uniform_bits", BF16, rng.integers(0, 65536, 100003).astype(np.uint16), 2048
    yield "uniform_bits_e5m2", E5M2, rng.integers(0, 256, 100003).astype(np.uint8), 512
    yield "fp16_cache", FP16, W.kv_cache_layer_fp16(7, 3, tokens=40).numpy().view(np.uint16), 4096
    yield "uniform_bits_fp16", FP16, rng.integers(0, 65536, 100003).astype(np.uint16), 1024


@pytest.mark.parametrize("case", list(_random_cases()), ids=lambda c: c[0])
def test_escape_count_size_ratio_roundtrip(case):
    _, dtype, x, chunk = case
    h = oracle.histogram(x, dtype)
    cb = oracle.calibrate(h, dtype)
    blob = oracle.encode(x, dtype, cb, chunk)
    st, hdr = oracle.parse_header(blob)
    assert st == oracle.OK
    n = x.size
    # escape count = histogram mass outside the Top-16 (exponents via floats)
    ef = {BF16: exponent_field_from_floats_bf16, E5M2: exponent_field_from_floats_e5m2,
          FP16: exponent_field_from_floats_fp16}[dtype](x)
    E = int(np.sum(~np.isin(ef, cb)))
    assert hdr.total_escapes == E
    # per-chunk counts sum to E
    assert int(oracle.chunk_escape_counts(x, dtype, cb, chunk).sum()) == E
    # size: 4 bits + raw sign|mantissa per element, 24 bits per escape, plus
    # the 64 B header, 12 B of index per chunk and section padding (< 16 B each)
    C = -(-n // chunk)
    bits_sm = {BF16: 8, E5M2: 3, FP16: 11}[dtype]
    payload = n * (4 + bits_sm) / 8 + 3 * E
    overhead = blob.size - payload
    assert 64 + 12 * C <= overhead < 64 + 12 * C + 4 * 16 + 3
    # ratio bound: 16/12 for BF16, 8/7 for E5M2, 16/15 for FP16
    raw = n * (1 if dtype == E5M2 else 2)
    assert raw / blob.size <= {BF16: 4 / 3, E5M2: 8 / 7, FP16: 16 / 15}[dtype]
    np.testing.assert_array_equal(oracle.decode(blob, n, dtype), x)


@pytest.mark.parametrize("n", [0, 1, 2, 7, 8, 9, 63, 64, 65, 127, 4097])
@pytest.mark.parametrize("dtype", [BF16, E5M2, FP16])
def test_small_sizes_roundtrip(n, dtype):
    rng = np.random.default_rng(n)
    x = rng.integers(0, 256 if dtype == E5M2 else 65536, n).astype(np.uint8 if dtype == E5M2 else np.uint16)
    cb = np.arange(16, dtype=np.uint8) + (120 if dtype == BF16 else 8)
    blob = oracle.encode(x, dtype, cb, 64)
    assert blob.size == oracle.container_size(n, dtype, 64, oracle.parse_header(blob)[1].total_escapes)
    np.testing.assert_array_equal(oracle.decode(blob, n, dtype), x)


def test_empty_input_is_header_only():
    for dtype in (BF16, E5M2, FP16):
        x = np.zeros(0, dtype=np.uint8 if dtype == E5M2 else np.uint16)
        blob = oracle.encode(x, dtype, np.arange(16, dtype=np.uint8), 65536)
        assert blob.size == 64
        assert oracle.decode(blob, 0, dtype).size == 0


def test_all_escape_chunk():
    """A codebook holding none of the exponents present: every element of the
    chunk escapes and all nibbles are 0 (reading R5)."""
    x = np.full(65536, 0x3F80, dtype=np.uint16)
    cb = np.arange(16, dtype=np.uint8)
    blob = oracle.encode(x, BF16, cb, 65536)
    _, hdr = oracle.parse_header(blob)
    assert hdr.total_escapes == 65536
    assert blob.size == oracle.max_container_size(65536, BF16, 65536)
    nib_off = a16(64 + 12)
    assert not blob[nib_off : nib_off + 32768].any()
    np.testing.assert_array_equal(oracle.decode(blob, 65536, BF16), x)


# --------------------------------------------------------- corrupt containers

def _stress_blob():
    x = W.escape_stress(11, chunks=3, chunk_elems=4096).numpy().view(np.uint16)[:12000]
    cb = oracle.calibrate(oracle.histogram(x, BF16), BF16)
    return x, oracle.encode(x, BF16, cb, 4096)


def corruptions(blob):
    """(name, corrupted copy) pairs that a decoder must reject."""
    st, h = oracle.parse_header(blob)
    C, E, n = h.n_chunks, h.total_escapes, h.n
    nib_off = a16(64 + 12 * C)
    rec_off = nib_off + a16((n + 1) // 2) + a16(n)
    out = []

    def mut(name, f):
        b = blob.copy()
        f(b)
        out.append((name, b))

    mut("magic", lambda b: b.__setitem__(0, 0))
    mut("version", lambda b: b.__setitem__(4, 2))
    mut("dtype", lambda b: b.__setitem__(6, 1))
    mut("reserved", lambda b: b.__setitem__(50, 1))
    mut("chunk_not_pow2", lambda b: b.__setitem__(16, 0x01))
    mut("n_chunks", lambda b: b.__setitem__(20, C + 1))
    mut("escapes_gt_n", lambda b: b[24:32].__setitem__(slice(None), np.frombuffer(np.uint64(n + 1).tobytes(), np.uint8)))
    mut("codebook_dup", lambda b: b.__setitem__(33, b[32]))
    mut("offset_not_prefix", lambda b: b.__setitem__(64 + 8, b[64 + 8] ^ 1))
    mut("count_changed", lambda b: b.__setitem__(64 + 8 * C, b[64 + 8 * C] ^ 1))
    mut("pos_out_of_chunk", lambda b: b[rec_off : rec_off + 2].__setitem__(slice(None), [0xFF, 0xFF]))
    mut("pos_not_ascending", lambda b: b[rec_off + 3 : rec_off + 5].__setitem__(slice(None), b[rec_off : rec_off + 2]))
    out.append(("truncated", blob[:-1].copy()))
    return out


def test_corrupt_containers_rejected():
    x, blob = _stress_blob()
    assert oracle.decode_status(blob, x.size, BF16)[0] == oracle.OK
    for name, bad in corruptions(blob):
        st, _ = oracle.decode_status(bad, x.size, BF16)
        assert st == oracle.CORRUPT, name
    # caller's n or dtype disagreeing with the header
    assert oracle.decode_status(blob, x.size - 1, BF16)[0] == oracle.CORRUPT
    assert oracle.decode_status(blob, x.size, E5M2)[0] == oracle.CORRUPT
