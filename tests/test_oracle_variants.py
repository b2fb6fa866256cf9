"""Pins of the oracle's ablation variants (Results, "Ablation Studies": Top-8
with 3-bit codes, Top-15 with a sentinel code; READINGS V1-V3 in
oracle/splitzip_oracle.c).  Checked against what the readings and the
mathematics fix: exhaustive round trips, closed-form escape counts and sizes on
inputs whose histograms are known, bytes derived by hand for a small input,
and rejected corruptions."""
import numpy as np
import pytest

import oracle
from lossless_kv_cache_gb300 import workloads as W

V = (oracle.TOP8, oracle.TOP15_SENTINEL)


def cb_of(x, dtype, variant):
    return oracle.variant_codebook(oracle.calibrate(oracle.histogram(x, dtype), dtype), variant)


@pytest.mark.parametrize("variant", V)
@pytest.mark.parametrize("chunk", [64, 65536])
def test_all_bf16_patterns_round_trip(variant, chunk):
    x = np.arange(65536, dtype=np.uint16)
    cb = cb_of(x, oracle.BF16, variant)
    blob = oracle.encode_variant(x, oracle.BF16, cb, chunk, variant)
    assert np.array_equal(oracle.decode_variant(blob, x.size, oracle.BF16), x)


@pytest.mark.parametrize("variant", V)
def test_all_e5m2_patterns_round_trip(variant):
    x = np.arange(256, dtype=np.uint8)
    for chunk in (64, 65536):
        blob = oracle.encode_variant(x, oracle.E5M2, cb_of(x, oracle.E5M2, variant), chunk, variant)
        assert np.array_equal(oracle.decode_variant(blob, x.size, oracle.E5M2), x)


def test_uniform_histograms_closed_forms():
    # every exponent equally frequent: the first k exponents are coded and the
    # rest escape: E = n - k * (n / bins)
    x = np.arange(65536, dtype=np.uint16)  # 256 of each of the 256 BF16 exponents
    for variant, k, bytes_per_escape, code_bytes in ((oracle.TOP8, 8, 3, 3 * 8192),
                                                     (oracle.TOP15_SENTINEL, 15, 1, 32768)):
        cb = cb_of(x, oracle.BF16, variant)
        assert list(cb[:k]) == list(range(k)) and not cb[k:].any()
        blob = oracle.encode_variant(x, oracle.BF16, cb, 65536, variant)
        E = 65536 - k * 256
        assert int(blob[24:32].view(np.uint64)[0]) == E
        # header 64 + index 12 -> 80; codes; 65,536 sign|mantissa bytes; escapes
        assert blob.size == 80 + code_bytes + 65536 + bytes_per_escape * E
    assert 65536 - 8 * 256 == 63488 and 65536 - 15 * 256 == 61696
    y = np.arange(256, dtype=np.uint8)  # 8 of each of the 32 E5M2 exponents
    for variant, k in ((oracle.TOP8, 8), (oracle.TOP15_SENTINEL, 15)):
        blob = oracle.encode_variant(y, oracle.E5M2, cb_of(y, oracle.E5M2, variant), 64, variant)
        assert int(blob[24:32].view(np.uint64)[0]) == 256 - 8 * k


def test_escapes_are_the_mass_outside_the_codebook():
    x = W.escape_stress(3, chunks=2, chunk_elems=65536).numpy().view(np.uint16)[:100003]
    h = oracle.histogram(x, oracle.BF16)
    for variant, k in ((oracle.TOP8, 8), (oracle.TOP15_SENTINEL, 15)):
        cb = cb_of(x, oracle.BF16, variant)
        mass = int(h.sum() - h[cb[:k]].sum())
        blob = oracle.encode_variant(x, oracle.BF16, cb, 4096, variant)
        assert int(blob[24:32].view(np.uint64)[0]) == mass
        assert np.array_equal(oracle.decode_variant(blob, x.size, oracle.BF16), x)


# 1.0 (e 127, sm 0x00), 2.0 (e 128, sm 0x00), -2.0 (e 128, sm 0x80),
# the smallest subnormal 0x0001 (e 0, sm 0x01) and a NaN 0x7FC1 (e 255, sm 0x41)
FIVE = np.array([0x3F80, 0x4000, 0xC000, 0x0001, 0x7FC1], dtype=np.uint16)


def test_top8_bytes_by_hand():
    cb = np.array([128, 127, 0, 1, 2, 3, 4, 5] + [0] * 8, dtype=np.uint8)
    blob = oracle.encode_variant(FIVE, oracle.BF16, cb, 64, oracle.TOP8)
    # codes 1, 0, 0, 2 and an escape (code 0): bits 0..2 = 1, bits 9..11 = 2
    # -> 0x000401, three bytes LSB first, at 80 (header 64 + index 12 -> 80)
    assert list(blob[80:83]) == [0x01, 0x04, 0x00]
    assert list(blob[96:101]) == [0x00, 0x00, 0x80, 0x01, 0x41]   # sign|mantissa at 80 + 16
    assert list(blob[112:115]) == [0x04, 0x00, 0xFF]              # (position 4, exponent 255)
    assert blob.size == 115 and blob[7] == oracle.TOP8
    assert np.array_equal(oracle.decode_variant(blob, 5, oracle.BF16), FIVE)


def test_sentinel_bytes_by_hand():
    cb = np.array([128, 127, 0] + list(range(1, 13)) + [0], dtype=np.uint8)
    blob = oracle.encode_variant(FIVE, oracle.BF16, cb, 64, oracle.TOP15_SENTINEL)
    # codes 1, 0, 0, 2, 15 (the sentinel), two per byte, even element low
    assert list(blob[80:83]) == [0x01, 0x20, 0x0F]
    assert list(blob[96:101]) == [0x00, 0x00, 0x80, 0x01, 0x41]
    assert list(blob[112:113]) == [0xFF]                          # the exponent only
    assert blob.size == 113 and blob[7] == oracle.TOP15_SENTINEL
    assert np.array_equal(oracle.decode_variant(blob, 5, oracle.BF16), FIVE)


def test_variant_corruptions_are_rejected():
    x = W.escape_stress(4, chunks=1, chunk_elems=65536).numpy().view(np.uint16)[:5000]
    for variant in V:
        blob = oracle.encode_variant(x, oracle.BF16, cb_of(x, oracle.BF16, variant), 1024, variant)
        for name, bad in (("variant 3", lambda b: b.__setitem__(7, 3)),
                          ("codebook tail", lambda b: b.__setitem__(47, 1)),
                          ("offset + 1", lambda b: b.__setitem__(64 + 8 * 5, b[64 + 8 * 5] + 1))):
            b = blob.copy()
            bad(b)
            st, _ = oracle.decode_variant_status(b, x.size, oracle.BF16)
            assert st == oracle.CORRUPT, (variant, name)
    # a sentinel without an escape byte left in its chunk
    cb = np.array([128, 127, 0] + list(range(1, 13)) + [0], dtype=np.uint8)
    blob = oracle.encode_variant(FIVE, oracle.BF16, cb, 64, oracle.TOP15_SENTINEL)
    b = blob.copy()
    b[81] = 0xF0  # element 3 becomes a sentinel too: two sentinels, one escape
    assert oracle.decode_variant_status(b, 5, oracle.BF16)[0] == oracle.CORRUPT


def test_variants_are_defined_for_bf16_and_e5m2_only():
    """The ablation formats (readings V1-V3) are defined for the page's two
    dtypes; the oracle refuses FP16 for them."""
    x = np.arange(4096, dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.encode_variant(x, oracle.FP16, oracle.variant_codebook(np.arange(16), oracle.TOP8), 4096, oracle.TOP8)
