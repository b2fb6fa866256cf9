"""CPU: the whole-container comparison used by the full-size GPU parity tests
catches a one-bit difference anywhere in the compared sections.

The GPU tests compare every chunk of the two 4.3 GB containers against the
oracle with _compare_all_chunks.  Here the oracle's own container stands in
for the GPU's: it must pass unchanged, and a single flipped bit planted in it
(nibbles, sign|mantissa, counts, records) must be reported.
"""
import numpy as np
import pytest

import oracle
from lossless_kv_cache_gb300 import workloads as W
from tests.test_gpu_parity import _compare_all_chunks, _expected_header, _layout


def _case(dtype):
    if dtype == 0:
        return W.escape_stress(0, chunks=40, chunk_elems=4096).numpy().view(np.uint16)[: 40 * 4096 - 1000]
    if dtype == 2:
        return W.kv_cache_layer_fp16(0, 1, tokens=80).numpy().view(np.uint16)[:-40]
    return W.kv_cache_layer_e5m2(0, 1, tokens=100).numpy()[:-24]


@pytest.mark.parametrize("dtype", [0, 1, 2])
def test_checker_accepts_the_oracle_and_catches_planted_bits(dtype):
    chunk = 4096
    x = _case(dtype)
    cb = oracle.calibrate(oracle.histogram(x, dtype), dtype)
    blob = oracle.encode(x, dtype, cb, chunk)
    E = oracle.parse_header(blob)[1].total_escapes
    L = _layout(x.size, dtype, chunk, E)
    assert blob.size == L["size"]
    np.testing.assert_array_equal(blob[:64], _expected_header(x.size, dtype, chunk, L["C"], E, cb))
    cnt = blob[L["counts"]: L["counts"] + 4 * L["C"]].view(np.uint32).astype(np.uint64)
    off = blob[64: 64 + 8 * L["C"]].view(np.uint64)
    assert _compare_all_chunks(blob, x, dtype, cb, chunk, L, off, cnt, block_chunks=3) == L["C"]
    for pos in (L["nib"] + 5000, L["sm"] + 777, L["counts"] + 4 * 7, L["rec"] + 3 * int(E // 2) + 1, L["size"] - 1):
        bad = blob.copy()
        bad[pos] ^= 1
        with pytest.raises(AssertionError):
            _compare_all_chunks(bad, x, dtype, cb, chunk, L, off, cnt, block_chunks=3)
