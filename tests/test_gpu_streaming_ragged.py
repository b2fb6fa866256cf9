"""GPU parity of the persistent streaming encoder and decoder on ragged sizes.

A call with at most 8,192 tiles (a tile is 16 KB of input, or one chunk when
chunks are smaller) takes the small-tensor kernels, so the ragged sizes of
test_gpu_parity.py and test_gpu_fp16.py never reach the streaming encoder.
These cases have more tiles than that, so they exercise the streaming
encoder's partial-tile body: a ragged last tile, the last bytes past the
tensor map's whole 128-byte rows, tiles smaller than 16 KB throughout (chunks
of 64 and 4,096 elements), and FP16's per-thread stores beside its
shared-memory transpose.  Every case is also above 2^21 elements, so its
decode is the streaming decoder's too.  Each container must equal the
oracle's byte for byte, and both containers must decode on the GPU to the
input (tolerance 0: integer work).
"""
import numpy as np
import pytest
import torch

import lossless_kv_cache_gb300 as sz
from lossless_kv_cache_gb300 import workloads as W
from tests.test_gpu_parity import roundtrip_vs_oracle

pytestmark = pytest.mark.gpu

SMALL_PATH_MAX_TILES = 8192  # the C ABI's small-tensor encode threshold (tiles of one call)
SMALL_DECODE_MAX_ELEMS = 1 << 21  # and its small-tensor decode threshold
TILE_BYTES = 16384


@pytest.fixture(scope="module", autouse=True)
def _lib(splitzip_lib):
    assert torch.cuda.is_available()
    return splitzip_lib


def _tile_elems(dtype, chunk):
    return min(chunk, TILE_BYTES // (1 if dtype == sz.FP8_E5M2 else 2))


def _input(dtype, n, seed):
    """KV-cache-like bits of the dtype with 2 % arbitrary patterns (escapes of
    every kind)."""
    layer_tokens = -(-n // (2 * 8 * 128))
    if dtype == sz.BF16:
        x = W.kv_cache_layer_bf16(seed, 1, layer_tokens).numpy().view(np.uint16)[:n].copy()
        cb = [127, 126, 128, 125, 124, 129, 123, 130, 122, 131, 121, 132, 120, 119, 133, 118]
        bits = np.uint16
    elif dtype == sz.FP16:
        x = W.kv_cache_layer_fp16(seed, 1, layer_tokens).numpy().view(np.uint16)[:n].copy()
        cb = [15, 14, 16, 13, 12, 17, 11, 18, 10, 9, 19, 8, 7, 20, 6, 5]
        bits = np.uint16
    else:
        x = W.kv_cache_layer_e5m2(seed, 1, layer_tokens).numpy()[:n].copy()
        cb = [15, 14, 16, 13, 17, 12, 18, 11, 19, 10, 20, 9, 21, 8, 22, 7]
        bits = np.uint8
    rng = np.random.default_rng(seed)
    k = rng.integers(0, n, size=n // 50)
    x[k] = rng.integers(0, np.iinfo(bits).max + 1, size=k.size).astype(bits)
    return x, cb


@pytest.mark.parametrize("dtype", [sz.BF16, sz.FP8_E5M2, sz.FP16])
@pytest.mark.parametrize("chunk,extra", [(64, 37), (4096, 5), (65536, 777)])
def test_streaming_encoder_ragged(dtype, chunk, extra):
    te = _tile_elems(dtype, chunk)
    # past both small-tensor limits, then a ragged tail
    n = max((SMALL_PATH_MAX_TILES + 1) * te, SMALL_DECODE_MAX_ELEMS) + extra
    assert -(-n // te) > SMALL_PATH_MAX_TILES and n > SMALL_DECODE_MAX_ELEMS
    x, cb = _input(dtype, n, seed=chunk + dtype)
    roundtrip_vs_oracle(x, dtype, cb, chunk)
