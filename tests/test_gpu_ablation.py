"""GPU: the ablation formats (Top-16, Top-8, Top-15 + sentinel) of the plain
kernel family against the oracle's variants, byte for byte, and their
decoders bit for bit, on GPU and oracle containers alike; corrupt containers
are reported."""
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


def inputs():
    return [
        ("bf16 stress", sz.BF16, W.escape_stress(8, chunks=5, chunk_elems=65536)[:300001]),
        ("bf16 cache layer", sz.BF16, W.kv_cache_layer_bf16(2, 4, tokens=150)),
        ("bf16 all patterns", sz.BF16, W.all_bf16_patterns()),
        ("e5m2 cache layer", sz.FP8_E5M2, W.kv_cache_layer_e5m2(2, 4, tokens=170)[:340001]),
        ("e5m2 all patterns", sz.FP8_E5M2, W.all_e5m2_patterns()),
        ("bf16 one", sz.BF16, W.all_bf16_patterns()[12345:12346]),
        ("e5m2 thirty-three", sz.FP8_E5M2, W.all_e5m2_patterns()[100:133]),
    ]


def host(t, dtype):
    a = t.numpy()
    return a.view(np.uint16) if dtype == sz.BF16 else a


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("case", range(7))
@pytest.mark.parametrize("chunk", [64, 4096, 65536])
def test_ablation_formats_match_oracle(variant, case, chunk):
    name, dtype, x = inputs()[case]
    h = host(x, dtype)
    cb16 = oracle.calibrate(oracle.histogram(h, dtype), dtype)
    ocb = oracle.variant_codebook(cb16, variant)
    cb = sz.ablation_codebook(sz.Codebook.make(dtype, [int(e) for e in cb16]), variant)
    assert list(cb.exps) == [int(e) for e in ocb]
    xd = x.cuda()
    blob = sz.ablation_encode(xd, cb, dtype, variant, chunk)
    ref = oracle.encode_variant(h, dtype, ocb, chunk, variant)
    assert np.array_equal(blob.cpu().numpy(), ref), (name, variant, chunk)
    if variant == 0:  # the main format: also the production encoder's container
        assert np.array_equal(ref, oracle.encode(h, dtype, cb16, chunk))
    for b in (blob, torch.from_numpy(ref).cuda()):
        st, y = sz.ablation_decode_status(b, x.numel(), dtype, variant)
        assert st == sz.OK, (name, variant, chunk)
        assert torch.equal(y, xd), (name, variant, chunk)


def test_ablation_corrupt_containers_are_reported():
    x = W.escape_stress(9, chunks=1, chunk_elems=65536)[:20000]
    h = host(x, sz.BF16)
    cb16 = oracle.calibrate(oracle.histogram(h, sz.BF16), sz.BF16)
    for variant in (0, 1, 2):
        ref = oracle.encode_variant(h, sz.BF16, oracle.variant_codebook(cb16, variant), 1024, variant)
        # decoded as another variant
        other = (variant + 1) % 3
        st, _ = sz.ablation_decode_status(torch.from_numpy(ref).cuda(), x.numel(), sz.BF16, other)
        assert st == sz.ERR_CORRUPT
        # an index offset off by one
        bad = ref.copy()
        bad[64 + 8 * 3] += 1
        st, _ = sz.ablation_decode_status(torch.from_numpy(bad).cuda(), x.numel(), sz.BF16, variant)
        assert st == sz.ERR_CORRUPT
    # a sentinel with no escape byte left for it in its chunk
    ref = oracle.encode_variant(h, sz.BF16, oracle.variant_codebook(cb16, 2), 1024, 2)
    L_code = 64 + 12 * 20  # header + index of 20 chunks, already 16-aligned
    bad = ref.copy()
    bad[L_code] |= 0x0F  # element 0 becomes a sentinel
    if (ref[L_code] & 0x0F) != 0x0F:
        st, _ = sz.ablation_decode_status(torch.from_numpy(bad).cuda(), x.numel(), sz.BF16, 2)
        assert st == sz.ERR_CORRUPT
