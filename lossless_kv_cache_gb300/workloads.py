"""Seeded synthetic KV-cache tensors shaped like the SplitZip page's workloads.

This module only draws random numbers and rounds them to BF16 / FP8-E5M2; it
holds none of the codec's arithmetic, so both the CUDA path (through the tests
and the benchmark) and the CPU oracle can take their inputs from it.

The page ("SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
Serving", Contributions 2 and Results) measures on real BF16 / E5M2 KV
activations of Qwen, Llama and Phi models, which are not available here; the
tensors below stand in for them.  Layout is contiguous
[layer][K,V][token][kv_head][head_dim], channel = kv_head * 128 + dim.

Every tensor is returned as raw bits: BF16 and FP16 as torch.int16, E5M2 as
torch.uint8.
Per-layer generators use seed ``seed * 1000 + layer`` so a 32-layer cache can be
produced one layer at a time.  The random numbers are always drawn with the CPU
generator (torch.Generator on the CPU, the seeds above), whatever device the
result is for; the 32-layer caches are then moved to the device as float32 and
rounded there (round to nearest even, no saturation: the same result as on the
CPU), one layer at a time.
"""
import torch

HEADS = 8
HEAD_DIM = 128
CHANNELS = HEADS * HEAD_DIM


def _gen(seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _lognormal(shape, sigma, g, device):
    return torch.exp(sigma * torch.randn(shape, generator=g, device=device))


def to_bf16_bits(x):
    return x.to(torch.bfloat16).view(torch.int16)


def to_e5m2_bits(x):
    # torch rounds to nearest even and does not saturate (overflow -> inf)
    return x.to(torch.float8_e5m2).view(torch.uint8)


def to_fp16_bits(x):
    # round to nearest even; values beyond 65504 would become inf (the
    # recipes' scales stay far below it)
    return x.to(torch.float16).view(torch.int16)


def kv_tile_k_only(seed, tokens=1024, device="cpu"):
    """One layer, K only: N(0,1) x per-channel lognormal(0,1) scale."""
    g = _gen(seed, device)
    chan = _lognormal((CHANNELS,), 1.0, g, device)
    x = torch.randn((tokens, CHANNELS), generator=g, device=device) * chan
    return to_bf16_bits(x).reshape(-1)


def llama_layer_kv(seed, tokens=8192, device="cpu"):
    """One Llama-3-8B-like layer, K and V.

    K = N(0,1) x per-channel lognormal(0,1.5) with 4 outlier channels x20;
    V = N(0, 0.5)."""
    g = _gen(seed, device)
    chan = _lognormal((CHANNELS,), 1.5, g, device)
    outliers = torch.randperm(CHANNELS, generator=g, device=device)[:4]
    chan[outliers] *= 20.0
    k = torch.randn((tokens, CHANNELS), generator=g, device=device) * chan
    v = 0.5 * torch.randn((tokens, CHANNELS), generator=g, device=device)
    return to_bf16_bits(torch.stack([k, v])).reshape(-1)


def kv_cache_layer_f32(seed, layer, tokens, device="cpu"):
    """One layer (K and V) of the 32-layer cache, float32, before rounding.

    Per layer: scale_l ~ lognormal(0,1); per K/V and channel a lognormal(0,1)
    scale (the single-layer scheme); values N(0,1) x channel scale x scale_l."""
    g = _gen(seed * 1000 + layer, device)
    scale_l = _lognormal((1,), 1.0, g, device)
    chan = _lognormal((2, 1, CHANNELS), 1.0, g, device)
    x = torch.randn((2, tokens, CHANNELS), generator=g, device=device)
    return x * (chan * scale_l)


def kv_cache_layer_bf16(seed, layer, tokens=32768, device="cpu"):
    return to_bf16_bits(kv_cache_layer_f32(seed, layer, tokens).to(device)).reshape(-1)


def kv_cache_layer_e5m2(seed, layer, tokens=65536, device="cpu"):
    return to_e5m2_bits(kv_cache_layer_f32(seed, layer, tokens).to(device)).reshape(-1)


def kv_cache_layer_fp16(seed, layer, tokens=32768, device="cpu"):
    return to_fp16_bits(kv_cache_layer_f32(seed, layer, tokens).to(device)).reshape(-1)


def escape_stress(seed, chunks=64, chunk_elems=65536, sigma=3.0, device="cpu"):
    """Heavy-tailed values: Student-t(df=2) x per-element lognormal(0, sigma).

    t(2) = Z / sqrt(W / 2) with W ~ chi-square(2) = -2 ln U."""
    g = _gen(seed, device)
    n = chunks * chunk_elems
    z = torch.randn(n, generator=g, device=device)
    u = torch.rand(n, generator=g, device=device).clamp_min(1e-30)
    t = z / torch.sqrt(-torch.log(u))
    s = _lognormal((n,), sigma, g, device)
    return to_bf16_bits(t * s)


def special_bf16_patterns():
    """Sign/zero/inf/NaN/subnormal bit patterns and their neighbours (BF16)."""
    pats = [0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x7FC1, 0x7F81, 0xFFFF,
            0x0001, 0x8001, 0x007F, 0x807F, 0x0080, 0x8080, 0x7F7F, 0xFF7F, 0x3F80, 0xBF80]
    return torch.tensor(pats, dtype=torch.int32).to(torch.int16)


def special_e5m2_patterns():
    pats = [0x00, 0x80, 0x7C, 0xFC, 0x7D, 0x7E, 0x7F, 0xFF, 0x01, 0x81, 0x03, 0x83,
            0x04, 0x84, 0x7B, 0xFB, 0x3C, 0xBC]
    return torch.tensor(pats, dtype=torch.uint8)


def special_fp16_patterns():
    """Sign/zero/inf/NaN/subnormal bit patterns and their neighbours (FP16)."""
    pats = [0x0000, 0x8000, 0x7C00, 0xFC00, 0x7E00, 0xFE00, 0x7E01, 0x7C01, 0xFFFF,
            0x0001, 0x8001, 0x03FF, 0x83FF, 0x0400, 0x8400, 0x7BFF, 0xFBFF, 0x3C00, 0xBC00]
    return torch.tensor(pats, dtype=torch.int32).to(torch.int16)


def all_bf16_patterns():
    return torch.arange(65536, dtype=torch.int32).to(torch.int16)


def all_e5m2_patterns():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8)


# --------------------------------------------------------------------------
# the five workloads, by name

WORKLOADS = {
    # name: (dtype, n, description)
    "kv_tile_1x1024x8x128_bf16": (0, 1024 * CHANNELS,
                                  "BF16 1 layer K only, 1024 tok x 8 heads x 128"),
    "llama_layer_2x8192x8x128_bf16": (0, 2 * 8192 * CHANNELS,
                                      "BF16 1 layer K+V, 8192 tok x 8 heads x 128"),
    "kv_cache_32x2x32768x8x128_bf16": (0, 32 * 2 * 32768 * CHANNELS,
                                       "BF16 32 layers K+V, 32768 tok x 8 heads x 128"),
    "escape_stress_64x65536_bf16": (0, 64 * 65536,
                                    "BF16 Student-t(2) x lognormal(0,3), 64 chunks of 65536"),
    "kv_cache_32x2x65536x8x128_e5m2": (1, 32 * 2 * 65536 * CHANNELS,
                                       "FP8-E5M2 32 layers K+V, 65536 tok x 8 heads x 128"),
    # beyond the five: the BF16 cache recipe rounded to FP16 instead
    "kv_cache_32x2x32768x8x128_fp16": (2, 32 * 2 * 32768 * CHANNELS,
                                       "FP16 32 layers K+V, 32768 tok x 8 heads x 128"),
}


def layers_of(name):
    """(n_layers, per-layer generator(seed, layer, device)) for the cache workloads."""
    if name == "kv_cache_32x2x32768x8x128_bf16":
        return 32, lambda seed, layer, device="cpu": kv_cache_layer_bf16(seed, layer, 32768, device)
    if name == "kv_cache_32x2x65536x8x128_e5m2":
        return 32, lambda seed, layer, device="cpu": kv_cache_layer_e5m2(seed, layer, 65536, device)
    if name == "kv_cache_32x2x32768x8x128_fp16":
        return 32, lambda seed, layer, device="cpu": kv_cache_layer_fp16(seed, layer, 32768, device)
    raise KeyError(name)


def make(name, seed, device="cpu"):
    """Whole tensor of a workload (raw bits, flat), on `device`; drawn with the
    CPU generator."""
    if name == "kv_tile_1x1024x8x128_bf16":
        return kv_tile_k_only(seed).to(device)
    if name == "llama_layer_2x8192x8x128_bf16":
        return llama_layer_kv(seed).to(device)
    if name == "escape_stress_64x65536_bf16":
        return escape_stress(seed).to(device)
    n_layers, layer = layers_of(name)
    return make_layers(name, seed, n_layers, device)


def make_layers(name, seed, n_layers, device="cpu", first=0):
    """Layers first .. first + n_layers - 1 of a 32-layer cache, filled one
    layer at a time."""
    _, layer = layers_of(name)
    head = layer(seed, first, device)
    out = torch.empty(n_layers * head.numel(), dtype=head.dtype, device=device)
    out[: head.numel()].copy_(head)
    del head
    per = out.numel() // n_layers
    for l in range(1, n_layers):
        out[l * per: (l + 1) * per].copy_(layer(seed, first + l, device))
    return out


def calibration_tensor(name, device="cpu"):
    """The tensor each workload's codebook is calibrated on: seed 1 of the same
    recipe (for the 32-layer caches: layer 0 of seed 1)."""
    if name in ("kv_cache_32x2x32768x8x128_bf16", "kv_cache_32x2x65536x8x128_e5m2",
                "kv_cache_32x2x32768x8x128_fp16"):
        _, layer = layers_of(name)
        return layer(1, 0, device)
    return make(name, 1, device)


def dtype_of(name):
    return WORKLOADS[name][0]


def numel(name):
    return WORKLOADS[name][1]


def bytes_per_element(dtype):
    return 1 if dtype == 1 else 2


def gigabytes(n_bytes):
    return n_bytes / 1e9

