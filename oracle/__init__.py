"""ctypes wrapper around the SplitZip CPU oracle (oracle/splitzip_oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use it; the product package never does.

Arrays are numpy arrays of raw bits: BF16 and FP16 as ``uint16``, FP8-E5M2 as
``uint8``.
"""
import ctypes

import numpy as np

from . import build_oracle

BF16 = 0
E5M2 = 1
FP16 = 2
OK, INVALID, CAPACITY, CORRUPT = 0, 1, 2, 3

_lib = None


class Header(ctypes.Structure):
    _fields_ = [
        ("n", ctypes.c_uint64),
        ("total_escapes", ctypes.c_uint64),
        ("size", ctypes.c_uint64),
        ("chunk_elems", ctypes.c_uint32),
        ("n_chunks", ctypes.c_uint32),
        ("dtype", ctypes.c_uint8),
        ("codebook", ctypes.c_uint8 * 16),
    ]


def lib():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        L = ctypes.CDLL(path)
        u64, u32, i32, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p
        L.oracle_container_size.restype = u64
        L.oracle_container_size.argtypes = [u64, i32, u32, u64]
        L.oracle_histogram.restype = i32
        L.oracle_histogram.argtypes = [vp, u64, i32, vp]
        L.oracle_calibrate.restype = i32
        L.oracle_calibrate.argtypes = [vp, i32, vp]
        L.oracle_chunk_escape_counts.restype = i32
        L.oracle_chunk_escape_counts.argtypes = [vp, u64, i32, vp, u32, vp]
        L.oracle_encode.restype = i32
        L.oracle_encode.argtypes = [vp, u64, i32, vp, u32, vp, u64, ctypes.POINTER(u64)]
        L.oracle_decode.restype = i32
        L.oracle_decode.argtypes = [vp, u64, vp, u64, i32]
        L.oracle_parse_header.restype = i32
        L.oracle_parse_header.argtypes = [vp, u64, ctypes.POINTER(Header)]
        L.oracle_variant_size.restype = u64
        L.oracle_variant_size.argtypes = [u64, i32, u32, i32, u64]
        L.oracle_encode_variant.restype = i32
        L.oracle_encode_variant.argtypes = [vp, u64, i32, vp, u32, i32, vp, u64, ctypes.POINTER(u64)]
        L.oracle_decode_variant.restype = i32
        L.oracle_decode_variant.argtypes = [vp, u64, vp, u64, i32]
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None and a.size else None


def _check_bits(x, dtype):
    want = np.uint8 if dtype == E5M2 else np.uint16
    x = np.ascontiguousarray(x)
    if x.dtype != want:
        raise TypeError("dtype %d wants %s bits, got %s" % (dtype, want.__name__, x.dtype))
    return x.reshape(-1)


def container_size(n, dtype, chunk_elems, total_escapes):
    return int(lib().oracle_container_size(n, dtype, chunk_elems, total_escapes))


def max_container_size(n, dtype, chunk_elems):
    return container_size(n, dtype, chunk_elems, n)


def histogram(x, dtype):
    x = _check_bits(x, dtype)
    h = np.zeros(256, dtype=np.uint64)
    st = lib().oracle_histogram(_ptr(x), x.size, dtype, _ptr(h))
    if st != OK:
        raise ValueError("oracle_histogram status %d" % st)
    return h


def calibrate(hist, dtype):
    hist = np.ascontiguousarray(hist, dtype=np.uint64)
    assert hist.size == 256
    cb = np.zeros(16, dtype=np.uint8)
    st = lib().oracle_calibrate(_ptr(hist), dtype, _ptr(cb))
    if st != OK:
        raise ValueError("oracle_calibrate status %d" % st)
    return cb


def chunk_escape_counts(x, dtype, codebook, chunk_elems):
    x = _check_bits(x, dtype)
    cb = np.ascontiguousarray(codebook, dtype=np.uint8)
    C = (x.size + chunk_elems - 1) // chunk_elems
    counts = np.zeros(max(C, 1), dtype=np.uint32)
    st = lib().oracle_chunk_escape_counts(_ptr(x), x.size, dtype, _ptr(cb), chunk_elems, _ptr(counts))
    if st != OK:
        raise ValueError("oracle_chunk_escape_counts status %d" % st)
    return counts[:C]


def encode(x, dtype, codebook, chunk_elems=65536):
    """Return the container bytes (numpy uint8) for ``x``."""
    x = _check_bits(x, dtype)
    cb = np.ascontiguousarray(codebook, dtype=np.uint8)
    cap = max_container_size(x.size, dtype, chunk_elems)
    out = np.zeros(cap, dtype=np.uint8)
    size = ctypes.c_uint64(0)
    st = lib().oracle_encode(_ptr(x), x.size, dtype, _ptr(cb), chunk_elems, _ptr(out), cap, ctypes.byref(size))
    if st != OK:
        raise ValueError("oracle_encode status %d" % st)
    return out[: size.value].copy()


def decode_status(blob, n, dtype):
    """Decode ``blob``; return (status, decoded bits)."""
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    out = np.zeros(n, dtype=np.uint8 if dtype == E5M2 else np.uint16)
    st = lib().oracle_decode(_ptr(blob), blob.size, _ptr(out), n, dtype)
    return st, out


def decode(blob, n, dtype):
    st, out = decode_status(blob, n, dtype)
    if st != OK:
        raise ValueError("oracle_decode status %d" % st)
    return out


def parse_header(blob):
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    h = Header()
    st = lib().oracle_parse_header(_ptr(blob), blob.size, ctypes.byref(h))
    return st, h


# ---------------------------------------------------------------- ablation variants
# (Results, "Ablation Studies"): 1 = Top-8 with 3-bit codes, 2 = Top-15 with a
# sentinel code; 0 = the main format.  See READINGS V1-V3 in splitzip_oracle.c.
TOP16, TOP8, TOP15_SENTINEL = 0, 1, 2


def variant_codebook(codebook16, variant):
    """The variant's codebook: the first k exponents of the Top-16 order (the
    same selection stopped at k), the remaining bytes zero."""
    k = {TOP16: 16, TOP8: 8, TOP15_SENTINEL: 15}[variant]
    cb = np.zeros(16, dtype=np.uint8)
    cb[:k] = np.asarray(codebook16, dtype=np.uint8)[:k]
    return cb


def variant_size(n, dtype, chunk_elems, variant, total_escapes):
    return int(lib().oracle_variant_size(n, dtype, chunk_elems, variant, total_escapes))


def encode_variant(x, dtype, codebook, chunk_elems, variant):
    x = _check_bits(x, dtype)
    cb = np.ascontiguousarray(codebook, dtype=np.uint8)
    cap = variant_size(x.size, dtype, chunk_elems, variant, x.size)
    out = np.zeros(max(cap, 1), dtype=np.uint8)
    size = ctypes.c_uint64(0)
    st = lib().oracle_encode_variant(_ptr(x), x.size, dtype, _ptr(cb), chunk_elems, variant, _ptr(out), cap,
                                     ctypes.byref(size))
    if st != OK:
        raise ValueError("oracle_encode_variant status %d" % st)
    return out[: size.value].copy()


def decode_variant_status(blob, n, dtype):
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    out = np.zeros(n, dtype=np.uint16 if dtype == BF16 else np.uint8)
    st = lib().oracle_decode_variant(_ptr(blob), blob.size, _ptr(out), n, dtype)
    return st, out


def decode_variant(blob, n, dtype):
    st, out = decode_variant_status(blob, n, dtype)
    if st != OK:
        raise ValueError("oracle_decode_variant status %d" % st)
    return out
