"""SplitZip lossless KV-cache codec for GB300 (sm_103a).

Thin ctypes binding of the C ABI in include/splitzip.h: the ``splitzip_*``
functions below take the same arguments as the C entry points (device
pointers as Python ints, a CUDA stream handle as an int) and return the same
status codes.  Every step of the codec runs in the CUDA kernels of
``libsplitzip.so``; this module only marshals arguments.  The torch helpers at
the end (``calibrate``, ``encode``, ``decode``) allocate device memory with
torch and call the same entry points.

Method: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
Serving", section "Method: SplitZip".
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsplitzip.so")

BF16 = 0
FP8_E5M2 = 1
FP16 = 2
OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_CORRUPT, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = range(7)
DEFAULT_CHUNK_ELEMS = 65536
HEADER_BYTES = 64
NOALLOC_SCRATCH_BYTES = 32 << 20  # SPLITZIP_NOALLOC_SCRATCH_BYTES


class SplitZipError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, splitzip_status_string(status), status))


class Codebook(ctypes.Structure):
    """splitzip_codebook_t: code i stands for exponent exps[i]."""
    _fields_ = [("dtype", ctypes.c_uint8), ("exps", ctypes.c_uint8 * 16)]

    def values(self):
        return list(self.exps)

    @classmethod
    def make(cls, dtype, exps):
        cb = cls()
        cb.dtype = dtype
        for i, e in enumerate(exps):
            cb.exps[i] = int(e)
        return cb


class Header(ctypes.Structure):
    """splitzip_header_t."""
    _fields_ = [
        ("n_elems", ctypes.c_uint64),
        ("total_escapes", ctypes.c_uint64),
        ("size", ctypes.c_uint64),
        ("index_off", ctypes.c_uint64),
        ("counts_off", ctypes.c_uint64),
        ("nibble_off", ctypes.c_uint64),
        ("signmant_off", ctypes.c_uint64),
        ("escrec_off", ctypes.c_uint64),
        ("chunk_elems", ctypes.c_uint32),
        ("n_chunks", ctypes.c_uint32),
        ("dtype", ctypes.c_uint8),
        ("codebook", ctypes.c_uint8 * 16),
    ]


class EncodeItem(ctypes.Structure):
    """splitzip_encode_item_t."""
    _fields_ = [("d_in", ctypes.c_void_p), ("n", ctypes.c_uint64), ("d_out", ctypes.c_void_p),
                ("out_capacity", ctypes.c_uint64), ("d_out_size", ctypes.c_void_p)]


class DecodeItem(ctypes.Structure):
    """splitzip_decode_item_t."""
    _fields_ = [("d_in", ctypes.c_void_p), ("in_bytes", ctypes.c_uint64), ("d_out", ctypes.c_void_p),
                ("n", ctypes.c_uint64)]


MAX_BATCH = 256                 # SPLITZIP_MAX_BATCH
MAX_BATCH_ITEM_ELEMS = 1 << 26  # SPLITZIP_MAX_BATCH_ITEM_ELEMS


class _Address(ctypes.c_void_p):
    """A pointer argument: an integer address, None (NULL), or an object with
    data_ptr() (a torch tensor).  Anything else -- notably a str or bytes, which
    plain c_void_p would turn into the address of its host buffer -- is a
    TypeError, so a wrong value never reaches a kernel as an address."""

    @classmethod
    def from_param(cls, obj):
        if obj is None or isinstance(obj, bool):
            if obj is None:
                return None
            raise TypeError("pointer argument: expected an address, got bool")
        if isinstance(obj, int):
            return ctypes.c_void_p(obj)
        if isinstance(obj, ctypes.c_void_p):
            return obj
        if hasattr(obj, "data_ptr"):
            return ctypes.c_void_p(obj.data_ptr())
        raise TypeError("pointer argument: expected an integer address, None or a tensor, got %s"
                        % type(obj).__name__)


_u64, _u32, _int, _vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, _Address
_P_u64 = ctypes.POINTER(ctypes.c_uint64)

# name -> (restype, argtypes); mirrors include/splitzip.h
SIGNATURES = {
    "splitzip_status_string": (ctypes.c_char_p, [_int]),
    "splitzip_exponent_histogram": (_int, [_vp, _u64, _int, _vp, _vp]),
    "splitzip_calibrate": (_int, [_vp, _int, _int, ctypes.POINTER(Codebook)]),
    "splitzip_compressed_size": (_int, [_u64, _int, _u32, _u64, _P_u64]),
    "splitzip_max_compressed_size": (_int, [_u64, _int, _u32, _P_u64]),
    "splitzip_encode_workspace_size": (_int, [_u64, _int, _u32, _P_u64]),
    "splitzip_encode": (_int, [_vp, _u64, _int, ctypes.POINTER(Codebook), _u32, _vp, _u64, _vp, _u64, _vp,
                               _vp, _vp]),
    "splitzip_encode_noalloc": (_int, [_vp, _u64, _int, ctypes.POINTER(Codebook), _u32, _vp, _u64, _vp, _vp,
                                       _vp]),
    "splitzip_decode": (_int, [_vp, _u64, _vp, _u64, _int, _vp, _vp]),
    "splitzip_parse_header": (_int, [_vp, _u64, ctypes.POINTER(Header)]),
    "splitzip_calibrate_device": (_int, [_vp, _u64, _int, _vp, _vp, _vp]),
    "splitzip_ablation_max_size": (_int, [_u64, _int, _u32, _int, _P_u64]),
    "splitzip_ablation_encode": (_int, [_vp, _u64, _int, ctypes.POINTER(Codebook), _u32, _int, _vp, _u64, _vp, _vp,
                                        _vp]),
    "splitzip_ablation_decode": (_int, [_vp, _u64, _vp, _u64, _int, _int, _vp, _vp]),
    "splitzip_encode_paged": (_int, [_vp, _u64, _vp, _u64, _u64, _int, ctypes.POINTER(Codebook), _u32, _vp, _u64, _vp,
                                     _u64, _vp, _vp, _vp]),
    "splitzip_decode_paged": (_int, [_vp, _u64, _vp, _u64, _vp, _u64, _u64, _int, _vp, _vp]),
    "splitzip_encode_device_codebook": (_int, [_vp, _u64, _int, _vp, _u32, _vp, _u64, _vp, _u64, _vp, _vp, _vp]),
    "splitzip_transfer_scratch_size": (_int, [_u64, _int, _u32, _u64, _int, _P_u64, _P_u64]),
    "splitzip_transfer": (_int, [_vp, _vp, _u64, _int, ctypes.POINTER(Codebook), _u32, _u64, _int, _vp, _u64, _vp,
                                 _u64, _P_u64, ctypes.POINTER(ctypes.c_float), _vp]),
    "splitzip_selftest_bounded_wait": (_int, [_u64, _vp, _vp, _vp]),
    "splitzip_merge": (_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_uint64), _u32, _vp, _u64,
                              _P_u64]),
    "splitzip_encode_batch_workspace_size": (_int, [ctypes.POINTER(ctypes.c_uint64), _u32, _int, _u32, _P_u64]),
    "splitzip_encode_batch": (_int, [ctypes.POINTER(EncodeItem), _u32, _int, ctypes.POINTER(Codebook), _u32, _vp,
                                     _u64, _vp, _vp]),
    "splitzip_decode_batch": (_int, [ctypes.POINTER(DecodeItem), _u32, _int, _vp, _vp]),
}

_lib = None


def lib():
    """The loaded libsplitzip.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libsplitzip.so is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ---------------------------------------------------------------- C entry points

def splitzip_status_string(status):
    return lib().splitzip_status_string(status).decode()


def splitzip_exponent_histogram(d_x, n, dtype, d_hist256, stream):
    return lib().splitzip_exponent_histogram(d_x, n, dtype, d_hist256, stream)


def splitzip_calibrate(hist256, hist_is_device, dtype, out_cb):
    return lib().splitzip_calibrate(hist256, hist_is_device, dtype, ctypes.byref(out_cb))


def splitzip_compressed_size(n, dtype, chunk_elems, total_escapes, out_bytes):
    return lib().splitzip_compressed_size(n, dtype, chunk_elems, total_escapes, ctypes.byref(out_bytes))


def splitzip_max_compressed_size(n, dtype, chunk_elems, out_bytes):
    return lib().splitzip_max_compressed_size(n, dtype, chunk_elems, ctypes.byref(out_bytes))


def splitzip_encode_workspace_size(n, dtype, chunk_elems, out_bytes):
    return lib().splitzip_encode_workspace_size(n, dtype, chunk_elems, ctypes.byref(out_bytes))


def splitzip_encode(d_in, n, dtype, cb, chunk_elems, d_out, out_capacity, d_ws, ws_bytes, d_out_size,
                    d_status, stream):
    return lib().splitzip_encode(d_in, n, dtype, ctypes.byref(cb), chunk_elems, d_out, out_capacity, d_ws,
                                 ws_bytes, d_out_size, d_status, stream)


def splitzip_encode_noalloc(d_in, n, dtype, cb, chunk_elems, d_out, out_capacity, d_out_size, d_status, stream):
    return lib().splitzip_encode_noalloc(d_in, n, dtype, ctypes.byref(cb), chunk_elems, d_out, out_capacity,
                                         d_out_size, d_status, stream)


def splitzip_decode(d_in, in_bytes, d_out, n, dtype, d_status, stream):
    return lib().splitzip_decode(d_in, in_bytes, d_out, n, dtype, d_status, stream)


def splitzip_parse_header(h_blob, nbytes, out):
    return lib().splitzip_parse_header(h_blob, nbytes, ctypes.byref(out))


def splitzip_encode_paged(d_pool, pool_pages, d_pages, n_pages, page_elems, dtype, cb, chunk_elems, d_out,
                          out_capacity, d_ws, ws_bytes, d_out_size, d_status, stream):
    return lib().splitzip_encode_paged(d_pool, pool_pages, d_pages, n_pages, page_elems, dtype, ctypes.byref(cb),
                                       chunk_elems, d_out, out_capacity, d_ws, ws_bytes, d_out_size, d_status, stream)


def splitzip_decode_paged(d_in, in_bytes, d_pool, pool_pages, d_pages, n_pages, page_elems, dtype, d_status, stream):
    return lib().splitzip_decode_paged(d_in, in_bytes, d_pool, pool_pages, d_pages, n_pages, page_elems, dtype,
                                       d_status, stream)


def splitzip_ablation_max_size(n, dtype, chunk_elems, variant, out_bytes):
    return lib().splitzip_ablation_max_size(n, dtype, chunk_elems, variant, ctypes.byref(out_bytes))


def splitzip_ablation_encode(d_in, n, dtype, cb, chunk_elems, variant, d_out, out_capacity, d_out_size, d_status,
                             stream):
    return lib().splitzip_ablation_encode(d_in, n, dtype, ctypes.byref(cb), chunk_elems, variant, d_out,
                                          out_capacity, d_out_size, d_status, stream)


def splitzip_ablation_decode(d_in, in_bytes, d_out, n, dtype, variant, d_status, stream):
    return lib().splitzip_ablation_decode(d_in, in_bytes, d_out, n, dtype, variant, d_status, stream)


def splitzip_calibrate_device(d_x, n, dtype, d_hist256, d_cb, stream):
    return lib().splitzip_calibrate_device(d_x, n, dtype, d_hist256, d_cb, stream)


def splitzip_encode_device_codebook(d_in, n, dtype, d_cb, chunk_elems, d_out, out_capacity, d_ws, ws_bytes,
                                    d_out_size, d_status, stream):
    return lib().splitzip_encode_device_codebook(d_in, n, dtype, d_cb, chunk_elems, d_out, out_capacity, d_ws,
                                                 ws_bytes, d_out_size, d_status, stream)


def splitzip_transfer_scratch_size(n, dtype, chunk_elems, piece_elems, compress, out_device_bytes, out_host_bytes):
    return lib().splitzip_transfer_scratch_size(n, dtype, chunk_elems, piece_elems, compress,
                                                ctypes.byref(out_device_bytes), ctypes.byref(out_host_bytes))


def splitzip_transfer(d_src, d_dst, n, dtype, cb, chunk_elems, piece_elems, compress, d_scratch, d_scratch_bytes,
                      h_stage, h_stage_bytes, out_link_bytes, out_ms, stream):
    """out_link_bytes: ctypes.c_uint64 or None; out_ms: ctypes.c_float or None."""
    return lib().splitzip_transfer(d_src, d_dst, n, dtype, None if cb is None else ctypes.byref(cb), chunk_elems,
                                   piece_elems, compress, d_scratch, d_scratch_bytes, h_stage, h_stage_bytes,
                                   None if out_link_bytes is None else ctypes.byref(out_link_bytes),
                                   None if out_ms is None else ctypes.byref(out_ms), stream)


def splitzip_selftest_bounded_wait(limit_cycles, d_status, d_cycles, stream):
    return lib().splitzip_selftest_bounded_wait(limit_cycles, d_status, d_cycles, stream)


def splitzip_merge(h_parts, part_bytes, count, h_out, out_capacity, out_bytes):
    """h_parts: ctypes array of c_void_p; part_bytes: ctypes array of c_uint64."""
    return lib().splitzip_merge(h_parts, part_bytes, count, h_out, out_capacity, ctypes.byref(out_bytes))


def splitzip_encode_batch_workspace_size(h_n, count, dtype, chunk_elems, out_bytes):
    """h_n: ctypes array of c_uint64."""
    return lib().splitzip_encode_batch_workspace_size(h_n, count, dtype, chunk_elems, ctypes.byref(out_bytes))


def splitzip_encode_batch(h_items, count, dtype, cb, chunk_elems, d_ws, ws_bytes, d_status, stream):
    """h_items: ctypes array of EncodeItem."""
    return lib().splitzip_encode_batch(h_items, count, dtype, ctypes.byref(cb), chunk_elems, d_ws, ws_bytes, d_status,
                                       stream)


def splitzip_decode_batch(h_items, count, dtype, d_status, stream):
    """h_items: ctypes array of DecodeItem."""
    return lib().splitzip_decode_batch(h_items, count, dtype, d_status, stream)


# ------------------------------------------------------------ size helpers

def _size_call(fn, *args):
    out = ctypes.c_uint64(0)
    st = fn(*args, out)
    if st != OK:
        raise SplitZipError(st, fn.__name__)
    return out.value


def max_compressed_size(n, dtype, chunk_elems=DEFAULT_CHUNK_ELEMS):
    return _size_call(splitzip_max_compressed_size, n, dtype, chunk_elems)


def compressed_size(n, dtype, chunk_elems, total_escapes):
    return _size_call(splitzip_compressed_size, n, dtype, chunk_elems, total_escapes)


def workspace_size(n, dtype, chunk_elems=DEFAULT_CHUNK_ELEMS):
    return _size_call(splitzip_encode_workspace_size, n, dtype, chunk_elems)


def merge(parts):
    """Join host containers (numpy uint8 arrays, tensor order) of consecutive
    whole-chunk pieces into the container of the whole tensor (numpy uint8)."""
    import numpy as np
    arrs = [np.ascontiguousarray(p, dtype=np.uint8) for p in parts]
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    sizes = (ctypes.c_uint64 * len(arrs))(*[a.size for a in arrs])
    total = ctypes.c_uint64(0)
    _check(splitzip_merge(ptrs, sizes, len(arrs), None, 0, total), "splitzip_merge")
    out = np.empty(max(total.value, 1), dtype=np.uint8)
    _check(splitzip_merge(ptrs, sizes, len(arrs), out.ctypes.data, out.size, total), "splitzip_merge")
    return out[: total.value]


def parse_header(blob_bytes):
    """Header of a container held in host memory (bytes / numpy / torch CPU)."""
    import numpy as np
    buf = np.ascontiguousarray(np.frombuffer(bytes(blob_bytes), dtype=np.uint8)) \
        if isinstance(blob_bytes, (bytes, bytearray)) else np.ascontiguousarray(blob_bytes).view(np.uint8)
    h = Header()
    st = splitzip_parse_header(buf.ctypes.data, buf.size, h)
    if st != OK:
        raise SplitZipError(st, "splitzip_parse_header")
    return h


# ------------------------------------------------------------ torch helpers

def _torch():
    import torch
    return torch


def _stream_handle(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _bits_dtype(dtype):
    torch = _torch()
    return torch.uint8 if dtype == FP8_E5M2 else torch.int16


def _check(st, where):
    if st != OK:
        raise SplitZipError(st, where)


def calibrate(x, dtype, stream=None):
    """Exponent histogram of the device tensor ``x`` (raw bits) on the GPU,
    then the Top-16 codebook.  Synchronises."""
    torch = _torch()
    hist = torch.empty(256, dtype=torch.int64, device=x.device)
    _check(splitzip_exponent_histogram(x.data_ptr(), x.numel(), dtype, hist.data_ptr(), _stream_handle(stream)),
           "splitzip_exponent_histogram")
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    h = hist.cpu()
    cb = Codebook()
    _check(splitzip_calibrate(h.data_ptr(), 0, dtype, cb), "splitzip_calibrate")
    return cb, h


class EncodeBuffers:
    """Device buffers for one encode of n elements (capacity-sized)."""

    def __init__(self, n, dtype, chunk_elems=DEFAULT_CHUNK_ELEMS, device="cuda"):
        torch = _torch()
        self.n, self.dtype, self.chunk_elems = n, dtype, chunk_elems
        self.capacity = max_compressed_size(n, dtype, chunk_elems)
        self.ws_bytes = workspace_size(n, dtype, chunk_elems)
        self.out = torch.empty(self.capacity, dtype=torch.uint8, device=device)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
        self.size = torch.zeros(2, dtype=torch.int64, device=device)   # [0] = container bytes
        self.status = torch.zeros(4, dtype=torch.int32, device=device)  # [0] = status


def encode_into(x, cb, bufs, stream=None):
    """Enqueue the encode of device tensor ``x`` into ``bufs`` (asynchronous)."""
    _check(splitzip_encode(x.data_ptr(), x.numel(), bufs.dtype, cb, bufs.chunk_elems, bufs.out.data_ptr(),
                           bufs.capacity, bufs.ws.data_ptr(), bufs.ws_bytes, bufs.size.data_ptr(),
                           bufs.status.data_ptr(), _stream_handle(stream)), "splitzip_encode")


def encode(x, cb, dtype, chunk_elems=DEFAULT_CHUNK_ELEMS, stream=None):
    """Encode device tensor ``x``; returns the container as a uint8 device
    tensor of its exact size.  Synchronises to read the size."""
    bufs = EncodeBuffers(x.numel(), dtype, chunk_elems, device=x.device)
    encode_into(x, cb, bufs, stream)
    size, status = int(bufs.size[0].item()), int(bufs.status[0].item())
    _check(status, "splitzip_encode (device)")
    return bufs.out[:size]


def decode_into(blob, in_bytes, out, n, dtype, status, stream=None):
    _check(splitzip_decode(blob.data_ptr(), in_bytes, out.data_ptr() if n else 0, n, dtype, status.data_ptr(),
                           _stream_handle(stream)), "splitzip_decode")


def decode(blob, n, dtype, stream=None):
    """Decode a device container into a new device tensor of raw bits."""
    torch = _torch()
    out = torch.empty(max(n, 1), dtype=_bits_dtype(dtype), device=blob.device)
    status = torch.zeros(4, dtype=torch.int32, device=blob.device)
    decode_into(blob, blob.numel(), out, n, dtype, status, stream)
    _check(int(status[0].item()), "splitzip_decode (device)")
    return out[:n]


def batch_workspace_size(ns, dtype, chunk_elems=DEFAULT_CHUNK_ELEMS):
    arr = (ctypes.c_uint64 * len(ns))(*ns)
    out = ctypes.c_uint64(0)
    _check(splitzip_encode_batch_workspace_size(arr, len(ns), dtype, chunk_elems, out),
           "splitzip_encode_batch_workspace_size")
    return out.value


def encode_batch(xs, cb, dtype, chunk_elems=DEFAULT_CHUNK_ELEMS, stream=None):
    """Encode each device tensor of ``xs`` into its own container with one
    batched call; returns the containers (uint8 device tensors of their exact
    sizes).  Synchronises to read the sizes."""
    torch = _torch()
    dev = xs[0].device
    caps = [max_compressed_size(x.numel(), dtype, chunk_elems) for x in xs]
    outs = [torch.empty(c, dtype=torch.uint8, device=dev) for c in caps]
    sizes = torch.zeros(len(xs), dtype=torch.int64, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    ws_bytes = batch_workspace_size([x.numel() for x in xs], dtype, chunk_elems)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    items = (EncodeItem * len(xs))()
    for i, (x, o, c) in enumerate(zip(xs, outs, caps)):
        items[i] = EncodeItem(x.data_ptr() if x.numel() else 0, x.numel(), o.data_ptr(), c,
                              sizes.data_ptr() + 8 * i)
    _check(splitzip_encode_batch(items, len(xs), dtype, cb, chunk_elems, ws.data_ptr(), ws_bytes, status.data_ptr(),
                                 _stream_handle(stream)), "splitzip_encode_batch")
    _check(int(status[0].item()), "splitzip_encode_batch (device)")
    return [o[: int(n)] for o, n in zip(outs, sizes.cpu().tolist())]


def decode_batch_status(blobs, ns, dtype, stream=None):
    """Decode device containers ``blobs`` (element counts ``ns``) with one
    batched call; returns (device status, decoded tensors)."""
    torch = _torch()
    dev = blobs[0].device
    outs = [torch.empty(max(n, 1), dtype=_bits_dtype(dtype), device=dev) for n in ns]
    status = torch.full((4,), -1, dtype=torch.int32, device=dev)
    items = (DecodeItem * len(blobs))()
    for i, (b, o, n) in enumerate(zip(blobs, outs, ns)):
        items[i] = DecodeItem(b.data_ptr(), b.numel(), o.data_ptr() if n else 0, n)
    _check(splitzip_decode_batch(items, len(blobs), dtype, status.data_ptr(), _stream_handle(stream)),
           "splitzip_decode_batch")
    return int(status[0].item()), [o[:n] for o, n in zip(outs, ns)]


def transfer_scratch_size(n, dtype, piece_elems, compress=True, chunk_elems=DEFAULT_CHUNK_ELEMS):
    """(device bytes, pinned host bytes) that splitzip_transfer needs."""
    d, h = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check(splitzip_transfer_scratch_size(n, dtype, chunk_elems, piece_elems, int(compress), d, h),
           "splitzip_transfer_scratch_size")
    return d.value, h.value


class TransferBuffers:
    """Device scratch and pinned host staging for splitzip_transfer."""

    def __init__(self, n, dtype, piece_elems, compress=True, chunk_elems=DEFAULT_CHUNK_ELEMS, device="cuda"):
        torch = _torch()
        self.n, self.dtype, self.piece_elems = n, dtype, piece_elems
        self.compress, self.chunk_elems = bool(compress), chunk_elems
        d, h = transfer_scratch_size(n, dtype, piece_elems, compress, chunk_elems)
        self.device = torch.empty(max(d, 16), dtype=torch.uint8, device=device)
        self.host = torch.empty(max(h, 16), dtype=torch.uint8, pin_memory=True)


def transfer(src, dst, cb, bufs, stream=None):
    """Move device tensor src into dst across the GPU <-> host link (see
    splitzip_transfer); returns (GPU milliseconds, bytes over the link each way)."""
    link, ms = ctypes.c_uint64(0), ctypes.c_float(0.0)
    _check(splitzip_transfer(src.data_ptr(), dst.data_ptr(), bufs.n, bufs.dtype, cb if bufs.compress else None,
                             bufs.chunk_elems, bufs.piece_elems, int(bufs.compress), bufs.device.data_ptr(),
                             bufs.device.numel(), bufs.host.data_ptr(), bufs.host.numel(), link, ms,
                             _stream_handle(stream)), "splitzip_transfer")
    return ms.value, link.value


def calibrate_device(x, dtype, hist=None, cb=None, stream=None):
    """Online calibration on the device (no host synchronisation): returns
    (histogram, codebook) as device tensors (256 int64; 17 uint8 laid out as
    splitzip_codebook_t: dtype, then the 16 exponents)."""
    torch = _torch()
    hist = torch.empty(256, dtype=torch.int64, device=x.device) if hist is None else hist
    cb = torch.empty(32, dtype=torch.uint8, device=x.device) if cb is None else cb
    _check(splitzip_calibrate_device(x.data_ptr(), x.numel(), dtype, hist.data_ptr(), cb.data_ptr(),
                                     _stream_handle(stream)), "splitzip_calibrate_device")
    return hist, cb


def encode_into_device_codebook(x, d_cb, bufs, stream=None):
    """encode_into with the codebook in device memory (see calibrate_device)."""
    _check(splitzip_encode_device_codebook(x.data_ptr(), x.numel(), bufs.dtype, d_cb.data_ptr(), bufs.chunk_elems,
                                           bufs.out.data_ptr(), bufs.capacity, bufs.ws.data_ptr(), bufs.ws_bytes,
                                           bufs.size.data_ptr(), bufs.status.data_ptr(), _stream_handle(stream)),
           "splitzip_encode_device_codebook")


def encode_paged_into(pool, pages, page_elems, cb, bufs, stream=None):
    """Encode the pages `pages` (device int32 tensor) of `pool` (a device tensor
    of whole pages, raw bits) into `bufs` (sized for len(pages) * page_elems)."""
    _check(splitzip_encode_paged(pool.data_ptr(), pool.numel() // page_elems, pages.data_ptr(), pages.numel(),
                                 page_elems, bufs.dtype, cb, bufs.chunk_elems, bufs.out.data_ptr(), bufs.capacity,
                                 bufs.ws.data_ptr(), bufs.ws_bytes, bufs.size.data_ptr(), bufs.status.data_ptr(),
                                 _stream_handle(stream)), "splitzip_encode_paged")


def decode_paged_into(blob, in_bytes, pool, pages, page_elems, dtype, status, stream=None):
    """Decode a container into the pages `pages` of `pool`."""
    _check(splitzip_decode_paged(blob.data_ptr(), in_bytes, pool.data_ptr(), pool.numel() // page_elems,
                                 pages.data_ptr(), pages.numel(), page_elems, dtype, status.data_ptr(),
                                 _stream_handle(stream)), "splitzip_decode_paged")


# ablation formats (see splitzip_ablation_encode): 0 = Top-16, 1 = Top-8, 2 = Top-15 + sentinel
ABL_TOP16, ABL_TOP8, ABL_TOP15_SENTINEL = 0, 1, 2
ABL_CODES = {ABL_TOP16: 16, ABL_TOP8: 8, ABL_TOP15_SENTINEL: 15}


def ablation_codebook(cb16, variant):
    """The variant's codebook: the first k exponents of a Top-16 codebook, then zeros."""
    k = ABL_CODES[variant]
    vals = list(cb16.values())[:k]
    c = Codebook()
    c.dtype = cb16.dtype
    for i in range(16):
        c.exps[i] = vals[i] if i < k else 0
    return c


def ablation_max_size(n, dtype, variant, chunk_elems=DEFAULT_CHUNK_ELEMS):
    return _size_call(splitzip_ablation_max_size, n, dtype, chunk_elems, variant)


def ablation_encode(x, cb, dtype, variant, chunk_elems=DEFAULT_CHUNK_ELEMS, stream=None):
    """Encode device tensor x in an ablation format; returns the container
    (uint8 device tensor of its exact size).  Synchronises."""
    torch = _torch()
    cap = ablation_max_size(x.numel(), dtype, variant, chunk_elems)
    out = torch.empty(max(cap, 16), dtype=torch.uint8, device=x.device)
    size = torch.zeros(2, dtype=torch.int64, device=x.device)
    status = torch.zeros(4, dtype=torch.int32, device=x.device)
    _check(splitzip_ablation_encode(x.data_ptr(), x.numel(), dtype, cb, chunk_elems, variant, out.data_ptr(), cap,
                                    size.data_ptr(), status.data_ptr(), _stream_handle(stream)),
           "splitzip_ablation_encode")
    _check(int(status[0].item()), "splitzip_ablation_encode (device)")
    return out[: int(size[0].item())]


def ablation_decode_status(blob, n, dtype, variant, stream=None):
    torch = _torch()
    out = torch.empty(max(n, 1), dtype=_bits_dtype(dtype), device=blob.device)
    status = torch.full((4,), -1, dtype=torch.int32, device=blob.device)
    _check(splitzip_ablation_decode(blob.data_ptr(), blob.numel(), out.data_ptr() if n else 0, n, dtype, variant,
                                    status.data_ptr(), _stream_handle(stream)), "splitzip_ablation_decode")
    return int(status[0].item()), out[:n]
