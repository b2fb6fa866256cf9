"""Benchmark of the SplitZip GB300 codec.

One step = encode + decode of one KV tensor, inputs resident in HBM.  The
default workload is the 32-layer BF16 KV cache (32 x 2 x 32768 x 8 x 128 =
2,147,483,648 elements, 4.29 GB); `--workload` selects another of the five
workloads of lossless_kv_cache_gb300.workloads (for reporting; the default is
the headline line).

Prints one JSON line.  `value` is the round-trip throughput in GB/s of
uncompressed bytes (bytes of the tensor / (encode + decode time)); encode and
decode throughputs, the compression ratio, the escape rate and the derived
link-transfer model are reported beside it, with the end-to-end figure from
pinned host memory, the transfer path, online calibration, paged KV and the
ablation formats.  `cpu_baseline` and `--impl reference` time the CPU oracle
as it stands on a bounded sample of the same workload, in independent
containers on every host core (the single-thread figure beside it).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--layers L]
Under torchrun each rank encodes/decodes its own copy of the workload (chunks
are independent, no data exchange): weak scaling, max time over ranks.
"""
import argparse
import faulthandler
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "encode/decode GB/s (uncompressed) on 1 GB300, % HBM roofline, ratio"
DEFAULT_WORKLOAD = "kv_cache_32x2x32768x8x128_bf16"
CHUNK = 65536
LINKS_GBS = (50.0, 100.0)
L2_BYTES = 129 * 1000 * 1000
ELEMENT_DTYPE = {0: "bf16", 1: "fp8_e5m2", 2: "fp16"}


def signmant_bytes(dtype, n):
    """Bytes of the sign|mantissa stream: BF16 1 per element, E5M2 3 and FP16
    11 per 8 elements."""
    return n if dtype == 0 else (11 if dtype == 2 else 3) * (-(-n // 8))


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--cpu-seconds", type=float, default=8.0, help="oracle wall-time budget for cpu_baseline (all cores; half of it again single-threaded)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--ref-threads", type=int, default=0,
                   help="host threads for the oracle (cpu_baseline and --impl reference); 0 = every core")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-transfer", action="store_true", help="skip the GPU -> host -> GPU transfer leg")
    p.add_argument("--no-online", action="store_true", help="skip the online-calibration leg")
    p.add_argument("--no-paged", action="store_true", help="skip the paged-KV leg")
    p.add_argument("--no-ablation", action="store_true", help="skip the Top-8 / Top-15 + sentinel leg")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the per-workload object (the other four workloads, timed after the headline)")
    p.add_argument("--workload-steps", type=int, default=20, help="timed steps per workload of that object")
    p.add_argument("--no-batch", action="store_true", help="skip the batched-call leg")
    p.add_argument("--shard", action="store_true",
                   help="under torchrun: rank r encodes and decodes chunks [r C / N, (r + 1) C / N) of one tensor "
                        "(strong scaling) instead of a replica of the whole workload (weak scaling)")
    p.add_argument("--layers", type=int, default=32,
                   help="32-layer workloads: encode only L layers (a smaller case for profiling; "
                        "not a bench line)")
    p.add_argument("--first-layer", type=int, default=0,
                   help="with --layers: the first of the L layers (layers 1-2 have the cache's average escape "
                        "rate; layer 0 has the highest)")
    return p.parse_args()


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_over_ranks(x, world, device, op):
    """MAX or SUM of a float over the ranks (the value itself at world 1)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def shard_range(n, chunk, world, rank):
    """Elements [lo, hi) of rank `rank`: a contiguous range of whole chunks,
    chunks split as evenly as possible (the ranks' containers join into the
    container of the whole tensor)."""
    C = -(-n // chunk)
    c0, c1 = C * rank // world, C * (rank + 1) // world
    return min(n, c0 * chunk), min(n, c1 * chunk)


def exclusive_scan_over_ranks(v, world, rank, device):
    """Sum of `v` over the ranks below this one (0 on rank 0) and over all
    ranks: where this rank's escape records start in the joined container."""
    if world == 1:
        return 0, v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.int64, device=device)
    got = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(got, t)
    vals = [int(g.item()) for g in got]
    return sum(vals[:rank]), sum(vals)


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# each call on the full-size caches: the dominant kernels captured one at a
# time at full size (a one-pass metric), the two short index kernels on
# layers 1-2 scaled by tiles, as summarised in the named profile, with the
# SHA-256 of the kernel sources it was taken on.  A figure is reported only
# while the sources still hash to that value.
_ENC_SOURCES = ('encode.cu', 'encode_core.cuh', 'tma_pipeline.cuh', 'splitzip_internal.cuh')
_DEC_SOURCES = ('decode.cu', 'decode_core.cuh', 'tma_pipeline.cuh', 'splitzip_internal.cuh')
TRAFFIC = {
    ("kv_cache_32x2x32768x8x128_bf16", "encode"): {
        "bytes": 8094123264, "sources": _ENC_SOURCES,
        "sha256": "e20cbcf7be70cf4493210d5db80401d531b9d6386a6b9755f517282decc2d489",
        "profile": "profiles/launches_kv_cache_32x2x32768x8x128_bf16.md"},
    ("kv_cache_32x2x32768x8x128_bf16", "decode"): {
        "bytes": 7641231104, "sources": _DEC_SOURCES,
        "sha256": "77df22b2c26f6787138c817c4963244aacac423b302050ebec756faf753e9646",
        "profile": "profiles/launches_kv_cache_32x2x32768x8x128_bf16.md"},
    ("kv_cache_32x2x65536x8x128_e5m2", "encode"): {
        "bytes": 9082352384, "sources": _ENC_SOURCES,
        "sha256": "e20cbcf7be70cf4493210d5db80401d531b9d6386a6b9755f517282decc2d489",
        "profile": "profiles/launches_kv_cache_32x2x65536x8x128_e5m2.md"},
    ("kv_cache_32x2x65536x8x128_e5m2", "decode"): {
        "bytes": 8305438976, "sources": _DEC_SOURCES,
        "sha256": "77df22b2c26f6787138c817c4963244aacac423b302050ebec756faf753e9646",
        "profile": "profiles/launches_kv_cache_32x2x65536x8x128_e5m2.md"},
    ("kv_cache_32x2x32768x8x128_fp16", "encode"): {
        "bytes": 8899424000, "sources": _ENC_SOURCES,
        "sha256": "e20cbcf7be70cf4493210d5db80401d531b9d6386a6b9755f517282decc2d489",
        "profile": "profiles/launches_kv_cache_32x2x32768x8x128_fp16.md"},
    ("kv_cache_32x2x32768x8x128_fp16", "decode"): {
        "bytes": 8429386240, "sources": _DEC_SOURCES,
        "sha256": "77df22b2c26f6787138c817c4963244aacac423b302050ebec756faf753e9646",
        "profile": "profiles/launches_kv_cache_32x2x32768x8x128_fp16.md"},
}

E2E_BLOCKS = 7  # timed blocks of the end-to-end leg (the median one is reported)
TRANSFER_RUNS = 5  # runs of each kind in the transfer leg (medians reported)


def sources_sha256(names):
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "lossless_kv_cache_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload, op):
    """(bytes per launch, profile) when a capture of the current kernel sources exists, else (None, None)."""
    t = TRAFFIC.get((workload, op))
    if t is None or sources_sha256(t["sources"]) != t["sha256"]:
        return None, None
    return t["bytes"], t["profile"]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0}, "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, reasons, n = [], [], set(), 0
        window = [(t, l) for t, l in self.lines if t0 <= t <= t1 + 0.06]
        if not window:  # timed region shorter than the sampling period
            window = self.lines[-3:]
        for _, line in window:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


# ------------------------------------------------------------ workloads

class Workload:
    """One of the five workloads: raw-bit tensors and their sizes."""

    def __init__(self, name, layers=32, first_layer=0):
        from lossless_kv_cache_gb300 import workloads as W
        self.W = W
        self.name = name
        self.dtype = W.dtype_of(name)
        self.elem_bytes = W.bytes_per_element(self.dtype)
        self.layered = name in ("kv_cache_32x2x32768x8x128_bf16", "kv_cache_32x2x65536x8x128_e5m2",
                                "kv_cache_32x2x32768x8x128_fp16")
        self.layers = layers if self.layered else None
        self.first_layer = first_layer if self.layered else 0
        if self.layered and not (0 <= first_layer and layers >= 1 and first_layer + layers <= 32):
            raise SystemExit("--first-layer + --layers must stay within the 32 layers")
        full = W.numel(name)
        self.n = full // 32 * layers if self.layered else full

    def make(self, seed, device):
        if self.layered:
            return self.W.make_layers(self.name, seed, self.layers, device, first=self.first_layer)
        return self.W.make(self.name, seed, device)

    def calibration(self, device):
        return self.W.calibration_tensor(self.name, device)

    def make_range(self, seed, lo, hi, device):
        """Elements [lo, hi) of the workload (the layers that hold them are
        generated, the rest is not)."""
        if not self.layered:
            return self.make(seed, device)[lo:hi].contiguous()
        per = self.n // self.layers
        l0, l1 = lo // per, -(-hi // per)
        x = self.W.make_layers(self.name, seed, l1 - l0, device, first=self.first_layer + l0)
        return x[lo - l0 * per: hi - l0 * per].contiguous()

    def config(self, world, shard=False):
        label = self.name
        if self.layered and self.layers != 32:
            label = "%s (layers %d-%d only: profiling case)" % (self.name, self.first_layer,
                                                                self.first_layer + self.layers - 1)
        return {"workload": label, "elements": self.n,
                "element_dtype": ELEMENT_DTYPE[self.dtype], "chunk_elems": CHUNK,
                "codebook": "Top-16 from the seed-1 calibration tensor"
                            + (" (layer 0)" if self.layered else ""),
                "l2": ("inputs %.2f GB > 129 MB L2 (no flush needed)" % (self.n * self.elem_bytes / 1e9))
                if self.n * self.elem_bytes > L2_BYTES else "L2 flushed (512 MB write) before every step",
                "parallelism": ("chunk-range shards of one tensor, one container per GPU, no collective in the "
                                "data path" if shard else "replicas of the workload per GPU, no collective")
                if world > 1 else "single GPU"}

    def algorithmic_bytes(self, E, n=None):
        """(encode, decode) bytes the method must move for n elements (default:
        the workload's): the elements, the two dense streams, 3 bytes per
        escape record and 12 bytes of index per chunk."""
        n = self.n if n is None else n
        C = -(-n // CHUNK)
        streams = (n + 1) // 2 + signmant_bytes(self.dtype, n)
        moved = n * self.elem_bytes + streams + 3 * E + 12 * C
        return moved, moved


# ---------------------------------------------------- other workloads

def measure_workload(name, steps, warmup, device, hbm):
    """Encode + decode of one workload (seed 0, codebook from its calibration
    tensor), timed like the headline: CUDA events around each call on the
    launching stream, W untimed warm-up steps, a 512 MB L2 flush before every
    step when the input fits in L2; the round trip is checked bit for bit."""
    import lossless_kv_cache_gb300 as sz
    wl = Workload(name)
    n, dtype = wl.n, wl.dtype
    raw = wl.elem_bytes * n
    x = wl.make(0, device)
    cb, _ = sz.calibrate(wl.calibration(device), dtype)
    bufs = sz.EncodeBuffers(n, dtype, CHUNK, device=device)
    out = torch.empty(n, dtype=x.dtype, device=device)
    dstatus = torch.zeros(4, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()
    h = stream.cuda_stream
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device) if raw <= L2_BYTES else None

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        st = sz.splitzip_encode(x.data_ptr(), n, dtype, cb, CHUNK, bufs.out.data_ptr(), bufs.capacity,
                                bufs.ws.data_ptr(), bufs.ws_bytes, bufs.size.data_ptr(), bufs.status.data_ptr(), h)
        if st != sz.OK:
            raise sz.SplitZipError(st, "encode")
        if ev is not None:
            ev[1].record(stream)
        st = sz.splitzip_decode(bufs.out.data_ptr(), bufs.capacity, out.data_ptr(), n, dtype, dstatus.data_ptr(), h)
        if st != sz.OK:
            raise sz.SplitZipError(st, "decode")
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    out.fill_(0)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for ev in evs:
        if flush is not None:
            flush.fill_(7)
        step(ev)
    torch.cuda.synchronize()
    ok = int(bufs.status[0]) == sz.OK and int(dstatus[0]) == sz.OK and bool(torch.equal(out, x))
    enc = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    dec = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    size = int(bufs.size[0])
    E = int(bufs.out[24:32].cpu().numpy().view(np.uint64)[0])
    alg, _ = wl.algorithmic_bytes(E)
    link = {}
    for L in LINKS_GBS:
        t_plain = raw / (L * 1e9)
        link["%d_GBps" % int(L)] = round(t_plain / ((enc + dec) * 1e-3 + size / (L * 1e9)), 4)
    res = {"elements": n, "element_dtype": ELEMENT_DTYPE[dtype], "steps": steps,
           "encode_ms": round(enc, 5), "decode_ms": round(dec, 5),
           "encode_gbs": round(raw / (enc * 1e-3) / 1e9, 2), "decode_gbs": round(raw / (dec * 1e-3) / 1e9, 2),
           "round_trip_gbs": round(raw / ((enc + dec) * 1e-3) / 1e9, 2),
           "encode_hbm_frac": round(alg / (enc * 1e-3) / 1e9 / hbm, 4),
           "decode_hbm_frac": round(alg / (dec * 1e-3) / 1e9 / hbm, 4),
           "ratio": round(raw / size, 5), "escape_rate": round(E / n, 6),
           "link_model_speedup": link, "verified": ok,
           "l2": "flushed (512 MB write) before every step" if flush is not None else "inputs larger than L2"}
    del x, bufs, out, flush
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------- batches

def measure_batch(dtype, device, warmup, pieces=32, steps=10):
    """`pieces` tensors of 1,048,576 elements: per step all of them encoded
    and decoded by single calls, or by one splitzip_encode_batch and one
    splitzip_decode_batch; CUDA events on the launching stream, a 512 MB L2
    flush before every step; every piece checked bit for bit."""
    import ctypes
    import lossless_kv_cache_gb300 as sz
    from lossless_kv_cache_gb300 import workloads as W
    make = W.kv_tile_k_only if dtype == 0 else (lambda seed: W.kv_cache_layer_fp16(seed, 0, tokens=512))
    xs = [make(i).to(device) for i in range(pieces)]
    n = xs[0].numel()
    cb, _ = sz.calibrate(make(1000).to(device), dtype)
    stream = torch.cuda.current_stream()
    h = stream.cuda_stream
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    cap = sz.max_compressed_size(n, dtype)
    outs = torch.empty(pieces, cap, dtype=torch.uint8, device=device)
    sizes = torch.zeros(pieces, dtype=torch.int64, device=device)
    status = torch.zeros(4, dtype=torch.int32, device=device)
    ys = [torch.empty_like(x) for x in xs]
    ws1 = sz.workspace_size(n, dtype)
    ws = torch.empty(max(sz.batch_workspace_size([n] * pieces, dtype), ws1, 16), dtype=torch.uint8, device=device)
    enc_items = (sz.EncodeItem * pieces)(*[sz.EncodeItem(x.data_ptr(), n, outs[i].data_ptr(), cap,
                                                         sizes.data_ptr() + 8 * i) for i, x in enumerate(xs)])
    dec_items = (sz.DecodeItem * pieces)(*[sz.DecodeItem(outs[i].data_ptr(), cap, ys[i].data_ptr(), n)
                                           for i in range(pieces)])
    ws_batch = ws.numel()

    def singles():
        for i, x in enumerate(xs):
            st = sz.splitzip_encode(x.data_ptr(), n, dtype, cb, CHUNK, outs[i].data_ptr(), cap, ws.data_ptr(), ws1,
                                    sizes.data_ptr() + 8 * i, status.data_ptr(), h)
            st |= sz.splitzip_decode(outs[i].data_ptr(), cap, ys[i].data_ptr(), n, dtype, status.data_ptr() + 4, h)
            if st != sz.OK:
                raise sz.SplitZipError(st, "single calls")

    def batched():
        st = sz.splitzip_encode_batch(enc_items, pieces, dtype, cb, CHUNK, ws.data_ptr(), ws_batch, status.data_ptr(), h)
        st |= sz.splitzip_decode_batch(dec_items, pieces, dtype, status.data_ptr() + 4, h)
        if st != sz.OK:
            raise sz.SplitZipError(st, "batched calls")

    res = {}
    for label, fn in (("single_calls", singles), ("batched", batched)):
        for _ in range(max(warmup, 3)):
            fn()
        torch.cuda.synchronize()
        for y in ys:
            y.fill_(0)
        ts = []
        for _ in range(steps):
            flush.fill_(5)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ok = int(status[0]) == sz.OK and int(status[1]) == sz.OK and all(torch.equal(x, y) for x, y in zip(xs, ys))
        ms = statistics.median(ts)
        res[label] = {"ms_per_step": round(ms, 4), "us_per_piece": round(1e3 * ms / pieces, 3),
                      "round_trip_gbs": round(pieces * n * 2 / (ms * 1e-3) / 1e9, 2), "verified": ok}
    res["pieces"] = pieces
    res["piece_elems"] = n
    res["element_dtype"] = ELEMENT_DTYPE[dtype]
    res["speedup"] = round(res["single_calls"]["ms_per_step"] / res["batched"]["ms_per_step"], 3)
    res["what"] = ("per step every piece encoded and decoded (round trip), L2 flushed before the step; median of %d "
                   "steps" % steps)
    del xs, ys, outs, ws, flush
    torch.cuda.empty_cache()
    return res


# --------------------------------------------------------- CPU oracle

def host_cores():
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_block(n, threads):
    """Elements per oracle work item (one container): 16 chunks, fewer when
    the workload is too small to give every thread one, one chunk at least."""
    per_thread = n // max(threads, 1) // CHUNK * CHUNK
    return max(CHUNK, min(16 * CHUNK, per_thread))


def oracle_round_trips(pool, blocks, dtype, cb):
    """Encode + decode each host block with the scalar oracle as it stands,
    the blocks spread over the pool's threads (every block is its own
    container, so the blocks are independent, and the oracle's C calls
    release the GIL); every round trip is checked.  Returns wall seconds."""
    import oracle

    def one(xs):
        y = oracle.decode(oracle.encode(xs, dtype, cb, CHUNK), xs.size, dtype)
        if not np.array_equal(y, xs):
            raise RuntimeError("oracle round trip failed")

    t0 = time.perf_counter()
    list(pool.map(one, blocks))
    return time.perf_counter() - t0


def oracle_throughput(x_dev, dtype, cb_exps, seconds, threads):
    """The oracle on `threads` host threads over the first blocks of the
    workload, in passes over them until `seconds` of wall time are spent;
    returns (GB/s uncompressed, elements, seconds, distinct elements,
    elements per container)."""
    from concurrent.futures import ThreadPoolExecutor
    cb = np.asarray(cb_exps, dtype=np.uint8)
    eb = 1 if dtype == 1 else 2
    block = oracle_block(x_dev.numel(), threads)
    distinct = min(x_dev.numel(), 2 * threads * block)
    host = x_dev[:distinct].cpu().numpy()
    host = host if dtype == 1 else host.view(np.uint16)
    blocks = [host[i: i + block] for i in range(0, distinct, block)]
    done, t_total = 0, 0.0
    with ThreadPoolExecutor(threads) as pool:
        oracle_round_trips(pool, blocks[:threads], dtype, cb)  # warm-up: thread start, library load
        while t_total < seconds:
            t_total += oracle_round_trips(pool, blocks, dtype, cb)
            done += distinct
    return eb * done / t_total / 1e9, done, t_total, distinct, block


# ---------------------------------------------------------------- arms

def run_reference(args, world, rank):
    """The CPU oracle on a bounded sample of the workload, per step."""
    if rank != 0:
        return None
    import oracle
    wl = Workload(args.workload, args.layers, args.first_layer)
    if wl.layered:
        _, layer = wl.W.layers_of(wl.name)
        x = layer(0, 0, "cpu").numpy()  # layer 0 of seed 0
        cal = layer(1, 0, "cpu").numpy()
    else:
        x = wl.make(0, "cpu").numpy()
        cal = wl.calibration("cpu").numpy()
    if wl.dtype != 1:
        x, cal = x.view(np.uint16), cal.view(np.uint16)
    cb = oracle.calibrate(oracle.histogram(cal, wl.dtype), wl.dtype)
    from concurrent.futures import ThreadPoolExecutor
    threads = args.ref_threads or host_cores()
    block = min(oracle_block(x.size, threads), x.size)
    per_step = min(threads * block, x.size - x.size % block)
    times = []
    with ThreadPoolExecutor(threads) as pool:
        for s in range(args.warmup + args.steps):
            off = (s * per_step) % (x.size - per_step + 1)
            xs = x[off: off + per_step]
            blocks = [xs[i: i + block] for i in range(0, per_step, block)]
            dt = oracle_round_trips(pool, blocks, wl.dtype, cb)
            if s >= args.warmup:
                times.append(dt)
    total = sum(times)
    value = wl.elem_bytes * per_step * len(times) / total / 1e9
    sample = ("%d elements of %s per step in %d container(s) of %d elements, encode+decode+check, "
              "scalar C oracle, %d thread(s), one container each at a time" % (
                  per_step, "layer 0" if wl.layered else "the tensor", len(blocks), block, threads))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8" if wl.dtype == 1 else "u16",
        "data": "synthetic (seeded torch CPU generator)", "config": wl.config(world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_ours(args, world, rank, local):
    import lossless_kv_cache_gb300 as sz

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    sz.lib()  # fails loudly when the CUDA library is missing
    wl = Workload(args.workload, args.layers, args.first_layer)
    n, dtype = wl.n, wl.dtype
    raw_bytes = wl.elem_bytes * n

    if args.shard:
        # strong scaling: the ranks split one tensor (seed 0) by whole chunks
        lo, hi = shard_range(wl.n, CHUNK, world, rank)
        x = wl.make_range(0, lo, hi, device)
        n = hi - lo
        raw_bytes = wl.elem_bytes * n
        for leg in ("no_transfer", "no_online", "no_paged", "no_ablation", "no_workloads"):
            setattr(args, leg, True)  # these legs measure whole workloads
    else:
        x = wl.make(rank, device)  # weak scaling: every rank has its own workload
    assert x.numel() == n
    cb, _ = sz.calibrate(wl.calibration(device), dtype)

    bufs = sz.EncodeBuffers(n, dtype, CHUNK, device=device)
    out = torch.empty(n, dtype=x.dtype, device=device)
    dstatus = torch.zeros(4, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()
    h = stream.cuda_stream
    xp, op, wp, ws = x.data_ptr(), bufs.out.data_ptr(), bufs.ws.data_ptr(), bufs.ws_bytes
    cap = bufs.capacity
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device) if raw_bytes <= L2_BYTES else None

    def check(st, what):
        if st != sz.OK:
            raise sz.SplitZipError(st, what)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        check(sz.splitzip_encode(xp, n, dtype, cb, CHUNK, op, cap, wp, ws, bufs.size.data_ptr(),
                                 bufs.status.data_ptr(), h), "encode")
        if ev is not None:
            ev[1].record(stream)
        # decode bound: the buffer; the header carries the container's real size
        check(sz.splitzip_decode(op, cap, out.data_ptr(), n, dtype, dstatus.data_ptr(), h), "decode")
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize()
    assert int(bufs.status[0]) == sz.OK and int(dstatus[0]) == sz.OK
    verified = bool(torch.equal(out, x))
    blob_size = int(bufs.size[0])
    E = int(bufs.out[24:32].cpu().numpy().view(np.uint64)[0])

    # ---- timed region: K steps, CUDA events around each launch group ----
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for k in range(K):
        if flush is not None:
            flush.fill_(k & 0xFF)  # small inputs: evict them from L2 between steps
        step(evs[k])
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    clk = clocks.stop(t_wall0, t_wall1)
    enc = [e[0].elapsed_time(e[1]) for e in evs]
    dec = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms = evs[0][0].elapsed_time(evs[-1][2]) if flush is None else sum(enc) + sum(dec)
    total_ms = reduce_over_ranks(total_ms, world, device, "max")
    enc_ms, dec_ms = statistics.mean(enc), statistics.mean(dec)
    ms_per_step = total_ms / K
    all_bytes = reduce_over_ranks(raw_bytes * K, world, device, "sum")
    value = all_bytes / (total_ms * 1e-3) / 1e9

    # ---- roofline of the dominant kernel (algorithmic bytes / event time) ----
    # Each call is essentially one streaming kernel (encode adds two short
    # kernels and two small memsets, decode a 4-byte memset, inside the events).
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    alg_encode, alg_decode = wl.algorithmic_bytes(E, n)
    tag = {0: "bf16", 1: "e5m2", 2: "fp16"}[dtype]
    if enc_ms >= dec_ms:
        name, alg, ms = "encode_kernel<%s> (+ index and record kernels)" % tag, alg_encode, enc_ms
    else:
        name, alg, ms = "decode_kernel<%s>" % tag, alg_decode, dec_ms
    achieved = alg / (ms * 1e-3) / 1e9
    slower = "encode" if enc_ms >= dec_ms else "decode"
    traffic, traffic_src = measured_traffic(wl.name if wl.layers in (None, 32) else None, slower)
    roofline = {"bound": "hbm", "kernel": name, "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "peak_source": "%s hbm_gbs (copy)" % peak_kind,
                "algorithmic_bytes_per_launch": alg, "traffic": traffic}
    if traffic_src:
        roofline["traffic_source"] = traffic_src
    per_kernel = {
        "encode": {"ms": round(enc_ms, 4), "alg_bytes": alg_encode,
                   "gbs": round(alg_encode / (enc_ms * 1e-3) / 1e9, 1)},
        "decode": {"ms": round(dec_ms, 4), "alg_bytes": alg_decode,
                   "gbs": round(alg_decode / (dec_ms * 1e-3) / 1e9, 1)},
    }
    enc_gbs = raw_bytes / (enc_ms * 1e-3) / 1e9
    dec_gbs = raw_bytes / (dec_ms * 1e-3) / 1e9
    link = {}
    for L in LINKS_GBS:
        t_plain = raw_bytes / (L * 1e9)
        t_zip = (enc_ms + dec_ms) * 1e-3 + blob_size / (L * 1e9)
        link["%d_GBps" % int(L)] = {"t_uncompressed_ms": round(1e3 * t_plain, 3),
                                    "t_splitzip_ms": round(1e3 * t_zip, 3),
                                    "speedup": round(t_plain / t_zip, 4)}

    # ---- e2e: host pinned input -> H2D -> encode -> decode -> D2H ----
    # The step is cut into chunk-aligned pieces (one per layer on the layered
    # caches), each encoded into its own container and decoded through the C
    # ABI; H2D copies, the codec and D2H copies run on three streams, so piece
    # i's codec overlaps the copies of its neighbours.  Every byte of the
    # step's input crosses H2D and every byte of the decoded tensor crosses
    # D2H inside the timed region.
    e2e = None
    if not args.no_e2e:
        if wl.layered:
            pieces = max(1, n // (wl.n // wl.layers))
        else:
            pieces = int(max(1, min(32, raw_bytes // (64 << 20))))
        piece_n = -(-(-(-n // pieces)) // CHUNK) * CHUNK
        pieces = -(-n // piece_n)
        piece_cap = -(-sz.max_compressed_size(piece_n, dtype, CHUNK) // 16) * 16
        piece_ws = max(sz.workspace_size(piece_n, dtype, CHUNK), 16)
        boxes = torch.empty(pieces * piece_cap, dtype=torch.uint8, device=device)
        pws = torch.empty(piece_ws, dtype=torch.uint8, device=device)
        psize = torch.zeros(2, dtype=torch.int64, device=device)
        pstatus = torch.zeros(4, dtype=torch.int32, device=device)
        x_host = torch.empty(n, dtype=x.dtype, pin_memory=True)
        x_host.copy_(x)
        y_host = torch.empty(n, dtype=x.dtype, pin_memory=True)
        xin = torch.empty_like(x)
        s_in, s_codec, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        hc = s_codec.cuda_stream
        ev_enc = [torch.cuda.Event() for _ in range(pieces)]  # piece i's input consumed
        ev_d2h = [torch.cuda.Event() for _ in range(pieces)]  # piece i's output copied out
        ev_in = [torch.cuda.Event() for _ in range(pieces)]
        ev_dec = [torch.cuda.Event() for _ in range(pieces)]
        started = [False] * pieces
        status_ok = True

        def e2e_step():
            for i in range(pieces):
                lo, hi = i * piece_n, min(n, (i + 1) * piece_n)
                m = hi - lo
                box = boxes.data_ptr() + i * piece_cap
                with torch.cuda.stream(s_in):
                    if started[i]:
                        s_in.wait_event(ev_enc[i])
                    xin[lo:hi].copy_(x_host[lo:hi], non_blocking=True)
                    ev_in[i].record(s_in)
                s_codec.wait_event(ev_in[i])
                check(sz.splitzip_encode(xin.data_ptr() + lo * wl.elem_bytes, m, dtype, cb, CHUNK, box, piece_cap,
                                         pws.data_ptr(), piece_ws, psize.data_ptr(), pstatus.data_ptr(), hc),
                      "encode")
                ev_enc[i].record(s_codec)
                if started[i]:
                    s_codec.wait_event(ev_d2h[i])
                check(sz.splitzip_decode(box, piece_cap, out.data_ptr() + lo * wl.elem_bytes, m, dtype,
                                         dstatus.data_ptr(), hc), "decode")
                ev_dec[i].record(s_codec)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_dec[i])
                    y_host[lo:hi].copy_(out[lo:hi], non_blocking=True)
                    ev_d2h[i].record(s_out)
                started[i] = True

        torch.cuda.synchronize()
        e2e_step()
        torch.cuda.synchronize()
        status_ok = int(pstatus[0]) == sz.OK and int(dstatus[0]) == sz.OK
        # seven timed blocks of e2e_steps steps each; the median block is
        # reported (the host link is shared with the rest of the machine: a
        # block that meets another tenant's transfers takes ~2.5x as long, and
        # two of three blocks did so in one run)
        blocks_ms = []
        for _ in range(E2E_BLOCKS):
            barrier(world)
            ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            ea.record(s_in)
            s_codec.wait_event(ea)
            s_out.wait_event(ea)
            for _ in range(args.e2e_steps):
                e2e_step()
            s_out.wait_event(ev_dec[pieces - 1])
            eb.record(s_out)
            torch.cuda.synchronize()
            blocks_ms.append(reduce_over_ranks(ea.elapsed_time(eb), world, device, "max"))
        e2e_ms = statistics.median(blocks_ms)
        e2e_ok = bool(torch.equal(y_host, x_host)) and status_ok and int(pstatus[0]) == sz.OK and \
            int(dstatus[0]) == sz.OK
        e2e_bytes = reduce_over_ranks(raw_bytes * args.e2e_steps, world, device, "sum")
        e2e = {"value": round(e2e_bytes / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
               "h2d_bytes_per_step": raw_bytes, "d2h_bytes_per_step": raw_bytes,
               "ms_per_step": round(e2e_ms / args.e2e_steps, 3), "verified": e2e_ok,
               "pieces": pieces, "streams": "H2D / codec / D2H",
               "timing": "median of %d blocks of %d steps" % (E2E_BLOCKS, args.e2e_steps),
               "blocks_ms_per_step": [round(b / args.e2e_steps, 3) for b in blocks_ms]}
        del x_host, y_host, xin, boxes, pws

    # ---- transfer: GPU -> pinned host -> GPU through splitzip_transfer, the
    # codec on both ends of the link (compressed) against the raw bytes ----
    transfer = None
    if not args.no_transfer:
        if wl.layered:
            tpieces = wl.layers
        else:
            tpieces = int(max(1, min(32, raw_bytes // (64 << 20))))
        tpiece = -(-(-(-n // tpieces)) // CHUNK) * CHUNK
        y = torch.empty_like(x)
        # compressed and raw transfers alternate, so that both meet the same
        # state of the host link (shared with the machine's other GPUs)
        tbs = {c: sz.TransferBuffers(n, dtype, tpiece, c, CHUNK, device=device) for c in (True, False)}
        for c in (True, False):
            sz.transfer(x, y, cb, tbs[c])  # warm-up
        runs = {True: [], False: []}
        ok_all = True
        for _ in range(TRANSFER_RUNS):
            for c in (True, False):
                y.zero_()
                runs[c].append(sz.transfer(x, y, cb, tbs[c]))
                torch.cuda.synchronize()
                ok_all &= bool(torch.equal(y, x))
        del tbs
        z_ms, z_link = statistics.median(r[0] for r in runs[True]), runs[True][0][1]
        r_ms, r_link = statistics.median(r[0] for r in runs[False]), runs[False][0][1]
        transfer = {"pieces": -(-n // tpiece), "piece_elems": tpiece, "splitzip_ms": round(z_ms, 3),
                    "raw_ms": round(r_ms, 3), "speedup": round(r_ms / z_ms, 4),
                    "link_bytes_each_way": {"splitzip": z_link, "raw": r_link},
                    "raw_link_GBps_each_way": round(r_link / (r_ms * 1e-3) / 1e9, 1), "verified": ok_all,
                    "runs_ms": {"splitzip": [round(r[0], 3) for r in runs[True]],
                                "raw": [round(r[0], 3) for r in runs[False]]},
                    "path": "device -> pinned host -> device copies (cudaMemcpyAsync), encode / D2H / H2D / decode "
                            "on four streams; compressed and raw runs alternate, median of %d each" % TRANSFER_RUNS}
        del y

    # ---- online calibration: histogram + Top-16 on the device, then the
    # encode that reads that codebook, against the offline codebook's encode ----
    online = None
    if not args.no_online:
        hist_d = torch.empty(256, dtype=torch.int64, device=device)
        cb_d = torch.empty(32, dtype=torch.uint8, device=device)

        def online_step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            check(sz.splitzip_calibrate_device(xp, n, dtype, hist_d.data_ptr(), cb_d.data_ptr(), h), "calibrate")
            if ev is not None:
                ev[1].record(stream)
            check(sz.splitzip_encode_device_codebook(xp, n, dtype, cb_d.data_ptr(), CHUNK, op, cap, wp, ws,
                                                     bufs.size.data_ptr(), bufs.status.data_ptr(), h), "encode")
            if ev is not None:
                ev[2].record(stream)

        for _ in range(2):
            online_step()
        torch.cuda.synchronize()
        oevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(10)]
        for ev in oevs:
            if flush is not None:
                flush.fill_(1)
            online_step(ev)
        torch.cuda.synchronize()
        cal_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in oevs)
        oenc_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in oevs)
        on_ok = int(bufs.status[0]) == sz.OK
        on_size = int(bufs.size[0])
        on_E = int(bufs.out[24:32].cpu().numpy().view(np.uint64)[0])
        check(sz.splitzip_decode(op, cap, out.data_ptr(), n, dtype, dstatus.data_ptr(), h), "decode")
        torch.cuda.synchronize()
        on_ok = on_ok and int(dstatus[0]) == sz.OK and bool(torch.equal(out, x))
        online = {"calibrate_ms": round(cal_ms, 4), "encode_ms": round(oenc_ms, 4),
                  "total_ms": round(cal_ms + oenc_ms, 4), "offline_encode_ms": round(enc_ms, 4),
                  "slowdown_vs_offline": round((cal_ms + oenc_ms) / enc_ms, 4),
                  "escape_rate": round(on_E / n, 6), "ratio": round(raw_bytes / on_size, 5),
                  "codebook": [int(v) for v in cb_d[1:17].cpu().tolist()], "verified": on_ok,
                  "what": "per-tensor codebook calibrated on the device from the encoded tensor itself"}

    # ---- paged KV: the workload as a pool of 16,384-element pages (16 tokens
    # x 8 heads x 128 of one layer's K or V), encoded from a shuffled page
    # table and decoded into another shuffled one ----
    paged = None
    page_elems = 16384
    if not args.no_paged and n % page_elems == 0 and n // page_elems >= 2:
        pool_pages = n // page_elems
        g = torch.Generator()
        g.manual_seed(11)
        src_pages = torch.randperm(pool_pages, generator=g).to(torch.int32).to(device)
        dst_pages = torch.randperm(pool_pages, generator=g).to(torch.int32).to(device)

        def paged_step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            check(sz.splitzip_encode_paged(xp, pool_pages, src_pages.data_ptr(), pool_pages, page_elems, dtype, cb,
                                           CHUNK, op, cap, wp, ws, bufs.size.data_ptr(), bufs.status.data_ptr(), h),
                  "encode_paged")
            if ev is not None:
                ev[1].record(stream)
            check(sz.splitzip_decode_paged(op, cap, out.data_ptr(), pool_pages, dst_pages.data_ptr(), pool_pages,
                                           page_elems, dtype, dstatus.data_ptr(), h), "decode_paged")
            if ev is not None:
                ev[2].record(stream)

        for _ in range(2):
            paged_step()
        torch.cuda.synchronize()
        pevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(10)]
        for ev in pevs:
            if flush is not None:
                flush.fill_(2)
            paged_step(ev)
        torch.cuda.synchronize()
        penc = statistics.mean(e[0].elapsed_time(e[1]) for e in pevs)
        pdec = statistics.mean(e[1].elapsed_time(e[2]) for e in pevs)
        p_ok = int(bufs.status[0]) == sz.OK and int(dstatus[0]) == sz.OK and bool(torch.equal(
            out.view(pool_pages, page_elems)[dst_pages.long()], x.view(pool_pages, page_elems)[src_pages.long()]))
        paged = {"page_elems": page_elems, "pages": pool_pages, "page_tables": "two seeded random permutations",
                 "encode_ms": round(penc, 4), "decode_ms": round(pdec, 4),
                 "encode_gbs": round(raw_bytes / (penc * 1e-3) / 1e9, 2),
                 "decode_gbs": round(raw_bytes / (pdec * 1e-3) / 1e9, 2),
                 "vs_contiguous": {"encode": round(enc_ms / penc, 4), "decode": round(dec_ms / pdec, 4)},
                 "verified": p_ok}

    # ---- ablation formats: Top-16 / Top-8 / Top-15 + sentinel through one
    # plain kernel family (their differences are the formats'), next to the
    # production Top-16 kernels ----
    ablation = None
    if not args.no_ablation:
        ablation = {"kernels": "one plain kernel family for the three formats (no TMA ring); "
                               "production Top-16 decode: %.4f ms" % dec_ms}
        for variant, label in ((sz.ABL_TOP16, "top16"), (sz.ABL_TOP8, "top8"), (sz.ABL_TOP15_SENTINEL, "top15_sentinel")):
            vcb = sz.ablation_codebook(cb, variant)
            acap = sz.ablation_max_size(n, dtype, variant, CHUNK)

            def abl_step(ev=None):
                if ev is not None:
                    ev[0].record(stream)
                check(sz.splitzip_ablation_encode(xp, n, dtype, vcb, CHUNK, variant, op, acap, bufs.size.data_ptr(),
                                                  bufs.status.data_ptr(), h), "ablation encode")
                if ev is not None:
                    ev[1].record(stream)
                check(sz.splitzip_ablation_decode(op, acap, out.data_ptr(), n, dtype, variant, dstatus.data_ptr(),
                                                  h), "ablation decode")
                if ev is not None:
                    ev[2].record(stream)

            abl_step()
            torch.cuda.synchronize()
            aevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(5)]
            for ev in aevs:
                if flush is not None:
                    flush.fill_(3)
                abl_step(ev)
            torch.cuda.synchronize()
            aenc = statistics.mean(e[0].elapsed_time(e[1]) for e in aevs)
            adec = statistics.mean(e[1].elapsed_time(e[2]) for e in aevs)
            asize = int(bufs.size[0])
            aE = int(bufs.out[24:32].cpu().numpy().view(np.uint64)[0])
            a_ok = int(bufs.status[0]) == sz.OK and int(dstatus[0]) == sz.OK and bool(torch.equal(out, x))
            ablation[label] = {"encode_ms": round(aenc, 4), "decode_ms": round(adec, 4),
                               "encode_gbs": round(raw_bytes / (aenc * 1e-3) / 1e9, 1),
                               "decode_gbs": round(raw_bytes / (adec * 1e-3) / 1e9, 1),
                               "escape_rate": round(aE / n, 6), "ratio": round(raw_bytes / asize, 5),
                               "verified": a_ok}
        for label in ("top8", "top15_sentinel"):
            ablation[label]["decode_slowdown_vs_top16"] = round(ablation[label]["decode_ms"] /
                                                                ablation["top16"]["decode_ms"], 3)

    # ---- CPU oracle on a bounded sample (rank 0 only) ----
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cores = args.ref_threads or host_cores()
        gbs, elems, secs, distinct, block = oracle_throughput(x, dtype, cb.values(), args.cpu_seconds, cores)
        gbs1, elems1, secs1, distinct1, block1 = oracle_throughput(x, dtype, cb.values(), args.cpu_seconds / 2, 1)
        what = "encode+decode+check, scalar C oracle, containers of %d elements"
        cpu = {"value": round(gbs, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": "%d elements in %.1f s: passes over the first %d elements (%d chunks) of the workload, "
                         "%s, %d thread(s), one container each at a time" % (
                             elems, secs, distinct, distinct // CHUNK, what % block, cores),
               "single_thread": {"value": round(gbs1, 5), "cores": 1,
                                 "sample": "%d elements in %.1f s: passes over the first %d elements, %s" % (
                                     elems1, secs1, distinct1, what % block1)}}

    # ---- shards: where this rank's records start in the joined container
    # (an exclusive scan of the per-rank escape totals) and its size ----
    shard = None
    if args.shard:
        base, E_all = exclusive_scan_over_ranks(E, world, rank, device)
        joined = sz.compressed_size(wl.n, dtype, CHUNK, E_all)
        shard = {"elements": n, "range": list(shard_range(wl.n, CHUNK, world, rank)), "escape_base": base,
                 "joined_escapes": E_all, "joined_bytes": joined, "joined_ratio": round(wl.elem_bytes * wl.n / joined, 5)}

    # ---- batches: 32 per-layer K tiles of 1,048,576 elements (the kv-tile
    # recipe, seeds 0..31) as 32 single encode + decode calls against one
    # batched encode and one batched decode (L2 flushed before each step) ----
    batch = None
    if not args.no_batch and not args.shard:
        batch = measure_batch(dtype if dtype != 1 else 0, device, args.warmup)

    # ---- the other workloads (one line carries all five), timed after the
    # headline's buffers are released ----
    workloads = None
    if not args.no_workloads and wl.name == DEFAULT_WORKLOAD and wl.layers == 32:
        del x, out, bufs
        torch.cuda.empty_cache()
        workloads = {}
        for other in ("kv_tile_1x1024x8x128_bf16", "llama_layer_2x8192x8x128_bf16",
                      "escape_stress_64x65536_bf16", "kv_cache_32x2x65536x8x128_e5m2",
                      "kv_cache_32x2x32768x8x128_fp16"):
            workloads[other] = measure_workload(other, args.workload_steps, args.warmup, device, hbm)

    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "strong" if args.shard else "weak", "vs_baseline": None,
        "dtype": "u8" if dtype == 1 else "u16",
        "data": "synthetic (seeded torch CPU generator, rounded on the GPU; recipe of the workload module)",
        "config": wl.config(world, args.shard), "shard": shard,
        "encode_gbs": round(enc_gbs, 2), "decode_gbs": round(dec_gbs, 2),
        "encode_hbm_frac": round(alg_encode / (enc_ms * 1e-3) / 1e9 / hbm, 4),
        "decode_hbm_frac": round(alg_decode / (dec_ms * 1e-3) / 1e9 / hbm, 4),
        "ratio": round(raw_bytes / blob_size, 5), "compressed_bytes": blob_size, "escapes": E,
        "escape_rate": round(E / n, 6), "verified_bit_exact": verified,
        "per_kernel": per_kernel, "link_model": link,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
        "transfer": transfer, "online_calibration": online, "paged": paged, "ablation": ablation,
        "workloads": workloads, "batch": batch,
        "gpu_launches": 5 * K,  # timed steps: encode (streaming, group, index, records kernels) + decode
    }


def main():
    faulthandler.enable()  # a native crash prints the Python stack of every thread
    args = parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
