"""Multi-rank path on CPU: two gloo ranks.

The codec shards by whole chunks with no data exchange: each rank encodes its
own chunk range (bench.shard_range, as bench.py --shard does), and the only
cross-rank steps are the barrier, the max/sum reductions bench.py uses for
its timing and byte totals, and the exclusive scan of the per-rank escape
totals that places each rank's records in the joined container.  This test
runs those steps on two processes, encodes each rank's range with the CPU
oracle (no GPU here), and joins the gathered per-rank containers with the
library's splitzip_merge: the result must be the single-rank container, byte
for byte.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    import oracle
    from lossless_kv_cache_gb300 import workloads as W

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    mx = bench.reduce_over_ranks(float(rank + 1), w, "cpu", "max")
    sm = bench.reduce_over_ranks(float(rank + 1), w, "cpu", "sum")

    chunk = 4096
    x = W.escape_stress(0, chunks=6, chunk_elems=chunk, sigma=2.0).numpy().view(np.uint16)[:6 * chunk - 100]
    cb = oracle.calibrate(oracle.histogram(x, 0), 0)
    lo, hi = bench.shard_range(x.size, chunk, w, r)  # whole chunks per rank
    mine = oracle.encode(x[lo:hi], 0, cb, chunk)
    E_mine = oracle.parse_header(mine)[1].total_escapes
    base, E_all = bench.exclusive_scan_over_ranks(E_mine, w, r, "cpu")
    blobs = [None] * w
    dist.all_gather_object(blobs, mine)
    results[rank] = (mx, sm, blobs if rank == 0 else None, x if rank == 0 else None, cb, (lo, hi, E_mine, base, E_all))
    dist.destroy_process_group()


def _sections(blob):
    import oracle
    st, h = oracle.parse_header(blob)
    assert st == oracle.OK
    C, n, E = h.n_chunks, h.n, h.total_escapes
    a16 = lambda v: (v + 15) // 16 * 16
    nib = a16(64 + 12 * C)
    sm = nib + a16((n + 1) // 2)
    rec = sm + a16(n)
    return dict(n=n, C=C, E=E, counts=blob[64 + 8 * C: 64 + 12 * C].view(np.uint32),
                nib=blob[nib: nib + (n + 1) // 2], sm=blob[sm: sm + n], rec=blob[rec: rec + 3 * E])


@pytest.mark.timeout(300)
def test_two_gloo_ranks_reduce_and_shard():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(240)
        assert p.exitcode == 0
    mx, sm, blobs, x, cb, scan0 = results[0]
    scan1 = results[1][5]
    assert (mx, sm) == (2.0, 3.0) and results[1][:2] == (2.0, 3.0)
    # the ranks' ranges tile the tensor; the scan gives each rank its record base
    assert scan0[0] == 0 and scan0[1] == scan1[0] and scan1[1] == x.size
    assert scan0[3] == 0 and scan1[3] == scan0[2] and scan0[4] == scan1[4] == scan0[2] + scan1[2]

    import oracle
    import lossless_kv_cache_gb300 as sz
    whole_blob = oracle.encode(x, 0, cb, 4096)
    np.testing.assert_array_equal(sz.merge(blobs), whole_blob)
    whole = _sections(whole_blob)
    parts = [_sections(b) for b in blobs]
    assert whole["E"] == sum(p["E"] for p in parts)
    np.testing.assert_array_equal(whole["counts"], np.concatenate([p["counts"] for p in parts]))
    np.testing.assert_array_equal(whole["nib"], np.concatenate([p["nib"] for p in parts]))
    np.testing.assert_array_equal(whole["sm"], np.concatenate([p["sm"] for p in parts]))
    np.testing.assert_array_equal(whole["rec"], np.concatenate([p["rec"] for p in parts]))
