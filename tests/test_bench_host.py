"""Host-side pieces of bench.py: the traffic figures and their source hashes."""
import os

import bench


def test_traffic_entries_name_existing_profiles_and_sources():
    for (workload, op), t in bench.TRAFFIC.items():
        assert op in ("encode", "decode")
        assert os.path.isfile(os.path.join(bench.ROOT, t["profile"]))
        assert t["bytes"] > 0 and len(t["sha256"]) == 64
        bench.sources_sha256(t["sources"])  # every source file exists


def test_traffic_reported_only_for_the_captured_sources(monkeypatch):
    key = next(iter(bench.TRAFFIC))
    t = bench.TRAFFIC[key]
    monkeypatch.setattr(bench, "sources_sha256", lambda names: t["sha256"])
    assert bench.measured_traffic(*key) == (t["bytes"], t["profile"])
    monkeypatch.setattr(bench, "sources_sha256", lambda names: "0" * 64)
    assert bench.measured_traffic(*key) == (None, None)
    assert bench.measured_traffic("no_such_workload", "encode") == (None, None)


def test_threaded_oracle_round_trips_check_every_container(monkeypatch):
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np
    import oracle
    from lossless_kv_cache_gb300 import workloads as W

    x = W.escape_stress(5, chunks=5, chunk_elems=4096).numpy().view(np.uint16)
    cb = oracle.calibrate(oracle.histogram(x, oracle.BF16), oracle.BF16)
    blocks = [x[i: i + 6000] for i in range(0, x.size, 6000)]  # ragged last block
    with ThreadPoolExecutor(3) as pool:
        assert bench.oracle_round_trips(pool, blocks, oracle.BF16, cb) > 0
        real = oracle.decode

        def flip_last(blob, n, dtype):  # a planted mistake in the oracle's decode
            y = real(blob, n, dtype).copy()
            y[-1] ^= 1
            return y

        monkeypatch.setattr(oracle, "decode", flip_last)
        try:
            bench.oracle_round_trips(pool, blocks, oracle.BF16, cb)
        except RuntimeError as e:
            assert "round trip" in str(e)
        else:
            raise AssertionError("a wrong round trip went unnoticed")


def test_reference_arm_uses_the_requested_threads(capsys):
    import sys
    argv = ["bench.py", "--impl", "reference", "--workload", "escape_stress_64x65536_bf16",
            "--steps", "2", "--warmup", "1", "--ref-threads", "2"]
    old = sys.argv
    sys.argv = argv
    try:
        args = bench.parse_args()
    finally:
        sys.argv = old
    line = bench.run_reference(args, 1, 0)
    assert line["impl"] == "reference" and line["cpu_baseline"]["cores"] == 2
    assert line["value"] == line["cpu_baseline"]["value"] == line["e2e"]["value"] > 0
    assert "2 thread(s)" in line["cpu_baseline"]["sample"]


def test_oracle_containers_shrink_so_every_thread_has_one():
    C = bench.CHUNK
    assert bench.oracle_block(1 << 30, 16) == 16 * C
    assert bench.oracle_block(16 * C, 16) == C          # one chunk each
    assert bench.oracle_block(64 * C, 16) == 4 * C
    assert bench.oracle_block(C // 2, 16) == C          # never below one chunk
    assert bench.oracle_block(100 * C, 1) == 16 * C


def test_cpu_baseline_helper_on_host_bits():
    from lossless_kv_cache_gb300 import workloads as W
    import oracle
    x = W.escape_stress(6, chunks=8, chunk_elems=65536)  # raw BF16 bits
    cb = oracle.calibrate(oracle.histogram(x.numpy().view("uint16"), oracle.BF16), oracle.BF16)
    gbs, done, secs, distinct, block = bench.oracle_throughput(x, 0, cb, 0.01, 4)
    assert block == 2 * bench.CHUNK and distinct == x.numel() and done % distinct == 0
    assert gbs > 0 and secs > 0


def test_reference_arm_runs_on_rank_0_only():
    import sys
    old = sys.argv
    sys.argv = ["bench.py", "--impl", "reference", "--workload", "escape_stress_64x65536_bf16"]
    try:
        args = bench.parse_args()
    finally:
        sys.argv = old
    assert bench.run_reference(args, 2, 1) is None  # rank 1 of 2: no work, no line


def test_traffic_table_agrees_with_its_profiles():
    # the per-operation DRAM traffic that each launch-list profile prints (MB,
    # one decimal) is the figure the bench line reports
    for (workload, op), t in bench.TRAFFIC.items():
        with open(os.path.join(bench.ROOT, t["profile"])) as f:
            lines = f.readlines()
        header = [c.strip() for c in next(l for l in lines if l.startswith("| call |")).split("|")]
        col = header.index("DRAM traffic MB")
        rows = [line.split("|") for line in lines if line.startswith("| %s" % op)]
        assert len(rows) == 1, (workload, op)
        printed = float(rows[0][col].strip().split()[0].replace(",", ""))
        assert printed == round(t["bytes"] / 1e6, 1), (workload, op, printed, t["bytes"])
