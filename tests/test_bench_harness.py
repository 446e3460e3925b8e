"""The benchmark harness on CPU: the rank reduction of a replica run over
gloo (world size 2), and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    t, u = bench.aggregate(10.0 + 5.0 * rank, 100 * (rank + 1), ws, torch.device("cpu"))
    out[rank] = (t, u)
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    # the slowest rank's time and the units of both ranks, on every rank
    assert res[0] == res[1] == (15.0, 300.0)


def test_aggregate_single_rank_is_identity():
    assert bench.aggregate(3.5, 7, 1, None) == (3.5, 7.0)


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--layers", "4"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["steps"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    # the 4 sampled layers run on at most 4 threads
    assert line["cpu_baseline"]["kind"] == "oracle" and 1 <= line["cpu_baseline"]["cores"] <= 4


def test_threaded_oracle_step_equals_sequential():
    # the cpu_baseline runs the oracle's layers on a thread pool: the results
    # must be those of the sequential loop, bit for bit
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    from speculative_decode_hybrid_gb300 import workloads as W
    oracle.build()
    wl = W.make_workload(0, seed=3, layers=6)
    layers = list(range(6))
    seq = oracle.verify_request(wl, 0, layers=layers)
    with ThreadPoolExecutor(max_workers=4) as pool:
        par = list(pool.map(lambda y: oracle.verify_request(wl, 0, layers=[y])[0], layers))
    for a, b in zip(seq, par):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
    # and the full step (verify + accept + restore) runs through the pool
    with ThreadPoolExecutor(max_workers=4) as pool:
        k_pool = bench.oracle_full_step(wl, layers, pool=pool)
    assert k_pool == bench.oracle_full_step(wl, layers)


def test_recorded_traffic_is_per_workload_and_kernel():
    # each committed capture names its workload, layers, verify kind and
    # sources; the traffic is reported only for that configuration, and only
    # while the sources hash to the recorded value
    seen = set()
    for path in bench.TRAFFIC_FILES:
        vals = bench.read_traffic_file(path)
        key = (int(vals["workload"]), int(vals["layers"]), vals["verify"])
        assert key not in seen
        seen.add(key)
        got = bench.recorded_traffic(*key)
        fresh = vals["source_sha256"] == bench.sources_sha(vals["sources"].split())
        assert got == (int(vals["dram_bytes_per_launch"]) if fresh else None)
        assert int(vals["dram_bytes_per_launch"]) == int(vals["dram_bytes_read"]) + int(vals["dram_bytes_write"])
    assert bench.recorded_traffic(4, 48, "checkpoint") is None
    assert bench.recorded_traffic(2, 12, "checkpoint") is None
