"""Multi-rank host logic of bench.py, run as two gloo ranks on the CPU.

The layer shards by request and KV group with no exchange step, so several GPUs run
independent replicas ("weak" scaling). What the ranks share is host logic: the job's time is
the slowest rank's (a max all-reduce), the job's throughput counts every rank's replica, and
the reference arm works and prints on rank 0 only.
"""
import contextlib
import io
import os
import socket
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, ws: int, port: int, out):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        # rank r measured [1 + r, 10 - r, 5]: the job sees the max of each
        vals = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 5.0], ws, torch.device("cpu"))
        thr = bench.job_throughput(1000.0, vals[0], ws)
        printed = ""
        if rank != 0:
            # the reference arm returns at once, without work or output, on ranks other than 0
            buf = io.StringIO()
            with contextlib.redirect_stdout(buf):
                bench.run_reference(None, ws, rank, 0)
            printed = buf.getvalue()
        torch.distributed.barrier()
        out.put((rank, vals, thr, printed))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_every_replica():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(ws):
        rank, vals, thr, printed = q.get(timeout=120)
        results[rank] = (vals, thr, printed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(ws):
        vals, thr, printed = results[rank]
        assert vals == [2.0, 10.0, 5.0]
        # 1000 units per rank, 2 ranks, 2 ms: 1e6 units/s
        assert abs(thr - 1.0e6) < 1e-6
    assert results[1][2] == ""


def test_one_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks([3, 4.5], 1, torch.device("cpu")) == [3.0, 4.5]
    assert bench.job_throughput(10.0, 5.0, 1) == 2000.0


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` on one rank: the oracle timed on the host cores, one JSON
    line with the keys the benchmark contract asks of the reference arm."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
