"""Multi-process replica path of bench.py on CPU (gloo, world size 2).

Under torchrun every rank runs the full workload on its own GPU and the job's
time is the slowest rank's.  This checks the rank aggregation (all-reduce MAX
over a real process group) and that the reference arm runs on rank 0 only.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as tdist
    import bench
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [100.0, 150.0][rank]
    value, max_ms = bench.replica_throughput(local_ms, 1e12, 10, world,
                                             bench.reduce_max_fn(world, "cpu"))
    results[rank] = (value, max_ms)
    tdist.barrier()
    tdist.destroy_process_group()


def test_replica_throughput_max_over_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    expect = world * 1e12 * 10 / 0.150 / 1e12
    for rank in range(world):
        value, max_ms = res[rank]
        assert max_ms == 150.0
        assert value == pytest.approx(expect)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    value, max_ms = bench.replica_throughput(50.0, 2e12, 4, 1, bench.reduce_max_fn(1))
    assert max_ms == 50.0 and value == pytest.approx(2e12 * 4 / 0.05 / 1e12)


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_one_json_line():
    import json
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
