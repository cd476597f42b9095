"""The multi-rank timing logic of bench.py on CPU: two gloo ranks, each with
its own timings; both must see the element-wise maximum, and the job
throughput counts the work of every rank against the slowest rank's time."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
    got = bench.max_over_ranks(mine, dist)
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == [2.0, 5.0, 0.5]


def test_job_throughput_and_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], None) == [3.0, 4.0]
    # 2 ranks x 1e9 units in 2 ms (slowest rank) -> 1e12 units/s
    assert bench.job_throughput(1e9, 2, 2.0) == pytest.approx(1e12)
    assert bench.visible_pairs(4, 4) == 10            # square causal: 1+2+3+4
    assert bench.visible_pairs(2, 5) == 4 + 5         # delta = 3: rows see 4 and 5 keys
    assert bench.visible_pairs(5, 2) == 0 + 0 + 0 + 1 + 2


def test_reference_arm_under_torchrun_prints_one_line():
    """`bench.py --impl reference` launched as two ranks: rank 0 alone times
    the oracle and prints one JSON line; the other rank exits 0 without
    output."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
