"""Host side of bench.py's multi-GPU mode (independent replicas, no
collective on the data path), run as two gloo ranks on the CPU: rank/world
discovery, the barriers around the timed region, the max over ranks of the
elapsed time, whole-job throughput, and the reference arm printing on rank 0
only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo")
    try:
        got = bench.dist_setup()
        bench.barrier(torch, got[0])
        slowest = bench.max_over_ranks(torch, got[0], 1.5 + rank, "cpu")
        bench.barrier(torch, got[0])
        with open(os.path.join(outdir, "rank%d.json" % rank), "w") as f:
            json.dump({"setup": list(got), "max": slowest}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        with open(tmp_path / ("rank%d.json" % rank)) as f:
            r = json.load(f)
        assert r["setup"] == [world, rank, rank]
        assert r["max"] == pytest.approx(1.5 + world - 1)


def test_replica_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # the headline step: W 33,030,144 B + x 57,344 B + y 16,384 B = 33,103,872 B
    step = bench.gemv_bytes("q4_0", 4096, 14336, 1)
    assert step == 33_030_144 + 4 * 14336 + 4 * 4096 == 33_103_872
    one = bench.replica_value(step, 1000, 1, 0.0128)
    two = bench.replica_value(step, 1000, 2, 0.0128)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(33_103_872 * 1000 / 0.0128 / 1e9)


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
