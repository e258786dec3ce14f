"""The N > 1 bench path on CPU: two ranks on the gloo backend.

The decode path has no cross-GPU exchange, so N GPUs run N independent replicas; what the
multi-process code owns is the rendezvous, the barrier around the timed region, the max of the
step time over ranks and the whole-job aggregate.  These tests run that host logic with
world_size 2 and no GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank reports its own step time; every rank must see the slowest one
    ms = bench.max_over_ranks(1.25 + 0.5 * rank, w)
    bench.barrier(w)
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"max_ms": ms}, f)
    dist.destroy_process_group()


def test_gloo_world2_barrier_and_max(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        with open(tmp_path / ("rank%d.json" % r)) as f:
            assert json.load(f)["max_ms"] == pytest.approx(1.75)


def test_aggregate_is_sum_over_slowest():
    sys.path.insert(0, ROOT)
    import bench
    b = 68_157_440  # K/V bytes of one decode_32k step
    one = bench.aggregate_gbs(b, 0.02, 1)
    assert one == pytest.approx(b / 0.02e-3 / 1e9)
    # two replicas, the slower taking 0.025 ms: twice the bytes over the slower time
    assert bench.aggregate_gbs(b, 0.025, 2) == pytest.approx(2 * b / 0.025e-3 / 1e9)
    assert bench.aggregate_gbs(b, 0.02, 4) == pytest.approx(4 * one)


def test_reference_arm_under_torchrun_world2():
    """`bench.py --impl reference` launched like the N = 2 driver run: rank 0 alone times the
    oracle and prints one JSON line; rank 1 exits 0 without work."""
    env = dict(os.environ, KVQ_REF_HEADS="1", CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference"
    assert res["n_gpus"] == 2
    assert res["value"] > 0 and res["e2e"]["value"] == res["value"]
    assert res["cpu_baseline"]["kind"] == "oracle"
