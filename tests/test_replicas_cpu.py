"""Host logic of the multi-GPU bench on the CPU: N independent replicas under
torchrun, joined only by a gloo group for barriers and the max over ranks of
the timings (no collective on the data path).  Two gloo ranks, no GPU."""

import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    # rank r's own timings: total ms and host seconds
    mine = [10.0 + 5.0 * rank, 3.0 - rank]
    got = bench.max_over_ranks(mine, world)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(" ".join(repr(v) for v in got))


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        vals = [float(v) for v in (tmp_path / f"rank{r}.txt").read_text().split()]
        assert vals == [15.0, 3.0], f"rank {r} saw {vals}"


def test_whole_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench

    # 64 tokens per replica, 2 ms per step (slowest replica), 4 replicas
    assert bench.replica_throughput(64, 4, 2.0) == 64 * 4 / 2e-3
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
