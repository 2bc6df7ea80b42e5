"""Multi-rank host logic of bench.py, on CPU with the gloo backend (two ranks).

bench.py runs one replica of the workload per GPU: the timed region is the
maximum over ranks, and the whole-job time per call divides it by the number of
calls all ranks made. The reference arm prints from rank 0 only; the other ranks
exit 0 without work.
"""
import json
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # Rank r measured 10 (r + 1) ms for 100 calls of its replica.
        res = bench.aggregate_ranks(10.0 * (rank + 1), 100, world)
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(list(res), f)


def test_timed_region_is_max_over_ranks_and_value_is_per_whole_job_call(tmp_path):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        ms, us_per_call, value = json.load(open(tmp_path / f"rank{rank}.json"))
        assert ms == 20.0              # the slower rank
        assert us_per_call == 200.0    # 20 ms / 100 calls
        assert value == 100.0          # 2 x 100 calls in 20 ms


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_ranks(5.0, 50, 1) == (5.0, 100.0, 100.0)


def test_reference_arm_prints_from_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "2", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
