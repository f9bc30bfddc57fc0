"""The multi-rank (N > 1) path of bench.py on CPU with the gloo backend and two
ranks: each rank draws its own pack (no data-path collective), the step time is
the maximum over ranks and the work the sum, and the reference arm runs on rank 0
only."""
import json
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


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = bench.rank_workload("mixed_50k", 0, rank, budget=6000)
        # each rank reports a different step time and its own pack's work
        ms = 10.0 + 5.0 * rank
        got = bench.reduce_over_ranks(ms, wl.flops_fwd(), world)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"specs": wl.specs, "flops": wl.flops_fwd(), "got": got}, f)
    finally:
        dist.destroy_process_group()


def test_two_rank_reduction_and_independent_packs(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn")
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    assert r[0]["specs"] != r[1]["specs"]                      # each rank its own pack
    assert r[0]["got"] == r[1]["got"]                          # every rank sees the same totals
    ms_max, flops_all = r[0]["got"]
    assert ms_max == 15.0                                      # max over ranks
    assert flops_all == pytest.approx(r[0]["flops"] + r[1]["flops"], rel=1e-12)


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.5, 7.0, 1) == (3.5, 7.0)


def test_rank_packs_are_deterministic():
    sys.path.insert(0, ROOT)
    import bench
    a = bench.rank_workload("mixed_50k", 0, 1, budget=8000)
    b = bench.rank_workload("mixed_50k", 0, 1, budget=8000)
    assert a.specs == b.specs


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
