"""The bench's multi-rank host logic on CPU: two gloo ranks (the layout the
bench runs under torchrun, one process per GPU, replicas with no data-path
collective). Checks the barrier, the max over ranks that sets the job's pace,
the whole-job aggregate, and that only rank 0 runs and prints the CPU
reference arm."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup(None)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # rank r took 1 + r ms per step: the job runs at the slowest rank's pace
    value, ms = bench.whole_job_tflops(w, 2e9, 1.0 + rank)
    assert ms == float(world)
    assert abs(value - world * 2e9 / (world * 1e-3) / 1e12) < 1e-9
    # reference arm: rank 0 alone does the (stubbed) CPU work and returns a line
    bench.cpu_baseline = lambda wl, budget: {"value": 1.0, "seconds": 0.01, "sample": "stub"}

    class A:
        workload, steps, warmup = "gpt2_small", 2, 3
    res = bench.run_reference(A, w, r)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write("none" if res is None else f"{res['impl']} {res['n_gpus']} {res['value']}")
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    assert (tmp_path / "rank0.txt").read_text() == "reference 2 1.0"
    assert (tmp_path / "rank1.txt").read_text() == "none"
