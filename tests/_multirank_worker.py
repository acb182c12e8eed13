"""One rank of the multi-process check of bench.py's N>1 logic (gloo on the host).

Launched by tests/test_multirank.py through torch.distributed.run; every check
is an assert, so a wrong rank exits non-zero and fails the launch.
"""
import argparse
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main() -> None:
    dist.init_process_group("gloo")
    rank, world, local = bench._dist_env()
    assert dist.get_rank() == rank and dist.get_world_size() == world and world >= 2
    # the slowest rank's step time decides the job's time; a sum sees every rank
    local_ms = 1.0 + 0.5 * rank
    slowest = bench.max_over_ranks(local_ms)
    assert slowest == 1.0 + 0.5 * (world - 1), slowest
    assert bench.sum_over_ranks(float(rank + 1)) == world * (world + 1) / 2
    bench.barrier()
    # weak scaling: every rank processed its own batch, so the job moved world x the bytes
    per_rank = 582_307_988.0
    value = bench.job_throughput(per_rank, slowest, world)
    assert abs(value - per_rank * world / (slowest * 1e-3) / 1e9) < 1e-9
    agreed = bench.max_over_ranks(value)
    assert agreed == value                      # every rank computed the same number
    # the reference arm: only rank 0 works and prints; the others return at once
    if rank != 0:
        bench.run_reference(argparse.Namespace(steps=1, warmup=3))
    bench.barrier()
    if rank == 0:
        print(f"MULTIRANK_OK world={world} value={value:.3f}", flush=True)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
